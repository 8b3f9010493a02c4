// The decode block: input preparation, the h1 finalisation between O and
// gate/up, and the host-side orchestration of the seven kernels (prep, QKV,
// attention, O, mid, gate/up, down) on the caller's stream, chained with
// programmatic dependent launch so each projection's weight stream starts while
// its predecessor finishes.
#include <algorithm>
#include <cmath>

#include "ft_block.cuh"

namespace ft {

// Encodes 8 consecutive inputs 8 ch .. 8 ch + 7 of row t into the grouped
// operand buffer `op` of B rows (op_index) and returns their contribution to
// the group offset S.
__device__ __forceinline__ float encode_chunk8(const float (&v)[8], int ch, int t, int B, __half* op) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float s0, s1;
    const int k = 8 * ch + 2 * i;  // k and k + 1 share one 8-value chunk of the row
    const __half h0 = op_encode(v[2 * i], k, s0);
    const __half h1 = op_encode(v[2 * i + 1], k + 1, s1);
    *reinterpret_cast<__half2*>(op + op_index(t, k, B)) = __halves2half2(h0, h1);
    s += s0 + s1;
  }
  return s;
}

// Sums a per-thread value over the 16 consecutive threads that hold one group
// (16 chunks of 8 = 128 inputs) and returns it in every lane of the 16.
__device__ __forceinline__ float group16_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Loads chunk ch (inputs 8 ch .. 8 ch + 7) of a BF16 or FP32 row.
__device__ __forceinline__ void load_chunk8(const void* row, int dtype, int ch, float (&v)[8]) {
  if (dtype == FT_F32) {
    const float4* src = reinterpret_cast<const float4*>(row) + 2 * ch;
    const float4 a = __ldcg(src), d = __ldcg(src + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = d.x; v[5] = d.y; v[6] = d.z; v[7] = d.w;
  } else {
    const uint4 a = __ldcg(reinterpret_cast<const uint4*>(row) + ch);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// One row part: chunk ch of the row -> FP32 copy, FP16 operand + group offsets,
// and the part's sum of squares (written by thread 0).  kPrepThreads threads,
// one chunk each; a part is a whole number of 128-input groups.
__device__ __forceinline__ bool row_part(const float (&v)[8], bool valid, int ch, int b, int B, float* copy,
                                         __half* op, sfix_t* s_grp, float* ssq_out) {
  __shared__ float red[kPrepThreads / 32];
  float ss = 0.0f, sterm = 0.0f;
  bool bad = false;
  if (valid) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ss = fmaf(v[k], v[k], ss);
      bad |= !(fabsf(v[k]) <= 65504.0f);
    }
    if (copy) {
      float4* dst = reinterpret_cast<float4*>(copy) + 2 * ch;
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    sterm = encode_chunk8(v, ch, b, B, op);
  }
  // warps stay converged: a group is 16 chunks and parts start on group boundaries
  const float gs = group16_sum(sterm);  // fixed shuffle order: deterministic
  if (valid && (ch & 15) == 0) s_grp[(ch >> 4) * 32 + b] = f32_to_sfix(gs);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kPrepThreads / 32; ++w) t += red[w];
    *ssq_out = t;
  }
  return bad;
}

// Block input -> QKV operand + offsets, partial sums of x^2 (the consumers form
// rho1 from them and apply it after the QKV accumulation, summary page
// "어떻게 동작하나"), an FP32 copy of x (the residual), and this call's
// accumulators cleared.  Grid (parts, B).
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepParams p) {
  griddep_launch();  // the QKV kernel may start streaming its weights
  griddep_wait();    // the previous kernel may have produced x_in or still read the workspace
  const int part = blockIdx.x, parts = gridDim.x, b = blockIdx.y, tid = threadIdx.x;
  const int first = part * kPrepThreads + tid, step = parts * kPrepThreads;
  for (int i = first; i < p.nkg_o; i += step) p.s_o[i * 32 + b] = 0;
  for (int i = first; i < p.nkg_a; i += step) p.s_a[i * 32 + b] = 0;
  if (b == 0)
    for (int i = first; i < p.ntick; i += step) p.tick[i] = 0u;
  const int ch = first;
  const bool valid = ch < p.H / 8;
  float v[8];
  const size_t esz = p.act_dtype == FT_F32 ? 4 : 2;
  if (valid) load_chunk8(static_cast<const uint8_t*>(p.x_in) + (size_t)b * p.H * esz, p.act_dtype, ch, v);
  const bool bad =
      row_part(v, valid, ch, b, p.B, p.xres + (size_t)b * p.H, p.x_h, p.s_x, p.ssq + b * parts + part);
  if (bad) set_status(p.status, FT_DEV_RANGE);
}

// h1 = x + the O projection (its pieces' slabs added in slab order) -> h1,
// the gate/up operand + offsets and partial sums of h1^2 (rho2 is formed and
// applied after the gate/up accumulation).  Grid (parts, B).
__global__ void __launch_bounds__(kPrepThreads) mid_kernel(const MidParams p) {
  griddep_launch();  // the gate/up kernel may start streaming its weights
  const int part = blockIdx.x, parts = gridDim.x, b = blockIdx.y;
  const int ch = part * kPrepThreads + threadIdx.x;
  const bool valid = ch < p.H / 8;
  // before the wait (no dependence on earlier kernels): the 8 rows of a chunk
  // lie in one row-tile set of the O projection, so they share its piece count
  const GemvPlan& pl = p.o_plan;
  const int np = valid ? plan_pieces(pl, (8 * ch) / (pl.RT * kRowTile)) : 0;
  const size_t slab4 = (size_t)p.B * pl.N / 4;
  const float4* q = reinterpret_cast<const float4*>(p.o_part + (size_t)b * pl.N + 8 * (valid ? ch : 0));
  griddep_wait();
  float v[8];
  if (valid) {
    // x and the first pieces of W_o o, loaded together
    float4 xa[kPieceBatch], xc[kPieceBatch];
    pieces_load<kPieceBatch>(q, slab4, np, xa);
    pieces_load<kPieceBatch>(q + 1, slab4, np, xc);
    load_chunk8(p.xres + (size_t)b * p.H, FT_F32, ch, v);
    // h1 = x + W_o o, the pieces added in slab order
    const float4 a = pieces_sum<kPieceBatch>(q, slab4, np, xa), c = pieces_sum<kPieceBatch>(q + 1, slab4, np, xc);
    const float o[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] += o[k];
  }
  const bool bad =
      row_part(v, valid, ch, b, p.B, p.h1 + (size_t)b * p.H, p.h1_h, p.s_h1, p.ssq + b * parts + part);
  if (bad) set_status(p.status, FT_DEV_RANGE);
}

// Gate/up slabs (tensor-core path) -> the down projection's operand: a =
// silu(rho2 g) * (rho2 u) for 128 columns (one group of the operand) and up to 8
// tokens per CTA; the group offsets are summed over the CTA's four warps in a
// fixed order and stored (one CTA owns a (group, token)).  Gate row g and up row
// g + 8 of a 16-row packed tile give column 8 T + g.
__global__ void __launch_bounds__(128) swiglu_kernel(const SwigluParams p) {
  __shared__ float wsum[4][8];
  __shared__ float rho2_s[8];
  griddep_launch();  // the down projection may start streaming its weights
  const int grp = blockIdx.x, t0 = 8 * blockIdx.y, c = threadIdx.x, warp = c >> 5, lane = c & 31;
  const int kcol = grp * kWGroup + c;
  const int T = kcol >> 3, r = kcol & 7;
  const int row_g = 16 * T + r, row_u = row_g + 8;
  const GemvPlan& pl = p.plan;
  const int np = plan_pieces(pl, row_g / (pl.RT * kRowTile));
  const size_t slab = (size_t)p.B * pl.N;
  griddep_wait();
  float xg[8][kPieceBatch], xu[8][kPieceBatch];
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // every slab load of the CTA's tokens in flight together
    const int t = t0 + i;
    const int n = t < p.B ? np : 0;
    pieces_load<kPieceBatch>(p.part + (size_t)t * pl.N + row_g, slab, n, xg[i]);
    pieces_load<kPieceBatch>(p.part + (size_t)t * pl.N + row_u, slab, n, xu[i]);
  }
  if (c < 8) {  // the RMSNorm row factor of each of the CTA's tokens, once
    float a = 0.0f;
    if (t0 + c < p.B)
      for (int k = 0; k < p.nssq; ++k) a += __ldcg(p.ssq2 + (t0 + c) * p.nssq + k);
    rho2_s[c] = rsqrtf(a * p.inv_h + p.eps);
  }
  __syncthreads();
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + i;
    float st = 0.0f;
    if (t < p.B) {
      const float rho2 = rho2_s[i];
      const float gv = rho2 * pieces_sum<kPieceBatch>(p.part + (size_t)t * pl.N + row_g, slab, np, xg[i]);
      const float uv = rho2 * pieces_sum<kPieceBatch>(p.part + (size_t)t * pl.N + row_u, slab, np, xu[i]);
      const float a = gv / (1.0f + expf(-gv)) * uv;
      bad |= !(fabsf(a) <= 65504.0f);
      p.out_h[op_index(t, kcol, p.B)] = op_encode(a, kcol, st);
    }
    st = warp_sum(st);
    if (lane == 0) wsum[warp][i] = st;
  }
  __syncthreads();
  if (c < 8 && t0 + c < p.B) {
    const float st = ((wsum[0][c] + wsum[1][c]) + wsum[2][c]) + wsum[3][c];  // fixed order
    p.s_out[grp * 32 + t0 + c] = f32_to_sfix(st);
  }
  if (bad) set_status(p.status, FT_DEV_RANGE);
}

// Down slabs (tensor-core path) + h1 -> the block output; 4 rows of one token
// per thread.
__global__ void __launch_bounds__(128) post_kernel(const PostParams p) {
  griddep_launch();
  const GemvPlan& pl = p.plan;
  const int t = blockIdx.y, row = 512 * blockIdx.x + 4 * threadIdx.x;
  const bool on = row < pl.N;
  const int np = on ? plan_pieces(pl, row / (pl.RT * kRowTile)) : 0;
  const size_t at = (size_t)t * pl.N + (on ? row : 0), slab4 = (size_t)p.B * pl.N / 4;
  const float4* q = reinterpret_cast<const float4*>(p.part + at);
  griddep_wait();
  if (!on) return;
  float4 x[kPieceBatch];
  pieces_load<kPieceBatch>(q, slab4, np, x);
  const float4 h = __ldcg(reinterpret_cast<const float4*>(p.resid + at));
  float4 y = pieces_sum<kPieceBatch>(q, slab4, np, x);
  piece_add(y, h);
  GemvParams gp = {};
  gp.out_final = p.out_final;
  gp.out_dtype = p.out_dtype;
  down_out4(gp, at, y);
}

struct WsPlan {
  GemvPlan g[4];
  int nsplit;
  int kv_slots;  // attention: K/V tiles in flight per warp
  int parts;  // prep / mid CTAs per request
  size_t x_h, s_x, rho1, ssq1, xres, h1, qkv, qkv_part, o_part, o_h, s_o, h1_h, s_h1, ssq2, a_h, s_a, gu_part,
      down_part, tick, total;
};

// Splits per (request, KV head): as many as keep every attention CTA resident in
// one wave (a second, partial wave would double the kernel's time).
static int attn_splits(int B, int nkv, int G, int d, int max_ctx, int sms, int npmax) {
  const int pairs = B * nkv;
  const int per_sm = attn_ctas_per_sm(G, d, npmax);
  const int target = (per_sm > 0 ? per_sm : 4) * (sms > 0 ? sms : 148);
  int ns = target / pairs;
  const int cap = (max_ctx + 63) / 64;
  if (ns > cap) ns = cap;
  const int maxc = attn_max_cluster(G, d);  // the splits of one (request, KV head) form one cluster
  if (ns > maxc) ns = maxc;
  if (ns < 1) ns = 1;
  return ns;
}

static WsPlan make_plan(const ft_block_cfg& c, int B, int max_ctx) {
  WsPlan w;
  int sms = ft_host::num_sms();
  if (sms <= 0) sms = 148;
  const int nqkv = (c.n_q + 2 * c.n_kv) * c.head_dim;
  // batches of 17-32 run the projections on the tensor cores (tcgen05); INT4 and E4M3
  // weights alike
  const int fmt = c.weight_format;
  auto plan = [&](int role, int N, int K, int B_, int sms_, int budget) {
    return B_ > 16 ? make_umma_plan(role, N, K, B_, sms_, budget, fmt)
                   : make_gemv_plan(role, N, K, B_, sms_, budget, fmt);
  };
  // the partition (hence the QKV pieces attention stages) does not depend on the budget
  const int np_qkv = plan(kRoleQKV, nqkv, c.hidden, B, sms, 200 * 1024).npmax;
  w.nsplit = attn_splits(B, c.n_kv, c.n_q / c.n_kv, c.head_dim, max_ctx, sms, np_qkv);
  // shared-memory budget of one GEMV CTA (ring + reduction area); the QKV and O
  // CTAs leave room for one attention CTA on their SM, so that attention CTAs
  // start (and load their first K/V tiles) while QKV still runs, and O CTAs
  // start (and fill their rings) while attention runs
  const int bud = 200 * 1024;
  const int per_sm = ft_host::smem_per_sm();
  // attention K/V: a warp with a tile or two loads them straight into registers (kv_slots
  // 0: a bulk copy's longer latency would only add to the kernel's); longer shares stream
  // through a ring no deeper than the share, deep where every attention CTA has an SM to
  // itself (long contexts at small batch: few CTAs, each streaming far)
  {
    const int tiles = (max_ctx + 15) / 16, per_cta = (tiles + w.nsplit - 1) / w.nsplit;
    const int per_warp = (per_cta + kAttnWarps - 1) / kAttnWarps;
    const long ctas = (long)B * c.n_kv * w.nsplit;
    const int cap = ctas <= sms ? kAttnMaxSlots : kAttnSharedSlots;
    w.kv_slots = per_warp <= 2 ? 0 : std::min(cap, per_warp);
  }
  const int attn = attn_smem_bytes(c.n_q / c.n_kv, w.nsplit, c.head_dim, np_qkv, w.kv_slots);
  const int bud_att = per_sm > 0 ? std::min(bud, per_sm - attn - 3 * 1024) : bud;
  w.g[kRoleQKV] = plan(kRoleQKV, nqkv, c.hidden, B, sms, bud_att);
  w.g[kRoleO] = plan(kRoleO, c.hidden, c.n_q * c.head_dim, B, sms, bud_att);
  w.g[kRoleGU] = plan(kRoleGU, 2 * c.inter, c.hidden, B, sms, bud);
  w.g[kRoleDown] = plan(kRoleDown, c.hidden, c.inter, B, sms, bud);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t sfx = sizeof(sfix_t);
  w.x_h = take((size_t)B * c.hidden * 2);
  w.s_x = take((size_t)(c.hidden / 128) * 32 * sfx);
  w.parts = rms_parts(c.hidden);
  w.rho1 = take((size_t)B * 4);
  w.ssq1 = take((size_t)B * w.parts * 4);
  w.xres = take((size_t)B * c.hidden * 4);
  w.h1 = take((size_t)B * c.hidden * 4);
  w.qkv = take((size_t)B * nqkv * 4);
  w.qkv_part = take((size_t)w.g[kRoleQKV].npmax * B * nqkv * 4);
  w.o_part = take((size_t)w.g[kRoleO].npmax * B * c.hidden * 4);
  w.o_h = take((size_t)B * c.n_q * c.head_dim * 2);
  w.s_o = take((size_t)(c.n_q * c.head_dim / 128) * 32 * sfx);
  w.h1_h = take((size_t)B * c.hidden * 2);
  w.s_h1 = take((size_t)(c.hidden / 128) * 32 * sfx);
  w.ssq2 = take((size_t)B * w.parts * 4);
  w.a_h = take((size_t)B * c.inter * 2);
  w.s_a = take((size_t)(c.inter / 128) * 32 * sfx);
  // tensor-core path: gate/up writes slabs too (the SwiGLU kernel finishes them)
  w.gu_part = w.g[kRoleGU].umma ? take((size_t)w.g[kRoleGU].npmax * B * 2 * c.inter * 4) : 0;
  w.down_part = w.g[kRoleDown].whole ? 0 : take((size_t)w.g[kRoleDown].npmax * B * c.hidden * 4);
  w.tick = take((size_t)w.g[kRoleDown].NSET * 4);
  w.total = off;
  return w;
}

// inv_freq[i] = base^(-2i/d) (FP64) divided by 2 pi and scaled by 2^64: the
// RoPE angle of position p is p * turn[i] turns, reduced modulo one turn by
// unsigned 64-bit wrap-around.  Cached for the last (base, d) of this thread.
static void rope_turns(float base, int d, uint64_t (&turn)[64]) {
  thread_local float cb = -1.0f;
  thread_local int cd = -1;
  thread_local uint64_t ct[64];
  if (cb != base || cd != d) {
    for (int i = 0; i < 64; ++i) {
      const double inv_freq = (i < d / 2) ? std::pow((double)base, -2.0 * i / d) : 0.0;
      ct[i] = (uint64_t)std::ldexp(inv_freq / 6.283185307179586476925, 64);
    }
    cb = base;
    cd = d;
  }
  for (int i = 0; i < 64; ++i) turn[i] = ct[i];
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

static int run_block(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch, int max_ctx,
                     const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B, void* ws,
                     size_t ws_bytes, int32_t* status, unsigned mask, cudaStream_t st) {
  int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (!w || !cache || !x_in || !x_out || !pos || !ws) return FT_ERR_INVALID_ARG;
  if (!w->qkv || !w->o || !w->gateup || !w->down) return FT_ERR_INVALID_ARG;
  if (act_dtype != FT_BF16 && act_dtype != FT_F32) return FT_ERR_INVALID_ARG;
  if (B < 1 || max_batch < 1 || max_ctx < 1) return FT_ERR_INVALID_ARG;
  if (B > 32) return FT_ERR_UNSUPPORTED;
  if (B > max_batch) return FT_ERR_CAPACITY;
  if (!ft_host::aligned16(cache) || !ft_host::aligned16(ws) || !ft_host::aligned16(x_in) ||
      !ft_host::aligned16(x_out) || !ft_host::aligned16(w->qkv) || !ft_host::aligned16(w->o) ||
      !ft_host::aligned16(w->gateup) || !ft_host::aligned16(w->down))
    return FT_ERR_INVALID_ARG;
  const size_t act_bytes = (size_t)B * c->hidden * (act_dtype == FT_F32 ? 4 : 2);
  if (overlaps(x_in, act_bytes, x_out, act_bytes)) return FT_ERR_INVALID_ARG;
  const WsPlan P = make_plan(*c, B, max_ctx);
  for (int r = 0; r < 4; ++r)
    if (!P.g[r].divs_exact) return FT_ERR_UNSUPPORTED;
  if (P.g[kRoleQKV].npmax > kAttnMaxPieces) return FT_ERR_UNSUPPORTED;  // attention stages at most that many
  if (ws_bytes < P.total) return FT_ERR_WORKSPACE;
  if (overlaps(x_out, act_bytes, ws, ws_bytes) || overlaps(x_in, act_bytes, ws, ws_bytes)) return FT_ERR_INVALID_ARG;

  uint8_t* W = static_cast<uint8_t*>(ws);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(W + off); };
  auto Hh = [&](size_t off) { return reinterpret_cast<__half*>(W + off); };
  auto SF = [&](size_t off) { return reinterpret_cast<sfix_t*>(W + off); };
  const bool pdl = ft_host::pdl_enabled();
  const KVLayout L = kv_layout(*c, max_batch, max_ctx);

  if (mask & FT_STAGE_PREP) {
    PrepParams pp = {};
    pp.x_in = x_in;
    pp.act_dtype = act_dtype;
    pp.B = B;
    pp.H = c->hidden;
    pp.x_h = Hh(P.x_h);
    pp.s_x = SF(P.s_x);
    pp.ssq = F(P.ssq1);
    pp.xres = F(P.xres);
    pp.s_o = SF(P.s_o);
    pp.nkg_o = c->n_q * c->head_dim / 128;
    pp.s_a = SF(P.s_a);
    pp.nkg_a = c->inter / 128;
    pp.tick = reinterpret_cast<uint32_t*>(W + P.tick);
    pp.ntick = P.g[kRoleDown].whole ? 0 : P.g[kRoleDown].NSET;
    pp.status = status;
    if (launch_ex(prep_kernel, dim3(P.parts, B), dim3(kPrepThreads), 0, st, pdl, pp) != cudaSuccess)
      return FT_ERR_CUDA;
  }

  auto gemv = [&](int role, const void* wptr, size_t xoff, size_t soff) {
    GemvParams g = {};
    g.plan = P.g[role];
    g.w = static_cast<const uint8_t*>(wptr);
    g.x = Hh(xoff);
    g.s_in = SF(soff);
    g.B = B;
    g.status = status;
    switch (role) {
      case kRoleQKV: g.part = F(P.qkv_part); break;
      case kRoleO: g.part = F(P.o_part); break;
      case kRoleGU:
        g.part = P.g[kRoleGU].umma ? F(P.gu_part) : nullptr;
        g.out_h = Hh(P.a_h);
        g.s_out = SF(P.s_a);
        g.ssq2 = F(P.ssq2);
        g.nssq = P.parts;
        g.inv_h = 1.0f / (float)c->hidden;
        g.eps = c->rms_eps;
        break;
      case kRoleDown:
        // whole sets add the residual h1 directly; split sets store partial
        // sums that the last piece of each set adds to h1
        g.resid = F(P.h1);
        g.part = P.g[kRoleDown].whole ? nullptr : F(P.down_part);
        g.tick = reinterpret_cast<uint32_t*>(W + P.tick);
        g.out_final = x_out;
        g.out_dtype = act_dtype;
        break;
    }
    return launch_gemv(role, g, st, pdl);
  };

  if (mask & FT_STAGE_QKV) {
    if (gemv(kRoleQKV, w->qkv, P.x_h, P.s_x) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_ATTN) {
    AttnParams a;
    a.qkv_part = F(P.qkv_part);
    a.qkv_plan = P.g[kRoleQKV];
    a.qkv = F(P.qkv);
    a.ssq1 = F(P.ssq1);
    a.nssq = P.parts;
    a.inv_h = 1.0f / (float)c->hidden;
    a.eps = c->rms_eps;
    a.rho1 = F(P.rho1);
    a.cache = static_cast<uint8_t*>(cache);
    a.L = L;
    a.pos = pos;
    a.B = B;
    a.nq = c->n_q;
    a.nkv = c->n_kv;
    a.G = c->n_q / c->n_kv;
    a.hb = c->had_block;
    a.nsplit = P.nsplit;
    a.kv_slots = P.kv_slots;
    a.Nqkv = (c->n_q + 2 * c->n_kv) * c->head_dim;
    a.qscale = (float)(1.4426950408889634 / std::sqrt((double)c->head_dim));
    a.o_h = Hh(P.o_h);
    a.s_o = SF(P.s_o);
    a.status = status;
    rope_turns(c->rope_base, c->head_dim, a.rope_turn);
    if (launch_attn(a, c->head_dim, st, pdl) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_O) {
    if (gemv(kRoleO, w->o, P.o_h, P.s_o) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_MID) {
    MidParams mp = {};
    mp.xres = F(P.xres);
    mp.o_part = F(P.o_part);
    mp.o_plan = P.g[kRoleO];
    mp.B = B;
    mp.H = c->hidden;
    mp.h1 = F(P.h1);
    mp.h1_h = Hh(P.h1_h);
    mp.s_h1 = SF(P.s_h1);
    mp.ssq = F(P.ssq2);
    mp.status = status;
    if (launch_ex(mid_kernel, dim3(P.parts, B), dim3(kPrepThreads), 0, st, pdl, mp) != cudaSuccess)
      return FT_ERR_CUDA;
  }
  const bool umma = P.g[kRoleGU].umma != 0;
  if (mask & FT_STAGE_GU) {
    if (gemv(kRoleGU, w->gateup, P.h1_h, P.s_h1) != cudaSuccess) return FT_ERR_CUDA;
    if (umma) {
      SwigluParams sp = {};
      sp.part = F(P.gu_part);
      sp.plan = P.g[kRoleGU];
      sp.B = B;
      sp.ssq2 = F(P.ssq2);
      sp.nssq = P.parts;
      sp.inv_h = 1.0f / (float)c->hidden;
      sp.eps = c->rms_eps;
      sp.out_h = Hh(P.a_h);
      sp.s_out = SF(P.s_a);
      sp.status = status;
      if (launch_ex(swiglu_kernel, dim3(c->inter / kWGroup, (B + 7) / 8), dim3(128), 0, st, pdl, sp) != cudaSuccess)
        return FT_ERR_CUDA;
    }
  }
  if (mask & FT_STAGE_DOWN) {
    if (gemv(kRoleDown, w->down, P.a_h, P.s_a) != cudaSuccess) return FT_ERR_CUDA;
    if (umma) {
      PostParams op = {};
      op.part = F(P.down_part);
      op.plan = P.g[kRoleDown];
      op.resid = F(P.h1);
      op.out_final = x_out;
      op.out_dtype = act_dtype;
      op.B = B;
      if (launch_ex(post_kernel, dim3((c->hidden + 511) / 512, B), dim3(128), 0, st, pdl, op) != cudaSuccess)
        return FT_ERR_CUDA;
    }
  }
  return FT_OK;
}

}  // namespace ft

extern "C" {

size_t ft_decode_workspace_bytes(const ft_block_cfg* c, int B, int max_ctx) {
  if (ft_host::check_cfg(c) != FT_OK || B < 1 || B > 32 || max_ctx < 1) return 0;
  return ft::make_plan(*c, B, max_ctx).total;
}

int ft_decode_workspace_layout(const ft_block_cfg* c, int B, int max_ctx, ft_ws_layout* out) {
  const int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (!out || B < 1 || B > 32 || max_ctx < 1) return FT_ERR_INVALID_ARG;
  const ft::WsPlan P = ft::make_plan(*c, B, max_ctx);
  out->qkv = P.qkv;
  out->rho1 = P.rho1;
  out->o = P.o_h;
  out->h1 = P.h1;
  out->a = P.a_h;
  out->n_split = P.nsplit;
  return FT_OK;
}

int ft_decode_plan_info(const ft_block_cfg* c, int B, int max_ctx, int role, ft_gemv_info* out) {
  const int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (!out || B < 1 || B > 32 || max_ctx < 1 || role < FT_W_QKV || role > FT_W_DOWN) return FT_ERR_INVALID_ARG;
  const ft::WsPlan P = ft::make_plan(*c, B, max_ctx);
  const int r = role == FT_W_QKV ? ft::kRoleQKV : role == FT_W_O ? ft::kRoleO : role == FT_W_GATEUP ? ft::kRoleGU
                                                                                                     : ft::kRoleDown;
  const ft::GemvPlan& g = P.g[r];
  out->ctas = g.C;
  out->row_tiles = g.RT;
  out->warps = g.umma ? ft::ft_umma_warps() : g.NCW + 2;
  out->col_tiles = g.NT;
  out->whole = g.whole;
  out->tensor_core = g.umma;
  out->stages = g.stages;
  out->groups_per_stage = g.ng;
  out->smem_bytes = g.smem;
  return FT_OK;
}

int ft_decode_block(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch, int max_ctx,
                    const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B, void* ws,
                    size_t ws_bytes, int32_t* status, ft_stream stream) {
  return ft::run_block(c, w, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, ws, ws_bytes, status,
                       FT_STAGE_ALL, (cudaStream_t)stream);
}

int ft_decode_block_stages(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch, int max_ctx,
                           const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B, void* ws,
                           size_t ws_bytes, int32_t* status, unsigned mask, ft_stream stream) {
  if (mask == 0 || (mask & ~(unsigned)FT_STAGE_ALL)) return FT_ERR_INVALID_ARG;
  return ft::run_block(c, w, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, ws, ws_bytes, status, mask,
                       (cudaStream_t)stream);
}

int ft_decode_block_launches(const ft_block_cfg* c, int B) {
  if (ft_host::check_cfg(c) != FT_OK || B < 1 || B > 32) return 0;
  return B > 16 ? 9 : 7;
}

}  // extern "C"
