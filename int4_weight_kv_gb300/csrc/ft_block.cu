// The decode block: input preparation and the host-side orchestration of the
// six kernels (prep, QKV, attention, O, gate/up, down) on the caller's stream,
// chained with programmatic dependent launch so each kernel's weight stream
// starts while its predecessor finishes.
#include <cmath>

#include "ft_block.cuh"

namespace ft {

// Block input -> FP16 MMA operand, RMSNorm row factor rho1 (applied later in
// the QKV epilogue, summary page "어떻게 동작하나"), and the per-call counters
// cleared.  One CTA per request.
__global__ void __launch_bounds__(256) prep_kernel(const PrepParams p) {
  griddep_wait();  // the previous block's kernels may still read the workspace
  griddep_launch();
  __shared__ float red[8];
  const int b = blockIdx.x, tid = threadIdx.x;
  for (int i = b * 256 + tid; i < p.nzero; i += gridDim.x * 256) p.zero[i] = 0u;
  float ss = 0.0f;
  bool bad = false;
  for (int i = tid; i < p.H; i += 256) {
    const float x = (p.act_dtype == FT_F32) ? static_cast<const float*>(p.x_in)[(size_t)b * p.H + i]
                                            : bf16_bits_to_f32(static_cast<const uint16_t*>(p.x_in)[(size_t)b * p.H + i]);
    ss = fmaf(x, x, ss);
    bad |= !(fabsf(x) <= 65504.0f);
    p.x_h[(size_t)b * p.H + i] = __float2half_rn(x);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.0f;
    for (int w = 0; w < 8; ++w) t += red[w];
    p.rho1[b] = rsqrtf(t / (float)p.H + p.eps);
  }
  if (bad) set_status(p.status, FT_DEV_RANGE);
}

struct WsPlan {
  GemvPlan g[4];
  int nsplit;
  size_t x_h, rho1, zero, nzero_words, sumsq2, attn_tick, gtick[4], qkv, o_h, h1, h1_h, a_h, attn_part, slots, total;
};

static int attn_splits(int B, int nkv, int max_ctx, int sms) {
  const int pairs = B * nkv;
  const int target = 4 * (sms > 0 ? sms : 148);
  int ns = (target + pairs - 1) / pairs;
  const int cap = (max_ctx + 63) / 64;
  if (ns > cap) ns = cap;
  if (ns > 48) ns = 48;
  if (ns < 1) ns = 1;
  return ns;
}

static WsPlan make_plan(const ft_block_cfg& c, int B, int max_ctx) {
  WsPlan w;
  int sms = ft_host::num_sms();
  if (sms <= 0) sms = 148;
  const int nqkv = (c.n_q + 2 * c.n_kv) * c.head_dim;
  w.g[kRoleQKV] = make_gemv_plan(nqkv, c.hidden, B, sms);
  w.g[kRoleO] = make_gemv_plan(c.hidden, c.n_q * c.head_dim, B, sms);
  w.g[kRoleGU] = make_gemv_plan(2 * c.inter, c.hidden, B, sms);
  w.g[kRoleDown] = make_gemv_plan(c.hidden, c.inter, B, sms);
  w.nsplit = attn_splits(B, c.n_kv, max_ctx, sms);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  w.x_h = take((size_t)B * c.hidden * 2);
  w.rho1 = take((size_t)B * 4);
  // counters cleared by the prep kernel every call: sumsq2, attention tickets, GEMV tickets
  w.zero = off;
  size_t z = 0;
  w.sumsq2 = off + z;
  z += (size_t)B * 4;
  w.attn_tick = off + z;
  z += (size_t)B * c.n_kv * 4;
  for (int r = 0; r < 4; ++r) {
    w.gtick[r] = off + z;
    z += (size_t)w.g[r].NMB * 4;
  }
  w.nzero_words = z / 4;
  take(z);
  w.qkv = take((size_t)B * nqkv * 4);
  w.o_h = take((size_t)B * c.n_q * c.head_dim * 2);
  w.h1 = take((size_t)B * c.hidden * 4);
  w.h1_h = take((size_t)B * c.hidden * 2);
  w.a_h = take((size_t)B * c.inter * 2);
  w.attn_part = take((size_t)B * c.n_kv * w.nsplit * (16 + 8 * c.head_dim) * 4);
  size_t sl = 0;
  for (int r = 0; r < 4; ++r) {
    const size_t s = (size_t)w.g[r].NMB * w.g[r].maxp * w.g[r].slotf * 4;
    if (s > sl) sl = s;
  }
  w.slots = take(sl);
  w.total = off;
  return w;
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
  if (ws_bytes < P.total) return FT_ERR_WORKSPACE;
  if (overlaps(x_out, act_bytes, ws, ws_bytes) || overlaps(x_in, act_bytes, ws, ws_bytes)) return FT_ERR_INVALID_ARG;

  uint8_t* W = static_cast<uint8_t*>(ws);
  const bool pdl = ft_host::pdl_enabled();
  const KVLayout L = kv_layout(*c, max_batch, max_ctx);
  cudaError_t err = cudaSuccess;

  if (mask & FT_STAGE_PREP) {
    PrepParams pp;
    pp.x_in = x_in;
    pp.act_dtype = act_dtype;
    pp.B = B;
    pp.H = c->hidden;
    pp.eps = c->rms_eps;
    pp.x_h = reinterpret_cast<__half*>(W + P.x_h);
    pp.rho1 = reinterpret_cast<float*>(W + P.rho1);
    pp.zero = reinterpret_cast<uint32_t*>(W + P.zero);
    pp.nzero = (int)P.nzero_words;
    pp.status = status;
    err = launch_ex(prep_kernel, dim3(B), dim3(256), 0, st, pdl, pp);
    if (err != cudaSuccess) return FT_ERR_CUDA;
  }

  auto gemv = [&](int role, const void* wptr, size_t xoff) {
    GemvParams g = {};
    g.plan = P.g[role];
    g.w = static_cast<const uint8_t*>(wptr);
    g.x = reinterpret_cast<const __half*>(W + xoff);
    g.B = B;
    g.tick = reinterpret_cast<uint32_t*>(W + P.gtick[role]);
    g.slots = reinterpret_cast<float*>(W + P.slots);
    g.H = c->hidden;
    g.eps = c->rms_eps;
    g.status = status;
    g.sumsq = reinterpret_cast<float*>(W + P.sumsq2);
    switch (role) {
      case kRoleQKV:
        g.rho = reinterpret_cast<const float*>(W + P.rho1);
        g.out_f32 = reinterpret_cast<float*>(W + P.qkv);
        break;
      case kRoleO:
        g.out_f32 = reinterpret_cast<float*>(W + P.h1);
        g.out_h = reinterpret_cast<__half*>(W + P.h1_h);
        g.resid = x_in;
        g.resid_dtype = act_dtype;
        break;
      case kRoleGU:
        g.out_h = reinterpret_cast<__half*>(W + P.a_h);
        break;
      case kRoleDown:
        g.resid = W + P.h1;
        g.resid_dtype = FT_F32;
        g.out_final = x_out;
        g.out_dtype = act_dtype;
        break;
    }
    return launch_gemv(role, g, st, pdl);
  };

  if (mask & FT_STAGE_QKV) {
    if ((err = gemv(kRoleQKV, w->qkv, P.x_h)) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_ATTN) {
    AttnParams a;
    a.qkv = reinterpret_cast<const float*>(W + P.qkv);
    a.cache = static_cast<uint8_t*>(cache);
    a.L = L;
    a.pos = pos;
    a.B = B;
    a.nq = c->n_q;
    a.nkv = c->n_kv;
    a.G = c->n_q / c->n_kv;
    a.hb = c->had_block;
    a.nsplit = P.nsplit;
    a.Nqkv = (c->n_q + 2 * c->n_kv) * c->head_dim;
    a.qscale = (float)(1.4426950408889634 / std::sqrt((double)c->head_dim));
    a.part = reinterpret_cast<float*>(W + P.attn_part);
    a.tick = reinterpret_cast<uint32_t*>(W + P.attn_tick);
    a.o_h = reinterpret_cast<__half*>(W + P.o_h);
    a.status = status;
    for (int i = 0; i < 64; ++i)
      a.inv_freq[i] = (i < c->head_dim / 2) ? std::pow((double)c->rope_base, -2.0 * i / c->head_dim) : 0.0;
    if ((err = launch_attn(a, c->head_dim, st, pdl)) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_O) {
    if ((err = gemv(kRoleO, w->o, P.o_h)) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_GU) {
    if ((err = gemv(kRoleGU, w->gateup, P.h1_h)) != cudaSuccess) return FT_ERR_CUDA;
  }
  if (mask & FT_STAGE_DOWN) {
    if ((err = gemv(kRoleDown, w->down, P.a_h)) != cudaSuccess) return FT_ERR_CUDA;
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
  out->o = P.o_h;
  out->h1 = P.h1;
  out->a = P.a_h;
  out->n_split = P.nsplit;
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

int ft_decode_block_launches(void) { return 6; }

}  // extern "C"
