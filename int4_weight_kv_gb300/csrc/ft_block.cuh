// Declarations shared by the decode block's kernels and its host orchestration:
// the workspace plan, the split-K GEMV work partition and kernel parameters.
#pragma once

#include "ft_internal.cuh"

namespace ft {

enum GemvRole { kRoleQKV = 0, kRoleO = 1, kRoleGU = 2, kRoleDown = 3 };

// Streaming GEMV work partition for one projection.
// Units are (row-tile set, input group) pairs, set-major; a set is RT
// consecutive 16-row tiles processed together so each activation B fragment is
// reused RT times.  CTA c owns the contiguous unit range [u0(c), u1(c)); with
// `whole` the ranges are whole sets (no set is split across CTAs).
struct GemvPlan {
  int N, K, NTILE, NKG;        // rows, inputs, 16-row tiles, 128-input groups
  int NT, RT, NCW, NSET;       // 8-token column tiles, row tiles per set, consumer warps, sets
  int whole, C, per, rem;      // partition of units over C CTAs
  int ng;                      // groups per stage
  int stages, slot, xoff, soff, xstride;  // ring geometry (bytes)
  int redoff, zerooff, slotoff, smem;  // shared-memory map
  // split partitions: the most pieces (CTAs) any set is divided into
  int npmax;
  // ceil(2^32 / (per + 1)) and ceil(2^32 / per): plan_owner divides with a
  // multiply-high, exact because units * (per + 1) <= 2^32 (checked on the host)
  unsigned long long rcp_per1, rcp_per;
  int divs_exact;  // 0: the partition is too large for that division (refused)
  int umma;        // 1: the tensor-core (tcgen05) kernel, 128-row sets, every role may split sets
  int slab;        // bytes of one (row tile, group) slab: kSlabBytes (INT4) or kSlabBytesE4 (E4M3)
};

__host__ __device__ __forceinline__ int plan_u0(const GemvPlan& p, int c) {
  const int u = c * p.per + (c < p.rem ? c : p.rem);
  return p.whole ? u * p.NKG : u;
}
// CTA owning unit u (split partitions only).  floor(n M / 2^32) with
// M = ceil(2^32 / d) equals floor(n / d) whenever n d <= 2^32.
__host__ __device__ __forceinline__ int plan_owner(const GemvPlan& p, int u) {
  const int big = p.rem * (p.per + 1);
  if (u < big) return (int)(((unsigned long long)u * p.rcp_per1) >> 32);
  return p.rem + (int)(((unsigned long long)(u - big) * p.rcp_per) >> 32);
}
// Split partitions: the first CTA of set s, and how many CTAs (pieces) share it.
__host__ __device__ __forceinline__ int plan_first(const GemvPlan& p, int s) { return plan_owner(p, s * p.NKG); }
__host__ __device__ __forceinline__ int plan_pieces(const GemvPlan& p, int s) {
  return plan_owner(p, s * p.NKG + p.NKG - 1) - plan_first(p, s) + 1;
}
// Split partitions write each piece's partial sums to its own slab: piece j of
// a set to part[j][t][row] (slabs of B x N floats), so every piece writes whole
// 32-byte sectors.  Consumers add the pieces of an output in slab order, so a
// sum does not depend on which CTA finished first.  kPieceBatch pieces are
// loaded together with no branch (absent pieces read as 0, which adds
// exactly); more (large batches split sets into up to about 8 pieces) are added
// one by one.
constexpr int kPieceBatch = 4;
template <int NB, typename T>
__device__ __forceinline__ void pieces_load(const T* src, size_t slab, int np, T (&x)[NB]) {
#pragma unroll
  for (int u = 0; u < NB; ++u) x[u] = (u < np) ? __ldcg(src + u * slab) : T{};
}
__device__ __forceinline__ void piece_add(float& a, float b) { a += b; }
__device__ __forceinline__ void piece_add(float4& a, const float4& b) {
  a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
template <int NB, typename T>
__device__ __forceinline__ T pieces_sum(const T* src, size_t slab, int np, const T (&x)[NB]) {
  T v = x[0];
#pragma unroll
  for (int u = 1; u < NB; ++u) piece_add(v, x[u]);
  for (int j = NB; j < np; ++j) piece_add(v, __ldcg(src + j * slab));
  return v;
}

// Walks a CTA's unit range stage by stage (set, first group, group count) with
// no divisions in the loop; every warp role runs the same walk.
struct StageWalk {
  int u, u1, set, kg, ng, NKG, cap;
  __device__ __forceinline__ StageWalk(const GemvPlan& pl, int u0, int u1_) {
    u = u0;
    u1 = u1_;
    NKG = pl.NKG;
    cap = pl.ng;
    set = u0 / NKG;
    kg = u0 - set * NKG;
    ng = min(min(cap, NKG - kg), u1 - u);
  }
  __device__ __forceinline__ bool valid() const { return u < u1; }
  // true if the stage just finished ends this CTA's piece of its set
  __device__ __forceinline__ bool piece_end() const { return u + ng >= u1 || kg + ng == NKG; }
  __device__ __forceinline__ void next() {
    u += ng;
    kg += ng;
    if (kg == NKG) {
      kg = 0;
      ++set;
    }
    ng = min(min(cap, NKG - kg), u1 - u);
  }
};

struct GemvParams {
  GemvPlan plan;
  const uint8_t* w;   // packed weights of this role
  const __half* x;    // activation operand, grouped layout of B rows (op_index)
  const sfix_t* s_in; // its group offsets [K/128][32]
  int B;
  uint32_t* tick;     // DOWN (split sets): per-set completion tickets [NSET]
  float* part;        // QKV, O, DOWN split sets: piece slabs [npmax][B][N]
  const float* resid; // DOWN: h1, the residual added to the block output
  __half* out_h;      // GU: a operand [B][I]
  sfix_t* s_out;      // GU: a's group offsets [I/128][32] (accumulated, exact)
  const float* ssq2;  // GU: partial sums of h1^2 [B][nssq], giving the RMSNorm row factor rho2
  int nssq;
  float inv_h, eps;   // GU: 1 / hidden, RMSNorm epsilon
  void* out_final;    // DOWN: block output (h1 + W_down a, BF16 or FP32)
  int out_dtype;
  int32_t* status;
};

// Down projection, split set `set` whose last piece just finished here: the
// block output of its rows is the pieces' slabs added in slab order, plus h1.
// Threads take 4 consecutive rows of one token at a time.
__device__ __forceinline__ void down_out4(const GemvParams& p, size_t at, const float4& y) {
  if (p.out_dtype == FT_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out_final) + at) = y;
  } else {
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.x)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.y)) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.z)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(y.w)) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out_final) + at) = make_uint2(lo, hi);
  }
}
__device__ __forceinline__ void down_finish_set(const GemvParams& p, int set, int rows, int first_row, int i0,
                                                int stride) {
  const GemvPlan& pl = p.plan;
  const int np = plan_pieces(pl, set);
  const size_t slab4 = (size_t)p.B * pl.N / 4;
  const int r4 = rows / 4, n = r4 * p.B;
  for (int i = i0; i < n; i += stride) {
    const size_t at = (size_t)(i / r4) * pl.N + first_row + 4 * (i % r4);  // 4 rows of one token
    const float4* q = reinterpret_cast<const float4*>(p.part + at);
    float4 x[kPieceBatch];
    pieces_load<kPieceBatch>(q, slab4, np, x);
    const float4 h = __ldcg(reinterpret_cast<const float4*>(p.resid + at));
    float4 y = pieces_sum<kPieceBatch>(q, slab4, np, x);
    piece_add(y, h);
    down_out4(p, at, y);
  }
}

struct AttnParams {
  const float* qkv_part;  // QKV piece slabs, before rho1 and RoPE
  GemvPlan qkv_plan;      // the QKV partition that wrote them
  float* qkv;         // [B][Nqkv] the summed projection, recorded for inspection
  const float* ssq1;  // [B][nssq] partial sums of x^2, giving the RMSNorm row factor rho1
  int nssq;
  float inv_h, eps;
  float* rho1;        // [B] rho1, recorded for inspection
  uint8_t* cache;
  KVLayout L;
  const int32_t* pos;
  int B, nq, nkv, G, hb, nsplit, Nqkv;
  int kv_slots;       // K/V tiles each warp keeps in flight in a shared-memory ring (1..kAttnMaxSlots),
                      // or 0: plain loads into registers, one tile ahead
  float qscale;       // log2(e) / sqrt(d), folded into the rotated query
  __half* o_h;        // attention output, grouped operand layout of B rows (op_index)
  sfix_t* s_o;        // its group offsets [nq d / 128][32] (accumulated, exact)
  int32_t* status;
  uint64_t rope_turn[64];  // inv_freq[i] / (2 pi) as 64-bit binary fractions (RoPE angles in turns)
};

// Block input -> QKV operand, partial sums of x^2, an FP32 copy of x (the
// residual), and the accumulators of this call cleared.  CTA (part, request)
// covers 512 inputs (kPrepThreads chunks of 8).
struct PrepParams {
  const void* x_in;
  int act_dtype, B, H;
  __half* x_h;       // operand, grouped layout (op_index)
  sfix_t* s_x;       // [H/128][32]
  float* ssq;        // [B][parts] partial sums of x^2
  float* xres;       // [B][H] <- x
  sfix_t* s_o;       // [NKG_o][32] <- 0 (column b)
  int nkg_o;
  sfix_t* s_a;       // [NKG_a][32] <- 0 (column b)
  int nkg_a;
  uint32_t* tick;    // down completion tickets <- 0 (split sets only)
  int ntick;
  int32_t* status;
};

// Between O and gate/up: h1 = x + the O projection's pieces, its operand and
// offsets, and partial sums of h1^2.  CTA (part, request) covers 512 inputs.
struct MidParams {
  const float* xres;    // [B][H] block input (FP32 copy)
  const float* o_part;  // O piece slabs
  GemvPlan o_plan;
  int B, H;
  float* h1;         // [B][H] <- x + W_o o
  __half* h1_h;      // operand, grouped layout (op_index)
  sfix_t* s_h1;      // [H/128][32]
  float* ssq;        // [B][parts] partial sums of h1^2
  int32_t* status;
};

// Batches of 17-32 (tensor-core projections, every set split into slabs):
// gate/up slabs -> a = silu(rho2 g) (rho2 u), the down projection's operand and
// its group offsets.  CTA (group of 128 columns, 8 tokens), one column per thread.
struct SwigluParams {
  const float* part;  // gate/up piece slabs [npmax][B][2I]
  GemvPlan plan;      // the gate/up partition that wrote them
  int B;
  const float* ssq2;  // [B][nssq] partial sums of h1^2 (rho2)
  int nssq;
  float inv_h, eps;
  __half* out_h;      // a operand (op_index)
  sfix_t* s_out;      // its group offsets [I/128][32] (written, exact)
  int32_t* status;
};
// down slabs + h1 -> block output.  CTA (512 rows, token), 4 rows per thread.
struct PostParams {
  const float* part;  // down piece slabs [npmax][B][H]
  GemvPlan plan;
  const float* resid; // h1 [B][H]
  void* out_final;
  int out_dtype, B;
};

constexpr int kPrepThreads = 64;  // threads (chunks of 8 inputs) per prep / mid CTA
__host__ __device__ __forceinline__ int rms_parts(int H) { return (H / 8 + kPrepThreads - 1) / kPrepThreads; }

// host-side launchers (ft_gemv.cu / ft_umma.cu / ft_attn.cu / ft_block.cu)
cudaError_t launch_gemv(int role, const GemvParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_umma(int role, const GemvParams& p, cudaStream_t st, bool pdl);
// Partition for the tensor-core kernel (batches of 17-32): 128-row sets.
GemvPlan make_umma_plan(int role, int N, int K, int B, int sms, int smem_budget, int weight_format);
int ft_umma_warps();  // warps per CTA of the tensor-core kernel
cudaError_t launch_attn(const AttnParams& p, int head_dim, cudaStream_t st, bool pdl);
constexpr int kAttnWarps = 4;  // warps per attention CTA (16-position tiles strided over them)
// The attention kernel stages the QKV pieces it needs (G query heads, k and v:
// (G + 2) d channels of each of at most kAttnMaxPieces pieces) in the area
// that later holds its warps' partials.
constexpr int kAttnMaxPieces = 8;
__host__ __device__ __forceinline__ int attn_stage_floats(int G, int d, int npmax) { return (G + 2) * d * npmax; }
// K/V tiles in flight per attention warp: at most kAttnMaxSlots where every
// attention CTA has an SM to itself, else at most kAttnSharedSlots (the ring
// size that still lets four CTAs share an SM)
constexpr int kAttnMaxSlots = 8, kAttnSharedSlots = 3;
// Dynamic shared memory of one attention CTA: the warps' partials of G heads
// (or, before the main loop, the staged QKV pieces), the inbox of
// n_split * ceil(G / n_split) pushed partials, (d + 4) floats each, then
// (128-byte aligned, at float offset attn_ring_off) each warp's ring of
// kv_slots K/V tiles of 16 positions (16 d bytes: K entries, then V entries).
__host__ __device__ __forceinline__ int attn_ring_off(int G, int nsplit, int d, int npmax) {
  const int mrg = kAttnWarps * G * (d + 4), stage = attn_stage_floats(G, d, npmax);
  const int f = (mrg > stage ? mrg : stage) + nsplit * ((G + nsplit - 1) / nsplit) * (d + 4);
  return (f + 31) & ~31;
}
__host__ __device__ __forceinline__ int attn_dyn_smem(int G, int nsplit, int d, int npmax, int kv_slots) {
  return attn_ring_off(G, nsplit, d, npmax) * 4 + kAttnWarps * kv_slots * 16 * d;
}
// Static + dynamic shared memory of one attention CTA (host).
int attn_smem_bytes(int G, int nsplit, int d, int npmax, int kv_slots);
// Attention CTAs resident per SM (registers, shared memory) with npmax staged
// QKV pieces, 0 if unknown (host).
int attn_ctas_per_sm(int G, int d, int npmax);
// Largest cluster of attention CTAs the device schedules: 16 where the
// non-portable size is allowed and fits, else 8 (host).
int attn_max_cluster(int G, int d);
// Gate/up CTAs own whole row-tile sets; QKV and O split sets over CTAs along K
// (each piece's partial sums go to its own slab); down does either.
GemvPlan make_gemv_plan(int role, int N, int K, int B, int sms, int smem_budget, int weight_format);

template <typename... Args>
cudaError_t launch_ex(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace ft
