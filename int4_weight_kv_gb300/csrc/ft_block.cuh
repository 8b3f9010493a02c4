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
  // tile-split consumers (large batches): each consumer warp owns tpw of the
  // set's RT = tpw * NCW row tiles over all of a stage's groups, so one stage
  // of activations serves RT tiles (no cross-warp reduction)
  int ts, tpw;
};

__host__ __device__ __forceinline__ int plan_u0(const GemvPlan& p, int c) {
  const int u = c * p.per + (c < p.rem ? c : p.rem);
  return p.whole ? u * p.NKG : u;
}
// CTA owning unit u (split partitions only).
__host__ __device__ __forceinline__ int plan_owner(const GemvPlan& p, int u) {
  const int big = p.rem * (p.per + 1);
  return (u < big) ? u / (p.per + 1) : p.rem + (u - big) / p.per;
}

struct GemvParams {
  GemvPlan plan;
  const uint8_t* w;   // packed weights of this role
  const __half* x;    // activation operand, grouped layout of B rows (op_index)
  const float* s_in;  // its group offsets [K/128][32]
  int B;
  uint32_t* tick;     // DOWN (split sets): per-set completion tickets [NSET]
  float* out_f32;     // QKV: qkv acc;  O: h1 acc;  DOWN: h1 (whole sets) or its copy accumulating split sets
  __half* out_h;      // GU: a operand [B][I]
  float* s_out;       // GU: a's group offsets [I/128][32] (accumulated)
  const float* ssq2;  // GU: partial sums of h1^2 [B][nssq], giving the RMSNorm row factor rho2
  int nssq;
  float inv_h, eps;   // GU: 1 / hidden, RMSNorm epsilon
  void* out_final;    // DOWN: block output (h1 + W_down a, BF16 or FP32)
  int out_dtype;
  int32_t* status;
};

struct AttnParams {
  const float* qkv;   // [B][Nqkv] accumulated projections, before rho1 and RoPE
  const float* ssq1;  // [B][nssq] partial sums of x^2, giving the RMSNorm row factor rho1
  int nssq;
  float inv_h, eps;
  float* rho1;        // [B] rho1, recorded for inspection
  uint8_t* cache;
  KVLayout L;
  const int32_t* pos;
  int B, nq, nkv, G, hb, nsplit, Nqkv;
  float qscale;       // log2(e) / sqrt(d), folded into the rotated query
  __half* o_h;        // attention output, grouped operand layout of B rows (op_index)
  float* s_o;         // its group offsets [nq d / 128][32] (accumulated)
  int32_t* status;
  uint64_t rope_turn[64];  // inv_freq[i] / (2 pi) as 64-bit binary fractions (RoPE angles in turns)
};

// Block input -> QKV operand, partial sums of x^2, h1 accumulator initialised
// to x, and the accumulators of this call cleared.  CTA (part, request) covers
// 512 inputs (kPrepChunk chunks of 8).
struct PrepParams {
  const void* x_in;
  int act_dtype, B, H;
  __half* x_h;       // operand, grouped layout (op_index)
  float* s_x;        // [H/128][32]
  float* ssq;        // [B][parts] partial sums of x^2
  float* h1;         // [B][H] <- x
  float* qkv;        // [B][Nqkv] <- 0
  int nqkv;
  float* s_o;        // [NKG_o][32] <- 0 (column b)
  int nkg_o;
  float* s_a;        // [NKG_a][32] <- 0 (column b)
  int nkg_a;
  uint32_t* tick;    // down completion tickets <- 0 (split sets only)
  int ntick;
  int32_t* status;
};

// Between O and gate/up: h1 -> its operand and offsets, partial sums of h1^2
// and (split down sets) the down accumulator.  CTA (part, request) covers 512
// inputs.
struct MidParams {
  const float* h1;   // [B][H] complete after O
  int B, H;
  __half* h1_h;      // operand, grouped layout (op_index)
  float* s_h1;       // [H/128][32]
  float* ssq;        // [B][parts] partial sums of h1^2
  float* out_acc;    // [B][H] <- h1 (down accumulator of split sets) or null
  int32_t* status;
};

constexpr int kPrepThreads = 64;  // threads (chunks of 8 inputs) per prep / mid CTA
__host__ __device__ __forceinline__ int rms_parts(int H) { return (H / 8 + kPrepThreads - 1) / kPrepThreads; }

// host-side launchers (ft_gemv.cu / ft_attn.cu / ft_block.cu)
cudaError_t launch_gemv(int role, const GemvParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_attn(const AttnParams& p, int head_dim, cudaStream_t st, bool pdl);
constexpr int kAttnWarps = 4;  // warps per attention CTA (16-position tiles strided over them)
// Dynamic shared memory of one attention CTA: the warps' partials of G heads and
// the inbox of n_split * ceil(G / n_split) pushed partials, (d + 4) floats each.
__host__ __device__ __forceinline__ int attn_dyn_smem(int G, int nsplit, int d) {
  return (kAttnWarps * G + nsplit * ((G + nsplit - 1) / nsplit)) * (d + 4) * 4;
}
// Static + dynamic shared memory of one attention CTA (host).
int attn_smem_bytes(int G, int nsplit, int d);
// Attention CTAs resident per SM (registers, shared memory), 0 if unknown (host).
int attn_ctas_per_sm(int G, int d);
// Largest cluster of attention CTAs the device schedules: 16 where the
// non-portable size is allowed and fits, else 8 (host).
int attn_max_cluster(int G, int d);
// Gate/up and down CTAs own whole row-tile sets; QKV and O split sets over
// CTAs along K (partial sums red.add-ed into an FP32 accumulator).
GemvPlan make_gemv_plan(int role, int N, int K, int B, int sms, int smem_budget);

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
