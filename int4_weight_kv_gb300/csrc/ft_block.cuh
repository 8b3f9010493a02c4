// Declarations shared by the decode block's kernels and its host orchestration:
// the workspace plan, the split-K GEMV work partition and kernel parameters.
#pragma once

#include "ft_internal.cuh"

namespace ft {

enum GemvRole { kRoleQKV = 0, kRoleO = 1, kRoleGU = 2, kRoleDown = 3 };

// Streaming GEMV work partition for one projection.
// Units are (macro block mb, input group kg) pairs, mb-major, where a macro
// block is RB consecutive 128-row blocks processed together (RB = NT, the
// number of 8-token MMA column tiles, so B-fragments are reused RB times).
// CTA c owns the contiguous unit range [u0(c), u1(c)); a macro block cut by a
// range boundary is a split-K reduction: each piece writes its partial sums to
// a slot and the last piece to finish (atomic ticket) sums the slots in piece
// order and runs the epilogue.
struct GemvPlan {
  int N, K, NRB, NKG, RB, NT, NMB;
  int U, C, per, rem, maxp;
  int slotf;  // floats per partial slot (8 warps x RB x NT x 128)
};

__host__ __device__ __forceinline__ int plan_u0(const GemvPlan& p, int c) {
  return c * p.per + (c < p.rem ? c : p.rem);
}
__host__ __device__ __forceinline__ int plan_owner(const GemvPlan& p, int u) {
  const int big = p.rem * (p.per + 1);
  return (u < big) ? u / (p.per + 1) : p.rem + (u - big) / p.per;
}

struct GemvParams {
  GemvPlan plan;
  const uint8_t* w;  // packed weights of this role
  const __half* x;   // FP16 activation operand [B][K]
  int B;
  uint32_t* tick;    // [NMB]
  float* slots;      // [NMB][maxp][slotf]
  // epilogue operands
  const float* rho;     // QKV: rho1[B]
  float* out_f32;       // QKV: qkv [B][N];  O: h1 [B][N]
  __half* out_h;        // O: h1 as FP16;  GU: a [B][I]
  const void* resid;    // O: block input (act dtype);  DOWN: h1 FP32
  int resid_dtype;
  float* sumsq;         // O: accumulates sum h1^2;  GU: reads it
  void* out_final;      // DOWN: block output (act dtype)
  int out_dtype;
  int H;
  float eps;
  int32_t* status;
};

struct AttnParams {
  const float* qkv;   // [B][Nqkv], rho1 applied, before RoPE
  uint8_t* cache;
  KVLayout L;
  const int32_t* pos;
  int B, nq, nkv, G, hb, nsplit, Nqkv;
  float qscale;       // log2(e) / sqrt(d), folded into the rotated query
  float* part;        // [B][nkv][nsplit][16 + 8 d]
  uint32_t* tick;     // [B * nkv]
  __half* o_h;        // [B][nq d]
  int32_t* status;
  double inv_freq[64];
};

struct PrepParams {
  const void* x_in;
  int act_dtype, B, H;
  float eps;
  __half* x_h;
  float* rho1;
  uint32_t* zero;  // counters cleared every call
  int nzero;
  int32_t* status;
};

// host-side launchers (ft_gemv.cu / ft_attn.cu / ft_block.cu)
cudaError_t launch_gemv(int role, const GemvParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_attn(const AttnParams& p, int head_dim, cudaStream_t st, bool pdl);
GemvPlan make_gemv_plan(int N, int K, int B, int sms);
size_t gemv_smem_bytes(int NT);

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
