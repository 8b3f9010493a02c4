// Declarations of the persistent decode-block kernel: the split-K work
// partition of the four INT4 projections, the shared-memory map and the
// kernel parameters.
#pragma once

#include "ft_internal.cuh"

namespace ft {

enum GemvRole { kRoleQKV = 0, kRoleO = 1, kRoleGU = 2, kRoleDown = 3 };

// RT row tiles per set share every activation fragment (RT x NT independent
// MMA chains per warp); NCW consumer warps split a stage's groups.
template <int NT>
struct GemvShape;
template <> struct GemvShape<1> { static constexpr int RT = 4, NCW = 12; };
template <> struct GemvShape<2> { static constexpr int RT = 4, NCW = 8; };
template <> struct GemvShape<3> { static constexpr int RT = 4, NCW = 4; };
template <> struct GemvShape<4> { static constexpr int RT = 4, NCW = 4; };

// Streaming work partition of one projection.  Units are (row-tile set, input
// group) pairs, set-major; a set is RT consecutive 16-row tiles processed
// together so each activation B fragment is reused RT times.  CTA c < C owns
// the contiguous unit range [u0(c), u0(c+1)); with `whole` the ranges are
// whole sets (no set is split across CTAs).  A stage of the ring carries up
// to ng groups of the RT tiles of one set, the activation chunk of those
// groups for every token and their offsets.
struct GemvPlan {
  int N, K, NTILE, NKG;        // rows, inputs, 16-row tiles, 128-input groups
  int NT, RT, NCW, NSET;       // 8-token column tiles, row tiles per set, consumer warps, sets
  int whole, C, per, rem;      // partition of units over C CTAs
  int ng;                      // groups per stage
  int slot, xoff, soff, xstride;  // stage layout (bytes)
};

__host__ __device__ __forceinline__ int plan_u0(const GemvPlan& p, int c) {
  if (c >= p.C) c = p.C;
  const int u = c * p.per + (c < p.rem ? c : p.rem);
  return p.whole ? u * p.NKG : u;
}
// CTA owning unit u (split partitions only).
__host__ __device__ __forceinline__ int plan_owner(const GemvPlan& p, int u) {
  const int big = p.rem * (p.per + 1);
  return (u < big) ? u / (p.per + 1) : p.rem + (u - big) / p.per;
}

constexpr int kMaxStages = 16;
constexpr int kZeroRowBytes = 16 * 128 * 2;  // one activation row of the largest stage (16 groups)
constexpr int kAttMaxG = 8;   // query heads per KV head handled by one piece

// Per-CTA control block at the start of dynamic shared memory (after the
// mbarriers).
// Attention work: request b has nt[b] tiles of 16 positions per KV head (0 if
// its position is invalid); each (request, KV head) pair is cut into np[b]
// pieces of sz[b] tiles (the last may be shorter); pieces are numbered
// request-major, head, piece (first piece of request b: pb[b]) and piece i
// goes to CTA i mod C.
struct Ctrl {
  double inv_freq[64];  // RoPE frequencies, copied from the parameters
  int nt[32], np[32], sz[32];
  int pb[33];
  int lb[32];          // L_b
  int P;               // pieces in total
  int flag;
  float rho1[32], rho2[32];
};

struct BlockParams {
  int B, H, I, nq, nkv, D, G, hb, nqkv;
  float eps, qscale;   // RMSNorm epsilon; log2(e)/sqrt(d) folded into the rotated query
  float hscale;        // 1/sqrt(had_block)
  int C;               // CTAs (one per SM, all co-resident)
  GemvPlan g[4];
  int stages, stride;  // ring: stages x stride bytes
  int ctrl_off, att_off, red_off, zero_off, ring_off, smem;
  int tps;             // attention tiles (16 positions) per ring stage
  int tmin;            // fewest tiles in one attention piece (shorter contexts are not split)
  const uint8_t* w[4];
  uint8_t* cache;
  KVLayout L;
  const int32_t* pos;
  const void* x_in;
  void* x_out;
  int act_dtype;
  // workspace
  uint32_t* sync;      // [0..5] arrivals at grid barriers G0..G5, [6] exits, [7] abort flag
  __half* x_h;         // [B][H] block input as the QKV operand
  float* s_x;          // [H/128][32] its group offsets
  float* ss1;          // [H/128][32] per-group sums of x^2
  float* rho1;         // [B] (written by CTA 0 for inspection)
  float* qkv;          // [B][nqkv] QKV accumulators (before rho1 and RoPE)
  float* part;         // attention partials, one per piece [(C + B n_kv)][16 + G d]
  uint32_t* att_tick;  // [B n_kv]
  __half* o_h;         // [B][nq d] attention output as the O operand
  float* s_o;          // [nq d / 128][32]
  float* h1;           // [B][H] x + attention delta
  __half* h1_h;        // [B][H] h1 as the gate/up operand
  float* s_h1;         // [H/128][32]
  float* ss2;          // [32] sums of h1^2
  __half* a_h;         // [B][I] SwiGLU output as the down operand
  float* s_a;          // [I/128][32]
  float* out_acc;      // [B][H] down accumulator (x_out itself for FP32 output)
  int32_t* status;
  double inv_freq[64];
};

GemvPlan make_gemv_plan(int N, int K, int B, int C, bool whole_sets);

}  // namespace ft
