// Internal helpers shared by the library's kernels: inline-PTX wrappers for
// sm_103a (bulk async copies, mbarriers, programmatic dependent launch,
// tensor-core MMA, warp matrix transpose), nibble decoding, the packed-weight
// and KV-entry layouts, and host-side launch utilities.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "ft.h"

namespace ft {

// ------------------------------------------------------------------ layout
constexpr int kWGroup = 128;         // weight group along the input axis
constexpr int kRowTile = 16;         // rows per MMA tile
constexpr int kSlabCodes = 1024;     // nibbles of one (row tile, group): 16 x 128 / 2
constexpr int kSlabBytes = 1056;     // + 16 BF16 scales
constexpr int kSlabCodesE4 = 2048;   // E4M3 codes of one (row tile, group): 16 x 128 bytes
constexpr int kSlabBytesE4 = 2080;   // + 16 BF16 scales
__host__ __device__ __forceinline__ int slab_bytes_of(int weight_format) {
  return weight_format == FT_WFMT_E4M3 ? kSlabBytesE4 : kSlabBytes;
}

// bounded waits: a wait that exceeds this many nanoseconds gives up
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Waits for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// Orders this thread's generic-proxy shared-memory accesses before its later
// async-proxy ones (a bulk copy into memory that was just read or written).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 1-D bulk copy global -> shared, completion signalled on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), no register holds the
// data in flight; cp_async_wait_all() waits for this thread's copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// L2 load issued where it stands (volatile: the compiler may not sink it to
// its first use), for values fetched early and consumed much later.
__device__ __forceinline__ float ld_cg_early(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

// Streamed read-once data (KV cache): skip L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Data written by an earlier kernel of the same dependent chain or by another
// CTA of this kernel: read at L2 (coherent point), never from L1.
__device__ __forceinline__ float ld_cg_f32(const float* p) { return __ldcg(p); }

// D = A(16x16, f16, row) * B(16x8, f16, col) + C  (FP32 accumulate)
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Same with C = 0.
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// Split cluster barrier: arrive (release) early, wait (acquire) before the
// first access to a peer's shared memory, which must have started executing
// and initialised what the access relies on.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
// Asynchronous store of 4 floats into the shared memory of CTA `rank` of this
// cluster, at the offset of the 16-byte aligned local shared address `local`;
// its 16 bytes complete on that CTA's mbarrier at the offset of `local_bar`.
__device__ __forceinline__ void st_async_v4(uint32_t local, uint32_t local_bar, uint32_t rank, float4 v) {
  uint32_t remote, remote_bar;
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote_bar) : "r"(local_bar), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t lop3_or_and(uint32_t x, uint32_t mask, uint32_t orv) {
  // (x & mask) | orv
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(x), "r"(mask), "r"(orv));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Nibble decode.  A 4-bit code c placed in the low mantissa bits of FP16
// 1024.0 (0x6400, mantissa step 1) reads as 1024 + c; placed at bits 4..7 of
// the half it reads as 1024 + 16 c.  Both are exact.  The offset (1024 + 8 for
// the first kind, 1024 + 128 after dividing the activation by 16 for the
// second) is not subtracted per weight: every k-step of 16 uses the first kind
// for k = 0..7 and the second for k = 8..15, the activation operand holds
// x (k < 8) and x / 16 (k >= 8), and each group's accumulation starts at -S
// with S = 1032 * sum_{k<8} x + 1152 * sum_{k>=8} (x / 16) (kOffLo / kOffHi).
// From one 32-bit word with nibbles n0..n7 (bits 4i..4i+3) four integer ops
// and one shift give the four f16x2 registers
//   r0 = (n0, n4),  r1 = 16 (n1, n5),  r2 = (n2, n6),  r3 = 16 (n3, n7)
// (low half first, before the offsets).
constexpr uint32_t kH1024 = 0x64006400u;   // (1024, 1024)
constexpr float kOffLo = 1032.0f;          // 1024 + 8
constexpr float kOffHi = 1152.0f;          // (1024 + 16 * 8) with x / 16: 1024 + 128
constexpr uint32_t kHOffLo = 0x64086408u;  // (1032, 1032) in FP16
constexpr uint32_t kHOffHi = 0x64806480u;  // (1152, 1152) in FP16

__device__ __forceinline__ void magic_word(uint32_t w, uint32_t (&r)[4]) {
  const uint32_t w8 = w >> 8;
  r[0] = lop3_or_and(w, 0x000F000Fu, kH1024);
  r[1] = lop3_or_and(w, 0x00F000F0u, kH1024);
  r[2] = lop3_or_and(w8, 0x000F000Fu, kH1024);
  r[3] = lop3_or_and(w8, 0x00F000F0u, kH1024);
}

// Four f16x2 registers (n_i of the low half, n_i of the high half) from a
// register holding nibbles n0..n3 in each 16-bit half: at the unscaled
// position (1024 + c) or at bits 4..7 (1024 + 16 c).
__device__ __forceinline__ void magic_low4(uint32_t r, uint32_t (&o)[4]) {
  o[0] = lop3_or_and(r, 0x000F000Fu, kH1024);
  o[1] = lop3_or_and(r >> 4, 0x000F000Fu, kH1024);
  o[2] = lop3_or_and(r >> 8, 0x000F000Fu, kH1024);
  o[3] = lop3_or_and(r >> 12, 0x000F000Fu, kH1024);
}
__device__ __forceinline__ void magic_high4(uint32_t r, uint32_t (&o)[4]) {
  o[0] = lop3_or_and(r << 4, 0x00F000F0u, kH1024);
  o[1] = lop3_or_and(r, 0x00F000F0u, kH1024);
  o[2] = lop3_or_and(r >> 4, 0x00F000F0u, kH1024);
  o[3] = lop3_or_and(r >> 8, 0x00F000F0u, kH1024);
}

// Activation operand layout.  Within each chunk of 16 consecutive inputs the
// FP16 values are stored in the order 0,1,8,9, 2,3,10,11, 4,5,12,13, 6,7,14,15
// (so lane tig's four B-fragment values are one 8-byte load), and inputs
// 8..15 of the chunk hold x / 16.  op_slot(k) is the storage index of input k.
__host__ __device__ __forceinline__ int op_slot(int k) {
  const int c = k & 15, base = k & ~15;
  return base + ((c < 8) ? (4 * (c >> 1) + (c & 1)) : (4 * ((c - 8) >> 1) + 2 + (c & 1)));
}
__host__ __device__ __forceinline__ bool op_high(int k) { return (k & 15) >= 8; }
// Grouped operand buffer of B rows: the B rows' values of each 64-input half
// group are stored together ([K/64][B][64] FP16, one 128-byte row per token), so
// a stage of consecutive groups is one contiguous copy; within a 128-byte row
// the 8 chunks of 8 values (op_slot order) are XOR-permuted by (row & 7).  That
// is the 128-byte-swizzled K-major layout the tensor cores read through a
// shared-memory descriptor (8-row, 1024-byte atoms), and it keeps the
// B-fragment loads of 8 rows on different shared-memory banks.  op_index(t, k,
// B) is the element index of input k of row t.
__host__ __device__ __forceinline__ int op_index(int t, int k, int B) {
  const int p = op_slot(k & 63);
  return ((k >> 6) * B + t) * 64 + (((p >> 3) ^ (t & 7)) << 3) + (p & 7);
}
// Byte offset, within a 128-byte half-group row, of lane tig's 8-byte B fragment
// of k-step ks (0..3 within the half) for a row whose (row & 7) is `key`.
__device__ __forceinline__ int op_frag_off(int ks, int tig, int key) {
  return ((((2 * ks) + (tig >> 1)) ^ key) << 4) + ((tig & 1) << 3);
}
// Group offsets S.  Every FP16 value is a multiple of 2^-24 (the smallest
// subnormal), so each term 1032 h or 1152 h is an exact FP32 value and an
// integer number of 2^-24 units.  Terms are first summed in FP32 inside one
// warp in a fixed order (deterministic), then converted once to a 64-bit count
// of 2^-24 units; sums of those integers, across warps, CTAs and atomics, do
// not depend on the order of their terms, so S is the same whichever CTA
// finishes first.  It is rounded once more, to FP32, where an MMA chain starts
// at -S.
typedef long long sfix_t;
// FP32 -> count of 2^-24 units (nearest), with 32-bit conversions only: the
// value w = v 2^24 splits exactly into hi 2^32 + rem, 0 <= rem < 2^32.
__device__ __forceinline__ sfix_t f32_to_sfix(float v) {
  const float w = v * 16777216.0f;                         // exact (power of two)
  const float hi = floorf(v * 0.00390625f);                // floor(w / 2^32), exact scaling
  const float rem = fmaf(-hi, 4294967296.0f, w);           // the low bits of w: exact
  return (sfix_t)((unsigned long long)(long long)__float2int_rn(hi) << 32) +
         (sfix_t)__float2uint_rn(rem);
}
// Count of 2^-24 units -> FP32 from its two 32-bit halves (32-bit conversions
// only); deterministic, within 2 FP32 ulps of the exact value.
__device__ __forceinline__ float sfix_to_f32(sfix_t s) {
  const float hi = __int2float_rn((int)(s >> 32)), lo = __uint2float_rn((unsigned)(unsigned long long)s);
  return fmaf(hi, 4294967296.0f, lo) * 5.9604644775390625e-08f;  // x 2^-24
}

// FP16 operand value of input k and its contribution to the group offset S
// (exact in FP32: an 11-bit significand times 1032 or 1152).
__device__ __forceinline__ __half op_encode(float x, int k, float& s_term) {
  const __half h = __float2half_rn(op_high(k) ? x * 0.0625f : x);
  s_term = (op_high(k) ? kOffHi : kOffLo) * __half2float(h);
  return h;
}
__device__ __forceinline__ void sfix_atomic_add(sfix_t* p, sfix_t v) {
  atomicAdd(reinterpret_cast<unsigned long long*>(p), (unsigned long long)v);
}

// ------------------------------------------------------------------ packed weights
// Row-tile-major: [row tile T][group kg] -> one 1056-byte slab: 1024 bytes of
// nibbles (two 512-byte halves for k-steps 0-3 and 4-7, 16 bytes per lane)
// followed by 8 x (bf16 s[g], bf16 s[g+8]).  Nibble i of the word for
// (lane = 4g + tig, k-step ks) holds
//   row  g + (i & 2 ? 8 : 0),  column  16 ks + 2 tig + (i & 1 ? 8 : 0) + (i & 4 ? 1 : 0)
// so that magic_word() yields the m16n8k16 A fragment {r0, r2, r1, r3}.
__host__ __device__ __forceinline__ int wslab_word_offset(int lane, int ks) {
  return (ks >> 2) * 512 + lane * 16 + (ks & 3) * 4;
}
__host__ __device__ __forceinline__ int wnib_row(int g, int i) { return g + ((i & 2) ? 8 : 0); }
__host__ __device__ __forceinline__ int wnib_col(int ks, int tig, int i) {
  return 16 * ks + 2 * tig + ((i & 1) ? 8 : 0) + ((i & 4) ? 1 : 0);
}

// Logical row of packed row r (0..15) of global row tile T for a role.
__host__ __device__ __forceinline__ int64_t packed_row_to_logical(int role, int inter, int64_t T, int r) {
  if (role == FT_W_GATEUP) return (r < 8) ? (8 * T + r) : (int64_t)inter + 8 * T + (r - 8);
  return T * kRowTile + r;
}

// ------------------------------------------------------------------ KV entries
// K entry (d/2 bytes): chunk tig (d/8 bytes) word j, nibble i holds channel
//   16 (2j + ((i >> 1) & 1)) + 2 tig + (i & 1 ? 8 : 0) + ((i >> 2) & 1)
// V entry (d/2 bytes): chunk g (d/16 bytes) word j, nibble i holds channel
//   16 (4j + (i >> 1)) + g + (i & 1 ? 8 : 0)
__host__ __device__ __forceinline__ int kv_k_channel(int tig, int j, int i) {
  return 16 * (2 * j + ((i >> 1) & 1)) + 2 * tig + ((i & 1) ? 8 : 0) + ((i >> 2) & 1);
}
__host__ __device__ __forceinline__ int kv_v_channel(int g, int j, int i) {
  return 16 * (4 * j + (i >> 1)) + g + ((i & 1) ? 8 : 0);
}

struct KVLayout {
  int d, nkv, max_batch, max_ctx;
  size_t entry;        // d/2 bytes of one K (or V) entry
  size_t kc, vc, ks, vs, total;
  __host__ __device__ size_t row(int b, int h, int p) const {
    return ((size_t)(b * nkv + h) * (size_t)max_ctx + (size_t)p);
  }
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline KVLayout kv_layout(const ft_block_cfg& c, int max_batch, int max_ctx) {
  KVLayout L;
  L.d = c.head_dim;
  L.nkv = c.n_kv;
  L.max_batch = max_batch;
  L.max_ctx = max_ctx;
  L.entry = (size_t)c.head_dim / 2;
  const size_t n = (size_t)max_batch * c.n_kv * (size_t)max_ctx;
  L.kc = 0;
  L.vc = align_up(n * L.entry, 256);
  L.ks = L.vc + align_up(n * L.entry, 256);
  L.vs = L.ks + align_up(n * 2, 256);
  L.total = L.vs + align_up(n * 2, 256);
  return L;
}

// ------------------------------------------------------------------ misc device
__device__ __forceinline__ void set_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Symmetric INT4 quantiser decision (FP32): s = bf16_rne(amax / 7); code =
// clamp(rne(x / s), -8, 7) + 8; s = 0 gives code 8.
__device__ __forceinline__ uint16_t quant_scale_bits(float amax) {
  const float q = __fdiv_rn(amax, 7.0f);
  return __bfloat16_as_ushort(__float2bfloat16_rn(q));
}
__device__ __forceinline__ uint32_t quant_code(float x, float s) {
  if (s == 0.0f) return 8u;
  float t = rintf(__fdiv_rn(x, s));
  t = fminf(fmaxf(t, -8.0f), 7.0f);
  return (uint32_t)((int)t + 8);
}

// E4M3 decode weights: s = bf16(amax / 448) (448 = the largest E4M3 magnitude),
// code = E4M3(x / s) rounded to nearest even, saturating at +-448; s = 0 gives 0.
__device__ __forceinline__ uint16_t quant_scale_bits_e4m3(float amax) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(__fdiv_rn(amax, 448.0f)));
}
__device__ __forceinline__ uint32_t quant_code_e4m3(float x, float s) {
  if (s == 0.0f) return 0u;
  return (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3);
}
// Two E4M3 codes (low byte first) -> an FP16 pair (every E4M3 value is exact in FP16).
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xFFFFu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
// The four A-fragment registers of one k-step from its 8 packed E4M3 codes
// (lo: row g inputs c, c+1, c+8, c+9; hi: row g+8, the same inputs), in the
// order the INT4 decode produces them (rows g | g+8 x inputs c.. | c+8..), the
// inputs 8..15 of the step scaled by 16 to match the activation operand (x / 16).
__device__ __forceinline__ void e4m3_words(uint32_t lo, uint32_t hi, uint32_t* r) {
  const __half2 x16 = __floats2half2_rn(16.0f, 16.0f);
  const uint32_t u1 = e4m3x2_to_h2(lo >> 16), u3 = e4m3x2_to_h2(hi >> 16);
  const __half2 a2 = __hmul2(*reinterpret_cast<const __half2*>(&u1), x16);
  const __half2 a3 = __hmul2(*reinterpret_cast<const __half2*>(&u3), x16);
  r[0] = e4m3x2_to_h2(lo);
  r[1] = *reinterpret_cast<const uint32_t*>(&a2);
  r[2] = e4m3x2_to_h2(hi);
  r[3] = *reinterpret_cast<const uint32_t*>(&a3);
}

// Fast Walsh-Hadamard transform of a d-vector held stride-32 across a warp:
// lane l owns channels l + 32 m (m < NPL = d / 32).  Butterflies for strides
// < hb give the natural-order Sylvester transform on each hb block; the
// result is scaled by 1 / sqrt(hb).
template <int NPL>
__device__ __forceinline__ void warp_fwht(float (&v)[NPL], int hb) {
  const int lane = threadIdx.x & 31;
  for (int s = 1; s < hb && s < 32; s <<= 1) {
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      const float o = __shfl_xor_sync(0xffffffffu, v[m], s);
      v[m] = (lane & s) ? (o - v[m]) : (v[m] + o);
    }
  }
#pragma unroll
  for (int sm = 1; sm < NPL; sm <<= 1) {
    if (sm * 32 >= hb) break;
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      if (m & sm) continue;
      const float a = v[m], b = v[m + sm];
      v[m] = a + b;
      v[m + sm] = a - b;
    }
  }
  const float sc = __frsqrt_rn((float)hb);
#pragma unroll
  for (int m = 0; m < NPL; ++m) v[m] *= sc;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


// Quantise one rotated d-vector (stride-32 ownership, kv_group = d) and write
// its K- or V-entry nibbles and BF16 scale.  Returns the decoded values
// (c - 8) * s in v.  `codes` is a warp-private staging area of d bytes.
template <int NPL>
__device__ __forceinline__ void warp_quant_store(float (&v)[NPL], bool is_k, uint8_t* codes,
                                                 uint8_t* entry, uint16_t* scale_out) {
  const int lane = threadIdx.x & 31;
  constexpr int D = NPL * 32;
  float am = 0.0f;
#pragma unroll
  for (int m = 0; m < NPL; ++m) am = fmaxf(am, fabsf(v[m]));
  am = warp_max(am);
  const uint16_t sb = quant_scale_bits(am);
  const float s = bf16_bits_to_f32(sb);
#pragma unroll
  for (int m = 0; m < NPL; ++m) {
    const uint32_t c = quant_code(v[m], s);
    codes[lane + 32 * m] = (uint8_t)c;
    v[m] = (float)((int)c - 8) * s;
  }
  __syncwarp();
  constexpr int WORDS = D / 8;  // 32-bit words per entry
  if (lane < WORDS) {
    uint32_t w = 0;
    if (is_k) {
      const int tig = lane / (D / 32), j = lane % (D / 32);
#pragma unroll
      for (int i = 0; i < 8; ++i) w |= (uint32_t)codes[kv_k_channel(tig, j, i)] << (4 * i);
      *reinterpret_cast<uint32_t*>(entry + tig * (D / 8) + 4 * j) = w;
    } else {
      const int g = lane / (D / 64), j = lane % (D / 64);
#pragma unroll
      for (int i = 0; i < 8; ++i) w |= (uint32_t)codes[kv_v_channel(g, j, i)] << (4 * i);
      *reinterpret_cast<uint32_t*>(entry + g * (D / 16) + 4 * j) = w;
    }
  }
  if (lane == 0) *scale_out = sb;
  __syncwarp();
}

}  // namespace ft

// ------------------------------------------------------------------ host utils
namespace ft_host {

int num_sms();
int smem_per_sm();  // shared memory per SM in bytes (0 if unknown)
bool pdl_enabled();
int check_cfg(const ft_block_cfg* c);
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace ft_host
