// KV cache: rotate, quantise and place new K/V entries (summary page, "무엇과
// 다른가": a block-diagonal Hadamard transform before INT4 cache quantisation;
// "어떻게 동작하나": direct placement at offset(request, head, position, channel)).
//
// Cache layout for one layer (KVLayout): four regions
//   K nibbles [max_batch][n_kv][max_ctx][d/2], V nibbles (same),
//   K scales  [max_batch][n_kv][max_ctx] BF16, V scales (same).
// Within an entry the nibbles are permuted (kv_k_channel / kv_v_channel) so that
// the attention kernel's 16-byte / 8-byte loads land directly in tensor-core
// fragment order: K as the A operand of q.K (rows = positions), V as the A
// operand of P.V (rows = channels, two positions per register).
#include "ft_internal.cuh"

namespace ft {

template <int NPL>
__global__ void __launch_bounds__(128) kv_append_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                                        const int32_t* __restrict__ pos, uint8_t* __restrict__ cache,
                                                        KVLayout L, int B, int T, int hb, int32_t* status) {
  constexpr int D = NPL * 32;
  __shared__ uint8_t stage[4][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;
  if (idx >= B * T * L.nkv) return;
  const int h = idx % L.nkv, t = (idx / L.nkv) % T, b = idx / (L.nkv * T);
  const int p0 = pos[b];
  if (p0 < 0 || p0 + T > L.max_ctx) {
    if (lane == 0 && t == 0 && h == 0) set_status(status, FT_DEV_CAPACITY);
    return;
  }
  const int p = p0 + t;
  const size_t src = ((size_t)(b * T + t) * L.nkv + h) * D;
  const size_t row = L.row(b, h, p);
  float x[NPL];
#pragma unroll
  for (int m = 0; m < NPL; ++m) x[m] = bf16_bits_to_f32(k[src + lane + 32 * m]);
  warp_fwht<NPL>(x, hb);
  warp_quant_store<NPL>(x, true, stage[warp], cache + L.kc + row * L.entry,
                        reinterpret_cast<uint16_t*>(cache + L.ks) + row);
#pragma unroll
  for (int m = 0; m < NPL; ++m) x[m] = bf16_bits_to_f32(v[src + lane + 32 * m]);
  warp_fwht<NPL>(x, hb);
  warp_quant_store<NPL>(x, false, stage[warp], cache + L.vc + row * L.entry,
                        reinterpret_cast<uint16_t*>(cache + L.vs) + row);
}

// Ragged placement: packed token i (rows of all requests back to back, request b
// owning rows cu[b] .. cu[b+1]-1) goes to position pos[b] + i - cu[b] of request b.
// One warp per (token, head) finds b by binary search over the prefix sums and
// checks its bracket, so every write stays inside request b's cache row.
template <int NPL>
__global__ void __launch_bounds__(128) kv_append_ragged_kernel(const uint16_t* __restrict__ k,
                                                               const uint16_t* __restrict__ v,
                                                               const int32_t* __restrict__ cu,
                                                               const int32_t* __restrict__ pos,
                                                               uint8_t* __restrict__ cache, KVLayout L, int B,
                                                               int total, int hb, int32_t* status) {
  constexpr int D = NPL * 32;
  __shared__ uint8_t stage[4][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;
  if (idx >= total * L.nkv) return;
  const int h = idx % L.nkv, i = idx / L.nkv;
  if (cu[0] != 0 || cu[B] != total) {  // not a prefix-sum map of `total` rows
    if (lane == 0) set_status(status, FT_DEV_RANGE);
    return;
  }
  int lo = 0, hi = B;  // cu[lo] <= i < cu[hi] for a non-decreasing map
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= i) lo = mid; else hi = mid;
  }
  const int b = lo, c0 = cu[b], c1 = cu[b + 1];
  if (!(c0 <= i && i < c1)) {  // the map decreases somewhere
    if (lane == 0) set_status(status, FT_DEV_RANGE);
    return;
  }
  const int p0 = pos[b];
  if (p0 < 0 || p0 > L.max_ctx - (c1 - c0)) {
    if (lane == 0 && i == c0 && h == 0) set_status(status, FT_DEV_CAPACITY);
    return;
  }
  const size_t src = ((size_t)i * L.nkv + h) * D;
  const size_t row = L.row(b, h, p0 + (i - c0));
  float x[NPL];
#pragma unroll
  for (int m = 0; m < NPL; ++m) x[m] = bf16_bits_to_f32(k[src + lane + 32 * m]);
  warp_fwht<NPL>(x, hb);
  warp_quant_store<NPL>(x, true, stage[warp], cache + L.kc + row * L.entry,
                        reinterpret_cast<uint16_t*>(cache + L.ks) + row);
#pragma unroll
  for (int m = 0; m < NPL; ++m) x[m] = bf16_bits_to_f32(v[src + lane + 32 * m]);
  warp_fwht<NPL>(x, hb);
  warp_quant_store<NPL>(x, false, stage[warp], cache + L.vc + row * L.entry,
                        reinterpret_cast<uint16_t*>(cache + L.vs) + row);
}

__global__ void kv_unpack_kernel(const uint8_t* __restrict__ cache, KVLayout L, int B, int len,
                                 uint8_t* __restrict__ kc, uint8_t* __restrict__ vc, uint16_t* __restrict__ ks,
                                 uint16_t* __restrict__ vs) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)B * L.nkv * len) return;
  const int p = (int)(idx % len), h = (int)((idx / len) % L.nkv), b = (int)(idx / ((int64_t)len * L.nkv));
  const size_t row = L.row(b, h, p);
  const int D = L.d;
  const uint8_t* ke = cache + L.kc + row * L.entry;
  const uint8_t* ve = cache + L.vc + row * L.entry;
  uint8_t* ko = kc + idx * D;
  uint8_t* vo = vc + idx * D;
  for (int tig = 0; tig < 4; ++tig)
    for (int j = 0; j < D / 32; ++j) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(ke + tig * (D / 8) + 4 * j);
      for (int i = 0; i < 8; ++i) ko[kv_k_channel(tig, j, i)] = (uint8_t)((w >> (4 * i)) & 0xF);
    }
  for (int g = 0; g < 8; ++g)
    for (int j = 0; j < D / 64; ++j) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(ve + g * (D / 16) + 4 * j);
      for (int i = 0; i < 8; ++i) vo[kv_v_channel(g, j, i)] = (uint8_t)((w >> (4 * i)) & 0xF);
    }
  ks[idx] = reinterpret_cast<const uint16_t*>(cache + L.ks)[row];
  vs[idx] = reinterpret_cast<const uint16_t*>(cache + L.vs)[row];
}

}  // namespace ft

extern "C" {

size_t ft_kv_cache_bytes(const ft_block_cfg* c, int max_batch, int max_ctx) {
  if (ft_host::check_cfg(c) != FT_OK || max_batch <= 0 || max_ctx <= 0) return 0;
  return ft::kv_layout(*c, max_batch, max_ctx).total;
}

int ft_kv_append_int4(const ft_block_cfg* c, void* cache, int max_batch, int max_ctx, const uint16_t* k_bf16,
                      const uint16_t* v_bf16, const int32_t* pos, int B, int T, int32_t* dev_status,
                      ft_stream stream) {
  int st = ft_host::check_cfg(c);
  if (st != FT_OK) return st;
  if (!cache || !k_bf16 || !v_bf16 || !pos || !ft_host::aligned16(cache)) return FT_ERR_INVALID_ARG;
  if (max_batch <= 0 || max_ctx <= 0 || B <= 0 || T <= 0) return FT_ERR_INVALID_ARG;
  if (B > max_batch) return FT_ERR_CAPACITY;
  if (T > max_ctx) return FT_ERR_CAPACITY;
  const ft::KVLayout L = ft::kv_layout(*c, max_batch, max_ctx);
  const int64_t warps = (int64_t)B * T * c->n_kv;
  if (warps > (int64_t)INT32_MAX) return FT_ERR_UNSUPPORTED;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  auto* cp = static_cast<uint8_t*>(cache);
  if (c->head_dim == 128)
    ft::kv_append_kernel<4><<<blocks, 128, 0, (cudaStream_t)stream>>>(k_bf16, v_bf16, pos, cp, L, B, T, c->had_block,
                                                                      dev_status);
  else
    ft::kv_append_kernel<2><<<blocks, 128, 0, (cudaStream_t)stream>>>(k_bf16, v_bf16, pos, cp, L, B, T, c->had_block,
                                                                      dev_status);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_kv_append_ragged_int4(const ft_block_cfg* c, void* cache, int max_batch, int max_ctx,
                             const uint16_t* k_bf16, const uint16_t* v_bf16, const int32_t* cu_seqlens,
                             const int32_t* pos, int B, int total, int32_t* dev_status, ft_stream stream) {
  int st = ft_host::check_cfg(c);
  if (st != FT_OK) return st;
  if (!cache || !cu_seqlens || !pos || !ft_host::aligned16(cache)) return FT_ERR_INVALID_ARG;
  if (max_batch <= 0 || max_ctx <= 0 || B <= 0 || total < 0) return FT_ERR_INVALID_ARG;
  if (B > max_batch) return FT_ERR_CAPACITY;
  if (total == 0) return FT_OK;
  if (!k_bf16 || !v_bf16) return FT_ERR_INVALID_ARG;
  const ft::KVLayout L = ft::kv_layout(*c, max_batch, max_ctx);
  const int64_t warps = (int64_t)total * c->n_kv;
  if (warps > (int64_t)INT32_MAX) return FT_ERR_UNSUPPORTED;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  auto* cp = static_cast<uint8_t*>(cache);
  if (c->head_dim == 128)
    ft::kv_append_ragged_kernel<4><<<blocks, 128, 0, (cudaStream_t)stream>>>(k_bf16, v_bf16, cu_seqlens, pos, cp, L,
                                                                             B, total, c->had_block, dev_status);
  else
    ft::kv_append_ragged_kernel<2><<<blocks, 128, 0, (cudaStream_t)stream>>>(k_bf16, v_bf16, cu_seqlens, pos, cp, L,
                                                                             B, total, c->had_block, dev_status);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_kv_unpack_int4(const ft_block_cfg* c, const void* cache, int max_batch, int max_ctx, int B, int len,
                      uint8_t* k_codes, uint8_t* v_codes, uint16_t* k_scales, uint16_t* v_scales, ft_stream stream) {
  int st = ft_host::check_cfg(c);
  if (st != FT_OK) return st;
  if (!cache || !k_codes || !v_codes || !k_scales || !v_scales) return FT_ERR_INVALID_ARG;
  if (B <= 0 || len <= 0 || B > max_batch || len > max_ctx) return FT_ERR_INVALID_ARG;
  const ft::KVLayout L = ft::kv_layout(*c, max_batch, max_ctx);
  const int64_t n = (int64_t)B * c->n_kv * len;
  ft::kv_unpack_kernel<<<(unsigned)((n + 127) / 128), 128, 0, (cudaStream_t)stream>>>(
      static_cast<const uint8_t*>(cache), L, B, len, k_codes, v_codes, k_scales, v_scales);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

}  // extern "C"
