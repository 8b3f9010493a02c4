// Weight packing: RMSNorm-gain folding, symmetric INT4 group quantisation with
// BF16 scales, and the kernel-native layout (summary page, "어떻게 동작하나":
// W' = gamma W before quantisation; "무엇과 다른가": INT4 values with group
// scales, stored in the order the decode kernels consume them).
//
// Layout of a packed role with N_out rows and K_in inputs (row-tile-major):
//   [row tile T < N/16][group kg < K/128] -> one 1056-byte slab
//   slab = 1024 bytes of nibbles (two 512-byte halves: k-steps 0-3 and 4-7,
//          lane-major 16 bytes each) + 8 x (bf16 s[g], bf16 s[g+8]).
// A row tile's whole input range is contiguous, so the GEMV streams any run
// of (row tile, group) units with one bulk copy per row tile.
#include "ft_internal.cuh"

namespace ft {

__global__ void __launch_bounds__(256) pack_kernel(const float* __restrict__ W, const float* __restrict__ gamma,
                                                   uint8_t* __restrict__ out, int role, int inter, int K, int NKG) {
  __shared__ float wv[16][129];
  __shared__ float srow[16];
  __shared__ uint16_t sbits[16];
  const int T = blockIdx.x, kg = blockIdx.y, t = threadIdx.x;
  // pass 1: W' = W * gamma (FP32) and the per-row group amax
  {
    const int r = t >> 4, part = t & 15;
    const int64_t row = packed_row_to_logical(role, inter, T, r);
    const float* src = W + row * (int64_t)K + (int64_t)kg * kWGroup + part * 8;
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float w = src[i];
      if (gamma) w = __fmul_rn(w, gamma[kg * kWGroup + part * 8 + i]);
      wv[r][part * 8 + i] = w;
      am = fmaxf(am, fabsf(w));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (part == 0) {
      const uint16_t b = quant_scale_bits(am);
      sbits[r] = b;
      srow[r] = bf16_bits_to_f32(b);
    }
  }
  __syncthreads();
  uint8_t* slab = out + ((size_t)T * NKG + kg) * kSlabBytes;
  // pass 2: one 32-bit word of 8 nibbles per thread, in A-fragment order
  {
    const int ks = t >> 5, lane = t & 31, g = lane >> 2, tig = lane & 3;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = wnib_row(g, i), c = wnib_col(ks, tig, i);
      w |= quant_code(wv[r][c], srow[r]) << (4 * i);
    }
    *reinterpret_cast<uint32_t*>(slab + wslab_word_offset(lane, ks)) = w;
  }
  if (t < 8) {
    const uint32_t pair = (uint32_t)sbits[t] | ((uint32_t)sbits[t + 8] << 16);
    *reinterpret_cast<uint32_t*>(slab + kSlabCodes + 4 * t) = pair;
  }
}

__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ codes,
                                                     uint16_t* __restrict__ scales, int role, int inter, int K,
                                                     int NKG) {
  const int T = blockIdx.x, kg = blockIdx.y, t = threadIdx.x;
  const uint8_t* slab = in + ((size_t)T * NKG + kg) * kSlabBytes;
  const int ks = t >> 5, lane = t & 31, g = lane >> 2, tig = lane & 3;
  const uint32_t w = *reinterpret_cast<const uint32_t*>(slab + wslab_word_offset(lane, ks));
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = wnib_row(g, i), c = wnib_col(ks, tig, i);
    const int64_t row = packed_row_to_logical(role, inter, T, r);
    codes[row * (int64_t)K + (int64_t)kg * kWGroup + c] = (uint8_t)((w >> (4 * i)) & 0xF);
  }
  if (t < 16) {
    const uint16_t b = *reinterpret_cast<const uint16_t*>(slab + kSlabCodes + 4 * (t & 7) + 2 * (t >> 3));
    const int64_t row = packed_row_to_logical(role, inter, T, t);
    scales[row * (int64_t)NKG + kg] = b;
  }
}

// E4M3 decode weights: the same pass 1 (gain folding, group amax) with s =
// bf16(amax / 448); pass 2 writes per (128-input half, lane, k-step) 8 codes:
// row g inputs c, c+1, c+8, c+9, then row g+8 the same, c = 16 ks + 2 tig
// (ks the k-step of the group, g = lane / 4, tig = lane % 4), at half * 1024 +
// lane * 32 + (ks % 4) * 8: a decoder lane reads its half's 32 bytes with two
// 16-byte loads.  Scales as for INT4, after the 2048 bytes of codes.
__global__ void __launch_bounds__(256) pack_e4m3_kernel(const float* __restrict__ W, const float* __restrict__ gamma,
                                                        uint8_t* __restrict__ out, int role, int inter, int K,
                                                        int NKG) {
  __shared__ float wv[16][129];
  __shared__ float srow[16];
  __shared__ uint16_t sbits[16];
  const int T = blockIdx.x, kg = blockIdx.y, t = threadIdx.x;
  {
    const int r = t >> 4, part = t & 15;
    const int64_t row = packed_row_to_logical(role, inter, T, r);
    const float* src = W + row * (int64_t)K + (int64_t)kg * kWGroup + part * 8;
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float w = src[i];
      if (gamma) w = __fmul_rn(w, gamma[kg * kWGroup + part * 8 + i]);
      wv[r][part * 8 + i] = w;
      am = fmaxf(am, fabsf(w));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (part == 0) {
      const uint16_t b = quant_scale_bits_e4m3(am);
      sbits[r] = b;
      srow[r] = bf16_bits_to_f32(b);
    }
  }
  __syncthreads();
  uint8_t* slab = out + ((size_t)T * NKG + kg) * kSlabBytesE4;
  {
    const int half = t >> 7, lane = (t >> 2) & 31, ks = t & 3, g = lane >> 2, tig = lane & 3;
    const int c = 16 * (4 * half + ks) + 2 * tig;
    const int cols[4] = {c, c + 1, c + 8, c + 9};
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lo |= quant_code_e4m3(wv[g][cols[j]], srow[g]) << (8 * j);
      hi |= quant_code_e4m3(wv[g + 8][cols[j]], srow[g + 8]) << (8 * j);
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(slab + half * 1024 + lane * 32 + ks * 8);
    dst[0] = lo;
    dst[1] = hi;
  }
  if (t < 8) {
    const uint32_t pair = (uint32_t)sbits[t] | ((uint32_t)sbits[t + 8] << 16);
    *reinterpret_cast<uint32_t*>(slab + kSlabCodesE4 + 4 * t) = pair;
  }
}

__global__ void __launch_bounds__(256) unpack_e4m3_kernel(const uint8_t* __restrict__ in, uint8_t* __restrict__ codes,
                                                          uint16_t* __restrict__ scales, int role, int inter, int K,
                                                          int NKG) {
  const int T = blockIdx.x, kg = blockIdx.y, t = threadIdx.x;
  const uint8_t* slab = in + ((size_t)T * NKG + kg) * kSlabBytesE4;
  const int half = t >> 7, lane = (t >> 2) & 31, ks = t & 3, g = lane >> 2, tig = lane & 3;
  const int c = 16 * (4 * half + ks) + 2 * tig;
  const int cols[4] = {c, c + 1, c + 8, c + 9};
  const uint32_t* src = reinterpret_cast<const uint32_t*>(slab + half * 1024 + lane * 32 + ks * 8);
  const uint32_t lo = src[0], hi = src[1];
  const int64_t r0 = packed_row_to_logical(role, inter, T, g), r1 = packed_row_to_logical(role, inter, T, g + 8);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    codes[r0 * (int64_t)K + (int64_t)kg * kWGroup + cols[j]] = (uint8_t)(lo >> (8 * j));
    codes[r1 * (int64_t)K + (int64_t)kg * kWGroup + cols[j]] = (uint8_t)(hi >> (8 * j));
  }
  if (t < 16) {
    const uint16_t b = *reinterpret_cast<const uint16_t*>(slab + kSlabCodesE4 + 4 * (t & 7) + 2 * (t >> 3));
    const int64_t row = packed_row_to_logical(role, inter, T, t);
    scales[row * (int64_t)NKG + kg] = b;
  }
}

}  // namespace ft

extern "C" {

int ft_pack_weights_int4(const ft_block_cfg* c, int role, const float* W, const float* gamma, void* packed,
                         size_t packed_bytes, ft_stream stream) {
  int32_t n, k;
  int st = ft_weight_shape(c, role, &n, &k);
  if (st != FT_OK) return st;
  if (!W || !packed || !ft_host::aligned16(packed) || !ft_host::aligned16(W)) return FT_ERR_INVALID_ARG;
  if (c->weight_format != FT_WFMT_INT4) return FT_ERR_INVALID_ARG;
  if (packed_bytes < ft_packed_weight_bytes(c, role)) return FT_ERR_WORKSPACE;
  dim3 grid(n / ft::kRowTile, k / ft::kWGroup);
  ft::pack_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(W, gamma, static_cast<uint8_t*>(packed), role, c->inter,
                                                          k, k / ft::kWGroup);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_unpack_weights_int4(const ft_block_cfg* c, int role, const void* packed, uint8_t* codes,
                           uint16_t* scales_bf16, ft_stream stream) {
  int32_t n, k;
  int st = ft_weight_shape(c, role, &n, &k);
  if (st != FT_OK) return st;
  if (!packed || !codes || !scales_bf16 || !ft_host::aligned16(packed)) return FT_ERR_INVALID_ARG;
  if (c->weight_format != FT_WFMT_INT4) return FT_ERR_INVALID_ARG;
  dim3 grid(n / ft::kRowTile, k / ft::kWGroup);
  ft::unpack_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(static_cast<const uint8_t*>(packed), codes, scales_bf16,
                                                            role, c->inter, k, k / ft::kWGroup);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_pack_weights_e4m3(const ft_block_cfg* c, int role, const float* W, const float* gamma, void* packed,
                         size_t packed_bytes, ft_stream stream) {
  int32_t n, k;
  int st = ft_weight_shape(c, role, &n, &k);
  if (st != FT_OK) return st;
  if (!W || !packed || !ft_host::aligned16(packed) || !ft_host::aligned16(W)) return FT_ERR_INVALID_ARG;
  if (c->weight_format != FT_WFMT_E4M3) return FT_ERR_INVALID_ARG;
  if (packed_bytes < ft_packed_weight_bytes(c, role)) return FT_ERR_WORKSPACE;
  dim3 grid(n / ft::kRowTile, k / ft::kWGroup);
  ft::pack_e4m3_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(W, gamma, static_cast<uint8_t*>(packed), role,
                                                               c->inter, k, k / ft::kWGroup);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_unpack_weights_e4m3(const ft_block_cfg* c, int role, const void* packed, uint8_t* codes,
                           uint16_t* scales_bf16, ft_stream stream) {
  int32_t n, k;
  int st = ft_weight_shape(c, role, &n, &k);
  if (st != FT_OK) return st;
  if (!packed || !codes || !scales_bf16 || !ft_host::aligned16(packed)) return FT_ERR_INVALID_ARG;
  if (c->weight_format != FT_WFMT_E4M3) return FT_ERR_INVALID_ARG;
  dim3 grid(n / ft::kRowTile, k / ft::kWGroup);
  ft::unpack_e4m3_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(static_cast<const uint8_t*>(packed), codes,
                                                                 scales_bf16, role, c->inter, k, k / ft::kWGroup);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

}  // extern "C"
