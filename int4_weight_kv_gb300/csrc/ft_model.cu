// Full-model step helpers around the decode block (a complete Llama-3.1-8B
// decode step at batch 1 is quoted on the summary page, "전제와 한계"):
// BF16 embedding gather and the final RMSNorm fused into a BF16 LM-head GEMV.
//
// LM head (HBM-bound: V x H BF16 weights streamed once).  Each warp streams
// 16-row tiles of W straight into registers with 16-byte non-allocating loads
// and runs mma.m16n8k16 (BF16 operands, FP32 accumulate).  Within every 32
// inputs the MMA's k order is permuted so that one 16-byte load of a row feeds
// the A fragments of two MMAs; the normalised activation z = gamma * rho(x) * x
// sits in shared memory as a BF16 (hi, lo) pair with the same permutation, so
// the product is accurate to ~2^-16 relative while W is read once per chunk of
// up to 8 tokens.  Work units are (row tile, quarter of H), strided over all
// warps for balance; the four quarters of a row tile always fall to four
// consecutive warps of one CTA, which add their partial sums through shared
// memory in quarter order and store the logits (no atomics: the result does
// not depend on timing).
#include <algorithm>

#include "ft_internal.cuh"

namespace ft {

__global__ void __launch_bounds__(256) embed_kernel(const uint16_t* __restrict__ table,
                                                    const int32_t* __restrict__ tokens, float* __restrict__ out,
                                                    int V, int H, int32_t* status) {
  const int b = blockIdx.x;
  const int tok = tokens[b];
  const bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) set_status(status, FT_DEV_RANGE);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    out[(size_t)b * H + i] = ok ? bf16_bits_to_f32(table[(size_t)tok * H + i]) : 0.0f;
}

// z[b, :] = bf16(gamma * rho_b * x[b, :]), rho_b = (mean_i x[b, i]^2 + eps)^-1/2.
// One CTA per row: sum of squares (FP32, tree over warps), then the scaled row.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                                                      uint16_t* __restrict__ z, int H, float eps) {
  __shared__ float red[8];
  const int b = blockIdx.x, tid = threadIdx.x;
  const float* row = x + (size_t)b * H;
  float ss = 0.0f;
  for (int i = tid; i < H; i += 256) {
    const float v = __ldcg(row + i);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) t += red[w];
  const float rho = rsqrtf(t / (float)H + eps);
  for (int i = tid; i < H; i += 256)
    z[(size_t)b * H + i] = __bfloat16_as_ushort(__float2bfloat16_rn(gamma[i] * (rho * __ldcg(row + i))));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kHeadWarps = 16;
constexpr int kHeadKSplit = 4;  // quarters of H: warps 4j .. 4j + 3 of a CTA share a row tile
static_assert(kHeadWarps % kHeadKSplit == 0, "row tiles are split within groups of warps");
constexpr int kHeadLook = 4;  // 32-input chunks in flight per warp

// z rows in shared memory: [B][H] hi then [B][H] lo (BF16 bits), natural order.
__global__ void __launch_bounds__(kHeadWarps * 32, 1) lm_head_kernel(const float* __restrict__ x,
                                                                     const float* __restrict__ gamma,
                                                                     const uint16_t* __restrict__ W,
                                                                     float* __restrict__ logits, int B, int V, int H,
                                                                     float eps) {
  extern __shared__ __align__(16) uint16_t zs[];
  __shared__ float red[kHeadWarps];
  __shared__ float part[kHeadWarps][4][32];  // [warp][output register][lane]
  __shared__ float rho[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  // final RMSNorm of every token row, then z = gamma * rho * x as BF16 hi + lo
  for (int b = 0; b < B; ++b) {
    float ss = 0.0f;
    for (int i = tid; i < H; i += blockDim.x) {
      const float v = __ldcg(x + (size_t)b * H + i);
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.0f;
      for (int w = 0; w < kHeadWarps; ++w) t += red[w];
      rho[b] = rsqrtf(t / (float)H + eps);
    }
    __syncthreads();
  }
  for (int i = tid; i < B * H; i += blockDim.x) {
    const int b = i / H, k = i - b * H;
    const float z = gamma[k] * (rho[b] * __ldcg(x + i));
    const __nv_bfloat16 hi = __float2bfloat16_rn(z);
    const __nv_bfloat16 lo = __float2bfloat16_rn(z - __bfloat162float(hi));
    zs[i] = __bfloat16_as_ushort(hi);
    zs[B * H + i] = __bfloat16_as_ushort(lo);
  }
  __syncthreads();

  const int ntile = (V + 15) / 16;
  const int kq = H / kHeadKSplit;  // inputs per unit (a multiple of 32)
  const int nunit = ntile * kHeadKSplit;
  // unit % kHeadKSplit == warp % kHeadKSplit (nw is a multiple of it): quarter q of row tile T
  // runs on warp kHeadKSplit * j + q of the CTA that holds the tile, in the same iteration
  const int gw = blockIdx.x * kHeadWarps + warp, nw = gridDim.x * kHeadWarps;
  const int grp = warp / kHeadKSplit;
  const int zrow = min(g, B - 1);
  const bool zvalid = g < B;
  for (int unit = gw; unit < nunit; unit += nw) {
    const int T = unit / kHeadKSplit, q = unit - T * kHeadKSplit;
    const int r0 = min(T * 16 + g, V - 1), r1 = min(T * 16 + g + 8, V - 1);
    const uint16_t* w0 = W + (size_t)r0 * H + q * kq + 8 * tig;
    const uint16_t* w1 = W + (size_t)r1 * H + q * kq + 8 * tig;
    const uint16_t* zh = zs + zrow * H + q * kq + 8 * tig;
    const uint16_t* zl = zs + B * H + zrow * H + q * kq + 8 * tig;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int nchunk = kq / 32;
    uint4 a[kHeadLook][2];
#pragma unroll
    for (int c = 0; c < kHeadLook; ++c) {
      if (c < nchunk) {
        a[c][0] = ld_stream_v4(w0 + 32 * c);
        a[c][1] = ld_stream_v4(w1 + 32 * c);
      }
    }
    for (int c0 = 0; c0 < nchunk; c0 += kHeadLook) {
#pragma unroll
      for (int c = 0; c < kHeadLook; ++c) {
        const int ch = c0 + c;
        if (ch >= nchunk) break;
        const uint4 p0 = a[c][0], p1 = a[c][1];
        if (ch + kHeadLook < nchunk) {
          a[c][0] = ld_stream_v4(w0 + 32 * (ch + kHeadLook));
          a[c][1] = ld_stream_v4(w1 + 32 * (ch + kHeadLook));
        }
        uint4 bh = *reinterpret_cast<const uint4*>(zh + 32 * ch);
        uint4 bl = *reinterpret_cast<const uint4*>(zl + 32 * ch);
        if (!zvalid) bh = bl = make_uint4(0u, 0u, 0u, 0u);
        // k-slots (2tig, 2tig+1 | 2tig+8, 2tig+9) of step 0 <-> inputs 8tig+0..3, of step 1 <-> 8tig+4..7
        mma_bf16(acc, p0.x, p1.x, p0.y, p1.y, bh.x, bh.y);
        mma_bf16(acc, p0.z, p1.z, p0.w, p1.w, bh.z, bh.w);
        mma_bf16(acc, p0.x, p1.x, p0.y, p1.y, bl.x, bl.y);
        mma_bf16(acc, p0.z, p1.z, p0.w, p1.w, bl.z, bl.w);
      }
    }
    // the quarters' partial sums, added in quarter order: warp q of the group finishes output
    // register q (c0 = (row g, token 2tig), c1 = (row g, token 2tig+1), c2, c3: row g + 8)
#pragma unroll
    for (int r = 0; r < 4; ++r) part[warp][r][lane] = acc[r];
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kHeadKSplit * 32) : "memory");
    {
      const int r = q;
      float v = part[grp * kHeadKSplit][r][lane];
#pragma unroll
      for (int j = 1; j < kHeadKSplit; ++j) v += part[grp * kHeadKSplit + j][r][lane];
      const int t = 2 * tig + (r & 1);
      const int row = T * 16 + g + ((r & 2) ? 8 : 0);
      if (t < B && row < V) logits[(size_t)t * V + row] = v;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "n"(kHeadKSplit * 32) : "memory");  // part is reused
  }
}

}  // namespace ft

extern "C" {

int ft_embed_bf16(const uint16_t* table, const int32_t* tokens, float* x_out, int B, int V, int H,
                  int32_t* dev_status, ft_stream stream) {
  if (!table || !tokens || !x_out || B < 1 || V < 1 || H < 1) return FT_ERR_INVALID_ARG;
  ft::embed_kernel<<<B, 256, 0, (cudaStream_t)stream>>>(table, tokens, x_out, V, H, dev_status);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_rmsnorm_bf16(const float* x, const float* gamma, uint16_t* z_out, int B, int H, float eps, ft_stream stream) {
  if (!x || !gamma || !z_out || B < 1 || H < 1 || !(eps >= 0.0f)) return FT_ERR_INVALID_ARG;
  ft::rmsnorm_kernel<<<B, 256, 0, (cudaStream_t)stream>>>(x, gamma, z_out, H, eps);
  return cudaGetLastError() == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_read_device_status(const int32_t* dev_status, int32_t* host_out, ft_stream stream) {
  if (!dev_status || !host_out) return FT_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(host_out, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
      cudaSuccess)
    return FT_ERR_CUDA;
  return cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

int ft_lm_head_bf16(const float* x, const float* gamma, const uint16_t* W, float* logits, int B, int V, int H,
                    float eps, ft_stream stream) {
  if (!x || !gamma || !W || !logits || B < 1 || V < 1 || H < 1) return FT_ERR_INVALID_ARG;
  if (!ft_host::aligned16(W) || !ft_host::aligned16(x)) return FT_ERR_INVALID_ARG;
  if (B > 32 || H % (32 * ft::kHeadKSplit)) return FT_ERR_UNSUPPORTED;
  // tokens in chunks of up to 8 (one MMA column tile) whose z rows fit in shared memory
  const int bc = std::min(8, (int)((160 * 1024) / ((size_t)H * 4)));
  if (bc < 1) return FT_ERR_UNSUPPORTED;
  const size_t smem = (size_t)std::min(B, bc) * H * 4;
  static int attr_smem[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FT_ERR_CUDA;
  if (attr_smem[dev] < (int)smem) {
    if (cudaFuncSetAttribute(ft::lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return FT_ERR_CUDA;
    attr_smem[dev] = (int)smem;
  }
  const int sms = ft_host::num_sms();
  for (int c0 = 0; c0 < B; c0 += bc) {
    const int nb = std::min(bc, B - c0);
    ft::lm_head_kernel<<<sms > 0 ? sms : 1, ft::kHeadWarps * 32, (size_t)nb * H * 4, (cudaStream_t)stream>>>(
        x + (size_t)c0 * H, gamma, W, logits + (size_t)c0 * V, nb, V, H, eps);
    if (cudaGetLastError() != cudaSuccess) return FT_ERR_CUDA;
  }
  return FT_OK;
}

}  // extern "C"
