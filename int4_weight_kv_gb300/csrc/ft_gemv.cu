// Streaming INT4 projection (decode GEMV / skinny GEMM, 1 <= B <= 32 tokens).
//
// y[t, o] = sum_g s[o, g] * sum_{i in g} (c[o, i] - 8) * x[t, i]
// with the group scale applied after each 128-input partial sum (summary page,
// "무엇과 다른가"), followed by a role-specific epilogue: the RMSNorm row
// factor (QKV, "어떻게 동작하나": rho applied after accumulation), the residual
// (O, down) or SwiGLU (gate/up).
//
// GB300 design:
//  * one CTA per SM, 9 warps: warp 8 is a producer that streams the CTA's
//    contiguous run of packed weight slabs with 1-D bulk async copies
//    (cp.async.bulk, mbarrier completion) into a ring of STAGES slots, and
//    copies the matching 128-input chunks of the FP16 activation rows next to
//    them.  Weights do not depend on earlier kernels, so the producer fills the
//    whole ring BEFORE waiting on the previous kernel (programmatic dependent
//    launch): the weight stream overlaps the previous kernel's tail.
//  * warps 0-7 consume: each owns one 16-row tile of every 128-row block in the
//    macro block, dequantises nibbles in registers into FP16 tensor-core A
//    fragments (exact: (c-8) is representable) and runs mma.m16n8k16 with FP32
//    accumulation; activation B fragments are read from shared memory once per
//    k-step and reused across the RB row tiles.  Tensor cores here reduce the
//    per-weight instruction count (one MMA replaces 256 FMAs); the kernel is
//    bound by HBM bandwidth.
//  * split-K across CTAs with deterministic reduction: partial sums go to
//    per-piece slots and the last piece (atomic ticket, no waiting) adds them
//    in piece order.
#include "ft_block.cuh"

namespace ft {

template <int NT>
struct GemvCfg {
  static constexpr int RB = NT;
  static constexpr int NGS = (RB == 1) ? 2 : 1;                // groups per stage
  static constexpr int STAGES = (RB <= 2) ? 5 : 4;
  static constexpr int WBYTES = RB * NGS * kBlockGroupBytes;     // weight bytes per slot
  static constexpr int XROW = NGS * kWGroup + 8;                 // halfs per activation row
  static constexpr int XBYTES = 8 * NT * XROW * 2;
  static constexpr int SLOT = WBYTES + XBYTES;
  static constexpr int SMEM = 128 + SLOT * STAGES;
  static constexpr int THREADS = 288;
};

struct ConsumerSync {
  uint32_t bar;
  uint32_t phase;
  // bounded barrier of the 8 consumer warps (an mbarrier with count 8)
  __device__ __forceinline__ bool sync() {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase);
    phase ^= 1;
    __syncwarp();
    return ok;
  }
};

template <int NT, int ROLE>
__device__ __forceinline__ void gemv_epilogue(const GemvParams& p, int mb, int nrb, float (&tot)[NT][NT][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int N = p.plan.N;
  bool range_bad = false;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    float sq[2] = {0.0f, 0.0f};
#pragma unroll
    for (int rb = 0; rb < NT; ++rb) {
      if (rb >= nrb) continue;
      const int rbg = mb * NT + rb;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = r & 1;
        const int t = 8 * j + 2 * tig + e;
        if (t >= p.B) continue;
        const float val = tot[rb][j][r];
        const int row = rbg * kRowBlock + warp * kRowTile + g + ((r & 2) ? 8 : 0);
        if (ROLE == kRoleQKV) {
          p.out_f32[(size_t)t * N + row] = p.rho[t] * val;
        } else if (ROLE == kRoleO) {
          const float xin = (p.resid_dtype == FT_F32)
                                ? ld_cg_f32(static_cast<const float*>(p.resid) + (size_t)t * N + row)
                                : bf16_bits_to_f32(static_cast<const uint16_t*>(p.resid)[(size_t)t * N + row]);
          const float h1 = xin + val;
          p.out_f32[(size_t)t * N + row] = h1;
          p.out_h[(size_t)t * N + row] = __float2half_rn(h1);
          range_bad |= !(fabsf(h1) <= 65504.0f);
          sq[e] += h1 * h1;
        } else if (ROLE == kRoleDown) {
          const float y = ld_cg_f32(static_cast<const float*>(p.resid) + (size_t)t * N + row) + val;
          if (p.out_dtype == FT_F32)
            static_cast<float*>(p.out_final)[(size_t)t * N + row] = y;
          else
            static_cast<uint16_t*>(p.out_final)[(size_t)t * N + row] =
                __bfloat16_as_ushort(__float2bfloat16_rn(y));
        }
      }
      if (ROLE == kRoleGU) {
        // rows g (gate) and g + 8 (up) of global tile T hold a-column 8 T + g
        const int T = rbg * kTilesPerBlock + warp;
        const int inter = N / 2;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * j + 2 * tig + e;
          if (t >= p.B) continue;
          const float rho2 = rsqrtf(ld_cg_f32(p.sumsq + t) / (float)p.H + p.eps);
          const float gv = rho2 * tot[rb][j][e];
          const float uv = rho2 * tot[rb][j][2 + e];
          const float a = gv / (1.0f + expf(-gv)) * uv;
          range_bad |= !(fabsf(a) <= 65504.0f);
          p.out_h[(size_t)t * inter + 8 * T + g] = __float2half_rn(a);
        }
      }
    }
    if (ROLE == kRoleO) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = sq[e];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        const int t = 8 * j + 2 * tig + e;
        if (g == 0 && t < p.B) atomicAdd(p.sumsq + t, v);
      }
    }
  }
  if (range_bad) set_status(p.status, FT_DEV_RANGE);
}

template <int NT, int ROLE>
__global__ void __launch_bounds__(288, 1) gemv_kernel(const GemvParams p) {
  using C = GemvCfg<NT>;
  constexpr int RB = C::RB;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GemvPlan& pl = p.plan;
  const int cta = blockIdx.x;
  const int u0 = plan_u0(pl, cta), u1 = plan_u0(pl, cta + 1);
  const uint32_t full0 = smem_u32(smem), empty0 = full0 + 8 * C::STAGES, sync_bar = empty0 + 8 * C::STAGES;
  uint8_t* slots = smem + 128;
  volatile uint32_t* flag = reinterpret_cast<volatile uint32_t*>(smem + 8 * (2 * C::STAGES + 1));

  griddep_launch();
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 8);
    }
    mbar_init(sync_bar, 8);
    mbar_fence_init();
  }
  // activation rows of tokens >= B are never copied: keep them zero
  {
    const int padrows = 8 * NT - p.B;
    const int words = padrows * (C::XROW / 2);
    for (int i = tid; i < C::STAGES * words; i += C::THREADS) {
      const int s = i / words, k = i % words;
      uint32_t* xs = reinterpret_cast<uint32_t*>(slots + s * C::SLOT + C::WBYTES);
      xs[p.B * (C::XROW / 2) + k] = 0u;
    }
  }
  __syncthreads();

  if (warp == 8) {
    // ---------------- producer
    auto issue_x = [&](int slot, int kg, int ng) {
      if (lane < p.B) {
        const uint32_t dst = smem_u32(slots + slot * C::SLOT + C::WBYTES) + lane * C::XROW * 2;
        bulk_g2s(dst, p.x + (size_t)lane * pl.K + (size_t)kg * kWGroup, ng * kWGroup * 2, full0 + 8 * slot);
      }
    };
    bool waited = false;
    int s = 0;
    for (int u = u0; u < u1; ++s) {
      const int mb = u / pl.NKG, kg = u - mb * pl.NKG;
      const int ng = min(min(C::NGS, pl.NKG - kg), u1 - u);
      const int slot = s % C::STAGES;
      if (s >= C::STAGES && !mbar_wait(empty0 + 8 * slot, ((s / C::STAGES) - 1) & 1)) {
        set_status(p.status, FT_DEV_TIMEOUT);
        break;
      }
      const int nrb = min(RB, pl.NRB - mb * RB);
      const uint32_t sb = smem_u32(slots + slot * C::SLOT);
      if (lane == 0) {
        mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)(nrb * ng * kBlockGroupBytes + p.B * ng * kWGroup * 2));
        for (int rb = 0; rb < nrb; ++rb)
          bulk_g2s(sb + rb * ng * kBlockGroupBytes,
                   p.w + ((size_t)(mb * RB + rb) * pl.NKG + kg) * kBlockGroupBytes, ng * kBlockGroupBytes,
                   full0 + 8 * slot);
      }
      __syncwarp();
      if (waited) issue_x(slot, kg, ng);
      u += ng;
      if (!waited && (s == C::STAGES - 1 || u >= u1)) {
        // the ring is full of weights: now wait for the activations' producer
        griddep_wait();
        waited = true;
        int uu = u0;
        for (int ss = 0; ss <= s; ++ss) {
          const int mb2 = uu / pl.NKG, kg2 = uu - mb2 * pl.NKG;
          const int ng2 = min(min(C::NGS, pl.NKG - kg2), u1 - uu);
          issue_x(ss, kg2, ng2);
          uu += ng2;
        }
      }
    }
    if (!waited) griddep_wait();
    return;
  }

  // ---------------- consumers (warps 0..7)
  griddep_wait();
  ConsumerSync cs{sync_bar, 0};
  const int g = lane >> 2, tig = lane & 3;
  float tot[RB][NT][4];
#pragma unroll
  for (int a = 0; a < RB; ++a)
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int r = 0; r < 4; ++r) tot[a][b][r] = 0.0f;

  int s = 0, piece_kg0 = -1;
  for (int u = u0; u < u1; ++s) {
    const int mb = u / pl.NKG, kg = u - mb * pl.NKG;
    const int ng = min(min(C::NGS, pl.NKG - kg), u1 - u);
    if (piece_kg0 < 0) piece_kg0 = kg;
    const int slot = s % C::STAGES;
    if (!mbar_wait(full0 + 8 * slot, (s / C::STAGES) & 1)) {
      set_status(p.status, FT_DEV_TIMEOUT);
      return;
    }
    const int nrb = min(RB, pl.NRB - mb * RB);
    const uint8_t* sw = slots + slot * C::SLOT;
    const uint8_t* sx = sw + C::WBYTES;
    for (int kgl = 0; kgl < ng; ++kgl) {
      float acc[RB][NT][4];
      uint32_t sc[RB];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // nibble words of k-steps 4 half .. 4 half + 3 for each row tile
        uint32_t wd[RB][4];
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          if (rb < nrb) {
            const uint8_t* slab = sw + ((rb * ng + kgl) * kTilesPerBlock + warp) * kSlabBytes;
            const uint4 q = *reinterpret_cast<const uint4*>(slab + half * 512 + lane * 16);
            wd[rb][0] = q.x; wd[rb][1] = q.y; wd[rb][2] = q.z; wd[rb][3] = q.w;
            if (half == 0) sc[rb] = *reinterpret_cast<const uint32_t*>(slab + kSlabCodes + 4 * g);
          } else {
            wd[rb][0] = wd[rb][1] = wd[rb][2] = wd[rb][3] = 0x88888888u;
            if (half == 0) sc[rb] = 0u;
          }
        }
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int ks = 4 * half + kq;
          uint32_t b0[NT], b1[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint8_t* xr = sx + ((8 * j + g) * C::XROW + kgl * kWGroup + ks * 16 + 2 * tig) * 2;
            b0[j] = *reinterpret_cast<const uint32_t*>(xr);
            b1[j] = *reinterpret_cast<const uint32_t*>(xr + 16);
          }
#pragma unroll
          for (int rb = 0; rb < RB; ++rb) {
            if (rb < nrb) {
              uint32_t a[4];
              dequant_word(wd[rb][kq], a);
#pragma unroll
              for (int j = 0; j < NT; ++j) {
                if (ks == 0)
                  mma_f16_zc(acc[rb][j], a, b0[j], b1[j]);
                else
                  mma_f16(acc[rb][j], a, b0[j], b1[j]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        if (rb < nrb) {
          const float slo = bf16_bits_to_f32((uint16_t)(sc[rb] & 0xFFFFu));
          const float shi = bf16_bits_to_f32((uint16_t)(sc[rb] >> 16));
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            tot[rb][j][0] = fmaf(slo, acc[rb][j][0], tot[rb][j][0]);
            tot[rb][j][1] = fmaf(slo, acc[rb][j][1], tot[rb][j][1]);
            tot[rb][j][2] = fmaf(shi, acc[rb][j][2], tot[rb][j][2]);
            tot[rb][j][3] = fmaf(shi, acc[rb][j][3], tot[rb][j][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    u += ng;

    if (u >= u1 || u % pl.NKG == 0) {
      // ---- end of a piece of macro block mb
      const bool full = (piece_kg0 == 0) && (u == (mb + 1) * pl.NKG);
      piece_kg0 = -1;
      if (!full) {
        const int first = plan_owner(pl, mb * pl.NKG);
        const int np = plan_owner(pl, mb * pl.NKG + pl.NKG - 1) - first + 1;
        const int pidx = cta - first;
        float* base = p.slots + ((size_t)mb * pl.maxp) * pl.slotf;
        float* mine = base + (size_t)pidx * pl.slotf;
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r)
              __stcg(mine + (((warp * RB + rb) * NT + j) * 4 + r) * 32 + lane, tot[rb][j][r]);
        __threadfence();
        if (!cs.sync()) { set_status(p.status, FT_DEV_TIMEOUT); return; }
        if (tid == 0) *flag = (atomicAdd(p.tick + mb, 1u) == (uint32_t)(np - 1)) ? 1u : 0u;
        if (!cs.sync()) { set_status(p.status, FT_DEV_TIMEOUT); return; }
        const bool last = *flag != 0;
        if (last) {
          __threadfence();
#pragma unroll
          for (int rb = 0; rb < RB; ++rb)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
              for (int r = 0; r < 4; ++r) tot[rb][j][r] = 0.0f;
          for (int q = 0; q < np; ++q) {
            const float* src = base + (size_t)q * pl.slotf;
#pragma unroll
            for (int rb = 0; rb < RB; ++rb)
#pragma unroll
              for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int r = 0; r < 4; ++r)
                  tot[rb][j][r] += __ldcg(src + (((warp * RB + rb) * NT + j) * 4 + r) * 32 + lane);
          }
          if (tid == 0) p.tick[mb] = 0u;
          gemv_epilogue<NT, ROLE>(p, mb, nrb, tot);
        }
        // a later piece may reuse the flag word
        if (!cs.sync()) { set_status(p.status, FT_DEV_TIMEOUT); return; }
      } else {
        gemv_epilogue<NT, ROLE>(p, mb, nrb, tot);
      }
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) tot[rb][j][r] = 0.0f;
    }
  }
}

template <int NT, int ROLE>
static cudaError_t launch_one(const GemvParams& p, cudaStream_t st, bool pdl) {
  using C = GemvCfg<NT>;
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NT, ROLE>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  return launch_ex(gemv_kernel<NT, ROLE>, dim3(p.plan.C), dim3(C::THREADS), (size_t)C::SMEM, st, pdl, p);
}

template <int ROLE>
static cudaError_t launch_role(const GemvParams& p, cudaStream_t st, bool pdl) {
  switch (p.plan.NT) {
    case 1: return launch_one<1, ROLE>(p, st, pdl);
    case 2: return launch_one<2, ROLE>(p, st, pdl);
    case 3: return launch_one<3, ROLE>(p, st, pdl);
    case 4: return launch_one<4, ROLE>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemv(int role, const GemvParams& p, cudaStream_t st, bool pdl) {
  switch (role) {
    case kRoleQKV: return launch_role<kRoleQKV>(p, st, pdl);
    case kRoleO: return launch_role<kRoleO>(p, st, pdl);
    case kRoleGU: return launch_role<kRoleGU>(p, st, pdl);
    case kRoleDown: return launch_role<kRoleDown>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

GemvPlan make_gemv_plan(int N, int K, int B, int sms) {
  GemvPlan p;
  p.N = N;
  p.K = K;
  p.NT = (B + 7) / 8;
  p.RB = p.NT;
  p.NRB = N / kRowBlock;
  p.NKG = K / kWGroup;
  p.NMB = (p.NRB + p.RB - 1) / p.RB;
  p.U = p.NMB * p.NKG;
  p.C = sms < p.U ? sms : p.U;
  if (p.C < 1) p.C = 1;
  p.per = p.U / p.C;
  p.rem = p.U % p.C;
  const int mp = (p.NKG + p.per - 1) / p.per + 1;
  p.maxp = mp < p.NKG ? mp : p.NKG;
  p.slotf = 8 * p.RB * p.NT * 128;
  return p;
}

size_t gemv_smem_bytes(int NT) {
  switch (NT) {
    case 1: return GemvCfg<1>::SMEM;
    case 2: return GemvCfg<2>::SMEM;
    case 3: return GemvCfg<3>::SMEM;
    default: return GemvCfg<4>::SMEM;
  }
}

}  // namespace ft
