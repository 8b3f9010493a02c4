// Streaming INT4 projection (decode GEMV / skinny GEMM, 1 <= B <= 32 tokens).
//
// y[t, o] = sum_g s[o, g] * sum_{i in g} (c[o, i] - 8) * x[t, i]
// with the group scale applied after each 128-input partial sum (summary page,
// "무엇과 다른가"), followed by a role epilogue.  The RMSNorm row factors are
// not applied here: the consumer of each output applies them after the
// accumulation (summary page, "어떻게 동작하나").
//
// GB300 design:
//  * one CTA per SM: one producer warp streams the CTA's contiguous run of
//    (row tile, group) slabs with 1-D bulk async copies (cp.async.bulk, mbarrier
//    completion; one copy per row tile, issued from parallel lanes) into a ring
//    of stages sized at launch, next to the matching chunk of the FP16
//    activation operand (one copy: the grouped layout keeps a stage's B rows
//    contiguous) and its group offsets.  Weights do not depend on earlier
//    kernels, so the ring fills BEFORE the producer waits on its predecessor
//    (programmatic dependent launch).
//  * NCW consumer warps split each stage's groups; each keeps RT row tiles x
//    NT eight-token column tiles in registers.  Nibbles become FP16 A fragments
//    with four logic ops and a shift per 8 weights (magic_word: the 1024-offset
//    mantissa trick) and run through mma.m16n8k16 with FP32 accumulation; the
//    offset is removed by starting each group's chain at -S (see ft_internal).
//  * warps reduce through shared memory at the end of a row-tile set.  QKV and
//    O split sets along K across CTAs; each CTA's piece of a set stores its
//    partial sums in its own slab and the next kernel adds the slabs in a fixed
//    order (no floating-point atomics: results do not depend on which CTA
//    finished first).  Gate/up CTAs own whole row-tile sets (SwiGLU in the
//    epilogue); down owns whole sets where that balances (block output written
//    directly) and otherwise splits them, the last piece of each set adding the
//    slabs to h1 and writing the output (completion ticket, never waits).
//  * batches of 17-32 run on the tensor-core kernel (tcgen05, ft_umma.cu)
//    instead; this kernel serves 1-16 tokens (one or two column tiles).
//  * E4M3 decode weights (summary page, "전제와 한계") take the same path with
//    2080-byte slabs: two codes at a time convert exactly to an FP16 pair, and
//    there is no decode offset to remove.
#include <algorithm>

#include "ft_block.cuh"

namespace ft {

// RT row tiles per set share every activation fragment (RT x NT independent
// MMA chains per warp); NCW consumer warps split a stage's groups.
template <int NT>
struct GemvShape;
template <> struct GemvShape<1> { static constexpr int RT = 4, NCW = 8; };
template <> struct GemvShape<2> { static constexpr int RT = 4, NCW = 8; };
// The down projection uses sets of two row tiles: fine enough that whole sets
// (no split-K, output written directly with the residual added) balance over
// the SMs for the 8B-class shapes; where whole sets would leave CTAs too
// unequal (long K, many sets), it splits sets along K like QKV and O.
constexpr int kDownRT = 2;
template <int NT, int ROLE>
constexpr int gemv_rt() { return ROLE == kRoleDown ? kDownRT : GemvShape<NT>::RT; }

// Epilogue of one (row tile, column tile) of fully reduced values.
// v[0] = (row g, token t0), v[1] = (row g, t0+1), v[2] = (row g+8, t0), v[3] = (row g+8, t0+1).
// rho2_lane: lane t holds the RMSNorm row factor of token t (gate/up only).
// direct: the piece is a whole set (down: write the block output);
// piece: otherwise, this CTA's piece index within the set (its slab).
template <int ROLE>
__device__ __forceinline__ bool gemv_epi(const GemvParams& p, int T, int j, const float (&v)[4], bool direct,
                                         float rho2_lane, int piece) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int N = p.plan.N;
  const int r0 = T * kRowTile + g, r1 = r0 + 8;
  bool bad = false;
  if constexpr (ROLE == kRoleGU) {
    const int kcol = 8 * T + g;  // a column produced by packed rows g (gate) and g + 8 (up)
    const int grp = kcol / kWGroup;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 8 * j + 2 * tig + e;
      float st = 0.0f;
      const float rho2 = __shfl_sync(0xffffffffu, rho2_lane, t & 31);
      if (t < p.B) {
        const float gv = rho2 * v[e], uv = rho2 * v[2 + e];
        const float a = gv / (1.0f + expf(-gv)) * uv;
        bad |= !(fabsf(a) <= 65504.0f);
        p.out_h[op_index(t, kcol, p.B)] = op_encode(a, kcol, st);
      }
      st += __shfl_xor_sync(0xffffffffu, st, 4);
      st += __shfl_xor_sync(0xffffffffu, st, 8);
      st += __shfl_xor_sync(0xffffffffu, st, 16);
      // the 16 row tiles of a group add exact integers: any order gives the same S
      if (g == 0 && t < p.B) sfix_atomic_add(p.s_out + grp * 32 + t, f32_to_sfix(st));
    }
    return bad;
  } else {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 8 * j + 2 * tig + (r & 1);
      if (t >= p.B) continue;
      const int row = (r & 2) ? r1 : r0;
      if (ROLE == kRoleDown && direct) {
        const float y = __ldcg(p.resid + (size_t)t * N + row) + v[r];
        if (p.out_dtype == FT_F32)
          static_cast<float*>(p.out_final)[(size_t)t * N + row] = y;
        else
          static_cast<uint16_t*>(p.out_final)[(size_t)t * N + row] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
      } else {
        __stcg(p.part + ((size_t)piece * p.B + t) * N + row, v[r]);
      }
    }
    return bad;
  }
}

// Programmatic dependent launch.  Every kernel of the block waits for its
// predecessor before it exits, so a kernel's completion implies that of the
// whole chain before it.  Most kernels let their successor launch at entry, so
// its weight stream starts early.  The QKV projection lets the attention kernel
// launch only after its own wait (every warp triggers after waiting): the prep kernel of
// this call has then completed, hence the previous call on the stream too, and
// the attention kernel's history loads issued before its own wait can never
// overlap a previous call that wrote the same cache.
//
// Producer warp: streams the CTA's (row-tile set, group) units stage by stage
// into the ring, with the matching activation chunk and group offsets.  The
// first `stages` stages of weights are issued before waiting on the previous
// kernel (weights do not depend on it); their activation chunks right after.
template <int RT>
__device__ __forceinline__ void gemv_produce(const GemvParams& p, uint8_t* slots, uint32_t full0, uint32_t empty0,
                                             int u0, int u1, bool trigger_after_wait) {
  const GemvPlan& pl = p.plan;
  const int lane = threadIdx.x & 31;
  const int S = pl.stages;
  auto issue_x = [&](int slot, int kg, int ng) {
    uint8_t* sb = slots + slot * pl.slot;
    // the B rows of groups kg .. kg + ng - 1 are contiguous in the grouped layout
    if (lane == 0)
      bulk_g2s(smem_u32(sb + pl.xoff), p.x + (size_t)kg * p.B * kWGroup, p.B * ng * kWGroup * 2, full0 + 8 * slot);
    if (lane == 31) bulk_g2s(smem_u32(sb + pl.soff), p.s_in + (size_t)kg * 32, ng * 256, full0 + 8 * slot);
  };
  bool waited = false;
  int s = 0, slot = 0, round = 0;
  for (StageWalk st(pl, u0, u1); st.valid(); st.next(), ++s) {
    if (round > 0 && !mbar_wait(empty0 + 8 * slot, (round - 1) & 1)) {
      set_status(p.status, FT_DEV_TIMEOUT);
      break;
    }
    const int nrt = min(RT, pl.NTILE - st.set * RT);
    if (lane == 0)
      mbar_arrive_expect_tx(full0 + 8 * slot,
                            (uint32_t)(nrt * st.ng * pl.slab + p.B * st.ng * kWGroup * 2 + st.ng * 256));
    __syncwarp();
    // one bulk copy per row tile, issued by lane rt (a single thread issuing them
    // one after another limits the stage rate for wide sets)
    const uint32_t sb = smem_u32(slots + slot * pl.slot);
    for (int rt = lane; rt < nrt; rt += 32)
      bulk_g2s(sb + rt * pl.ng * pl.slab, p.w + ((size_t)(st.set * RT + rt) * pl.NKG + st.kg) * pl.slab,
               st.ng * pl.slab, full0 + 8 * slot);
    __syncwarp();
    if (waited) issue_x(slot, st.kg, st.ng);
    if (!waited && (s == S - 1 || st.u + st.ng >= u1)) {
      griddep_wait();  // the activation operand comes from the previous kernel
      if (trigger_after_wait) griddep_launch();
      waited = true;
      int ss = 0;
      for (StageWalk s2(pl, u0, u1); ss <= s; s2.next(), ++ss) issue_x(ss, s2.kg, s2.ng);
    }
    if (++slot == S) {
      slot = 0;
      ++round;
    }
  }
  if (!waited) {
    griddep_wait();
    if (trigger_after_wait) griddep_launch();
  }
}

// FMT: FT_WFMT_INT4 (nibbles, FP16 magic-number decode, each group's chain started at
// -S) or FT_WFMT_E4M3 (bytes converted exactly to FP16, chains start at 0).
template <int NT, int ROLE, int FMT>
__global__ void __launch_bounds__((GemvShape<NT>::NCW + 2) * 32, 1) gemv_kernel(const GemvParams p) {
  constexpr bool E4 = FMT == FT_WFMT_E4M3;
  constexpr int kSlab = E4 ? kSlabBytesE4 : kSlabBytes, kCodes = E4 ? kSlabCodesE4 : kSlabCodes;
  constexpr int RT = gemv_rt<NT, ROLE>(), NCW = GemvShape<NT>::NCW;
  constexpr int PRODUCER = NCW, EPILOGUE = NCW + 1;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GemvPlan& pl = p.plan;
  const int cta = blockIdx.x;
  const int u0 = plan_u0(pl, cta), u1 = plan_u0(pl, cta + 1);
  const int S = pl.stages;
  // barriers: full[S], empty[S], red_full, red_empty
  const uint32_t full0 = smem_u32(smem), empty0 = full0 + 8 * S;
  const uint32_t red_full = empty0 + 8 * S, red_empty = red_full + 8;
  float* red = reinterpret_cast<float*>(smem + pl.redoff);
  uint8_t* zero_row = smem + pl.zerooff;  // stands in for activation rows of absent tokens
  uint8_t* slots = smem + pl.slotoff;

  if (ROLE != kRoleQKV) griddep_launch();  // QKV: every warp after its own wait (see the note on programmatic dependent launch)
  for (int i = tid; i < pl.ng * kWGroup * 2 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(zero_row)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, NCW);
    }
    mbar_init(red_full, NCW);
    mbar_init(red_empty, 1);
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == PRODUCER) {
    gemv_produce<RT>(p, slots, full0, empty0, u0, u1, ROLE == kRoleQKV);
    return;
  }

  if (warp == EPILOGUE) {
    // ------------------------------------------------------------ epilogue
    // Reduces each finished piece over the consumer warps and applies the role
    // epilogue while the consumers already stream the next piece.
    griddep_wait();
    if (ROLE == kRoleQKV) griddep_launch();
    // loaded once: a dependent global load per epilogue call would sit on the
    // critical path of every piece
    float rho2_lane = 0.0f;
    if (ROLE == kRoleGU && lane < p.B) {
      float t = 0.0f;
      for (int k = 0; k < p.nssq; ++k) t += __ldcg(p.ssq2 + lane * p.nssq + k);
      rho2_lane = rsqrtf(t * p.inv_h + p.eps);
    }
    bool bad = false;
    int k = 0, piece_kg0 = -1;
    for (StageWalk st(pl, u0, u1); st.valid(); st.next()) {
      if (piece_kg0 < 0) piece_kg0 = st.kg;
      if (!st.piece_end()) continue;
      const bool whole = (piece_kg0 == 0) && (st.kg + st.ng == pl.NKG);
      piece_kg0 = -1;
      const int piece = cta - plan_first(pl, st.set);  // split sets: this piece's slab
      const int nrt = min(RT, pl.NTILE - st.set * RT);
      if (!mbar_wait(red_full, k & 1)) {
        set_status(p.status, FT_DEV_TIMEOUT);
        return;
      }
      for (int q = 0; q < RT * NT; ++q) {
        const int rt = q / NT, j = q % NT;
        if (rt >= nrt) continue;
        float v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float a = 0.0f;
#pragma unroll
          for (int w = 0; w < NCW; ++w) a += red[((w * RT * NT + q) * 4 + r) * 32 + lane];
          v[r] = a;
        }
        bad |= gemv_epi<ROLE>(p, st.set * RT + rt, j, v, whole, rho2_lane, piece);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_empty);
      if (ROLE == kRoleDown && !whole) {
        // split set: the last of its pieces writes the block output from h1
        // and the pieces' slabs (completion ticket, never waits)
        __threadfence();
        __syncwarp();
        const int np = plan_pieces(pl, st.set);
        uint32_t last = 0;
        if (lane == 0) last = (atomicAdd(p.tick + st.set, 1u) == (uint32_t)(np - 1)) ? 1u : 0u;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          down_finish_set(p, st.set, nrt * kRowTile, st.set * RT * kRowTile, lane, 32);
          if (lane == 0) p.tick[st.set] = 0u;
        }
      }
      ++k;
    }
    if (bad) set_status(p.status, FT_DEV_RANGE);
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  if (ROLE == kRoleQKV) griddep_launch();
  const int g = lane >> 2, tig = lane & 3;
  float tot[RT][NT][4];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int r = 0; r < 4; ++r) tot[a][b][r] = 0.0f;

  // Every projection has a multiple of 64 output rows (hidden, inter, n_q d and
  // (n_q + 2 n_kv) d are multiples of 128), so every set has RT full tiles.
  int slot = 0, fphase = 0, k = 0;
  for (StageWalk st(pl, u0, u1); st.valid(); st.next()) {
    if (!mbar_wait(full0 + 8 * slot, fphase)) {
      set_status(p.status, FT_DEV_TIMEOUT);
      return;
    }
    const uint8_t* sw = slots + slot * pl.slot;
    const sfix_t* ss = reinterpret_cast<const sfix_t*>(sw + pl.soff);
    for (int kgl = warp; kgl < st.ng; kgl += NCW) {
      // activation rows of this lane's B fragments (tokens >= B read zeros) and
      // the group offsets -S for the lane's two token columns
      const uint8_t* xr[NT];  // row of half 0; half 1 is xh bytes further
      int xh[NT];
      float c0[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int row = 8 * j + g, t = 8 * j + 2 * tig;
        // row `row` of group kgl in the stage's half-group rows; absent tokens read zeros
        const bool on = row < p.B;
        xr[j] = on ? sw + pl.xoff + (2 * kgl * p.B + row) * 128 : zero_row + kgl * (kWGroup * 2);
        xh[j] = on ? p.B * 128 : 128;
        const longlong2 sv = *reinterpret_cast<const longlong2*>(ss + kgl * 32 + t);
        c0[j][0] = (!E4 && t < p.B) ? -sfix_to_f32(sv.x) : 0.0f;
        c0[j][1] = (!E4 && t + 1 < p.B) ? -sfix_to_f32(sv.y) : 0.0f;
      }
      const uint8_t* slab0 = sw + kgl * kSlab;
      // k-steps 0-3 and 4-7 of the group run as two independent MMA chains
      // (the second starts at 0) where registers allow, halving the chain depth
      constexpr bool kTwoChains = NT <= 2;
      uint32_t sc[RT];
      float acc[RT][NT][4];
      float acc2[kTwoChains ? RT : 1][kTwoChains ? NT : 1][4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t wd[RT][E4 ? 8 : 4];  // INT4: one word per k-step; E4M3: two
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
          const uint8_t* slab = slab0 + rt * pl.ng * kSlab;
          if constexpr (E4) {
            const uint4* q = reinterpret_cast<const uint4*>(slab + half * 1024 + lane * 32);
            const uint4 qa = q[0], qb = q[1];
            wd[rt][0] = qa.x; wd[rt][1] = qa.y; wd[rt][2] = qa.z; wd[rt][3] = qa.w;
            wd[rt][4] = qb.x; wd[rt][5] = qb.y; wd[rt][6] = qb.z; wd[rt][7] = qb.w;
          } else {
            const uint4 q = *reinterpret_cast<const uint4*>(slab + half * 512 + lane * 16);
            wd[rt][0] = q.x; wd[rt][1] = q.y; wd[rt][2] = q.z; wd[rt][3] = q.w;
          }
          if (half == 0) sc[rt] = *reinterpret_cast<const uint32_t*>(slab + kCodes + 4 * g);
        }
#pragma unroll
        for (int kq = 0; kq < 4; ++kq) {
          const int ks = 4 * half + kq;
          uint32_t b0[NT], b1[NT];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            const uint2 bv = *reinterpret_cast<const uint2*>(xr[j] + half * xh[j] + op_frag_off(kq, tig, g));
            b0[j] = bv.x;
            b1[j] = bv.y;
          }
#pragma unroll
          for (int rt = 0; rt < RT; ++rt) {
            uint32_t r[4];
            if constexpr (E4)
              e4m3_words(wd[rt][2 * kq], wd[rt][2 * kq + 1], r);
            else
              magic_word(wd[rt][kq], r);
            const uint32_t a[4] = {r[0], r[2], r[1], r[3]};
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              if (ks == 0) {
                float* d = acc[rt][j];
                d[0] = c0[j][0]; d[1] = c0[j][1]; d[2] = c0[j][0]; d[3] = c0[j][1];
              }
              if (kTwoChains && half == 1) {
                float (&d2)[4] = acc2[kTwoChains ? rt : 0][kTwoChains ? j : 0];
                if (kq == 0)
                  mma_f16_zc(d2, a, b0[j], b1[j]);
                else
                  mma_f16(d2, a, b0[j], b1[j]);
              } else {
                mma_f16(acc[rt][j], a, b0[j], b1[j]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int rt = 0; rt < RT; ++rt) {
        const float slo = bf16_bits_to_f32((uint16_t)(sc[rt] & 0xFFFFu));
        const float shi = bf16_bits_to_f32((uint16_t)(sc[rt] >> 16));
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = kTwoChains ? acc[rt][j][r] + acc2[kTwoChains ? rt : 0][kTwoChains ? j : 0][r]
                                       : acc[rt][j][r];
            tot[rt][j][r] = fmaf((r & 2) ? shi : slo, a, tot[rt][j][r]);
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    if (++slot == S) {
      slot = 0;
      fphase ^= 1;
    }

    if (st.piece_end()) {
      // ---- end of this CTA's piece of a set: hand the partial sums to the epilogue warp
      if (k > 0 && !mbar_wait(red_empty, (k - 1) & 1)) {
        set_status(p.status, FT_DEV_TIMEOUT);
        return;
      }
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            red[(((warp * RT + rt) * NT + j) * 4 + r) * 32 + lane] = tot[rt][j][r];
            tot[rt][j][r] = 0.0f;
          }
      __syncwarp();
      if (lane == 0) mbar_arrive(red_full);
      ++k;
    }
  }
}

template <int NT, int ROLE, int FMT>
static cudaError_t launch_one(const GemvParams& p, cudaStream_t st, bool pdl) {
  constexpr int THREADS = (GemvShape<NT>::NCW + 2) * 32;
  static int attr_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_smem[dev] < p.plan.smem) {
    cudaError_t e =
        cudaFuncSetAttribute(gemv_kernel<NT, ROLE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.plan.smem);
    if (e != cudaSuccess) return e;
    attr_smem[dev] = p.plan.smem;
  }
  return launch_ex(gemv_kernel<NT, ROLE, FMT>, dim3(p.plan.C), dim3(THREADS), (size_t)p.plan.smem, st, pdl, p);
}

template <int ROLE, int FMT>
static cudaError_t launch_role_fmt(const GemvParams& p, cudaStream_t st, bool pdl) {
  switch (p.plan.NT) {
    case 1: return launch_one<1, ROLE, FMT>(p, st, pdl);
    case 2: return launch_one<2, ROLE, FMT>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

template <int ROLE>
static cudaError_t launch_role(const GemvParams& p, cudaStream_t st, bool pdl) {
  if (p.plan.slab == kSlabBytesE4) return launch_role_fmt<ROLE, FT_WFMT_E4M3>(p, st, pdl);
  if (p.plan.slab == kSlabBytes) return launch_role_fmt<ROLE, FT_WFMT_INT4>(p, st, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(int role, const GemvParams& p, cudaStream_t st, bool pdl) {
  if (p.plan.umma) return launch_umma(role, p, st, pdl);
  switch (role) {
    case kRoleQKV: return launch_role<kRoleQKV>(p, st, pdl);
    case kRoleO: return launch_role<kRoleO>(p, st, pdl);
    case kRoleGU: return launch_role<kRoleGU>(p, st, pdl);
    case kRoleDown: return launch_role<kRoleDown>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

static void shape_of(int NT, int& RT, int& NCW) {
  switch (NT) {
    case 1: RT = GemvShape<1>::RT; NCW = GemvShape<1>::NCW; break;
    case 2: RT = GemvShape<2>::RT; NCW = GemvShape<2>::NCW; break;
    default: RT = GemvShape<2>::RT; NCW = GemvShape<2>::NCW; break;
  }
}

GemvPlan make_gemv_plan(int role, int N, int K, int B, int sms, int smem_budget, int weight_format) {
  GemvPlan p = {};
  p.slab = slab_bytes_of(weight_format);
  p.N = N;
  p.K = K;
  p.NT = (B + 7) / 8;
  shape_of(p.NT, p.RT, p.NCW);
  if (role == kRoleDown) p.RT = kDownRT;
  p.NTILE = N / kRowTile;
  p.NKG = K / kWGroup;
  p.NSET = (p.NTILE + p.RT - 1) / p.RT;
  bool whole_sets = role == kRoleGU;
  if (role == kRoleDown) {
    // whole sets unless the busiest CTA would stream > 64 KB more weights than
    // the average CTA of the split partition (the split costs a completion
    // ticket round trip at the end of each split set)
    const long units = (long)p.NSET * p.NKG;
    const long c_split = std::min<long>(sms, units), c_whole = std::min<long>(sms, p.NSET);
    const double avg = (double)units / (double)c_split;
    const long max_whole = (p.NSET + c_whole - 1) / c_whole * (long)p.NKG;
    whole_sets = ((double)max_whole - avg) * p.RT * p.slab <= 64.0 * 1024.0;
  }
  p.whole = whole_sets ? 1 : 0;
  const int units = whole_sets ? p.NSET : p.NSET * p.NKG;
  p.C = sms < units ? sms : units;
  if (p.C < 1) p.C = 1;
  p.per = units / p.C;
  p.rem = units % p.C;
  p.rcp_per1 = ((1ull << 32) + (unsigned long long)p.per) / (unsigned long long)(p.per + 1);  // ceil
  p.rcp_per = ((1ull << 32) + (unsigned long long)p.per - 1) / (unsigned long long)p.per;     // ceil
  p.divs_exact = (unsigned long long)units * (unsigned long long)(p.per + 1) <= (1ull << 32) ? 1 : 0;
  p.npmax = 1;
  if (!whole_sets)
    for (int set = 0; set < p.NSET; ++set) p.npmax = std::max(p.npmax, plan_pieces(p, set));
  p.ng = p.NCW * 4 / p.RT;  // stages of 4 row tiles x NCW groups (a group per warp for RT = 4)
  if (p.ng > p.NKG) p.ng = p.NKG;
  // (E4M3 slabs are twice as large: where two such stages would not fit, stages carry fewer
  // groups, and some consumer warps sit out a stage)
  for (;;) {
    p.xstride = p.ng * kWGroup * 2;  // bytes of one token row of a stage (grouped rows, no padding)
    const int wbytes = p.RT * p.ng * p.slab;
    p.xoff = (int)align_up((size_t)wbytes, 16);
    p.soff = (int)align_up((size_t)p.xoff + (size_t)B * p.xstride, 16);
    p.slot = (int)align_up((size_t)p.soff + (size_t)p.ng * 256, 128);
    p.redoff = 256;
    const int redbytes = p.NCW * p.RT * p.NT * 128 * 4;
    p.zerooff = (int)align_up((size_t)p.redoff + (size_t)redbytes, 128);
    p.slotoff = (int)align_up((size_t)p.zerooff + (size_t)p.ng * kWGroup * 2, 128);
    if (p.ng == 1 || p.slotoff + 2 * p.slot <= smem_budget) break;
    p.ng = (p.ng + 1) / 2;
  }
  int stages = (smem_budget - p.slotoff) / p.slot;
  if (stages > 8) stages = 8;
  if (stages < 2) stages = 2;
  p.stages = stages;
  p.smem = p.slotoff + stages * p.slot;
  return p;
}

}  // namespace ft
