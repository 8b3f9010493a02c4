// Tensor-core projection for batches of 17-32 tokens (fifth-generation tensor
// cores, tcgen05, sm_103a).
//
// Computes the same y[t, o] = sum_g s[o, g] * sum_{i in g} (c[o, i] - 8) x[t, i]
// as the streaming GEMV (group scale after each 128-input partial sum, summary
// page "무엇과 다른가"), from the same packed weights, activation operand and
// group offsets, with the skinny contraction on the tensor cores:
//  * a CTA per SM owns a contiguous run of (128-row block, 128-input group)
//    units; a producer warp streams each stage's weight slabs (one bulk copy
//    per 16-row tile), activation half-groups (32-row, 128-byte-swizzled tiles
//    of 64 inputs; rows of absent tokens stay zero) and group offsets into a
//    ring of shared-memory stages;
//  * eight decoder warps turn each group's nibbles into FP16 (1024 + c, or
//    1024 + 16 c for the upper 8 inputs of every 16, the activation holding
//    x / 16 there) and store them straight into tensor memory as the A operand:
//    the packed fragment order is the 16x256b tensor-memory layout, with K
//    permuted exactly as the activation operand's storage order;
//  * two threads (groups taken in turn) issue tcgen05.mma kind::f16 (M = 128
//    rows, N = 32 tokens, K = 16), A from tensor memory, B from shared memory
//    through a 128-byte-swizzle descriptor, FP32 accumulation in tensor
//    memory, one accumulator per group (four groups' A tiles and eight
//    accumulators in flight);
//  * four epilogue warps read each group's accumulator (one row per thread),
//    remove the decode offset S of each token and apply the row's group scale
//    in FP32 (scales and offsets stashed by the decoders), and at the end of
//    the CTA's piece of a block write its partial sums to the piece's slab;
//    units are spread evenly over the CTAs, and the next kernel adds the slabs
//    of each row in slab order (attention for QKV, mid for O, the SwiGLU kernel
//    for gate/up, the output kernel for down).
// Every wait is an mbarrier wait bounded by %globaltimer; on a timeout the
// kernel sets FT_DEV_TIMEOUT, stops issuing, waits (bounded) for its own
// tensor-core work and copies, frees its tensor memory and returns.
#include <algorithm>

#include "ft_block.cuh"

namespace ft {

namespace umma {

constexpr int kDecWarps = 8, kEpiWarps = 4;
// Two issuing warps, group gi issued by issuer gi % 2: a thread stalls while its MMAs run, so
// the other's bookkeeping and waits overlap them and the tensor core stays fed.  Warp w runs on
// scheduler w % 4; the roles are placed so that each scheduler carries two decoder warps and
// at most two others (the decoders' pace sets the tensor core's).
constexpr int kIssuers = 2;
constexpr int kMma2 = 0, kMma = 1, kDec0 = 2, kEpi0 = kDec0 + kDecWarps, kProducer = kEpi0 + kEpiWarps;
constexpr int kWarps = kProducer + 1, kThreads = kWarps * 32;
constexpr int kNBuf = 4;         // A tiles in flight (groups)
constexpr int kNAcc = 8;         // accumulators (and stashed scales / offsets) in flight (groups)
static_assert(kNAcc % kIssuers == 0, "each issuer owns the accumulators of its own groups");
constexpr int kTmemCols = 512;  // D: kNAcc x 32 columns, A: kNBuf x 64 columns
constexpr int kAccCol = 0, kACol = 32 * kNAcc;
constexpr int kXTile = 32 * 128;  // one 64-input half group of 32 token rows

// ---- tcgen05 / async-proxy wrappers
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "n"(kTmemCols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kTmemCols));
}
__device__ __forceinline__ void tmem_st16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld32x32b_x32(uint32_t taddr, uint32_t (&d)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7]), "=r"(d[8]),
        "=r"(d[9]), "=r"(d[10]), "=r"(d[11]), "=r"(d[12]), "=r"(d[13]), "=r"(d[14]), "=r"(d[15]), "=r"(d[16]),
        "=r"(d[17]), "=r"(d[18]), "=r"(d[19]), "=r"(d[20]), "=r"(d[21]), "=r"(d[22]), "=r"(d[23]), "=r"(d[24]),
        "=r"(d[25]), "=r"(d[26]), "=r"(d[27]), "=r"(d[28]), "=r"(d[29]), "=r"(d[30]), "=r"(d[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// D (+)= A (tensor memory) * B (shared memory descriptor), kind::f16
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.u32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on the mbarrier once every tcgen05 operation this thread issued before it has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Instruction descriptor: FP32 accumulator, FP16 A and B, both K-major, N and M.
constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Shared-memory descriptor of a K-major, 128-byte-swizzled tile: rows 128 B
// apart inside 8-row 1024-byte atoms, atoms 1024 B apart (stride byte offset).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Shared-memory map (offsets from a 1024-byte aligned base).
struct Smem {
  static constexpr int kBars = 0;          // full[8], empty[8], a_full[8], mma_done[8], acc_empty[8]
  static constexpr int kTmemSlot = 448;    // u32 tensor-memory base
  static constexpr int kScl = 1024;        // float[kNAcc][128] row scales of the groups in flight
  static constexpr int kSof = 5120;        // float[kNAcc][32] token offsets S of the groups in flight
  static constexpr int kSlots = 6144;      // ring of stages
};

}  // namespace umma

using namespace umma;

// FMT: FT_WFMT_INT4 (nibbles decoded by the FP16 magic-number trick, offsets S
// removed per token) or FT_WFMT_E4M3 (bytes converted exactly to FP16, no offset).
template <int ROLE, int FMT>
__global__ void __launch_bounds__(kThreads, 1) umma_kernel(const GemvParams p) {
  constexpr bool E4 = FMT == FT_WFMT_E4M3;
  constexpr int kSlab = E4 ? kSlabBytesE4 : kSlabBytes, kCodes = E4 ? kSlabCodesE4 : kSlabCodes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024 - (raw & 1023)) & 1023);  // 1024-byte aligned (swizzle atoms)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const GemvPlan& pl = p.plan;
  const int cta = blockIdx.x;
  const int u0 = plan_u0(pl, cta), u1 = plan_u0(pl, cta + 1);
  const int S = pl.stages;
  const uint32_t bar0 = smem_u32(sm + Smem::kBars);
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 64 + 8 * s; };
  // per group gi, indexed by a = gi % kNAcc (the A tile by gi % kNBuf): a_full[a]: the decoders
  // filled the A tile and stashed the scales and offsets; mma_done[a]: the tensor core finished the
  // group (A tile free, accumulator a ready); acc_empty[a]: the epilogue read accumulator a and stash a
  const uint32_t a_full = bar0 + 128, mma_done = a_full + 8 * kNAcc, acc_empty = mma_done + 8 * kNAcc;
  uint8_t* slots = sm + Smem::kSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::kTmemSlot);
  float* scl = reinterpret_cast<float*>(sm + Smem::kScl);
  float* sof = reinterpret_cast<float*>(sm + Smem::kSof);

  if (ROLE != kRoleQKV) griddep_launch();  // QKV: after its wait (see the gemv kernel's note)
  // zero the activation rows of absent tokens (t >= B) once: copies never write them
  {
    const int per_tile = (32 - p.B) * 8;  // 16-byte chunks of rows B..31
    for (int i = tid; i < S * 2 * pl.ng * per_tile; i += kThreads) {
      const int tile = i / per_tile, k = i % per_tile;
      uint8_t* t0 = slots + (tile / (2 * pl.ng)) * pl.slot + pl.xoff + (tile % (2 * pl.ng)) * kXTile;
      reinterpret_cast<uint4*>(t0 + p.B * 128)[k] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      // decoders (weights, scales and offsets read) and the tensor core (activations read)
      mbar_init(empty(s), kDecWarps + kIssuers);
    }
    for (int b = 0; b < kNAcc; ++b) {
      mbar_init(a_full + 8 * b, kDecWarps);
      mbar_init(mma_done + 8 * b, 1);
      mbar_init(acc_empty + 8 * b, kEpiWarps);
    }
    mbar_fence_init();
  }
  if (warp == kMma) tmem_alloc(smem_u32(tmem_slot));
  fence_proxy_async();  // the zeroed tiles, before the tensor core reads them
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == kProducer) {
    // ------------------------------------------------------------ producer
    bool waited = false;
    int si = 0;
    auto issue_x = [&](int slot, int kg, int ng) {
      uint8_t* sb = slots + slot * pl.slot;
      for (int hh = lane; hh < 2 * ng; hh += 32)  // one 64-input half group (B rows of 128 B) per copy
        bulk_g2s(smem_u32(sb + pl.xoff + hh * kXTile), p.x + ((size_t)(2 * kg + hh) * p.B) * 64, p.B * 128,
                 full(slot));
      if (lane == 31) bulk_g2s(smem_u32(sb + pl.soff), p.s_in + (size_t)kg * 32, ng * 256, full(slot));
    };
    for (StageWalk st(pl, u0, u1); st.valid(); st.next(), ++si) {
      const int slot = si % S, round = si / S;
      if (round > 0 && !mbar_wait(empty(slot), (round - 1) & 1)) {
        ok = false;
        break;
      }
      if (lane == 0)
        mbar_arrive_expect_tx(full(slot), (uint32_t)(8 * st.ng * kSlab + 2 * st.ng * p.B * 128 + st.ng * 256));
      __syncwarp();
      const uint32_t sb = smem_u32(slots + slot * pl.slot);
      if (lane < 8)
        bulk_g2s(sb + lane * pl.ng * kSlab, p.w + ((size_t)(st.set * 8 + lane) * pl.NKG + st.kg) * kSlab,
                 st.ng * kSlab, full(slot));
      __syncwarp();
      if (waited) issue_x(slot, st.kg, st.ng);
      if (!waited && (si == S - 1 || st.u + st.ng >= u1)) {
        griddep_wait();  // the activation operand and its offsets come from the previous kernel
        if (ROLE == kRoleQKV) griddep_launch();
        waited = true;
        int s2i = 0;
        for (StageWalk s2(pl, u0, u1); s2i <= si; s2.next(), ++s2i) issue_x(s2i, s2.kg, s2.ng);
      }
    }
    if (!waited) {
      griddep_wait();
      if (ROLE == kRoleQKV) griddep_launch();
      int s2i = 0;  // stages issued before a timeout still expect their activation bytes
      for (StageWalk s2(pl, u0, u1); s2i < si && s2.valid(); s2.next(), ++s2i) issue_x(s2i, s2.kg, s2.ng);
    }
    // every copy this warp issued has landed before the CTA may leave
    for (int k = 0; k < S && k < si; ++k) {
      const int sj = si - 1 - k;
      if (!mbar_wait(full(sj % S), (sj / S) & 1)) ok = false;
    }
  } else if (warp == kMma || warp == kMma2) {
    // ------------------------------------------------------------ tensor-core issue (one thread per
    // issuing warp; issuer i takes the groups gi with gi % kIssuers == i)
    griddep_wait();
    if (ROLE == kRoleQKV) griddep_launch();
    const int issuer = warp == kMma ? 0 : 1;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(128, 32);
      int si = 0, gi = 0, last = -1;
      for (StageWalk st(pl, u0, u1); ok && st.valid(); st.next(), ++si) {
        const int slot = si % S;
        if (!mbar_wait(full(slot), (si / S) & 1)) {
          ok = false;
          break;
        }
        const uint32_t xs = smem_u32(slots + slot * pl.slot + pl.xoff);
        for (int kgl = 0; kgl < st.ng; ++kgl, ++gi) {
          if (gi % kIssuers != issuer) continue;
          const int a = gi % kNAcc, ua = gi / kNAcc, ab = gi % kNBuf;
          // A tile filled (decoders); accumulator a drained (epilogue, group gi - kNAcc)
          if (!mbar_wait(a_full + 8 * a, ua & 1) || (ua > 0 && !mbar_wait(acc_empty + 8 * a, (ua - 1) & 1))) {
            ok = false;
            break;
          }
          fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_f16_ts(tmem + kAccCol + 32 * a, tmem + kACol + 64 * ab + 8 * ks,
                       desc_sw128(xs + (2 * kgl + (ks >> 2)) * kXTile + 32 * (ks & 3)), idesc, ks > 0 ? 1u : 0u);
          mma_commit(mma_done + 8 * a);
          last = gi;
        }
        if (!ok) break;
        mma_commit(empty(slot));  // this thread's reads of the stage's activation tiles are done
      }
      // the tensor core has finished everything issued here before tensor memory is freed (the
      // issuers use disjoint accumulators and barriers)
      if (last >= 0 && !mbar_wait(mma_done + 8 * (last % kNAcc), (last / kNAcc) & 1)) ok = false;
    }
    __syncwarp();
  } else if (warp < kEpi0) {
    // ------------------------------------------------------------ decoders
    griddep_wait();
    if (ROLE == kRoleQKV) griddep_launch();
    const int q = warp & 3, half = (warp - kDec0) >> 2;  // lane quarter (tensor-memory lanes 32q..), input half
    int si = 0, gi = 0;
    for (StageWalk st(pl, u0, u1); ok && st.valid(); st.next(), ++si) {
      const int slot = si % S;
      if (!mbar_wait(full(slot), (si / S) & 1)) {
        ok = false;
        break;
      }
      const uint8_t* ws = slots + slot * pl.slot;
      // all of the stage's groups are decoded before one wait for the tensor-memory stores (the
      // wait's latency, not the decoding, would otherwise set the pace)
      for (int kgl = 0; kgl < st.ng; ++kgl) {
        const int g = gi + kgl, a = g % kNAcc, ua = g / kNAcc, ab = g % kNBuf;
        // A tile ab: the tensor core finished group g - kNBuf; stash a: the epilogue drained
        // group g - kNAcc
        if ((g >= kNBuf && !mbar_wait(mma_done + 8 * ((g - kNBuf) % kNAcc), ((g - kNBuf) / kNAcc) & 1)) ||
            (ua > 0 && !mbar_wait(acc_empty + 8 * a, (ua - 1) & 1))) {
          ok = false;
          break;
        }
        if (half == 0) {  // this quarter's 32 row scales of the group, for the epilogue
          const int rr = lane & 15;
          const uint16_t sb = *reinterpret_cast<const uint16_t*>(
              ws + ((2 * q + (lane >> 4)) * pl.ng + kgl) * kSlab + kCodes + 4 * (rr & 7) + 2 * (rr >> 3));
          scl[a * 128 + 32 * q + lane] = bf16_bits_to_f32(sb);
        } else if (q == 3) {  // the group's token offsets S (one per token; absent tokens 0)
          const sfix_t* ss = reinterpret_cast<const sfix_t*>(ws + pl.soff);
          sof[a * 32 + lane] = lane < p.B ? sfix_to_f32(ss[kgl * 32 + lane]) : 0.0f;
        }
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int T = 2 * q + s2;  // row tile: rows 16 T .. 16 T + 15 = tensor-memory lanes
          uint32_t r[16];
          if constexpr (E4) {  // 4 k-steps x 8 codes: two 16-byte loads
            const uint4* w8 = reinterpret_cast<const uint4*>(ws + (T * pl.ng + kgl) * kSlab + half * 1024 + lane * 32);
            const uint4 wa = w8[0], wb = w8[1];
            e4m3_words(wa.x, wa.y, r);
            e4m3_words(wa.z, wa.w, r + 4);
            e4m3_words(wb.x, wb.y, r + 8);
            e4m3_words(wb.z, wb.w, r + 12);
          } else {
            const uint4 w4 = *reinterpret_cast<const uint4*>(ws + (T * pl.ng + kgl) * kSlab + half * 512 + lane * 16);
            const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              uint32_t m[4];
              magic_word(wv[ks], m);
              r[4 * ks] = m[0];
              r[4 * ks + 1] = m[1];
              r[4 * ks + 2] = m[2];
              r[4 * ks + 3] = m[3];
            }
          }
          tmem_st16x256b_x4(tmem + kACol + 64 * ab + 32 * half + ((uint32_t)(16 * T) << 16), r);
        }
      }
      if (!ok) break;
      tmem_wait_st();
      fence_before();
      __syncwarp();
      if (lane == 0) {
        for (int kgl = 0; kgl < st.ng; ++kgl) mbar_arrive(a_full + 8 * ((gi + kgl) % kNAcc));
        mbar_arrive(empty(slot));
      }
      gi += st.ng;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    griddep_wait();
    if (ROLE == kRoleQKV) griddep_launch();
    const int q = warp & 3, te = tid - kEpi0 * 32;  // lane quarter; epilogue thread 0..127
    const int rblk = 32 * q + lane;                  // this thread's row of the 128-row block
    const int T = rblk >> 4, rr = rblk & 15;
    float tot[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) tot[t] = 0.0f;
    int gi = 0;
    for (StageWalk st(pl, u0, u1); ok && st.valid(); st.next()) {
      for (int kgl = 0; kgl < st.ng; ++kgl, ++gi) {
        const int a = gi % kNAcc, ua = gi / kNAcc;
        // the group's accumulator is complete; a_full (already complete) orders the decoders'
        // stash writes before these reads
        if (!mbar_wait(mma_done + 8 * a, ua & 1) || !mbar_wait(a_full + 8 * a, ua & 1)) {
          ok = false;
          break;
        }
        fence_after();
        uint32_t acc[32];
        tmem_ld32x32b_x32(tmem + kAccCol + 32 * a + ((uint32_t)(32 * q) << 16), acc);
        const float sc = scl[a * 128 + rblk];
        float s4[32];
#pragma unroll
        for (int t4 = 0; t4 < 8; ++t4) {
          const float4 v = E4 ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : reinterpret_cast<const float4*>(sof + a * 32)[t4];
          s4[4 * t4] = v.x;
          s4[4 * t4 + 1] = v.y;
          s4[4 * t4 + 2] = v.z;
          s4[4 * t4 + 3] = v.w;
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty + 8 * a);  // accumulator and stash entries free
#pragma unroll
        for (int t = 0; t < 32; ++t) tot[t] = fmaf(sc, __uint_as_float(acc[t]) - s4[t], tot[t]);
      }
      if (!ok) break;
      if (!st.piece_end()) continue;

      // ---- end of this CTA's piece of block st.set: its partial sums to the piece's slab (the
      // next kernel adds the slabs of a row in slab order)
      const int row = st.set * 128 + rblk;
      const int piece = cta - plan_first(pl, st.set);
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < p.B) __stcg(p.part + ((size_t)piece * p.B + t) * pl.N + row, tot[t]);
#pragma unroll
      for (int t = 0; t < 32; ++t) tot[t] = 0.0f;
    }
  }
  if (!ok) set_status(p.status, FT_DEV_TIMEOUT);
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == kMma) tmem_dealloc(tmem);
}

template <int ROLE, int FMT>
static cudaError_t launch_umma_role(const GemvParams& p, cudaStream_t st, bool pdl) {
  static int attr_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_smem[dev] < p.plan.smem) {
    cudaError_t e =
        cudaFuncSetAttribute(umma_kernel<ROLE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.plan.smem);
    if (e != cudaSuccess) return e;
    attr_smem[dev] = p.plan.smem;
  }
  return launch_ex(umma_kernel<ROLE, FMT>, dim3(p.plan.C), dim3(kThreads), (size_t)p.plan.smem, st, pdl, p);
}

template <int FMT>
static cudaError_t launch_umma_fmt(int role, const GemvParams& p, cudaStream_t st, bool pdl) {
  switch (role) {
    case kRoleQKV: return launch_umma_role<kRoleQKV, FMT>(p, st, pdl);
    case kRoleO: return launch_umma_role<kRoleO, FMT>(p, st, pdl);
    case kRoleGU: return launch_umma_role<kRoleGU, FMT>(p, st, pdl);
    case kRoleDown: return launch_umma_role<kRoleDown, FMT>(p, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_umma(int role, const GemvParams& p, cudaStream_t st, bool pdl) {
  if (p.plan.slab == kSlabBytesE4) return launch_umma_fmt<FT_WFMT_E4M3>(role, p, st, pdl);
  if (p.plan.slab == kSlabBytes) return launch_umma_fmt<FT_WFMT_INT4>(role, p, st, pdl);
  return cudaErrorInvalidValue;
}

int ft_umma_warps() { return kWarps; }

// Partition of a projection for the tensor-core kernel: 128-row blocks as
// sets, 3 groups per stage, units (set, group) spread evenly over the CTAs
// (sets split along K); every piece writes its partial sums to its own slab.
GemvPlan make_umma_plan(int role, int N, int K, int B, int sms, int smem_budget, int weight_format) {
  GemvPlan p = {};
  p.slab = slab_bytes_of(weight_format);
  p.N = N;
  p.K = K;
  p.NT = 4;
  p.RT = 8;
  p.NCW = 0;
  p.umma = 1;
  p.NTILE = N / kRowTile;
  p.NKG = K / kWGroup;
  p.NSET = (p.NTILE + p.RT - 1) / p.RT;
  const bool whole_sets = false;
  (void)role;
  p.whole = whole_sets ? 1 : 0;
  const int units = whole_sets ? p.NSET : p.NSET * p.NKG;
  p.C = sms < units ? sms : units;
  if (p.C < 1) p.C = 1;
  p.per = units / p.C;
  p.rem = units % p.C;
  p.rcp_per1 = ((1ull << 32) + (unsigned long long)p.per) / (unsigned long long)(p.per + 1);
  p.rcp_per = ((1ull << 32) + (unsigned long long)p.per - 1) / (unsigned long long)p.per;
  p.divs_exact = (unsigned long long)units * (unsigned long long)(p.per + 1) <= (1ull << 32) ? 1 : 0;
  p.npmax = 1;
  if (!whole_sets)
    for (int set = 0; set < p.NSET; ++set) p.npmax = std::max(p.npmax, plan_pieces(p, set));
  // 3 groups per stage: fewer ring hand-offs than 1 or 2 at the same depth (4 leaves 3 coarse
  // stages); E4M3 slabs are twice as large, so 2 groups keep 3 stages
  p.ng = std::min(weight_format == FT_WFMT_E4M3 ? 2 : 3, p.NKG);
  // slot: weight slabs of 8 tiles, activation half-group tiles (1024-aligned), offsets
  p.xoff = (int)align_up((size_t)8 * p.ng * p.slab, 1024);
  p.soff = p.xoff + 2 * p.ng * kXTile;
  p.slot = (int)align_up((size_t)p.soff + (size_t)p.ng * 256, 1024);
  p.xstride = 0;
  p.redoff = 0;
  p.zerooff = 0;
  p.slotoff = Smem::kSlots;
  int stages = (smem_budget - 1024 - p.slotoff) / p.slot;  // 1024: alignment slack
  if (stages > 8) stages = 8;
  if (stages < 2) stages = 2;
  p.stages = stages;
  p.smem = 1024 + p.slotoff + stages * p.slot;
  (void)B;
  return p;
}

}  // namespace ft
