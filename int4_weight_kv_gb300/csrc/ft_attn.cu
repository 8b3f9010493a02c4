// Decode attention over the Hadamard-rotated INT4 KV cache, with RoPE, the
// rotation of q, the new token's cache write, split-KV and the inverse rotation
// of the output (summary page, "무엇과 다른가": rotation of K/V, q and the
// output, split-KV reduction for long contexts; "전제와 한계": the 8-head INT4
// cache is read directly by the query heads, no head expansion).
//
// One CTA (kAttnWarps warps) per (request b, KV head h, split): the G = n_q / n_kv query
// heads of the group share every K/V byte the CTA reads.  Per 16-position tile
// a warp computes
//   S[pos][head]  = K^(16 x d) . q~ (d x 8 heads)       (A = K codes, FP16 exact)
//   online softmax in FP32 (exp2 domain, log2(e)/sqrt(d) folded into q~)
//   O[ch][head] += V^T(d x 16) . (P * s_v)(16 x 8)      (A = V codes, B = P via
//                                                        movmatrix transpose)
// The K entry's nibbles are stored so that a 16-byte load per thread is the
// A fragment of two k-steps; the V entry's nibbles so that two positions' bytes
// combine (prmt) into A fragments of V^T.  Per-position scales multiply the
// scores (K) and the probabilities (V).  The n_split CTAs of one (b, h) form a
// thread-block cluster.  CTA r merges heads r, r + n_split, ...: every CTA
// pushes its (max, sum, acc) partial of each head into the merging CTA's shared
// memory with asynchronous distributed-shared-memory stores that complete on
// the merger's mbarrier (no cluster-wide barrier at the end), and the merger
// combines them from its own shared memory with the new token, undoes the
// rotation and writes o.  The new token's k and v are loaded before the main
// loop and quantised (written to the cache at L_b by CTA 0) and decoded by the
// merging CTAs while their peers' partials arrive.
#include <atomic>

#include "ft_block.cuh"

namespace ft {

template <int D>
struct TileRegs {
  uint32_t k[2][D / 32];  // K words of positions g and g+8 (chunk tig)
  uint32_t v[4][D / 64];  // V words of positions 2tig, 2tig+1, 2tig+8, 2tig+9 (chunk g)
  uint16_t ks[2], vs[2];  // K / V scales of positions g and g+8
};

// K / V scales of positions p + g and p + g + 8 (clamped into the cache row).
__device__ __forceinline__ void load_scales(uint16_t (&ks)[2], uint16_t (&vs)[2], const uint8_t* cache,
                                            const KVLayout& L, int b, int h, int p, int g) {
  const int last = L.max_ctx - 1;
  const size_t r0 = L.row(b, h, min(p + g, last)), r1 = L.row(b, h, min(p + g + 8, last));
  const uint16_t* ksb = reinterpret_cast<const uint16_t*>(cache + L.ks);
  const uint16_t* vsb = reinterpret_cast<const uint16_t*>(cache + L.vs);
  ks[0] = ld_stream_u16(ksb + r0);
  ks[1] = ld_stream_u16(ksb + r1);
  vs[0] = ld_stream_u16(vsb + r0);
  vs[1] = ld_stream_u16(vsb + r1);
}

// Fragments and scales of one 16-position tile straight from the cache into
// registers (short contexts: a warp has a tile or two, nothing to pipeline).
template <int D>
__device__ __forceinline__ void load_tile(TileRegs<D>& r, const uint8_t* cache, const KVLayout& L, int b, int h, int p,
                                          int g, int tig) {
  const int last = L.max_ctx - 1;
  const int pk0 = min(p + g, last), pk1 = min(p + g + 8, last);
  const uint8_t* kb = cache + L.kc;
  const uint8_t* vb = cache + L.vc;
  const size_t r0 = L.row(b, h, pk0), r1 = L.row(b, h, pk1);
  if constexpr (D == 128) {
    const uint4 a = ld_stream_v4(kb + r0 * L.entry + tig * 16);
    const uint4 c = ld_stream_v4(kb + r1 * L.entry + tig * 16);
    r.k[0][0] = a.x; r.k[0][1] = a.y; r.k[0][2] = a.z; r.k[0][3] = a.w;
    r.k[1][0] = c.x; r.k[1][1] = c.y; r.k[1][2] = c.z; r.k[1][3] = c.w;
  } else {
    const uint2 a = ld_stream_v2(kb + r0 * L.entry + tig * 8);
    const uint2 c = ld_stream_v2(kb + r1 * L.entry + tig * 8);
    r.k[0][0] = a.x; r.k[0][1] = a.y;
    r.k[1][0] = c.x; r.k[1][1] = c.y;
  }
  const int pv[4] = {p + 2 * tig, p + 2 * tig + 1, p + 2 * tig + 8, p + 2 * tig + 9};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const size_t rv = L.row(b, h, min(pv[q], last));
    if constexpr (D == 128) {
      const uint2 a = ld_stream_v2(vb + rv * L.entry + g * 8);
      r.v[q][0] = a.x;
      r.v[q][1] = a.y;
    } else {
      r.v[q][0] = ld_stream_u32(vb + rv * L.entry + g * 4);
    }
  }
  load_scales(r.ks, r.vs, cache, L, b, h, p, g);
}

// Fragments of one 16-position tile from its ring slot: K entries of positions
// 0..15 (d/2 bytes each), then V entries.  Positions past the copied ones hold
// stale codes; the caller masks them (scores -inf, V scales 0).
template <int D>
__device__ __forceinline__ void tile_from_smem(TileRegs<D>& r, const uint8_t* s, int g, int tig) {
  constexpr int E = D / 2;
  const uint8_t* ks = s;
  const uint8_t* vs = s + 16 * E;
  if constexpr (D == 128) {
    const uint4 a = *reinterpret_cast<const uint4*>(ks + g * E + tig * 16);
    const uint4 c = *reinterpret_cast<const uint4*>(ks + (g + 8) * E + tig * 16);
    r.k[0][0] = a.x; r.k[0][1] = a.y; r.k[0][2] = a.z; r.k[0][3] = a.w;
    r.k[1][0] = c.x; r.k[1][1] = c.y; r.k[1][2] = c.z; r.k[1][3] = c.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(ks + g * E + tig * 8);
    const uint2 c = *reinterpret_cast<const uint2*>(ks + (g + 8) * E + tig * 8);
    r.k[0][0] = a.x; r.k[0][1] = a.y;
    r.k[1][0] = c.x; r.k[1][1] = c.y;
  }
  const int pv[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr (D == 128) {
      const uint2 a = *reinterpret_cast<const uint2*>(vs + pv[q] * E + g * 8);
      r.v[q][0] = a.x;
      r.v[q][1] = a.y;
    } else {
      r.v[q][0] = *reinterpret_cast<const uint32_t*>(vs + pv[q] * E + g * 4);
    }
  }
}


__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// RoPE at position pos on a d-vector held stride-32 (lane owns l + 32 m).
// turn[i] is inv_freq[i] / (2 pi) as a 64-bit binary fraction, so pos * turn[i]
// modulo 2^64 is the angle in turns reduced exactly modulo one turn; its top 32
// bits, read as a signed fraction in [-1/2, 1/2), feed sincospif.
template <int NPL>
__device__ __forceinline__ void warp_rope(float (&v)[NPL], int pos, const uint64_t* turn) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < NPL / 2; ++m) {
    const int i = lane + 32 * m;
    const uint64_t t = (uint64_t)(uint32_t)pos * turn[i];
    const float half_turns = (float)(int32_t)(uint32_t)(t >> 32) * 4.656612873077393e-10f;  // x 2^-31
    float sn, cs;
    sincospif(half_turns, &sn, &cs);
    const float x1 = v[m], x2 = v[m + NPL / 2];
    v[m] = x1 * cs - x2 * sn;
    v[m + NPL / 2] = x2 * cs + x1 * sn;
  }
}

// Lazy rescaling threshold of the online softmax (log2 units): weights up to
// 2^4 = 16 times the running max's keep P = weight * V scale within FP16 for V
// scales up to 4094.
constexpr float kLazyLog2 = 4.0f;

template <int D>
__global__ void __launch_bounds__(kAttnWarps * 32, 4) attn_kernel(const AttnParams p) {
  constexpr int NPL = D / 32;
  constexpr int KT = D / 16;  // k-tiles of q.K == m-tiles of P.V
  constexpr int PW = D + 4;             // one partial: running max, sum, 2 pad, acc[D] (16-byte rows)
  __shared__ float qt[8][D];            // rotated, scaled query (FP16 values)
  __shared__ float qoff[8];             // its operand offsets (magic-number decode)
  __shared__ float knew[D], vnew[D];
  __shared__ float fac[8][1 + kAttnWarps];  // per head: CTA max, then each warp's rescale factor
  __shared__ __align__(8) uint64_t inbox_bar;  // completes when every partial of this CTA's heads arrived
  __shared__ __align__(8) uint64_t kv_bar[kAttnWarps][kAttnMaxSlots];  // a warp's ring slot has landed
  // dynamic: mrg[4][G * PW], each warp's partial of every head (before the main
  // loop the same area holds the staged QKV pieces), then, after the larger of
  // the two, inbox[n_split * ceil(G / n_split)][PW], the partials of the heads
  // this CTA merges, pushed by every CTA of the cluster (slot j * n_split + r
  // holds CTA r's partial of head split + j * n_split)
  extern __shared__ __align__(16) float dyn[];
  __shared__ uint8_t stage[2][D];
  __shared__ __align__(16) uint8_t stage_out[2][D / 2];
  __shared__ uint16_t stage_sc[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int split = blockIdx.x % p.nsplit;
  const int bh = blockIdx.x / p.nsplit;
  const int h = bh % p.nkv, b = bh / p.nkv;
  const int G = p.G;
  const int Lb = p.pos[b];
  if (Lb < 0 || Lb >= p.L.max_ctx) {
    // every CTA of this cluster serves the same request, so all leave here together;
    // they still wait for the QKV kernel, so that this kernel's completion implies
    // its predecessor's (the next kernels rely on that chain)
    if (tid == 0 && split == 0 && h == 0) set_status(p.status, FT_DEV_CAPACITY);
    griddep_launch();
    griddep_wait();
    return;
  }
  const int ntiles = (Lb + 15) / 16;
  const int tps = (ntiles + p.nsplit - 1) / p.nsplit;
  const int t0 = split * tps, t1 = min(t0 + tps, ntiles);
  const int p1 = min(16 * t1, Lb);

  // heads this CTA merges: split, split + n_split, ...; the inbox barrier
  // expects the partials of all n_split CTAs for each
  int nloc = 0;
  for (int hh = split; hh < G; hh += p.nsplit) ++nloc;
  if (tid == 0) {
    mbar_init(smem_u32(&inbox_bar), 1);
    mbar_fence_init();
    if (nloc) mbar_arrive_expect_tx(smem_u32(&inbox_bar), (uint32_t)(nloc * p.nsplit * PW * 4));
  }
  cluster_arrive();  // paired with cluster_wait() before the first push into a peer

  // history K/V do not depend on earlier kernels: start streaming now.  Each warp
  // owns tiles t0 + warp + k kAttnWarps (k = 0, 1, ...) and a ring of kv_slots
  // slots; lane 0 bulk-copies tile k into slot k % kv_slots (the K entries of
  // its 16 positions are contiguous in the cache, and so are the V entries) and
  // refills the slot with tile k + kv_slots once the warp has used it.
  const int ns = p.kv_slots;
  const uint32_t kvb0 = smem_u32(&kv_bar[warp][0]);
  uint8_t* ring = reinterpret_cast<uint8_t*>(dyn + attn_ring_off(G, p.nsplit, D, p.qkv_plan.npmax)) +
                  warp * ns * 16 * D;
  auto issue_tile = [&](int k) {
    const int tile = t0 + warp + k * kAttnWarps;
    if (tile >= t1) return;
    const int p0 = 16 * tile, n = min(16, p.L.max_ctx - p0);  // positions in the cache row
    const uint32_t bar = kvb0 + 8 * (k % ns);
    const size_t r = p.L.row(b, h, p0);
    const uint32_t dst = smem_u32(ring + (k % ns) * 16 * D);
    mbar_arrive_expect_tx(bar, (uint32_t)(n * D));
    bulk_g2s(dst, p.cache + p.L.kc + r * p.L.entry, (uint32_t)(n * (D / 2)), bar);
    bulk_g2s(dst + 8 * D, p.cache + p.L.vc + r * p.L.entry, (uint32_t)(n * (D / 2)), bar);
  };
  if (lane == 0 && ns > 0) {
    for (int s2 = 0; s2 < ns; ++s2) mbar_init(kvb0 + 8 * s2, 1);
    mbar_fence_init();
    for (int k = 0; k < ns; ++k) issue_tile(k);
  }
  __syncwarp();
  int ti = t0 + warp;
  uint16_t ksn[2] = {0, 0}, vsn[2] = {0, 0};  // ring: scales of the warp's next tile
  TileRegs<D> reg_cur;                        // no ring (kv_slots 0): the warp's first tile
  if (ti < t1) {
    if (ns > 0)
      load_scales(ksn, vsn, p.cache, p.L, b, h, 16 * ti, g);
    else
      load_tile<D>(reg_cur, p.cache, p.L, b, h, 16 * ti, g, tig);
  }

  griddep_wait();

  // The QKV projection arrives as piece slabs (one per CTA that shared a row
  // set), added here in slab order.  The CTA first stages the pieces it needs
  // (its G query heads and, in merging CTAs, k and v) in shared memory with
  // asynchronous copies, each 16-byte chunk of each piece once (no register
  // holds the data in flight; the RMSNorm partial sums load meanwhile), in the
  // area that later holds the warps' partials.  Sets are multiples of 32 rows,
  // so a 16-byte chunk lies in one set.
  const GemvPlan& qp = p.qkv_plan;
  const bool merger = split < G;
  const int npm = qp.npmax;
  float* qkv_st = dyn;  // [segment (q heads, then k and v)][piece][D]
  {
    const int srows = qp.RT * kRowTile, nseg = G + (merger ? 2 : 0);
    const size_t slab = (size_t)p.B * qp.N;
    const float* src0 = p.qkv_part + (size_t)b * qp.N;
    for (int i = tid; i < nseg * npm * (D / 4); i += kAttnWarps * 32) {
      const int c4 = i % (D / 4), sj = i / (D / 4), j = sj % npm, sg = sj / npm;
      const int row = (sg < G ? h * G + sg : p.nq + (sg - G) * p.nkv + h) * D + 4 * c4;
      if (j < plan_pieces(qp, row / srows)) cp_async16(smem_u32(qkv_st + sj * D + 4 * c4), src0 + j * slab + row);
    }
  }
  float rho1;  // RMSNorm row factor of the block input, from the prep kernel's partial sums
  {
    float t = 0.0f;
    for (int k = lane; k < p.nssq; k += 32) t += __ldcg(p.ssq1 + b * p.nssq + k);
    rho1 = rsqrtf(warp_sum(t) * p.inv_h + p.eps);
    if (tid == 0 && h == 0 && split == 0) p.rho1[b] = rho1;
  }
  cp_async_wait_all();
  __syncthreads();
  // sums of the staged pieces of channels lane + 32 m of segment sg, in slab order
  auto staged_sum = [&](int sg, int base, float (&v)[NPL]) {
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      const int np = plan_pieces(qp, (base + 32 * m) / (qp.RT * kRowTile));
      const float* q = qkv_st + sg * npm * D + lane + 32 * m;
      float a = q[0];
      for (int j = 1; j < np; ++j) a += q[j * D];
      v[m] = a;
    }
  };
  // ---- rotated, scaled query of each head (rho1, RoPE, Hadamard, softmax scale)
  for (int u = warp; u < G; u += kAttnWarps) {
    float v[NPL];
    const int qbase = (h * G + u) * D;
    staged_sum(u, qbase, v);
    if (split == 0) {  // the summed projection, recorded for inspection
#pragma unroll
      for (int m = 0; m < NPL; ++m) p.qkv[(size_t)b * p.Nqkv + qbase + lane + 32 * m] = v[m];
    }
#pragma unroll
    for (int m = 0; m < NPL; ++m) v[m] *= rho1;
    warp_rope<NPL>(v, Lb, p.rope_turn);
    warp_fwht<NPL>(v, p.hb);
    // q~ as the FP16 B operand (channels c % 16 >= 8 hold q / 16) and its offset
    float sq = 0.0f;
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      const int c = lane + 32 * m;
      const float q = __half2float(__float2half_rn(v[m] * p.qscale));
      qt[u][c] = q;
      float st;
      (void)op_encode(q, c, st);
      sq += st;
    }
    sq = warp_sum(sq);  // one warp, fixed order: deterministic
    if (lane == 0) qoff[u] = sq;
  }
  // the new token's k (warp 0) or v (warp 1) of the merging CTAs, with rho1 applied
  float kvraw[NPL];
  if (merger && warp < 2) {
    const int kvbase = (p.nq + warp * p.nkv + h) * D;
    staged_sum(G + warp, kvbase, kvraw);
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      if (split == 0) p.qkv[(size_t)b * p.Nqkv + kvbase + lane + 32 * m] = kvraw[m];  // for inspection
      kvraw[m] *= rho1;
    }
  }
  __syncthreads();
  uint32_t bq[KT][2];
#pragma unroll
  for (int kt = 0; kt < KT; ++kt) {
    if (g < G) {
      const int c = 16 * kt + 2 * tig;
      bq[kt][0] = pack_half2(qt[g][c], qt[g][c + 1]);
      bq[kt][1] = pack_half2(qt[g][c + 8] * 0.0625f, qt[g][c + 9] * 0.0625f);
    } else {
      bq[kt][0] = bq[kt][1] = 0u;
    }
  }
  const float qo0 = (2 * tig < G) ? qoff[2 * tig] : 0.0f;
  const float qo1 = (2 * tig + 1 < G) ? qoff[2 * tig + 1] : 0.0f;

  float acc[KT][4];
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
  // offset accumulator: the same P.V product with every V code replaced by its
  // decode offset (rows of constant 1032 / 1152), rescaled like acc
  float kacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const uint32_t kappa[4] = {kHOffLo, kHOffLo, kHOffHi, kHOffHi};
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

  // one 16-position tile of this warp: scores, online softmax, P.V
  auto tile_step = [&](const TileRegs<D>& cur, int ti, bool lazy) {
    const int p0 = 16 * ti;
    // S = K . q~   (rows: positions g, g+8; columns: heads 2tig, 2tig+1)
    float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      uint32_t dg[4], dg8[4];
      magic_word(cur.k[0][j], dg);
      magic_word(cur.k[1][j], dg8);
      const uint32_t a0[4] = {dg[0], dg8[0], dg[1], dg8[1]};
      const uint32_t a1[4] = {dg[2], dg8[2], dg[3], dg8[3]};
      mma_f16(sacc, a0, bq[2 * j][0], bq[2 * j][1]);
      mma_f16(sacc, a1, bq[2 * j + 1][0], bq[2 * j + 1][1]);
    }
    const bool va = (p0 + g) < p1, vb = (p0 + g + 8) < p1;
    const float ks0 = bf16_bits_to_f32(cur.ks[0]), ks1 = bf16_bits_to_f32(cur.ks[1]);
    const float s0 = va ? (sacc[0] - qo0) * ks0 : -INFINITY;
    const float s1 = va ? (sacc[1] - qo1) * ks0 : -INFINITY;
    const float s2 = vb ? (sacc[2] - qo0) * ks1 : -INFINITY;
    const float s3 = vb ? (sacc[3] - qo1) * ks1 : -INFINITY;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    // With `lazy` (long shares) the running max moves (and the sums are rescaled) only when
    // a score exceeds it by more than kLazyLog2 (warp-uniform decision): the result is the
    // same softmax, the unnormalised weights stay below 2^kLazyLog2, and most tiles of a
    // long context skip the rescale.  Every tile holds a valid position, so the first one
    // always moves it.
    if (!lazy || __any_sync(0xffffffffu, mx0 > m0 + kLazyLog2 || mx1 > m1 + kLazyLog2)) {
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int mt = 0; mt < KT; ++mt) {
        acc[mt][0] *= al0;
        acc[mt][1] *= al1;
        acc[mt][2] *= al0;
        acc[mt][3] *= al1;
      }
      kacc[0] *= al0;
      kacc[1] *= al1;
      kacc[2] *= al0;
      kacc[3] *= al1;
    }
    const float e0 = exp2f(s0 - m0), e1 = exp2f(s1 - m1), e2 = exp2f(s2 - m0), e3 = exp2f(s3 - m1);
    l0 += e0 + e2;
    l1 += e1 + e3;
    const float vs0 = va ? bf16_bits_to_f32(cur.vs[0]) : 0.0f;
    const float vs1 = vb ? bf16_bits_to_f32(cur.vs[1]) * 0.0625f : 0.0f;  // positions 8..15: operand / 16
    const uint32_t P0 = pack_half2(e0 * vs0, e1 * vs0);  // position g,   heads 2tig, 2tig+1
    const uint32_t P1 = pack_half2(e2 * vs1, e3 * vs1);  // position g+8
    const uint32_t pb0 = movmatrix_trans(P0);            // positions 2tig, 2tig+1 of head g
    const uint32_t pb1 = movmatrix_trans(P1);            // positions 2tig+8, 2tig+9
    // O += V^T . P  (positions 2tig, 2tig+1 decode at 1024 + c, positions +8 at 1024 + 16 c)
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
      uint32_t lo01[4], hi01[4], lo23[4], hi23[4];
      magic_low4(prmt(cur.v[0][j], cur.v[1][j], 0x5410u), lo01);
      magic_low4(prmt(cur.v[0][j], cur.v[1][j], 0x7632u), hi01);
      magic_high4(prmt(cur.v[2][j], cur.v[3][j], 0x5410u), lo23);
      magic_high4(prmt(cur.v[2][j], cur.v[3][j], 0x7632u), hi23);
      const uint32_t A0[4] = {lo01[0], lo01[1], lo23[0], lo23[1]};
      const uint32_t A1[4] = {lo01[2], lo01[3], lo23[2], lo23[3]};
      const uint32_t A2[4] = {hi01[0], hi01[1], hi23[0], hi23[1]};
      const uint32_t A3[4] = {hi01[2], hi01[3], hi23[2], hi23[3]};
      mma_f16(acc[4 * j + 0], A0, pb0, pb1);
      mma_f16(acc[4 * j + 1], A1, pb0, pb1);
      mma_f16(acc[4 * j + 2], A2, pb0, pb1);
      mma_f16(acc[4 * j + 3], A3, pb0, pb1);
    }
    mma_f16(kacc, kappa, pb0, pb1);
  };
  int kt_done = 0;  // tiles of this warp consumed (ring)
  bool kv_ok = true;
  if (ns == 0) {
    for (; ti < t1; ti += kAttnWarps) {  // plain loads, the next tile in flight in registers
      TileRegs<D> nxt;
      const bool more = ti + kAttnWarps < t1;
      if (more) load_tile<D>(nxt, p.cache, p.L, b, h, 16 * (ti + kAttnWarps), g, tig);
      tile_step(reg_cur, ti, false);
      if (more) reg_cur = nxt;
    }
  }
  for (; ns > 0 && ti < t1; ti += kAttnWarps, ++kt_done) {
    TileRegs<D> cur;
    cur.ks[0] = ksn[0], cur.ks[1] = ksn[1], cur.vs[0] = vsn[0], cur.vs[1] = vsn[1];
    if (ti + kAttnWarps < t1) load_scales(ksn, vsn, p.cache, p.L, b, h, 16 * (ti + kAttnWarps), g);
    if (!mbar_wait(kvb0 + 8 * (kt_done % ns), (kt_done / ns) & 1)) {
      kv_ok = false;
      break;
    }
    tile_from_smem<D>(cur, ring + (kt_done % ns) * 16 * D, g, tig);
    tile_step(cur, ti, true);
    // the slot's fragments are consumed (the MMAs above used them): refill it
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async_smem();
      issue_tile(kt_done + ns);
    }
  }
  if (!kv_ok) {  // a copy never landed: flag it, and wait (bounded) for the ones still in flight
    if (lane == 0) {
      set_status(p.status, FT_DEV_TIMEOUT);
      for (int k = kt_done; k < kt_done + ns; ++k)
        if (t0 + warp + k * kAttnWarps < t1) mbar_wait(kvb0 + 8 * (k % ns), (k / ns) & 1);
    }
    __syncwarp();
  }
  griddep_launch();

  // remove the decode offsets (every row of kacc carries the same value)
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) {
    acc[mt][0] -= kacc[0];
    acc[mt][1] -= kacc[1];
    acc[mt][2] -= kacc[0];
    acc[mt][3] -= kacc[1];
  }

  // ---- merge the warps of the CTA into this CTA's partial (kept in smem)
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  float* mrg = dyn;                       // [4][G * PW]
  // [n_split * ceil(G / n_split)][PW], after the larger of the partials and the
  // staged QKV pieces (peers push into it while this CTA may still read those)
  float* inbox = dyn + max(kAttnWarps * G * PW, attn_stage_floats(G, D, npm));
  float* mw = mrg + warp * G * PW;
  const bool c0ok = 2 * tig < G, c1ok = 2 * tig + 1 < G;  // this lane's two head columns exist
  float* h0 = mw + (2 * tig) * PW;
  float* h1 = mw + (2 * tig + 1) * PW;
  if (g == 0) {
    if (c0ok) h0[0] = m0, h0[1] = l0;
    if (c1ok) h1[0] = m1, h1[1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < KT; ++mt) {
    const int c0 = 16 * mt + g, c1 = c0 + 8;
    if (c0ok) h0[4 + c0] = acc[mt][0], h0[4 + c1] = acc[mt][2];
    if (c1ok) h1[4 + c0] = acc[mt][1], h1[4 + c1] = acc[mt][3];
  }
  __syncthreads();
  if (tid < G) {  // per head: the CTA max and each warp's rescale factor
    float mx[kAttnWarps], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mx[w] = mrg[(w * G + tid) * PW]);
    fac[tid][0] = M;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) fac[tid][1 + w] = (mx[w] == -INFINITY) ? 0.0f : exp2f(mx[w] - M);
  }
  __syncthreads();
  // ---- this CTA's partial of every head, pushed into the inbox of the CTA that
  // merges the head (asynchronous DSMEM stores completing on its inbox barrier)
  cluster_wait();  // every CTA of the cluster has started (arrived at entry)
  const uint32_t inbox0 = smem_u32(inbox);
  constexpr int PW4 = PW / 4;
  for (int i = tid; i < G * PW4; i += kAttnWarps * 32) {
    const int hh = i / PW4, e4 = i - hh * PW4;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float4 a = reinterpret_cast<const float4*>(mrg + (w * G + hh) * PW)[e4];
      const float f = fac[hh][1 + w];
      v.x = fmaf(a.x, f, v.x);
      v.y = fmaf(a.y, f, v.y);
      v.z = fmaf(a.z, f, v.z);
      v.w = fmaf(a.w, f, v.w);
    }
    if (e4 == 0) v = make_float4(fac[hh][0], v.y, 0.0f, 0.0f);  // (max, sum)
    const int slot = (hh / p.nsplit) * p.nsplit + split;
    st_async_v4(inbox0 + 16 * (slot * PW4 + e4), smem_u32(&inbox_bar), (uint32_t)(hh % p.nsplit), v);
  }

  // ---- the new token (merging CTAs): RoPE on k, rotation, INT4 (cache write at
  // L_b by split 0), decode; overlaps the peers' pushes
  if (merger && warp < 2) {
    float v[NPL];
#pragma unroll
    for (int m = 0; m < NPL; ++m) v[m] = kvraw[m];
    if (warp == 0) warp_rope<NPL>(v, Lb, p.rope_turn);
    warp_fwht<NPL>(v, p.hb);
    const size_t row = p.L.row(b, h, Lb);
    uint8_t* entry = (split == 0) ? p.cache + (warp == 0 ? p.L.kc : p.L.vc) + row * p.L.entry : stage_out[warp];
    uint16_t* sc = (split == 0) ? reinterpret_cast<uint16_t*>(p.cache + (warp == 0 ? p.L.ks : p.L.vs)) + row
                                : &stage_sc[warp];
    warp_quant_store<NPL>(v, warp == 0, stage[warp], entry, sc);
    float* dst = (warp == 0) ? knew : vnew;
#pragma unroll
    for (int m = 0; m < NPL; ++m) dst[lane + 32 * m] = v[m];
  }
  if (nloc == 0) return;  // nothing to merge; nobody pushes into this CTA
  __syncthreads();          // knew / vnew
  if (!mbar_wait(smem_u32(&inbox_bar), 0)) {  // every partial of this CTA's heads has arrived
    if (tid == 0) set_status(p.status, FT_DEV_TIMEOUT);
    return;
  }

  // ---- CTA r merges heads r, r + n_split, ...: the new token and the n_split partials
  for (int j = warp; split + p.nsplit * j < G; j += kAttnWarps) {
    const int hh = split + p.nsplit * j;
    float sn = 0.0f;
#pragma unroll
    for (int m = 0; m < NPL; ++m) sn += qt[hh][lane + 32 * m] * knew[lane + 32 * m];
    sn = warp_sum(sn);
    float M = sn;
    for (int r = 0; r < p.nsplit; ++r) M = fmaxf(M, inbox[(j * p.nsplit + r) * PW]);
    const float wn = exp2f(sn - M);
    float lsum = wn;
    float o[NPL];
#pragma unroll
    for (int m = 0; m < NPL; ++m) o[m] = wn * vnew[lane + 32 * m];
    for (int r = 0; r < p.nsplit; ++r) {
      const float* part = inbox + (j * p.nsplit + r) * PW;
      const float ms = part[0];
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      lsum += w * part[1];
#pragma unroll
      for (int m = 0; m < NPL; ++m) o[m] += w * part[4 + lane + 32 * m];
    }
    const float inv = 1.0f / lsum;
#pragma unroll
    for (int m = 0; m < NPL; ++m) o[m] *= inv;
    warp_fwht<NPL>(o, p.hb);
    const int kbase = (h * G + hh) * D;  // input index of channel 0 of this head in the O projection
    bool bad = false;
    float so = 0.0f;
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      const int k = kbase + lane + 32 * m;
      bad |= !(fabsf(o[m]) <= 65504.0f);
      float st;
      p.o_h[op_index(b, k, p.B)] = op_encode(o[m], k, st);
      so += st;
    }
    so = warp_sum(so);  // a head (d <= 128 channels) lies inside one 128-input group
    // the heads of a group (two at d = 64) add exact integers: any order
    if (lane == 0) sfix_atomic_add(p.s_o + (kbase / kWGroup) * 32 + b, f32_to_sfix(so));
    if (bad) set_status(p.status, FT_DEV_RANGE);
  }
}

// Per-device caches of the kernel attributes the host plan needs (the queries
// cost microseconds; every block call plans).  Benign races: equal values.
static std::atomic<int> g_attn_static[64][2];
static std::atomic<int> g_attn_occ[64][2][9][kAttnMaxPieces + 1];

static const void* attn_fn(int d) { return d == 128 ? (const void*)attn_kernel<128> : (const void*)attn_kernel<64>; }

int attn_smem_bytes(int G, int nsplit, int d, int npmax, int kv_slots) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  const int di = d == 128 ? 1 : 0;
  int stat = g_attn_static[dev][di].load(std::memory_order_relaxed);
  if (stat <= 0) {
    cudaFuncAttributes fa = {};
    const cudaError_t e = cudaFuncGetAttributes(&fa, attn_fn(d));
    stat = (e == cudaSuccess) ? (int)fa.sharedSizeBytes : 8 * 1024;
    if (e == cudaSuccess) g_attn_static[dev][di].store(stat, std::memory_order_relaxed);
  }
  return stat + attn_dyn_smem(G, nsplit, d, npmax, kv_slots);
}

int attn_ctas_per_sm(int G, int d, int npmax) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || G < 1 || G > 8) return 0;
  if (npmax < 1 || npmax > kAttnMaxPieces) return 0;
  const int di = d == 128 ? 1 : 0;
  int n = g_attn_occ[dev][di][G][npmax].load(std::memory_order_relaxed);
  if (n > 0) return n;
  // this many staged QKV pieces, the largest inbox (16 splits) and the ring of CTAs sharing an SM
  const size_t dyn = (size_t)attn_dyn_smem(G, 16, d, npmax, kAttnSharedSlots);
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_fn(d), kAttnWarps * 32, dyn);
  if (e != cudaSuccess) return 0;
  g_attn_occ[dev][di][G][npmax].store(n, std::memory_order_relaxed);
  return n;
}

static std::atomic<int> g_attn_cl[64][2][9];

// Allows the largest dynamic shared memory an attention CTA can ask for (G = 8,
// 16 splits, kAttnMaxPieces staged pieces, d = 128, the deepest ring: about
// 114 KB, above the default 48 KB).  Idempotent; false if the runtime refuses.
static bool attn_allow_smem(const void* fn) {
  const int most = attn_dyn_smem(8, 16, 128, kAttnMaxPieces, kAttnMaxSlots);
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, most) == cudaSuccess;
}

int attn_max_cluster(int G, int d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || G < 1 || G > 8) return 8;
  const int di = d == 128 ? 1 : 0;
  int c = g_attn_cl[dev][di][G].load(std::memory_order_relaxed);
  if (c > 0) return c;
  c = 8;
  const void* fn = attn_fn(d);
  if (attn_allow_smem(fn) && cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(kAttnWarps * 32);
    cfg.dynamicSmemBytes = attn_dyn_smem(G, 16, d, kAttnMaxPieces, kAttnSharedSlots);
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = 16;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0) c = 16;
  }
  cudaGetLastError();  // a refused query leaves no sticky state behind
  g_attn_cl[dev][di][G].store(c, std::memory_order_relaxed);
  return c;
}

cudaError_t launch_attn(const AttnParams& p, int head_dim, cudaStream_t st, bool pdl) {
  static std::atomic<int> allowed[64][2];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int di = head_dim == 128 ? 1 : 0;
  if (!allowed[dev][di].load(std::memory_order_relaxed)) {
    if (!attn_allow_smem(attn_fn(head_dim))) return cudaErrorInvalidValue;
    allowed[dev][di].store(1, std::memory_order_relaxed);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.nkv * p.nsplit));
  cfg.blockDim = dim3(kAttnWarps * 32);
  cfg.dynamicSmemBytes = attn_dyn_smem(p.G, p.nsplit, head_dim, p.qkv_plan.npmax, p.kv_slots);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.nsplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_kernel<128>, p);
  return cudaLaunchKernelEx(&cfg, attn_kernel<64>, p);
}

}  // namespace ft
