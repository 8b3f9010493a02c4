// The decode block as ONE persistent kernel (summary page, "어떻게 동작하나":
// the INT4 projections with RMSNorm gains folded into the weights and the row
// factors applied after accumulation; "무엇과 다른가": per-group scales,
// rotated INT4 KV cache, rotated query and inverse rotation of the output,
// split-KV attention for long contexts; "전제와 한계": the INT4 cache read
// directly by the query heads of each KV head).
//
// GB300 design.  One CTA per SM, all co-resident (cooperative launch).  Each
// CTA has a producer warp and NCW consumer warps, and one ring of shared-memory
// stages that never drains between phases: the producer streams, in order,
// this CTA's share of
//     QKV weights | KV-cache tiles for attention | O weights | gate/up weights | down weights
// with 1-D bulk async copies (mbarrier completion).  None of these bytes depend
// on earlier phases, so HBM streaming runs ahead across phase boundaries; only
// each GEMV stage's activation chunk (tens of bytes per token) waits for the
// grid barrier that publishes it and is issued into the already-armed stage.
//
// Phases and grid barriers (G0..G5, one arrival counter each in the workspace):
//   P0  input -> FP16 operand + group offsets, per-group sums of x^2, this
//       call's accumulators cleared                                        -> G0
//   P1  QKV: split-K units, red.add into FP32 accumulators                 -> G1
//   P2  attention: each (request, KV head) pair is cut into pieces of at
//       least tmin 16-position tiles (short contexts: one piece), pieces go to
//       CTAs round-robin; the piece holding position L_b also takes the new
//       token -- rotated, quantised, written to the cache and read back; a
//       pair of several pieces is merged by its last piece (atomic ticket);
//       o is written as the O operand                                      -> G2
//   P3  O: whole row sets per CTA; the epilogue forms h1 = x + W_o o and
//       writes the gate/up operand, its offsets and sums of h1^2           -> G3
//   P4  gate/up: whole row sets per CTA, SwiGLU in the epilogue with rho2    -> G4
//   P5  down: red.add into the output accumulator                          -> G5
//       (a BF16 output is then converted by every CTA).
// At the end of a CTA's piece of a row set the consumer warps reduce their
// partial sums together through shared memory and apply the role epilogue.
// Every wait (mbarrier or grid barrier) is bounded; a wait that gives up sets
// FT_DEV_TIMEOUT and a workspace abort flag that ends every other wait, and
// the kernel still leaves through its normal exit (named barriers are always
// reached, copies in flight are waited for).  The last CTA to leave resets
// the counters, so the workspace is ready for the next call.
#include <cmath>
#include <mutex>

#include "ft_block.cuh"

namespace ft {

constexpr int kSetRows = 64;  // rows of a row-tile set (RT = 4 tiles of 16)
static_assert(GemvShape<1>::RT * kRowTile == kSetRows && GemvShape<4>::RT * kRowTile == kSetRows,
              "sets of 64 rows: half of a 128-input group of the next projection");

// ------------------------------------------------------------------ waits
// Workspace words: one arrival counter per grid barrier (an early arrival at a
// later barrier can never complete an earlier one), the exit counter and the
// abort flag.
constexpr int kNumGridBars = 6;
constexpr int kSyncExit = kNumGridBars, kSyncAbort = kNumGridBars + 1;

__device__ __forceinline__ void raise_abort(const BlockParams& p) {
  atomicExch(p.sync + kSyncAbort, 1u);
  set_status(p.status, FT_DEV_TIMEOUT);
}

__device__ bool mbar_wait_ab(uint32_t bar, uint32_t parity, const uint32_t* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (ld_volatile_u32(abort) != 0u) return false;
      if (globaltimer() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Warp-wide bounded mbarrier wait with one outcome for every lane; raises the
// abort flag when it gives up.
__device__ bool warp_wait(const BlockParams& p, uint32_t bar, uint32_t parity) {
  bool r = mbar_wait_ab(bar, parity, p.sync + kSyncAbort);
  r = __all_sync(0xffffffffu, r);
  if (!r && (threadIdx.x & 31) == 0) raise_abort(p);
  return r;
}

// One thread per CTA arrives at grid barrier k, after the CTA's writers of
// the phase synchronised.
__device__ __forceinline__ void grid_arrive(const BlockParams& p, int k) {
  __threadfence();
  atomicAdd(p.sync + k, 1u);
}

// Warp-wide wait for grid barrier k to complete; false (abort raised) on
// timeout.
__device__ __noinline__ bool grid_wait_warp(const BlockParams& p, int k) {
  const uint32_t target = (uint32_t)p.C;
  uint32_t ok = 1u;
  if ((threadIdx.x & 31) == 0) {
    if (ld_acquire_u32(p.sync + k) < target) {
      const unsigned long long t0 = globaltimer();
      for (uint32_t it = 1;; ++it) {
        if (ld_acquire_u32(p.sync + k) >= target) break;
        if ((it & 15u) == 0 &&
            (ld_volatile_u32(p.sync + kSyncAbort) != 0u || globaltimer() - t0 > kWaitLimitNs)) {
          ok = 0u;
          raise_abort(p);
          break;
        }
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0u;
}

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// RoPE at position pos on a d-vector held stride-32 (lane owns l + 32 m);
// angles pos * inv_freq[i] are formed and reduced modulo 2 pi in FP64.
template <int NPL>
__device__ __forceinline__ void warp_rope(float (&v)[NPL], int pos, const double* inv_freq) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < NPL / 2; ++m) {
    const int i = lane + 32 * m;
    const double ang = (double)pos * inv_freq[i];
    const double r = fma(-6.283185307179586476925, rint(ang * 0.15915494309189533577), ang);
    float sn, cs;
    sincosf((float)r, &sn, &cs);
    const float x1 = v[m], x2 = v[m + NPL / 2];
    v[m] = x1 * cs - x2 * sn;
    v[m + NPL / 2] = x2 * cs + x1 * sn;
  }
}

// Encodes 8 consecutive inputs 8 ch .. 8 ch + 7 of one row into the operand
// layout (op_slot) and returns their contribution to the group offset S.
__device__ __forceinline__ float encode_chunk8(const float (&v)[8], int ch, __half* row) {
  const bool high = (ch & 1) != 0;
  const int base = (ch >> 1) * 16 + (high ? 2 : 0);
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float s0, s1;
    const __half h0 = op_encode(v[2 * i], 8 * ch + 2 * i, s0);
    const __half h1 = op_encode(v[2 * i + 1], 8 * ch + 2 * i + 1, s1);
    *reinterpret_cast<__half2*>(row + base + 4 * i) = __halves2half2(h0, h1);
    s += s0 + s1;
  }
  return s;
}

// Sum over the 16 consecutive lanes that hold one 128-input group.
__device__ __forceinline__ float group16_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Walks a CTA's unit range stage by stage (set, first group, group count) with
// no divisions in the loop; every warp role runs the same walk.
struct StageWalk {
  int u, u1, set, kg, ng, NKG, cap;
  __device__ __forceinline__ StageWalk(const GemvPlan& pl, int u0, int u1_) {
    u = u0;
    u1 = u1_;
    NKG = pl.NKG;
    cap = pl.ng;
    set = u0 / NKG;
    kg = u0 - set * NKG;
    ng = min(min(cap, NKG - kg), u1 - u);
  }
  __device__ __forceinline__ bool valid() const { return u < u1; }
  // true if the stage just finished ends this CTA's piece of its set
  __device__ __forceinline__ bool piece_end() const { return u + ng >= u1 || kg + ng == NKG; }
  __device__ __forceinline__ void next() {
    u += ng;
    kg += ng;
    if (kg == NKG) {
      kg = 0;
      ++set;
    }
    ng = min(min(cap, NKG - kg), u1 - u);
  }
};

// Attention piece i (see Ctrl): request b, KV head h, piece j of np, tiles [ta, tb).
struct Piece {
  int b, h, j, np, ta, tb;
};
__device__ __forceinline__ Piece att_piece(const Ctrl* ctl, int i, int nkv) {
  Piece r;
  int b = 0;
  while (ctl->pb[b + 1] <= i) ++b;
  const int np = ctl->np[b], local = i - ctl->pb[b];
  r.b = b;
  r.h = local / np;
  r.j = local - r.h * np;
  r.np = np;
  r.ta = r.j * ctl->sz[b];
  r.tb = min(ctl->nt[b], r.ta + ctl->sz[b]);
  return r;
}

// ------------------------------------------------------------------ P0
// Worker warps gw of TW: input rows -> operand, offsets, sums of squares;
// this call's accumulators and tickets cleared.
__device__ void prep_phase(const BlockParams& p, int gw, int TW, bool& bad) {
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const int nkg = p.H / kWGroup;
  const int items = p.B * nkg;
  for (int base = 2 * gw; base < items; base += 2 * TW) {
    const int it = base + (lane >> 4);
    const bool ok = it < items;
    const int b = ok ? it / nkg : 0, kg = ok ? it - b * nkg : 0;
    const int ch = kg * 16 + hl;  // chunk of 8 inputs
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    if (ok) {
      if (p.act_dtype == FT_F32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x_in) + (size_t)b * p.H) + 2 * ch;
        const float4 a = __ldcg(src), d = __ldcg(src + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = d.x; v[5] = d.y; v[6] = d.z; v[7] = d.w;
      } else {
        const uint4 a = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x_in) + (size_t)b * p.H) + ch);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[2 * k] = __uint_as_float(w[k] << 16);
          v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
      }
    }
    float ss = 0.0f, sterm = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      ss = fmaf(v[i], v[i], ss);
      bad |= !(fabsf(v[i]) <= 65504.0f);
    }
    if (ok) sterm = encode_chunk8(v, ch, p.x_h + (size_t)b * p.H);
    const float gs = group16_sum(sterm), gss = group16_sum(ss);
    if (ok && hl == 0) {
      p.s_x[kg * 32 + b] = gs;
      p.ss1[kg * 32 + b] = gss;
    }
  }
  const int tid = gw * 32 + lane, nth = TW * 32;
  for (int i = tid; i < p.B * p.nqkv; i += nth) p.qkv[i] = 0.0f;
  const int nso = p.nq * p.D / kWGroup * 32, nsh = p.H / kWGroup * 32, nsa = p.I / kWGroup * 32;
  for (int i = tid; i < nso; i += nth) p.s_o[i] = 0.0f;
  for (int i = tid; i < nsh; i += nth) p.s_h1[i] = 0.0f;
  for (int i = tid; i < nsa; i += nth) p.s_a[i] = 0.0f;
  if (tid < 32) p.ss2[tid] = 0.0f;
  for (int i = tid; i < p.B * p.nkv; i += nth) p.att_tick[i] = 0u;
}

// ------------------------------------------------------------------ GEMV epilogues
// One (row tile T, column tile j) of fully reduced values:
// v[0] = (row g, token t0), v[1] = (row g, t0+1), v[2] = (row g+8, t0), v[3] = (row g+8, t0+1).
// QKV: red.add into the accumulators (split-K).  O (whole sets): h1 = x + v,
// kept, written as the gate/up operand with its group offsets and the sums of
// h1^2, and copied into the down accumulator.  Gate/up (whole sets): SwiGLU
// with rho2, written as the down operand with its offsets.  Down: red.add into
// the output accumulator, or the final value when the piece is the whole row
// (FP32 output).
template <int ROLE>
__device__ __forceinline__ void gemv_epi(const BlockParams& p, const GemvPlan& pl, const Ctrl* ctl, int T, int j,
                                         const float (&v)[4], bool whole, bool& bad) {
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const int N = pl.N;
  const int r0 = T * kRowTile + g, r1 = r0 + 8;
  if constexpr (ROLE == kRoleGU) {
    const int inter = N / 2;
    const int kcol = 8 * T + g;  // the column produced by packed rows g (gate) and g + 8 (up)
    const int grp = kcol / kWGroup;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 8 * j + 2 * tig + e;
      float st = 0.0f;
      if (t < p.B) {
        const float rho2 = ctl->rho2[t];
        const float gv = rho2 * v[e], uv = rho2 * v[2 + e];
        // silu(g) = g / (1 + e^-g); below -80 it is 0 to FP32 precision of the product
        const float sg = (gv < -80.0f) ? 0.0f : __fdividef(gv, 1.0f + __expf(-gv));
        const float a = sg * uv;
        bad |= !(fabsf(a) <= 65504.0f);
        p.a_h[(size_t)t * inter + op_slot(kcol)] = op_encode(a, kcol, st);
      }
      st += __shfl_xor_sync(0xffffffffu, st, 4);
      st += __shfl_xor_sync(0xffffffffu, st, 8);
      st += __shfl_xor_sync(0xffffffffu, st, 16);
      if (g == 0 && t < p.B) atomicAdd(p.s_a + grp * 32 + t, st);
    }
  } else if constexpr (ROLE == kRoleO) {
    const int grp = (T * kRowTile) / kWGroup;  // all 16 rows of the tile lie in one group
    float sh[2] = {0.0f, 0.0f}, sq[2] = {0.0f, 0.0f};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 8 * j + 2 * tig + (r & 1);
      if (t >= p.B) continue;
      const int row = (r & 2) ? r1 : r0;
      const size_t idx = (size_t)t * N + row;
      const float x = (p.act_dtype == FT_F32) ? __ldcg(static_cast<const float*>(p.x_in) + idx)
                                              : bf16_bits_to_f32(__ldcg(static_cast<const uint16_t*>(p.x_in) + idx));
      const float h = x + v[r];
      bad |= !(fabsf(h) <= 65504.0f);
      p.h1[idx] = h;
      p.out_acc[idx] = h;
      float st;
      p.h1_h[(size_t)t * N + op_slot(row)] = op_encode(h, row, st);
      sh[r & 1] += st;
      sq[r & 1] = fmaf(h, h, sq[r & 1]);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        sh[e] += __shfl_xor_sync(0xffffffffu, sh[e], o);
        sq[e] += __shfl_xor_sync(0xffffffffu, sq[e], o);
      }
      const int t = 8 * j + 2 * tig + e;
      if (g == 0 && t < p.B) {
        atomicAdd(p.s_h1 + grp * 32 + t, sh[e]);
        atomicAdd(p.ss2 + t, sq[e]);
      }
    }
  } else {
    float* out = (ROLE == kRoleQKV) ? p.qkv : p.out_acc;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int t = 8 * j + 2 * tig + (r & 1);
      if (t >= p.B) continue;
      const int row = (r & 2) ? r1 : r0;
      float* acc = out + (size_t)t * N + row;
      if (ROLE == kRoleDown && whole && p.act_dtype == FT_F32)
        static_cast<float*>(p.x_out)[(size_t)t * N + row] = __ldcg(acc) + v[r];
      else
        atomicAdd(acc, v[r]);
    }
  }
}

__device__ __noinline__ void piece_epilogue(const BlockParams& p, int role, const Ctrl* ctl, int T, int j,
                                            const float* vv, bool whole, bool& bad) {
  const float v[4] = {vv[0], vv[1], vv[2], vv[3]};
  const GemvPlan& pl = p.g[role];
  switch (role) {
    case kRoleQKV: gemv_epi<kRoleQKV>(p, pl, ctl, T, j, v, whole, bad); break;
    case kRoleO: gemv_epi<kRoleO>(p, pl, ctl, T, j, v, whole, bad); break;
    case kRoleGU: gemv_epi<kRoleGU>(p, pl, ctl, T, j, v, whole, bad); break;
    default: gemv_epi<kRoleDown>(p, pl, ctl, T, j, v, whole, bad); break;
  }
}

// ------------------------------------------------------------------ GEMV consumer
// NCW warps split each stage's groups; RT row tiles x NT column tiles of MMA
// chains per warp.  At the end of this CTA's piece of a row set the warps
// leave their partial sums in shared memory, then reduce them together (warp
// w takes tiles w, w + NCW, ...) and apply the role epilogue.  After a wait
// fails every warp still walks the same pieces, so the named barriers match.
// Every projection has a multiple of 64 output rows (hidden, inter, n_q d and
// (n_q + 2 n_kv) d are multiples of 128), so every set has RT full tiles.
template <int NT>
__device__ bool gemv_consume(const BlockParams& p, int role, int cta, const Ctrl* ctl, const uint8_t* ring,
                             const uint8_t* zero_row, uint32_t full0, uint32_t empty0, float* red, int& slot,
                             uint32_t& fphase, bool ok, bool& bad) {
  constexpr int RT = GemvShape<NT>::RT, NCW = GemvShape<NT>::NCW;
  const GemvPlan& pl = p.g[role];
  if (cta >= pl.C) return ok;
  const int u0 = plan_u0(pl, cta), u1 = plan_u0(pl, cta + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  float tot[RT][NT][4];
#pragma unroll
  for (int a = 0; a < RT; ++a)
#pragma unroll
    for (int b = 0; b < NT; ++b)
#pragma unroll
      for (int r = 0; r < 4; ++r) tot[a][b][r] = 0.0f;

  int piece_kg0 = -1;
  for (StageWalk st(pl, u0, u1); st.valid(); st.next()) {
    if (piece_kg0 < 0) piece_kg0 = st.kg;
    if (ok) ok = warp_wait(p, full0 + 8 * slot, fphase);
    if (ok) {
      const uint8_t* sw = ring + (size_t)slot * p.stride;
      const float* ss = reinterpret_cast<const float*>(sw + pl.soff);
      for (int kgl = warp; kgl < st.ng; kgl += NCW) {
        // activation rows of this lane's B fragments; tokens >= B read zeros
        const uint8_t* xr[NT];
        float c0[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int row = 8 * j + g, t = 8 * j + 2 * tig;
          xr[j] = (row < p.B ? sw + pl.xoff + row * pl.xstride : zero_row) + (kgl * kWGroup + 4 * tig) * 2;
          const float2 sv = *reinterpret_cast<const float2*>(ss + kgl * 32 + t);
          c0[j][0] = (t < p.B) ? -sv.x : 0.0f;
          c0[j][1] = (t + 1 < p.B) ? -sv.y : 0.0f;
        }
        const uint8_t* slab0 = sw + kgl * kSlabBytes;
        // k-steps 0-3 and 4-7 of the group run as two independent MMA chains
        // (the second starts at 0) where registers allow, halving the chain depth
        constexpr bool kTwoChains = NT <= 2;
        uint32_t sc[RT];
        float acc[RT][NT][4];
        float acc2[kTwoChains ? RT : 1][kTwoChains ? NT : 1][4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t wd[RT][4];
#pragma unroll
          for (int rt = 0; rt < RT; ++rt) {
            const uint8_t* slab = slab0 + rt * pl.ng * kSlabBytes;
            const uint4 q = *reinterpret_cast<const uint4*>(slab + half * 512 + lane * 16);
            wd[rt][0] = q.x; wd[rt][1] = q.y; wd[rt][2] = q.z; wd[rt][3] = q.w;
            if (half == 0) sc[rt] = *reinterpret_cast<const uint32_t*>(slab + kSlabCodes + 4 * g);
          }
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int ks = 4 * half + kq;
            uint32_t b0[NT], b1[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              const uint2 bv = *reinterpret_cast<const uint2*>(xr[j] + ks * 32);
              b0[j] = bv.x;
              b1[j] = bv.y;
            }
#pragma unroll
            for (int rt = 0; rt < RT; ++rt) {
              uint32_t r[4];
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
    }
    if (++slot == p.stages) {
      slot = 0;
      fphase ^= 1u;
    }

    if (st.piece_end()) {
      const bool whole = (piece_kg0 == 0) && (st.kg + st.ng == pl.NKG);
      piece_kg0 = -1;
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            red[(((warp * RT + rt) * NT + j) * 4 + r) * 32 + lane] = tot[rt][j][r];
            tot[rt][j][r] = 0.0f;
          }
      named_bar(1, NCW * 32);
      if (ok) {
        for (int q = warp; q < RT * NT; q += NCW) {
          const int rt = q / NT, j = q - (q / NT) * NT;
          float v[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float a = 0.0f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) a += red[((w * RT * NT + q) * 4 + r) * 32 + lane];
            v[r] = a;
          }
          piece_epilogue(p, role, ctl, st.set * RT + rt, j, v, whole, bad);
        }
      }
      named_bar(1, NCW * 32);
    }
  }
  return ok;
}

// After down with a BF16 output: every CTA converts its share of the output
// accumulator (all pieces added, grid barrier G5).
__device__ __noinline__ void convert_out(const BlockParams& p, int cta, int tid, int nth) {
  const int n = p.B * p.H;
  const int per = (n + p.C - 1) / p.C;
  const int i0 = cta * per, i1 = min(n, i0 + per);
  for (int i = i0 + tid; i < i1; i += nth)
    static_cast<uint16_t*>(p.x_out)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(__ldcg(p.out_acc + i)));
}

// ------------------------------------------------------------------ attention
struct AttSmem {
  float* qt;     // [kAttMaxG][D] rotated, scaled query (FP16 values)
  float* qoff;   // [kAttMaxG] its operand offsets (magic-number decode)
  float* knew;   // [D] decoded new K (rotated)
  float* vnew;   // [D]
  uint8_t* codes;  // [2][D] staging for the new entry's codes
  const double* inv_freq;  // [d/2] RoPE frequencies (shared-memory copy of the parameter)
  float* mrg;    // [NCW][16 + G D] per-warp partials
};

// One 16-position tile of a staged run: K codes as A of S = K q~, online
// softmax (exp2 domain), V codes as A of O += V^T (P s_v).
template <int D>
__device__ __forceinline__ void att_tile(const uint8_t* st, int npos, int i, int p0, int Lb,
                                         const uint32_t (&bq)[D / 16][2], float qo0, float qo1,
                                         float (&acc)[D / 16][4], float (&kacc)[4], float& m0, float& m1, float& l0,
                                         float& l1) {
  constexpr int E = D / 2, KT = D / 16;
  const int lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
  const uint8_t* Kp = st;
  const uint8_t* Vp = st + npos * E;
  const uint16_t* Ks = reinterpret_cast<const uint16_t*>(st + 2 * npos * E);
  const uint16_t* Vs = Ks + npos;
  const int r = 16 * i;
  uint32_t kw[2][D / 32];
  uint32_t vw[4][(D / 64) > 0 ? D / 64 : 1];
  if constexpr (D == 128) {
    const uint4 a = *reinterpret_cast<const uint4*>(Kp + (r + g) * E + tig * 16);
    const uint4 c = *reinterpret_cast<const uint4*>(Kp + (r + g + 8) * E + tig * 16);
    kw[0][0] = a.x; kw[0][1] = a.y; kw[0][2] = a.z; kw[0][3] = a.w;
    kw[1][0] = c.x; kw[1][1] = c.y; kw[1][2] = c.z; kw[1][3] = c.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(Kp + (r + g) * E + tig * 8);
    const uint2 c = *reinterpret_cast<const uint2*>(Kp + (r + g + 8) * E + tig * 8);
    kw[0][0] = a.x; kw[0][1] = a.y;
    kw[1][0] = c.x; kw[1][1] = c.y;
  }
  const int pv[4] = {r + 2 * tig, r + 2 * tig + 1, r + 2 * tig + 8, r + 2 * tig + 9};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr (D == 128) {
      const uint2 a = *reinterpret_cast<const uint2*>(Vp + pv[q] * E + g * 8);
      vw[q][0] = a.x;
      vw[q][1] = a.y;
    } else {
      vw[q][0] = *reinterpret_cast<const uint32_t*>(Vp + pv[q] * E + g * 4);
    }
  }
  // S = K . q~   (rows: positions g, g+8; columns: heads 2tig, 2tig+1)
  float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int j = 0; j < D / 32; ++j) {
    uint32_t dg[4], dg8[4];
    magic_word(kw[0][j], dg);
    magic_word(kw[1][j], dg8);
    const uint32_t a0[4] = {dg[0], dg8[0], dg[1], dg8[1]};
    const uint32_t a1[4] = {dg[2], dg8[2], dg[3], dg8[3]};
    mma_f16(sacc, a0, bq[2 * j][0], bq[2 * j][1]);
    mma_f16(sacc, a1, bq[2 * j + 1][0], bq[2 * j + 1][1]);
  }
  const bool va = (p0 + g) < Lb, vb = (p0 + g + 8) < Lb;
  const float ks0 = bf16_bits_to_f32(Ks[r + g]), ks1 = bf16_bits_to_f32(Ks[r + g + 8]);
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
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  // an all-masked tile before any valid one keeps m = -inf: use 0 for the rescale
  const float al0 = (mn0 == -INFINITY) ? 1.0f : exp2f(m0 - mn0);
  const float al1 = (mn1 == -INFINITY) ? 1.0f : exp2f(m1 - mn1);
  m0 = mn0;
  m1 = mn1;
  const float e0 = va ? exp2f(s0 - mn0) : 0.0f, e1 = va ? exp2f(s1 - mn1) : 0.0f;
  const float e2 = vb ? exp2f(s2 - mn0) : 0.0f, e3 = vb ? exp2f(s3 - mn1) : 0.0f;
  l0 = l0 * al0 + e0 + e2;
  l1 = l1 * al1 + e1 + e3;
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
  const float vs0 = va ? bf16_bits_to_f32(Vs[r + g]) : 0.0f;
  const float vs1 = vb ? bf16_bits_to_f32(Vs[r + g + 8]) * 0.0625f : 0.0f;  // positions 8..15: operand / 16
  const uint32_t P0 = pack_half2(e0 * vs0, e1 * vs0);  // position g,   heads 2tig, 2tig+1
  const uint32_t P1 = pack_half2(e2 * vs1, e3 * vs1);  // position g+8
  const uint32_t pb0 = movmatrix_trans(P0);            // positions 2tig, 2tig+1 of head g
  const uint32_t pb1 = movmatrix_trans(P1);            // positions 2tig+8, 2tig+9
  const uint32_t kappa[4] = {kHOffLo, kHOffLo, kHOffHi, kHOffHi};
  // O += V^T . P  (positions 2tig, 2tig+1 decode at 1024 + c, positions +8 at 1024 + 16 c)
#pragma unroll
  for (int j = 0; j < (D / 64 > 0 ? D / 64 : 1); ++j) {
    uint32_t lo01[4], hi01[4], lo23[4], hi23[4];
    magic_low4(prmt(vw[0][j], vw[1][j], 0x5410u), lo01);
    magic_low4(prmt(vw[0][j], vw[1][j], 0x7632u), hi01);
    magic_high4(prmt(vw[2][j], vw[3][j], 0x5410u), lo23);
    magic_high4(prmt(vw[2][j], vw[3][j], 0x7632u), hi23);
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
}

// The vectors of pair (b, h) the attention needs, one per warp task: task
// hh < G is the rotated query of head hh (rho1, RoPE, rotation, softmax scale,
// rounded to the FP16 operand, with its decode offset for the K codes);
// task G / G + 1 is the new token's K (with RoPE) / V: rho1, rotation, INT4
// quantisation, cache write at L_b, and the decoded values kept so the token
// attends to its own INT4 entry.
template <int D>
__device__ __noinline__ void att_prepare(const BlockParams& p, const AttSmem& sm, int task, int b, int h, int Lb,
                                         float rho1) {
  constexpr int NPL = D / 32;
  const int lane = threadIdx.x & 31;
  const bool isq = task < p.G;
  const int off = isq ? (h * p.G + task) * D : (task == p.G ? (p.nq + h) * D : (p.nq + p.nkv + h) * D);
  const float* src = p.qkv + (size_t)b * p.nqkv + off;
  float v[NPL];
#pragma unroll
  for (int m = 0; m < NPL; ++m) v[m] = __ldcg(src + lane + 32 * m) * rho1;
  if (task <= p.G) warp_rope<NPL>(v, Lb, sm.inv_freq);
  warp_fwht<NPL>(v, p.hb, p.hscale);
  if (isq) {
    // channels c % 16 >= 8 enter the B operand as q / 16
    float sq = 0.0f;
#pragma unroll
    for (int m = 0; m < NPL; ++m) {
      const int c = lane + 32 * m;
      const float qv = __half2float(__float2half_rn(v[m] * p.qscale));
      sm.qt[task * D + c] = qv;
      float st;
      (void)op_encode(qv, c, st);
      sq += st;
    }
    sq = warp_sum(sq);
    if (lane == 0) sm.qoff[task] = sq;
  } else {
    const int which = task - p.G;
    const size_t row = p.L.row(b, h, Lb);
    uint8_t* entry = p.cache + (which == 0 ? p.L.kc : p.L.vc) + row * p.L.entry;
    uint16_t* sc = reinterpret_cast<uint16_t*>(p.cache + (which == 0 ? p.L.ks : p.L.vs)) + row;
    warp_quant_store<NPL>(v, which == 0, sm.codes + which * D, entry, sc);
    float* dst = (which == 0) ? sm.knew : sm.vnew;
#pragma unroll
    for (int m = 0; m < NPL; ++m) dst[lane + 32 * m] = v[m];
  }
}

// Normalised output of one query head -> inverse rotation -> O operand and
// its group offset.
template <int D>
__device__ __noinline__ void att_emit(const BlockParams& p, float* o, float l, int b, int h, int hh, bool& bad) {
  constexpr int NPL = D / 32;
  const int lane = threadIdx.x & 31;
  const float inv = 1.0f / l;
  float v[NPL];
#pragma unroll
  for (int m = 0; m < NPL; ++m) v[m] = o[m] * inv;
  warp_fwht<NPL>(v, p.hb, p.hscale);
  const int kbase = (h * p.G + hh) * D;  // input index of channel 0 of this head in the O projection
  __half* dst = p.o_h + (size_t)b * p.nq * D;
  float so = 0.0f;
#pragma unroll
  for (int m = 0; m < NPL; ++m) {
    const int k = kbase + lane + 32 * m;
    bad |= !(fabsf(v[m]) <= 65504.0f);
    float st;
    dst[op_slot(k)] = op_encode(v[m], k, st);
    so += st;
  }
  so = warp_sum(so);  // a head (d <= 128 channels) lies inside one 128-input group
  if (lane == 0) atomicAdd(p.s_o + (kbase / kWGroup) * 32 + b, so);
}

// Merge of the np partials of pair (b, h) (pieces i0 .. i0 + np - 1) for
// query head hh, one pass with a running maximum; then emit.
template <int D>
__device__ __noinline__ void att_merge_head(const BlockParams& p, int i0, int np, int b, int h, int hh, bool& bad) {
  constexpr int NPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int PS = 16 + p.G * D;
  float M = -INFINITY, l = 0.0f, o[NPL];
#pragma unroll
  for (int m = 0; m < NPL; ++m) o[m] = 0.0f;
#pragma unroll 4
  for (int j = 0; j < np; ++j) {
    const float* pj = p.part + (size_t)(i0 + j) * PS;
    const float mj = __ldcg(pj + hh), lj = __ldcg(pj + 8 + hh);
    float oj[NPL];
#pragma unroll
    for (int m = 0; m < NPL; ++m) oj[m] = __ldcg(pj + 16 + hh * D + lane + 32 * m);
    const float Mn = fmaxf(M, mj);
    if (Mn == -INFINITY) continue;
    const float a = (M == -INFINITY) ? 0.0f : exp2f(M - Mn);
    const float e = (mj == -INFINITY) ? 0.0f : exp2f(mj - Mn);
    l = l * a + lj * e;
#pragma unroll
    for (int m = 0; m < NPL; ++m) o[m] = o[m] * a + oj[m] * e;
    M = Mn;
  }
  att_emit<D>(p, o, l, b, h, hh, bad);
}

// P2 on the consumer warps: this CTA's pieces (i = cta, cta + C, ...), in ring
// stages of up to tps tiles.  A pair's last piece (whose last tile contains
// position L_b) takes the new token: it writes the token's cache entry and
// folds the token into its result.  A pair of one piece is finished here;
// otherwise each piece leaves a partial (max, sum, output) in global memory
// and the last piece to finish (atomic ticket) merges them.
template <int D, int NCW>
__device__ __noinline__ bool att_consume(const BlockParams& p, int cta, Ctrl* ctl, const AttSmem& sm,
                                         const uint8_t* ring, uint32_t full0, uint32_t empty0, int& slot,
                                         uint32_t& fphase, bool& bad) {
  constexpr int NPL = D / 32, KT = D / 16;
  constexpr int CT = NCW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int G = p.G, PS = 16 + G * D;
  bool ok = true;
  for (int i = cta; i < ctl->P; i += p.C) {
    const Piece pc = att_piece(ctl, i, p.nkv);
    const int b = pc.b, h = pc.h;
    const int q = b * p.nkv + h;
    const int Lb = ctl->lb[b];
    const float rho1 = ctl->rho1[b];
    const bool last_piece = (pc.j == pc.np - 1);

    // ---- rotated queries of the G heads (and the new token, last piece)
    named_bar(1, CT);
    const int ntask = G + (last_piece ? 2 : 0);
    for (int task = warp; task < ntask; task += NCW) att_prepare<D>(p, sm, task, b, h, Lb, rho1);
    named_bar(1, CT);
    uint32_t bq[KT][2];
#pragma unroll
    for (int kt = 0; kt < KT; ++kt) {
      if (g < G) {
        const int c = 16 * kt + 2 * tig;
        bq[kt][0] = pack_half2(sm.qt[g * D + c], sm.qt[g * D + c + 1]);
        bq[kt][1] = pack_half2(sm.qt[g * D + c + 8] * 0.0625f, sm.qt[g * D + c + 9] * 0.0625f);
      } else {
        bq[kt][0] = bq[kt][1] = 0u;
      }
    }
    const float qo0 = (2 * tig < G) ? sm.qoff[2 * tig] : 0.0f;
    const float qo1 = (2 * tig + 1 < G) ? sm.qoff[2 * tig + 1] : 0.0f;

    float acc[KT][4];
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    float kacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;

    for (int s0 = pc.ta; s0 < pc.tb; s0 += p.tps) {
      const int n = min(p.tps, pc.tb - s0);
      if (ok && !warp_wait(p, full0 + 8 * slot, fphase)) ok = false;
      if (ok) {
        const uint8_t* st = ring + (size_t)slot * p.stride;
        for (int it = warp; it < n; it += NCW)
          att_tile<D>(st, 16 * n, it, 16 * (s0 + it), Lb, bq, qo0, qo1, acc, kacc, m0, m1, l0, l1);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      }
      if (++slot == p.stages) {
        slot = 0;
        fphase ^= 1u;
      }
    }

    // ---- this warp's partial: remove the decode offsets, sum over the rows
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      acc[mt][0] -= kacc[0];
      acc[mt][1] -= kacc[1];
      acc[mt][2] -= kacc[0];
      acc[mt][3] -= kacc[1];
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    float* mw = sm.mrg + warp * PS;
    const bool h0 = 2 * tig < G, h1v = 2 * tig + 1 < G;
    if (g == 0) {
      if (h0) {
        mw[2 * tig] = m0;
        mw[8 + 2 * tig] = l0;
      }
      if (h1v) {
        mw[2 * tig + 1] = m1;
        mw[8 + 2 * tig + 1] = l1;
      }
    }
#pragma unroll
    for (int mt = 0; mt < KT; ++mt) {
      const int c0 = 16 * mt + g, c1 = c0 + 8;
      if (h0) {
        mw[16 + (2 * tig) * D + c0] = acc[mt][0];
        mw[16 + (2 * tig) * D + c1] = acc[mt][2];
      }
      if (h1v) {
        mw[16 + (2 * tig + 1) * D + c0] = acc[mt][1];
        mw[16 + (2 * tig + 1) * D + c1] = acc[mt][3];
      }
    }
    named_bar(1, CT);

    // ---- the piece's result per head (warp hh): merge of the warps (+ the new token)
    const bool single = (pc.np == 1);
    for (int hh = warp; hh < G; hh += NCW) {
      float sn = -INFINITY;
      if (last_piece) {
        float d = 0.0f;
#pragma unroll
        for (int m = 0; m < NPL; ++m) d += sm.qt[hh * D + lane + 32 * m] * sm.knew[lane + 32 * m];
        sn = warp_sum(d);
      }
      float M = sn;
      for (int w = 0; w < NCW; ++w) M = fmaxf(M, sm.mrg[w * PS + hh]);
      float o[NPL], l;
      const float wn = last_piece ? exp2f(sn - M) : 0.0f;
#pragma unroll
      for (int m = 0; m < NPL; ++m) o[m] = last_piece ? wn * sm.vnew[lane + 32 * m] : 0.0f;
      l = wn;
      for (int w = 0; w < NCW; ++w) {
        const float mw2 = sm.mrg[w * PS + hh];
        if (mw2 == -INFINITY) continue;
        const float e = exp2f(mw2 - M);
        l = fmaf(e, sm.mrg[w * PS + 8 + hh], l);
#pragma unroll
        for (int m = 0; m < NPL; ++m) o[m] = fmaf(e, sm.mrg[w * PS + 16 + hh * D + lane + 32 * m], o[m]);
      }
      if (single) {
        att_emit<D>(p, o, l, b, h, hh, bad);
      } else {
        float* dstp = p.part + (size_t)i * PS;
        if (lane == 0) {
          dstp[hh] = M;
          dstp[8 + hh] = l;
        }
#pragma unroll
        for (int m = 0; m < NPL; ++m) dstp[16 + hh * D + lane + 32 * m] = o[m];
      }
    }
    if (!single) {
      __threadfence();
      named_bar(1, CT);
      if (tid == 0) ctl->flag = (atomicAdd(p.att_tick + q, 1u) == (uint32_t)(pc.np - 1)) ? 1 : 0;
      named_bar(1, CT);
      if (ctl->flag) {
        __threadfence();
        const int i0 = i - pc.j;
        for (int hh = warp; hh < G; hh += NCW) att_merge_head<D>(p, i0, pc.np, b, h, hh, bad);
      }
    }
  }
  return ok;
}

// ------------------------------------------------------------------ producer
// Ring cursor and the queue of armed GEMV stages whose activation copy waits
// for a grid barrier (entry e lives in lane e % 32 of the producer warp).
struct Prod {
  int slot, round, issued;
  int qh, qt;
  int r_role, r_kg, r_ng, r_slot;
  uint32_t passed;  // bit k: grid barrier k known complete
};

// the grid barrier that publishes a role's activation operand
__device__ __forceinline__ int act_barrier(int role) {
  return role == kRoleQKV ? 0 : role == kRoleO ? 2 : role == kRoleGU ? 3 : 4;
}

// Issues the queued activation copies whose barrier is known complete (all of
// them when `force`).  Every lane acquired the barrier counter itself, and a
// proxy fence orders that view before the bulk copies.
__device__ __noinline__ void prod_service(const BlockParams& p, Prod& ps, uint8_t* ring, uint32_t full0, bool force) {
  const int lane = threadIdx.x & 31;
  bool fenced = false;
  while (ps.qh < ps.qt) {
    const int e = ps.qh & 31;
    const int role = __shfl_sync(0xffffffffu, ps.r_role, e);
    const int kg = __shfl_sync(0xffffffffu, ps.r_kg, e);
    const int ng = __shfl_sync(0xffffffffu, ps.r_ng, e);
    const int sl = __shfl_sync(0xffffffffu, ps.r_slot, e);
    if (!force && !(ps.passed & (1u << act_barrier(role)))) break;
    if (!fenced) {
      fence_proxy_async_global();
      fenced = true;
    }
    const GemvPlan& pl = p.g[role];
    const __half* x = role == kRoleQKV ? p.x_h : role == kRoleO ? p.o_h : role == kRoleGU ? p.h1_h : p.a_h;
    const float* sv = role == kRoleQKV ? p.s_x : role == kRoleO ? p.s_o : role == kRoleGU ? p.s_h1 : p.s_a;
    const uint32_t sb = smem_u32(ring + (size_t)sl * p.stride);
    const uint32_t bar = full0 + 8 * sl;
    if (lane < p.B)
      bulk_g2s(sb + pl.xoff + lane * pl.xstride, x + (size_t)lane * pl.K + (size_t)kg * kWGroup, ng * kWGroup * 2, bar);
    if (lane == 31) bulk_g2s(sb + pl.soff, sv + (size_t)kg * 32, ng * 128, bar);
    ++ps.qh;
  }
}

// Acquires the barrier of the head of the queue, if any.
__device__ __forceinline__ void prod_refresh(const BlockParams& p, Prod& ps) {
  if (ps.qh >= ps.qt) return;
  const int k = act_barrier(__shfl_sync(0xffffffffu, ps.r_role, ps.qh & 31));
  uint32_t v = ld_acquire_u32(p.sync + k);
  v = __shfl_sync(0xffffffffu, v, 0);
  if (v >= (uint32_t)p.C) ps.passed |= 1u << k;
}

__device__ __noinline__ bool prod_give_up(const BlockParams& p, unsigned long long t0) {
  int stop = 0;
  if ((threadIdx.x & 31) == 0)
    stop = (ld_volatile_u32(p.sync + kSyncAbort) != 0u || globaltimer() - t0 > kWaitLimitNs) ? 1 : 0;
  return __shfl_sync(0xffffffffu, stop, 0) != 0;
}

// Waits until the next slot is free, issuing queued activation copies as their
// barriers complete; false on timeout or abort.
__device__ __noinline__ bool prod_acquire(const BlockParams& p, Prod& ps, uint8_t* ring, uint32_t full0,
                                          uint32_t empty0) {
  if (ps.round == 0) return true;
  const uint32_t bar = empty0 + 8 * ps.slot, par = (uint32_t)(ps.round - 1) & 1u;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ps.qh < ps.qt) {
      if (__shfl_sync(0xffffffffu, mbar_test(bar, par) ? 1 : 0, 0)) return true;
      prod_refresh(p, ps);
      prod_service(p, ps, ring, full0, false);
    } else if (__shfl_sync(0xffffffffu, mbar_try_wait(bar, par) ? 1 : 0, 0)) {
      return true;
    }
    if ((it & 15u) == 0 && prod_give_up(p, t0)) return false;
  }
}

__device__ __forceinline__ void prod_advance(const BlockParams& p, Prod& ps) {
  ++ps.issued;
  if (++ps.slot == p.stages) {
    ps.slot = 0;
    ++ps.round;
  }
}

// Streams this CTA's stages in order: QKV | attention tiles | O | gate/up | down.
template <int D>
__device__ void producer(const BlockParams& p, int cta, const Ctrl* ctl, uint8_t* ring, uint32_t full0,
                         uint32_t empty0) {
  constexpr int E = D / 2;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  Prod ps = {};
  bool ok = true;
#pragma unroll 1
  for (int ph = 0; ph < 5 && ok; ++ph) {
    if (ph == 1) {
      // attention: the tile runs of this CTA's pieces, no activation
      for (int i = cta; ok && i < ctl->P; i += p.C) {
        const Piece pc = att_piece(ctl, i, p.nkv);
        const int b = pc.b, h = pc.h;
        for (int s0 = pc.ta; s0 < pc.tb; s0 += p.tps) {
          const int npos = 16 * min(p.tps, pc.tb - s0);
          if (!prod_acquire(p, ps, ring, full0, empty0)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = full0 + 8 * ps.slot;
            mbar_arrive_expect_tx(bar, (uint32_t)(npos * (2 * E + 4)));
            const uint32_t sb = smem_u32(ring + (size_t)ps.slot * p.stride);
            const size_t row = p.L.row(b, h, 16 * s0);
            bulk_g2s(sb, p.cache + p.L.kc + row * E, npos * E, bar);
            bulk_g2s(sb + npos * E, p.cache + p.L.vc + row * E, npos * E, bar);
            bulk_g2s(sb + 2 * npos * E, p.cache + p.L.ks + row * 2, npos * 2, bar);
            bulk_g2s(sb + 2 * npos * E + 2 * npos, p.cache + p.L.vs + row * 2, npos * 2, bar);
          }
          __syncwarp();
          prod_advance(p, ps);
        }
      }
      continue;
    }
    const int role = ph == 0 ? kRoleQKV : ph - 1;
    const GemvPlan& pl = p.g[role];
    if (cta >= pl.C) continue;
    const int u0 = plan_u0(pl, cta), u1 = plan_u0(pl, cta + 1);
    const uint8_t* W = p.w[role];
    for (StageWalk st(pl, u0, u1); st.valid(); st.next()) {
      if (!prod_acquire(p, ps, ring, full0, empty0)) {
        ok = false;
        break;
      }
      const int nrt = min(pl.RT, pl.NTILE - st.set * pl.RT);
      if (lane == 0) {
        const uint32_t bar = full0 + 8 * ps.slot;
        mbar_arrive_expect_tx(bar, (uint32_t)(nrt * st.ng * kSlabBytes + p.B * st.ng * kWGroup * 2 + st.ng * 128));
        const uint32_t sb = smem_u32(ring + (size_t)ps.slot * p.stride);
        for (int rt = 0; rt < nrt; ++rt)
          bulk_g2s(sb + rt * pl.ng * kSlabBytes, W + ((size_t)(st.set * pl.RT + rt) * pl.NKG + st.kg) * kSlabBytes,
                   st.ng * kSlabBytes, bar);
      }
      __syncwarp();
      if (lane == (ps.qt & 31)) {
        ps.r_role = role;
        ps.r_kg = st.kg;
        ps.r_ng = st.ng;
        ps.r_slot = ps.slot;
      }
      ++ps.qt;
      if (ps.passed & (1u << act_barrier(role))) prod_service(p, ps, ring, full0, false);
      prod_advance(p, ps);
    }
  }
  if (ok) {
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1; ps.qh < ps.qt; ++it) {
      prod_refresh(p, ps);
      prod_service(p, ps, ring, full0, false);
      if ((it & 15u) == 0 && ps.qh < ps.qt && prod_give_up(p, t0)) {
        ok = false;
        break;
      }
    }
  }
  if (!ok) {
    if (lane == 0) raise_abort(p);
    prod_service(p, ps, ring, full0, true);  // every armed stage gets all its bytes
    for (int i = max(0, ps.issued - S); i < ps.issued; ++i)
      (void)mbar_wait(full0 + 8 * (i % S), (uint32_t)(i / S) & 1u);
  }
}

// ------------------------------------------------------------------ the kernel
template <int NT, int D>
__global__ void __launch_bounds__((GemvShape<NT>::NCW + 1) * 32, 1) block_kernel(const BlockParams p) {
  constexpr int NCW = GemvShape<NT>::NCW;
  constexpr int PRODUCER = NCW;
  constexpr int CT = NCW * 32;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  const int S = p.stages;
  const uint32_t full0 = smem_u32(smem), empty0 = full0 + 8 * S;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + p.ctrl_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  uint8_t* zero_row = smem + p.zero_off;  // stands in for activation rows of absent tokens
  uint8_t* ring = smem + p.ring_off;
  AttSmem sm;
  sm.qt = reinterpret_cast<float*>(smem + p.att_off);
  sm.qoff = sm.qt + kAttMaxG * D;
  sm.knew = sm.qoff + kAttMaxG;
  sm.vnew = sm.knew + D;
  sm.codes = reinterpret_cast<uint8_t*>(sm.vnew + D);
  sm.inv_freq = ctl->inv_freq;
  sm.mrg = red;  // the piece reduction area is idle during attention

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, NCW);
    }
    mbar_fence_init();
  }
  if (tid < 32) {
    int n = 0, lb = 0;
    if (tid < p.B) {
      lb = p.pos[tid];
      if (lb >= 0 && lb < p.L.max_ctx) {
        n = lb / 16 + 1;
      } else if (cta == 0) {
        set_status(p.status, FT_DEV_CAPACITY);
      }
    }
    ctl->nt[tid] = n;
    ctl->lb[tid] = lb;
    if (tid == 0) ctl->flag = 0;
  }
  if (tid >= 32 && tid < 96) ctl->inv_freq[tid - 32] = p.inv_freq[tid - 32];
  for (int i = tid; i < kZeroRowBytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(zero_row)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  if (tid == 0) {
    // piece length: at least tmin tiles, else the even share of all CTAs
    int TT = 0;
    for (int b = 0; b < 32; ++b) TT += p.nkv * ctl->nt[b];
    const int tp = max(p.tmin, (TT + p.C - 1) / p.C);
    int acc = 0;
    for (int b = 0; b < 32; ++b) {
      const int n = ctl->nt[b];
      const int np = (n + tp - 1) / tp;
      ctl->np[b] = np;
      ctl->sz[b] = np > 0 ? (n + np - 1) / np : 0;
      ctl->pb[b] = acc;
      acc += p.nkv * np;
    }
    ctl->pb[32] = acc;
    ctl->P = acc;
  }
  __syncthreads();

  // Phases, one call site each: P0 -> G0; QKV -> G1; attention -> G2; O -> G3;
  // gate/up -> G4; down -> G5 (a BF16 output is converted after G5).
  bool bad = false;
  if (warp == PRODUCER) {
    producer<D>(p, cta, ctl, ring, full0, empty0);
  } else {
    prep_phase(p, cta * NCW + warp, p.C * NCW, bad);
    named_bar(1, CT);
    if (tid == 0) grid_arrive(p, 0);
    int slot = 0;
    uint32_t fphase = 0;
    bool ok = true;
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
      if (r == kRoleGU) {
        // rho2 of every request from the sums of h1^2 (complete at G3)
        if (warp == 0) {
          if (grid_wait_warp(p, 3) && lane < p.B) ctl->rho2[lane] = rsqrtf(__ldcg(p.ss2 + lane) / (float)p.H + p.eps);
        }
        named_bar(1, CT);
      }
      ok = gemv_consume<NT>(p, r, cta, ctl, ring, zero_row, full0, empty0, red, slot, fphase, ok, bad);
      named_bar(1, CT);
      if (tid == 0) grid_arrive(p, r == kRoleQKV ? 1 : r == kRoleO ? 3 : r == kRoleGU ? 4 : 5);
      if (r == kRoleQKV) {
        // rho1 of every request from the per-group sums of x^2
        if (warp == 0) {
          if (grid_wait_warp(p, 0) && lane < p.B) {
            const int nkg = p.H / kWGroup;
            float s = 0.0f;
            for (int kg = 0; kg < nkg; ++kg) s += __ldcg(p.ss1 + kg * 32 + lane);
            const float rr = rsqrtf(s / (float)p.H + p.eps);
            ctl->rho1[lane] = rr;
            if (cta == 0) p.rho1[lane] = rr;
          }
        }
        named_bar(1, CT);
        if (ok) ok = grid_wait_warp(p, 1);
        if (!att_consume<D, NCW>(p, cta, ctl, sm, ring, full0, empty0, slot, fphase, bad)) ok = false;
        named_bar(1, CT);
        if (tid == 0) grid_arrive(p, 2);
      }
    }
    if (p.act_dtype != FT_F32 && grid_wait_warp(p, 5)) convert_out(p, cta, tid, CT);
  }
  if (bad) set_status(p.status, FT_DEV_RANGE);

  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.sync + kSyncExit, 1u) == (uint32_t)(p.C - 1)) {
      for (int k = 0; k < kNumGridBars; ++k) atomicExch(p.sync + k, 0u);
      atomicExch(p.sync + kSyncAbort, 0u);
      atomicExch(p.sync + kSyncExit, 0u);
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------ host side
GemvPlan make_gemv_plan(int N, int K, int B, int C, bool whole_sets) {
  GemvPlan p = {};
  p.N = N;
  p.K = K;
  p.NT = (B + 7) / 8;
  switch (p.NT) {
    case 1: p.RT = GemvShape<1>::RT; p.NCW = GemvShape<1>::NCW; break;
    case 2: p.RT = GemvShape<2>::RT; p.NCW = GemvShape<2>::NCW; break;
    case 3: p.RT = GemvShape<3>::RT; p.NCW = GemvShape<3>::NCW; break;
    default: p.RT = GemvShape<4>::RT; p.NCW = GemvShape<4>::NCW; break;
  }
  p.NTILE = N / kRowTile;
  p.NKG = K / kWGroup;
  p.NSET = (p.NTILE + p.RT - 1) / p.RT;
  p.whole = whole_sets ? 1 : 0;
  const int units = whole_sets ? p.NSET : p.NSET * p.NKG;
  p.C = C < units ? C : units;
  if (p.C < 1) p.C = 1;
  p.per = units / p.C;
  p.rem = units % p.C;
  p.ng = p.NCW;  // one group per consumer warp per stage
  if (p.ng > p.NKG) p.ng = p.NKG;
  p.xstride = p.ng * kWGroup * 2 + 16;
  const int wbytes = p.RT * p.ng * kSlabBytes;
  p.xoff = (int)align_up((size_t)wbytes, 16);
  p.soff = (int)align_up((size_t)p.xoff + (size_t)B * p.xstride, 16);
  p.slot = (int)align_up((size_t)p.soff + (size_t)p.ng * 128, 128);
  return p;
}

struct WsPlan {
  BlockParams bp;  // geometry part (no pointers)
  size_t x_h, s_x, ss1, rho1, qkv, part, att_tick, o_h, s_o, h1, h1_h, s_h1, ss2, a_h, s_a, out_acc;
  size_t total;
  bool ok;
};

static int grid_ctas() {
  const int sms = ft_host::num_sms();
  return sms > 0 ? sms : 148;
}

static int smem_optin() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 227 * 1024;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || v <= 0)
    return 227 * 1024;
  return v;
}

static WsPlan make_plan(const ft_block_cfg& c, int B, int max_ctx) {
  WsPlan w = {};
  BlockParams& P = w.bp;
  const int C = grid_ctas();
  P.B = B;
  P.H = c.hidden;
  P.I = c.inter;
  P.nq = c.n_q;
  P.nkv = c.n_kv;
  P.D = c.head_dim;
  P.G = c.n_q / c.n_kv;
  P.hb = c.had_block;
  P.hscale = hadamard_scale(c.had_block);
  P.nqkv = (c.n_q + 2 * c.n_kv) * c.head_dim;
  P.eps = c.rms_eps;
  P.qscale = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  P.C = C;
  P.g[kRoleQKV] = make_gemv_plan(P.nqkv, c.hidden, B, C, false);
  P.g[kRoleO] = make_gemv_plan(c.hidden, c.n_q * c.head_dim, B, C, true);
  P.g[kRoleGU] = make_gemv_plan(2 * c.inter, c.hidden, B, C, true);
  P.g[kRoleDown] = make_gemv_plan(c.hidden, c.inter, B, C, false);
  w.ok = P.G <= kAttMaxG;
  // shared memory: mbarriers | Ctrl | attention scratch | piece handoff / attention partials | ring
  const int NCW = P.g[0].NCW, RT = P.g[0].RT, NT = P.g[0].NT;
  int stride = 0;
  for (int r = 0; r < 4; ++r) stride = stride > P.g[r].slot ? stride : P.g[r].slot;
  const int tile_bytes = 16 * (P.D + 4);
  if (stride < 2 * tile_bytes) stride = 2 * tile_bytes;
  stride = (int)align_up((size_t)stride, 128);
  P.ctrl_off = 16 * kMaxStages + 16;
  P.att_off = (int)align_up((size_t)P.ctrl_off + sizeof(Ctrl), 128);
  const size_t att_bytes = (size_t)(kAttMaxG * P.D + kAttMaxG + 2 * P.D) * 4 + 2 * P.D;
  P.red_off = (int)align_up((size_t)P.att_off + att_bytes, 128);
  const size_t red_bytes = (size_t)NCW * RT * NT * 128 * 4;
  const size_t mrg_bytes = (size_t)NCW * (16 + P.G * P.D) * 4;
  P.zero_off = (int)align_up((size_t)P.red_off + (red_bytes > mrg_bytes ? red_bytes : mrg_bytes), 128);
  P.ring_off = (int)align_up((size_t)P.zero_off + kZeroRowBytes, 1024);
  const int budget = smem_optin();
  int stages = (budget - P.ring_off) / stride;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) w.ok = false;
  P.stages = stages;
  P.stride = stride;
  P.smem = P.ring_off + stages * stride;
  P.tps = stride / tile_bytes;
  P.tmin = 16;  // pieces of at least 256 positions
  for (int i = 0; i < 64; ++i)
    P.inv_freq[i] = (i < c.head_dim / 2) ? std::pow((double)c.rope_base, -2.0 * i / c.head_dim) : 0.0;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  (void)take(256);  // sync counters at offset 0
  const int nkg_h = c.hidden / 128, nkg_o = c.n_q * c.head_dim / 128, nkg_a = c.inter / 128;
  w.x_h = take((size_t)B * c.hidden * 2);
  w.s_x = take((size_t)nkg_h * 32 * 4);
  w.ss1 = take((size_t)nkg_h * 32 * 4);
  w.rho1 = take(32 * 4);
  w.qkv = take((size_t)B * P.nqkv * 4);
  w.part = take((size_t)(C + B * c.n_kv) * (16 + P.G * P.D) * 4);
  w.att_tick = take((size_t)B * c.n_kv * 4);
  w.o_h = take((size_t)B * c.n_q * c.head_dim * 2);
  w.s_o = take((size_t)nkg_o * 32 * 4);
  w.h1 = take((size_t)B * c.hidden * 4);
  w.h1_h = take((size_t)B * c.hidden * 2);
  w.s_h1 = take((size_t)nkg_h * 32 * 4);
  w.ss2 = take(32 * 4);
  w.a_h = take((size_t)B * c.inter * 2);
  w.s_a = take((size_t)nkg_a * 32 * 4);
  w.out_acc = take((size_t)B * c.hidden * 4);
  w.total = off;
  return w;
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

template <int NT, int D>
static cudaError_t launch_block(const BlockParams& p, cudaStream_t st) {
  constexpr int THREADS = (GemvShape<NT>::NCW + 1) * 32;
  static std::mutex mu;
  static int attr_smem[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (attr_smem[dev] < p.smem) {
      e = cudaFuncSetAttribute(block_kernel<NT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
      if (e != cudaSuccess) return e;
      attr_smem[dev] = p.smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.C);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, block_kernel<NT, D>, p);
}

template <int D>
static cudaError_t launch_nt(const BlockParams& p, cudaStream_t st) {
  switch (p.g[0].NT) {
    case 1: return launch_block<1, D>(p, st);
    case 2: return launch_block<2, D>(p, st);
    case 3: return launch_block<3, D>(p, st);
    case 4: return launch_block<4, D>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

static int run_block(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch, int max_ctx,
                     const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B, void* ws,
                     size_t ws_bytes, int32_t* status, cudaStream_t st) {
  int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (!w || !cache || !x_in || !x_out || !pos || !ws) return FT_ERR_INVALID_ARG;
  if (!w->qkv || !w->o || !w->gateup || !w->down) return FT_ERR_INVALID_ARG;
  if (act_dtype != FT_BF16 && act_dtype != FT_F32) return FT_ERR_INVALID_ARG;
  if (B < 1 || max_batch < 1 || max_ctx < 1) return FT_ERR_INVALID_ARG;
  if (B > 32) return FT_ERR_UNSUPPORTED;
  if (B > max_batch) return FT_ERR_CAPACITY;
  if (!ft_host::aligned16(cache) || !ft_host::aligned16(ws) || !ft_host::aligned16(x_in) ||
      !ft_host::aligned16(x_out) || !ft_host::aligned16(w->qkv) || !ft_host::aligned16(w->o) ||
      !ft_host::aligned16(w->gateup) || !ft_host::aligned16(w->down))
    return FT_ERR_INVALID_ARG;
  const size_t act_bytes = (size_t)B * c->hidden * (act_dtype == FT_F32 ? 4 : 2);
  if (overlaps(x_in, act_bytes, x_out, act_bytes)) return FT_ERR_INVALID_ARG;
  WsPlan P = make_plan(*c, B, max_ctx);
  if (!P.ok) return FT_ERR_UNSUPPORTED;
  if (ws_bytes < P.total) return FT_ERR_WORKSPACE;
  if (overlaps(x_out, act_bytes, ws, ws_bytes) || overlaps(x_in, act_bytes, ws, ws_bytes)) return FT_ERR_INVALID_ARG;

  uint8_t* W = static_cast<uint8_t*>(ws);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(W + off); };
  auto Hh = [&](size_t off) { return reinterpret_cast<__half*>(W + off); };
  BlockParams& p = P.bp;
  p.w[kRoleQKV] = static_cast<const uint8_t*>(w->qkv);
  p.w[kRoleO] = static_cast<const uint8_t*>(w->o);
  p.w[kRoleGU] = static_cast<const uint8_t*>(w->gateup);
  p.w[kRoleDown] = static_cast<const uint8_t*>(w->down);
  p.cache = static_cast<uint8_t*>(cache);
  p.L = kv_layout(*c, max_batch, max_ctx);
  p.pos = pos;
  p.x_in = x_in;
  p.x_out = x_out;
  p.act_dtype = act_dtype;
  p.sync = reinterpret_cast<uint32_t*>(W);
  p.x_h = Hh(P.x_h);
  p.s_x = F(P.s_x);
  p.ss1 = F(P.ss1);
  p.rho1 = F(P.rho1);
  p.qkv = F(P.qkv);
  p.part = F(P.part);
  p.att_tick = reinterpret_cast<uint32_t*>(W + P.att_tick);
  p.o_h = Hh(P.o_h);
  p.s_o = F(P.s_o);
  p.h1 = F(P.h1);
  p.h1_h = Hh(P.h1_h);
  p.s_h1 = F(P.s_h1);
  p.ss2 = F(P.ss2);
  p.a_h = Hh(P.a_h);
  p.s_a = F(P.s_a);
  p.out_acc = (act_dtype == FT_F32) ? static_cast<float*>(x_out) : F(P.out_acc);
  p.status = status;
  const cudaError_t ce = (c->head_dim == 128) ? launch_nt<128>(p, st) : launch_nt<64>(p, st);
  return ce == cudaSuccess ? FT_OK : FT_ERR_CUDA;
}

}  // namespace ft

extern "C" {

size_t ft_decode_workspace_bytes(const ft_block_cfg* c, int B, int max_ctx) {
  if (ft_host::check_cfg(c) != FT_OK || B < 1 || B > 32 || max_ctx < 1) return 0;
  return ft::make_plan(*c, B, max_ctx).total;
}

int ft_decode_workspace_layout(const ft_block_cfg* c, int B, int max_ctx, ft_ws_layout* out) {
  const int e = ft_host::check_cfg(c);
  if (e != FT_OK) return e;
  if (!out || B < 1 || B > 32 || max_ctx < 1) return FT_ERR_INVALID_ARG;
  const ft::WsPlan P = ft::make_plan(*c, B, max_ctx);
  out->qkv = P.qkv;
  out->rho1 = P.rho1;
  out->o = P.o_h;
  out->h1 = P.h1;
  out->a = P.a_h;
  out->n_split = P.bp.C;
  return FT_OK;
}

int ft_decode_block(const ft_block_cfg* c, const ft_layer_weights* w, void* cache, int max_batch, int max_ctx,
                    const void* x_in, void* x_out, int act_dtype, const int32_t* pos, int B, void* ws,
                    size_t ws_bytes, int32_t* status, ft_stream stream) {
  return ft::run_block(c, w, cache, max_batch, max_ctx, x_in, x_out, act_dtype, pos, B, ws, ws_bytes, status,
                       (cudaStream_t)stream);
}

int ft_decode_block_launches(void) { return 1; }

}  // extern "C"
