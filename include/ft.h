/*
 * ft.h -- C ABI of the INT4-weight / Hadamard-rotated INT4-KV decode block.
 *
 * One Llama-style Transformer block, one new token per request, on one GPU
 * (sm_103a).  The operations follow the statement of the problem on the pages
 * "FuTransformer: FP8 prefill and INT4 decode for Llama-style inference on
 * Hopper" (summary page on onedev.kr, sections "어떻게 동작하나" / how it
 * works, "무엇과 다른가" / what differs, "전제와 한계" / premises and limits).
 *
 * Conventions (all calls):
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise.  The
 *    caller allocates and owns all memory; the library never allocates.
 *  - Calls are asynchronous on the caller's stream and return an ft_status
 *    code.  Host-side argument checks happen before anything is enqueued; a
 *    failed check enqueues nothing.
 *  - Conditions only the device can see (a position beyond the cache capacity,
 *    an activation outside the FP16 range, a bounded wait that ran out) are
 *    OR-ed into the caller's int32 device status word (may be NULL) as
 *    FT_DEV_* bits; read it after synchronising.  Kernels never trap.
 *  - No exception or abort crosses this boundary.
 */
#ifndef FT_H_
#define FT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *ft_stream;

/* ---- status codes ------------------------------------------------------ */
enum {
  FT_OK = 0,
  FT_ERR_INVALID_ARG = -1, /* NULL/misaligned pointer, bad size, overlap    */
  FT_ERR_UNSUPPORTED = -2, /* shape or option this build does not implement */
  FT_ERR_WORKSPACE = -3,   /* workspace or packed buffer too small          */
  FT_ERR_CAPACITY = -4,    /* batch larger than the cache's max_batch       */
  FT_ERR_CUDA = -5         /* a CUDA runtime call failed (launch, attrs)    */
};

/* bits OR-ed into the device status word */
enum {
  FT_DEV_CAPACITY = 1, /* pos[b] (+T) outside [0, max_ctx): that request skipped */
  FT_DEV_TIMEOUT = 2,  /* a bounded pipeline wait ran out; outputs invalid       */
  FT_DEV_RANGE = 4     /* an activation exceeded the FP16 operand range          */
};

/* activation dtypes of the block input/output */
enum { FT_BF16 = 0, FT_F32 = 1 };

/* decode-weight formats (ft_block_cfg.weight_format): INT4 codes, or E4M3 codes
 * (summary page, "전제와 한계": E4M3 decode weights as the FP8 variant of the
 * decode path), both with one BF16 scale per (output row, 128 inputs) */
enum { FT_WFMT_INT4 = 0, FT_WFMT_E4M3 = 1 };

/* ---- configuration ------------------------------------------------------ */
typedef struct {
  int32_t hidden;    /* H; multiple of 128                                      */
  int32_t n_q;       /* query heads; multiple of n_kv, n_q / n_kv <= 8          */
  int32_t n_kv;      /* KV heads                                               */
  int32_t head_dim;  /* d in {64, 128}                                          */
  int32_t inter;     /* SwiGLU intermediate I; multiple of 128                  */
  int32_t w_group;   /* weight group along the input axis; must be 128         */
  int32_t had_block; /* Hadamard block h_b: power of two dividing d (1 = none) */
  int32_t kv_group;  /* channels per KV scale; must equal head_dim             */
  float rms_eps;     /* RMSNorm epsilon                                        */
  float rope_base;   /* RoPE base                                              */
  int32_t weight_format; /* FT_WFMT_INT4 (0) or FT_WFMT_E4M3                    */
} ft_block_cfg;

/* Projection roles.  Weights are given in the logical row-major [N_out, K_in]
 * orientation:  QKV [(n_q+2 n_kv) d, H] (q rows, then k, then v);
 * O [H, n_q d];  GATEUP [2 I, H] (I gate rows, then I up rows);  DOWN [H, I]. */
typedef enum { FT_W_QKV = 0, FT_W_O = 1, FT_W_GATEUP = 2, FT_W_DOWN = 3 } ft_wrole;

/* Describes a status code; never NULL. */
const char *ft_status_string(int status);

/* Host-only check of a configuration (FT_OK, FT_ERR_INVALID_ARG, FT_ERR_UNSUPPORTED). */
int ft_validate_cfg(const ft_block_cfg *cfg);

/* Logical shape [n_out, k_in] of a role's weight matrix (host pointers out). */
int ft_weight_shape(const ft_block_cfg *cfg, int role, int32_t *n_out, int32_t *k_in);

/* ---- weights ------------------------------------------------------------
 * Packing (summary page, "어떻게 동작하나": the fixed RMSNorm gain is folded
 * into the weights before quantisation, W' = gamma W; "무엇과 다른가": INT4
 * values with group scales applied after accumulation, stored in the order the
 * kernel consumes them).  For each output row o and each group of 128
 * consecutive input channels: W'[o,i] = W[o,i] * gamma[i] (FP32 product),
 * s = bf16_rne(amax / 7), code = clamp(rne(W' / s), -8, 7) + 8 (FP32
 * decisions; s = 0 gives code 8).  The packed buffer is opaque: 128-row blocks,
 * 16-row tiles, per (tile, group) 1024 bytes of nibbles in the tensor-core
 * fragment order the decode kernels read, followed by the 16 BF16 scales. */

/* Bytes of one packed role in the configuration's weight format: INT4 codes
 * P/2 + scales P/64, or E4M3 codes P + scales P/64, for P = N_out * K_in. */
size_t ft_packed_weight_bytes(const ft_block_cfg *cfg, int role);

/* W: FP32 [N_out, K_in] row-major.  gamma: FP32 [K_in] or NULL (treated as 1);
 * use gamma_attn for QKV and gamma_ffn for GATEUP.  packed: >= 16-byte aligned,
 * packed_bytes >= ft_packed_weight_bytes().  Overwrites packed entirely.
 * cfg->weight_format must be FT_WFMT_INT4 (else FT_ERR_INVALID_ARG). */
int ft_pack_weights_int4(const ft_block_cfg *cfg, int role, const float *W, const float *gamma,
                         void *packed, size_t packed_bytes, ft_stream stream);

/* Inverse view for tests: codes uint8 [N_out, K_in] in [0,15] (value code-8)
 * and scales as BF16 bits [N_out, K_in/128], logical orientation. */
int ft_unpack_weights_int4(const ft_block_cfg *cfg, int role, const void *packed, uint8_t *codes,
                           uint16_t *scales_bf16, ft_stream stream);

/* E4M3 decode weights (summary page, "전제와 한계"; the abstract page compares
 * the INT4 decode path with an FP8 one).  For each output row o and group of 128
 * consecutive inputs: W'[o,i] = W[o,i] * gamma[i] (FP32), s = bf16_rne(amax /
 * 448), code = E4M3(W' / s) rounded to nearest, ties to even, saturating at
 * +-448, the sign of zero kept (FP32 division; s = 0 gives code 0x00).  Same
 * row-tile-major layout as INT4 with 2048 bytes of codes per (tile, group) in
 * the tensor-core fragment order, then the 16 BF16 scales.  Arguments as for
 * ft_pack_weights_int4; cfg->weight_format must be FT_WFMT_E4M3. */
int ft_pack_weights_e4m3(const ft_block_cfg *cfg, int role, const float *W, const float *gamma, void *packed,
                         size_t packed_bytes, ft_stream stream);

/* Inverse layout transform of ft_pack_weights_e4m3 (for tests): codes as E4M3
 * bytes [N_out, K_in] and scales as BF16 bits [N_out, K_in/128]. */
int ft_unpack_weights_e4m3(const ft_block_cfg *cfg, int role, const void *packed, uint8_t *codes,
                           uint16_t *scales_bf16, ft_stream stream);

/* ---- KV cache -----------------------------------------------------------
 * One layer's cache for max_batch requests x n_kv heads x max_ctx positions.
 * Entry (request, head, position) holds d/2 bytes of K nibbles, d/2 bytes of V
 * nibbles and one BF16 scale each for K and V (kv_group = d), addressed by
 * offset(request, head, position, channel) (summary page, "어떻게 동작하나":
 * direct placement, no dense K/V tensors).  Within an entry the nibbles are
 * permuted into the tensor-core fragment order of the attention kernel; the
 * buffer is opaque to callers. */

size_t ft_kv_cache_bytes(const ft_block_cfg *cfg, int max_batch, int max_ctx);

/* Append T tokens per request (summary page, "무엇과 다른가": block-diagonal
 * Hadamard rotation of the new K and V, then INT4 quantisation with BF16
 * scales; H is the normalised Sylvester matrix of order had_block).
 * k_bf16, v_bf16: BF16 bits [B, T, n_kv, d] (post-RoPE).  pos: device int32
 * [B], first position of request b.  Positions pos[b]..pos[b]+T-1 are written;
 * a request with pos[b] < 0 or pos[b]+T > max_ctx is skipped and sets
 * FT_DEV_CAPACITY.  B <= max_batch or FT_ERR_CAPACITY. */
int ft_kv_append_int4(const ft_block_cfg *cfg, void *cache, int max_batch, int max_ctx,
                      const uint16_t *k_bf16, const uint16_t *v_bf16, const int32_t *pos, int B,
                      int T, int32_t *dev_status, ft_stream stream);

/* Append packed variable-length requests: the K/V rows the prefill side
 * produces for a batch of prompts of different lengths, placed straight at
 * offset(request, head, position, channel) (summary page, "어떻게 동작하나":
 * the QKV epilogue writes the KV cache directly; requests of different lengths
 * are packed).  The prefill GEMM itself is not part of this library; this call
 * is its placement step, with the same rotation and quantiser as
 * ft_kv_append_int4.
 *   k_bf16, v_bf16: BF16 bits [total, n_kv, d] (post-RoPE), the rows of request
 *     0, then request 1, ... back to back.
 *   cu_seqlens: device int32 [B + 1], the prefix sums of the request lengths
 *     (cu_seqlens[0] = 0, cu_seqlens[B] = total, non-decreasing); request b
 *     owns rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (a zero-length request owns
 *     none).
 *   pos: device int32 [B], the first position written for request b.
 * Row cu_seqlens[b] + t goes to position pos[b] + t of request b.  A request
 * whose positions fall outside 0 .. max_ctx-1 is skipped and sets
 * FT_DEV_CAPACITY; a map that is not such a prefix sum writes nothing and sets
 * FT_DEV_RANGE.  B <= max_batch or FT_ERR_CAPACITY; total = 0 enqueues nothing. */
int ft_kv_append_ragged_int4(const ft_block_cfg *cfg, void *cache, int max_batch, int max_ctx,
                             const uint16_t *k_bf16, const uint16_t *v_bf16, const int32_t *cu_seqlens,
                             const int32_t *pos, int B, int total, int32_t *dev_status, ft_stream stream);

/* Inverse view for tests: positions [0, len) of requests [0, B).  codes uint8
 * [B, n_kv, len, d] in logical channel order; scales BF16 bits [B, n_kv, len, 1]. */
int ft_kv_unpack_int4(const ft_block_cfg *cfg, const void *cache, int max_batch, int max_ctx, int B,
                      int len, uint8_t *k_codes, uint8_t *v_codes, uint16_t *k_scales,
                      uint16_t *v_scales, ft_stream stream);

/* ---- the decode block ---------------------------------------------------
 * One token per request b < B at position pos[b] (= L_b, its history length):
 *   rho1 = (mean x^2 + eps)^-1/2;  [q;k;v] = rho1 * W'_qkv x      (row factor
 *      applied after the projection's accumulation, "어떻게 동작하나")
 *   RoPE(q, k) at L_b;  k~ = H k, v~ = H v quantised and written at L_b
 *   q~ = H q;  per query head h (KV head h / G, no head expansion,
 *      "전제와 한계"): softmax over positions 0..L_b of q~.k^/sqrt(d) against
 *      the INT4 cache (split across CTAs and merged for long contexts,
 *      "무엇과 다른가"), o = H o~ (inverse rotation)
 *   h1 = x + W_o o;  rho2 = (mean h1^2 + eps)^-1/2;
 *   a = silu(rho2 W'_g h1) * (rho2 W'_u h1);  out = h1 + W_down a.
 * The new token's K/V are written before attending; attention covers
 * positions 0..pos[b] inclusive; the caller advances pos.
 * x_in, x_out: [B, H] of act_dtype (FT_BF16 bits or FT_F32), must not overlap.
 * Arithmetic: tensor-core FP16 operands (codes exact, activations rounded to
 * FP16), FP32 accumulation, epilogues and softmax.  Activations must stay
 * within the FP16 range (|x| < 65504; FT_DEV_RANGE otherwise).
 * The projection weights are in cfg->weight_format (INT4 or E4M3 codes).
 * 1 <= B <= min(32, max_batch); larger B -> FT_ERR_UNSUPPORTED. */
typedef struct {
  const void *qkv, *o, *gateup, *down; /* each from the pack call of cfg->weight_format */
} ft_layer_weights;

size_t ft_decode_workspace_bytes(const ft_block_cfg *cfg, int B, int max_ctx);

int ft_decode_block(const ft_block_cfg *cfg, const ft_layer_weights *w, void *cache, int max_batch,
                    int max_ctx, const void *x_in, void *x_out, int act_dtype, const int32_t *pos,
                    int B, void *workspace, size_t ws_bytes, int32_t *dev_status, ft_stream stream);

/* Stage selection for ft_decode_block_stages (bit mask). */
enum {
  FT_STAGE_PREP = 1,  /* input -> FP16 operand, sums of squares, zero counters */
  FT_STAGE_QKV = 2,   /* QKV projection (x rho1)                             */
  FT_STAGE_ATTN = 4,  /* RoPE, rotation, cache write, split-KV attention     */
  FT_STAGE_O = 8,     /* O projection + residual                              */
  FT_STAGE_MID = 16,  /* h1 -> gate/up operand, sums of squares, down acc.   */
  FT_STAGE_GU = 32,   /* gate/up projection + SwiGLU                          */
  FT_STAGE_DOWN = 64, /* down projection + residual -> x_out                  */
  FT_STAGE_ALL = 127
};

/* Runs a subset of the block's stages on a workspace left by a previous full
 * call with the same arguments (each stage reads what the earlier stages
 * wrote there).  Used to time one stage alone; FT_STAGE_ALL equals
 * ft_decode_block. */
int ft_decode_block_stages(const ft_block_cfg *cfg, const ft_layer_weights *w, void *cache,
                           int max_batch, int max_ctx, const void *x_in, void *x_out, int act_dtype,
                           const int32_t *pos, int B, void *workspace, size_t ws_bytes,
                           int32_t *dev_status, unsigned stage_mask, ft_stream stream);

/* Byte offsets of intermediate tensors inside the workspace (host struct out),
 * for tests:  qkv FP32 [B, (n_q+2n_kv) d] (the projection before rho1 and
 * RoPE);  rho1 FP32 [B];  o FP16, n_q d values per request (attention output
 * after the inverse rotation);  h1 FP32 [B, H];  a FP16, I values per request
 * (SwiGLU output).  o and a are stored in the projections' grouped operand
 * layout: [inputs / 64][B][64], i.e. the B requests' values of each half group
 * of 64 inputs together (one 128-byte row per request); within a request's 64
 * values the order is 0,1,8,9,2,3,10,11,4,5,12,13,6,7,14,15 per 16 inputs,
 * inputs 8..15 of each 16 hold value / 16, and the 8 runs of 8 stored values
 * are permuted: run r is stored at position r XOR (request mod 8). */
typedef struct {
  size_t qkv, rho1, o, h1, a;
  int32_t n_split; /* split-KV chunks per (request, KV head) */
} ft_ws_layout;

int ft_decode_workspace_layout(const ft_block_cfg *cfg, int B, int max_ctx, ft_ws_layout *out);

/* How ft_decode_block partitions one projection (role FT_W_*) for this batch
 * on the current device (148 SMs assumed when no device is visible): ctas
 * launched; rows per set (row_tiles x 16); warps per CTA; 8-token column tiles;
 * whole = 1 when every CTA owns whole sets (no split along the inputs);
 * tensor_core = 1 for the tcgen05 kernel of batches 17-32 (128-row sets, the
 * contraction on the fifth-generation tensor cores), 0 for the streaming
 * mma.sync kernel of batches 1-16; ring stages, groups (128 inputs) per stage
 * and dynamic shared memory per CTA in bytes. */
typedef struct {
  int32_t ctas, row_tiles, warps, col_tiles, whole, tensor_core, stages, groups_per_stage, smem_bytes;
} ft_gemv_info;
int ft_decode_plan_info(const ft_block_cfg *cfg, int B, int max_ctx, int role, ft_gemv_info *out);

/* ---- full decode step helpers (BF16, not INT4) ----------------------------
 * A complete Llama-style decode step is: embedding gather, the decode block
 * per layer (FT_F32 residual between layers), final RMSNorm, LM head (summary
 * page, "전제와 한계": the full Llama-3.1-8B step at batch 1). */

/* x_out[b, :] = table[tokens[b], :] widened to FP32.  table: BF16 bits [V, H];
 * tokens: device int32 [B]; x_out: FP32 [B, H].  A token outside [0, V) gives a
 * zero row and sets FT_DEV_RANGE. */
int ft_embed_bf16(const uint16_t *table, const int32_t *tokens, float *x_out, int B, int V, int H,
                  int32_t *dev_status, ft_stream stream);

/* Final RMSNorm on its own (ft_lm_head_bf16 applies it fused):
 * z[b, :] = bf16(gamma * rho_b * x[b, :]), rho_b = (mean x[b, :]^2 + eps)^-1/2.
 * x: FP32 [B, H]; gamma: FP32 [H]; z_out: BF16 bits [B, H]. */
int ft_rmsnorm_bf16(const float *x, const float *gamma, uint16_t *z_out, int B, int H, float eps,
                    ft_stream stream);

/* Copies the device status word that the calls above OR their asynchronous
 * FT_DEV_* conditions into to *host_out, after waiting for `stream` (every
 * call enqueued before it has finished).  FT_OK, or FT_ERR_CUDA if the copy or
 * the wait fails. */
int ft_read_device_status(const int32_t *dev_status, int32_t *host_out, ft_stream stream);

/* logits[b, v] = sum_k W[v, k] * z[b, k] with z = gamma * rho(x_b) * x_b,
 * rho = (mean x^2 + eps)^-1/2.  x: FP32 [B, H]; gamma: FP32 [H]; W: BF16 bits
 * [V, H] (16-byte aligned); logits: FP32 [B, V] (overwritten; every element
 * is written once, no accumulation, so repeated calls give the same bits).
 * B <= 32 and H a multiple of 128, else FT_ERR_UNSUPPORTED.  Tokens run in
 * chunks of min(8, 160 KiB / (4 H)) (one launch each, W streamed once per
 * chunk).  z enters the tensor cores as a BF16 (hi, lo) pair. */
int ft_lm_head_bf16(const float *x, const float *gamma, const uint16_t *W, float *logits, int B, int V, int H,
                    float eps, ft_stream stream);

/* ft_decode_block without a caller-provided workspace.  The FuTransformer paper
 * has no counterpart to this call; it exists for callers that cannot allocate
 * device memory when they run a step (a pool or allocation policy that forbids
 * new device allocations after start-up, a host that hands over only input and
 * output buffers, or a loop that must not pay for an allocation).  The scratch
 * space is a fixed 48 MiB device array inside this library, held by every GPU
 * that loads it until the process exits; problems needing more (see
 * ft_decode_workspace_bytes; the 70B layer shape at batch 32 needs about
 * 33 MiB) return FT_ERR_WORKSPACE and enqueue nothing.  No memory is allocated
 * by this call.  The array is shared by all calls on a device and keeps the
 * previous call's contents (the block clears what it needs itself); calls that
 * overlap on the GPU race on it.  The first call on each device looks up the
 * array's address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept for the process's
 * life: do not use this call on a device after cudaDeviceReset in the same
 * process.  Arguments and results are otherwise those of ft_decode_block. */
int ft_decode_block_static_ws(const ft_block_cfg *cfg, const ft_layer_weights *w, void *cache, int max_batch,
                              int max_ctx, const void *x_in, void *x_out, int act_dtype, const int32_t *pos, int B,
                              int32_t *dev_status, ft_stream stream);

/* Number of kernels one ft_decode_block call with batch B launches: 7 for
 * INT4 weights and B <= 16; 9 where the projections run on the tensor cores
 * (17 <= B <= 32, or E4M3 weights at any batch) and two small kernels finish
 * gate/up (SwiGLU) and the block output from the per-piece partial sums.
 * 0 for an invalid configuration. */
int ft_decode_block_launches(const ft_block_cfg *cfg, int B);

/* Programmatic dependent launch between the block's kernels (default on).
 * Returns the previous setting. */
int ft_set_pdl(int enabled);

#ifdef __cplusplus
}
#endif

#endif /* FT_H_ */
