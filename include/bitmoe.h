/*
 * bitmoe.h -- C ABI of the int4 mixture-of-experts layer and int4 LM head
 * for NVIDIA B300 (sm_103a).
 *
 * What is computed.  One sparse MoE layer of a 256-expert, top-k coding model
 * with 4-bit weights ("Flint 40B : Best Mid Sized LLM", video transcript
 * 02:35: 256 routed experts per mixture layer, a small router picks a few per
 * token; 06:11: dedicated kernels for low-bit projections and mixture-of-
 * experts routing), and the 4-bit output projection (same transcript 03:36
 * and 05:39; "Recursive_SI's First Model Unveiled!", section "Quantization"):
 *
 *   logits l = x Wr^T + b          softmax p = softmax(l)     top-k ids, gates w
 *   rows grouped by expert (stable)                              [moe_permute]
 *   a = x Wg^T, u = x Wu^T, h = silu(a) * u, y = h Wd^T          [moe_expert_ffn_int4]
 *   out = residual + sum_j w_j y_j                               [moe_combine]
 *   z = h Wlm^T, argmax z                                        [lmhead_int4_gemv]
 *
 * Conventions.
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; nothing is
 *    freed or retained by the library.  bf16 and fp16 tensors are passed as
 *    raw 16-bit patterns (uint16_t).  All tensors are dense row-major.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and returns a bitmoe_status_t synchronously.  A call that
 *    returns an error launched nothing.
 *  - Scratch memory comes from a caller-provided workspace whose size is given
 *    by the matching *_workspace_size() function; pass the workspace of the
 *    same shape to every call that needs one.  Calls sharing one workspace must
 *    be ordered on one stream.
 *  - int4 weights are used in the library's packed tile layout, produced once
 *    by bitmoe_pack_int4() from the canonical layout below.
 *  - Device-side checks (forced expert ids out of range, a bounded wait that
 *    ran out) do not fault: they set a status word inside the workspace, read
 *    with bitmoe_get_device_status().
 *
 * Canonical int4 layout (input of bitmoe_pack_int4).  A bank of n_mats
 * matrices, each rows x K: q [n_mats, rows, K/2] bytes, element 2b of a row in
 * the low nibble of byte b and 2b+1 in the high nibble, two's complement in
 * [-8, 7]; scale [n_mats, rows, K/group] fp16.  W[n,i] = q[n,i] * s[n, i/group]
 * (symmetric, no zero point).  The expert banks are gate [E, I, d],
 * up [E, I, d] and down [E, d, I]; the LM head is one matrix [V, d].
 */
#ifndef BITMOE_H_
#define BITMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bitmoe_status {
  BITMOE_OK = 0,
  BITMOE_ERR_INVALID_ARG = 1,  /* null pointer, bad shape, misaligned pointer, k > E ... */
  BITMOE_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels handle (see each call) */
  BITMOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than *_workspace_size() */
  BITMOE_ERR_CUDA = 4,         /* a launch failed; bitmoe_last_cuda_error() has the code */
  BITMOE_ERR_TIMEOUT = 5,      /* device status: a bounded wait ran out */
  BITMOE_ERR_DEVICE_CHECK = 6  /* device status: an input failed a device-side check (an
                                  out-of-range or repeated forced expert id, or an expert
                                  intermediate outside the fp16 range, see moe_forward) */
} bitmoe_status_t;

/* Shape of one MoE layer.  d: hidden size; E: routed experts; k: routed
 * experts per token; I: expert intermediate size; group: the weights' scale
 * group (32 for the int4 calls, 16 for the NVFP4 ones); renormalize: 1 = gates
 * are the chosen softmax probabilities rescaled
 * to sum 1, 0 = the raw probabilities; n_shared: 0, or 1 for a shared expert
 * that every token uses with gate weight 1 besides its k routed ones ("Flint
 * 40B : Best Mid Sized LLM", transcript 02:35: six routed experts of 256 plus
 * one shared expert that is always on).  The shared expert is entry E of each
 * expert bank (the banks then hold E + 1 experts; the router still scores the
 * E routed ones), and every per-token array below -- topk_ids, topk_w, the
 * forced selection, the rows of the permutation -- has kt = k + n_shared
 * entries per token, the shared one last (id E, weight 1).  k = 0 with
 * n_shared = 1 is a dense SwiGLU layer (the stack's two leading layers in the
 * same transcript): the bank's one entry serves every token with weight 1 and
 * there is no router (w_router may be NULL; E is normally 0).  Supported: d and
 * I multiples of 128, group == 32 (int4) or 16 (NVFP4), 1 <= k <= E or k = 0 with n_shared = 1,
 * k + n_shared <= 32, E + n_shared <= 1024.  (n_shared fills what was padding: the struct's size
 * is that of the version without it, where it read as 0 when zero-filled.) */
typedef struct bitmoe_moe_shape {
  int64_t d, E, k, I, group;
  int32_t renormalize;
  int32_t n_shared;
} bitmoe_moe_shape_t;

/* Packed expert banks (bitmoe_pack_int4 output, 16-byte aligned) and the
 * router: w_router [E, d] fp32, b_router [E] fp32 or NULL (no bias). */
typedef struct bitmoe_moe_weights {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
} bitmoe_moe_weights_t;

/* NVFP4 expert banks (bitmoe_pack_nvfp4 output, 16-byte aligned), their fp32
 * tensor scales gate_scale / up_scale / down_scale [E + n_shared] (device, one
 * per bank entry, finite) and the router as in bitmoe_moe_weights_t. */
typedef struct bitmoe_moe_weights_nvfp4 {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* gate_scale;
  const float* up_scale;
  const float* down_scale;
  const float* w_router;
  const float* b_router;
} bitmoe_moe_weights_nvfp4_t;

/* ------------------------------------------------------------ utilities */

const char* bitmoe_status_string(bitmoe_status_t status);
/* cudaError_t code of the last failed launch in this thread (0 if none). */
int bitmoe_last_cuda_error(void);
const char* bitmoe_version(void);

/* Tracing (off by default): while a device buffer is set, every fused decode
 * launch writes 32 stamps per CTA into it, as uint64 [gridDim][32]: slots
 * 0..30 hold the SM's cycle counter (clock64) at 0 start, 1 after the
 * grid-dependency wait, 2 logits done, 3 after barrier A, 4 routing done,
 * 5 gate/up done, 6 after barrier B, 7 end; 8 first gate/up unit computed,
 * 9 second unit's tiles landed, 10 grouping ranks done, 11 routing tables
 * done, 12 first gate/up tiles landed, 13 h staged, 14 down projection done,
 * 15 first unit's h stored, 16 x landed, 17 router rows landed, 18 router dot
 * products done, 19 first W_down stage landed, 20 first W_down stage done,
 * 22 / 23 barrier A / B arrival counted; slot 31 holds the global timer (ns)
 * at point 0 (0 = not reached).
 * The buffer must hold gridDim (= SM count) * 256 bytes, else tracing is skipped.
 * Pass NULL, 0 to turn it off.  Process-wide; not for concurrent callers. */
bitmoe_status_t bitmoe_set_trace_buffer(void* device_buf, size_t bytes);

/* Bytes of a packed bank of n_mats matrices of rows x K (rows % 16 == 0,
 * K % 128 == 0, group == 32); 0 for an unsupported shape.  Equal to the
 * canonical size q + scale: n_mats * rows * K * 9 / 16. */
size_t bitmoe_packed_int4_bytes(int64_t n_mats, int64_t rows, int64_t K, int64_t group);

/* Reorder a canonical int4 bank (device q, scale) into the packed tile layout
 * the kernels stream: 16-row tiles, each a run of 128-column chunks holding
 * the nibbles of every (row, 32-column group) in the order one mma fragment
 * consumes them, followed by the chunk's fp16 scales.  Off the timed path.
 * q 4-byte aligned, scale 2-byte aligned; packed: a 16-byte aligned device
 * buffer of bitmoe_packed_int4_bytes().  The packed bank holds the same bytes as q + scale
 * (nothing added), so a 4-bit weight with a 16-bit scale per 32 weights costs
 * 4.5 bits, as the pages' ~23 GB 4-bit release of the 39.8B model implies.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 07:15 (four-bit and
 * integer-four builds, GGUF files around 23 GB); "Recursive_SI's First Model
 * Unveiled!", section "Quantization" (4-bit weights, the output layer too). */
bitmoe_status_t bitmoe_pack_int4(const uint8_t* q, const uint16_t* scale, int64_t n_mats, int64_t rows,
                                 int64_t K, int64_t group, uint8_t* packed, void* stream);

/* ------------------------------------------------------------ attention decode step
 *
 * The attention layer beside each mixture layer, for one token of a decode step:
 * grouped-query attention over a bf16 key/value cache with a sliding window or the
 * whole context, per-head RMS norm on queries and keys, rotary encoding and learned
 * sinks.
 *   q | k | v = Wqkv x                    (int4 group-32, rows stacked: nq*128 | nkv*128 | nkv*128)
 *   q_h, k_g <- RMSNorm per head (unit gain, eps), then rotated by the position when
 *               rope: pairs (i, i + 64) by the angle pos * rope_theta^(-2i/128)
 *   cache row pos <- bf16(k), bf16(v)
 *   o_h = sum_j e^(s_j) v_j / (sum_j e^(s_j) + e^(sink_h)),  s_j = q_h . k_j / sqrt(128),
 *         j over the window [max(0, pos - window + 1), pos] (window 0: [0, pos]) of key/value
 *         head g = h / (nq / nkv); no sinks: the plain softmax
 *   out = residual + Wo bf16(o)           (bf16 out; out_f32 the unrounded sum, nullable)
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 03:05 (32 query / 4 key-value heads of
 * 128, a 513-token sliding window on 35 layers with rotary encoding, whole-context attention
 * without it on the others) and 03:36 (per-head RMS norm on q and k, learned attention sinks);
 * the pages give no formula: rope_theta, eps, the sink form and the bf16 cache are readings.
 * Supported: head_dim 128, nq = 8 nkv, d % 128 == 0; else BITMOE_ERR_UNSUPPORTED.  x, residual,
 * out [d] bf16 (one token); k_cache, v_cache [nkv, max_len, 128] bf16, head-major (each
 * head's rows contiguous, so a span of positions is one run of memory), with rows 0 .. pos - 1
 * of every head filled by earlier steps and row pos written by this one (0 <= pos < max_len,
 * else BITMOE_ERR_INVALID_ARG); all 16-byte aligned.  d and nq * 128 at most 16384.  Workspace: attn_workspace_size() bytes,
 * zero-filled before first use. */
typedef struct bitmoe_attn_shape {
  int64_t d;          /* hidden size */
  int64_t n_q_heads;  /* query heads (32) */
  int64_t n_kv_heads; /* key/value heads (4) */
  int64_t head_dim;   /* 128 */
  int64_t max_len;    /* cache rows */
  int64_t window;     /* attended tokens including the current one (513); 0: the whole context */
  int32_t rope;       /* 1: rotary encoding of q and k; 0: none */
  float eps;          /* RMS-norm epsilon (1e-6) */
  double rope_theta;  /* rotary base (1e6) */
} bitmoe_attn_shape_t;

typedef struct bitmoe_attn_weights {
  const uint8_t* wqkv; /* packed int4 [(nq + 2 nkv) * 128, d] (bitmoe_pack_int4, group 32) */
  const uint8_t* wo;   /* packed int4 [d, nq * 128] */
  const float* sinks;  /* [nq] fp32 sink logits, or NULL */
} bitmoe_attn_weights_t;

size_t attn_workspace_size(const bitmoe_attn_shape_t* shape);
/* x the block's input (the normalised residual); out may alias residual, not x. */
bitmoe_status_t attn_decode_step(const uint16_t* x, const uint16_t* residual, int64_t pos,
                                 const bitmoe_attn_shape_t* shape, const bitmoe_attn_weights_t* weights,
                                 uint16_t* k_cache, uint16_t* v_cache, uint16_t* out, float* out_f32,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* The pre-norm attention block of a decoder layer, as the stack's MoE block
 * (moe_forward_prenorm): x = bf16(residual / sqrt(mean(residual^2) + eps)) with the shape's
 * eps (unit gain; the norm is formed inside the q|k|v projection launch), then
 * out = residual + Attn(x) as attn_decode_step.  out may alias residual (in-place update
 * of the residual stream).  A decoder layer is this call followed by moe_forward_prenorm.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 03:05 (every mixture layer has an
 * attention block before its experts); the pre-norm placement and unit gain are readings. */
bitmoe_status_t attn_decode_step_prenorm(const uint16_t* residual, int64_t pos, const bitmoe_attn_shape_t* shape,
                                         const bitmoe_attn_weights_t* weights, uint16_t* k_cache,
                                         uint16_t* v_cache, uint16_t* out, float* out_f32, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Read (and clear, when clear != 0) the device status word of a workspace.
 * Synchronises `stream`.  *status_out receives BITMOE_OK, BITMOE_ERR_TIMEOUT
 * or BITMOE_ERR_DEVICE_CHECK. */
bitmoe_status_t bitmoe_get_device_status(void* workspace, int clear, int32_t* status_out, void* stream);

/* ------------------------------------------------------------ NVFP4 weights
 *
 * The pages name "four-bit NVFP" builds of the model beside the integer-four
 * ones and an NVFP4 final model ("Flint 40B : Best Mid Sized LLM", transcript
 * 07:15; "Recursive_SI's First Model Unveiled!", section "Quantization") but do
 * not define the format; this library takes its public definition:
 *   W[n,i] = e2m1(q[n,i]) * e4m3(s[n, i/16]) * ts
 * with q an FP4 E2M1 code (bit 3 sign, 2 exponent bits with bias 1, 1 mantissa
 * bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), s an FP8 E4M3 scale byte for
 * every 16 consecutive weights of a row (finite; NVFP4 scales are >= 0), and ts
 * one fp32 tensor scale per matrix.
 * Canonical NVFP4 layout (input of bitmoe_pack_nvfp4): q [n_mats, rows, K/2]
 * bytes, element 2b in the low nibble of byte b; s [n_mats, rows, K/16] bytes.
 * The packed bank has the int4 bank's tile geometry and size (4.5 bits per
 * weight); tensor scales are passed to the compute calls, not packed.
 */

/* Bytes of a packed NVFP4 bank (rows % 16 == 0, K % 128 == 0; else 0):
 * n_mats * rows * K * 9 / 16. */
size_t bitmoe_packed_nvfp4_bytes(int64_t n_mats, int64_t rows, int64_t K);

/* Reorder a canonical NVFP4 bank (device q, s) into the packed tile layout:
 * 16-row tiles of 128-column chunks, each chunk the 16 x 128 codes in the
 * order one mma fragment takes them (a 32-bit word per lane and 32-column
 * group, byte j holding the two codes of fragment register j) and then the 16
 * rows' 8 block-scale bytes.  q 4-byte aligned; packed 16-byte aligned, of
 * bitmoe_packed_nvfp4_bytes().  Off the timed path.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 07:15. */
bitmoe_status_t bitmoe_pack_nvfp4(const uint8_t* q, const uint8_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                                  uint8_t* packed, void* stream);

/* ------------------------------------------------------------ MoE layer */

/* Workspace bytes for any MoE call below on T tokens of this shape.  A
 * workspace must be zero-filled before its first use (it holds the device
 * status word and the fused decode kernel's grid-barrier counter, which
 * carry state from one call to the next); after that, pass it unchanged to
 * every call of this shape, on one stream. */
size_t moe_workspace_size(const bitmoe_moe_shape_t* shape, int64_t T);

/*
 * Router: logits l[t,e] = sum_i x[t,i] w_router[e,i] + b_router[e] in fp32;
 * softmax over the E experts; the k largest logits (descending, equal
 * logits -> lower expert index) give topk_ids [T, kt] int32; topk_w [T, kt]
 * fp32 are their softmax probabilities, renormalised to sum 1 if
 * shape->renormalize, followed (n_shared = 1) by the shared expert, id E with
 * weight 1.  x [T, d] bf16.  logits_out [T, E] fp32 may be NULL.  T = 0 is a
 * no-op.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35 (the router picks
 * a few of 256 experts per token).
 */
bitmoe_status_t moe_route(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape, const float* w_router,
                          const float* b_router, int32_t* topk_ids, float* topk_w, float* logits_out,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Token -> expert grouping (the dispatch step of the mixture-of-experts
 * kernels).  Row r = t*kt + j of topk_ids is placed at
 * position inv_rows[r]; sorted_rows[p] = r; expert e owns positions
 * [expert_offsets[e], expert_offsets[e+1]); inside one expert the rows keep
 * ascending r (a stable counting sort, so the result is unique).  With
 * Et = E + n_shared bank entries: expert_offsets [Et+1], sorted_rows [T*kt],
 * inv_rows [T*kt], all int32.  Rows whose id is outside [0, Et) are left out
 * (inv_rows[r] = -1) and flag BITMOE_ERR_DEVICE_CHECK in the device status
 * word.  The workspace supplies the counting sort's scratch.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35 (each token goes
 * to six of 256 routed experts) and 06:11 (dedicated kernels for mixture-of-
 * experts routing); "Recursive_SI's First Model Unveiled!", section "Inference
 * Kernel" (kernels for MoE operations).
 */
bitmoe_status_t moe_permute(const int32_t* topk_ids, int64_t T, const bitmoe_moe_shape_t* shape,
                            int32_t* expert_offsets, int32_t* sorted_rows, int32_t* inv_rows, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Expert FFNs of every grouped row: for position p holding row r = t*kt + j of
 * expert e, a = Wg[e] x[t], u = Wu[e] x[t], h = a / (1 + exp(-a)) * u and
 * y_rows[p] = Wd[e] h (fp32 [T*kt, d], sorted order), with int4 weights
 * dequantised group by group.  expert_offsets / sorted_rows are moe_permute's.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35 and 06:11.
 */
bitmoe_status_t moe_expert_ffn_int4(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape,
                                    const bitmoe_moe_weights_t* weights, const int32_t* expert_offsets,
                                    const int32_t* sorted_rows, float* y_rows, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Gate-weighted combine into the residual:
 * out_f32[t,c] = residual[t,c] + sum_{j=0}^{kt-1} topk_w[t,j] * y_rows[inv_rows[t*kt+j], c]
 * summed in ascending j in fp32; out [T, d] bf16 = round-to-nearest-even of
 * out_f32.  out_f32 may be NULL.  out may alias residual.  y_rows [T*kt, d]
 * fp32 in grouped order (moe_expert_ffn_int4's output); inv_rows and topk_w
 * [T*kt]; residual [T, d] bf16; all 16-byte aligned except inv_rows / topk_w.
 * A row whose inv_rows entry is negative (left out by moe_permute) adds
 * nothing.  No workspace.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35 (a token's output
 * is the mix of the experts the router chose for it) and 06:11 (mixture-of-
 * experts kernels); "Recursive_SI's First Model Unveiled!", section "Inference
 * Kernel" (kernels for MoE operations).  The gate-weighted sum is the plain
 * reading of a top-k mixture; the pages print no formula.
 */
bitmoe_status_t moe_combine(const float* y_rows, const int32_t* inv_rows, const float* topk_w,
                            const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape, uint16_t* out,
                            float* out_f32, void* stream);

/*
 * The whole layer: route (unless forced), group, expert FFNs, combine.
 * residual may equal x.  forced_ids [T, kt] / forced_w [T, kt] (both or
 * neither) replace the router's choice; forced ids are range-checked on the
 * device.  topk_ids_out / topk_w_out are [T, kt].
 * topk_ids_out / topk_w_out / out_f32 may be NULL.  out may alias residual but
 * not x.  Batches of T <= 8 tokens run one fused decode kernel, other batches
 * with T*k < 512 routed rows the streaming kernels (both exact int4 x bf16 with
 * fp32 sums); T*k >= 512 runs the tcgen05 grouped GEMM (fp16 operands).
 * The projections carry the SwiGLU output h in fp16 (an exact hi + lo pair on the
 * fused and streaming paths, one fp16 value on the grouped-GEMM path, which keeps the
 * y rows in fp16 too): an h (or grouped-GEMM y) of magnitude 65520 or more, or a NaN,
 * cannot be represented and flags BITMOE_ERR_DEVICE_CHECK in the device status word
 * (inputs of the scale of a normalised residual stay far below it).
 * The fused decode kernel is one persistent launch of one CTA per SM whose
 * CTAs wait on each other; it runs only where the occupancy query says every
 * CTA of the grid can be resident at once (else the call takes the unfused
 * kernels), and it should not share the device with concurrent kernels that
 * occupy SMs for long (its CTAs would then wait, up to the 2 s limit, for SMs
 * that another kernel holds).
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35 (the MoE layer:
 * 256 routed experts, a few per token), 06:11 (kernels for low-bit projections
 * and mixture-of-experts routing) and 06:43 (the whole decode pass fused into
 * one launch on Apple GPUs; here one launch per layer step); "Recursive_SI's
 * First Model Unveiled!", section "Inference Kernel".
 */
bitmoe_status_t moe_forward(const uint16_t* x, const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                            const bitmoe_moe_weights_t* weights, const int32_t* forced_ids, const float* forced_w,
                            int32_t* topk_ids_out, float* topk_w_out, uint16_t* out, float* out_f32,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_forward with NVFP4 expert banks (see the NVFP4 section above):
 * shape->group must be 16 (the NVFP4 block), weights the packed NVFP4 banks
 * with their per-expert tensor scales; everything else as moe_forward.  Each
 * code times its E4M3 block scale is an exact fp16 weight, so the projections
 * keep exact products and fp32 sums; the tensor scale multiplies each
 * projection's fp32 result.  The kernels are those of moe_forward (fused
 * decode for T <= 8, streaming, tcgen05 grouped GEMM), each with an NVFP4
 * dequantisation step.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35, 06:43 and 07:15
 * (the four-bit NVFP builds); "Recursive_SI's First Model Unveiled!", section
 * "Quantization" (the NVFP4 model).
 */
bitmoe_status_t moe_forward_nvfp4(const uint16_t* x, const uint16_t* residual, int64_t T,
                                  const bitmoe_moe_shape_t* shape, const bitmoe_moe_weights_nvfp4_t* weights,
                                  const int32_t* forced_ids, const float* forced_w, int32_t* topk_ids_out,
                                  float* topk_w_out, uint16_t* out, float* out_f32, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* moe_expert_ffn_int4 over NVFP4 banks (shape->group == 16).  Source as
 * moe_forward_nvfp4. */
bitmoe_status_t moe_expert_ffn_nvfp4(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape,
                                     const bitmoe_moe_weights_nvfp4_t* weights, const int32_t* expert_offsets,
                                     const int32_t* sorted_rows, float* y_rows, void* workspace,
                                     size_t workspace_bytes, void* stream);

/*
 * One pre-norm layer step of a decode stack: xh = RMSNorm(residual) with unit
 * gain (y = x / sqrt(mean(x^2) + eps), fp32, rounded to bf16), then
 * out = residual + MoE(xh), as moe_forward(xh, residual, ...) computes it.
 * For T <= 8 the normalisation runs inside the fused decode kernel (no extra
 * launch); other T normalise first into xh_out (or the workspace).  xh_out
 * [T, d] bf16 may be NULL; out may alias residual.  Forced ids/gates as in
 * moe_forward.  Source: "Flint 40B : Best Mid Sized LLM", transcript 02:35
 * (the 49-layer decoder stack of MoE layers) and 03:36 (RMS norm is the
 * model's normalisation); the pre-norm placement, unit gain and eps are this
 * library's reading (the pages give none), and attention is left out.
 */
bitmoe_status_t moe_forward_prenorm(const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                                    const bitmoe_moe_weights_t* weights, float eps, const int32_t* forced_ids,
                                    const float* forced_w, int32_t* topk_ids_out, float* topk_w_out, uint16_t* xh_out,
                                    uint16_t* out, float* out_f32, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * A whole decode step of a stack of pre-norm MoE layers in ONE launch:
 *   for l = 0 .. n_layers-1:  residual = residual + MoE_l(RMSNorm(residual))
 * (each layer exactly as moe_forward_prenorm computes it, the residual kept in
 * bf16 and updated in place), then, when lm_packed is given,
 *   argmax[t] = the lowest v maximising (RMSNorm(residual) Wlm^T)[t, v]
 * with the LM head of lmhead_int4_gemv (logits [T, V] written when not NULL).
 * One persistent kernel: the layers follow each other through grid-wide
 * barriers instead of kernel boundaries, and each layer's router rows are
 * fetched while the previous layer's down projection runs.
 * residual [T, d] bf16 (in/out).  layers: a HOST array of n_layers weight sets
 * (each as moe_forward's; all layers share `shape`).  topk_ids_out (nullable)
 * [n_layers, T, kt] int32.  lm_packed: the packed [V, d] LM head or NULL (then
 * argmax / logits are unused).  The workspace is moe_stack_workspace_size()
 * bytes, zero-filled before its first use, as for moe_forward.
 * Supported: T <= 8, n_layers <= 64, the fused decode kernel's shapes (those
 * of moe_forward's batch <= 8 path), V % 16 == 0; otherwise
 * BITMOE_ERR_UNSUPPORTED, and the caller steps the layers with
 * moe_forward_prenorm, then bitmoe_rmsnorm and lmhead_int4_gemv, which compute
 * the same bits.  Its CTAs wait on each other across all layers, so it should
 * not share the device with concurrent kernels that occupy SMs for long.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 06:43 (a kernel that
 * fuses the entire decode pass into a single launch, written there for Apple
 * GPUs; here the 49-layer MoE stack and the output layer on B300) and 02:35
 * (the 49-layer decoder); "Recursive_SI's First Model Unveiled!", section
 * "Inference Kernel".
 */
size_t moe_stack_workspace_size(const bitmoe_moe_shape_t* shape, int64_t T);
bitmoe_status_t moe_stack_decode(uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                                 const bitmoe_moe_weights_t* layers, int64_t n_layers, float eps,
                                 const uint8_t* lm_packed, int64_t V, float* logits, int32_t* argmax,
                                 int32_t* topk_ids_out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------ LM head */

size_t lmhead_workspace_size(int64_t T, int64_t d, int64_t V);

/*
 * 4-bit output projection: logits[t,v] = sum_i Wlm[v,i] h[t,i] (fp32) and
 * argmax[t] = the lowest v reaching the maximum.  h [T, d] bf16; w_packed is
 * the packed [V, d] bank; logits [T, V] may be NULL.  V % 16 == 0, T <= 64,
 * d % 128 == 0 and small enough that a CTA stages min(T, 16) tokens beside two
 * 16-row weight tiles in shared memory (d = 2048: any T; d = 8192: T <= 4),
 * else BITMOE_ERR_UNSUPPORTED.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 03:36 and 05:39.
 */
bitmoe_status_t lmhead_int4_gemv(const uint16_t* h, int64_t T, int64_t d, int64_t V, int64_t group,
                                 const uint8_t* w_packed, float* logits, int32_t* argmax, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * The LM head over an NVFP4 matrix: logits[t,v] = sum_i Wlm[v,i] h[t,i] with
 * Wlm = e2m1(q) * e4m3(s) * tensor_scale (see the NVFP4 section above), fp32
 * sums, argmax as lmhead_int4_gemv.  w_packed is bitmoe_pack_nvfp4's [V, d]
 * bank; tensor_scale must be finite.  Shapes, workspace and errors as
 * lmhead_int4_gemv.  Each code times its block scale is an exact fp16 value,
 * so the products with the (exactly scaled) fp16 tokens are exact.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 03:36, 05:39 (the 4-bit
 * output layer) and 07:15 (the NVFP4 builds); "Recursive_SI's First Model
 * Unveiled!", section "Quantization".
 */
bitmoe_status_t lmhead_nvfp4_gemv(const uint16_t* h, int64_t T, int64_t d, int64_t V, const uint8_t* w_packed,
                                  float tensor_scale, float* logits, int32_t* argmax, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * lmhead_int4_gemv_static: the int4 LM head (lmhead_int4_gemv) without a workspace argument.
 * For callers that cannot allocate device memory: code embedded in another
 * runtime that owns all device memory through its own pool and hands this
 * library only the pointers of its inputs and outputs, or a per-token loop
 * that must not call cudaMalloc, which can synchronise the whole device.
 * The paper has no counterpart to this entry point.
 *
 * Arguments, layout and results are those of lmhead_int4_gemv.  The scratch
 * (a status word and one arg-max key per token) lives in a fixed 1 KiB device
 * array inside the library, which every GPU that loads the library holds until
 * the process exits; lmhead_static_scratch_bytes() returns its size.  T <= 64
 * (768 bytes of it); a larger T returns BITMOE_ERR_WORKSPACE before any launch.
 * The call allocates nothing.
 *
 * The first call on a device looks up the array's device address on that
 * device (the current device); make that first call before any stream
 * capture.  Each call clears the status word and the keys it uses itself.
 * All calls share the one array: two calls whose work overlaps on the GPU
 * (different streams, or different host threads, without ordering between
 * them) race and may return wrong arg-max values.  If a bounded device-side
 * wait runs out, every argmax[t] is set to -1.
 *
 * The looked-up address is kept for the life of the process: after
 * cudaDeviceReset() (or any teardown of the device's primary context) it is
 * stale, so do not call this entry point on a device that was reset.
 */
size_t lmhead_static_scratch_bytes(void);
bitmoe_status_t lmhead_int4_gemv_static(const uint16_t* h, int64_t T, int64_t d, int64_t V, int64_t group,
                                        const uint8_t* w_packed, float* logits, int32_t* argmax, void* stream);

/* RMSNorm with unit gain between stacked layers: y = x / sqrt(mean(x^2) + eps),
 * computed in fp32, rounded to bf16.  x, y [T, d] bf16, 16-byte aligned
 * (y may alias x); d % 8 == 0.  No workspace.
 * Source: "Flint 40B : Best Mid Sized LLM", transcript 03:36 (RMS norm is the
 * model's normalisation; the page names it for the attention heads).  Its
 * place before each stacked MoE layer, the unit gain and eps are this
 * library's reading: the pages give none of them. */
bitmoe_status_t bitmoe_rmsnorm(const uint16_t* x, int64_t T, int64_t d, float eps, uint16_t* y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BITMOE_H_ */
