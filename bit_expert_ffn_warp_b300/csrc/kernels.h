// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace bitmoe {

// ---------------------------------------------------------------- routing (route.cu)
// Router logits.  From kRouterTcMinT tokens on the product runs on tcgen05 and needs
// w_split (router_split_bytes: the router rows split into three bf16 parts per call);
// with fewer tokens, or w_split null, the mma.sync kernels run.  st: status word for
// the tcgen05 kernel's bounded waits.
constexpr int kRouterTcMinT = 256;
bool router_uses_tc(int T);
size_t router_split_bytes(int E, int d);
cudaError_t launch_router_logits(const uint16_t* x, int T, int d, int E, const float* w_router,
                                 const float* b_router, float* logits, uint16_t* w_split, DevStatus* st,
                                 cudaStream_t s);
// ids / w rows of k + n_shared entries: the k routed experts, then (n_shared = 1)
// the shared expert, bank entry E, with weight 1.
cudaError_t launch_topk_gates(const float* logits, int T, int E, int k, int renorm, int n_shared, int32_t* ids,
                              float* w, cudaStream_t s);
cudaError_t launch_forced_select(const int32_t* forced_ids, const float* forced_w, int T, int E, int k,
                                 int32_t* ids, float* w, DevStatus* st, cudaStream_t s);

// ---------------------------------------------------------------- permutation (permute.cu)
// Scratch needed by launch_permute (bytes), for R = T*k rows.
size_t permute_scratch_bytes(int64_t R, int E);
// Stable counting sort of R ids into E buckets; also writes blk_prefix[E+1]:
// exclusive prefix of ceil(count_e / kTokBlock).
cudaError_t launch_permute(const int32_t* ids, int R, int E, int32_t* offsets, int32_t* sorted_rows, int32_t* inv,
                           int32_t* blk_prefix, void* scratch, DevStatus* st, cudaStream_t s);
// blk_prefix from offsets only (standalone expert-FFN entry point).
cudaError_t launch_blk_prefix(const int32_t* offsets, int E, int32_t* blk_prefix, cudaStream_t s);

// ---------------------------------------------------------------- expert FFN (ffn.cu)
struct FfnArgs {
  const uint16_t* x;  // [T, d] bf16
  int T, d, I, E, k;
  const uint8_t* gate;  // packed banks
  const uint8_t* up;
  const uint8_t* down;
  const float* gate_ts;        // NVFP4 banks: tensor scale per bank entry; null = int4 banks
  const float* up_ts;
  const float* down_ts;
  const int32_t* offsets;      // [E+1]
  const int32_t* sorted_rows;  // [R]
  const int32_t* blk_prefix;   // [E+1]
  __half* h_hi;                // [R, I]
  __half* h_lo;                // [R, I]
  float* y_rows;               // [R, d]
  DevStatus* st;
};
cudaError_t launch_ffn_up(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_ffn_down(const FfnArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- prefill grouped GEMMs (prefill.cu)
// tcgen05 path for many routed rows: writes fp16 h into a.h_hi and y rows
// into y16 (fp16) when given, else a.y_rows (fp32); nb_prefix [E+1 + T*k/128
// + E + 1] and xs [T*k, d] fp16 (the routed rows in grouped order) are scratch.
bool prefill_eligible(int d, int I);
cudaError_t launch_prefill_ffn(const FfnArgs& a, int32_t* nb_prefix, __half* xs, __half* y16, cudaStream_t s);
cudaError_t launch_combine_f16(const __half* y_rows, const int32_t* inv, const float* w, const uint16_t* resid, int T,
                               int d, int k, uint16_t* out, float* out_f32, cudaStream_t s);

// ---------------------------------------------------------------- fused decode step (decode.cu)
struct DecodeLaunch {
  const uint16_t* x;
  const uint16_t* resid;
  int T, d, E, k, I, renorm;  // E, k: routed experts and routed experts per token
  int n_shared;               // 1: bank entry E is a shared expert every token uses with weight 1
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
  const float* gate_ts;       // NVFP4 banks: tensor scale per bank entry; null = int4 banks
  const float* up_ts;
  const float* down_ts;
  const int32_t* forced_ids;  // null = route; else [T, k + n_shared]
  const float* forced_w;
  uint16_t* out;
  float* out_f32;   // may be null
  int32_t* ids_out;  // may be null
  float* w_out;      // may be null
  float* logits;     // scratch [T, E]
  __half* h_hi;      // scratch [T*k, I]
  __half* h_lo;
  unsigned* gbar;    // grid-barrier words (arrivals, epoch), arrivals 0 at launch
  DevStatus* st;
  int pdl;           // launch with programmatic dependent launch
  int prenorm;       // x is the residual: the layer runs on RMSNorm(x) (unit gain, eps)
  float eps;
  uint16_t* xh_out;  // optional [T, d] copy of RMSNorm(x)
};
bool decode_fused_eligible(int T, int d, int E, int k, int I, int n_shared);
// Optional phase-timestamp buffer for the fused decode kernel (null = off).
extern void* g_trace_buf;
extern size_t g_trace_bytes;
cudaError_t launch_decode_fused(const DecodeLaunch& L, cudaStream_t s);
// Whole decode stack in one launch: n_layers pre-norm layers (L.prenorm = 1, x,
// resid and out all the residual, updated in place), then (lm_w != null)
// RMSNorm, the LM head over V rows and the arg-max.  The weights of L are unused;
// layer l's come from layers[l].
struct StackLayer {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
};
bool decode_stack_eligible(int T, int d, int E, int k, int I, int n_shared, int n_layers, int V);
cudaError_t launch_decode_stack(const DecodeLaunch& L, const StackLayer* layers, int n_layers, const uint8_t* lm_w,
                                int V, float* lm_logits, unsigned long long* lm_keys, int32_t* lm_argmax,
                                cudaStream_t s);

// ---------------------------------------------------------------- combine / norm / pack (misc.cu)
cudaError_t launch_combine(const float* y_rows, const int32_t* inv, const float* w, const uint16_t* resid, int T,
                           int d, int k, uint16_t* out, float* out_f32, cudaStream_t s);
cudaError_t launch_rmsnorm(const uint16_t* x, int T, int d, float eps, uint16_t* y, cudaStream_t s);
cudaError_t launch_pack_int4(const uint8_t* q, const uint16_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                             uint8_t* packed, cudaStream_t s);
cudaError_t launch_pack_nvfp4(const uint8_t* q, const uint8_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                              uint8_t* packed, cudaStream_t s);

// ---------------------------------------------------------------- LM head (lmhead.cu)
size_t lmhead_scratch_bytes(int T);
// Whether one launch can stage min(T, 16) tokens and at least two weight tiles of width d.
bool lmhead_supported(int d, int T);
cudaError_t launch_lmhead(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float* logits,
                          int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s);
// The same over a packed NVFP4 bank with tensor scale ts.
cudaError_t launch_lmhead_nvfp4(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float ts,
                                float* logits, int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s);

// ---------------------------------------------------------------- C-ABI helpers (api.cu)
// Records e as the thread's last CUDA error (read by bitmoe_last_cuda_error) and maps it to a status.
bitmoe_status_t api_cuda_status(cudaError_t e);

// ---------------------------------------------------------------- attention decode step (attn.cu)
constexpr int kAttnHeadDim = 128;  // head dimension the kernels are built for
constexpr int kAttnGroup = 8;      // query heads per key/value head
constexpr int kAttnPart = 4 + kAttnHeadDim;  // floats per (query head, split) partial result
constexpr int kAttnMaxSplits = 128;          // splits of the attended span per key/value head, at most
// How the split kernel cuts `span` attended positions for nkv key/value heads: `chunk`
// positions per CTA (a multiple of 64) and `nsplit` <= kAttnMaxSplits CTAs per head,
// about two CTAs per SM in all.
struct AttnPlan {
  int64_t chunk;
  int nsplit;
};
AttnPlan attn_plan(int64_t span, int nkv);
struct AttnLaunch {
  const uint16_t* x;      // [d] bf16 (the normalised residual; unused with prenorm)
  const uint16_t* resid;  // [d] bf16
  int prenorm;            // 1: x = bf16(RMSNorm(resid)) with eps, formed in the projection
  int64_t pos;            // the token's position (its cache row)
  int d, nq, nkv;
  int64_t window;         // 0: the whole context
  int rope;
  double theta;
  float eps;
  const uint8_t* wqkv;    // packed int4 [(nq + 2 nkv) * 128, d]
  const uint8_t* wo;      // packed int4 [d, nq * 128]
  const float* sinks;     // [nq] or null
  uint16_t* k_cache;      // [nkv, max_len, 128] bf16
  uint16_t* v_cache;
  int64_t max_len;
  uint16_t* out;          // [d] bf16
  float* out_f32;         // [d] or null
  // scratch
  float* qkv;             // [(nq + 2 nkv) * 128]
  float* part;            // [nq * kAttnMaxSplits * kAttnPart]
  uint16_t* attn;         // [nq * 128] bf16
};
cudaError_t launch_attn_decode(const AttnLaunch& L, cudaStream_t s);

}  // namespace bitmoe
