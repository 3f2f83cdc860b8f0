// C ABI of the int4 MoE layer and LM head: argument checks, workspace layout
// and the launch sequence of each entry point.  See include/bitmoe.h.
#include <string.h>

#include <cmath>

#include "kernels.h"

using namespace bitmoe;

namespace {

thread_local int g_last_cuda_error = 0;

bitmoe_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return BITMOE_OK;
  g_last_cuda_error = (int)e;
  return BITMOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxRows = int64_t(1) << 22;  // T*k limit (int32 positions with headroom)

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Bank entries (routed + shared) and rows per token (routed + shared).
int64_t bank_experts(const bitmoe_moe_shape_t* sh) { return sh->E + sh->n_shared; }
int64_t rows_per_token(const bitmoe_moe_shape_t* sh) { return sh->k + sh->n_shared; }

// Workspace carve-up shared by every MoE entry point.
struct MoeWs {
  DevStatus* st;
  int32_t* ids;
  float* w;
  float* logits;
  int32_t* offsets;
  int32_t* sorted_rows;
  int32_t* inv;
  int32_t* blk_prefix;
  void* perm_scratch;
  __half* h_hi;
  __half* h_lo;
  float* y_rows;
  __half* xs;         // [R, d] routed rows in grouped order, fp16 (grouped-GEMM path)
  int32_t* nb_prefix;  // [E+1] 128-row blocks per expert, then the block list (grouped-GEMM path)
  uint16_t* xh;        // [T, d] bf16 RMSNorm of the residual (pre-norm step, unfused path)
  uint16_t* w_split;   // [3E, d] bf16 parts of the router rows (tcgen05 router, many tokens; else null)
  size_t total;
};

MoeWs moe_layout(const bitmoe_moe_shape_t* sh, int64_t T, void* base) {
  const int64_t R = T * rows_per_token(sh), Et = bank_experts(sh);
  char* p = static_cast<char*>(base);
  size_t off = 0;
  MoeWs w;
  auto take = [&](size_t bytes) {
    char* q = p ? p + off : nullptr;
    off += align256(bytes);
    return q;
  };
  w.st = reinterpret_cast<DevStatus*>(take(256));
  w.ids = reinterpret_cast<int32_t*>(take((size_t)R * 4));
  w.w = reinterpret_cast<float*>(take((size_t)R * 4));
  w.logits = reinterpret_cast<float*>(take((size_t)T * sh->E * 4));
  w.offsets = reinterpret_cast<int32_t*>(take((size_t)(Et + 1) * 4));
  w.sorted_rows = reinterpret_cast<int32_t*>(take((size_t)R * 4));
  w.inv = reinterpret_cast<int32_t*>(take((size_t)R * 4));
  w.blk_prefix = reinterpret_cast<int32_t*>(take((size_t)(Et + 1) * 4));
  w.perm_scratch = take(permute_scratch_bytes(R, (int)Et));
  w.h_hi = reinterpret_cast<__half*>(take((size_t)R * sh->I * 2));
  w.h_lo = reinterpret_cast<__half*>(take((size_t)R * sh->I * 2));
  w.y_rows = reinterpret_cast<float*>(take((size_t)R * sh->d * 4));
  w.xs = reinterpret_cast<__half*>(take((size_t)R * sh->d * 2));
  // prefix of 128-row expert blocks [E+1], then the blocks widest first [R/128 + E]
  w.nb_prefix = reinterpret_cast<int32_t*>(take((size_t)(Et + 1) * 4 + (size_t)(R / 128 + Et + 1) * 4));
  w.xh = reinterpret_cast<uint16_t*>(take((size_t)T * sh->d * 2));
  w.w_split = (sh->k > 0 && router_uses_tc((int)T))
                  ? reinterpret_cast<uint16_t*>(take(router_split_bytes((int)sh->E, (int)sh->d)))
                  : nullptr;
  w.total = off;
  return w;
}

bitmoe_status_t check_shape(const bitmoe_moe_shape_t* sh, int64_t T) {
  if (sh == nullptr || T < 0) return BITMOE_ERR_INVALID_ARG;
  if (sh->d <= 0 || sh->E < 0 || sh->k < 0 || sh->I <= 0) return BITMOE_ERR_INVALID_ARG;
  // k = 0 routed experts is a dense layer: the shared expert alone, no router
  if (sh->k == 0 && sh->n_shared != 1) return BITMOE_ERR_INVALID_ARG;
  if (sh->k > 0 && sh->E == 0) return BITMOE_ERR_INVALID_ARG;
  if (sh->n_shared < 0 || sh->n_shared > 1) return BITMOE_ERR_INVALID_ARG;
  if (sh->k > sh->E || rows_per_token(sh) > kMaxK) return BITMOE_ERR_INVALID_ARG;
  if (sh->group != kGroup && sh->group != kFp4Block) return BITMOE_ERR_UNSUPPORTED;  // int4 or NVFP4 banks
  if (sh->d % kChunkK || sh->I % kChunkK) return BITMOE_ERR_UNSUPPORTED;
  if (bank_experts(sh) > kMaxE || sh->d > 16384 || sh->I > 16384) return BITMOE_ERR_UNSUPPORTED;
  if (T * rows_per_token(sh) > kMaxRows) return BITMOE_ERR_UNSUPPORTED;
  return BITMOE_OK;
}

bitmoe_status_t check_ws(const bitmoe_moe_shape_t* sh, int64_t T, void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned16(ws)) return BITMOE_ERR_WORKSPACE;
  if (ws_bytes < moe_layout(sh, T, nullptr).total) return BITMOE_ERR_WORKSPACE;
  return BITMOE_OK;
}


// A layer's weights in either format (tensor scales null: int4 banks).
struct LayerW {
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
  const float* gate_ts;
  const float* up_ts;
  const float* down_ts;
  bool nvfp4() const { return gate_ts != nullptr; }
};

LayerW layer_w(const bitmoe_moe_weights_t* wt) {
  return LayerW{wt->gate, wt->up, wt->down, wt->w_router, wt->b_router, nullptr, nullptr, nullptr};
}

LayerW layer_w(const bitmoe_moe_weights_nvfp4_t* wt) {
  return LayerW{wt->gate, wt->up, wt->down, wt->w_router, wt->b_router, wt->gate_scale, wt->up_scale, wt->down_scale};
}

// The shape's scale group names the format: 32 for int4 calls, 16 for NVFP4 ones.
bitmoe_status_t check_format(const bitmoe_moe_shape_t* sh, bool nvfp4) {
  return sh->group == (nvfp4 ? kFp4Block : kGroup) ? BITMOE_OK : BITMOE_ERR_UNSUPPORTED;
}

// nvfp4: the call takes NVFP4 banks, whose three tensor-scale arrays must be given.
bitmoe_status_t check_layer(const LayerW& wt, bool need_router, bool nvfp4) {
  if (!wt.gate || !wt.up || !wt.down) return BITMOE_ERR_INVALID_ARG;
  if (!aligned16(wt.gate) || !aligned16(wt.up) || !aligned16(wt.down)) return BITMOE_ERR_INVALID_ARG;
  if (need_router && (!wt.w_router || !aligned16(wt.w_router))) return BITMOE_ERR_INVALID_ARG;
  if (nvfp4 && (!wt.gate_ts || !wt.up_ts || !wt.down_ts)) return BITMOE_ERR_INVALID_ARG;
  return BITMOE_OK;
}

bitmoe_status_t check_weights(const bitmoe_moe_weights_t* wt, bool need_router) {
  return wt ? check_layer(layer_w(wt), need_router, false) : BITMOE_ERR_INVALID_ARG;
}

FfnArgs ffn_args(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* sh, const LayerW& wt,
                 const int32_t* offsets, const int32_t* sorted_rows, const int32_t* blk_prefix, const MoeWs& w,
                 float* y_rows) {
  FfnArgs a;
  a.x = x;
  a.T = (int)T;
  a.d = (int)sh->d;
  a.I = (int)sh->I;
  a.E = (int)bank_experts(sh);
  a.k = (int)rows_per_token(sh);
  a.gate = wt.gate;
  a.up = wt.up;
  a.down = wt.down;
  a.gate_ts = wt.gate_ts;
  a.up_ts = wt.up_ts;
  a.down_ts = wt.down_ts;
  a.offsets = offsets;
  a.sorted_rows = sorted_rows;
  a.blk_prefix = blk_prefix;
  a.h_hi = w.h_hi;
  a.h_lo = w.h_lo;
  a.y_rows = y_rows;
  a.st = w.st;
  return a;
}

// Expert FFNs of the grouped rows: the tcgen05 grouped GEMMs when the batch
// routes more than 512 rows (a dense contraction per expert), else the
// streaming mma.sync kernels.
// y16 (optional): write fp16 y rows there instead of fp32 a.y_rows (grouped-GEMM path only).
bool uses_grouped_gemm(const FfnArgs& a) { return (int64_t)a.T * a.k >= 512 && prefill_eligible(a.d, a.I); }

cudaError_t run_expert_ffn(const FfnArgs& a, const MoeWs& w, __half* y16, cudaStream_t s) {
  if (uses_grouped_gemm(a)) return launch_prefill_ffn(a, w.nb_prefix, w.xs, y16, s);
  cudaError_t e = launch_ffn_up(a, s);
  if (e == cudaSuccess) e = launch_ffn_down(a, s);
  return e;
}

}  // namespace

namespace bitmoe {
bitmoe_status_t api_cuda_status(cudaError_t e) { return cuda_status(e); }
}  // namespace bitmoe

namespace {

// One layer step.  prenorm: x is the residual and the layer runs on RMSNorm(x) (unit gain,
// eps), optionally copied to xh_out.
bitmoe_status_t forward_impl(const uint16_t* x, const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                             const LayerW& weights, const int32_t* forced_ids, const float* forced_w,
                             int32_t* topk_ids_out, float* topk_w_out, uint16_t* out, float* out_f32,
                             void* workspace, size_t workspace_bytes, void* stream, int prenorm, float eps,
                             uint16_t* xh_out, bool nvfp4) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if ((st = check_format(shape, nvfp4)) != BITMOE_OK) return st;
  if (T == 0) return BITMOE_OK;
  if ((forced_ids == nullptr) != (forced_w == nullptr)) return BITMOE_ERR_INVALID_ARG;
  if ((st = check_layer(weights, forced_ids == nullptr && shape->k > 0, nvfp4)) != BITMOE_OK) return st;
  if (!x || !residual || !out || !aligned16(x) || !aligned16(residual) || !aligned16(out) ||
      (out_f32 && !aligned16(out_f32)) || (xh_out && !aligned16(xh_out)) || !(eps >= 0.f))
    return BITMOE_ERR_INVALID_ARG;
  if ((st = check_ws(shape, T, workspace, workspace_bytes)) != BITMOE_OK) return st;
  const MoeWs w = moe_layout(shape, T, workspace);
  cudaStream_t s = (cudaStream_t)stream;
  const int Ti = (int)T, d = (int)shape->d, E = (int)shape->E, k = (int)shape->k;
  const int ns = (int)shape->n_shared, Et = E + ns, kt = k + ns;
  cudaError_t e;
  if (decode_fused_eligible(Ti, d, E, k, (int)shape->I, ns)) {
    DecodeLaunch L;
    L.x = x;
    L.resid = residual;
    L.T = Ti;
    L.d = d;
    L.E = E;
    L.k = k;
    L.I = (int)shape->I;
    L.renorm = shape->renormalize;
    L.n_shared = ns;
    L.gate = weights.gate;
    L.up = weights.up;
    L.down = weights.down;
    L.w_router = weights.w_router;
    L.b_router = weights.b_router;
    L.gate_ts = weights.gate_ts;
    L.up_ts = weights.up_ts;
    L.down_ts = weights.down_ts;
    L.forced_ids = forced_ids;
    L.forced_w = forced_w;
    L.out = out;
    L.out_f32 = out_f32;
    L.ids_out = topk_ids_out;
    L.w_out = topk_w_out;
    L.logits = w.logits;
    L.h_hi = w.h_hi;
    L.h_lo = w.h_lo;
    L.gbar = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(w.st) + 64);
    L.st = w.st;
    L.pdl = 1;
    L.prenorm = prenorm;
    L.eps = eps;
    L.xh_out = xh_out;
    e = launch_decode_fused(L, s);
    if (e != cudaErrorNotSupported) return cuda_status(e);
    (void)cudaGetLastError();
  }
  if (prenorm) {  // the unfused path normalises first, into xh_out or the workspace
    uint16_t* xh = xh_out ? xh_out : w.xh;
    e = launch_rmsnorm(x, Ti, d, eps, xh, s);
    if (e != cudaSuccess) return cuda_status(e);
    x = xh;
  }
  if (forced_ids) {
    e = launch_forced_select(forced_ids, forced_w, Ti, Et, kt, w.ids, w.w, w.st, s);
  } else {
    e = k > 0 ? launch_router_logits(x, Ti, d, E, weights.w_router, weights.b_router, w.logits, w.w_split, w.st, s)
              : cudaSuccess;
    if (e == cudaSuccess) e = launch_topk_gates(w.logits, Ti, E, k, shape->renormalize, ns, w.ids, w.w, s);
  }
  if (e == cudaSuccess)
    e = launch_permute(w.ids, Ti * kt, Et, w.offsets, w.sorted_rows, w.inv, w.blk_prefix, w.perm_scratch, w.st, s);
  const FfnArgs a = ffn_args(x, T, shape, weights, w.offsets, w.sorted_rows, w.blk_prefix, w, w.y_rows);
  // the grouped-GEMM path keeps y in fp16 (half the bytes through HBM twice), except
  // with a shared expert: its rows enter the combine with weight 1, not a gate of
  // about 1/k, and fp16's rounding of y (half an ulp is 1/64 at |y| in [32, 64))
  // would then reach the output undamped
  __half* y16 = (uses_grouped_gemm(a) && ns == 0) ? reinterpret_cast<__half*>(w.y_rows) : nullptr;
  if (e == cudaSuccess) e = run_expert_ffn(a, w, y16, s);
  if (e == cudaSuccess) {
    if (y16) e = launch_combine_f16(y16, w.inv, w.w, residual, Ti, d, kt, out, out_f32, s);
    else e = launch_combine(w.y_rows, w.inv, w.w, residual, Ti, d, kt, out, out_f32, s);
  }
  if (e == cudaSuccess && topk_ids_out)
    e = cudaMemcpyAsync(topk_ids_out, w.ids, (size_t)T * kt * 4, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && topk_w_out)
    e = cudaMemcpyAsync(topk_w_out, w.w, (size_t)T * kt * 4, cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

bitmoe_status_t expert_ffn_impl(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape, const LayerW& weights,
                                const int32_t* expert_offsets, const int32_t* sorted_rows, float* y_rows,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !expert_offsets || !sorted_rows || !y_rows || !aligned16(x) || !aligned16(y_rows))
    return BITMOE_ERR_INVALID_ARG;
  bitmoe_status_t st = check_ws(shape, T, workspace, workspace_bytes);
  if (st != BITMOE_OK) return st;
  const MoeWs w = moe_layout(shape, T, workspace);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_blk_prefix(expert_offsets, (int)bank_experts(shape), w.blk_prefix, s);
  const FfnArgs a = ffn_args(x, T, shape, weights, expert_offsets, sorted_rows, w.blk_prefix, w, y_rows);
  if (e == cudaSuccess) e = run_expert_ffn(a, w, nullptr, s);
  return cuda_status(e);
}

}  // namespace

namespace {

// Workspace carve-up of the attention decode step.
struct AttnWs {
  DevStatus* st;
  float* qkv;
  float* part;
  uint16_t* attn;
  size_t total;
};

bitmoe_status_t check_attn_shape(const bitmoe_attn_shape_t* sh) {
  if (sh == nullptr || sh->d <= 0 || sh->n_q_heads <= 0 || sh->n_kv_heads <= 0 || sh->max_len <= 0 ||
      sh->window < 0 || !(sh->eps >= 0.f) || (sh->rope && !(sh->rope_theta > 0.0)))
    return BITMOE_ERR_INVALID_ARG;
  if (sh->head_dim != kAttnHeadDim || sh->n_q_heads != kAttnGroup * sh->n_kv_heads || sh->d % kChunkK ||
      sh->d > 16384 || sh->n_q_heads * kAttnHeadDim > 16384 || sh->max_len > (int64_t(1) << 31))
    return BITMOE_ERR_UNSUPPORTED;
  return BITMOE_OK;
}

AttnWs attn_layout(const bitmoe_attn_shape_t* sh, void* base) {
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* q = p ? p + off : nullptr;
    off += align256(bytes);
    return q;
  };
  const int64_t nq = sh->n_q_heads, nkv = sh->n_kv_heads, hd = kAttnHeadDim;
  AttnWs w;
  w.st = reinterpret_cast<DevStatus*>(take(256));
  w.qkv = reinterpret_cast<float*>(take((size_t)(nq + 2 * nkv) * hd * 4));
  w.part = reinterpret_cast<float*>(take((size_t)nq * kAttnMaxSplits * kAttnPart * 4));
  w.attn = reinterpret_cast<uint16_t*>(take((size_t)nq * hd * 2));
  w.total = off;
  return w;
}

// One attention decode step: x the block input (with prenorm, x = residual and the
// projection normalises it).
bitmoe_status_t attn_step(const uint16_t* x, const uint16_t* residual, int prenorm, int64_t pos,
                          const bitmoe_attn_shape_t* shape, const bitmoe_attn_weights_t* weights,
                          uint16_t* k_cache, uint16_t* v_cache, uint16_t* out, float* out_f32, void* workspace,
                          size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_attn_shape(shape);
  if (st != BITMOE_OK) return st;
  if (pos < 0 || pos >= shape->max_len || !weights) return BITMOE_ERR_INVALID_ARG;
  if (!x || !residual || !out || !k_cache || !v_cache || !weights->wqkv || !weights->wo)
    return BITMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(weights->wqkv) || !aligned16(weights->wo) || (out_f32 && !aligned16(out_f32)))
    return BITMOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < attn_layout(shape, nullptr).total)
    return BITMOE_ERR_WORKSPACE;
  const AttnWs w = attn_layout(shape, workspace);
  AttnLaunch L;
  L.x = x;
  L.resid = residual;
  L.prenorm = prenorm;
  L.pos = pos;
  L.d = (int)shape->d;
  L.nq = (int)shape->n_q_heads;
  L.nkv = (int)shape->n_kv_heads;
  L.window = shape->window;
  L.rope = shape->rope ? 1 : 0;
  L.theta = shape->rope_theta;
  L.eps = shape->eps;
  L.wqkv = weights->wqkv;
  L.wo = weights->wo;
  L.sinks = weights->sinks;
  L.k_cache = k_cache;
  L.v_cache = v_cache;
  L.max_len = shape->max_len;
  L.out = out;
  L.out_f32 = out_f32;
  L.qkv = w.qkv;
  L.part = w.part;
  L.attn = w.attn;
  return cuda_status(launch_attn_decode(L, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

const char* bitmoe_status_string(bitmoe_status_t status) {
  switch (status) {
    case BITMOE_OK: return "ok";
    case BITMOE_ERR_INVALID_ARG: return "invalid argument";
    case BITMOE_ERR_UNSUPPORTED: return "unsupported shape";
    case BITMOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case BITMOE_ERR_CUDA: return "CUDA launch error";
    case BITMOE_ERR_TIMEOUT: return "device wait timed out";
    case BITMOE_ERR_DEVICE_CHECK: return "device-side input check failed";
  }
  return "unknown status";
}

int bitmoe_last_cuda_error(void) { return g_last_cuda_error; }

bitmoe_status_t bitmoe_set_trace_buffer(void* device_buf, size_t bytes) {
  if ((device_buf == nullptr) != (bytes == 0)) return BITMOE_ERR_INVALID_ARG;
  if (device_buf && (reinterpret_cast<uintptr_t>(device_buf) & 7u)) return BITMOE_ERR_INVALID_ARG;
  g_trace_buf = device_buf;
  g_trace_bytes = bytes;
  return BITMOE_OK;
}

const char* bitmoe_version(void) { return "bitmoe 0.1 (sm_103a)"; }

size_t bitmoe_packed_int4_bytes(int64_t n_mats, int64_t rows, int64_t K, int64_t group) {
  if (n_mats <= 0 || rows <= 0 || K <= 0 || group != kGroup || rows % kTileRows || K % kChunkK) return 0;
  return (size_t)n_mats * (size_t)(rows / kTileRows) * (size_t)tile_bytes(K);
}

bitmoe_status_t bitmoe_pack_int4(const uint8_t* q, const uint16_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                                 int64_t group, uint8_t* packed, void* stream) {
  if (!q || !scale || !packed) return BITMOE_ERR_INVALID_ARG;
  if (bitmoe_packed_int4_bytes(n_mats, rows, K, group) == 0) return BITMOE_ERR_UNSUPPORTED;
  if (!aligned16(packed) || (reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(scale) & 1u))
    return BITMOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_int4(q, scale, n_mats, rows, K, packed, (cudaStream_t)stream));
}

size_t bitmoe_packed_nvfp4_bytes(int64_t n_mats, int64_t rows, int64_t K) {
  return bitmoe_packed_int4_bytes(n_mats, rows, K, kGroup);  // same geometry: 4.5 bits per weight
}

bitmoe_status_t bitmoe_pack_nvfp4(const uint8_t* q, const uint8_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                                  uint8_t* packed, void* stream) {
  if (!q || !scale || !packed) return BITMOE_ERR_INVALID_ARG;
  if (bitmoe_packed_nvfp4_bytes(n_mats, rows, K) == 0) return BITMOE_ERR_UNSUPPORTED;
  if (!aligned16(packed) || (reinterpret_cast<uintptr_t>(q) & 3u)) return BITMOE_ERR_INVALID_ARG;
  return cuda_status(launch_pack_nvfp4(q, scale, n_mats, rows, K, packed, (cudaStream_t)stream));
}

bitmoe_status_t bitmoe_get_device_status(void* workspace, int clear, int32_t* status_out, void* stream) {
  if (!workspace || !status_out) return BITMOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  DevStatus hs;
  cudaError_t e = cudaMemcpyAsync(&hs, workspace, sizeof(hs), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    e = cudaMemsetAsync(workspace, 0, 256, s);  // status word and grid-barrier words
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return cuda_status(e);
  *status_out = hs.code;
  return BITMOE_OK;
}

size_t moe_workspace_size(const bitmoe_moe_shape_t* shape, int64_t T) {
  if (check_shape(shape, T) != BITMOE_OK) return 0;
  return moe_layout(shape, T, nullptr).total;
}

bitmoe_status_t moe_route(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape, const float* w_router,
                          const float* b_router, int32_t* topk_ids, float* topk_w, float* logits_out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if (T == 0) return BITMOE_OK;
  const bool scored = shape->k > 0;  // k = 0: a dense layer, only the shared expert's column
  if (!x || (scored && !w_router) || !topk_ids || !topk_w) return BITMOE_ERR_INVALID_ARG;
  if (!aligned16(x) || (scored && !aligned16(w_router))) return BITMOE_ERR_INVALID_ARG;
  if ((st = check_ws(shape, T, workspace, workspace_bytes)) != BITMOE_OK) return st;
  const MoeWs w = moe_layout(shape, T, workspace);
  cudaStream_t s = (cudaStream_t)stream;
  float* logits = logits_out ? logits_out : w.logits;
  cudaError_t e = scored ? launch_router_logits(x, (int)T, (int)shape->d, (int)shape->E, w_router, b_router, logits,
                                              w.w_split, w.st, s)
                         : cudaSuccess;
  if (e == cudaSuccess)
    e = launch_topk_gates(logits, (int)T, (int)shape->E, (int)shape->k, shape->renormalize, (int)shape->n_shared,
                          topk_ids, topk_w, s);
  return cuda_status(e);
}

bitmoe_status_t moe_permute(const int32_t* topk_ids, int64_t T, const bitmoe_moe_shape_t* shape,
                            int32_t* expert_offsets, int32_t* sorted_rows, int32_t* inv_rows, void* workspace,
                            size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if (!expert_offsets || (T > 0 && (!topk_ids || !sorted_rows || !inv_rows))) return BITMOE_ERR_INVALID_ARG;
  if ((st = check_ws(shape, T, workspace, workspace_bytes)) != BITMOE_OK) return st;
  const MoeWs w = moe_layout(shape, T, workspace);
  return cuda_status(launch_permute(topk_ids, (int)(T * rows_per_token(shape)), (int)bank_experts(shape),
                                    expert_offsets, sorted_rows, inv_rows, w.blk_prefix, w.perm_scratch, w.st,
                                    (cudaStream_t)stream));
}

bitmoe_status_t moe_expert_ffn_int4(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape,
                                    const bitmoe_moe_weights_t* weights, const int32_t* expert_offsets,
                                    const int32_t* sorted_rows, float* y_rows, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if ((st = check_format(shape, false)) != BITMOE_OK) return st;
  if (T == 0) return BITMOE_OK;
  if ((st = check_weights(weights, false)) != BITMOE_OK) return st;
  return expert_ffn_impl(x, T, shape, layer_w(weights), expert_offsets, sorted_rows, y_rows, workspace,
                         workspace_bytes, stream);
}

bitmoe_status_t moe_expert_ffn_nvfp4(const uint16_t* x, int64_t T, const bitmoe_moe_shape_t* shape,
                                     const bitmoe_moe_weights_nvfp4_t* weights, const int32_t* expert_offsets,
                                     const int32_t* sorted_rows, float* y_rows, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if ((st = check_format(shape, true)) != BITMOE_OK) return st;
  if (T == 0) return BITMOE_OK;
  if (!weights || (st = check_layer(layer_w(weights), false, true)) != BITMOE_OK) return BITMOE_ERR_INVALID_ARG;
  return expert_ffn_impl(x, T, shape, layer_w(weights), expert_offsets, sorted_rows, y_rows, workspace,
                         workspace_bytes, stream);
}

bitmoe_status_t moe_combine(const float* y_rows, const int32_t* inv_rows, const float* topk_w,
                            const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape, uint16_t* out,
                            float* out_f32, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if (T == 0) return BITMOE_OK;
  if (!y_rows || !inv_rows || !topk_w || !residual || !out) return BITMOE_ERR_INVALID_ARG;
  if (!aligned16(y_rows) || !aligned16(residual) || !aligned16(out) || (out_f32 && !aligned16(out_f32)))
    return BITMOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y_rows, inv_rows, topk_w, residual, (int)T, (int)shape->d,
                                    (int)rows_per_token(shape), out, out_f32, (cudaStream_t)stream));
}

bitmoe_status_t moe_forward(const uint16_t* x, const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                            const bitmoe_moe_weights_t* weights, const int32_t* forced_ids, const float* forced_w,
                            int32_t* topk_ids_out, float* topk_w_out, uint16_t* out, float* out_f32,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(x, residual, T, shape, weights ? layer_w(weights) : LayerW{}, forced_ids, forced_w, topk_ids_out,
                      topk_w_out, out, out_f32, workspace, workspace_bytes, stream, 0, 0.f, nullptr, false);
}

bitmoe_status_t moe_forward_nvfp4(const uint16_t* x, const uint16_t* residual, int64_t T,
                                  const bitmoe_moe_shape_t* shape, const bitmoe_moe_weights_nvfp4_t* weights,
                                  const int32_t* forced_ids, const float* forced_w, int32_t* topk_ids_out,
                                  float* topk_w_out, uint16_t* out, float* out_f32, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return forward_impl(x, residual, T, shape, weights ? layer_w(weights) : LayerW{}, forced_ids, forced_w, topk_ids_out,
                      topk_w_out, out, out_f32, workspace, workspace_bytes, stream, 0, 0.f, nullptr, true);
}

bitmoe_status_t moe_forward_prenorm(const uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                                    const bitmoe_moe_weights_t* weights, float eps, const int32_t* forced_ids,
                                    const float* forced_w, int32_t* topk_ids_out, float* topk_w_out, uint16_t* xh_out,
                                    uint16_t* out, float* out_f32, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return forward_impl(residual, residual, T, shape, weights ? layer_w(weights) : LayerW{}, forced_ids, forced_w,
                      topk_ids_out, topk_w_out, out, out_f32, workspace, workspace_bytes, stream, 1, eps, xh_out,
                      false);
}

size_t moe_stack_workspace_size(const bitmoe_moe_shape_t* shape, int64_t T) {
  if (check_shape(shape, T) != BITMOE_OK) return 0;
  return moe_layout(shape, T, nullptr).total + 256;  // + the arg-max keys
}

bitmoe_status_t moe_stack_decode(uint16_t* residual, int64_t T, const bitmoe_moe_shape_t* shape,
                                 const bitmoe_moe_weights_t* layers, int64_t n_layers, float eps,
                                 const uint8_t* lm_packed, int64_t V, float* logits, int32_t* argmax,
                                 int32_t* topk_ids_out, void* workspace, size_t workspace_bytes, void* stream) {
  bitmoe_status_t st = check_shape(shape, T);
  if (st != BITMOE_OK) return st;
  if ((st = check_format(shape, false)) != BITMOE_OK) return st;
  if (!layers || n_layers < 1 || !(eps >= 0.f) || V < 0) return BITMOE_ERR_INVALID_ARG;
  if (T == 0) return BITMOE_OK;
  if (!residual || !aligned16(residual)) return BITMOE_ERR_INVALID_ARG;
  for (int64_t l = 0; l < n_layers; ++l)
    if ((st = check_weights(&layers[l], shape->k > 0)) != BITMOE_OK) return st;
  if (lm_packed && (!argmax || !aligned16(lm_packed) || V <= 0 || (logits && !aligned16(logits))))
    return BITMOE_ERR_INVALID_ARG;
  if (!decode_stack_eligible((int)T, (int)shape->d, (int)shape->E, (int)shape->k, (int)shape->I,
                             (int)shape->n_shared, (int)n_layers, lm_packed ? (int)V : 0) ||
      V > (int64_t(1) << 30))
    return BITMOE_ERR_UNSUPPORTED;
  if (!workspace || !aligned16(workspace) || workspace_bytes < moe_stack_workspace_size(shape, T))
    return BITMOE_ERR_WORKSPACE;
  const MoeWs w = moe_layout(shape, T, workspace);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + w.total);
  StackLayer tab[64];
  for (int64_t l = 0; l < n_layers; ++l)
    tab[l] = StackLayer{layers[l].gate, layers[l].up, layers[l].down, layers[l].w_router, layers[l].b_router};
  DecodeLaunch L = {};
  L.x = residual;
  L.resid = residual;
  L.out = residual;
  L.T = (int)T;
  L.d = (int)shape->d;
  L.E = (int)shape->E;
  L.k = (int)shape->k;
  L.I = (int)shape->I;
  L.renorm = shape->renormalize;
  L.n_shared = (int)shape->n_shared;
  L.ids_out = topk_ids_out;
  L.logits = w.logits;
  L.h_hi = w.h_hi;
  L.h_lo = w.h_lo;
  L.gbar = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(w.st) + 64);
  L.st = w.st;
  L.pdl = 1;
  L.prenorm = 1;
  L.eps = eps;
  return cuda_status(launch_decode_stack(L, tab, (int)n_layers, lm_packed, (int)V, logits, keys, argmax,
                                         (cudaStream_t)stream));
}

size_t attn_workspace_size(const bitmoe_attn_shape_t* shape) {
  if (check_attn_shape(shape) != BITMOE_OK) return 0;
  return attn_layout(shape, nullptr).total;
}

bitmoe_status_t attn_decode_step(const uint16_t* x, const uint16_t* residual, int64_t pos,
                                 const bitmoe_attn_shape_t* shape, const bitmoe_attn_weights_t* weights,
                                 uint16_t* k_cache, uint16_t* v_cache, uint16_t* out, float* out_f32,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!x) return BITMOE_ERR_INVALID_ARG;
  return attn_step(x, residual, 0, pos, shape, weights, k_cache, v_cache, out, out_f32, workspace, workspace_bytes,
                   stream);
}

bitmoe_status_t attn_decode_step_prenorm(const uint16_t* residual, int64_t pos, const bitmoe_attn_shape_t* shape,
                                         const bitmoe_attn_weights_t* weights, uint16_t* k_cache,
                                         uint16_t* v_cache, uint16_t* out, float* out_f32, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return attn_step(residual, residual, 1, pos, shape, weights, k_cache, v_cache, out, out_f32, workspace,
                   workspace_bytes, stream);
}

size_t lmhead_workspace_size(int64_t T, int64_t d, int64_t V) {
  if (T < 0 || d <= 0 || V <= 0) return 0;
  return 256 + align256(lmhead_scratch_bytes((int)T));
}

bitmoe_status_t lmhead_int4_gemv(const uint16_t* h, int64_t T, int64_t d, int64_t V, int64_t group,
                                 const uint8_t* w_packed, float* logits, int32_t* argmax, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (T < 0 || d <= 0 || V <= 0) return BITMOE_ERR_INVALID_ARG;
  if (group != kGroup || d % kChunkK || V % kTileRows || T > 64 || d > 16384 || V > (int64_t(1) << 30))
    return BITMOE_ERR_UNSUPPORTED;
  if (T == 0) return BITMOE_OK;
  if (!lmhead_supported((int)d, (int)T)) return BITMOE_ERR_UNSUPPORTED;
  if (!h || !w_packed || !argmax || !aligned16(h) || !aligned16(w_packed)) return BITMOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < lmhead_workspace_size(T, d, V))
    return BITMOE_ERR_WORKSPACE;
  DevStatus* st = static_cast<DevStatus*>(workspace);
  void* keys = static_cast<char*>(workspace) + 256;
  return cuda_status(launch_lmhead(h, (int)T, (int)d, (int)V, w_packed, logits, argmax, keys, st,
                                   (cudaStream_t)stream));
}

bitmoe_status_t lmhead_nvfp4_gemv(const uint16_t* h, int64_t T, int64_t d, int64_t V, const uint8_t* w_packed,
                                  float tensor_scale, float* logits, int32_t* argmax, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (T < 0 || d <= 0 || V <= 0 || !std::isfinite(tensor_scale)) return BITMOE_ERR_INVALID_ARG;
  if (d % kChunkK || V % kTileRows || T > 64 || d > 16384 || V > (int64_t(1) << 30)) return BITMOE_ERR_UNSUPPORTED;
  if (T == 0) return BITMOE_OK;
  if (!lmhead_supported((int)d, (int)T)) return BITMOE_ERR_UNSUPPORTED;
  if (!h || !w_packed || !argmax || !aligned16(h) || !aligned16(w_packed)) return BITMOE_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) || workspace_bytes < lmhead_workspace_size(T, d, V))
    return BITMOE_ERR_WORKSPACE;
  DevStatus* st = static_cast<DevStatus*>(workspace);
  void* keys = static_cast<char*>(workspace) + 256;
  return cuda_status(launch_lmhead_nvfp4(h, (int)T, (int)d, (int)V, w_packed, tensor_scale, logits, argmax, keys,
                                         st, (cudaStream_t)stream));
}

bitmoe_status_t bitmoe_rmsnorm(const uint16_t* x, int64_t T, int64_t d, float eps, uint16_t* y, void* stream) {
  if (T < 0 || d <= 0 || d % 8 || !(eps >= 0.f)) return BITMOE_ERR_INVALID_ARG;
  if (T == 0) return BITMOE_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return BITMOE_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm(x, (int)T, (int)d, eps, y, (cudaStream_t)stream));
}

}  // extern "C"
