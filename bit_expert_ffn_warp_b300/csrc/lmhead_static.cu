// LM head with its scratch in a fixed array inside the library, for callers
// that cannot allocate device memory.  The arithmetic is the LM-head kernel of
// lmhead.cu, unchanged; only where its scratch lives differs.
#include <mutex>

#include "kernels.h"

using namespace bitmoe;

namespace {

// Scratch of one call: the device status word (256 B, as at the head of every
// workspace) followed by one 64-bit arg-max key per token.  T <= 64 needs
// 256 + 64 * 8 = 768 bytes; the array is 1 KiB.  Every GPU that loads the
// library holds it until the process exits.
constexpr size_t kStaticScratchBytes = 1024;
constexpr size_t kStatusBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_lmhead_scratch[kStaticScratchBytes];

// Device address of g_lmhead_scratch on each device, looked up once per device.
// In host code the array's name is only a host-side stand-in, so kernels get
// this address, never the name.
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lmhead_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

// A bounded wait that ran out leaves no valid arg-max: mark every token -1 so
// that the caller, who has no workspace to read the status from, sees it.
__global__ void status_to_argmax_kernel(const DevStatus* st, int T, int32_t* argmax) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T && st->code != 0) argmax[t] = -1;
}

}  // namespace

extern "C" {

size_t lmhead_static_scratch_bytes(void) { return kStaticScratchBytes; }

bitmoe_status_t lmhead_int4_gemv_static(const uint16_t* h, int64_t T, int64_t d, int64_t V, int64_t group,
                                        const uint8_t* w_packed, float* logits, int32_t* argmax, void* stream) {
  if (T < 0 || d <= 0 || V <= 0) return BITMOE_ERR_INVALID_ARG;
  if (group != kGroup || d % kChunkK || V % kTileRows || d > 16384 || V > (int64_t(1) << 30))
    return BITMOE_ERR_UNSUPPORTED;
  // the scratch this call needs must fit the fixed array
  if (T > 64 || kStatusBytes + lmhead_scratch_bytes((int)T) > kStaticScratchBytes) return BITMOE_ERR_WORKSPACE;
  if (T == 0) return BITMOE_OK;
  if (!lmhead_supported((int)d, (int)T)) return BITMOE_ERR_UNSUPPORTED;
  const uintptr_t a16 = 15u;
  if (!h || !w_packed || !argmax || (reinterpret_cast<uintptr_t>(h) & a16) ||
      (reinterpret_cast<uintptr_t>(w_packed) & a16))
    return BITMOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  void* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  // the array keeps the previous call's contents: the status word must start
  // at zero (launch_lmhead zeroes the arg-max keys itself)
  if (e == cudaSuccess) e = cudaMemsetAsync(scratch, 0, kStatusBytes, s);
  DevStatus* st = static_cast<DevStatus*>(scratch);
  if (e == cudaSuccess)
    e = launch_lmhead(h, (int)T, (int)d, (int)V, w_packed, logits, argmax, static_cast<char*>(scratch) + kStatusBytes,
                      st, s);
  if (e == cudaSuccess) {
    status_to_argmax_kernel<<<1, 64, 0, s>>>(st, (int)T, argmax);
    e = cudaGetLastError();
  }
  return api_cuda_status(e);
}

}  // extern "C"
