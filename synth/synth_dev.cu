// Device twin of the uniform generators in synth/__init__.py.
//
// Draws the same bits as the numpy code: the i-th SplitMix64 output from a
// stream key (Steele, Lea and Flood, OOPSLA 2014), mapped to packed int4
// bytes, to fp16 scales RNE_fp16(0.005 + 0.015 * u) or to E4M3 block-scale
// bytes 0x58 + (h >> 60).  It exists so that the
// multi-GB weight banks can be written straight into HBM; it holds none of the
// MoE layer's arithmetic.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t hash_word(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ull) * 0x9E3779B97F4A7C15ull);
}

__global__ void fill_int4_kernel(uint8_t* dst, uint64_t count, uint64_t key, uint64_t start) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < count; b += stride) {
    uint64_t g = start + b;
    uint64_t w = hash_word(key, g >> 3);
    dst[b] = (uint8_t)(w >> (8 * (g & 7)));
  }
}

__global__ void fill_scales_kernel(uint16_t* dst, uint64_t count, uint64_t key, uint64_t start) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    uint64_t h = hash_word(key, start + i);
    double u = (double)(h >> 11) * 0x1p-53;
    double v = __dadd_rn(0.005, __dmul_rn(0.015, u));
    __half hv = __double2half(v);
    dst[i] = __half_as_ushort(hv);
  }
}

// E4M3 block-scale bytes: 0x58 + (h >> 60).
__global__ void fill_e4m3_kernel(uint8_t* dst, uint64_t count, uint64_t key, uint64_t start) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    dst[i] = (uint8_t)(0x58u + (uint32_t)(hash_word(key, start + i) >> 60));
}

int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 148ull * 32) g = 148ull * 32;
  if (g == 0) g = 1;
  return (int)g;
}

}  // namespace

extern "C" int synth_fill_int4_bytes(void* dst, uint64_t count, uint64_t key, uint64_t start, void* stream) {
  if (count == 0) return 0;
  if (dst == nullptr) return (int)cudaErrorInvalidValue;
  fill_int4_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>((uint8_t*)dst, count, key, start);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_f16_scales(void* dst, uint64_t count, uint64_t key, uint64_t start, void* stream) {
  if (count == 0) return 0;
  if (dst == nullptr) return (int)cudaErrorInvalidValue;
  fill_scales_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>((uint16_t*)dst, count, key, start);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_e4m3_scales(void* dst, uint64_t count, uint64_t key, uint64_t start, void* stream) {
  if (count == 0) return 0;
  if (dst == nullptr) return (int)cudaErrorInvalidValue;
  fill_e4m3_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>((uint8_t*)dst, count, key, start);
  return (int)cudaGetLastError();
}
