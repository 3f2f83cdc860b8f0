// Combine into the residual, RMSNorm between stacked layers, weight packing.
#include "kernels.h"

namespace bitmoe {
namespace {

// out[t,c] = resid[t,c] + sum_j w[t,j] * y[inv[t*k+j], c]  (j ascending, fp32),
// bf16 = round-to-nearest-even of that fp32 value.  8 columns per thread.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, const uint16_t* resid, int d, int k,
                                                      uint16_t* out, float* __restrict__ out_f32) {
  pdl_enter();
  const int t = blockIdx.y;
  for (int c8 = (blockIdx.x * blockDim.x + threadIdx.x) * 8; c8 < d; c8 += gridDim.x * blockDim.x * 8) {
    // the residual, then each batch of 8 rows' positions and gates, then their y
    // pieces, are requested together; the sum still runs in ascending j
    const uint4 r = *reinterpret_cast<const uint4*>(resid + (size_t)t * d + c8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      int pos[8];
      float wj[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + i;
        pos[i] = j < k ? inv[(size_t)t * k + j] : -1;
        wj[i] = j < k ? w[(size_t)t * k + j] : 0.f;
      }
      float4 y0[8], y1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (pos[i] >= 0) {
          y0[i] = *reinterpret_cast<const float4*>(y + (size_t)pos[i] * d + c8);
          y1[i] = *reinterpret_cast<const float4*>(y + (size_t)pos[i] * d + c8 + 4);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (pos[i] < 0) continue;
        acc[0] = fmaf(wj[i], y0[i].x, acc[0]);
        acc[1] = fmaf(wj[i], y0[i].y, acc[1]);
        acc[2] = fmaf(wj[i], y0[i].z, acc[2]);
        acc[3] = fmaf(wj[i], y0[i].w, acc[3]);
        acc[4] = fmaf(wj[i], y1[i].x, acc[4]);
        acc[5] = fmaf(wj[i], y1[i].y, acc[5]);
        acc[6] = fmaf(wj[i], y1[i].z, acc[6]);
        acc[7] = fmaf(wj[i], y1[i].w, acc[7]);
      }
    }
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
    float o[8];
    uint32_t ob[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(rw[i] << 16) + acc[2 * i];
      o[2 * i + 1] = __uint_as_float(rw[i] & 0xffff0000u) + acc[2 * i + 1];
      ob[i] = (uint32_t)float_to_bf16_bits(o[2 * i]) | ((uint32_t)float_to_bf16_bits(o[2 * i + 1]) << 16);
    }
    if (out_f32) {
      *reinterpret_cast<float4*>(out_f32 + (size_t)t * d + c8) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(out_f32 + (size_t)t * d + c8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * d + c8) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// The same combine reading fp16 y rows (grouped-GEMM path).
__global__ void __launch_bounds__(256) combine_f16_kernel(const __half* __restrict__ y, const int32_t* __restrict__ inv,
                                                          const float* __restrict__ w, const uint16_t* resid, int d,
                                                          int k, uint16_t* out, float* __restrict__ out_f32) {
  pdl_enter();
  const int t = blockIdx.y;
  for (int c8 = (blockIdx.x * blockDim.x + threadIdx.x) * 8; c8 < d; c8 += gridDim.x * blockDim.x * 8) {
    // as combine_kernel: residual, positions and gates, then y pieces requested together
    const uint4 r = *reinterpret_cast<const uint4*>(resid + (size_t)t * d + c8);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {
      int pos[8];
      float wj[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = j0 + i;
        pos[i] = j < k ? inv[(size_t)t * k + j] : -1;
        wj[i] = j < k ? w[(size_t)t * k + j] : 0.f;
      }
      uint4 yv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (pos[i] >= 0) yv[i] = *reinterpret_cast<const uint4*>(y + (size_t)pos[i] * d + c8);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (pos[i] < 0) continue;
        const uint32_t yw[4] = {yv[i].x, yv[i].y, yv[i].z, yv[i].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&yw[q]));
          acc[2 * q] = fmaf(wj[i], f.x, acc[2 * q]);
          acc[2 * q + 1] = fmaf(wj[i], f.y, acc[2 * q + 1]);
        }
      }
    }
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
    float o[8];
    uint32_t ob[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(rw[i] << 16) + acc[2 * i];
      o[2 * i + 1] = __uint_as_float(rw[i] & 0xffff0000u) + acc[2 * i + 1];
      ob[i] = (uint32_t)float_to_bf16_bits(o[2 * i]) | ((uint32_t)float_to_bf16_bits(o[2 * i + 1]) << 16);
    }
    if (out_f32) {
      *reinterpret_cast<float4*>(out_f32 + (size_t)t * d + c8) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(out_f32 + (size_t)t * d + c8 + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * d + c8) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// y = x / sqrt(mean(x^2) + eps) with unit gain; fp32 sums in a fixed tree order.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* x, int d, float eps, uint16_t* y) {
  pdl_enter();
  __shared__ float part[8];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * d;
  float ss = 0.f;
  for (int c8 = threadIdx.x * 8; c8 < d; c8 += blockDim.x * 8) {
    const uint4 r = *reinterpret_cast<const uint4*>(xr + c8);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(rw[i] << 16), b = __uint_as_float(rw[i] & 0xffff0000u);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += part[i];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  for (int c8 = threadIdx.x * 8; c8 < d; c8 += blockDim.x * 8) {
    const uint4 r = *reinterpret_cast<const uint4*>(xr + c8);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
    uint32_t ob[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = __uint_as_float(rw[i] << 16) * inv, b = __uint_as_float(rw[i] & 0xffff0000u) * inv;
      ob[i] = (uint32_t)float_to_bf16_bits(a) | ((uint32_t)float_to_bf16_bits(b) << 16);
    }
    // each thread rewrites only the elements it read, so y may alias x
    *reinterpret_cast<uint4*>(y + (size_t)t * d + c8) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
}

// Canonical int4 bank -> packed tiles.  Packed word (row r, group G, quarter c)
// holds the 8 values at columns 32G + 8c + m, m = 0..7: value m = 2p at bits
// [4p, 4p+4), value m = 2p+1 at bits [16+4p, 20+4p).  Inside a 128-column
// chunk the words are ordered [row][quarter][group-in-chunk], then the chunk's
// fp16 scales as [row][group-in-chunk].
__global__ void pack_int4_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ scale, int64_t n_mats,
                                 int64_t rows, int64_t K, uint8_t* __restrict__ packed) {
  const int64_t nch = K / kChunkK;
  const int64_t tiles = n_mats * (rows / kTileRows);
  const int64_t items = tiles * nch * kTileRows;  // one (tile, chunk, row) per thread
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(it % kTileRows);
    const int64_t ch = (it / kTileRows) % nch;
    const int64_t tile = it / (kTileRows * nch);
    const int64_t grow = tile * kTileRows + r;  // row index over the whole bank (n_mats * rows)
    const uint8_t* qrow = q + grow * (K / 2);
    const uint16_t* srow = scale + grow * (K / kGroup);
    uint8_t* chunk = packed + tile * tile_bytes(K) + ch * kChunkBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t words[4];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int64_t k0 = (ch * 4 + gg) * kGroup + c * 8;
        const uint32_t src = *reinterpret_cast<const uint32_t*>(qrow + k0 / 2);
        uint32_t wv = 0;
#pragma unroll
        for (int pr = 0; pr < 4; ++pr) {
          const uint32_t byte = (src >> (8 * pr)) & 0xffu;
          wv |= (byte & 0xfu) << (4 * pr);
          wv |= (byte >> 4) << (16 + 4 * pr);
        }
        words[gg] = wv;
      }
      *reinterpret_cast<uint4*>(chunk + (r * 4 + c) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    }
    uint16_t* sdst = reinterpret_cast<uint16_t*>(chunk + kChunkQBytes + r * 8);
#pragma unroll
    for (int gg = 0; gg < 4; ++gg) sdst[gg] = srow[ch * 4 + gg];
  }
}

// NVFP4 bank -> packed tiles: the same geometry as the int4 tiles.  A lane's
// word holds the 8 codes of columns 8c .. 8c+7 of a 32-column group in their
// canonical byte order (byte j = columns 8c+2j and 8c+2j+1, low nibble first),
// which is the pair order the hardware E2M1 conversion gives fragment register
// j; the chunk's scale block is each row's 8 E4M3 bytes.
__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ scale, int64_t n_mats,
                                  int64_t rows, int64_t K, uint8_t* __restrict__ packed) {
  const int64_t nch = K / kChunkK;
  const int64_t tiles = n_mats * (rows / kTileRows);
  const int64_t items = tiles * nch * kTileRows;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(it % kTileRows);
    const int64_t ch = (it / kTileRows) % nch;
    const int64_t tile = it / (kTileRows * nch);
    const int64_t grow = tile * kTileRows + r;
    const uint8_t* qrow = q + grow * (K / 2);
    const uint8_t* srow = scale + grow * (K / kFp4Block);
    uint8_t* chunk = packed + tile * tile_bytes(K) + ch * kChunkBytes;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t words[4];
#pragma unroll
      for (int gg = 0; gg < 4; ++gg)
        words[gg] = *reinterpret_cast<const uint32_t*>(qrow + ((ch * 4 + gg) * kGroup + c * 8) / 2);
      *reinterpret_cast<uint4*>(chunk + (r * 4 + c) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    }
    uint8_t* sdst = chunk + kChunkQBytes + r * 8;
#pragma unroll
    for (int b = 0; b < 8; ++b) sdst[b] = srow[ch * 8 + b];
  }
}

}  // namespace

cudaError_t launch_combine(const float* y_rows, const int32_t* inv, const float* w, const uint16_t* resid, int T,
                           int d, int k, uint16_t* out, float* out_f32, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  // 64 threads x 8 columns per CTA, one token per grid row (at most 65535 rows per launch)
  for (int t0 = 0; t0 < T; t0 += 65535) {
    const int n = T - t0 < 65535 ? T - t0 : 65535;
    const size_t o = (size_t)t0 * d;
    const cudaError_t e = launch_pdl(combine_kernel, dim3(ceil_div(d, 512), n), dim3(64), 0, s, y_rows,
                                     inv + (size_t)t0 * k, w + (size_t)t0 * k, resid + o, d, k, out + o,
                                     out_f32 ? out_f32 + o : nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_f16(const __half* y_rows, const int32_t* inv, const float* w, const uint16_t* resid, int T,
                               int d, int k, uint16_t* out, float* out_f32, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  for (int t0 = 0; t0 < T; t0 += 65535) {
    const int n = T - t0 < 65535 ? T - t0 : 65535;
    const size_t o = (size_t)t0 * d;
    const cudaError_t e = launch_pdl(combine_f16_kernel, dim3(ceil_div(d, 512), n), dim3(64), 0, s, y_rows,
                                     inv + (size_t)t0 * k, w + (size_t)t0 * k, resid + o, d, k, out + o,
                                     out_f32 ? out_f32 + o : nullptr);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t* x, int T, int d, float eps, uint16_t* y, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (cudaError_t e_ = launch_pdl(rmsnorm_kernel, dim3(T), dim3(256), 0, s, x, d, eps, y)) return e_;
  return cudaGetLastError();
}

cudaError_t launch_pack_int4(const uint8_t* q, const uint16_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                             uint8_t* packed, cudaStream_t s) {
  const int64_t items = n_mats * (rows / kTileRows) * (K / kChunkK) * kTileRows;
  if (items == 0) return cudaSuccess;
  const int grid = (int)(ceil_div<int64_t>(items, 256) < 148 * 64 ? ceil_div<int64_t>(items, 256) : 148 * 64);
  pack_int4_kernel<<<grid, 256, 0, s>>>(q, scale, n_mats, rows, K, packed);
  return cudaGetLastError();
}

}  // namespace bitmoe

namespace bitmoe {

cudaError_t launch_pack_nvfp4(const uint8_t* q, const uint8_t* scale, int64_t n_mats, int64_t rows, int64_t K,
                              uint8_t* packed, cudaStream_t s) {
  const int64_t items = n_mats * (rows / kTileRows) * (K / kChunkK) * kTileRows;
  if (items == 0) return cudaSuccess;
  const int grid = (int)(ceil_div<int64_t>(items, 256) < 148 * 64 ? ceil_div<int64_t>(items, 256) : 148 * 64);
  pack_nvfp4_kernel<<<grid, 256, 0, s>>>(q, scale, n_mats, rows, K, packed);
  return cudaGetLastError();
}

}  // namespace bitmoe
