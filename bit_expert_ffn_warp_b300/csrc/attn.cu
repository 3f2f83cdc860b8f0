// One decode step of the attention layer that sits beside each MoE layer: grouped-query
// attention over a bf16 key/value cache with a sliding window (or the whole context),
// per-head RMS norm on queries and keys, rotary encoding and learned sinks.
//
// "Flint 40B : Best Mid Sized LLM", transcript 03:05 (32 query heads, 4 key/value
// heads of 128; 35 of the mixture layers attend over a window of 513 tokens with rotary
// encoding, the rest over the whole context without it) and 03:36 (per-head RMS norm on
// queries and keys, learned attention sinks); 06:11 (dedicated attention kernels).
//
// For one token the step is a chain of weight and cache streams:
//   1. q|k|v = Wqkv x          the int4 projection rows stacked, on the LM-head GEMV kernel
//   2. prep                    RMS norm per head, rotation, k and v appended to the cache
//   3. split                   the window cut into 256-position chunks; a CTA per
//                              (key/value head, chunk) runs the 8 query heads that share
//                              the key/value head (one warp each) over its chunk with an
//                              online softmax, and leaves (max, sum, partial output)
//   4. combine                 per query head the chunks and the sink merge into one
//                              output, rounded to bf16
//   5. y = Wo attn, out = residual + y
// Step 3 reads the window's keys and values once per key/value head (the 8 query heads
// of a group share each staged tile), so at long context it is the HBM-bound part.
#include <math.h>

#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kHd = kAttnHeadDim;  // 128
constexpr int kQPerKv = kAttnGroup;  // query heads per key/value head
constexpr int kTilePos = 32;         // positions per staged tile (one per lane)
constexpr int kRowPad = 8;           // bf16 padding per staged row (bank spread)
constexpr int kPrepThreads = 512;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// qkv [(nq + 2 nkv) * 128] fp32 -> q (normalised, rotated) fp32 [nq * 128]; the k row
// (normalised, rotated) and the v row go to cache row pos in bf16.  One warp per head;
// lane l holds elements l, l + 32, l + 64, l + 96, so both members of each rotated pair
// (i, i + 64) sit in the same lane.  The angles pos * theta^(-2i/128) are formed and
// rotated in fp64 (positions reach 10^5 radians), once per launch.
__global__ void __launch_bounds__(kPrepThreads) attn_prep_kernel(const float* __restrict__ qkv, int nq, int nkv,
                                                                 int64_t pos, int rope, double theta, float eps,
                                                                 float* __restrict__ q_out,
                                                                 uint16_t* __restrict__ k_cache,
                                                                 uint16_t* __restrict__ v_cache) {
  pdl_enter();
  __shared__ float cs[kHd / 2], sn[kHd / 2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (rope && tid < kHd / 2) {
    const double ang = (double)pos * pow(theta, -2.0 * (double)tid / (double)kHd);
    double s, c;
    sincos(ang, &s, &c);
    cs[tid] = (float)c;
    sn[tid] = (float)s;
  }
  __syncthreads();
  const size_t row = (size_t)pos * nkv;
  for (int h = warp; h < nq + 2 * nkv; h += kPrepThreads / 32) {
    const float* src = qkv + (size_t)h * kHd;
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = src[lane + 32 * i];
    if (h < nq + nkv) {  // q or k: RMS norm, then the rotation
      const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
      const float r = 1.0f / sqrtf(ss / (float)kHd + eps);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] *= r;
      if (rope) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {  // pairs (lane + 32i, lane + 32i + 64)
          const float c = cs[lane + 32 * i], s = sn[lane + 32 * i];
          const float a = v[i], b = v[i + 2];
          v[i] = a * c - b * s;
          v[i + 2] = a * s + b * c;
        }
      }
    }
    if (h < nq) {
#pragma unroll
      for (int i = 0; i < 4; ++i) q_out[(size_t)h * kHd + lane + 32 * i] = v[i];
    } else {
      uint16_t* dst = (h < nq + nkv) ? k_cache + (row + (h - nq)) * kHd : v_cache + (row + (h - nq - nkv)) * kHd;
#pragma unroll
      for (int i = 0; i < 4; ++i) dst[lane + 32 * i] = f2bf(v[i]);
    }
  }
}

struct SplitArgs {
  const float* q;          // [nq * 128] normalised, rotated
  const uint16_t* k_cache;  // [L, nkv, 128] bf16
  const uint16_t* v_cache;
  int nkv;
  int64_t lo, hi;          // positions lo .. hi - 1 are attended
  int chunk;               // positions per CTA
  float scale;             // 1 / sqrt(128)
  float* part;             // [nq][nchunks][kAttnPart]: max, sum, 2 unused, unnormalised output
  int nchunks;
};

// grid (nkv, nchunks), kQPerKv warps: warp w runs query head g * kQPerKv + w over the CTA's
// chunk, 32 positions at a time (one per lane for the scores), with an online softmax;
// lane l accumulates output dimensions 4l .. 4l + 3.
__global__ void __launch_bounds__(kQPerKv * 32) attn_split_kernel(const __grid_constant__ SplitArgs a) {
  pdl_enter();
  __shared__ __align__(16) float qs[kQPerKv][kHd];
  __shared__ __align__(16) uint16_t ks[kTilePos][kHd + kRowPad];
  __shared__ __align__(16) uint16_t vs[kTilePos][kHd + kRowPad];
  const int g = blockIdx.x, c = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = g * kQPerKv + warp;
  for (int i = tid; i < kQPerKv * kHd; i += kQPerKv * 32) qs[i / kHd][i % kHd] = a.q[(size_t)g * kQPerKv * kHd + i];
  const int64_t c0 = a.lo + (int64_t)c * a.chunk;
  const int64_t c1 = min(a.hi, c0 + a.chunk);
  float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t t0 = c0; t0 < c1; t0 += kTilePos) {
    __syncthreads();  // the previous tile is consumed (and, first time, q is staged)
    // stage 32 key and value rows: 2 x 32 x 16 uint4, two of each per thread
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int idx = tid + rep * kQPerKv * 32;  // 0 .. 511
      const int r = idx >> 4, q16 = idx & 15;
      const int64_t j = t0 + r;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (j < c1) {
        const size_t off = ((size_t)j * a.nkv + g) * kHd + (size_t)q16 * 8;
        kv = *reinterpret_cast<const uint4*>(a.k_cache + off);
        vv = *reinterpret_cast<const uint4*>(a.v_cache + off);
      }
      *reinterpret_cast<uint4*>(&ks[r][q16 * 8]) = kv;
      *reinterpret_cast<uint4*>(&vs[r][q16 * 8]) = vv;
    }
    __syncthreads();
    // score of position t0 + lane
    float s = 0.f;
#pragma unroll 4
    for (int d8 = 0; d8 < kHd / 8; ++d8) {
      const uint4 kk = *reinterpret_cast<const uint4*>(&ks[lane][d8 * 8]);
      const float4 qa = *reinterpret_cast<const float4*>(&qs[warp][d8 * 8]);
      const float4 qb = *reinterpret_cast<const float4*>(&qs[warp][d8 * 8 + 4]);
      s = fmaf(qa.x, bf16f((uint16_t)(kk.x & 0xffffu)), s);
      s = fmaf(qa.y, bf16f((uint16_t)(kk.x >> 16)), s);
      s = fmaf(qa.z, bf16f((uint16_t)(kk.y & 0xffffu)), s);
      s = fmaf(qa.w, bf16f((uint16_t)(kk.y >> 16)), s);
      s = fmaf(qb.x, bf16f((uint16_t)(kk.z & 0xffffu)), s);
      s = fmaf(qb.y, bf16f((uint16_t)(kk.z >> 16)), s);
      s = fmaf(qb.z, bf16f((uint16_t)(kk.w & 0xffffu)), s);
      s = fmaf(qb.w, bf16f((uint16_t)(kk.w >> 16)), s);
    }
    const bool valid = t0 + lane < c1;
    s = valid ? s * a.scale : -INFINITY;
    const float mt = warp_max(s);
    const float mn = fmaxf(m, mt);
    const float corr = expf(m - mn);  // m = -inf at the first tile: corr = 0
    const float p = valid ? expf(s - mn) : 0.f;
    l = l * corr + warp_sum(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] *= corr;
    m = mn;
    const int nv = (int)min((int64_t)kTilePos, c1 - t0);
    for (int jj = 0; jj < nv; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const uint2 vv = *reinterpret_cast<const uint2*>(&vs[jj][lane * 4]);
      o[0] = fmaf(pj, bf16f((uint16_t)(vv.x & 0xffffu)), o[0]);
      o[1] = fmaf(pj, bf16f((uint16_t)(vv.x >> 16)), o[1]);
      o[2] = fmaf(pj, bf16f((uint16_t)(vv.y & 0xffffu)), o[2]);
      o[3] = fmaf(pj, bf16f((uint16_t)(vv.y >> 16)), o[3]);
    }
  }
  float* dst = a.part + ((size_t)h * a.nchunks + c) * kAttnPart;
  if (lane == 0) {
    dst[0] = m;
    dst[1] = l;
  }
  *reinterpret_cast<float4*>(dst + 4 + lane * 4) = make_float4(o[0], o[1], o[2], o[3]);
}

// One CTA per query head, one thread per output dimension: the chunks' partial results
// and the sink merge into out = sum_c e^(m_c - M) o_c / (e^(sink - M) + sum_c e^(m_c - M) l_c).
__global__ void __launch_bounds__(kHd) attn_combine_kernel(const float* __restrict__ part, int nchunks,
                                                          const float* __restrict__ sinks,
                                                          uint16_t* __restrict__ attn) {
  pdl_enter();
  const int h = blockIdx.x, d = threadIdx.x;
  const float* ph = part + (size_t)h * nchunks * kAttnPart;
  const float sink = sinks ? sinks[h] : -INFINITY;
  float M = sink;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, ph[(size_t)c * kAttnPart]);
  float L = sinks ? expf(sink - M) : 0.f, acc = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const float* pc = ph + (size_t)c * kAttnPart;
    const float w = expf(pc[0] - M);
    L = fmaf(w, pc[1], L);
    acc = fmaf(w, pc[4 + d], acc);
  }
  attn[(size_t)h * kHd + d] = f2bf(acc / L);
}

__global__ void attn_residual_kernel(const uint16_t* __restrict__ resid, const float* __restrict__ y, int d,
                                     uint16_t* __restrict__ out, float* __restrict__ out_f32) {
  pdl_enter();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d) return;
  const float v = bf16f(resid[i]) + y[i];
  if (out_f32) out_f32[i] = v;
  out[i] = f2bf(v);
}

}  // namespace

int attn_chunks(int64_t span) { return (int)((span + kAttnChunk - 1) / kAttnChunk); }

cudaError_t launch_attn_decode(const AttnLaunch& L, cudaStream_t s) {
  const int nq = L.nq, nkv = L.nkv, rows = (nq + 2 * nkv) * kHd;
  // 1. q | k | v
  cudaError_t e = launch_lmhead(L.x, 1, L.d, rows, L.wqkv, L.qkv, L.am_scratch, L.keys_scratch, L.st, s);
  if (e != cudaSuccess) return e;
  // 2. norm, rotation, cache rows
  if ((e = launch_pdl(attn_prep_kernel, dim3(1), dim3(kPrepThreads), 0, s, (const float*)L.qkv, nq, nkv, L.pos,
                      L.rope, L.theta, L.eps, L.q, L.k_cache, L.v_cache)) != cudaSuccess)
    return e;
  // 3. chunks of the window
  const int64_t lo = L.window > 0 ? (L.pos - L.window + 1 > 0 ? L.pos - L.window + 1 : 0) : 0;
  const int64_t hi = L.pos + 1;
  SplitArgs a;
  a.q = L.q;
  a.k_cache = L.k_cache;
  a.v_cache = L.v_cache;
  a.nkv = nkv;
  a.lo = lo;
  a.hi = hi;
  a.chunk = kAttnChunk;
  a.scale = 1.0f / sqrtf((float)kHd);
  a.part = L.part;
  a.nchunks = attn_chunks(hi - lo);
  if ((e = launch_pdl(attn_split_kernel, dim3(nkv, a.nchunks), dim3(kQPerKv * 32), 0, s, a)) != cudaSuccess) return e;
  // 4. merge with the sinks
  if ((e = launch_pdl(attn_combine_kernel, dim3(nq), dim3(kHd), 0, s, (const float*)L.part, a.nchunks, L.sinks,
                      L.attn)) != cudaSuccess)
    return e;
  // 5. output projection and residual
  if ((e = launch_lmhead(L.attn, 1, nq * kHd, L.d, L.wo, L.y, L.am_scratch, L.keys_scratch, L.st, s)) != cudaSuccess)
    return e;
  if ((e = launch_pdl(attn_residual_kernel, dim3(ceil_div(L.d, 256)), dim3(256), 0, s, L.resid, (const float*)L.y,
                      L.d, L.out, L.out_f32)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace bitmoe
