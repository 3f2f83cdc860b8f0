// Router: logits = x Wr^T + b (fp32), then per-token top-k and gate weights.
//
// "Flint 40B : Best Mid Sized LLM", transcript 02:35: a small router picks a
// few of the 256 routed experts for every token.  Softmax over all experts,
// the k largest (equal logits -> lower expert), gates renormalised over the
// chosen k unless disabled.
#include <float.h>

#include "kernels.h"

namespace bitmoe {
namespace {

// ---------------------------------------------------------------- decode-size router GEMV
//
// One CTA per pair of experts, so the 2 MB router matrix is read by every SM
// at once; each warp owns (token, expert) dot products and reduces them with
// shuffles.  Lanes read 8 consecutive elements (16 B of x, 32 B of Wr).
constexpr int kRouteEB = 2;

__global__ void __launch_bounds__(256) router_gemv_kernel(const uint16_t* __restrict__ x, int T, int d, int E,
                                                          const float* __restrict__ Wr,
                                                          const float* __restrict__ b, float* __restrict__ logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * kRouteEB;
  const int pairs = T * kRouteEB;
  for (int pr = warp; pr < pairs; pr += 8) {
    const int t = pr / kRouteEB;
    const int e = e0 + pr % kRouteEB;
    if (e >= E) continue;
    const uint16_t* xr = x + (size_t)t * d;
    const float* wr = Wr + (size_t)e * d;
    float acc = 0.f;
#pragma unroll 4
    for (int i = lane * 8; i < d; i += 256) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xr + i);
      const float4 w0 = *reinterpret_cast<const float4*>(wr + i);
      const float4 w1 = *reinterpret_cast<const float4*>(wr + i + 4);
      acc = fmaf(__uint_as_float(xv.x << 16), w0.x, acc);
      acc = fmaf(__uint_as_float(xv.x & 0xffff0000u), w0.y, acc);
      acc = fmaf(__uint_as_float(xv.y << 16), w0.z, acc);
      acc = fmaf(__uint_as_float(xv.y & 0xffff0000u), w0.w, acc);
      acc = fmaf(__uint_as_float(xv.z << 16), w1.x, acc);
      acc = fmaf(__uint_as_float(xv.z & 0xffff0000u), w1.y, acc);
      acc = fmaf(__uint_as_float(xv.w << 16), w1.z, acc);
      acc = fmaf(__uint_as_float(xv.w & 0xffff0000u), w1.w, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) logits[(size_t)t * E + e] = acc + (b ? b[e] : 0.f);
  }
}

// ---------------------------------------------------------------- prefill-size router GEMM
//
// 64 tokens x 64 experts per CTA, 32-column slabs of x (bf16 -> fp32) and Wr
// in shared memory, 4x4 outputs per thread, fp32 FMA in ascending column order.
constexpr int kRtM = 64, kRtN = 64, kRtK = 32;

__global__ void __launch_bounds__(256) router_gemm_kernel(const uint16_t* __restrict__ x, int T, int d, int E,
                                                          const float* __restrict__ Wr,
                                                          const float* __restrict__ b, float* __restrict__ logits) {
  __shared__ float xs[kRtK][kRtM + 4];
  __shared__ float ws[kRtK][kRtN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kRtM, e0 = blockIdx.y * kRtN;
  float acc[4][4] = {};
  // load mapping: row = tid / 4 (0..63), 8 columns at (tid % 4) * 8
  const int lr = tid >> 2, lc = (tid & 3) * 8;
  for (int k0 = 0; k0 < d; k0 += kRtK) {
    {
      const int t = t0 + lr;
      uint4 xv = make_uint4(0, 0, 0, 0);
      if (t < T) xv = *reinterpret_cast<const uint4*>(x + (size_t)t * d + k0 + lc);
      const uint32_t wv[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs[lc + 2 * i][lr] = __uint_as_float(wv[i] << 16);
        xs[lc + 2 * i + 1][lr] = __uint_as_float(wv[i] & 0xffff0000u);
      }
      const int e = e0 + lr;
      float4 a = make_float4(0, 0, 0, 0), c = make_float4(0, 0, 0, 0);
      if (e < E) {
        a = *reinterpret_cast<const float4*>(Wr + (size_t)e * d + k0 + lc);
        c = *reinterpret_cast<const float4*>(Wr + (size_t)e * d + k0 + lc + 4);
      }
      ws[lc + 0][lr] = a.x; ws[lc + 1][lr] = a.y; ws[lc + 2][lr] = a.z; ws[lc + 3][lr] = a.w;
      ws[lc + 4][lr] = c.x; ws[lc + 5][lr] = c.y; ws[lc + 6][lr] = c.z; ws[lc + 7][lr] = c.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kRtK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (b ? b[e] : 0.f);
    }
  }
}

// ---------------------------------------------------------------- top-k + gates
//
// One warp per token.  Lane l holds logits e = l, l+32, ...; k rounds of a
// warp arg-max over (value desc, index asc) pick the experts in order.  Gates:
// exp(l_j - l_max) normalised over the chosen k (renorm) or over all E.
__global__ void __launch_bounds__(256) topk_gates_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  float v[kMaxE / 32];
  const int nper = (E + 31) / 32;
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = i * 32 + lane;
    v[i] = (i < nper && e < E) ? l[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float my_sel = -INFINITY;
  int my_id = 0;
  float vmax = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = i * 32 + lane;
      if (i < nper && e < E && !((taken >> i) & 1u)) {
        if (v[i] > bv || (v[i] == bv && e < bi)) {
          bv = v[i];
          bi = e;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) vmax = bv;
    if (j == lane) {
      my_sel = bv;
      my_id = bi;
    }
  }
  const float my_e = (lane < k) ? expf(my_sel - vmax) : 0.f;
  float z = 0.f;
  if (renorm) {
    z = my_e;
  } else {
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = i * 32 + lane;
      if (i < nper && e < E) z += expf(v[i] - vmax);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = my_e / z;
  }
}

// ---------------------------------------------------------------- forced selection
//
// Copies caller-given ids / gates into the working arrays.  Ids outside [0, E)
// become -1 (left out of the permutation) and flag kStatusCheck; a token that
// lists one expert twice also flags kStatusCheck.
__global__ void forced_select_kernel(const int32_t* __restrict__ fid, const float* __restrict__ fw, int T, int E,
                                     int k, int32_t* __restrict__ ids, float* __restrict__ w, DevStatus* st) {
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= T * k) return;
  int e = fid[r];
  if (e < 0 || e >= E) {
    record_status(st, kStatusCheck, 1, r);
    e = -1;
  } else {
    const int t = r / k, j = r % k;
    for (int jj = 0; jj < j; ++jj)
      if (fid[t * k + jj] == e) record_status(st, kStatusCheck, 2, r);
  }
  ids[r] = e;
  w[r] = fw[r];
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, int T, int d, int E, const float* w_router,
                                 const float* b_router, float* logits, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (T <= 64) {
    router_gemv_kernel<<<ceil_div(E, kRouteEB), 256, 0, s>>>(x, T, d, E, w_router, b_router, logits);
  } else {
    dim3 grid(ceil_div(T, kRtM), ceil_div(E, kRtN));
    router_gemm_kernel<<<grid, 256, 0, s>>>(x, T, d, E, w_router, b_router, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_gates(const float* logits, int T, int E, int k, int renorm, int32_t* ids, float* w,
                              cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  topk_gates_kernel<<<ceil_div(T, 8), 256, 0, s>>>(logits, T, E, k, renorm, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_forced_select(const int32_t* forced_ids, const float* forced_w, int T, int E, int k,
                                 int32_t* ids, float* w, DevStatus* st, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  forced_select_kernel<<<ceil_div(T * k, 256), 256, 0, s>>>(forced_ids, forced_w, T, E, k, ids, w, st);
  return cudaGetLastError();
}

}  // namespace bitmoe
