// Expert FFN kernels: a = Wg x, u = Wu x, h = silu(a) * u, y = Wd h, with int4
// group-32 weights ("Flint 40B : Best Mid Sized LLM", transcript 06:11:
// kernels for low-bit matrix projections; 02:35: experts of a mixture layer).
//
// Work unit = (expert e, 16-row weight tile, block of up to 16 of e's grouped
// rows).  One elected thread stages the unit with TMA bulk copies (the weight
// tiles in the packed layout and the unit's activation rows) on an mbarrier;
// four warps split the reduction dimension by 128-column chunks.
//
// Arithmetic.  The int4 values are turned into exact 16-bit integers (bf16 for
// the bf16 activations, fp16 for h) and multiplied on the tensor cores with
// mma.sync m16n8k16 (weights = A, up to 8 tokens = B).  Each mma pair covers
// exactly one 32-column group, so its fp32 result is the group's exact-input
// partial sum, which is then scaled by the group's fp16 scale in fp32: the
// dequantised weight q*s is never rounded.  h enters the down projection as
// an fp16 pair hi + lo (about 22 significant bits).
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kFfnThreads = 128;
constexpr int kNT = kTokBlock / 8;  // n-tiles of 8 tokens per unit

__device__ __forceinline__ float scale_at(uint2 s, int gg) {
  const uint32_t w = (gg < 2) ? s.x : s.y;
  const uint16_t b = (gg & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
  return __half2float(__ushort_as_half(b));
}

// A fragments of two k16 steps for rows g (word w0) and g+8 (word w1).
__device__ __forceinline__ void frag_bf16(uint32_t w0, uint32_t w1, uint32_t (&a)[2][4]) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    a[s][0] = nib_pair_bf16(w0, 2 * s);
    a[s][1] = nib_pair_bf16(w1, 2 * s);
    a[s][2] = nib_pair_bf16(w0, 2 * s + 1);
    a[s][3] = nib_pair_bf16(w1, 2 * s + 1);
  }
}

__device__ __forceinline__ void frag_f16(uint32_t w0, uint32_t w1, uint32_t (&a)[2][4]) {
  uint32_t p0[4], p1[4];
  nib_pairs4_f16(w0, p0);
  nib_pairs4_f16(w1, p1);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    a[s][0] = p0[2 * s];
    a[s][1] = p1[2 * s];
    a[s][2] = p0[2 * s + 1];
    a[s][3] = p1[2 * s + 1];
  }
}

__device__ __forceinline__ uint32_t word_at(const uint4& q, int gg) {
  return gg == 0 ? q.x : gg == 1 ? q.y : gg == 2 ? q.z : q.w;
}

// Expert owning token block b: the e with blk_prefix[e] <= b < blk_prefix[e+1].
__device__ __forceinline__ int expert_of_block(const int32_t* __restrict__ blk_prefix, int E, int b) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (blk_prefix[mid] <= b) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------- gate/up + SwiGLU

__global__ void __launch_bounds__(kFfnThreads) ffn_up_kernel(FfnArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const int d = p.d, I = p.I;
  const int tbytes = (int)tile_bytes(d);
  unsigned char* sg = smem + 128;
  unsigned char* su = sg + tbytes;
  unsigned char* sx = su + tbytes;
  const int xstride = 2 * d + kSmemRowPad;
  float* red = reinterpret_cast<float*>(sx + kTokBlock * xstride);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int RT = I / kTileRows;
  const int n_units = RT * p.blk_prefix[p.E];
  const int nch = d / kChunkK;
  uint32_t phase = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int b = u / RT, rt = u - b * RT;
    const int e = expert_of_block(p.blk_prefix, p.E, b);
    const int p0 = p.offsets[e] + (b - p.blk_prefix[e]) * kTokBlock;
    const int nval = min(kTokBlock, p.offsets[e + 1] - p0);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, 2u * tbytes + (uint32_t)nval * 2u * d);
      const size_t toff = ((size_t)e * RT + rt) * tbytes;
      bulk_g2s(sg, p.gate + toff, tbytes, bar);
      bulk_g2s(su, p.up + toff, tbytes, bar);
      for (int i = 0; i < nval; ++i) {
        const int t = p.sorted_rows[p0 + i] / p.k;
        bulk_g2s(sx + i * xstride, p.x + (size_t)t * d, 2 * d, bar);
      }
    }
    const bool ok = mbar_wait(bar, phase, p.st, 10);
    if (__syncthreads_or(!ok)) return;  // uniform exit: every thread leaves together
    phase ^= 1;

    float acc_g[kNT][4], acc_u[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc_g[nt][i] = acc_u[nt][i] = 0.f;

    for (int ch = warp; ch < nch; ch += kFfnThreads / 32) {
      const unsigned char* cg = sg + ch * kChunkBytes;
      const unsigned char* cu = su + ch * kChunkBytes;
      const uint4 qg0 = *reinterpret_cast<const uint4*>(cg + (g * 4 + c) * 16);
      const uint4 qg1 = *reinterpret_cast<const uint4*>(cg + ((g + 8) * 4 + c) * 16);
      const uint4 qu0 = *reinterpret_cast<const uint4*>(cu + (g * 4 + c) * 16);
      const uint4 qu1 = *reinterpret_cast<const uint4*>(cu + ((g + 8) * 4 + c) * 16);
      const uint2 sg0 = *reinterpret_cast<const uint2*>(cg + kChunkQBytes + g * 8);
      const uint2 sg1 = *reinterpret_cast<const uint2*>(cg + kChunkQBytes + (g + 8) * 8);
      const uint2 su0 = *reinterpret_cast<const uint2*>(cu + kChunkQBytes + g * 8);
      const uint2 su1 = *reinterpret_cast<const uint2*>(cu + kChunkQBytes + (g + 8) * 8);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        uint32_t ag[2][4], au[2][4];
        frag_bf16(word_at(qg0, gg), word_at(qg1, gg), ag);
        frag_bf16(word_at(qu0, gg), word_at(qu1, gg), au);
        const float s_g0 = scale_at(sg0, gg), s_g1 = scale_at(sg1, gg);
        const float s_u0 = scale_at(su0, gg), s_u1 = scale_at(su1, gg);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const int tok = nt * 8 + g;
          uint4 xb = make_uint4(0, 0, 0, 0);
          if (tok < nval) xb = *reinterpret_cast<const uint4*>(sx + tok * xstride + col * 2);
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float dg[4], du[4];
          mma_bf16(dg, ag[0], xb.x, xb.y, z);
          mma_bf16(dg, ag[1], xb.z, xb.w, dg);
          mma_bf16(du, au[0], xb.x, xb.y, z);
          mma_bf16(du, au[1], xb.z, xb.w, du);
          acc_g[nt][0] = fmaf(s_g0, dg[0], acc_g[nt][0]);
          acc_g[nt][1] = fmaf(s_g0, dg[1], acc_g[nt][1]);
          acc_g[nt][2] = fmaf(s_g1, dg[2], acc_g[nt][2]);
          acc_g[nt][3] = fmaf(s_g1, dg[3], acc_g[nt][3]);
          acc_u[nt][0] = fmaf(s_u0, du[0], acc_u[nt][0]);
          acc_u[nt][1] = fmaf(s_u0, du[1], acc_u[nt][1]);
          acc_u[nt][2] = fmaf(s_u1, du[2], acc_u[nt][2]);
          acc_u[nt][3] = fmaf(s_u1, du[3], acc_u[nt][3]);
        }
      }
    }
    float* my = red + (size_t)(warp * 32 + lane) * (8 * kNT);
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        my[nt * 4 + i] = acc_g[nt][i];
        my[4 * kNT + nt * 4 + i] = acc_u[nt][i];
      }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = 0.f, uu = 0.f;
#pragma unroll
          for (int w = 0; w < kFfnThreads / 32; ++w) {
            a += red[(size_t)(w * 32 + lane) * (8 * kNT) + nt * 4 + i];
            uu += red[(size_t)(w * 32 + lane) * (8 * kNT) + 4 * kNT + nt * 4 + i];
          }
          const int row = rt * kTileRows + ((i < 2) ? g : g + 8);
          const int tok = nt * 8 + 2 * c + (i & 1);
          if (tok < nval) {
            const float h = silu_mul(a, uu);
            const __half hi = __float2half_rn(h);
            const __half lo = __float2half_rn(h - __half2float(hi));
            p.h_hi[(size_t)(p0 + tok) * I + row] = hi;
            p.h_lo[(size_t)(p0 + tok) * I + row] = lo;
          }
        }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- down projection

__global__ void __launch_bounds__(kFfnThreads) ffn_down_kernel(FfnArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
  const int d = p.d, I = p.I;
  const int tbytes = (int)tile_bytes(I);
  unsigned char* sw = smem + 128;
  const int hstride = 2 * I + kSmemRowPad;
  unsigned char* shh = sw + tbytes;
  unsigned char* shl = shh + kTokBlock * hstride;
  float* red = reinterpret_cast<float*>(shl + kTokBlock * hstride);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int CT = d / kTileRows;
  const int n_units = CT * p.blk_prefix[p.E];
  const int nch = I / kChunkK;
  uint32_t phase = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int b = u / CT, ct = u - b * CT;
    const int e = expert_of_block(p.blk_prefix, p.E, b);
    const int p0 = p.offsets[e] + (b - p.blk_prefix[e]) * kTokBlock;
    const int nval = min(kTokBlock, p.offsets[e + 1] - p0);
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)tbytes + (uint32_t)nval * 4u * I);
      bulk_g2s(sw, p.down + ((size_t)e * CT + ct) * tbytes, tbytes, bar);
      for (int i = 0; i < nval; ++i) {
        bulk_g2s(shh + i * hstride, p.h_hi + (size_t)(p0 + i) * I, 2 * I, bar);
        bulk_g2s(shl + i * hstride, p.h_lo + (size_t)(p0 + i) * I, 2 * I, bar);
      }
    }
    const bool ok = mbar_wait(bar, phase, p.st, 11);
    if (__syncthreads_or(!ok)) return;  // uniform exit: every thread leaves together
    phase ^= 1;

    float acc[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

    for (int ch = warp; ch < nch; ch += kFfnThreads / 32) {
      const unsigned char* cw = sw + ch * kChunkBytes;
      const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
      const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
      const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        uint32_t a[2][4];
        frag_f16(word_at(q0, gg), word_at(q1, gg), a);
        const float sc0 = scale_at(s0, gg), sc1 = scale_at(s1, gg);
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt) {
          const int tok = nt * 8 + g;
          uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
          if (tok < nval) {
            bh = *reinterpret_cast<const uint4*>(shh + tok * hstride + col * 2);
            bl = *reinterpret_cast<const uint4*>(shl + tok * hstride + col * 2);
          }
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float dd[4];
          mma_f16(dd, a[0], bh.x, bh.y, z);
          mma_f16(dd, a[0], bl.x, bl.y, dd);
          mma_f16(dd, a[1], bh.z, bh.w, dd);
          mma_f16(dd, a[1], bl.z, bl.w, dd);
          acc[nt][0] = fmaf(sc0, dd[0], acc[nt][0]);
          acc[nt][1] = fmaf(sc0, dd[1], acc[nt][1]);
          acc[nt][2] = fmaf(sc1, dd[2], acc[nt][2]);
          acc[nt][3] = fmaf(sc1, dd[3], acc[nt][3]);
        }
      }
    }
    float* my = red + (size_t)(warp * 32 + lane) * (4 * kNT);
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) my[nt * 4 + i] = acc[nt][i];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kFfnThreads / 32; ++w) v += red[(size_t)(w * 32 + lane) * (4 * kNT) + nt * 4 + i];
          const int col = ct * kTileRows + ((i < 2) ? g : g + 8);
          const int tok = nt * 8 + 2 * c + (i & 1);
          if (tok < nval) p.y_rows[(size_t)(p0 + tok) * d + col] = v;
        }
    }
    __syncthreads();
  }
}

size_t up_smem(int d) {
  return 128 + 2 * (size_t)tile_bytes(d) + (size_t)kTokBlock * (2 * d + kSmemRowPad) +
         (size_t)kFfnThreads * 8 * kNT * sizeof(float);
}
size_t down_smem(int I) {
  return 128 + (size_t)tile_bytes(I) + 2 * (size_t)kTokBlock * (2 * I + kSmemRowPad) +
         (size_t)kFfnThreads * 4 * kNT * sizeof(float);
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// Upper bound on the token blocks of R rows over E experts (grid sizing only).
int max_blocks(int R, int E) { return min(R, E) + R / kTokBlock + 1; }

}  // namespace

cudaError_t launch_ffn_up(const FfnArgs& a, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) return cudaSuccess;
  const size_t sm = up_smem(a.d);
  static int attr_set[64] = {};
  cudaError_t err = ensure_smem_attr(ffn_up_kernel, sm, attr_set);
  if (err != cudaSuccess) return err;
  const long units = (long)(a.I / kTileRows) * max_blocks(R, a.E);
  const int grid = (int)(units < 2L * num_sms() ? units : 2L * num_sms());
  ffn_up_kernel<<<grid, kFfnThreads, sm, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_ffn_down(const FfnArgs& a, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) return cudaSuccess;
  const size_t sm = down_smem(a.I);
  static int attr_set[64] = {};
  cudaError_t err = ensure_smem_attr(ffn_down_kernel, sm, attr_set);
  if (err != cudaSuccess) return err;
  const long units = (long)(a.d / kTileRows) * max_blocks(R, a.E);
  const int grid = (int)(units < 4L * num_sms() ? units : 4L * num_sms());
  ffn_down_kernel<<<grid, kFfnThreads, sm, s>>>(a);
  return cudaGetLastError();
}

}  // namespace bitmoe
