// 4-bit LM head: logits = h Wlm^T and the argmax over the vocabulary.
//
// "Flint 40B : Best Mid Sized LLM", transcript 03:36 (the output layer maps
// hidden states to a ~150k-token vocabulary) and 05:39 (it is quantised to
// four bits); "Recursive_SI's First Model Unveiled!", section "Quantization"
// (the output layer is a large share of the weights read per token).
//
// The bank is 151 MB at V = 131072 and is read once per call, so the kernel is
// a weight stream: one CTA per SM, a producer warp keeps a ring of 16-row tiles
// in flight with TMA bulk copies (full / empty mbarriers per stage), eight
// consumer warps split each tile's 2048 columns, reduce through shared memory
// and fold every logit into a per-token running arg-max.  The final arg-max is
// an atomicMax on a 64-bit key (order-preserving logit bits, then the inverted
// row index so that the lowest row wins ties).
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kLmThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 6;
constexpr int kLmTok = 16;  // tokens per launch (two n-tiles)

struct LmArgs {
  const uint16_t* h;  // [T, d] bf16, this launch's first token
  int ntok, d, V, tok0;
  const uint8_t* w;
  float* logits;            // [T_total, V] or null
  unsigned long long* keys;  // [T_total]
  DevStatus* st;
};

__device__ __forceinline__ float scale_at(uint2 s, int gg) {
  const uint32_t w = (gg < 2) ? s.x : s.y;
  const uint16_t b = (gg & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t word_at(const uint4& q, int gg) {
  return gg == 0 ? q.x : gg == 1 ? q.y : gg == 2 ? q.z : q.w;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32)); }

template <int NT>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_kernel(LmArgs p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  uint64_t* xbar = empty + kStages;
  const int d = p.d;
  const int tbytes = (int)tile_bytes(d);
  const int xstride = 2 * d + kSmemRowPad;
  unsigned char* stages = smem + 256;
  unsigned char* sx = stages + (size_t)kStages * tbytes;
  float* red = reinterpret_cast<float*>(sx + (size_t)kLmTok * xstride);  // [2][8 warps][32][8]
  float* bestv = red + 2 * kConsumerWarps * 32 * 8;                      // [256]
  int* besti = reinterpret_cast<int*>(bestv + kConsumerWarps * 32);       // [256]
  int* fail_flag = besti + kConsumerWarps * 32;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
    *fail_flag = 0;
  }
  __syncthreads();

  const int VT = p.V / kTileRows;
  const int my_tiles = (VT > (int)blockIdx.x) ? (VT - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == kConsumerWarps) {
    // ---------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(xbar, (uint32_t)p.ntok * 2u * d);
      for (int i = 0; i < p.ntok; ++i) bulk_g2s(sx + i * xstride, p.h + (size_t)i * d, 2 * d, xbar);
      for (int i = 0; i < my_tiles; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1, p.st, 20)) return;
        mbar_arrive_expect_tx(&full[s], (uint32_t)tbytes);
        const size_t vt = (size_t)blockIdx.x + (size_t)i * gridDim.x;
        bulk_g2s(stages + (size_t)s * tbytes, p.w + vt * tbytes, tbytes, &full[s]);
      }
    }
    return;
  }

  // ---------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int nch = d / kChunkK;
  float best_v = -INFINITY;
  int best_i = 0x7fffffff;
  // reducer mapping: consumer thread -> (row, token) of the 16 x 16 tile output
  const int rrow = tid >> 4, rtok = tid & 15;
  const int r_nt = rtok >> 3, r_tl = rtok & 7;
  const int r_lane = (rrow & 7) * 4 + (r_tl >> 1);
  const int r_idx = r_nt * 4 + ((rrow >= 8) ? 2 : 0) + (r_tl & 1);

  // A wait that runs out sets fail_flag; every consumer reads the flag after
  // the same barrier, so all of them leave the loop together.
  bool ok = mbar_wait(xbar, 0, p.st, 21);
  if (!ok) atomicOr(fail_flag, 1);
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kStages;
    if (ok && !mbar_wait(&full[s], (i / kStages) & 1, p.st, 22)) {
      ok = false;
      atomicOr(fail_flag, 1);
    }
    const unsigned char* tile = stages + (size_t)s * tbytes;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;
    for (int ch = warp; ch < nch; ch += kConsumerWarps) {
      const unsigned char* cw = tile + ch * kChunkBytes;
      const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
      const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
      const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        uint32_t a[2][4];
        const uint32_t w0 = word_at(q0, gg), w1 = word_at(q1, gg);
#pragma unroll
        for (int st = 0; st < 2; ++st) {
          a[st][0] = nib_pair_bf16(w0, 2 * st);
          a[st][1] = nib_pair_bf16(w1, 2 * st);
          a[st][2] = nib_pair_bf16(w0, 2 * st + 1);
          a[st][3] = nib_pair_bf16(w1, 2 * st + 1);
        }
        const float sc0 = scale_at(s0, gg), sc1 = scale_at(s1, gg);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int tok = nt * 8 + g;
          uint4 xb = make_uint4(0, 0, 0, 0);
          if (tok < p.ntok) xb = *reinterpret_cast<const uint4*>(sx + tok * xstride + col * 2);
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float dd[4];
          mma_bf16(dd, a[0], xb.x, xb.y, z);
          mma_bf16(dd, a[1], xb.z, xb.w, dd);
          acc[nt][0] = fmaf(sc0, dd[0], acc[nt][0]);
          acc[nt][1] = fmaf(sc0, dd[1], acc[nt][1]);
          acc[nt][2] = fmaf(sc1, dd[2], acc[nt][2]);
          acc[nt][3] = fmaf(sc1, dd[3], acc[nt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    float* my = red + ((size_t)(i & 1) * kConsumerWarps * 32 + warp * 32 + lane) * 8;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) my[nt * 4 + j] = (nt < NT) ? acc[nt][j] : 0.f;
    consumer_sync();
    if (*(volatile int*)fail_flag) break;
    if (rtok < p.ntok) {
      const float* rb = red + (size_t)(i & 1) * kConsumerWarps * 32 * 8;
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v += rb[(w * 32 + r_lane) * 8 + r_idx];
      const int vrow = (int)(((size_t)blockIdx.x + (size_t)i * gridDim.x) * kTileRows) + rrow;
      if (p.logits) p.logits[(size_t)(p.tok0 + rtok) * p.V + vrow] = v;
      if (v > best_v || (v == best_v && vrow < best_i)) {
        best_v = v;
        best_i = vrow;
      }
    }
  }
  if (*(volatile int*)fail_flag) return;
  // per-token arg-max over the 16 rows each thread folded, then one atomic per token
  bestv[tid] = best_v;
  besti[tid] = best_i;
  consumer_sync();
  if (tid < p.ntok) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int r = 0; r < kTileRows; ++r) {
      const float v = bestv[r * 16 + tid];
      const int ix = besti[r * 16 + tid];
      if (v > bv || (v == bv && ix < bi)) {
        bv = v;
        bi = ix;
      }
    }
    if (bi != 0x7fffffff) {
      const unsigned long long key = ((unsigned long long)float_order_key(bv) << 32) | (0xffffffffu - (uint32_t)bi);
      atomicMax(&p.keys[p.tok0 + tid], key);
    }
  }
}

__global__ void argmax_finalize_kernel(const unsigned long long* keys, int T, int32_t* argmax) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) argmax[t] = (int32_t)(0xffffffffu - (uint32_t)(keys[t] & 0xffffffffull));
}

size_t lm_smem(int d) {
  return 256 + (size_t)kStages * tile_bytes(d) + (size_t)kLmTok * (2 * d + kSmemRowPad) +
         (size_t)2 * kConsumerWarps * 32 * 8 * 4 + (size_t)kConsumerWarps * 32 * 8 + 16;
}

}  // namespace

size_t lmhead_scratch_bytes(int T) { return (size_t)T * sizeof(unsigned long long); }

cudaError_t launch_lmhead(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float* logits,
                          int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  unsigned long long* keys = static_cast<unsigned long long*>(scratch);
  cudaError_t err = cudaMemsetAsync(keys, 0, (size_t)T * sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  const size_t sm = lm_smem(d);
  static int attr1[64] = {}, attr2[64] = {};
  err = ensure_smem_attr(lmhead_kernel<1>, sm, attr1);
  if (err != cudaSuccess) return err;
  err = ensure_smem_attr(lmhead_kernel<2>, sm, attr2);
  if (err != cudaSuccess) return err;
  static int sm_count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (sm_count[dev] == 0) cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
  const int sms = sm_count[dev] > 0 ? sm_count[dev] : 148;
  const int VT = V / kTileRows;
  const int grid = VT < sms ? VT : sms;
  for (int t0 = 0; t0 < T; t0 += kLmTok) {
    LmArgs a;
    a.h = h + (size_t)t0 * d;
    a.ntok = (T - t0) < kLmTok ? (T - t0) : kLmTok;
    a.d = d;
    a.V = V;
    a.tok0 = t0;
    a.w = w_packed;
    a.logits = logits;
    a.keys = keys;
    a.st = st;
    if (a.ntok <= 8)
      lmhead_kernel<1><<<grid, kLmThreads, sm, s>>>(a);
    else
      lmhead_kernel<2><<<grid, kLmThreads, sm, s>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  argmax_finalize_kernel<<<ceil_div(T, 128), 128, 0, s>>>(keys, T, argmax);
  return cudaGetLastError();
}

}  // namespace bitmoe
