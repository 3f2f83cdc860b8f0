// 4-bit LM head: logits = h Wlm^T and the argmax over the vocabulary, with
// int4 (fp16 scale per 32 weights) or NVFP4 (E2M1 codes, E4M3 scale per 16
// weights, fp32 tensor scale) weights.
//
// "Flint 40B : Best Mid Sized LLM", transcript 03:36 (the output layer maps
// hidden states to a ~150k-token vocabulary) and 05:39 (it is quantised to
// four bits); "Recursive_SI's First Model Unveiled!", section "Quantization"
// (the output layer is a large share of the weights read per token).
//
// The bank is 151 MB at V = 131072 and is read once per call, so the kernel is
// a weight stream that has to keep HBM busy: one CTA per SM, a producer warp
// keeps a ring of 16-row tiles in flight with TMA bulk copies, and each
// consumer warp owns whole tiles -- it multiplies its tile's 16 rows over the
// full reduction on its own, so no consumer waits for another -- and its own
// ring stages.  A warp folds
// its logits into a per-token running arg-max in registers; at the end the
// warps' maxima meet in shared memory and one 64-bit atomicMax per token and
// CTA (order-preserving logit bits, then the inverted row index so that the
// lowest row wins ties) publishes them.
//
// Dequantisation costs more instructions than anything else here, so the
// weights become fp16 (the magic-number conversion needs one shift per 8
// nibbles) and the activations are fed to the tensor cores as fp16 too.  To
// keep every product exact, token t is multiplied by 2^s_t first, s_t chosen
// so that its largest |h| lands in [2^14, 2^15): a power-of-two scale is
// exact, the scaled bf16 values fit fp16 without rounding (only elements below
// 2^-24 of the token's largest would round), and the fp32 logit is scaled back
// by 2^-s_t, again exactly.
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kLmConsumers = 12;                // consumer warps, each owning whole tiles
constexpr int kLmThreads = (kLmConsumers + 1) * 32;
constexpr int kLmTok = 16;                      // tokens per launch (two mma n-tiles)
constexpr int kLmMaxStages = 16;
constexpr int kLmSmemBudget = 227 * 1024;

struct LmArgs {
  const uint16_t* h;  // [T, d] bf16, this launch's first token
  int ntok, d, V, tok0, nstages;
  int nwarps;  // consumer warps that take tiles (nstages is a multiple of it)
  const uint8_t* w;
  float ts;                  // NVFP4: the matrix's tensor scale
  float* logits;             // [T_total, V] or null
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

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kLmConsumers * 32)); }


// Shared memory: barriers (256 B), the per-token scale exponents and arg-max
// partials, the fp16 tokens [8 * NT][d + pad] and one zeroed row, then the tile ring.
struct LmSmem {
  static constexpr int kBars = 0;                                   // full[16], empty[16], xbar
  static constexpr int kExp = 384;                                  // int [16]
  static constexpr int kBestV = kExp + 64;                          // float [warps][16 tokens]
  static constexpr int kBestI = kBestV + kLmConsumers * kLmTok * 4; // int   [warps][16 tokens]
  static constexpr int kFail = kBestI + kLmConsumers * kLmTok * 4;  // int
  static constexpr int kX = 2304;                                   // fp16 tokens
  __host__ __device__ static int xstride(int d) { return 2 * d + kSmemRowPad; }
  // the launch's ntok token rows, then one zeroed pad row
  __host__ __device__ static int ring(int d, int ntok) { return kX + (((ntok + 1) * xstride(d) + 127) / 128) * 128; }
};
static_assert((2 * kLmMaxStages + 1) * 8 <= LmSmem::kExp, "lm head barriers");
static_assert(LmSmem::kFail + 4 <= LmSmem::kX, "lm head smem header");

// kFp4: the bank is NVFP4 (codes times block scale become exact fp16 weights
// before the MMA, whose fp32 sums run over the whole row; the tensor scale
// multiplies the logit); else int4 with fp16 group scales applied per group.
template <int NT, bool kFp4>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_kernel(LmArgs p) {
  pdl_enter();
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LmSmem::kBars);
  uint64_t* empty = full + kLmMaxStages;
  uint64_t* xbar = empty + kLmMaxStages;
  int* sexp = reinterpret_cast<int*>(smem + LmSmem::kExp);
  float* bestv_s = reinterpret_cast<float*>(smem + LmSmem::kBestV);
  int* besti_s = reinterpret_cast<int*>(smem + LmSmem::kBestI);
  int* fail_flag = reinterpret_cast<int*>(smem + LmSmem::kFail);
  const int d = p.d;
  const int xstride = LmSmem::xstride(d);
  unsigned char* sx = smem + LmSmem::kX;
  unsigned char* ring = smem + LmSmem::ring(d, p.ntok);
  const int tbytes = (int)tile_bytes(d);
  const int NS = p.nstages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // the one warp that consumed the tile
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
    *fail_flag = 0;
  }
  __syncthreads();

  const int VT = p.V / kTileRows;
  const int my_tiles = (VT > (int)blockIdx.x) ? (VT - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == kLmConsumers) {
    // ---------------- producer: the tokens, then this CTA's tiles in order
    if (lane == 0) {
      mbar_arrive_expect_tx(xbar, (uint32_t)p.ntok * 2u * d);
      for (int i = 0; i < p.ntok; ++i) bulk_g2s(sx + i * xstride, p.h + (size_t)i * d, 2 * d, xbar);
      int issued = 0;
      for (int i = 0; i < my_tiles; ++i) {
        const int s = i % NS;
        if (i >= NS) {
          // a stage is free once its consumer released it; stop early if a
          // consumer gave up (it will not release any more stages)
          bool ok = false;
          const uint32_t par = ((i / NS) - 1) & 1;
          const uint64_t t0 = globaltimer_ns();
          while (!(ok = mbar_try_wait(&empty[s], par))) {
            if (*(volatile int*)fail_flag) break;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              record_status(p.st, kStatusTimeout, 20, (int)blockIdx.x);
              atomicOr(fail_flag, 1);
              break;
            }
          }
          if (!ok) break;
        }
        mbar_arrive_expect_tx(&full[s], (uint32_t)tbytes);
        const size_t vt = (size_t)blockIdx.x + (size_t)i * gridDim.x;
        bulk_g2s(ring + (size_t)s * tbytes, p.w + vt * tbytes, tbytes, &full[s]);
        issued = i + 1;
      }
      // every copy this thread started lands before the CTA can exit
      for (int n = (issued > NS ? issued - NS : 0); n < issued; ++n)
        mbar_wait(&full[n % NS], (n / NS) & 1, p.st, 23);
      mbar_wait(xbar, 0, p.st, 24);
    }
    return;
  }

  // ---------------- consumers: stage the tokens as scaled fp16
  bool ok = mbar_wait(xbar, 0, p.st, 21);
  if (!ok) atomicOr(fail_flag, 1);
  {  // the pad row read for absent tokens
    uint4* pad = reinterpret_cast<uint4*>(sx + p.ntok * xstride);
    for (int c = tid; c < d / 8; c += kLmConsumers * 32) pad[c] = make_uint4(0, 0, 0, 0);
  }
  consumer_sync();
  if (*(volatile int*)fail_flag == 0) {
    // per token (one warp each, two passes for 16 tokens over 12 warps): largest
    // |h| -> exponent e; scale 2^(14 - e) puts the largest element in [2^14, 2^15)
    for (int t = warp; t < p.ntok; t += kLmConsumers) {
      uint16_t* xr = reinterpret_cast<uint16_t*>(sx + t * xstride);
      uint32_t m = 0;
      for (int c = lane * 8; c < d; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) m = max(m, max(w4[i] & 0x7fffu, (w4[i] >> 16) & 0x7fffu));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      // bf16 exponent field of the largest magnitude (0 for an all-zero or
      // subnormal-only token); both 2^s and 2^-s stay normal floats
      const int ef = (int)(m >> 7);
      const int s = (ef == 0) ? 0 : min(126, max(-126, 14 - (ef - 127)));
      if (lane == 0) sexp[t] = s;
      const float f = pow2i(s);
      for (int c = lane * 8; c < d; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[i] << 16) * f,
                                               __uint_as_float(w4[i] & 0xffff0000u) * f);
          o[i] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(xr + c) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  consumer_sync();

  const int g = lane >> 2, c = lane & 3;
  const int nch = d / kChunkK;
  // running arg-max of the lane's token slots: tokens nt*8 + 2c + b, rows g and g+8
  float best_v[NT][2];
  int best_i[NT][2];
  float unscale[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      best_v[nt][b] = -INFINITY;
      best_i[nt][b] = 0x7fffffff;
      const int tok = nt * 8 + 2 * c + b;
      unscale[nt][b] = (tok < p.ntok) ? pow2i(-sexp[tok]) : 0.f;
    }

  // the activation row of each lane's n-tile token; lanes past the last token
  // read the zeroed pad row after the tokens, so the load needs no branch
  const unsigned char* xrow[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tok = nt * 8 + g;
    xrow[nt] = sx + (tok < p.ntok ? tok : p.ntok) * xstride;
  }
  // Stage s always belongs to warp s % nw (the stage count is a multiple of
  // nw), so a warp waits on a stage's phases strictly in order: a parity wait
  // two phases ahead would alias the earlier phase and return at once.
  const int nw = p.nwarps;
  for (int i = warp; warp < nw && i < my_tiles && *(volatile int*)fail_flag == 0; i += nw) {
    const int s = i % NS;
    if (!mbar_wait(&full[s], (i / NS) & 1, p.st, 22)) {
      atomicOr(fail_flag, 1);
      break;
    }
    const unsigned char* tile = ring + (size_t)s * tbytes;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[nt][j] = 0.f;
#pragma unroll 2
    for (int ch = 0; ch < nch; ++ch) {
      const unsigned char* cw = tile + ch * kChunkBytes;
      const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
      const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
      const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
      if constexpr (kFp4) {
        // the chunk's 8 MMA steps chain in the tensor core's accumulator; the
        // chunks are then added in fp32 (a chain over the whole row would
        // drift: the tensor core does not round its additions to nearest)
        const uint32_t sl0 = fp4_lane_scales(s0, c), sl1 = fp4_lane_scales(s1, c);
        float dd[NT][4];
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int col = (ch * 4 + gg) * kGroup + c * 8;
          uint32_t p0[4], p1[4];
          e2m1x8_f16_scaled(word_at(q0, gg), e4m3_pair_f16((sl0 >> (8 * gg)) & 0xffu), p0);
          e2m1x8_f16_scaled(word_at(q1, gg), e4m3_pair_f16((sl1 >> (8 * gg)) & 0xffu), p1);
          const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]};
          const uint32_t a1[4] = {p0[2], p1[2], p0[3], p1[3]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 xb = *reinterpret_cast<const uint4*>(xrow[nt] + col * 2);
            if (gg == 0)
              mma_f16_z(dd[nt], a0, xb.x, xb.y);
            else
              mma_f16(dd[nt], a0, xb.x, xb.y, dd[nt]);
            mma_f16(dd[nt], a1, xb.z, xb.w, dd[nt]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[nt][j] += dd[nt][j];
        continue;
      }
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        uint32_t p0[4], p1[4];
        nib_pairs4_f16(word_at(q0, gg), p0);
        nib_pairs4_f16(word_at(q1, gg), p1);
        const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]};
        const uint32_t a1[4] = {p0[2], p1[2], p0[3], p1[3]};
        const float sc0 = scale_at(s0, gg), sc1 = scale_at(s1, gg);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 xb = *reinterpret_cast<const uint4*>(xrow[nt] + col * 2);
          float dd[4];
          mma_f16_z(dd, a0, xb.x, xb.y);
          mma_f16(dd, a1, xb.z, xb.w, dd);
          acc[nt][0] = fmaf(sc0, dd[0], acc[nt][0]);
          acc[nt][1] = fmaf(sc0, dd[1], acc[nt][1]);
          acc[nt][2] = fmaf(sc1, dd[2], acc[nt][2]);
          acc[nt][3] = fmaf(sc1, dd[3], acc[nt][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // every lane has read the stage
    const int vrow0 = (int)(((size_t)blockIdx.x + (size_t)i * gridDim.x) * kTileRows);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int b = j & 1;
        const int tok = nt * 8 + 2 * c + b;
        const int vrow = vrow0 + g + ((j >= 2) ? 8 : 0);
        if (tok < p.ntok) {
          const float v = kFp4 ? acc[nt][j] * (unscale[nt][b] * p.ts) : acc[nt][j] * unscale[nt][b];
          if (p.logits) p.logits[(size_t)(p.tok0 + tok) * p.V + vrow] = v;
          if (v > best_v[nt][b] || (v == best_v[nt][b] && vrow < best_i[nt][b])) {
            best_v[nt][b] = v;
            best_i[nt][b] = vrow;
          }
        }
      }
  }
  // the warp's arg-max per token: reduce over the eight row groups g (lanes
  // with the same c), then over the warps in shared memory
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float v = best_v[nt][b];
      int ix = best_i[nt][b];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, off);
        if (ov > v || (ov == v && oi < ix)) {
          v = ov;
          ix = oi;
        }
      }
      if (g == 0) {
        bestv_s[warp * kLmTok + nt * 8 + 2 * c + b] = v;
        besti_s[warp * kLmTok + nt * 8 + 2 * c + b] = ix;
      }
    }
  consumer_sync();
  if (*(volatile int*)fail_flag) return;
  if (tid < p.ntok) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int w = 0; w < kLmConsumers; ++w) {
      const float v = bestv_s[w * kLmTok + tid];
      const int ix = besti_s[w * kLmTok + tid];
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
  pdl_enter();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < T) argmax[t] = (int32_t)(0xffffffffu - (uint32_t)(keys[t] & 0xffffffffull));
}

int lm_stages(int d, int ntok) {
  const int n = (kLmSmemBudget - LmSmem::ring(d, ntok)) / (int)tile_bytes(d);
  return n < kLmMaxStages ? n : kLmMaxStages;
}

size_t lm_smem(int d, int ntok) { return (size_t)LmSmem::ring(d, ntok) + (size_t)lm_stages(d, ntok) * tile_bytes(d); }

}  // namespace

size_t lmhead_scratch_bytes(int T) { return (size_t)T * sizeof(unsigned long long); }

bool lmhead_supported(int d, int T) { return lm_stages(d, T < kLmTok ? T : kLmTok) >= 2; }

template <bool kFp4>
cudaError_t launch_lmhead_fmt(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float ts,
                              float* logits, int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (!lmhead_supported(d, T)) return cudaErrorNotSupported;  // d too large for two tiles beside the tokens
  unsigned long long* keys = static_cast<unsigned long long*>(scratch);
  cudaError_t err = cudaMemsetAsync(keys, 0, (size_t)T * sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  static int attr1[64] = {}, attr2[64] = {};
  // every launch fits the budget whatever its token count (the ring takes the rest)
  err = ensure_smem_attr(lmhead_kernel<1, kFp4>, (size_t)kLmSmemBudget, attr1);
  if (err != cudaSuccess) return err;
  err = ensure_smem_attr(lmhead_kernel<2, kFp4>, (size_t)kLmSmemBudget, attr2);
  if (err != cudaSuccess) return err;
  static int sm_count[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
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
    const int nt = a.ntok <= 8 ? 1 : 2;
    const int ns = lm_stages(d, a.ntok);
    a.nwarps = ns < kLmConsumers ? ns : kLmConsumers;
    a.nstages = ns / a.nwarps * a.nwarps;
    a.w = w_packed;
    a.ts = ts;
    a.logits = logits;
    a.keys = keys;
    a.st = st;
    auto* kern = (nt == 1) ? lmhead_kernel<1, kFp4> : lmhead_kernel<2, kFp4>;
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kLmThreads), lm_smem(d, a.ntok), s, a);
    if (e != cudaSuccess) return e;
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cudaError_t e_ = launch_pdl(argmax_finalize_kernel, dim3(ceil_div(T, 128)), dim3(128), 0, s, keys, T,
                                  argmax)) return e_;
  return cudaGetLastError();
}

cudaError_t launch_lmhead(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float* logits,
                          int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s) {
  return launch_lmhead_fmt<false>(h, T, d, V, w_packed, 1.0f, logits, argmax, scratch, st, s);
}

cudaError_t launch_lmhead_nvfp4(const uint16_t* h, int T, int d, int V, const uint8_t* w_packed, float ts,
                                float* logits, int32_t* argmax, void* scratch, DevStatus* st, cudaStream_t s) {
  return launch_lmhead_fmt<true>(h, T, d, V, w_packed, ts, logits, argmax, scratch, st, s);
}

}  // namespace bitmoe
