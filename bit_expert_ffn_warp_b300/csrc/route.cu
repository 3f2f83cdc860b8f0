// Router: logits = x Wr^T + b (fp32 accuracy), then per-token top-k and gate weights.
//
// "Flint 40B : Best Mid Sized LLM", transcript 02:35: a small router picks a
// few of the 256 routed experts for every token.  Softmax over all experts,
// the k largest (equal logits -> lower expert), gates renormalised over the
// chosen k unless disabled.
#include <float.h>

#include "kernels.h"
#include "tc.cuh"

namespace bitmoe {
namespace {

// ---------------------------------------------------------------- router on the tensor cores
//
// logits = x Wr^T with mma.sync m16n8k16 (bf16 in, fp32 accumulate).  x is bf16
// already; every fp32 weight is split exactly into three bf16 parts
// w = hi + mid + lo (each part the truncation of what remains, which fp32
// holds exactly), so every product x * part is exact in fp32 and the logit
// carries only fp32 summation error, as a fp32 FMA chain would.  A warp owns
// 16 tokens x 8 experts over one eighth of K; the eight partial sums are added
// in a fixed order.
constexpr int kRmTok = 16, kRmExp = 8, kRmWarps = 8;

__device__ __forceinline__ void split3_bf16(float v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const uint32_t b0 = __float_as_uint(v);
  const float r1 = v - __uint_as_float(b0 & 0xffff0000u);
  const uint32_t b1 = __float_as_uint(r1);
  const float r2 = r1 - __uint_as_float(b1 & 0xffff0000u);
  hi = b0 >> 16;
  mid = b1 >> 16;
  lo = __float_as_uint(r2) >> 16;
}

__global__ void __launch_bounds__(kRmWarps * 32) router_mma_kernel(const uint16_t* __restrict__ x, int T, int d, int E,
                                                                   const float* __restrict__ Wr,
                                                                   const float* __restrict__ b,
                                                                   float* __restrict__ logits) {
  pdl_enter();
  __shared__ float part[kRmWarps][kRmTok][kRmExp];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int t0 = blockIdx.x * kRmTok, e0 = blockIdx.y * kRmExp;
  const int slice = d / kRmWarps;
  const int ta = t0 + g, tb = t0 + g + 8, ew = e0 + g;
  const bool va = ta < T, vb = tb < T;
  const uint32_t* xa = reinterpret_cast<const uint32_t*>(x + (size_t)(va ? ta : 0) * d);
  const uint32_t* xb = reinterpret_cast<const uint32_t*>(x + (size_t)(vb ? tb : 0) * d);
  const float* wr = Wr + (size_t)(ew < E ? ew : 0) * d;
  // the CTA's router rows are contiguous: one bulk prefetch pulls them into L2 at
  // full bandwidth, so the warps' small loads below meet L2 instead of DRAM
  if (threadIdx.x == 0) {
    const int ne = min(kRmExp, E - e0);
    bulk_prefetch_l2(Wr + (size_t)e0 * d, (uint32_t)ne * (uint32_t)d * 4u);
  }
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4  // four steps' loads in flight per round trip
  for (int kk = warp * slice; kk < (warp + 1) * slice; kk += 16) {
    uint32_t A[4];
    A[0] = va ? xa[(kk + 2 * c) >> 1] : 0u;
    A[1] = vb ? xb[(kk + 2 * c) >> 1] : 0u;
    A[2] = va ? xa[(kk + 8 + 2 * c) >> 1] : 0u;
    A[3] = vb ? xb[(kk + 8 + 2 * c) >> 1] : 0u;
    const float2 w0 = *reinterpret_cast<const float2*>(wr + kk + 2 * c);
    const float2 w1 = *reinterpret_cast<const float2*>(wr + kk + 8 + 2 * c);
    uint32_t h0, m0, l0, h1, m1, l1, h2, m2, l2, h3, m3, l3;
    split3_bf16(w0.x, h0, m0, l0);
    split3_bf16(w0.y, h1, m1, l1);
    split3_bf16(w1.x, h2, m2, l2);
    split3_bf16(w1.y, h3, m3, l3);
    // one 16-wide step summed from zero on the tensor core, then added in fp32
    float st[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16(st, A, h0 | (h1 << 16), h2 | (h3 << 16), st);
    mma_bf16(st, A, m0 | (m1 << 16), m2 | (m3 << 16), st);
    mma_bf16(st, A, l0 | (l1 << 16), l2 | (l3 << 16), st);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += st[i];
  }
  // D: acc[0..1] token g, experts 2c, 2c+1; acc[2..3] token g+8
  part[warp][g][2 * c] = acc[0];
  part[warp][g][2 * c + 1] = acc[1];
  part[warp][g + 8][2 * c] = acc[2];
  part[warp][g + 8][2 * c + 1] = acc[3];
  __syncthreads();
  if (threadIdx.x < kRmTok * kRmExp) {
    const int tok = threadIdx.x / kRmExp, ex = threadIdx.x % kRmExp;
    const int t = t0 + tok, e = e0 + ex;
    if (t < T && e < E) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kRmWarps; ++w) v += part[w][tok][ex];
      logits[(size_t)t * E + e] = v + (b ? b[e] : 0.f);
    }
  }
}

// The same product for many tokens: 64 tokens x 64 experts per CTA, K in chunks
// of 64 staged once in shared memory (x as bf16, Wr split into its three bf16
// parts), eight warps of 16 tokens x 32 experts.  Rows are padded to 72 elements
// so the fragment loads of a warp hit distinct banks.  Each 16-wide K step is
// summed on the tensor core from zero and added to the running fp32 sum, which
// keeps the logits as close to the exact value as a fp32 FMA chain.
constexpr int kRtT = 64, kRtE = 64, kRtK = 64, kRtPad = 72;

__global__ void __launch_bounds__(256) router_mma_tiled_kernel(const uint16_t* __restrict__ x, int T, int d, int E,
                                                               const float* __restrict__ Wr,
                                                               const float* __restrict__ b,
                                                               float* __restrict__ logits) {
  pdl_enter();
  __shared__ __align__(16) uint16_t xs[kRtT][kRtPad];
  __shared__ __align__(16) uint16_t wp[3][kRtE][kRtPad];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int wm = warp & 3, wn = warp >> 2;  // 16-token row block, 32-expert column block
  const int t0 = blockIdx.x * kRtT, e0 = blockIdx.y * kRtE;
  float acc[4][4] = {};
  // the next K chunk's global pieces are loaded into registers while the current
  // chunk is multiplied: x as two 16-byte pieces, Wr as four float4 per thread
  uint4 xr[2];
  float4 wr[4];
  auto load_chunk = [&](int k0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int piece = tid + i * 256, r = piece >> 3, c8 = (piece & 7) * 8;
      xr[i] = make_uint4(0, 0, 0, 0);
      if (t0 + r < T) xr[i] = *reinterpret_cast<const uint4*>(x + (size_t)(t0 + r) * d + k0 + c8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int piece = tid + i * 256, r = piece >> 4, c4 = (piece & 15) * 4;
      wr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < E) wr[i] = *reinterpret_cast<const float4*>(Wr + (size_t)(e0 + r) * d + k0 + c4);
    }
  };
  load_chunk(0);
  for (int k0 = 0; k0 < d; k0 += kRtK) {
    // x tile: 64 rows x 128 B
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int piece = tid + i * 256, r = piece >> 3, c8 = (piece & 7) * 8;
      *reinterpret_cast<uint4*>(&xs[r][c8]) = xr[i];
    }
    // Wr tile: 64 rows x 256 B, split into hi / mid / lo
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int piece = tid + i * 256, r = piece >> 4, c4 = (piece & 15) * 4;
      const float4 v = wr[i];
      uint32_t h[4], m[4], l[4];
      split3_bf16(v.x, h[0], m[0], l[0]);
      split3_bf16(v.y, h[1], m[1], l[1]);
      split3_bf16(v.z, h[2], m[2], l[2]);
      split3_bf16(v.w, h[3], m[3], l[3]);
      *reinterpret_cast<uint2*>(&wp[0][r][c4]) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
      *reinterpret_cast<uint2*>(&wp[1][r][c4]) = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
      *reinterpret_cast<uint2*>(&wp[2][r][c4]) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    }
    __syncthreads();
    if (k0 + kRtK < d) load_chunk(k0 + kRtK);
#pragma unroll
    for (int kk = 0; kk < kRtK; kk += 16) {
      uint32_t A[4];
      const int ra = wm * 16 + g;
      A[0] = *reinterpret_cast<const uint32_t*>(&xs[ra][kk + 2 * c]);
      A[1] = *reinterpret_cast<const uint32_t*>(&xs[ra + 8][kk + 2 * c]);
      A[2] = *reinterpret_cast<const uint32_t*>(&xs[ra][kk + 8 + 2 * c]);
      A[3] = *reinterpret_cast<const uint32_t*>(&xs[ra + 8][kk + 8 + 2 * c]);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int rb = wn * 32 + nt * 8 + g;
        // the three parts of one 16-wide step go into a fresh fragment, which is then
        // added in fp32: the tensor core's own accumulation never runs over long chains
        float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&wp[part][rb][kk + 2 * c]);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&wp[part][rb][kk + 8 + 2 * c]);
          mma_bf16(st, A, b0, b1, st);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] += st[i];
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int e = e0 + wn * 32 + nt * 8 + 2 * c;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int t = t0 + wm * 16 + g + 8 * h;
      if (t >= T) continue;
#pragma unroll
      for (int q = 0; q < 2; ++q)
        if (e + q < E) logits[(size_t)t * E + e + q] = acc[nt][2 * h + q] + (b ? b[e + q] : 0.f);
    }
  }
}

// ---------------------------------------------------------------- router on tcgen05 (many tokens)
//
// The same exact product on the 5th-generation tensor cores.  The fp32 router rows
// are first split once per call into their three bf16 parts, stored as a [3E, d]
// bf16 matrix (part p of expert e is row p*E + e).  A CTA owns 128 tokens (MMA M) x
// 64 experts: per 64-wide K block one TMA stage brings the token tile (16 KB) and the
// three part tiles (8 KB each) one after the other, so the stage's 192 weight rows
// are one MMA B operand (N = 192: columns 0-63 the hi parts, 64-127 mid, 128-191 lo)
// and the token tile is read once per K step.  One thread issues the block's four
// MMAs into a fresh tensor-memory accumulator; the four epilogue warps read each
// block's three part sums, add them (hi + mid) + lo, and add that to fp32 registers,
// so the tensor core's own accumulation never runs longer than one 64-wide block, as
// the short chains of the mma.sync kernels above.  Two accumulators alternate so the
// MMAs of block j + 1 run while block j is read.
// Roles: warp 0 TMA, warp 1 MMA issue and tensor-memory owner, warps 4-11 epilogue
// (warp 4 + 4h + q reads TMEM lanes 32q .. 32q + 31, one token each, for experts
// 32h .. 32h + 31 of the tile: one wait per block for all three parts).
constexpr int kRcM = 128, kRcN = 64, kRcK = 64, kRcStages = 4;
constexpr int kRcABytes = kRcM * kRcK * 2;            // 16 KB token tile
constexpr int kRcPBytes = kRcN * kRcK * 2;            // 8 KB per weight part
constexpr int kRcStageBytes = kRcABytes + 3 * kRcPBytes;
constexpr int kRcThreads = 384;
constexpr int kRcEpiWarps = 8;
constexpr int kRcCols = 3 * kRcN;                     // accumulator columns (three parts)
constexpr uint32_t kRcTmemCols = 512;                 // two accumulators of kRcCols
constexpr size_t kRcSmem = (size_t)kRcStages * kRcStageBytes + 1024 + 256;
static_assert(kRcStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(kRcSmem <= 227 * 1024, "shared memory budget");
static_assert(2 * kRcCols <= (int)kRcTmemCols, "tensor memory budget");

struct RouterTcArgs {
  CUtensorMap tmap_x;  // x [T, d] bf16, boxes of 64 K x 128 tokens
  CUtensorMap tmap_w;  // split router rows [3E, d] bf16, boxes of 64 K x 64 rows
  int T, d, E;
  const float* b;
  float* logits;
  DevStatus* st;
};

__global__ void router_split_kernel(const float* __restrict__ W, int64_t n, uint16_t* __restrict__ parts) {
  pdl_enter();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
    const float4 v = *reinterpret_cast<const float4*>(W + i);
    uint32_t h[4], m[4], l[4];
    split3_bf16(v.x, h[0], m[0], l[0]);
    split3_bf16(v.y, h[1], m[1], l[1]);
    split3_bf16(v.z, h[2], m[2], l[2]);
    split3_bf16(v.w, h[3], m[3], l[3]);
    *reinterpret_cast<uint2*>(parts + i) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    *reinterpret_cast<uint2*>(parts + n + i) = make_uint2(m[0] | (m[1] << 16), m[2] | (m[3] << 16));
    *reinterpret_cast<uint2*>(parts + 2 * n + i) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
  }
}

__global__ void __launch_bounds__(kRcThreads, 1) router_tc_kernel(const __grid_constant__ RouterTcArgs p) {
  pdl_enter();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(base + (size_t)kRcStages * kRcStageBytes);
  uint64_t* empty = full + kRcStages;  // MMA commit: the stage may be refilled
  uint64_t* accf = empty + kRcStages;  // [2] MMA commit: the block's sums are in TMEM
  uint64_t* acce = accf + 2;           // [2] one arrival per epilogue warp: the accumulator is free
  uint64_t* drain = acce + 2;          // MMA commit: every MMA done (before TMEM is freed)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kRcM, e0 = blockIdx.y * kRcN;
  const int nkb = p.d / kRcK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], kRcEpiWarps);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kRcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_x)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_w)) : "memory");
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kRcStages;
        if (kb >= kRcStages && !mbar_wait(&empty[s], ((kb / kRcStages) - 1) & 1, p.st, 60)) break;
        mbar_arrive_expect_tx(&full[s], (uint32_t)kRcStageBytes);
        const uint32_t dst = smem_u32(base + (size_t)s * kRcStageBytes);
        tma_load_2d(dst, &p.tmap_x, kb * kRcK, m0, &full[s]);
#pragma unroll
        for (int part = 0; part < 3; ++part)
          tma_load_2d(dst + (uint32_t)(kRcABytes + part * kRcPBytes), &p.tmap_w, kb * kRcK, part * p.E + e0,
                      &full[s]);
        issued = kb + 1;
      }
      // copies still in flight (only after a wait ran out) land before the CTA leaves
      for (int kb = issued > kRcStages ? issued - kRcStages : 0; kb < issued; ++kb)
        if (!mbar_wait(&full[kb % kRcStages], (kb / kRcStages) & 1, p.st, 61)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(kRcM, kRcCols);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kRcStages, b = kb & 1;
        if (!mbar_wait(&full[s], (kb / kRcStages) & 1, p.st, 62)) break;
        if (kb >= 2 && !mbar_wait(&acce[b], ((kb >> 1) - 1) & 1, p.st, 63)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(base + (size_t)s * kRcStageBytes);
        const uint32_t d = tmem_base + (uint32_t)(b * kRcCols);
#pragma unroll
        for (int ks = 0; ks < kRcK / 16; ++ks)
          umma_ss(d, umma_smem_desc(a0 + (uint32_t)(ks * 32)), umma_smem_desc(a0 + (uint32_t)(kRcABytes + ks * 32)),
                  idesc, ks != 0);
        umma_commit(&empty[s]);
        umma_commit(&accf[b]);
      }
      umma_commit(drain);
      mbar_wait(drain, 0, p.st, 64);
    }
  } else if (warp >= 4) {
    const int q = warp & 3, h = (warp - 4) >> 2;
    constexpr int kCols = kRcN / 2;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(h * kCols);
    float acc[kCols];
#pragma unroll
    for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int b = kb & 1;
      if (!mbar_wait(&accf[b], (kb >> 1) & 1, p.st, 65)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t hi[kCols], mid[kCols], lo[kCols];
      const uint32_t col = lane_addr + (uint32_t)(b * kRcCols);
      tmem_ld32(col, hi);
      tmem_ld32(col + kRcN, mid);
      tmem_ld32(col + 2 * kRcN, lo);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acce[b]);
#pragma unroll
      for (int i = 0; i < kCols; ++i)
        acc[i] += (__uint_as_float(hi[i]) + __uint_as_float(mid[i])) + __uint_as_float(lo[i]);
    }
    const int t = m0 + 32 * q + lane, eb = e0 + h * kCols;
    if (ok && t < p.T) {
      float* row = p.logits + (size_t)t * p.E;
#pragma unroll
      for (int i = 0; i < kCols; ++i)
        if (eb + i < p.E) row[eb + i] = acc[i] + (p.b ? p.b[eb + i] : 0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kRcTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------- top-k + gates
//
// One warp per token.  Lane l holds logits e = l, l+32, ...; k rounds of a
// warp arg-max over (value desc, index asc) pick the experts in order.  Gates:
// exp(l_j - l_max) normalised over the chosen k (renorm) or over all E.  With
// a shared expert (n_shared = 1) each token's row of ids / w has k + 1
// entries, the last naming bank entry E with weight 1.
template <int NPER>  // logits per lane: E <= 32 * NPER
__global__ void __launch_bounds__(256) topk_gates_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int renorm, int n_shared, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  float v[NPER];
  const int nper = (E + 31) / 32;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
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
    for (int i = 0; i < NPER; ++i) {
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
    for (int i = 0; i < NPER; ++i) {
      const int e = i * 32 + lane;
      if (i < nper && e < E) z += expf(v[i] - vmax);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  // rows of token t: its k routed experts, then the shared expert (bank entry E, weight 1)
  const int kt = k + n_shared;
  if (lane < k) {
    ids[(size_t)t * kt + lane] = my_id;
    w[(size_t)t * kt + lane] = my_e / z;
  } else if (lane < kt) {
    ids[(size_t)t * kt + lane] = E;
    w[(size_t)t * kt + lane] = 1.0f;
  }
}

// ---------------------------------------------------------------- forced selection
//
// Copies caller-given ids / gates into the working arrays.  Ids outside [0, E)
// become -1 (left out of the permutation) and flag kStatusCheck; a token that
// lists one expert twice also flags kStatusCheck.
__global__ void forced_select_kernel(const int32_t* __restrict__ fid, const float* __restrict__ fw, int T, int E,
                                     int k, int32_t* __restrict__ ids, float* __restrict__ w, DevStatus* st) {
  pdl_enter();
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

bool router_uses_tc(int T) { return T >= kRouterTcMinT; }

size_t router_split_bytes(int E, int d) { return (size_t)3 * E * d * 2; }

cudaError_t launch_router_logits(const uint16_t* x, int T, int d, int E, const float* w_router,
                                 const float* b_router, float* logits, uint16_t* w_split, DevStatus* st,
                                 cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (d % (kRmWarps * 16) || d % kRtK) return cudaErrorNotSupported;
  if (T <= 64) {
    const dim3 grid(ceil_div(T, kRmTok), ceil_div(E, kRmExp));
    if (cudaError_t e_ = launch_pdl(router_mma_kernel, dim3(grid), dim3(kRmWarps * 32), 0, s, x, T, d, E, w_router,
                                    b_router, logits)) return e_;
  } else if (!router_uses_tc(T) || w_split == nullptr) {
    const dim3 grid(ceil_div(T, kRtT), ceil_div(E, kRtE));
    if (cudaError_t e_ = launch_pdl(router_mma_tiled_kernel, dim3(grid), dim3(256), 0, s, x, T, d, E, w_router,
                                    b_router, logits)) return e_;
  } else {
    if (d % kRcK || (reinterpret_cast<uintptr_t>(w_split) & 15u)) return cudaErrorNotSupported;
    const int64_t n = (int64_t)E * d;
    const int64_t nthreads = n / 4;
    const int sg = (int)(nthreads / 256 < 148 * 8 ? (nthreads + 255) / 256 : 148 * 8);
    if (cudaError_t e_ = launch_pdl(router_split_kernel, dim3(sg), dim3(256), 0, s, w_router, n, w_split)) return e_;
    RouterTcArgs a = {};
    cudaError_t err = encode_rows_map(&a.tmap_x, x, T, d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kRcK, kRcM);
    if (err != cudaSuccess) return err;
    if ((err = encode_rows_map(&a.tmap_w, w_split, 3 * E, d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kRcK, kRcN)) !=
        cudaSuccess)
      return err;
    a.T = T;
    a.d = d;
    a.E = E;
    a.b = b_router;
    a.logits = logits;
    a.st = st;
    static int attr[64] = {};
    if ((err = ensure_smem_attr(router_tc_kernel, kRcSmem, attr)) != cudaSuccess) return err;
    const dim3 grid(ceil_div(T, kRcM), ceil_div(E, kRcN));
    if (cudaError_t e_ = launch_pdl(router_tc_kernel, dim3(grid), dim3(kRcThreads), kRcSmem, s, a)) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_topk_gates(const float* logits, int T, int E, int k, int renorm, int n_shared, int32_t* ids,
                              float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  auto* kern = (E <= 256) ? topk_gates_kernel<8> : topk_gates_kernel<kMaxE / 32>;
  const cudaError_t e =
      launch_pdl(kern, dim3(ceil_div(T, 8)), dim3(256), 0, s, logits, T, E, k, renorm, n_shared, ids, w);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_forced_select(const int32_t* forced_ids, const float* forced_w, int T, int E, int k,
                                 int32_t* ids, float* w, DevStatus* st, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (cudaError_t e_ = launch_pdl(forced_select_kernel, dim3(ceil_div(T * k, 256)), dim3(256), 0, s, forced_ids,
                                  forced_w, T, E, k, ids, w, st)) return e_;
  return cudaGetLastError();
}

}  // namespace bitmoe
