// One decode step of the attention layer that sits beside each MoE layer: grouped-query
// attention over a bf16 key/value cache with a sliding window (or the whole context),
// per-head RMS norm on queries and keys, rotary encoding and learned sinks.
//
// "Flint 40B : Best Mid Sized LLM", transcript 03:05 (32 query heads, 4 key/value
// heads of 128; 35 of the mixture layers attend over a window of 513 tokens with rotary
// encoding, the rest over the whole context without it) and 03:36 (per-head RMS norm on
// queries and keys, learned attention sinks); 06:11 (dedicated attention kernels).
//
// For one token the step is four launches, chained with programmatic dependent launch:
//   1. proj     q|k|v = Wqkv x (x the RMS-normalised residual in the pre-norm form, the
//               norm taken in the same launch): the int4 rows stacked; a CTA per 16-row tile, its eight
//               warps splitting the tile's 128-column chunks (so a short matrix still
//               spreads over every SM) and adding their sums in shared memory
//   2. split    a CTA per (key/value head, span of the window): RMS norm and rotation
//               of the group's 8 query heads (and, in the CTA that holds position pos,
//               of the new key, which it writes with the value into the cache), then an
//               online softmax over its span on the tensor cores; the four warps' results
//               merge into one (max, sum, output) record per query head
//   3. combine  per query head the records and the sink merge into one output, bf16
//   4. proj     out = residual + Wo attn, the residual added in the epilogue
// The cache is head-major, [key/value head][position][128], so the span one CTA attends is
// one contiguous run of rows per head.
// Step 2 reads the window's keys and values once per key/value head (the 8 query heads of
// a group share every staged tile), so at long context it is the HBM-bound part: its
// loads are cp.async into per-warp rings, and the first tiles are requested before the
// kernel waits for the projection (no cache row it reads there is written by it).
#include <math.h>

#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kHd = kAttnHeadDim;     // 128
constexpr int kQPerKv = kAttnGroup;   // query heads per key/value head
constexpr int kWarps = 4;             // warps per split CTA
constexpr int kTile = 16;             // positions per staged tile: one k16 step of P V
constexpr int kStages = 3;            // tiles in flight per warp
constexpr int kRowBytes = kHd * 2;    // one cache row of one head, bf16
constexpr int kTileBytes = kTile * kRowBytes;     // 4 KB of keys (or values)
constexpr int kStageBytes = 2 * kTileBytes;       // keys, then values
constexpr int kWarpRing = kStages * kStageBytes;  // 24 KB
constexpr int kRingBytes = kWarps * kWarpRing;    // 96 KB
// after the rings: normalised queries [8][128] f32, the new key and value rows [2][128]
// bf16, the rotation's cos and sin [2][64] f32
constexpr int kQnOff = kRingBytes;
constexpr int kKvNewOff = kQnOff + kQPerKv * kHd * 4;
constexpr int kRotOff = kKvNewOff + 2 * kHd * 2;
constexpr int kSplitSmem = kRotOff + kHd * 4;
static_assert(2 * (kSplitSmem + 1024) <= 228 * 1024, "two split CTAs per SM");
static_assert(kWarps * kQPerKv * (kHd + 2) * 4 <= kRingBytes, "the warp merge reuses the rings");
static_assert(kTile * kWarps == 64, "chunks are multiples of 64 positions");

constexpr int kProjWarps = 8;
constexpr int kProjBatch = 4;  // chunks a warp holds in registers at once

// 2 pi split for the reduction of the rotation angle (Cody and Waite): the double
// nearest 2 pi and the remainder.
constexpr double kTwoPiHi = 6.283185307179586;
constexpr double kTwoPiLo = 2.4492935982947064e-16;
constexpr double kInvTwoPi = 0.15915494309189535;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// (x0, x1) as a bf16 pair rounded to nearest (low half x0) and the pair of what it left.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 16-byte asynchronous copy global -> shared.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Byte offset of 16-byte piece ch (8 dimensions) of row r in a staged tile: the piece
// index is XOR-ed with the row's low three bits, so the eight rows one ldmatrix reads at
// the same piece fall in eight different bank groups.
__device__ __forceinline__ uint32_t tile_off(int r, int ch) { return r * kRowBytes + ((ch ^ (r & 7)) << 4); }

__device__ __forceinline__ float scale_at(uint2 s, int gg) {
  const uint32_t w = (gg < 2) ? s.x : s.y;
  const uint16_t b = (gg & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t word_at(const uint4& q, int gg) {
  return gg == 0 ? q.x : gg == 1 ? q.y : gg == 2 ? q.z : q.w;
}

// ---------------------------------------------------------------- projections

struct ProjArgs {
  const uint16_t* x;      // [K] bf16 (with prenorm: the residual, normalised here)
  const uint8_t* w;       // packed int4 [rows, K]
  int K, rows;
  int prenorm;            // x <- bf16(x / sqrt(mean(x^2) + eps)) before the product
  float eps;
  float* y;               // [rows] W x (fp32), or with resid the unrounded sum (nullable)
  const uint16_t* resid;  // [rows] bf16 or null: out = resid + W x
  uint16_t* out;          // [rows] bf16 (with resid)
  int early;              // the weights are read before the wait on the kernel before
};

// y = W x for one token.  CTA b takes tile b (rows 16b .. 16b + 15); warp w its chunks w,
// w + 8, ...  Each chunk is the LM head's fragment layout: per 32-column group two m16n8k16
// fp16 steps of the dequantised nibbles against x (every n column holds the token, so
// any lane's first column is the row sum), scaled by the group's fp16 scale in fp32.
// x is staged as fp16 times 2^s (largest magnitude in [2^14, 2^15): exact for bf16 input).
// With prenorm the residual is first RMS-normalised in fp32 and rounded to bf16, as a
// pre-norm layer feeds its block.
__global__ void __launch_bounds__(kProjWarps * 32) attn_proj_kernel(const __grid_constant__ ProjArgs a) {
  extern __shared__ __align__(16) unsigned char psm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(psm);
  __shared__ float red[kProjWarps][kTileRows];
  __shared__ uint32_t wmax[kProjWarps];
  __shared__ float wss[kProjWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int nch = a.K / kChunkK;
  const uint8_t* tile = a.w + (size_t)blockIdx.x * tile_bytes(a.K);
  uint4 q0[kProjBatch], q1[kProjBatch];
  uint2 s0[kProjBatch], s1[kProjBatch];
  auto load = [&](int base) {
#pragma unroll
    for (int i = 0; i < kProjBatch; ++i) {
      const int ch = base + i * kProjWarps;
      if (ch < nch) {
        const uint8_t* cw = tile + (size_t)ch * kChunkBytes;
        q0[i] = __ldg(reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16));
        q1[i] = __ldg(reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16));
        s0[i] = __ldg(reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8));
        s1[i] = __ldg(reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8));
      }
    }
  };
  if (a.early) {
    load(warp);
  } else if (tid == 0) {
    // the tile into L2 while the kernel before finishes: L2 is where every write lands,
    // so the loads after the wait see the current weights whatever that kernel wrote
    bulk_prefetch_l2(tile, (uint32_t)tile_bytes(a.K));
  }
  pdl_enter();
  if (!a.early) load(warp);

  // stage x: the largest magnitude (and with prenorm the sum of squares), then x 2^s as fp16
  uint32_t m = 0;
  float ss = 0.f;
  for (int i = tid * 8; i < a.K; i += kProjWarps * 32 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + i);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, max(w4[j] & 0x7fffu, (w4[j] >> 16) & 0x7fffu));
      const float lo = __uint_as_float(w4[j] << 16), hi = __uint_as_float(w4[j] & 0xffff0000u);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
  }
  if (lane == 0) {
    wmax[warp] = m;
    wss[warp] = ss;
  }
  __syncthreads();
  m = 0;
  ss = 0.f;
#pragma unroll
  for (int w = 0; w < kProjWarps; ++w) {
    m = max(m, wmax[w]);
    ss += wss[w];
  }
  // with prenorm every element becomes bf16(x / rms): rounding keeps order, so the largest
  // magnitude is bf16(max |x| / rms)
  const float inv = a.prenorm ? 1.0f / sqrtf(ss / (float)a.K + a.eps) : 1.0f;
  if (a.prenorm) m = (uint32_t)f2bf(bf16f((uint16_t)m) * inv) & 0x7fffu;
  const int se = f16_row_exponent(m);
  const float f = pow2i(se);
  for (int i = tid * 8; i < a.K; i += kProjWarps * 32 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + i);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float lo = __uint_as_float(w4[j] << 16), hi = __uint_as_float(w4[j] & 0xffff0000u);
      if (a.prenorm) {
        lo = bf16f(f2bf(lo * inv));
        hi = bf16f(f2bf(hi * inv));
      }
      const __half2 h2 = __floats2half2_rn(lo * f, hi * f);
      o[j] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(xs + i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();

  float acc[2] = {0.f, 0.f};  // rows g and g + 8
  for (int base = warp; base < nch; base += kProjWarps * kProjBatch) {
    if (base != warp) load(base);
#pragma unroll
    for (int i = 0; i < kProjBatch; ++i) {
      const int ch = base + i * kProjWarps;
      if (ch >= nch) break;
#pragma unroll
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        uint32_t p0[4], p1[4];
        nib_pairs4_f16(word_at(q0[i], gg), p0);
        nib_pairs4_f16(word_at(q1[i], gg), p1);
        const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]};
        const uint32_t a1[4] = {p0[2], p1[2], p0[3], p1[3]};
        const uint4 xb = *reinterpret_cast<const uint4*>(xs + col);
        float dd[4];
        mma_f16_z(dd, a0, xb.x, xb.y);
        mma_f16(dd, a1, xb.z, xb.w, dd);
        acc[0] = fmaf(scale_at(s0[i], gg), dd[0], acc[0]);
        acc[1] = fmaf(scale_at(s1[i], gg), dd[2], acc[1]);
      }
    }
  }
  if (c == 0) {
    red[warp][g] = acc[0];
    red[warp][g + 8] = acc[1];
  }
  __syncthreads();
  if (tid < kTileRows) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kProjWarps; ++w) v += red[w][tid];
    v *= pow2i(-se);
    const int row = blockIdx.x * kTileRows + tid;
    if (a.resid) {
      v += bf16f(a.resid[row]);
      a.out[row] = f2bf(v);
      if (a.y) a.y[row] = v;
    } else {
      a.y[row] = v;
    }
  }
}

// ---------------------------------------------------------------- split-KV attention

struct SplitArgs {
  const float* qkv;     // [(nq + 2 nkv) * 128] projections
  uint16_t* k_cache;    // [nkv, max_len, 128] bf16: each head's rows contiguous
  uint16_t* v_cache;
  int64_t max_len;
  int nq, nkv;
  int64_t lo, pos;      // positions lo .. pos are attended
  int64_t chunk;        // positions per CTA, a multiple of 64
  int nsplit;           // CTAs per key/value head
  int rope;
  float eps, scale2;    // RMS-norm epsilon, log2(e) / sqrt(128)
  float* part;          // [nq][nsplit][kAttnPart]: max, sum, 2 unused, unnormalised output
  double inv_freq[kHd / 2];  // rope_theta^(-2i/128)
};

// Grid (nkv, nsplit), 4 warps.  Warp w of CTA (g, sp) runs all 8 query heads of group g
// over its quarter of the CTA's span, 16 positions per step:
//   S = Q K^T   m16n8k16 bf16: A rows 0..7 the heads' queries rounded to bf16, rows 8..15
//               what that rounding left (so S = hi + lo carries q to about 2^-17), B the
//               staged keys (ldmatrix), two n tiles of 8 positions
//   online softmax per head (the four lanes of a quad hold one head's 16 scores)
//   O += P V    A = P split the same way into bf16 hi and lo rows (taken straight from the
//               S fragments), B the staged values (ldmatrix.trans), 16 n tiles of 8 dims
// Every position of the span belongs to exactly one warp.  A warp stages its tiles itself
// with cp.async (a tile of one head is 4 KB of contiguous keys and 4 KB of values); the
// rows past the span's end are zero-filled and masked out of the softmax.
__global__ void __launch_bounds__(kWarps * 32, 2) attn_split_kernel(const __grid_constant__ SplitArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* qn = reinterpret_cast<float*>(smem + kQnOff);
  uint16_t* kvnew = reinterpret_cast<uint16_t*>(smem + kKvNewOff);
  float* rot = reinterpret_cast<float*>(smem + kRotOff);
  const int g = blockIdx.x, sp = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int64_t hi = a.pos + 1;
  const int64_t c0 = a.lo + (int64_t)sp * a.chunk;
  const int64_t c1 = min(hi, c0 + a.chunk);
  const int64_t sub = a.chunk / kWarps;
  const int64_t w0 = c0 + (int64_t)warp * sub;
  const int64_t w1 = min(c1, w0 + sub);
  const int ntiles = w1 > w0 ? (int)((w1 - w0 + kTile - 1) / kTile) : 0;
  unsigned char* ring_p = smem + warp * kWarpRing;
  const uint32_t ring = smem_u32(ring_p);
  // lane l copies piece l % 16 of rows l / 16, l / 16 + 2, ..., l / 16 + 14 of a tile; row
  // r0 + 2j has low bits r0 | (2j & 6), so its swizzled piece is (piece ^ r0) ^ (2j & 6)
  const int r0 = lane >> 4, cx = (lane & 15) ^ r0;
  const size_t lane_src = ((size_t)g * a.max_len + r0) * kHd + (lane & 15) * 8;
  const uint16_t* kl = a.k_cache + lane_src;
  const uint16_t* vl = a.v_cache + lane_src;

  // tile t of this warp into stage t % kStages: 16 rows x 16 pieces of keys, then values
  auto issue = [&](int t) {
    const uint32_t st = ring + (t % kStages) * kStageBytes + r0 * kRowBytes;
    const int64_t p0 = w0 + (int64_t)t * kTile;
    const size_t src = (size_t)p0 * kHd;
    const bool full = p0 + kTile <= w1;
#pragma unroll
    for (int j = 0; j < kTile / 2; ++j) {
      const uint32_t dst = st + j * 2 * kRowBytes + ((cx ^ ((2 * j) & 6)) << 4);
      if (full || p0 + r0 + 2 * j < w1) {
        cp_async16(dst, kl + src + (size_t)j * 2 * kHd);
        cp_async16(dst + kTileBytes, vl + src + (size_t)j * 2 * kHd);
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst + kTileBytes), "r"(0u) : "memory");
      }
    }
  };
  // the first tiles stream in while the kernel before finishes: rows < pos were written
  // by earlier steps, and row pos (stale here) is replaced in shared memory below
#pragma unroll
  for (int t = 0; t < kStages; ++t) {
    if (t < ntiles) issue(t);
    cp_async_commit();
  }
  pdl_enter();

  // the heads this warp normalises (items w, w + 4, w + 8 of: the 8 query heads, then in
  // the CTA that holds pos the new key and value), loaded together
  const bool owns_pos = (sp == a.nsplit - 1);
  const int items = kQPerKv + (owns_pos ? 2 : 0);
  constexpr int kItemsPerWarp = (kQPerKv + 2 + kWarps - 1) / kWarps;
  float v[kItemsPerWarp][4];
#pragma unroll
  for (int k = 0; k < kItemsPerWarp; ++k) {
    const int it = warp + k * kWarps;
    if (it < items) {
      const int head = it < kQPerKv ? g * kQPerKv + it : (it == kQPerKv ? a.nq + g : a.nq + a.nkv + g);
      const float* src = a.qkv + (size_t)head * kHd;
#pragma unroll
      for (int i = 0; i < 4; ++i) v[k][i] = src[lane + 32 * i];
    }
  }
  // rotation angles: pos * inv_freq[i] reduced to [-pi, pi] in fp64, then sin and cos
  if (a.rope && tid < kHd / 2) {
    const double ang = (double)a.pos * a.inv_freq[tid];
    const double k = rint(ang * kInvTwoPi);
    const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, ang));
    float s, co;
    sincosf((float)r, &s, &co);
    rot[tid] = co;
    rot[kHd / 2 + tid] = s;
  }
  __syncthreads();
  // norm and rotation of the query heads and the new key (the value is stored as it is);
  // the key and value go to the cache and to shared memory as bf16.  Lane l holds
  // elements l, l + 32, l + 64, l + 96: each rotated pair (i, i + 64) in one lane.
#pragma unroll
  for (int k = 0; k < kItemsPerWarp; ++k) {
    const int it = warp + k * kWarps;
    if (it >= items) break;
    float* x = v[k];
    if (it <= kQPerKv) {
      const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
      const float rn = 1.0f / sqrtf(ss / (float)kHd + a.eps);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= rn;
      if (a.rope) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float co = rot[lane + 32 * i], s = rot[kHd / 2 + lane + 32 * i];
          const float x0 = x[i], x1 = x[i + 2];
          x[i] = x0 * co - x1 * s;
          x[i + 2] = x0 * s + x1 * co;
        }
      }
    }
    if (it < kQPerKv) {
#pragma unroll
      for (int i = 0; i < 4; ++i) qn[it * kHd + lane + 32 * i] = x[i];
    } else {
      const int which = it - kQPerKv;  // 0 key, 1 value
      uint16_t* dst = (which ? a.v_cache : a.k_cache) + ((size_t)g * a.max_len + (size_t)a.pos) * kHd;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint16_t b = f2bf(x[i]);
        dst[lane + 32 * i] = b;
        kvnew[which * kHd + lane + 32 * i] = b;
      }
    }
  }
  __syncthreads();

  // query fragments of the 8 k16 steps: rows gq (bf16 of q) and gq + 8 (the remainder)
  uint32_t qa[kHd / 16][4];
#pragma unroll
  for (int ks = 0; ks < kHd / 16; ++ks) {
    const float* qr = qn + gq * kHd + ks * 16 + 2 * cq;
    split_bf16x2(qr[0], qr[1], qa[ks][0], qa[ks][1]);
    split_bf16x2(qr[8], qr[9], qa[ks][2], qa[ks][3]);
  }

  float m = -INFINITY, l = 0.f;
  float o[kHd / 8][4];
#pragma unroll
  for (int nd = 0; nd < kHd / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

  // group k of this thread's copies holds tile k: before step t, kStages + t groups are
  // committed, so leaving the newest kStages - 1 pending completes tile t
  for (int t = 0; t < ntiles; ++t) {
    const int stg = t % kStages;
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint32_t kb = ring + stg * kStageBytes;
    const uint32_t vb = kb + kTileBytes;
    const int64_t p0 = w0 + (int64_t)t * kTile;
    if (owns_pos && a.pos >= p0 && a.pos < p0 + kTile) {  // the new row, as written to the cache
      const int r = (int)(a.pos - p0), which = lane >> 4, ch = lane & 15;
      const uint4 v = *reinterpret_cast<const uint4*>(kvnew + which * kHd + ch * 8);
      *reinterpret_cast<uint4*>(ring_p + stg * kStageBytes + which * kTileBytes + tile_off(r, ch)) = v;
      __syncwarp();
    }
    // scores of positions p0 + {2cq, 2cq + 1} (n tile 0) and p0 + 8 + {2cq, 2cq + 1} (n tile 1)
    float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kHd / 16; ++ks) {
      const int j = lane >> 3, r = 8 * (j >> 1) + (lane & 7);
      uint32_t b[4];
      ldsm_x4(b, kb + tile_off(r, 2 * ks + (j & 1)));
      mma_bf16(s0, qa[ks], b[0], b[1], s0);
      mma_bf16(s1, qa[ks], b[2], b[3], s1);
    }
    const int nv = (int)min((int64_t)kTile, w1 - p0);
    // scores in base 2: s log2(e), so e^(s - m) = 2^(s2 - m2)
    float sc[4] = {(s0[0] + s0[2]) * a.scale2, (s0[1] + s0[3]) * a.scale2, (s1[0] + s1[2]) * a.scale2,
                   (s1[1] + s1[3]) * a.scale2};
    const int pp[4] = {2 * cq, 2 * cq + 1, 8 + 2 * cq, 9 + 2 * cq};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (pp[i] >= nv) sc[i] = -INFINITY;
    float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);  // finite: the tile's first row is in the span
    const float corr = exp2f(m - mn);
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = exp2f(sc[i] - mn);
    l = fmaf(l, corr, (p[0] + p[1]) + (p[2] + p[3]));
    m = mn;
    if (__any_sync(0xffffffffu, corr != 1.0f)) {  // some head's running max moved
#pragma unroll
      for (int nd = 0; nd < kHd / 8; ++nd) {
        o[nd][0] *= corr;
        o[nd][1] *= corr;
        o[nd][2] *= corr;
        o[nd][3] *= corr;
      }
    }
    uint32_t pa[4];
    split_bf16x2(p[0], p[1], pa[0], pa[1]);
    split_bf16x2(p[2], p[3], pa[2], pa[3]);
#pragma unroll
    for (int pr = 0; pr < kHd / 16; ++pr) {
      const int j = lane >> 3, r = 8 * (j & 1) + (lane & 7);
      uint32_t b[4];
      ldsm_x4_t(b, vb + tile_off(r, 2 * pr + (j >> 1)));
      mma_bf16(o[2 * pr], pa, b[0], b[1], o[2 * pr]);
      mma_bf16(o[2 * pr + 1], pa, b[2], b[3], o[2 * pr + 1]);
    }
    __syncwarp();  // the stage is read before it is refilled with tile t + kStages
    if (t + kStages < ntiles) issue(t + kStages);
    cp_async_commit();
  }
  cp_async_wait<0>();
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);

  // merge the four warps: the rings become [warp][head] max, sum and output rows
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + kWarps * kQPerKv;
  float* ow = lw + kWarps * kQPerKv;
  if (cq == 0) {
    mw[warp * kQPerKv + gq] = m;
    lw[warp * kQPerKv + gq] = l;
  }
#pragma unroll
  for (int nd = 0; nd < kHd / 8; ++nd) {
    float* orow = ow + (warp * kQPerKv + gq) * kHd + nd * 8 + 2 * cq;
    orow[0] = o[nd][0] + o[nd][2];
    orow[1] = o[nd][1] + o[nd][3];
  }
  __syncthreads();
  const int hh = tid >> 4, d0 = (tid & 15) * 8;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * kQPerKv + hh]);
  float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float e = exp2f(mw[w * kQPerKv + hh] - M);  // 0 for a warp without positions
    L = fmaf(e, lw[w * kQPerKv + hh], L);
    const float* orow = ow + (w * kQPerKv + hh) * kHd + d0;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmaf(e, orow[i], acc[i]);
  }
  float* rec = a.part + ((size_t)(g * kQPerKv + hh) * a.nsplit + sp) * kAttnPart;
  if ((tid & 15) == 0) {
    rec[0] = M * 0.69314718055994531f;  // back to natural-log units
    rec[1] = L;
  }
  *reinterpret_cast<float4*>(rec + 4 + d0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
  *reinterpret_cast<float4*>(rec + 8 + d0) = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// One CTA of 16 warps per query head: warp w loads the records w, w + 16, ... at once
// (lane l dimensions 4l .. 4l + 3), the CTA takes the common max, then the warps' sums
// scaled to it and the sink:
//   out = sum_r e^(m_r - M) o_r / (e^(sink - M) + sum_r e^(m_r - M) l_r)
constexpr int kCombineWarps = 16;
constexpr int kRecPerWarp = (kAttnMaxSplits + kCombineWarps - 1) / kCombineWarps;
__global__ void __launch_bounds__(kCombineWarps * 32) attn_combine_kernel(const float* __restrict__ part, int nsplit,
                                                                         const float* __restrict__ sinks,
                                                                         uint16_t* __restrict__ attn) {
  pdl_enter();
  __shared__ __align__(16) float sacc[kCombineWarps][kHd];
  __shared__ float sl[kCombineWarps], smax[kCombineWarps];
  const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* ph = part + (size_t)h * nsplit * kAttnPart;
  float mr[kRecPerWarp], lr[kRecPerWarp];
  float4 vr[kRecPerWarp];
  float mloc = -INFINITY;
#pragma unroll
  for (int i = 0; i < kRecPerWarp; ++i) {
    const int r = warp + i * kCombineWarps;
    if (r < nsplit) {
      const float* pr = ph + (size_t)r * kAttnPart;
      mr[i] = pr[0];
      lr[i] = pr[1];
      vr[i] = *reinterpret_cast<const float4*>(pr + 4 + 4 * lane);
    } else {
      mr[i] = -INFINITY;
      lr[i] = 0.f;
      vr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    mloc = fmaxf(mloc, mr[i]);
  }
  if (lane == 0) smax[warp] = mloc;
  __syncthreads();
  const float sink = sinks ? sinks[h] : -INFINITY;
  float M = sink;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, smax[w]);  // finite: record 0 exists
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
#pragma unroll
  for (int i = 0; i < kRecPerWarp; ++i) {
    const float e = expf(mr[i] - M);  // 0 for an absent record
    L = fmaf(e, lr[i], L);
    acc.x = fmaf(e, vr[i].x, acc.x);
    acc.y = fmaf(e, vr[i].y, acc.y);
    acc.z = fmaf(e, vr[i].z, acc.z);
    acc.w = fmaf(e, vr[i].w, acc.w);
  }
  *reinterpret_cast<float4*>(&sacc[warp][4 * lane]) = acc;
  if (lane == 0) sl[warp] = L;
  __syncthreads();
  if (tid < kHd) {
    float A = 0.f, Lt = sinks ? expf(sink - M) : 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      A += sacc[w][tid];
      Lt += sl[w];
    }
    attn[(size_t)h * kHd + tid] = f2bf(A / Lt);
  }
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (n[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 148;
  }
  return n[dev];
}

}  // namespace

AttnPlan attn_plan(int64_t span, int nkv) {
  int target = 2 * sm_count() / (nkv > 0 ? nkv : 1);
  target = target < 1 ? 1 : (target > kAttnMaxSplits ? kAttnMaxSplits : target);
  int64_t chunk = (span + target - 1) / target;
  chunk = (chunk + 63) / 64 * 64;
  if (chunk < 64) chunk = 64;
  AttnPlan p;
  p.chunk = chunk;
  p.nsplit = (int)((span + chunk - 1) / chunk);
  return p;
}

cudaError_t launch_attn_decode(const AttnLaunch& L, cudaStream_t s) {
  const int nq = L.nq, nkv = L.nkv, rows = (nq + 2 * nkv) * kHd;
  // 1. q | k | v
  const ProjArgs p1 = {L.prenorm ? L.resid : L.x, L.wqkv, L.d, rows, L.prenorm, L.eps, L.qkv, nullptr, nullptr, 0};
  cudaError_t e =
      launch_pdl(attn_proj_kernel, dim3(rows / kTileRows), dim3(kProjWarps * 32), (size_t)L.d * 2, s, p1);
  if (e != cudaSuccess) return e;
  // 2. the window in splits
  static int attr[64] = {};
  if ((e = ensure_smem_attr(attn_split_kernel, (size_t)kSplitSmem, attr)) != cudaSuccess) return e;
  SplitArgs a;
  a.qkv = L.qkv;
  a.k_cache = L.k_cache;
  a.v_cache = L.v_cache;
  a.max_len = L.max_len;
  a.nq = nq;
  a.nkv = nkv;
  a.lo = L.window > 0 ? (L.pos - L.window + 1 > 0 ? L.pos - L.window + 1 : 0) : 0;
  a.pos = L.pos;
  const AttnPlan plan = attn_plan(L.pos + 1 - a.lo, nkv);
  a.chunk = plan.chunk;
  a.nsplit = plan.nsplit;
  a.rope = L.rope;
  a.eps = L.eps;
  a.scale2 = (float)(1.4426950408889634 / sqrt((double)kHd));
  a.part = L.part;
  {  // the angle steps of this base, kept per host thread while the base is unchanged
    thread_local double theta = -1.0;
    thread_local double inv[kHd / 2];
    if (L.rope && theta != L.theta) {
      for (int i = 0; i < kHd / 2; ++i) inv[i] = pow(L.theta, -2.0 * (double)i / (double)kHd);
      theta = L.theta;
    }
    for (int i = 0; i < kHd / 2; ++i) a.inv_freq[i] = L.rope ? inv[i] : 0.0;
  }
  if ((e = launch_pdl(attn_split_kernel, dim3(nkv, a.nsplit), dim3(kWarps * 32), (size_t)kSplitSmem, s, a)) !=
      cudaSuccess)
    return e;
  // 3. merge with the sinks
  if ((e = launch_pdl(attn_combine_kernel, dim3(nq), dim3(kCombineWarps * 32), 0, s, (const float*)L.part, a.nsplit,
                      L.sinks, L.attn)) != cudaSuccess)
    return e;
  // 4. output projection plus the residual
  const ProjArgs p2 = {L.attn, L.wo, nq * kHd, L.d, 0, 0.f, L.out_f32, L.resid, L.out, 1};
  if ((e = launch_pdl(attn_proj_kernel, dim3(L.d / kTileRows), dim3(kProjWarps * 32), (size_t)nq * kHd * 2, s,
                      p2)) != cudaSuccess)
    return e;
  return cudaGetLastError();
}

}  // namespace bitmoe
