// Expert FFN kernels: a = Wg x, u = Wu x, h = silu(a) * u, y = Wd h, with int4
// group-32 weights ("Flint 40B : Best Mid Sized LLM", transcript 06:11:
// kernels for low-bit matrix projections; 02:35: experts of a mixture layer).
//
// Work unit = (expert e, 16-row weight tile, block of up to 16 of e's grouped
// rows).  One elected thread stages the unit with TMA bulk copies (the weight
// tiles in the packed layout and the unit's activation rows) on an mbarrier;
// four warps split the reduction dimension by 128-column chunks.
//
// Arithmetic.  The int4 values are turned into exact fp16 integers (one shift
// per 8 nibbles with the magic-number conversion) and multiplied on the tensor
// cores with mma.sync m16n8k16 (weights = A, up to 8 tokens = B).  The bf16
// activation rows are staged as fp16 scaled by a power of two per row, which
// is exact (the largest |x| lands in [2^14, 2^15)) and undone on the sums.  Each mma pair covers
// exactly one 32-column group, so its fp32 result is the group's exact-input
// partial sum, which is then scaled by the group's fp16 scale in fp32: the
// dequantised weight q*s is never rounded.  h enters the down projection as
// an fp16 pair hi + lo (about 22 significant bits).
//
// NVFP4 banks (kFp4): each E2M1 code times its E4M3 block scale is an exact
// fp16 weight, so the weights enter the MMAs in fp16 with the scale already
// applied, a 128-column chunk's MMAs chain in the accumulator and the chunks
// add in fp32; the activation rows are turned into fp16 scaled by a power of
// two per row (exact, undone on the sums) and the tensor scale multiplies the
// result.
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kNT = kTokBlock / 8;  // n-tiles of 8 tokens per unit

__device__ __forceinline__ float scale_at(uint2 s, int gg) {
  const uint32_t w = (gg < 2) ? s.x : s.y;
  const uint16_t b = (gg & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
  return __half2float(__ushort_as_half(b));
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

// NVFP4: A fragments of two k16 steps for rows g (word w0, block scale byte s0)
// and g+8 (w1, s1), each weight the exact fp16 code times its block scale.
__device__ __forceinline__ void frag_fp4(uint32_t w0, uint32_t w1, uint32_t s0, uint32_t s1, uint32_t (&a)[2][4]) {
  uint32_t p0[4], p1[4];
  e2m1x8_f16_scaled(w0, e4m3_pair_f16(s0), p0);
  e2m1x8_f16_scaled(w1, e4m3_pair_f16(s1), p1);
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

// ---------------------------------------------------------------- pipeline plumbing
//
// Both kernels run one CTA per SM over a contiguous range of units.  Warp 8
// streams the units' weight tiles through a ring of stages (TMA bulk copies on
// full / empty mbarriers), warp 9 stages the activation rows of each token
// block once (x_full / x_empty), and consumer warps 0..7 compute, so the weight
// bytes of the next units are in flight while the current one is multiplied.
// Every wait is bounded.  A wait that runs out raises a CTA-wide flag that makes
// later waits give up at once; the consumers OR their failures into the
// per-unit barrier itself (bar.red.or), so all of them leave at the same unit,
// and the producers stop issuing and wait (bounded) for what they issued.

constexpr int kConsWarps = 8;

// Plain arrival (one count) on a shared-memory mbarrier.
__device__ __forceinline__ void mbar_arrive_one(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
constexpr int kPipeThreads = (kConsWarps + 2) * 32;
constexpr int kWProd = kConsWarps, kXProd = kConsWarps + 1;
constexpr int kMaxRing = 16;

struct Pipe {
  uint64_t* full;   // [kMaxRing]
  uint64_t* empty;  // [kMaxRing], one arrival per consumer warp
  uint64_t* xfull;
  uint64_t* xempty;  // one arrival per consumer warp
  int* dead;
};

// Barrier of the consumer warps that also ORs a per-thread flag across them.
__device__ __forceinline__ bool cons_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, %2, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsWarps * 32)
      : "memory");
  return r != 0;
}

// Bounded wait that gives up at once when the CTA is already aborting.
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, const Pipe& pp, DevStatus* st, int where) {
  if (*(volatile int*)pp.dead) return false;
  if (mbar_wait(bar, parity, st, where)) return true;
  *(volatile int*)pp.dead = 1;
  return false;
}

__device__ __forceinline__ Pipe pipe_init(unsigned char* smem, int ns) {
  Pipe pp;
  uint64_t* b = reinterpret_cast<uint64_t*>(smem);
  pp.full = b;
  pp.empty = b + kMaxRing;
  pp.xfull = b + 2 * kMaxRing;
  pp.xempty = b + 2 * kMaxRing + 1;
  pp.dead = reinterpret_cast<int*>(b + 2 * kMaxRing + 2);
  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(&pp.full[i], 1);
      mbar_init(&pp.empty[i], kConsWarps);
    }
    mbar_init(pp.xfull, 1);
    mbar_init(pp.xempty, kConsWarps);
    *pp.dead = 0;
    fence_mbar_init();
  }
  __syncthreads();
  return pp;
}

// The producer's last act: wait (bounded) until every copy it issued has landed.
__device__ __forceinline__ void drain(const Pipe& pp, int issued, int ns, DevStatus* st) {
  for (int i = issued - 1; i >= 0 && i >= issued - ns; --i) mbar_wait(&pp.full[i % ns], (i / ns) & 1, st, 19);
}

// Unit range of this CTA.
__device__ __forceinline__ void unit_range(int n_units, int& lo, int& hi) {
  lo = (int)((long)blockIdx.x * n_units / gridDim.x);
  hi = (int)((long)(blockIdx.x + 1) * n_units / gridDim.x);
}

struct Blk {
  int e, p0, nval;
};

// NVFP4 path: the block's bf16 activation rows, in place, as fp16 scaled by
// 2^sexp[r] (the largest |x| of row r in [2^14, 2^15), exact); consumer warp w
// takes rows w, w + 8.
__device__ __forceinline__ void rows_to_scaled_f16(unsigned char* sx, int nval, int d, int xstride, int* sexp,
                                                   int warp, int lane) {
  for (int r = warp; r < nval; r += kConsWarps) {
    uint16_t* xr = reinterpret_cast<uint16_t*>(sx + r * xstride);
    uint32_t m = 0;
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) m = max(m, max(w4[i] & 0x7fffu, (w4[i] >> 16) & 0x7fffu));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    const int sc = f16_row_exponent(m);
    if (lane == 0) sexp[r] = sc;
    const float f = pow2i(sc);
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[i] << 16) * f, __uint_as_float(w4[i] & 0xffff0000u) * f);
        o[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(xr + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

__device__ __forceinline__ Blk block_info(const FfnArgs& p, int b) {
  Blk k;
  k.e = expert_of_block(p.blk_prefix, p.E, b);
  k.p0 = p.offsets[k.e] + (b - p.blk_prefix[k.e]) * kTokBlock;
  k.nval = min(kTokBlock, p.offsets[k.e + 1] - k.p0);
  return k;
}

// ---------------------------------------------------------------- gate/up + SwiGLU
//
// Unit = (token block b, 16-row tile rt of W_gate and W_up); u = b * RT + rt.
// A stage holds the gate and the up tile (2 x 18 KB at d = 2048).  Consumer
// warp w takes the 128-column chunks w, w + 8, ...; partial sums meet in a
// double-buffered shared array and one thread per (row, token) applies SwiGLU.

template <bool kFp4>
__global__ void __launch_bounds__(kPipeThreads, 1) ffn_up_kernel(FfnArgs p, int ns) {
  pdl_enter();
  extern __shared__ __align__(128) unsigned char smem[];
  const int d = p.d, I = p.I;
  const int tbytes = (int)tile_bytes(d);
  const int xstride = 2 * d + kSmemRowPad;
  unsigned char* sx = smem + 1024;                                        // [16][xstride]
  float* red = reinterpret_cast<float*>(sx + kTokBlock * xstride);        // [2][8 warps][32][8 * kNT]
  unsigned char* ring = reinterpret_cast<unsigned char*>(red + 2 * kConsWarps * 32 * 8 * kNT);
  const Pipe pp = pipe_init(smem, ns);
  int* sexp = reinterpret_cast<int*>(smem + 512);  // [16] NVFP4: the rows' power-of-two scales
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int RT = I / kTileRows;
  int u_lo, u_hi;
  unit_range(RT * p.blk_prefix[p.E], u_lo, u_hi);
  if (u_lo >= u_hi) return;

  if (warp == kWProd) {  // weight tiles
    if (lane == 0) {
      int i = 0;
      for (int u = u_lo; u < u_hi; ++u, ++i) {
        const int s = i % ns;
        if (i >= ns && !pwait(&pp.empty[s], ((i / ns) - 1) & 1, pp, p.st, 12)) break;
        const int b = u / RT, rt = u - b * RT;
        const int e = expert_of_block(p.blk_prefix, p.E, b);
        const size_t toff = ((size_t)e * RT + rt) * tbytes;
        mbar_arrive_expect_tx(&pp.full[s], 2u * tbytes);
        bulk_g2s(ring + (size_t)s * 2 * tbytes, p.gate + toff, tbytes, &pp.full[s]);
        bulk_g2s(ring + (size_t)s * 2 * tbytes + tbytes, p.up + toff, tbytes, &pp.full[s]);
      }
      drain(pp, i, ns, p.st);
    }
    return;
  }
  if (warp == kXProd) {  // activation rows, once per token block
    if (lane == 0) {
      int j = 0;
      bool ok = true;
      for (int u = u_lo; u < u_hi && ok; ++j) {
        const int b = u / RT;
        if (j > 0 && !pwait(pp.xempty, (j - 1) & 1, pp, p.st, 13)) break;
        const Blk k = block_info(p, b);
        mbar_arrive_expect_tx(pp.xfull, (uint32_t)k.nval * 2u * d);
        for (int r = 0; r < k.nval; ++r) {
          const int t = p.sorted_rows[k.p0 + r] / p.k;
          bulk_g2s(sx + r * xstride, p.x + (size_t)t * d, 2 * d, pp.xfull);
        }
        if (!pwait(pp.xfull, j & 1, pp, p.st, 14)) ok = false;  // landed before the next refill
        u = min(u_hi, (b + 1) * RT);
      }
    }
    return;
  }

  // consumers
  const int nch = d / kChunkK;
  int cur_b = -1, j = 0, i = 0;
  Blk k{};
  float tsg = 1.f, tsu = 1.f;
  for (int u = u_lo; u < u_hi; ++u, ++i) {
    const int b = u / RT, rt = u - b * RT;
    bool ok = true;
    if (b != cur_b) {
      if (cur_b >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive_one(pp.xempty);
      }
      ok = pwait(pp.xfull, j & 1, pp, p.st, 15);
      ++j;
      cur_b = b;
      k = block_info(p, b);
      if constexpr (kFp4) {
        tsg = p.gate_ts[k.e];
        tsu = p.up_ts[k.e];
      }
      if (ok) rows_to_scaled_f16(sx, k.nval, d, xstride, sexp, warp, lane);
      if (cons_sync_or(!ok)) ok = false;  // every row converted before any warp reads one
    }
    const int s = i % ns;
    ok = ok && pwait(&pp.full[s], (i / ns) & 1, pp, p.st, 16);
    const unsigned char* sg = ring + (size_t)s * 2 * tbytes;
    const unsigned char* su = sg + tbytes;

    float acc_g[kNT][4], acc_u[kNT][4];
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc_g[nt][q] = acc_u[nt][q] = 0.f;
    const int nt_lim = (k.nval + 7) >> 3;  // n-tiles holding tokens (uniform in the CTA)
    if (ok) {
      for (int ch = warp; ch < nch; ch += kConsWarps) {
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
        if constexpr (kFp4) {
          const uint32_t lg0 = fp4_lane_scales(sg0, c), lg1 = fp4_lane_scales(sg1, c);
          const uint32_t lu0 = fp4_lane_scales(su0, c), lu1 = fp4_lane_scales(su1, c);
          float dg[kNT][4], du[kNT][4];
#pragma unroll
          for (int gg = 0; gg < 4; ++gg) {
            const int col = (ch * 4 + gg) * kGroup + c * 8;
            uint32_t ag[2][4], au[2][4];
            frag_fp4(word_at(qg0, gg), word_at(qg1, gg), (lg0 >> (8 * gg)) & 0xffu, (lg1 >> (8 * gg)) & 0xffu, ag);
            frag_fp4(word_at(qu0, gg), word_at(qu1, gg), (lu0 >> (8 * gg)) & 0xffu, (lu1 >> (8 * gg)) & 0xffu, au);
            uint4 xb[kNT];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              const int tok = nt * 8 + g;
              xb[nt] = make_uint4(0, 0, 0, 0);
              if (nt < nt_lim && tok < k.nval) xb[nt] = *reinterpret_cast<const uint4*>(sx + tok * xstride + col * 2);
            }
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              if (nt < nt_lim) {  // a chunk's MMAs chain in the accumulator; chunks add in fp32
                if (gg == 0) {
                  mma_f16(dg[nt], ag[0], xb[nt].x, xb[nt].y, z);
                  mma_f16(du[nt], au[0], xb[nt].x, xb[nt].y, z);
                } else {
                  mma_f16(dg[nt], ag[0], xb[nt].x, xb[nt].y, dg[nt]);
                  mma_f16(du[nt], au[0], xb[nt].x, xb[nt].y, du[nt]);
                }
              }
            }
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
              if (nt < nt_lim) {
                mma_f16(dg[nt], ag[1], xb[nt].z, xb[nt].w, dg[nt]);
                mma_f16(du[nt], au[1], xb[nt].z, xb[nt].w, du[nt]);
              }
            }
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            if (nt >= nt_lim) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              acc_g[nt][q] += dg[nt][q];
              acc_u[nt][q] += du[nt][q];
            }
          }
          continue;
        }
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int col = (ch * 4 + gg) * kGroup + c * 8;
          uint32_t ag[2][4], au[2][4];
          frag_f16(word_at(qg0, gg), word_at(qg1, gg), ag);
          frag_f16(word_at(qu0, gg), word_at(qu1, gg), au);
          const float s_g0 = scale_at(sg0, gg), s_g1 = scale_at(sg1, gg);
          const float s_u0 = scale_at(su0, gg), s_u1 = scale_at(su1, gg);
          uint4 xb[kNT];
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            const int tok = nt * 8 + g;
            xb[nt] = make_uint4(0, 0, 0, 0);
            if (nt < nt_lim && tok < k.nval) xb[nt] = *reinterpret_cast<const uint4*>(sx + tok * xstride + col * 2);
          }
          // the first halves of every n-tile, then the dependent second halves
          const float z[4] = {0.f, 0.f, 0.f, 0.f};
          float dg[kNT][4], du[kNT][4];
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            if (nt < nt_lim) {
              mma_f16(dg[nt], ag[0], xb[nt].x, xb[nt].y, z);
              mma_f16(du[nt], au[0], xb[nt].x, xb[nt].y, z);
            }
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            if (nt < nt_lim) {
              mma_f16(dg[nt], ag[1], xb[nt].z, xb[nt].w, dg[nt]);
              mma_f16(du[nt], au[1], xb[nt].z, xb[nt].w, du[nt]);
            }
          }
#pragma unroll
          for (int nt = 0; nt < kNT; ++nt) {
            if (nt >= nt_lim) continue;
            acc_g[nt][0] = fmaf(s_g0, dg[nt][0], acc_g[nt][0]);
            acc_g[nt][1] = fmaf(s_g0, dg[nt][1], acc_g[nt][1]);
            acc_g[nt][2] = fmaf(s_g1, dg[nt][2], acc_g[nt][2]);
            acc_g[nt][3] = fmaf(s_g1, dg[nt][3], acc_g[nt][3]);
            acc_u[nt][0] = fmaf(s_u0, du[nt][0], acc_u[nt][0]);
            acc_u[nt][1] = fmaf(s_u0, du[nt][1], acc_u[nt][1]);
            acc_u[nt][2] = fmaf(s_u1, du[nt][2], acc_u[nt][2]);
            acc_u[nt][3] = fmaf(s_u1, du[nt][3], acc_u[nt][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_one(&pp.empty[s]);  // the stage's bytes are in registers
    float* rb = red + (size_t)(i & 1) * kConsWarps * 32 * 8 * kNT;  // [warp][value][lane]
    float* my = rb + (size_t)warp * (8 * kNT) * 32 + lane;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        my[(nt * 4 + q) * 32] = acc_g[nt][q];
        my[(4 * kNT + nt * 4 + q) * 32] = acc_u[nt][q];
      }
    if (cons_sync_or(!ok)) break;  // the same decision in every consumer
    {  // one thread per (row, token) of the 16 x 16 tile
      const int row = tid >> 4, tok = tid & 15;
      if (tok < k.nval) {
        const int nt = tok >> 3, cc = (tok & 7) >> 1, q = ((row >= 8) ? 2 : 0) + (tok & 1);
        const int ln = (row & 7) * 4 + cc;
        float a = 0.f, uu = 0.f;
#pragma unroll
        for (int w = 0; w < kConsWarps; ++w) {
          a += rb[((size_t)w * (8 * kNT) + nt * 4 + q) * 32 + ln];
          uu += rb[((size_t)w * (8 * kNT) + 4 * kNT + nt * 4 + q) * 32 + ln];
        }
        {  // undo the row's power of two (and apply NVFP4 tensor scales)
          const float un = pow2i(-sexp[tok]);
          a *= un * tsg;
          uu *= un * tsu;
        }
        const float h = silu_mul(a, uu);
        const __half hi = __float2half_rn(h);
        const __half lo = __float2half_rn(h - __half2float(hi));
        const size_t o = (size_t)(k.p0 + tok) * I + rt * kTileRows + row;
        if (!(fabsf(h) < kF16Overflow)) record_status(p.st, kStatusCheck, 17, (int)o);
        p.h_hi[o] = hi;
        p.h_lo[o] = lo;
      }
    }
  }
}

// ---------------------------------------------------------------- down projection
//
// Unit = (token block b, pair cp of 16-row W_down tiles); u = b * CT2 + cp.  A
// stage holds the two tiles (2 x 4.6 KB at I = 512); the block's h rows (fp16 hi
// and lo) are staged once per block.  A block of at most 8 rows has one n-tile:
// warp w computes tile w >> 2 over chunks (w & 3) + 4m.  A larger block has two:
// warp w computes tile w >> 2, n-tile w & 1, over the chunk pairs
// {2 ((w >> 1) & 1), +1} + 4m.

__device__ __forceinline__ void down_chunk(const unsigned char* cw, const unsigned char* hh, const unsigned char* hl,
                                           bool has, int ch, int g, int c, float (&acc)[4]) {
  const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
  const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
  const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
  const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
#pragma unroll
  for (int gp = 0; gp < 4; gp += 2) {  // two groups at a time: four independent chains
    uint32_t a[2][2][4];
    uint4 bh[2], bl[2];
    float sc0[2], sc1[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gg = gp + h;
      const int col = (ch * 4 + gg) * kGroup + c * 8;
      frag_f16(word_at(q0, gg), word_at(q1, gg), a[h]);
      sc0[h] = scale_at(s0, gg);
      sc1[h] = scale_at(s1, gg);
      bh[h] = make_uint4(0, 0, 0, 0);
      bl[h] = make_uint4(0, 0, 0, 0);
      if (has) {
        bh[h] = *reinterpret_cast<const uint4*>(hh + col * 2);
        bl[h] = *reinterpret_cast<const uint4*>(hl + col * 2);
      }
    }
    const float z[4] = {0.f, 0.f, 0.f, 0.f};
    float dh[2][4], dl[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mma_f16(dh[h], a[h][0], bh[h].x, bh[h].y, z);
      mma_f16(dl[h], a[h][0], bl[h].x, bl[h].y, z);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mma_f16(dh[h], a[h][1], bh[h].z, bh[h].w, dh[h]);
      mma_f16(dl[h], a[h][1], bl[h].z, bl[h].w, dl[h]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      acc[0] = fmaf(sc0[h], dh[h][0] + dl[h][0], acc[0]);
      acc[1] = fmaf(sc0[h], dh[h][1] + dl[h][1], acc[1]);
      acc[2] = fmaf(sc1[h], dh[h][2] + dl[h][2], acc[2]);
      acc[3] = fmaf(sc1[h], dh[h][3] + dl[h][3], acc[3]);
    }
  }
}

// NVFP4 form of down_chunk: the chunk's MMAs chain in the accumulator (exact
// fp16 weights), then the hi and lo sums add into acc in fp32.
__device__ __forceinline__ void down_chunk_fp4(const unsigned char* cw, const unsigned char* hh,
                                               const unsigned char* hl, bool has, int ch, int g, int c,
                                               float (&acc)[4]) {
  const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
  const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
  const uint32_t l0 = fp4_lane_scales(*reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8), c);
  const uint32_t l1 = fp4_lane_scales(*reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8), c);
  float dh[4] = {0.f, 0.f, 0.f, 0.f}, dl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int gg = 0; gg < 4; ++gg) {
    const int col = (ch * 4 + gg) * kGroup + c * 8;
    uint32_t a[2][4];
    frag_fp4(word_at(q0, gg), word_at(q1, gg), (l0 >> (8 * gg)) & 0xffu, (l1 >> (8 * gg)) & 0xffu, a);
    uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
    if (has) {
      bh = *reinterpret_cast<const uint4*>(hh + col * 2);
      bl = *reinterpret_cast<const uint4*>(hl + col * 2);
    }
    mma_f16(dh, a[0], bh.x, bh.y, dh);
    mma_f16(dl, a[0], bl.x, bl.y, dl);
    mma_f16(dh, a[1], bh.z, bh.w, dh);
    mma_f16(dl, a[1], bl.z, bl.w, dl);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] += dh[q] + dl[q];
}

template <bool kFp4>
__global__ void __launch_bounds__(kPipeThreads, 1) ffn_down_kernel(FfnArgs p, int ns) {
  pdl_enter();
  extern __shared__ __align__(128) unsigned char smem[];
  const int d = p.d, I = p.I;
  const int tbytes = (int)tile_bytes(I);
  const int hstride = 2 * I + kSmemRowPad;
  unsigned char* shh = smem + 1024;
  unsigned char* shl = shh + kTokBlock * hstride;
  float* red = reinterpret_cast<float*>(shl + kTokBlock * hstride);  // [2][8 warps][4][32]
  unsigned char* ring = reinterpret_cast<unsigned char*>(red + 2 * kConsWarps * 32 * 4);
  const Pipe pp = pipe_init(smem, ns);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, c = lane & 3;
  const int CT = d / kTileRows, CT2 = CT / 2;
  int u_lo, u_hi;
  unit_range(CT2 * p.blk_prefix[p.E], u_lo, u_hi);
  if (u_lo >= u_hi) return;

  if (warp == kWProd) {
    if (lane == 0) {
      int i = 0;
      for (int u = u_lo; u < u_hi; ++u, ++i) {
        const int s = i % ns;
        if (i >= ns && !pwait(&pp.empty[s], ((i / ns) - 1) & 1, pp, p.st, 22)) break;
        const int b = u / CT2, cp = u - b * CT2;
        const int e = expert_of_block(p.blk_prefix, p.E, b);
        mbar_arrive_expect_tx(&pp.full[s], 2u * tbytes);
        bulk_g2s(ring + (size_t)s * 2 * tbytes, p.down + ((size_t)e * CT + 2 * cp) * tbytes, 2u * tbytes,
                 &pp.full[s]);
      }
      drain(pp, i, ns, p.st);
    }
    return;
  }
  if (warp == kXProd) {
    if (lane == 0) {
      int j = 0;
      bool ok = true;
      for (int u = u_lo; u < u_hi && ok; ++j) {
        const int b = u / CT2;
        if (j > 0 && !pwait(pp.xempty, (j - 1) & 1, pp, p.st, 23)) break;
        const Blk k = block_info(p, b);
        mbar_arrive_expect_tx(pp.xfull, (uint32_t)k.nval * 4u * I);
        for (int r = 0; r < k.nval; ++r) {
          bulk_g2s(shh + r * hstride, p.h_hi + (size_t)(k.p0 + r) * I, 2 * I, pp.xfull);
          bulk_g2s(shl + r * hstride, p.h_lo + (size_t)(k.p0 + r) * I, 2 * I, pp.xfull);
        }
        if (!pwait(pp.xfull, j & 1, pp, p.st, 24)) ok = false;
        u = min(u_hi, (b + 1) * CT2);
      }
    }
    return;
  }

  const int nch = I / kChunkK;
  const int tile = warp >> 2;
  int cur_b = -1, j = 0, i = 0;
  Blk k{};
  for (int u = u_lo; u < u_hi; ++u, ++i) {
    const int b = u / CT2, cp = u - b * CT2;
    bool ok = true;
    if (b != cur_b) {
      if (cur_b >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive_one(pp.xempty);
      }
      ok = pwait(pp.xfull, j & 1, pp, p.st, 25);
      ++j;
      cur_b = b;
      k = block_info(p, b);
    }
    const bool small = k.nval <= 8;  // one n-tile (uniform in the CTA)
    const int s = i % ns;
    ok = ok && pwait(&pp.full[s], (i / ns) & 1, pp, p.st, 26);
    const unsigned char* sw = ring + (size_t)s * 2 * tbytes + (size_t)tile * tbytes;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      if (small) {
        const bool has = g < k.nval;
        for (int ch = warp & 3; ch < nch; ch += 4) {
          if constexpr (kFp4)
            down_chunk_fp4(sw + ch * kChunkBytes, shh + g * hstride, shl + g * hstride, has, ch, g, c, acc);
          else
            down_chunk(sw + ch * kChunkBytes, shh + g * hstride, shl + g * hstride, has, ch, g, c, acc);
        }
      } else {
        const int nt = warp & 1, tok = nt * 8 + g;
        const bool has = tok < k.nval;
        for (int ch0 = 2 * ((warp >> 1) & 1); ch0 < nch; ch0 += 4)
          for (int ch = ch0; ch < ch0 + 2 && ch < nch; ++ch) {
            if constexpr (kFp4)
              down_chunk_fp4(sw + ch * kChunkBytes, shh + tok * hstride, shl + tok * hstride, has, ch, g, c, acc);
            else
              down_chunk(sw + ch * kChunkBytes, shh + tok * hstride, shl + tok * hstride, has, ch, g, c, acc);
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_one(&pp.empty[s]);
    const float tsd = kFp4 ? p.down_ts[k.e] : 1.f;
    float* rb = red + (size_t)(i & 1) * kConsWarps * 32 * 4;  // [warp][value][lane]
#pragma unroll
    for (int q = 0; q < 4; ++q) rb[((size_t)warp * 4 + q) * 32 + lane] = acc[q];
    if (cons_sync_or(!ok)) break;  // the same decision in every consumer
    {  // thread -> (tile, column, token low bits); four (small) or two partial sums per output
      const int tl = tid >> 7, col = (tid >> 3) & 15, t8 = tid & 7;
      const int cc = t8 >> 1, q = ((col >= 8) ? 2 : 0) + (t8 & 1), ln = (col & 7) * 4 + cc;
      const size_t ybase = (size_t)(2 * cp + tl) * kTileRows + col;
      if (small) {
        if (t8 < k.nval) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) v += rb[((size_t)(tl * 4 + w) * 4 + q) * 32 + ln];
          p.y_rows[(size_t)(k.p0 + t8) * d + ybase] = kFp4 ? v * tsd : v;
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int tk = nt * 8 + t8;
          if (tk < k.nval) {
            const float v = rb[((size_t)(tl * 4 + nt) * 4 + q) * 32 + ln] + rb[((size_t)(tl * 4 + 2 + nt) * 4 + q) * 32 + ln];
            p.y_rows[(size_t)(k.p0 + tk) * d + ybase] = kFp4 ? v * tsd : v;
          }
        }
      }
    }
  }
}

size_t up_fixed_smem(int d) {
  return 1024 + (size_t)kTokBlock * (2 * d + kSmemRowPad) + (size_t)2 * kConsWarps * 32 * 8 * kNT * sizeof(float);
}
size_t down_fixed_smem(int I) {
  return 1024 + 2 * (size_t)kTokBlock * (2 * I + kSmemRowPad) + (size_t)2 * kConsWarps * 32 * 4 * sizeof(float);
}
constexpr size_t kFfnSmemBudget = 227 * 1024;

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
  const size_t fixed = up_fixed_smem(a.d), stage = 2 * (size_t)tile_bytes(a.d);
  if (fixed + 2 * stage > kFfnSmemBudget) return cudaErrorNotSupported;
  int ns = (int)((kFfnSmemBudget - fixed) / stage);
  if (ns > kMaxRing) ns = kMaxRing;
  const size_t sm = fixed + (size_t)ns * stage;
  const long units = (long)(a.I / kTileRows) * max_blocks(R, a.E);
  const int grid = (int)(units < num_sms() ? units : num_sms());
  static int attr_set[64] = {}, attr_fp4[64] = {};
  cudaError_t err;
  if (a.gate_ts != nullptr) {
    if ((err = ensure_smem_attr(ffn_up_kernel<true>, sm, attr_fp4)) != cudaSuccess) return err;
    if (cudaError_t e_ = launch_pdl(ffn_up_kernel<true>, dim3(grid), dim3(kPipeThreads), sm, s, a, ns)) return e_;
  } else {
    if ((err = ensure_smem_attr(ffn_up_kernel<false>, sm, attr_set)) != cudaSuccess) return err;
    if (cudaError_t e_ = launch_pdl(ffn_up_kernel<false>, dim3(grid), dim3(kPipeThreads), sm, s, a, ns)) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_ffn_down(const FfnArgs& a, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) return cudaSuccess;
  if ((a.d / kTileRows) % 2) return cudaErrorNotSupported;
  const size_t fixed = down_fixed_smem(a.I), stage = 2 * (size_t)tile_bytes(a.I);
  if (fixed + 2 * stage > kFfnSmemBudget) return cudaErrorNotSupported;
  int ns = (int)((kFfnSmemBudget - fixed) / stage);
  if (ns > kMaxRing) ns = kMaxRing;
  const size_t sm = fixed + (size_t)ns * stage;
  const long units = (long)(a.d / kTileRows / 2) * max_blocks(R, a.E);
  const int grid = (int)(units < num_sms() ? units : num_sms());
  static int attr_set[64] = {}, attr_fp4[64] = {};
  cudaError_t err;
  if (a.down_ts != nullptr) {
    if ((err = ensure_smem_attr(ffn_down_kernel<true>, sm, attr_fp4)) != cudaSuccess) return err;
    if (cudaError_t e_ = launch_pdl(ffn_down_kernel<true>, dim3(grid), dim3(kPipeThreads), sm, s, a, ns)) return e_;
  } else {
    if ((err = ensure_smem_attr(ffn_down_kernel<false>, sm, attr_set)) != cudaSuccess) return err;
    if (cudaError_t e_ = launch_pdl(ffn_down_kernel<false>, dim3(grid), dim3(kPipeThreads), sm, s, a, ns)) return e_;
  }
  return cudaGetLastError();
}

}  // namespace bitmoe
