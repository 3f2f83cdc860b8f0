// Fused decode step of the int4 MoE layer: one persistent launch per token
// batch (T <= 8) runs router -> top-k -> grouping -> gate/up + SwiGLU ->
// down + combine.
//
// The pages' decode speed comes from a kernel that does the whole decode pass
// in one launch ("Flint 40B : Best Mid Sized LLM", transcript 06:43; "Recursive
// abre o Flint ...", section "O papel da quantizacao e dos kernels no
// lancamento").  That kernel was written for Apple GPUs; this one is built for
// B300.  One CTA per SM: a producer warp streams the CTA's share of the chosen
// experts' weights through a ring of TMA bulk copies (the ring holds a CTA's
// whole share at batch 1, so every byte of the step is requested at once), 16
// consumer warps run mma.sync, and two grid-wide barriers (bounded spins on a
// monotonic counter) separate the phases.  Programmatic dependent launch lets
// the next step's router rows be fetched before this step has drained.
//
// At batch 1 every phase runs once per launch, so the time goes to dependent
// latency (global round trips, CTA-wide barriers, instruction fetch) rather
// than to arithmetic: the phases below keep their serial chains short and their
// code compact.
//   P0  router logits of this CTA's experts, one warp per (token, expert) dot
//       product (W_r rows are fetched before the grid-dependency wait).  While
//       the grid barrier A is pending, the staged tokens are turned into fp16
//       scaled by a power of two per token (exact; see below).
//                                                            -- grid barrier A
//   P1  every CTA reads all logits and selects top-k per token: the k-th
//       largest of the 16 warp maxima bounds the k-th logit from below, so only
//       the few logits above it are ranked; for one token a single warp then
//       computes the gates and the (one row per expert) grouping, for several
//       tokens one warp per token selects and the grouping is a rank count.
//   P2  gate/up units (expert, 16-row tile), one 128-column chunk per warp;
//       h = silu(a) * u stored as an fp16 hi + lo pair.      -- grid barrier B
//       (the producer streams the CTA's W_down tiles meanwhile)
//   P3  16 output columns per CTA: four warps per expert tile (a K quarter
//       each), then out = resid + sum_j w_j y_j in ascending j.
//
// Both projections dequantise int4 to fp16 (the magic-number conversion takes
// one shift per eight weights, against three for bf16).  The gate/up inputs are
// bf16 tokens: token t is multiplied by 2^s_t so that its largest |x| lands in
// [2^14, 2^15), which makes every scaled value an exact fp16 (elements below
// 2^-24 of the token's largest would round); the fp32 dot products are scaled
// back by 2^-s_t, exactly, so the projections keep the exact products and fp32
// sums of the bf16 arithmetic.
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kDecWarps = 16;
constexpr int kConsumers = kDecWarps * 32;
constexpr int kDecThreads = kConsumers + 32;
constexpr int kMaxStages = 16;
constexpr int kDecMaxE = kConsumers;  // one logit per consumer thread
constexpr int kDecMaxK = kDecWarps;   // the warp-maxima bound needs k <= number of warps
constexpr int kDecMaxT = 8;
constexpr int kTracePoints = 32;
static_assert(kDecMaxT * (kDecMaxK + 1) <= kConsumers, "one routed row per consumer thread in the counts");

struct DecodeArgs {
  const uint16_t* x;
  const uint16_t* resid;
  int T, d, E, k, I, renorm;  // E, k: routed experts, routed experts per token
  int n_shared;               // 1: bank entry E is a shared expert, every token's last row, weight 1
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
  const float* gate_ts;  // NVFP4 banks: fp32 tensor scale per bank entry (null: int4 banks)
  const float* up_ts;
  const float* down_ts;
  const int32_t* forced_ids;
  const float* forced_w;
  uint16_t* out;
  float* out_f32;
  int32_t* ids_out;
  float* w_out;
  float* logits;  // [T, E] (global scratch)
  __half* h_hi;   // [R, I]
  __half* h_lo;
  unsigned* gbar;
  DevStatus* st;
  int nstages;
  int offA, offB, offR, offRing;  // shared-memory carve-up (bytes)
  int offX16;                      // fp16 tokens, from the start of region A
  unsigned long long* trace;       // optional [grid][kTracePoints] SM-clock stamps
  int prenorm;                     // x holds the residual: route and run the experts on RMSNorm(x)
  float eps;
  uint16_t* xh_out;                // optional [T, d] copy of RMSNorm(x) (CTA 0 writes it)
  // stack launches only
  int n_layers;                    // layers in the table
  const uint8_t* lm_w;             // packed LM head [V, d] after the layers (null: none)
  int lm_V;
  float* lm_logits;                // optional [T, V]
  unsigned long long* lm_keys;     // [T] arg-max keys (global scratch)
  int32_t* lm_argmax;              // [T]
};

struct LayerPtrs {  // one layer's weights
  const uint8_t* gate;
  const uint8_t* up;
  const uint8_t* down;
  const float* w_router;
  const float* b_router;
  const float* gate_ts;  // NVFP4 tensor scales (null for int4 banks)
  const float* up_ts;
  const float* down_ts;
};

constexpr int kMaxStackLayers = 64;
struct StackArgs {
  DecodeArgs base;
  LayerPtrs tab[kMaxStackLayers];
};

// Phase timestamps for the optional trace buffer (thread 0 of each CTA): the
// SM's cycle counter, which resolves single phases of a few hundred cycles;
// point 0 also records the global timer in the last slot, to line the CTAs up.
__device__ __forceinline__ void stamp(const unsigned long long* trace, int point) {
  if (trace != nullptr && threadIdx.x == 0) {
    unsigned long long* row = const_cast<unsigned long long*>(trace) + blockIdx.x * kTracePoints;
    row[point] = clock64();
    if (point == 0) row[kTracePoints - 1] = globaltimer_ns();
  }
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers)); }

// Barrier of the consumer warps that returns how many of their threads passed pred.
__device__ __forceinline__ int consumer_popc(bool pred) {
  int n;
  asm volatile("{ .reg .pred p; setp.ne.u32 p, %1, 0; bar.red.popc.u32 %0, 1, %2, p; }"
               : "=r"(n)
               : "r"((uint32_t)pred), "n"(kConsumers)
               : "memory");
  return n;
}

__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Grid-wide barrier over the consumer warps of every CTA, in two halves so that
// a CTA can work between its arrival and its wait.  gb[0] is a monotonic
// arrival counter: every launch passes each barrier once from every CTA, so a
// launch starts with gb[0] a multiple of gridDim.x and an arrival that returns
// `old` waits for the next multiple.  (A launch that timed out can leave it
// misaligned; clearing the device status word resets it.)  The release-add
// publishes the CTA's writes (made CTA-visible by the preceding bar.sync); the
// acquire fence after the poll makes the other CTAs' writes visible.
//
// grid_arrive: called by every consumer thread; returns the count to wait for
// (meaningful in thread 0 only).
__device__ __forceinline__ unsigned grid_arrive(unsigned* gb, const unsigned long long* trace, int arrived_point) {
  consumer_sync();
  unsigned target = 0;
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(gb) : "memory");
    stamp(trace, arrived_point);
    target = (old / gridDim.x + 1u) * gridDim.x;
  }
  return target;
}

// Bounded poll of thread 0 (out of line: it runs once per barrier).
__device__ __noinline__ void grid_poll(unsigned* gb, unsigned target, int* fail, DevStatus* st, int where) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gb) : "memory");
  if ((int)(v - target) < 0) {
    const uint64_t t0 = globaltimer_ns();
    do {
      asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gb) : "memory");
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        record_status(st, kStatusTimeout, where, blockIdx.x);
        *(volatile int*)fail = 1;
        break;
      }
    } while ((int)(v - target) < 0);
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// grid_wait: called by every consumer thread after grid_arrive; false on timeout.
__device__ __forceinline__ bool grid_wait(unsigned* gb, unsigned target, int* fail, DevStatus* st, int where) {
  if (threadIdx.x == 0) grid_poll(gb, target, fail, st, where);
  consumer_sync();
  return *(volatile int*)fail == 0;
}

__device__ __forceinline__ bool grid_barrier(unsigned* gb, int* fail, DevStatus* st, int where,
                                             const unsigned long long* trace, int arrived_point) {
  const unsigned target = grid_arrive(gb, trace, arrived_point);
  return grid_wait(gb, target, fail, st, where);
}


// Copies the T staged bf16 token rows into fp16 rows of dst, token t scaled by
// 2^sexp[t] so that its largest magnitude lands in [2^14, 2^15) (exact: bf16
// values carry 8 significant bits, fp16 holds 11).  One warp per token: warp
// w of nw handles tokens w, w + nw, ...
__device__ __noinline__ void stage_tokens_f16(const unsigned char* rows, unsigned char* dst, int T, int d, int xstride,
                                              int* sexp, int w, int nw, int lane) {
  for (int t = w; t < T; t += nw) {
    const uint16_t* xr = reinterpret_cast<const uint16_t*>(rows + t * xstride);
    uint16_t* xo = reinterpret_cast<uint16_t*>(dst + t * xstride);
    uint32_t m = 0;
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 v = *reinterpret_cast<const uint4*>(xr + c);
      m = max(m, max(max(v.x & 0x7fffu, v.x >> 16 & 0x7fffu), max(v.y & 0x7fffu, v.y >> 16 & 0x7fffu)));
      m = max(m, max(max(v.z & 0x7fffu, v.z >> 16 & 0x7fffu), max(v.w & 0x7fffu, v.w >> 16 & 0x7fffu)));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    const int ef = (int)(m >> 7);  // exponent field of the largest magnitude (0: zero / subnormal only)
    const int sc = (ef == 0) ? 0 : min(126, max(-126, 14 - (ef - 127)));
    if (lane == 0) sexp[t] = sc;
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
      *reinterpret_cast<uint4*>(xo + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Float value of an order-preserving arg-max key (inverse of float_order_key).
__device__ __forceinline__ float key_value(unsigned long long key) {
  const uint32_t u = (uint32_t)(key >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) { return a > b ? a : b; }

__device__ __forceinline__ float scale_at(uint2 s, int gg) {
  const uint32_t w = (gg < 2) ? s.x : s.y;
  const uint16_t b = (gg & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t word_at(const uint4& q, int gg) {
  return gg == 0 ? q.x : gg == 1 ? q.y : gg == 2 ? q.z : q.w;
}


struct Routing {  // shared-memory routing tables (identical in every CTA)
  int* ids;      // [R]   expert of row r (-1 = dropped)
  float* w;      // [R]
  int* pos;      // [R]   sorted position of row r (-1 = dropped)
  int* sorted;   // [R]   row at sorted position p
  int* first;    // [R]   1 + first position of the row's expert if r is its first row, else 0
  int* act_e;    // [R]   active experts, ascending
  int* act_off;  // [R+1] first sorted position of active expert a
  unsigned long long* wmax;  // [kDecWarps]
  unsigned long long* cand;  // [kConsumers]
  unsigned long long* sel;   // [kDecMaxT][kDecMaxK]
  float* zall;   // [kDecMaxT]
  float* part;   // [kDecWarps] partial sums
  int* sexp;     // [kDecMaxT] power-of-two scale of each staged fp16 token
  int* misc;     // [0] U, [1] fail flag, [2] candidate count, [3] tau slot
  float* tsd;    // [R] NVFP4: W_down tensor scale of active expert a
};

// Top-k of one token by one warp, for batches of several tokens (one warp per
// token, all tokens at once): lane l holds logits e = l, l + 32, ...; kr rounds
// of a warp arg-max over (value descending, index ascending) pick the experts in
// order; gates exp(l_j - l_max) over the chosen kr (renormalised) or over all E.
// Writes the token's rows t*k + j of the routing tables (the shared expert's
// row, if any, last with weight 1).
template <int NPER>  // logits per lane: E <= 32 * NPER
__device__ __noinline__ void warp_topk_token(const float* __restrict__ lrow, int E, int kr, int k, int renorm, int t, int* ids,
                                float* w, int lane) {
  float v[NPER];
  const int nper = (E + 31) / 32;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = i * 32 + lane;
    v[i] = (i < nper && e < E) ? __ldcg(lrow + e) : -INFINITY;
  }
  uint32_t taken = 0;
  float my_sel = -INFINITY, vmax = 0.f;
  int my_id = 0;
  for (int j = 0; j < kr; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
      const int e = i * 32 + lane;
      if (i < nper && e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
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
  const float my_e = (lane < kr) ? expf(my_sel - vmax) : 0.f;
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
  if (lane < kr) {
    ids[t * k + lane] = (my_id < E) ? my_id : -1;
    w[t * k + lane] = my_e / z;
  } else if (lane < k) {
    ids[t * k + lane] = E;
    w[t * k + lane] = 1.0f;
  }
}

// RMSNorm of the T staged bf16 rows in place (unit gain, eps), by the 512
// consumer threads: reduced exactly as the standalone RMSNorm kernel does (256
// threads per token, fp32 FMA chains, then eight warp partials in order), so
// both give the same bits; two tokens at a time.  xh_out (optional) receives a
// copy of the normalised rows.
__device__ __noinline__ void rmsnorm_rows(unsigned char* rows, int T, int d, int xstride, float eps, float* part,
                                          uint16_t* xh_out) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = tid >> 8, lt = tid & 255;
  for (int t0 = 0; t0 < T; t0 += 2) {
    const int t = t0 + half;
    uint16_t* xr = reinterpret_cast<uint16_t*>(rows + t * xstride);
    float ss = 0.f;
    if (t < T) {
      for (int c8 = lt * 8; c8 < d; c8 += 256 * 8) {
        const uint4 r = *reinterpret_cast<const uint4*>(xr + c8);
        const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = __uint_as_float(rw[i] << 16), b = __uint_as_float(rw[i] & 0xffff0000u);
          ss = fmaf(a, a, ss);
          ss = fmaf(b, b, ss);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) part[warp] = ss;
    consumer_sync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) tot += part[half * 8 + i];
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    if (t < T) {
      for (int c8 = lt * 8; c8 < d; c8 += 256 * 8) {
        const uint4 r = *reinterpret_cast<const uint4*>(xr + c8);
        const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
        uint32_t ob[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = __uint_as_float(rw[i] << 16) * inv, b = __uint_as_float(rw[i] & 0xffff0000u) * inv;
          ob[i] = (uint32_t)float_to_bf16_bits(a) | ((uint32_t)float_to_bf16_bits(b) << 16);
        }
        const uint4 o = make_uint4(ob[0], ob[1], ob[2], ob[3]);
        *reinterpret_cast<uint4*>(xr + c8) = o;
        if (xh_out) *reinterpret_cast<uint4*>(xh_out + (size_t)t * d + c8) = o;
      }
    }
    consumer_sync();  // the partials are read; the normalised rows are in place
  }
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// After the last layer of a stack: RMSNorm of the residual rows, then the LM
// head over all V rows and the arg-max (the arithmetic of lmhead.cu: fp16
// weights, tokens scaled by 2^s exactly, fp32 sums, lowest row wins ties).
// Tiles go to CTAs as in lmhead.cu (tile c, c + G, ...) and through the ring in
// the order of the layers' uses (ring_i onward); a stage belongs to one
// consumer warp here (nw = the stage count), so every warp waits on its own
// stage's phases in order, and releases it for all 16 layer-phase arrivals.
__device__ __noinline__ void lm_phase(const DecodeArgs& p, unsigned char* regA, unsigned char* x16,
                                      unsigned char* ring, uint64_t* full, uint64_t* empty, float* part,
                                      int* sexp, unsigned long long* wkey, int ring_i, int* fail) {
  const int T = p.T, d = p.d, V = p.lm_V, NS = p.nstages;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tbd = (int)tile_bytes(d), xstride = 2 * d + kSmemRowPad;
  const int VT = V / kTileRows;
  const int my_tiles = (VT > cta) ? (VT - 1 - cta) / G + 1 : 0;
  if (warp == kDecWarps) {
    if (lane == 0) {
      for (int j = 0; j < my_tiles; ++j) {
        const int i = ring_i + j, s = i % NS;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1, p.st, 44)) {
          *(volatile int*)fail = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], (uint32_t)tbd);
        bulk_g2s(ring + (size_t)s * tbd, p.lm_w + ((size_t)cta + (size_t)j * G) * tbd, (uint32_t)tbd, &full[s]);
      }
    }
    return;
  }
  // the final residual rows (written before barrier C), normalised, as scaled fp16
  for (int c8 = tid * 8; c8 < T * d; c8 += kConsumers * 8) {
    const int t = c8 / d, col = c8 - t * d;
    *reinterpret_cast<uint4*>(regA + t * xstride + col * 2) = __ldcg(reinterpret_cast<const uint4*>(p.x + c8));
  }
  {
    uint4* pad = reinterpret_cast<uint4*>(x16 + T * xstride);
    for (int c = tid; c < d / 8; c += kConsumers) pad[c] = make_uint4(0, 0, 0, 0);
  }
  consumer_sync();
  rmsnorm_rows(regA, T, d, xstride, p.eps, part, nullptr);
  stage_tokens_f16(regA, x16, T, d, xstride, sexp, warp, kDecWarps, lane);
  consumer_sync();

  const int g = lane >> 2, c = lane & 3;
  const int nw = NS;  // one stage per consumer warp (NS <= 16)
  const unsigned char* xrow = x16 + (g < T ? g : T) * xstride;
  const float un0 = (2 * c < T) ? pow2i(-sexp[2 * c]) : 0.f;
  const float un1 = (2 * c + 1 < T) ? pow2i(-sexp[2 * c + 1]) : 0.f;
  float best_v[2] = {-INFINITY, -INFINITY};
  int best_i[2] = {0x7fffffff, 0x7fffffff};
  bool ok = true;
  if (warp < nw) {
    const int j0 = ((warp - ring_i) % nw + nw) % nw;
    for (int j = j0; j < my_tiles && ok; j += nw) {
      const int i = ring_i + j, s = i % NS;
      ok = mbar_wait(&full[s], (i / NS) & 1, p.st, 45);
      if (!ok) break;
      const unsigned char* tile = ring + (size_t)s * tbd;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int ch = 0; ch < d / kChunkK; ++ch) {
        const unsigned char* cw = tile + ch * kChunkBytes;
        const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
        const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
        const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
        const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
#pragma unroll 2
        for (int gg = 0; gg < 4; ++gg) {
          const int col = (ch * 4 + gg) * kGroup + c * 8;
          uint32_t p0[4], p1[4];
          nib_pairs4_f16(word_at(q0, gg), p0);
          nib_pairs4_f16(word_at(q1, gg), p1);
          const uint32_t a0[4] = {p0[0], p1[0], p0[1], p1[1]}, a1[4] = {p0[2], p1[2], p0[3], p1[3]};
          const uint4 xb = *reinterpret_cast<const uint4*>(xrow + col * 2);
          float dd[4];
          mma_f16_z(dd, a0, xb.x, xb.y);
          mma_f16(dd, a1, xb.z, xb.w, dd);
          const float sc0 = scale_at(s0, gg), sc1 = scale_at(s1, gg);
          acc[0] = fmaf(sc0, dd[0], acc[0]);
          acc[1] = fmaf(sc0, dd[1], acc[1]);
          acc[2] = fmaf(sc1, dd[2], acc[2]);
          acc[3] = fmaf(sc1, dd[3], acc[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_n(&empty[s], kDecWarps);
      const int vrow0 = (cta + j * G) * kTileRows;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b = q & 1, tok = 2 * c + b, vrow = vrow0 + g + ((q >= 2) ? 8 : 0);
        if (tok < T) {
          const float v = acc[q] * (b ? un1 : un0);
          if (p.lm_logits) p.lm_logits[(size_t)tok * V + vrow] = v;
          if (v > best_v[b] || (v == best_v[b] && vrow < best_i[b])) {
            best_v[b] = v;
            best_i[b] = vrow;
          }
        }
      }
    }
  }
  if (!ok) *(volatile int*)fail = 1;
  // per token: the warp's best over its rows (lanes with the same c), then over
  // the warps as 64-bit keys (logit order, then the inverted row: lowest wins)
  // wkey: [16 warps][8 tokens]
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float v = best_v[b];
    int ix = best_i[b];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, off);
      const int oi = __shfl_xor_sync(0xffffffffu, ix, off);
      if (ov > v || (ov == v && oi < ix)) {
        v = ov;
        ix = oi;
      }
    }
    if (g == 0 && 2 * c + b < kDecMaxT)
      wkey[warp * kDecMaxT + 2 * c + b] =
          (ix == 0x7fffffff) ? 0ull : (((unsigned long long)float_order_key(v) << 32) | (0xffffffffu - (uint32_t)ix));
  }
  consumer_sync();
  if (tid < T && *(volatile int*)fail == 0) {
    unsigned long long key = 0ull;
    for (int w = 0; w < kDecWarps; ++w) key = umax64(key, wkey[w * kDecMaxT + tid]);
    if (key != 0ull) atomicMax(&p.lm_keys[tid], key);
  }
  // D: every CTA's keys folded; CTA 0 publishes the arg-max
  if (grid_barrier(p.gbar, fail, p.st, 43, nullptr, 0) && cta == 0 && tid < T)
    p.lm_argmax[tid] = (int32_t)(0xffffffffu - (uint32_t)(__ldcg(p.lm_keys + tid) & 0xffffffffull));
}

// The kernel body, one layer (kStack = false) or a stack of pre-norm layers
// followed by RMSNorm, the LM head and the arg-max (kStack = true; layer l's
// weights from tab[l], the residual updated in place).
// kFp4: the expert banks are NVFP4 (each code times its E4M3 block scale is an
// exact fp16 weight, the MMAs accumulate a whole row in fp32, and the tensor
// scale multiplies the sums); else int4 with fp16 scales applied per group.
template <bool kStack, bool kFp4>
__device__ __forceinline__ void decode_body(const DecodeArgs& p, const LayerPtrs* tab) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* xbar = empty + kMaxStages;
  uint64_t* wrbar = xbar + 1;
  uint64_t* hbar = wrbar + 1;
  unsigned char* regA = smem + p.offA;
  unsigned char* x16 = smem + p.offA + p.offX16;  // fp16 scaled tokens (P2), beside the bf16 ones
  unsigned char* regB = smem + p.offB;
  unsigned char* ring = smem + p.offRing;
  // kr routed experts per token; k rows per token (the shared expert's row last)
  const int T = p.T, d = p.d, E = p.E, kr = p.k, k = kr + p.n_shared, I = p.I, R = T * k;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tbd = (int)tile_bytes(d), tbi = (int)tile_bytes(I);
  const int dps = tbd / tbi;  // down tiles per ring stage
  const int RT = I / kTileRows, CT = d / kTileRows;
  const int xstride = 2 * d + kSmemRowPad;
  const int NS = p.nstages;
  // threads per output element in the combine: up to 8 (a power of two), all elements at once
  int cpe = 8;
  while (cpe > 1 && T * kTileRows * cpe > kConsumers) cpe >>= 1;

  Routing rt;
  {
    unsigned long long* q8 = reinterpret_cast<unsigned long long*>(smem + p.offR);
    rt.wmax = q8; q8 += kDecWarps;
    rt.cand = q8; q8 += kConsumers;
    rt.sel = q8; q8 += kDecMaxT * kDecMaxK;
    int* q = reinterpret_cast<int*>(q8);
    rt.zall = reinterpret_cast<float*>(q); q += kDecMaxT;
    rt.part = reinterpret_cast<float*>(q); q += kDecWarps;
    rt.sexp = q; q += kDecMaxT;
    rt.ids = q; q += R;
    rt.w = reinterpret_cast<float*>(q); q += R;
    rt.pos = q; q += R;
    rt.sorted = q; q += R;
    rt.first = q; q += R;
    rt.act_e = q; q += R;
    rt.act_off = q; q += R + 1;
    rt.misc = q; q += 4;
    rt.tsd = reinterpret_cast<float*>(q);
  }
  int* fail = rt.misc + 1;

  // experts whose router rows this CTA computes
  const int e_lo = (int)((long)cta * E / G), e_hi = (int)((long)(cta + 1) * E / G);
  const int nexp = e_hi - e_lo;
  float* wr_s = reinterpret_cast<float*>(regB);
  const bool routed = (p.forced_ids == nullptr);

  const bool lm = kStack && p.lm_w != nullptr;  // RMSNorm + LM head + arg-max after the layers
  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecWarps);
    }
    mbar_init(xbar, 1);
    mbar_init(wrbar, 1);
    mbar_init(hbar, 1);
    rt.misc[0] = 0;
    rt.misc[1] = 0;
    rt.misc[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long* trace = p.trace;  // layer 0 only
  stamp(trace, 0);
  if (tid == 0) grid_dep_launch();  // the next launch may be scheduled as SMs free up

  // router rows of the first layer (independent of the previous step)
  if (warp == kDecWarps && lane == 0 && routed && kr > 0 && nexp > 0) {
    const float* wr0 = kStack ? tab[0].w_router : p.w_router;
    mbar_arrive_expect_tx(wrbar, (uint32_t)nexp * d * 4u);
    bulk_g2s(wr_s, wr0 + (size_t)e_lo * d, (uint32_t)nexp * d * 4u, wrbar);
  }
  const int pairs = T * nexp;
  // warps per (token, expert) dot product: the largest power of two that keeps
  // every pair covered by the 16 consumer warps at once
  int wpp = 1;
  while (pairs > 0 && wpp < kDecWarps && wpp * 2 * pairs <= kDecWarps) wpp *= 2;
  int ring_i = 0;  // ring uses so far (the producer and the consumers count alike)
  const int L = kStack ? p.n_layers : 1;
  for (int l = 0; l < L; ++l) {
  const LayerPtrs lp = kStack ? tab[l]
                              : LayerPtrs{p.gate, p.up, p.down, p.w_router, p.b_router, p.gate_ts, p.up_ts, p.down_ts};
  int32_t* ids_out = (kStack && p.ids_out) ? p.ids_out + (size_t)l * R : p.ids_out;
  float* w_out = (kStack && p.w_out) ? p.w_out + (size_t)l * R : p.w_out;
  if (l > 0) trace = nullptr;
  const uint32_t lpar = (uint32_t)(l & 1);  // phase parity of the layer's single-use barriers
  // router bias of the logit this warp's lane 0 writes first (pair = warp), read now
  float bias0 = 0.f, biasA = 0.f;
  if (routed && lane == 0 && warp < kDecWarps && warp < pairs && lp.b_router != nullptr)
    bias0 = lp.b_router[e_lo + warp % nexp];
  if (routed && wpp > 1 && tid < pairs && lp.b_router != nullptr) biasA = lp.b_router[e_lo + tid % nexp];
  if (l == 0) {
    grid_dep_wait();  // the previous launch on this stream is complete and visible
    // arg-max keys: cleared once the previous launch (which may fold into them)
    // is done, before this launch's first grid barrier; read after its last
    if (lm && cta == 0 && tid < T) p.lm_keys[tid] = 0ull;
  }
  stamp(trace, 1);
  // residual of this CTA's first output tile, read now so that its latency is
  // off the combine at the end (one value per combine thread)
  // (the combine gives each output element cpe threads; the first of them adds the residual)
  uint16_t resid0 = 0;
  if (tid % cpe == 0 && tid / cpe < T * kTileRows && cta < CT) {
    const int el = tid / cpe;
    resid0 = p.resid[(size_t)(el >> 4) * d + (size_t)cta * kTileRows + (el & 15)];
  }
  if (tid == 0) {  // the layer's input rows (later layers: written by the combines before barrier C)
    if (l > 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      fence_proxy_async_smem();
    }
    mbar_arrive_expect_tx(xbar, (uint32_t)T * 2u * d);
    for (int t = 0; t < T; ++t) bulk_g2s(regA + t * xstride, p.x + (size_t)t * d, 2u * d, xbar);
  }

  if (warp < kDecWarps) {
    bool ok = mbar_wait(xbar, lpar, p.st, 30);
    stamp(trace, 16);
    if (p.prenorm)  // taken by every consumer thread alike (the function has barriers)
      rmsnorm_rows(regA, T, d, xstride, p.eps, rt.part, cta == 0 ? p.xh_out : nullptr);
    {  // the zeroed pad row after the fp16 tokens (read by lanes without a token)
      uint4* pad = reinterpret_cast<uint4*>(x16 + T * xstride);
      for (int c = tid; c < d / 8; c += kConsumers) pad[c] = make_uint4(0, 0, 0, 0);
    }
    if (routed && kr > 0) {  // (kr = 0: a dense layer, nothing to score)
      if (nexp > 0) ok = mbar_wait(wrbar, lpar, p.st, 31) && ok;
      stamp(trace, 17);
      if (!ok) *(volatile int*)fail = 1;
      // (token, expert) dot products: wpp warps per pair, each over a K slice
      // (two accumulators per lane), then the slices are added in order
      for (int pr = warp / wpp; pr < pairs; pr += kDecWarps / wpp) {
        const int t = pr / nexp, el = pr % nexp, sl = warp % wpp;
        const uint16_t* xr = reinterpret_cast<const uint16_t*>(regA + t * xstride);
        const float* wrow = wr_s + (size_t)el * d;
        const int ks = sl * (d / wpp), ke = ks + d / wpp;
        float acc0 = 0.f, acc1 = 0.f;
        for (int i = ks + lane * 8; i < ke; i += 512) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ii = i + h * 256;
            if (ii < ke) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xr + ii);
              const float4 w0 = *reinterpret_cast<const float4*>(wrow + ii);
              const float4 w1 = *reinterpret_cast<const float4*>(wrow + ii + 4);
              float a = h ? acc1 : acc0;
              a = fmaf(__uint_as_float(xv.x << 16), w0.x, a);
              a = fmaf(__uint_as_float(xv.x & 0xffff0000u), w0.y, a);
              a = fmaf(__uint_as_float(xv.y << 16), w0.z, a);
              a = fmaf(__uint_as_float(xv.y & 0xffff0000u), w0.w, a);
              a = fmaf(__uint_as_float(xv.z << 16), w1.x, a);
              a = fmaf(__uint_as_float(xv.z & 0xffff0000u), w1.y, a);
              a = fmaf(__uint_as_float(xv.w << 16), w1.z, a);
              a = fmaf(__uint_as_float(xv.w & 0xffff0000u), w1.w, a);
              if (h) acc1 = a; else acc0 = a;
            }
          }
        }
        float acc = acc0 + acc1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
          if (wpp == 1) {
            const float b = (pr == warp) ? bias0 : (lp.b_router ? lp.b_router[e_lo + el] : 0.f);
            p.logits[(size_t)t * E + e_lo + el] = acc + b;
          } else {
            rt.part[pr * wpp + sl] = acc;
          }
        }
      }
      stamp(trace, 24);
      if (wpp > 1) {
        consumer_sync();
        stamp(trace, 25);
        if (tid < pairs) {
          float acc = 0.f;
          for (int sl = 0; sl < wpp; ++sl) acc += rt.part[tid * wpp + sl];
          p.logits[(size_t)(tid / nexp) * E + e_lo + tid % nexp] = acc + biasA;
        }
      }
      stamp(trace, 18);
      stamp(trace, 2);
      // A: every logit written.  Between the arrival and the wait the staged
      // tokens become scaled fp16 (the router has read them).
      const unsigned tgt = grid_arrive(p.gbar, trace, 22);
      if (ok && warp > 0) stage_tokens_f16(regA, x16, T, d, xstride, rt.sexp, warp - 1, kDecWarps - 1, lane);
      grid_wait(p.gbar, tgt, fail, p.st, 32);
      stamp(trace, 3);
    } else {
      if (!ok) *(volatile int*)fail = 1;
      consumer_sync();  // (prenorm) every normalised row is in place
      if (ok) stage_tokens_f16(regA, x16, T, d, xstride, rt.sexp, warp, kDecWarps, lane);
    }

    // ---------------- P1: routing tables, replicated in every CTA
    bool grouped = false;  // the T = 1 path builds the grouping itself
    if (*(volatile int*)fail == 0) {
      if (routed && T > 1 && kr > 0) {
        // several tokens: one warp per token, all tokens at once
        if (warp < T) {
          if (E <= 256)
            warp_topk_token<8>(p.logits + (size_t)warp * E, E, kr, k, p.renorm, warp, rt.ids, rt.w, lane);
          else
            warp_topk_token<kDecMaxE / 32>(p.logits + (size_t)warp * E, E, kr, k, p.renorm, warp, rt.ids, rt.w,
                                            lane);
        }
      } else if (routed && kr > 0) {
        // One token.  Keys = order-preserving logit bits, then the inverted
        // expert index (equal logits put the lower expert first).  The kr-th
        // largest of the 16 warp maxima is a lower bound tau for the kr-th key
        // (kr distinct elements reach it), so only keys >= tau can be chosen;
        // ranking those few candidates against each other gives the top-kr.
        const unsigned long long key =
            (tid < E) ? (((unsigned long long)float_order_key(__ldcg(p.logits + tid)) << 32) |
                         (0xffffffffu - (uint32_t)tid))
                      : 0ull;
        stamp(trace, 26);
        unsigned long long m = key;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = umax64(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) rt.wmax[warp] = m;
        consumer_sync();
        stamp(trace, 27);
        // every warp finds tau itself: lanes 0..15 rank the 16 warp maxima
        // (independent shared-memory loads, no shuffle chain)
        const unsigned long long wm = (lane < kDecWarps) ? rt.wmax[lane] : 0ull;
        int rank = 0;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          const unsigned long long o = rt.wmax[w];
          rank += (o > wm) || (o == wm && w < lane);
        }
        const unsigned at_k = __ballot_sync(0xffffffffu, lane < kDecWarps && rank == kr - 1);
        const unsigned long long tau = __shfl_sync(0xffffffffu, wm, __ffs(at_k) - 1);
        // candidates (keys >= tau), compacted with one shared atomic per warp
        const bool is_cand = key != 0ull && key >= tau;
        const unsigned cb = __ballot_sync(0xffffffffu, is_cand);
        if (cb) {
          int base = 0;
          if (lane == 0) base = atomicAdd(&rt.misc[2], __popc(cb));
          base = __shfl_sync(0xffffffffu, base, 0);
          if (is_cand) rt.cand[base + __popc(cb & ((1u << lane) - 1u))] = key;
        }
        if (!p.renorm) {  // gates over all E: the softmax denominator, per warp
          const unsigned at_0 = __ballot_sync(0xffffffffu, lane < kDecWarps && rank == 0);
          const float vtop = key_value(__shfl_sync(0xffffffffu, wm, __ffs(at_0) - 1));
          float ez = (key != 0ull) ? expf(key_value(key) - vtop) : 0.f;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ez += __shfl_xor_sync(0xffffffffu, ez, off);
          if (lane == 0) rt.part[warp] = ez;
        }
        stamp(trace, 28);
        consumer_sync();
        stamp(trace, 29);
        if (is_cand) {
          const int nc = rt.misc[2];
          int r = 0;
          for (int j = 0; j < nc; ++j) r += rt.cand[j] > key;
          if (r < kr) rt.sel[r] = key;
        }
        consumer_sync();
        stamp(trace, 10);
        if (warp == 0) {
          // lane j < kr: the j-th chosen expert; lane kr (n_shared = 1): the
          // shared expert, bank entry E, weight 1.  One row per expert, so the
          // grouping sorts the kt = k ids (all distinct) ascending.
          int e = 0x7fffffff;
          float v = 0.f;
          if (lane < kr) {
            const unsigned long long sk = rt.sel[lane];
            e = (int)(0xffffffffu - (uint32_t)(sk & 0xffffffffull));
            v = key_value(sk);
          } else if (lane < k) {
            e = E;
          }
          const float vmax = __shfl_sync(0xffffffffu, v, 0);
          const float ez = (lane < kr) ? expf(v - vmax) : 0.f;
          float z = 0.f;
          if (p.renorm) {
            z = ez;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
          } else {
            for (int w = 0; w < kDecWarps; ++w) z += rt.part[w];
          }
          // rank of this lane's id among the k ids (all distinct), counted from
          // shared memory with independent loads (a loop of shuffles with a
          // varying source lane is a long serial chain here)
          if (lane < k) rt.act_e[lane] = e;
          __syncwarp();
          int pos = 0;
#pragma unroll 8
          for (int j = 0; j < k; ++j) pos += rt.act_e[j] < e;
          __syncwarp();
          if (lane < k) {
            const float wg = (lane < kr) ? ez / z : 1.0f;
            rt.ids[lane] = e;
            rt.w[lane] = wg;
            rt.pos[lane] = pos;
            rt.sorted[pos] = lane;
            rt.act_e[pos] = e;
            rt.act_off[pos] = pos;
            rt.first[lane] = pos + 1;
            if (cta == 0) {
              if (ids_out) ids_out[lane] = e;
              if (w_out) w_out[lane] = wg;
            }
          }
          if (lane == 0) {
            rt.misc[0] = k;
            rt.act_off[k] = k;
            rt.misc[2] = 0;
          }
        }
        grouped = true;
        stamp(trace, 11);
      } else if (routed) {
        // a dense layer (kr = 0): each token's one row is the shared expert
        for (int r = tid; r < R; r += kConsumers) {
          rt.ids[r] = E;
          rt.w[r] = 1.0f;
        }
      } else {
        for (int r = tid; r < R; r += kConsumers) {
          int e = p.forced_ids[r];
          if (e < 0 || e >= E + p.n_shared) {
            if (cta == 0) record_status(p.st, kStatusCheck, 33, r);
            e = -1;
          } else if (cta == 0) {
            const int t = r / k;
            for (int jj = t * k; jj < r; ++jj)
              if (p.forced_ids[jj] == e) record_status(p.st, kStatusCheck, 34, r);
          }
          rt.ids[r] = e;
          rt.w[r] = p.forced_w[r];
        }
      }
      if (!grouped) {
        consumer_sync();
        // stable grouping by ranks: row r goes to (rows of smaller experts) +
        // (earlier rows of its own expert); the first row of each expert also
        // places the expert in the ascending list of active experts
        for (int r = tid; r < R; r += kConsumers) {
          const int e = rt.ids[r];
          int less = 0, before = 0;
          if (e >= 0) {
#pragma unroll 8  // eight broadcast loads in flight (R is up to 136 rows)
            for (int rr = 0; rr < R; ++rr) {
              const int f = rt.ids[rr];
              less += (f >= 0 && f < e);
              before += (rr < r && f == e);
            }
            rt.pos[r] = less + before;
            rt.sorted[less + before] = r;
          } else {
            rt.pos[r] = -1;
          }
          rt.first[r] = (e >= 0 && before == 0) ? less + 1 : 0;
        }
        consumer_sync();
        stamp(trace, 10);
        for (int r = tid; r < R; r += kConsumers) {
          if (rt.first[r] > 0) {
            const int e = rt.ids[r];
            int a = 0;
#pragma unroll 8
            for (int rr = 0; rr < R; ++rr) a += (rt.first[rr] > 0 && rt.ids[rr] < e);
            rt.act_e[a] = e;
            rt.act_off[a] = rt.first[r] - 1;
          }
        }
        {  // active experts and routed rows, counted by the barrier itself (R <= kConsumers)
          const int U = consumer_popc(tid < R && rt.first[tid] > 0);
          const int Rv = consumer_popc(tid < R && rt.ids[tid] >= 0);
          if (tid == 0) {
            rt.misc[0] = U;
            rt.act_off[U] = Rv;
          }
        }
        consumer_sync();
        stamp(trace, 11);
        if (cta == 0) {
          for (int r = tid; r < R; r += kConsumers) {
            if (ids_out) ids_out[r] = rt.ids[r];
            if (w_out) w_out[r] = rt.w[r];
          }
        }
      }
    }
  }
  __syncthreads();  // routing tables visible to the producer warp
  stamp(trace, 4);
  if (*(volatile int*)fail) break;

  const int U = rt.misc[0];
  const int n_up = U * RT;
  const int u_lo = (int)((long)cta * n_up / G), u_hi = (int)((long)(cta + 1) * n_up / G);

  // ---------------- producer: this CTA's tiles, in consumption order
  if (warp == kDecWarps) {
    int i = ring_i;
    if (lane == 0) {
      bool pok = true;  // a wait that ran out stops the issue (consumers then time out too)
#pragma unroll 1
      for (int u = u_lo; u < u_hi && pok; ++u) {
        const int a = u / RT, r16 = u - a * RT;
        const size_t toff = ((size_t)rt.act_e[a] * RT + r16) * tbd;
#pragma unroll 1
        for (int m = 0; m < 2; ++m, ++i) {
          const int s = i % NS;
          if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1, p.st, 35)) {
            pok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], (uint32_t)tbd);
          bulk_g2s(ring + (size_t)s * tbd, (m == 0 ? lp.gate : lp.up) + toff, (uint32_t)tbd, &full[s]);
        }
      }
#pragma unroll 1
      for (int ct = cta; ct < CT && pok; ct += G) {
#pragma unroll 1
        for (int a0 = 0; a0 < U; a0 += dps, ++i) {
          const int s = i % NS;
          if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1, p.st, 36)) {
            pok = false;
            break;
          }
          const int n = min(dps, U - a0);
          mbar_arrive_expect_tx(&full[s], (uint32_t)n * tbi);
#pragma unroll 1
          for (int j = 0; j < n; ++j)
            bulk_g2s(ring + (size_t)s * tbd + (size_t)j * tbi,
                     lp.down + ((size_t)rt.act_e[a0 + j] * CT + ct) * tbi, (uint32_t)tbi, &full[s]);
        }
      }
      if (!pok) *(volatile int*)fail = 1;
    }
    ring_i = __shfl_sync(0xffffffffu, i, 0);
  } else {
  // ---------------- consumers
  const int g = lane >> 2, c = lane & 3;
  float* red = reinterpret_cast<float*>(regB);            // [2][16 warps][32][8]
  float* ypart = red + 2 * kDecWarps * 32 * 8;            // [4][R][16]
  int i = ring_i;
  bool ok = true;

  // NVFP4: this thread's active expert's W_down tensor scale, read now and
  // kept in shared memory for P3 (the load's latency hides behind P2)
  const float tsd_r = (kFp4 && tid < U) ? lp.down_ts[rt.act_e[tid]] : 1.0f;
  // P2: gate/up units, one 128-column chunk per warp
  for (int u = u_lo; u < u_hi; ++u) {
    const int a = u / RT, r16 = u - a * RT;
    const int na = rt.act_off[a + 1] - rt.act_off[a];
    const float tsg = kFp4 ? lp.gate_ts[rt.act_e[a]] : 1.0f, tsu = kFp4 ? lp.up_ts[rt.act_e[a]] : 1.0f;
    const int sg = i % NS, su = (i + 1) % NS;
    if (ok) ok = mbar_wait(&full[sg], (i / NS) & 1, p.st, 37) && mbar_wait(&full[su], ((i + 1) / NS) & 1, p.st, 38);
    if (u == u_lo) stamp(trace, 12);
    if (u == u_lo + 1) stamp(trace, 9);
    const unsigned char* tg = ring + (size_t)sg * tbd;
    const unsigned char* tu = ring + (size_t)su * tbd;
    // token row of this lane's B fragment (n = g)
    // (lanes past the expert's tokens read the zeroed pad row after the tokens)
    const unsigned char* xrow = x16 + (g < na ? rt.sorted[rt.act_off[a] + g] / k : T) * xstride;
    float ag4[4] = {0.f, 0.f, 0.f, 0.f}, au4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int ch = warp; ch < d / kChunkK; ch += kDecWarps) {
      const unsigned char* cg = tg + ch * kChunkBytes;
      const unsigned char* cu = tu + ch * kChunkBytes;
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
        float dg[4], du[4];
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
          const int col = (ch * 4 + gg) * kGroup + c * 8;
          const uint4 xb = *reinterpret_cast<const uint4*>(xrow + col * 2);
          uint32_t pg0[4], pg1[4], pu0[4], pu1[4];
          e2m1x8_f16_scaled(word_at(qg0, gg), e4m3_pair_f16((lg0 >> (8 * gg)) & 0xffu), pg0);
          e2m1x8_f16_scaled(word_at(qg1, gg), e4m3_pair_f16((lg1 >> (8 * gg)) & 0xffu), pg1);
          e2m1x8_f16_scaled(word_at(qu0, gg), e4m3_pair_f16((lu0 >> (8 * gg)) & 0xffu), pu0);
          e2m1x8_f16_scaled(word_at(qu1, gg), e4m3_pair_f16((lu1 >> (8 * gg)) & 0xffu), pu1);
          const uint32_t A0[4] = {pg0[0], pg1[0], pg0[1], pg1[1]}, A1[4] = {pg0[2], pg1[2], pg0[3], pg1[3]};
          const uint32_t B0[4] = {pu0[0], pu1[0], pu0[1], pu1[1]}, B1[4] = {pu0[2], pu1[2], pu0[3], pu1[3]};
          if (gg == 0) {  // a chunk's MMAs chain in the accumulator; chunks add in fp32
            mma_f16_z(dg, A0, xb.x, xb.y);
            mma_f16_z(du, B0, xb.x, xb.y);
          } else {
            mma_f16(dg, A0, xb.x, xb.y, dg);
            mma_f16(du, B0, xb.x, xb.y, du);
          }
          mma_f16(dg, A1, xb.z, xb.w, dg);
          mma_f16(du, B1, xb.z, xb.w, du);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          ag4[j] += dg[j];
          au4[j] += du[j];
        }
        continue;
      }
#pragma unroll 2
      for (int gg = 0; gg < 4; ++gg) {
        const int col = (ch * 4 + gg) * kGroup + c * 8;
        const uint4 xb = *reinterpret_cast<const uint4*>(xrow + col * 2);  // fp16, scaled
        uint32_t pg0[4], pg1[4], pu0[4], pu1[4];
        nib_pairs4_f16(word_at(qg0, gg), pg0);
        nib_pairs4_f16(word_at(qg1, gg), pg1);
        nib_pairs4_f16(word_at(qu0, gg), pu0);
        nib_pairs4_f16(word_at(qu1, gg), pu1);
        const uint32_t A0[4] = {pg0[0], pg1[0], pg0[1], pg1[1]}, A1[4] = {pg0[2], pg1[2], pg0[3], pg1[3]};
        const uint32_t B0[4] = {pu0[0], pu1[0], pu0[1], pu1[1]}, B1[4] = {pu0[2], pu1[2], pu0[3], pu1[3]};
        float dg[4], du[4];
        mma_f16_z(dg, A0, xb.x, xb.y);
        mma_f16_z(du, B0, xb.x, xb.y);
        mma_f16(dg, A1, xb.z, xb.w, dg);
        mma_f16(du, B1, xb.z, xb.w, du);
        const float s_g0 = scale_at(sg0, gg), s_g1 = scale_at(sg1, gg);
        const float s_u0 = scale_at(su0, gg), s_u1 = scale_at(su1, gg);
        ag4[0] = fmaf(s_g0, dg[0], ag4[0]);
        ag4[1] = fmaf(s_g0, dg[1], ag4[1]);
        ag4[2] = fmaf(s_g1, dg[2], ag4[2]);
        ag4[3] = fmaf(s_g1, dg[3], ag4[3]);
        au4[0] = fmaf(s_u0, du[0], au4[0]);
        au4[1] = fmaf(s_u0, du[1], au4[1]);
        au4[2] = fmaf(s_u1, du[2], au4[2]);
        au4[3] = fmaf(s_u1, du[3], au4[3]);
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive1(&empty[sg]);
      mbar_arrive1(&empty[su]);
    }
    i += 2;
    float* my = red + ((size_t)(u & 1) * kDecWarps * 32 + warp * 32 + lane) * 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      my[j] = ag4[j];
      my[4 + j] = au4[j];
    }
    if (!ok) *(volatile int*)fail = 1;
    if (u == u_lo) stamp(trace, 8);
    consumer_sync();
    // one thread per (row, token) output of the 16 x 8 tile
    if (tid < kTileRows * 8) {
      const int row = tid >> 3, tok = tid & 7;
      if (tok < na) {
        const int ln = (row & 7) * 4 + (tok >> 1);
        const int ix = ((row >= 8) ? 2 : 0) + (tok & 1);
        const float* rb = red + (size_t)(u & 1) * kDecWarps * 32 * 8;
        float av = 0.f, uv = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          av += rb[(w * 32 + ln) * 8 + ix];
          uv += rb[(w * 32 + ln) * 8 + 4 + ix];
        }
        const float un = pow2i(-rt.sexp[rt.sorted[rt.act_off[a] + tok] / k]);  // undo the token's scale
        const float h = silu_mul(av * (un * tsg), uv * (un * tsu));
        const __half hi = __float2half_rn(h);
        const __half lo = __float2half_rn(h - __half2float(hi));
        const size_t o = (size_t)(rt.act_off[a] + tok) * I + r16 * kTileRows + row;
        if (!(fabsf(h) < kF16Overflow)) record_status(p.st, kStatusCheck, 46, (int)o);
        p.h_hi[o] = hi;
        p.h_lo[o] = lo;
      }
    }
    if (u == u_lo) stamp(trace, 15);
  }
  if (kFp4 && tid < U) rt.tsd[tid] = tsd_r;  // read in P3, after the barrier's CTA-wide sync
  stamp(trace, 5);
  const bool passed_b = grid_barrier(p.gbar, fail, p.st, 39, trace, 23);  // B: every h written
  stamp(trace, 6);
  if (passed_b) {
  // the next layer's router rows, into region B while P3 runs (the P2 partials
  // there are dead; P3's partials sit above them)
  if (kStack && tid == 0 && l + 1 < L && routed && kr > 0 && nexp > 0) {
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(wrbar, (uint32_t)nexp * d * 4u);
    bulk_g2s(wr_s, tab[l + 1].w_router + (size_t)e_lo * d, (uint32_t)nexp * d * 4u, wrbar);
  }

  // P3: down projection of this CTA's 16-column tiles, then the combine
  const int Rv = rt.act_off[U];  // rows that reached an expert
  const int hstride = 2 * I;     // bytes per staged h row
  unsigned char* hhi = regA;
  unsigned char* hlo = regA + (size_t)Rv * hstride;
  bool h_loaded = false;
  for (int ct = cta; ct < CT; ct += G) {
    if (!h_loaded) {
      if (tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(hbar, (uint32_t)Rv * 2u * hstride);
        bulk_g2s(hhi, p.h_hi, (uint32_t)Rv * hstride, hbar);
        bulk_g2s(hlo, p.h_lo, (uint32_t)Rv * hstride, hbar);
      }
      if (ok) ok = mbar_wait(hbar, lpar, p.st, 40);
      h_loaded = true;
      stamp(trace, 13);
    }
    // W_down stages of this output tile in ring order; four warps per expert
    // tile, a quarter of the reduction each.  A warp releases a stage as soon
    // as its own tiles of it are done, so warps run ahead into later stages.
    const int nst = (U + dps - 1) / dps;
    const int quarter = warp & 3;
    for (int st = 0; st < nst; ++st) {
      const int s = (i + st) % NS;
      if (ok) ok = mbar_wait(&full[s], ((i + st) / NS) & 1, p.st, 41);
      if (st == 0 && ct == cta) stamp(trace, 19);
      for (int j = warp >> 2; j < dps; j += kDecWarps / 4) {
        const int a = st * dps + j;
        if (a >= U) break;
        const unsigned char* tw = ring + (size_t)s * tbd + (size_t)j * tbi;
        const int na = rt.act_off[a + 1] - rt.act_off[a];
        const int p0 = rt.act_off[a];
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const bool has = g < na;
        if constexpr (kFp4) {
          float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
          for (int ch = quarter; ch < I / kChunkK; ch += 4) {
            float dh[4], dl[4];  // a chunk's MMAs chain in the accumulator; chunks add in fp32
            const unsigned char* cw = tw + ch * kChunkBytes;
            const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
            const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
            const uint32_t l0 = fp4_lane_scales(*reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8), c);
            const uint32_t l1 = fp4_lane_scales(*reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8), c);
#pragma unroll
            for (int gg = 0; gg < 4; ++gg) {
              const int col = (ch * 4 + gg) * kGroup + c * 8;
              uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
              if (has) {
                bh = *reinterpret_cast<const uint4*>(hhi + (size_t)(p0 + g) * hstride + col * 2);
                bl = *reinterpret_cast<const uint4*>(hlo + (size_t)(p0 + g) * hstride + col * 2);
              }
              uint32_t w0[4], w1[4];
              e2m1x8_f16_scaled(word_at(q0, gg), e4m3_pair_f16((l0 >> (8 * gg)) & 0xffu), w0);
              e2m1x8_f16_scaled(word_at(q1, gg), e4m3_pair_f16((l1 >> (8 * gg)) & 0xffu), w1);
              const uint32_t A0[4] = {w0[0], w1[0], w0[1], w1[1]}, A1[4] = {w0[2], w1[2], w0[3], w1[3]};
              if (gg == 0) {
                mma_f16_z(dh, A0, bh.x, bh.y);
                mma_f16_z(dl, A0, bl.x, bl.y);
              } else {
                mma_f16(dh, A0, bh.x, bh.y, dh);
                mma_f16(dl, A0, bl.x, bl.y, dl);
              }
              mma_f16(dh, A1, bh.z, bh.w, dh);
              mma_f16(dl, A1, bl.z, bl.w, dl);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              sh[q] += dh[q];
              sl[q] += dl[q];
            }
          }
          const float tsd = rt.tsd[a];
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[q] = (sh[q] + sl[q]) * tsd;
        } else
        for (int ch = quarter; ch < I / kChunkK; ch += 4) {
          const unsigned char* cw = tw + ch * kChunkBytes;
          const uint4 q0 = *reinterpret_cast<const uint4*>(cw + (g * 4 + c) * 16);
          const uint4 q1 = *reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + c) * 16);
          const uint2 s0 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8);
          const uint2 s1 = *reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8);
#pragma unroll 2  // (full unrolling spills at the 96-register cap)
          for (int gg = 0; gg < 4; ++gg) {
            const int col = (ch * 4 + gg) * kGroup + c * 8;
            uint4 bh = make_uint4(0, 0, 0, 0), bl = make_uint4(0, 0, 0, 0);
            if (has) {
              bh = *reinterpret_cast<const uint4*>(hhi + (size_t)(p0 + g) * hstride + col * 2);
              bl = *reinterpret_cast<const uint4*>(hlo + (size_t)(p0 + g) * hstride + col * 2);
            }
            uint32_t A[2][4], p0[4], p1[4];
            nib_pairs4_f16(word_at(q0, gg), p0);
            nib_pairs4_f16(word_at(q1, gg), p1);
#pragma unroll
            for (int sp = 0; sp < 2; ++sp) {
              A[sp][0] = p0[2 * sp];
              A[sp][1] = p1[2 * sp];
              A[sp][2] = p0[2 * sp + 1];
              A[sp][3] = p1[2 * sp + 1];
            }
            // h = hi + lo: two independent chains of two MMAs, summed afterwards
            float dh[4], dl[4];
            mma_f16_z(dh, A[0], bh.x, bh.y);
            mma_f16_z(dl, A[0], bl.x, bl.y);
            mma_f16(dh, A[1], bh.z, bh.w, dh);
            mma_f16(dl, A[1], bl.z, bl.w, dl);
            const float sc0 = scale_at(s0, gg), sc1 = scale_at(s1, gg);
            acc[0] = fmaf(sc0, dh[0] + dl[0], acc[0]);
            acc[1] = fmaf(sc0, dh[1] + dl[1], acc[1]);
            acc[2] = fmaf(sc1, dh[2] + dl[2], acc[2]);
            acc[3] = fmaf(sc1, dh[3] + dl[3], acc[3]);
          }
        }
        // D rows g, g+8 (output columns) x tokens 2c, 2c+1 -> this quarter's partial
        float* yp = ypart + (size_t)quarter * R * kTileRows;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int tok = 2 * c + (q & 1);
          const int row = (q < 2) ? g : g + 8;
          if (tok < na) yp[(size_t)(p0 + tok) * kTileRows + row] = acc[q];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&empty[s]);
      if (st == 0 && ct == cta) stamp(trace, 20);
    }
    i += nst;
    if (!ok) *(volatile int*)fail = 1;
    consumer_sync();
    stamp(trace, 14);
    // combine: out[t, ct*16 + col] = resid + sum_j w_j * y_j.  cpe neighbouring threads
    // share an output element: thread `sub` sums rows j = sub, sub + cpe, ... in
    // ascending order, then a fixed shuffle tree adds the cpe partial sums (no serial
    // chain of k dependent shared-memory round trips)
    {
      const int el = tid / cpe, sub = tid % cpe;
      const bool mine = el < T * kTileRows;
      const int t = el >> 4, col = el & 15;
      float acc = 0.f;
      if (mine) {
        for (int j = sub; j < k; j += cpe) {
          const int ps = rt.pos[t * k + j];
          if (ps >= 0) {
            float y = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) y += ypart[((size_t)q * R + ps) * kTileRows + col];
            acc = fmaf(rt.w[t * k + j], y, acc);
          }
        }
      }
      for (int off = 1; off < cpe; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (mine && sub == 0) {
        const size_t o = (size_t)t * d + (size_t)ct * kTileRows + col;
        const float v = bf16_bits_to_float(ct == cta ? resid0 : p.resid[o]) + acc;
        if (*(volatile int*)fail == 0) {
          if (p.out_f32) p.out_f32[o] = v;
          p.out[o] = float_to_bf16_bits(v);
        }
      }
    }
    consumer_sync();
  }
  stamp(trace, 7);
  }  // passed_b
  ring_i = i;
  // C: every output column of the layer written before the next layer (or the
  // LM head) reads whole rows
  if (kStack && (l + 1 < L || lm)) grid_barrier(p.gbar, fail, p.st, 42, nullptr, 0);
  }  // consumers
  __syncthreads();
  if (*(volatile int*)fail) break;
  }  // layers
  if (lm && *(volatile int*)fail == 0)
    lm_phase(p, regA, x16, ring, full, empty, rt.part, rt.sexp, rt.cand, ring_i, fail);
}

template <bool kFp4>
__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(const __grid_constant__ DecodeArgs p) {
  decode_body<false, kFp4>(p, nullptr);
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_stack_kernel(const __grid_constant__ StackArgs a) {
  decode_body<true, false>(a.base, a.tab);
}

struct DecodePlan {
  int offA, offB, offR, offRing, offX16, nstages;
  size_t smem;
  bool ok;
};

// k: routed experts per token; n_shared: 0 or 1 (one more row per token)
DecodePlan plan(int T, int d, int E, int k, int I, int n_shared, int G) {
  DecodePlan pl{};
  pl.ok = false;
  const int R = T * (k + n_shared);
  if (T < 1 || T > kDecMaxT || k > kDecMaxK || E > kDecMaxE || I > d || d > 8192) return pl;
  if (tile_bytes(d) % tile_bytes(I)) return pl;
  const size_t xall = (size_t)T * (2 * d + kSmemRowPad);
  const size_t hall = (size_t)R * 2 * (2 * I);
  const size_t xall2 = (xall + 127) / 128 * 128 + (size_t)(T + 1) * (2 * d + kSmemRowPad);  // bf16, fp16 + pad
  const size_t regA = ((xall2 > hall ? xall2 : hall) + 127) / 128 * 128;
  pl.offX16 = (int)((xall + 127) / 128 * 128);
  const int nexp = (E + G - 1) / G;
  const size_t p0 = (size_t)nexp * d * 4 + (size_t)T * nexp * kDecWarps * 4;
  const size_t p2 = (size_t)2 * kDecWarps * 32 * 8 * 4 + (size_t)4 * R * kTileRows * 4;
  const size_t regB = ((p0 > p2 ? p0 : p2) + 127) / 128 * 128;
  const size_t regR = ((size_t)(kDecWarps + kConsumers + kDecMaxT * kDecMaxK) * 8 +
                       (size_t)(2 * kDecMaxT + kDecWarps + 8 * R + 1 + 4) * 4 + 127) / 128 * 128;
  pl.offA = 1024;
  pl.offB = pl.offA + (int)regA;
  pl.offR = pl.offB + (int)regB;
  pl.offRing = pl.offR + (int)regR;
  const size_t budget = 227 * 1024;
  if ((size_t)pl.offRing + 2 * tile_bytes(d) > budget) return pl;
  int ns = (int)((budget - pl.offRing) / tile_bytes(d));
  if (ns > kMaxStages) ns = kMaxStages;
  pl.nstages = ns;
  pl.smem = (size_t)pl.offRing + (size_t)ns * tile_bytes(d);
  pl.ok = true;
  return pl;
}

int sm_count() {
  static int cnt[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cnt[dev] == 0) cudaDeviceGetAttribute(&cnt[dev], cudaDevAttrMultiProcessorCount, dev);
  return cnt[dev] > 0 ? cnt[dev] : 148;
}

}  // namespace

void* g_trace_buf = nullptr;
size_t g_trace_bytes = 0;

bool decode_fused_eligible(int T, int d, int E, int k, int I, int n_shared) {
  return plan(T, d, E, k, I, n_shared, sm_count()).ok;
}

namespace {

// Shared-memory attribute and the one-CTA-per-SM residency check of a fused
// kernel, once per device and size.
template <typename K>
cudaError_t prepare_fused(K* kernel, size_t smem, int* attr_set, size_t* occ_ok) {
  cudaError_t err = ensure_smem_attr(kernel, smem, attr_set);
  if (err != cudaSuccess) return err;
  // The CTAs wait on each other at the grid barriers, so all G of them must be
  // resident at once: one per SM.  A device where they do not fit takes the
  // unfused kernels.
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  if (occ_ok[dev] < smem) {
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kDecThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorNotSupported;
    occ_ok[dev] = smem;
  }
  return cudaSuccess;
}

DecodeArgs fill_args(const DecodeLaunch& L, const DecodePlan& pl, int G) {
  DecodeArgs a = {};
  a.x = L.x;
  a.resid = L.resid;
  a.T = L.T;
  a.d = L.d;
  a.E = L.E;
  a.k = L.k;
  a.n_shared = L.n_shared;
  a.I = L.I;
  a.renorm = L.renorm;
  a.gate = L.gate;
  a.up = L.up;
  a.down = L.down;
  a.w_router = L.w_router;
  a.b_router = L.b_router;
  a.gate_ts = L.gate_ts;
  a.up_ts = L.up_ts;
  a.down_ts = L.down_ts;
  a.forced_ids = L.forced_ids;
  a.forced_w = L.forced_w;
  a.out = L.out;
  a.out_f32 = L.out_f32;
  a.ids_out = L.ids_out;
  a.w_out = L.w_out;
  a.logits = L.logits;
  a.h_hi = L.h_hi;
  a.h_lo = L.h_lo;
  a.gbar = L.gbar;
  a.st = L.st;
  a.nstages = pl.nstages;
  a.offA = pl.offA;
  a.offB = pl.offB;
  a.offR = pl.offR;
  a.offRing = pl.offRing;
  a.offX16 = pl.offX16;
  a.prenorm = L.prenorm;
  a.eps = L.eps;
  a.xh_out = L.xh_out;
  a.n_layers = 1;
  a.trace = static_cast<unsigned long long*>(g_trace_buf);
  if (a.trace && g_trace_bytes < (size_t)G * kTracePoints * sizeof(unsigned long long)) a.trace = nullptr;
  return a;
}

template <typename K, typename A>
cudaError_t launch_fused(K* kernel, const A& args, int G, size_t smem, int pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace

cudaError_t launch_decode_fused(const DecodeLaunch& L, cudaStream_t s) {
  const int G = sm_count();
  const DecodePlan pl = plan(L.T, L.d, L.E, L.k, L.I, L.n_shared, G);
  if (!pl.ok) return cudaErrorNotSupported;
  if (L.gate_ts != nullptr) {  // NVFP4 banks
    static int attr_set[64] = {};
    static size_t occ_ok[64] = {};
    cudaError_t err = prepare_fused(decode_layer_kernel<true>, pl.smem, attr_set, occ_ok);
    if (err != cudaSuccess) return err;
    return launch_fused(decode_layer_kernel<true>, fill_args(L, pl, G), G, pl.smem, L.pdl, s);
  }
  static int attr_set[64] = {};
  static size_t occ_ok[64] = {};
  cudaError_t err = prepare_fused(decode_layer_kernel<false>, pl.smem, attr_set, occ_ok);
  if (err != cudaSuccess) return err;
  return launch_fused(decode_layer_kernel<false>, fill_args(L, pl, G), G, pl.smem, L.pdl, s);
}

bool decode_stack_eligible(int T, int d, int E, int k, int I, int n_shared, int n_layers, int V) {
  const int G = sm_count();
  const DecodePlan pl = plan(T, d, E, k, I, n_shared, G);
  const int nexp = (E + G - 1) / G;
  // the next layer's router rows go below the down projection's partials in region B
  return pl.ok && n_layers >= 1 && n_layers <= kMaxStackLayers && (size_t)nexp * d * 4 <= (size_t)2 * kDecWarps * 32 * 8 * 4 &&
         (V == 0 || V % kTileRows == 0);
}

cudaError_t launch_decode_stack(const DecodeLaunch& L, const StackLayer* layers, int n_layers, const uint8_t* lm_w,
                                int V, float* lm_logits, unsigned long long* lm_keys, int32_t* lm_argmax,
                                cudaStream_t s) {
  const int G = sm_count();
  if (!decode_stack_eligible(L.T, L.d, L.E, L.k, L.I, L.n_shared, n_layers, V)) return cudaErrorNotSupported;
  const DecodePlan pl = plan(L.T, L.d, L.E, L.k, L.I, L.n_shared, G);
  static int attr_set[64] = {};
  static size_t occ_ok[64] = {};
  cudaError_t err = prepare_fused(decode_stack_kernel, pl.smem, attr_set, occ_ok);
  if (err != cudaSuccess) return err;
  StackArgs a;
  a.base = fill_args(L, pl, G);
  a.base.n_layers = n_layers;
  a.base.lm_w = lm_w;
  a.base.lm_V = V;
  a.base.lm_logits = lm_logits;
  a.base.lm_keys = lm_keys;
  a.base.lm_argmax = lm_argmax;
  for (int l = 0; l < kMaxStackLayers; ++l) {
    const StackLayer& w = layers[l < n_layers ? l : 0];
    a.tab[l] = LayerPtrs{w.gate, w.up, w.down, w.w_router, w.b_router};
  }
  return launch_fused(decode_stack_kernel, a, G, pl.smem, L.pdl, s);
}

}  // namespace bitmoe
