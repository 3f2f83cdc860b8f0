// Prefill expert FFN: grouped GEMMs on the 5th-generation tensor cores.
//
// "Flint 40B : Best Mid Sized LLM", transcript 06:11 (kernels for prompt
// processing and low-bit projections) -- here with B300's tcgen05.mma and
// tensor memory.  With thousands of routed rows per layer each expert's
// projection is a real dense contraction:
//   GEMM1  [n_e x d] x [d x 2I]   gate and up, SwiGLU in the epilogue -> h (fp16)
//   GEMM2  [n_e x I] x [I x d]    down -> y rows (fp16 inside the layer, fp32 standalone)
//
// Tile: M = 128 routed rows (tokens of one expert), N = 256 weight rows, K in
// blocks of 64.  For GEMM1 the 256 weight rows are 128 gate rows stacked on
// the same 128 up rows, so one MMA per k-step produces both halves and a
// thread of the epilogue holds gate and up of the same features.  Operands
// live in 128-byte-swizzled K-major shared memory:
//   A  fp16 token rows, copied with cp.async (activations converted once to
//      fp16; GEMM1 gathers the rows through the grouping, GEMM2 reads the h
//      rows of the expert, which are contiguous);
//   B  int4 weights dequantised by producer warps to fp16 RNE(q * s) -- the
//      dequantised weight rounded once -- one weight row per thread, with
//      the packed words of the next four k-blocks in flight in registers.
// One thread issues tcgen05.mma (kind::f16, fp32 accumulate) into tensor
// memory; the two 256-column accumulators alternate so that the epilogue of
// one tile runs under the MMAs of the next.  Shared memory carries each
// operand byte once in and once out (a single-thread MMA stream reaches the
// full tensor rate on this part; what limits a producer-fed GEMM is how much
// it asks of shared memory).  Roles per CTA (17 warps):
//   0-7 B producers (weights), 8 MMA issuer + TMEM owner, 9-12 A producers
//   (tokens), 13-16 epilogue.
// Every wait is bounded (status word + clean exit, TMEM freed).
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kPM = 128;        // routed rows per tile (MMA M)
constexpr int kPN = 256;        // weight rows per tile (MMA N)
constexpr int kPK = 64;         // K per stage (one 128-byte swizzle row of fp16)
constexpr int kPStages = 4;
constexpr int kPWarps = 17;
constexpr int kPThreads = kPWarps * 32;
constexpr int kABytes = kPM * kPK * 2;  // 16 KB token tile
constexpr int kBBytes = kPN * kPK * 2;  // 32 KB weight tile
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kPrefetch = 4;            // k-blocks of packed weight words in flight per producer thread
constexpr int kWarpMMA = 8, kWarpA0 = 9, kWarpEpi0 = 13;

struct PrefillArgs {
  int mode;            // 1 = gate/up + SwiGLU, 2 = down
  int T, d, I, E, k;   // shapes
  int Kdim;            // reduction length (d for mode 1, I for mode 2)
  int MT;              // weight tiles per expert (I/128 for mode 1, d/256 for mode 2)
  const uint8_t* wa;   // packed bank (gate for mode 1, down for mode 2)
  const uint8_t* wb;   // packed bank (up for mode 1)
  int wrows;           // rows per expert in the packed banks (I or d)
  const __half* x16;   // [T, d] fp16 copy of the activations (mode 1)
  const __half* hin;   // [R, I] fp16 (mode 2)
  const int32_t* offsets;      // [E+1]
  const int32_t* sorted_rows;  // [R]
  const int32_t* nb_prefix;    // [E+1] prefix of ceil(n_e / 128)
  __half* hout;        // [R, I] fp16 (mode 1 output)
  float* yout;         // [R, d] fp32 (mode 2 output, when y16 is null)
  __half* y16;         // [R, d] fp16 (mode 2 output)
  DevStatus* st;
  unsigned long long* trace;  // optional [grid][16] per-role cycle counters
};

// Optional per-role cycle counters (clock64) written per CTA when a trace
// buffer is set: 0 MMA waiting on tokens, 1 MMA waiting on weights, 2 MMA
// waiting for a free accumulator, 3 MMA total, 5 weight producers waiting for
// a free stage, 6 weight producers total, 7 token producers waiting for a free
// stage, 8 epilogue waiting for an accumulator, 9 epilogue total, 11 tiles.
__device__ __forceinline__ void ptrace(const PrefillArgs& p, int slot, unsigned long long v) {
  if (p.trace) p.trace[blockIdx.x * 16 + slot] = v;
}

// ---------------------------------------------------------------- tcgen05 helpers

__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr) {
  // K-major, 128-byte swizzle: 8-row atoms of 1024 bytes (SBO), version 1.
  uint64_t desc = 0;
  desc |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  desc |= (uint64_t)1 << 16;                     // leading byte offset (unused when swizzled)
  desc |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset
  desc |= (uint64_t)1 << 46;                     // descriptor version
  desc |= (uint64_t)2 << 61;                     // SWIZZLE_128B
  return desc;
}

__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N) {
  // kind::f16: D fp32 (bits 4-5 = 1), A fp16, B fp16 (0), K-major both, N>>3 at 17, M>>4 at 24.
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 16-byte chunk j (0..7) of operand row r inside a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t swz_off(int r, int j) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((j ^ (r & 7)) << 4));
}

__device__ __forceinline__ int expert_of(const int32_t* __restrict__ pre, int E, int b) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= b) lo = mid;
    else hi = mid;
  }
  return lo;
}

struct TileInfo {
  int e, m, p0, nval;
};

__device__ __forceinline__ TileInfo tile_info(const PrefillArgs& p, int tile) {
  TileInfo ti;
  const int b = tile / p.MT;
  ti.m = tile - b * p.MT;
  ti.e = expert_of(p.nb_prefix, p.E, b);
  ti.p0 = p.offsets[ti.e] + (b - p.nb_prefix[ti.e]) * kPM;
  const int rem = p.offsets[ti.e + 1] - ti.p0;
  ti.nval = rem < kPM ? rem : kPM;
  return ti;
}

// Dequantise the 8 int4 values of one packed word times scale s into 16 bytes of fp16.
__device__ __forceinline__ uint4 dequant_word_f16(uint32_t w, __half2 s2) {
  uint32_t o[4];
#pragma unroll
  for (int pr = 0; pr < 4; ++pr) {
    const uint32_t q = nib_pair_f16(w, pr);
    __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&q), s2);
    o[pr] = *reinterpret_cast<uint32_t*>(&v);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

struct WRaw {
  uint2 w[4];   // [quarter]: the two group words of this k-block
  uint32_t sc;  // the two fp16 group scales
};

// Packed words of row rr (inside its 16-row tile at `tile`) for k-block kb.
__device__ __forceinline__ void load_wraw(WRaw& a, const uint8_t* tile, int kb, int rr) {
  const uint8_t* c0 = tile + (size_t)(kb >> 1) * kChunkBytes;
  const int gg0 = (kb & 1) * 2;
  a.sc = __ldg(reinterpret_cast<const unsigned int*>(c0 + kChunkQBytes + rr * 8 + gg0 * 2));
#pragma unroll
  for (int c = 0; c < 4; ++c) a.w[c] = __ldg(reinterpret_cast<const uint2*>(c0 + (rr * 4 + c) * 16 + gg0 * 4));
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_gemm_kernel(PrefillArgs p) {
  extern __shared__ unsigned char smem_raw[];
  // 1024-byte aligned base for the swizzled operand tiles
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPStages * kStageBytes);
  uint64_t* a_full = bars;                 // [kPStages], one arrival per token-producer thread
  uint64_t* b_full = a_full + kPStages;    // [kPStages], one arrival per weight-producer warp
  uint64_t* s_empty = b_full + kPStages;   // [kPStages], MMA commit
  uint64_t* acc_full = s_empty + kPStages; // [2], MMA commit
  uint64_t* acc_empty = acc_full + 2;      // [2], one arrival per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* fail = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t kTmemCols = 2 * kPN;  // two 256-column accumulators

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&a_full[s], 128);
      mbar_init(&b_full[s], 8);
      mbar_init(&s_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int nblocks = p.nb_prefix[p.E];
  const int n_tiles = nblocks * p.MT;
  const int nkb = p.Kdim / kPK;
  const int wrow_tiles = p.wrows / kTileRows;  // packed 16-row tiles per expert
  const int tb = (int)tile_bytes(p.Kdim);       // bytes per packed 16-row tile

  if (warp < 8) {
    // ---------------- weight producers: one weight row per thread -> fp16 RNE(q*s) into the B tile
    const int brow = warp * 32 + lane;  // 0..255 inside the tile
    int it = 0;
    long long t_wait = 0;
    const long long t_start = clock64();
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const TileInfo ti = tile_info(p, tile);
      const uint8_t* bank;
      int wrow;
      if (p.mode == 1) {  // rows 0..127 gate, 128..255 up, same 128 features
        bank = (brow < 128) ? p.wa : p.wb;
        wrow = ti.m * 128 + (brow & 127);
      } else {
        bank = p.wa;
        wrow = ti.m * kPN + brow;
      }
      const uint8_t* tile16 = bank + ((size_t)ti.e * wrow_tiles + (wrow >> 4)) * tb;
      const int rr = wrow & 15;
      WRaw raw[kPrefetch];
#pragma unroll
      for (int j = 0; j < kPrefetch; ++j)
        if (j < nkb) load_wraw(raw[j], tile16, j, rr);
      for (int kb0 = 0; kb0 < nkb && ok; kb0 += kPrefetch) {
#pragma unroll
        for (int j = 0; j < kPrefetch; ++j) {
          const int kb = kb0 + j;
          if (kb >= nkb) break;
          const int s = it % kPStages;
          const long long w0 = clock64();
          if (it >= kPStages && !mbar_wait(&s_empty[s], ((it / kPStages) - 1) & 1, p.st, 50)) {
            *(volatile int*)fail = 1;
            ok = false;
            break;
          }
          t_wait += clock64() - w0;
          unsigned char* dst = stages + (size_t)s * kStageBytes + kABytes;
          const __half2 s0 = __half2half2(__ushort_as_half((uint16_t)(raw[j].sc & 0xffffu)));
          const __half2 s1 = __half2half2(__ushort_as_half((uint16_t)(raw[j].sc >> 16)));
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            // first group of the k-block -> k in [8c, 8c+8), second group -> [32+8c, ...)
            *reinterpret_cast<uint4*>(dst + swz_off(brow, c)) = dequant_word_f16(raw[j].w[c].x, s0);
            *reinterpret_cast<uint4*>(dst + swz_off(brow, 4 + c)) = dequant_word_f16(raw[j].w[c].y, s1);
          }
          if (kb + kPrefetch < nkb) load_wraw(raw[j], tile16, kb + kPrefetch, rr);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive_cta(&b_full[s]);
          ++it;
        }
      }
    }
    if (warp == 0 && lane == 0) {
      ptrace(p, 5, t_wait);
      ptrace(p, 6, clock64() - t_start);
    }
  } else if (warp >= kWarpA0 && warp < kWarpA0 + 4) {
    // ---------------- token producers: one routed row per thread, cp.async into the A tile;
    // a stage is published (proxy fence + arrival) once its copies have landed,
    // keeping up to kInFlight stages of copies outstanding
    constexpr int kInFlight = 2;
    const int n = (warp - kWarpA0) * 32 + lane;
    int it = 0, published = 0;
    long long t_wait = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const TileInfo ti = tile_info(p, tile);
      const bool valid = n < ti.nval;
      const int pos = ti.p0 + (valid ? n : 0);
      const __half* src = (p.mode == 1) ? p.x16 + (size_t)(p.sorted_rows[pos] / p.k) * p.d
                                        : p.hin + (size_t)pos * p.I;
      const uint32_t nbytes = valid ? 16u : 0u;  // 0 = zero fill
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kPStages;
        const long long w0 = clock64();
        if (it >= kPStages && !mbar_wait(&s_empty[s], ((it / kPStages) - 1) & 1, p.st, 51)) {
          *(volatile int*)fail = 1;
          ok = false;
          break;
        }
        t_wait += clock64() - w0;
        const uint32_t dst = smem_u32(stages + (size_t)s * kStageBytes);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + swz_off(n, j)),
                       "l"(src + kb * kPK + j * 8), "r"(nbytes)
                       : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        if (it + 1 - published > kInFlight) {
          asm volatile("cp.async.wait_group %0;" ::"n"(kInFlight) : "memory");
          fence_proxy_async_smem();
          mbar_arrive_cta(&a_full[published % kPStages]);
          ++published;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
    while (published < it) {
      mbar_arrive_cta(&a_full[published % kPStages]);
      ++published;
    }
    if (warp == kWarpA0 && lane == 0) ptrace(p, 7, t_wait);
  } else if (warp == kWarpMMA) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_f16(kPM, kPN);
      int it = 0, lt = 0;
      long long t_a = 0, t_b = 0, t_acc = 0;
      const long long t_start = clock64();
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const long long w0 = clock64();
        if (lt >= 2 && !mbar_wait(&acc_empty[buf], ((lt >> 1) - 1) & 1, p.st, 52)) {
          *(volatile int*)fail = 1;
          break;
        }
        t_acc += clock64() - w0;
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(buf * kPN);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kPStages;
          const long long w1 = clock64();
          const bool got_a = mbar_wait(&a_full[s], (it / kPStages) & 1, p.st, 53);
          const long long w2 = clock64();
          const bool got_b = got_a && mbar_wait(&b_full[s], (it / kPStages) & 1, p.st, 54);
          t_a += w2 - w1;
          t_b += clock64() - w2;
          if (!got_b) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t asm_ = smem_u32(stages + (size_t)s * kStageBytes);
          const uint32_t bsm = asm_ + (uint32_t)kABytes;
#pragma unroll
          for (int ks = 0; ks < kPK / 16; ++ks)
            umma_f16(d0, umma_smem_desc(asm_ + ks * 32), umma_smem_desc(bsm + ks * 32), idesc,
                     (kb > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&s_empty[s]);  // frees the stage once these MMAs have read it
        }
        if (!ok) {
          *(volatile int*)fail = 1;
          break;
        }
        umma_commit(&acc_full[buf]);
      }
      ptrace(p, 0, t_a);
      ptrace(p, 1, t_b);
      ptrace(p, 2, t_acc);
      ptrace(p, 3, clock64() - t_start);
      ptrace(p, 11, lt);
    }
  } else if (warp >= kWarpEpi0) {
    // ---------------- epilogue: TMEM -> registers -> outputs; one routed row per thread
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int n = q * 32 + lane;
    int lt = 0;
    long long t_wait = 0;
    const long long t_start = clock64();
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const long long w0 = clock64();
      if (!mbar_wait(&acc_full[buf], (lt >> 1) & 1, p.st, 55)) {
        *(volatile int*)fail = 1;
        break;
      }
      t_wait += clock64() - w0;
      tc_fence_after();
      const TileInfo ti = tile_info(p, tile);
      const bool valid = n < ti.nval;
      const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kPN);
      if (p.mode == 1) {
        __half* hrow = p.hout + (size_t)(ti.p0 + (valid ? n : 0)) * p.I + ti.m * 128;
        for (int c0 = 0; c0 < 128; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16(tq + (uint32_t)c0, g);
          tmem_ld16(tq + (uint32_t)(128 + c0), u);
          tmem_ld_wait();
          uint32_t hv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float h0 = silu_mul(__uint_as_float(g[2 * j]), __uint_as_float(u[2 * j]));
            const float h1 = silu_mul(__uint_as_float(g[2 * j + 1]), __uint_as_float(u[2 * j + 1]));
            __half2 h2 = __floats2half2_rn(h0, h1);
            hv[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          if (valid) {
            *reinterpret_cast<uint4*>(hrow + c0) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(hrow + c0 + 8) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
          }
        }
      } else {
        const size_t rowoff = (size_t)(ti.p0 + (valid ? n : 0)) * p.d + (size_t)ti.m * kPN;
        for (int c0 = 0; c0 < kPN; c0 += 16) {
          uint32_t g[16];
          tmem_ld16(tq + (uint32_t)c0, g);
          tmem_ld_wait();
          if (!valid) continue;
          if (p.y16) {
            uint32_t hv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              __half2 h2 = __floats2half2_rn(__uint_as_float(g[2 * j]), __uint_as_float(g[2 * j + 1]));
              hv[j] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(p.y16 + rowoff + c0) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4*>(p.y16 + rowoff + c0 + 8) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(p.yout + rowoff + c0 + 4 * j) =
                  make_uint4(g[4 * j], g[4 * j + 1], g[4 * j + 2], g[4 * j + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acc_empty[buf]);
    }
    if (warp == kWarpEpi0 && lane == 0) {
      ptrace(p, 8, t_wait);
      ptrace(p, 9, clock64() - t_start);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols) : "memory");
  }
}

__global__ void nb_prefix_kernel(const int32_t* __restrict__ offsets, int E, int32_t* __restrict__ pre) {
  // one thread: E <= 1024 small serial scan (prefill only)
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      pre[e] = run;
      run += (offsets[e + 1] - offsets[e] + kPM - 1) / kPM;
    }
    pre[E] = run;
  }
}

__global__ void bf16_to_f16_kernel(const uint16_t* __restrict__ x, size_t n8, __half* __restrict__ y) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __half2 h2 = __floats2half2_rn(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
      o[q] = *reinterpret_cast<uint32_t*>(&h2);
    }
    reinterpret_cast<uint4*>(y)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

constexpr size_t kPSmem = 1024 + (size_t)kPStages * kStageBytes + 256;

int sm_count_prefill() {
  static int cnt[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cnt[dev] == 0) cudaDeviceGetAttribute(&cnt[dev], cudaDevAttrMultiProcessorCount, dev);
  return cnt[dev] > 0 ? cnt[dev] : 148;
}

}  // namespace

bool prefill_eligible(int d, int I) { return d % 256 == 0 && I % 256 == 0; }

cudaError_t launch_prefill_ffn(const FfnArgs& a, int32_t* nb_prefix, __half* x16, __half* y16, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) return cudaSuccess;
  if (!prefill_eligible(a.d, a.I)) return cudaErrorNotSupported;
  nb_prefix_kernel<<<1, 32, 0, s>>>(a.offsets, a.E, nb_prefix);
  const size_t n8 = (size_t)a.T * a.d / 8;
  bf16_to_f16_kernel<<<(int)(n8 / 256 + 1 < 148 * 16 ? n8 / 256 + 1 : 148 * 16), 256, 0, s>>>(a.x, n8, x16);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  static int attr1[64] = {};
  if ((err = ensure_smem_attr(prefill_gemm_kernel, kPSmem, attr1)) != cudaSuccess) return err;
  const int G = sm_count_prefill();
  // upper bound on the 128-row blocks, for the grid size
  const long blocks = (long)R / kPM + (R < a.E ? R : a.E) + 1;
  const size_t need = (size_t)2 * G * 16 * sizeof(unsigned long long);
  unsigned long long* tr = (g_trace_buf && g_trace_bytes >= need) ? static_cast<unsigned long long*>(g_trace_buf) : nullptr;

  PrefillArgs p1 = {};
  p1.mode = 1;
  p1.T = a.T;
  p1.d = a.d;
  p1.I = a.I;
  p1.E = a.E;
  p1.k = a.k;
  p1.Kdim = a.d;
  p1.MT = a.I / 128;
  p1.wa = a.gate;
  p1.wb = a.up;
  p1.wrows = a.I;
  p1.x16 = x16;
  p1.offsets = a.offsets;
  p1.sorted_rows = a.sorted_rows;
  p1.nb_prefix = nb_prefix;
  p1.hout = a.h_hi;  // fp16 h, [R, I]
  p1.st = a.st;
  p1.trace = tr;
  const long g1 = blocks * p1.MT;
  prefill_gemm_kernel<<<(int)(g1 < G ? g1 : G), kPThreads, kPSmem, s>>>(p1);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;

  PrefillArgs p2 = p1;
  p2.mode = 2;
  p2.Kdim = a.I;
  p2.MT = a.d / kPN;
  p2.wa = a.down;
  p2.wb = nullptr;
  p2.wrows = a.d;
  p2.x16 = nullptr;
  p2.hin = a.h_hi;
  p2.hout = nullptr;
  p2.yout = a.y_rows;
  p2.y16 = y16;
  p2.trace = tr ? tr + (size_t)G * 16 : nullptr;
  const long g2 = blocks * p2.MT;
  prefill_gemm_kernel<<<(int)(g2 < G ? g2 : G), kPThreads, kPSmem, s>>>(p2);
  return cudaGetLastError();
}

}  // namespace bitmoe
