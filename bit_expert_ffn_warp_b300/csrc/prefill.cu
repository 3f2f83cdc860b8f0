// Prefill expert FFN: grouped GEMMs on the 5th-generation tensor cores.
//
// "Flint 40B : Best Mid Sized LLM", transcript 06:43 (kernels for prompt
// processing and low-bit projections) -- here with B300's tcgen05.mma and
// tensor memory.  With thousands of routed rows per layer each expert's
// projection is a real dense contraction:
//   GEMM1  h = silu(Wg x) * (Wu x)   per routed row, fp16 h
//   GEMM2  y = Wd h                  per routed row (fp16 inside the layer, fp32 standalone)
//
// Orientation: D[m, n] = sum_k W[m, k] * X[n, k].  The MMA's A side (M = 128) is 128
// weight rows held in tensor memory, its B side (N = the routed rows of one 128-row
// expert block, rounded up to 16) the fp16 activation rows in 128-byte-swizzled
// K-major shared memory.  A tile is one expert block times 256 weight rows, two M
// tiles into two accumulators D0, D1 of N columns: for GEMM1 128 gate rows and the
// same 128 up rows, so a thread of the epilogue holds gate and up of one feature for
// every routed row and writes h directly; for GEMM2 256 rows of W_down.
//   B  fp16 routed rows, contiguous in grouped order (GEMM1: the activations
//      gathered and converted once to fp16 by a small kernel; GEMM2: the h rows
//      GEMM1 wrote), loaded by 2-D TMA boxes of 64 rows x 64 K into a 4-stage ring;
//   A  int4 (or NVFP4) weights read by eight dequantising warps straight from global
//      memory in the packed tile order, converted in registers to fp16 RNE(q * s)
//      (NVFP4: code times block scale, exact) and stored into tensor memory with
//      tcgen05.st -- the dequantised weights never pass through shared memory, and an
//      expert block with few routed rows costs an MMA of that width only.
// One thread issues tcgen05.mma (kind::f16, A from tensor memory, fp32 accumulate).
// Tensor memory (512 columns): D0, D1 (128 columns each) and a 4-stage A ring
// (2 M tiles x 32 columns per stage).  The epilogue copies both accumulators into
// shared memory, converted and turned to row order, releases them, then writes h or y
// with 16-byte stores while the next tile's MMAs run.
// Roles per CTA (16 warps): 1 routed-row TMA, 2 MMA issuer + TMEM owner (on the third
// SM sub-partition, which the other roles load least), 4-11 dequantisation,
// 12-15 epilogue (one per TMEM lane quarter).
// Every wait is bounded (status word + clean exit, TMEM freed).

#include <cuda.h>

#include "kernels.h"
#include "tc.cuh"

namespace bitmoe {
namespace {

constexpr int kPM = 128;                  // weight rows per M tile (two M tiles per tile)
constexpr int kPN = 256;                  // weight rows per tile (GEMM 2; GEMM 1: 128 gate + 128 up)
constexpr int kPK = 64;                   // K per stage (one 128-byte swizzle row of fp16)
constexpr int kSubTiles = kPN / kTileRows;  // 16 packed 16-row tiles per weight tile
constexpr int kBoxRows = 64;              // routed rows per TMA box
constexpr int kRowsPerBlock = 128;        // routed rows per expert block (MMA N at most)

struct PrefillArgs {
  CUtensorMap tmap_a;  // routed rows [R, Kdim] fp16 (the MMA's B), box 64 x 64, 128-byte swizzle
  int mode;            // 1 = gate/up + SwiGLU, 2 = down
  int T, d, I, E, k;   // shapes
  int Kdim;            // reduction length (d for mode 1, I for mode 2)
  int FB;              // weight tiles per expert (I/128 for mode 1, d/256 for mode 2)
  const uint8_t* wa;   // packed bank (gate for mode 1, down for mode 2)
  const uint8_t* wb;   // packed bank (up for mode 1)
  const float* tsa;    // NVFP4 banks: tensor scales per expert of wa and wb (null: int4 banks)
  const float* tsb;
  int wrows;           // rows per expert in the packed banks (I or d)
  const int32_t* offsets;      // [E+1]
  const int32_t* nb_prefix;    // [E+1] prefix of ceil(n_e / 128)
  const int32_t* pair_list;    // [nb_prefix[E]] expert blocks, widest first
  __half* hout;        // [R, I] fp16 (mode 1 output)
  float* yout;         // [R, d] fp32 (mode 2 output, when y16 is null)
  __half* y16;         // [R, d] fp16 (mode 2 output)
  DevStatus* st;
  unsigned long long* trace;  // optional [grid][16] per-role cycle counters
};

// Optional per-role cycle counters (clock64) written per CTA when a trace buffer is
// set: 2 MMA waiting for free accumulators, 3 MMA total, 4 MMA waiting for a full
// stage, 6 dequantisation waiting for a free stage, 7 dequantisation total,
// 9 epilogue waiting for the accumulators, 10 epilogue total, 11 tiles, 12 sum of the
// tiles' N.
__device__ __forceinline__ void ptrace(const PrefillArgs& p, int slot, unsigned long long v) {
  if (p.trace) p.trace[blockIdx.x * 16 + slot] = v;
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
  int e;      // expert
  int f;      // weight tile inside the expert (0..FB-1)
  int p0;     // first grouped row of the tile
  int nval;   // routed rows in the tile (<= 128)
};

// The j-th tile a CTA takes: tiles are ordered widest block first and dealt out in a
// snake (c, then G-1-c, ...).
__device__ __forceinline__ int snake_tile(int j) {
  const int G = gridDim.x, c = blockIdx.x;
  return j * G + ((j & 1) ? G - 1 - c : c);
}

__device__ __forceinline__ TileInfo tile_info(const PrefillArgs& p, int sidx) {
  TileInfo ti;
  const int pi = sidx / p.FB;
  ti.f = sidx - pi * p.FB;
  const int b = p.pair_list[pi];
  ti.e = expert_of(p.nb_prefix, p.E, b);
  ti.p0 = p.offsets[ti.e] + (b - p.nb_prefix[ti.e]) * kRowsPerBlock;
  const int rem = p.offsets[ti.e + 1] - ti.p0;
  ti.nval = rem < kRowsPerBlock ? rem : kRowsPerBlock;
  return ti;
}

// Packed 16-row tile (inside the expert's bank) of sub-tile i (0..15) of weight tile f.
__device__ __forceinline__ const uint8_t* subtile_base(const PrefillArgs& p, const TileInfo& ti, int i) {
  const int rtiles = p.wrows / kTileRows;
  const uint8_t* bank;
  int rt;
  if (p.mode == 1) {  // sub-tiles 0-7: gate rows 128f.., 8-15: the same up rows
    bank = (i < 8) ? p.wa : p.wb;
    rt = ti.f * 8 + (i & 7);
  } else {
    bank = p.wa;
    rt = ti.f * 16 + i;
  }
  return bank + ((size_t)ti.e * rtiles + rt) * (size_t)tile_bytes(p.Kdim);
}

// ---------------------------------------------------------------- weights in tensor memory
//
// K order.  The dequantising warps read the packed tiles in the mma-fragment order
// (lane (g, c) holds rows g and g+8, columns 8c .. 8c+7 of every 32-column group) and
// store them with tcgen05.st.16x256b, whose thread t writes lanes t/4 and t/4 + 8,
// columns 2(t%4) and 2(t%4)+1 of each 8-column block.  So column p of a 16-column
// group (one 32-element K group, two K elements per column) holds the K pair
// P(p) = 4 ((p % 8) / 2) + p % 2 + 2 (p / 8); the B rows are stored with the same
// permutation inside every 32-element group (the gathered activations, and the h rows
// GEMM 1 writes for GEMM 2), so every product pairs the right elements.
constexpr int kQThreads = 16 * 32;
constexpr int kQWarpMMA = 2, kQWarpB = 1, kQWarpDq0 = 4, kQWarpEpi0 = 12;
constexpr int kQBStages = 4;                      // B ring (128 rows x 64 K fp16 = 16 KB each)
constexpr int kQAStages = kQBStages;              // A ring in tensor memory (2 tiles x 32 columns each):
                                                  // the same depth, so one MMA commit frees both
constexpr int kQBBytes = kPM * kPK * 2;
constexpr uint32_t kQTmemCols = 512;              // D0, D1 (128 columns each), then the A ring
constexpr int kQStageWarp = 2 * 128 * 32 * 4;     // per epilogue warp: [2 M tiles][128 routed rows][32] fp32 at most
constexpr int kQTileCache = 128;                  // tiles of a CTA whose TileInfo is computed once, up front
constexpr size_t kQSmem =
    (size_t)kQBStages * kQBBytes + 4 * (size_t)kQStageWarp + (size_t)kQTileCache * sizeof(TileInfo) + 1024 + 256;
static_assert(kQSmem <= 227 * 1024, "shared memory budget");
static_assert(256 + kQAStages * 2 * 32 <= (int)kQTmemCols, "tensor memory budget");

// Position of K pair P (0..15) inside its 32-element group (inverse of P(p) above).
__host__ __device__ constexpr int kpair_pos(int P) { return 2 * (P >> 2) + (P & 1) + 8 * ((P >> 1) & 1); }
// Column of element f of a row stored in that order.
__host__ __device__ constexpr int kperm(int f) { return (f & ~31) + 2 * kpair_pos((f & 31) >> 1) + (f & 1); }

__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_st16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ uint32_t word_at(const uint4& q, int gg) {
  return gg == 0 ? q.x : gg == 1 ? q.y : gg == 2 ? q.z : q.w;
}

// The eight weights of one packed word as fp16 pairs o[j] = columns 2j, 2j+1 of the lane's octet:
// int4: RNE(q * s) with the group's fp16 scale; NVFP4: code times block scale, exact.
template <bool kFp4>
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t scale_bits, uint32_t (&o)[4]) {
  if constexpr (kFp4) {
    e2m1x8_f16_scaled(w, e4m3_pair_f16(scale_bits), o);
  } else {
    uint32_t q[4];
    nib_pairs4_f16(w, q);
    const __half2 s2 = __half2half2(__ushort_as_half((uint16_t)scale_bits));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&q[j]), s2);
      o[j] = *reinterpret_cast<const uint32_t*>(&v);
    }
  }
}

template <bool kFp4>
__global__ void __launch_bounds__(kQThreads, 1) prefill_wa_kernel(const __grid_constant__ PrefillArgs p) {
  pdl_enter();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // the swizzled B tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) record_status(p.st, kStatusCheck, 80, (int)(smem_u32(smem_raw) & 1023u));
    return;
  }
  unsigned char* bst = smem_raw;  // [kQBStages] B stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)kQBStages * kQBBytes);
  // stage s is full once its B rows have landed (TMA transaction count, armed by the B
  // loader's arrival) and the eight dequantising warps have stored its A (eight more
  // arrivals): one barrier, so the MMA thread waits once per stage
  uint64_t* b_full = bars;                     // [kQBStages] 1 + 8 arrivals + B bytes
  uint64_t* b_empty = b_full + kQBStages;      // [kQBStages] MMA commit: B and A stage s free again
  uint64_t* a_full = b_full;                   // (the same barriers)
  uint64_t* a_empty = b_empty;
  uint64_t* d_full = b_empty + kQBStages;      // MMA commit: the tile's accumulators are complete
  uint64_t* d_empty = d_full + 1;              // one arrival per epilogue warp
  uint64_t* drain = d_empty + 1;               // MMA commit: every MMA of this CTA done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  unsigned char* epi_stage = smem_raw + (size_t)kQBStages * kQBBytes + 1024;  // [4 warps][kQStageWarp]
  TileInfo* tcache = reinterpret_cast<TileInfo*>(epi_stage + 4 * (size_t)kQStageWarp);  // [kQTileCache]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kQBStages; ++s) {
      mbar_init(&b_full[s], 1 + 8);
      mbar_init(&b_empty[s], 1);
    }
    mbar_init(d_full, 1);
    mbar_init(d_empty, 4);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == kQWarpMMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kQTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  const int n_tiles = p.nb_prefix[p.E] * p.FB;
  // every role walks the same tiles: their (expert, block, rows) are looked up once here,
  // in parallel, instead of by each role's single thread on its critical path
  for (int j = tid; j < kQTileCache; j += kQThreads) {
    const int tile = snake_tile(j);
    if (tile < n_tiles) tcache[j] = tile_info(p, tile);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto a_col = [](int s, int t) { return (uint32_t)(256 + (s * 2 + t) * 32); };
  auto tinfo = [&](int j, int tile) { return j < kQTileCache ? tcache[j] : tile_info(p, tile); };

  const int nchunks = p.Kdim / kChunkK;
  const int nkb = 2 * nchunks;  // 64-K stages per tile

  if (warp == kQWarpB) {
    // ---------------- B: the tile's routed rows, 64-row TMA boxes of 64 K (two per full block)
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_a)) : "memory");
      int it = 0;
      bool ok = true;
      // the dequantising warps read the packed weights straight from global memory, a
      // chunk ahead: pull each tile's weights into L2 one tile earlier, so that those
      // loads meet L2 rather than HBM
      auto prefetch_tile = [&](int jn, int tile) {
        if (tile >= n_tiles) return;
        const TileInfo tn = tinfo(jn, tile);
        for (int i = 0; i < kSubTiles; ++i)
          bulk_prefetch_l2(subtile_base(p, tn, i), (uint32_t)tile_bytes(p.Kdim));
      };
      prefetch_tile(0, snake_tile(0));
      for (int j = 0, tile = snake_tile(0); tile < n_tiles && ok; tile = snake_tile(++j)) {
        const TileInfo ti = tinfo(j, tile);
        prefetch_tile(j + 1, snake_tile(j + 1));
        const int nbox = (ti.nval + kBoxRows - 1) / kBoxRows;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kQBStages;
          if (it >= kQBStages && !mbar_wait(&b_empty[s], ((it / kQBStages) - 1) & 1, p.st, 81)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[s], (uint32_t)nbox * kBoxRows * kPK * 2);
          const uint32_t dst = smem_u32(bst + (size_t)s * kQBBytes);
          for (int i = 0; i < nbox; ++i)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                    dst + (uint32_t)(i * kBoxRows * kPK * 2)),
                "l"(reinterpret_cast<uint64_t>(&p.tmap_a)), "r"(kb * kPK), "r"(ti.p0 + i * kBoxRows),
                "r"(smem_u32(&b_full[s]))
                : "memory");
        }
      }
      for (int n = (it > kQBStages ? it - kQBStages : 0); n < it; ++n)
        mbar_wait(&b_full[n % kQBStages], (n / kQBStages) & 1, p.st, 82);
    }
  } else if (warp >= kQWarpDq0 && warp < kQWarpDq0 + 8) {
    // ---------------- dequantisation: warp (t, q) writes rows 32q .. 32q+31 of M tile t, that is
    // packed sub-tiles 8t + 2q and 8t + 2q + 1, into its own TMEM lane quarter q; the packed words
    // come straight from global memory (L2), a chunk ahead of their use
    const int q = warp & 3, t = (warp - kQWarpDq0) >> 2;
    const int g = lane >> 2, cl = lane & 3;
    uint4 w0[2], w1[2], n0[2], n1[2];  // rows g, g+8 of sub-tiles k = 0, 1: this chunk and the next
    uint2 s0[2], s1[2], m0[2], m1[2];
    TileInfo ti{};
    const uint8_t* sb[2] = {nullptr, nullptr};
    // the flat sequence of (tile, chunk) this CTA works through
    int jn = 0, cn = 0, tile_n = snake_tile(0);
    auto load = [&](int tile, int c, uint4 (&a0)[2], uint4 (&a1)[2], uint2 (&z0)[2], uint2 (&z1)[2]) {
      if (c == 0) {
        ti = tinfo(jn, tile);
        sb[0] = subtile_base(p, ti, 8 * t + 2 * q);
        sb[1] = subtile_base(p, ti, 8 * t + 2 * q + 1);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint8_t* cw = sb[k] + (size_t)c * kChunkBytes;
        a0[k] = __ldg(reinterpret_cast<const uint4*>(cw + (g * 4 + cl) * 16));
        a1[k] = __ldg(reinterpret_cast<const uint4*>(cw + ((g + 8) * 4 + cl) * 16));
        z0[k] = __ldg(reinterpret_cast<const uint2*>(cw + kChunkQBytes + g * 8));
        z1[k] = __ldg(reinterpret_cast<const uint2*>(cw + kChunkQBytes + (g + 8) * 8));
      }
    };
    if (tile_n < n_tiles) load(tile_n, 0, n0, n1, m0, m1);
    int it = 0;
    bool ok = true;
    long long t_wait = 0;
    const long long t_start = clock64();
    while (tile_n < n_tiles && ok) {
      const int c = cn;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        w0[k] = n0[k];
        w1[k] = n1[k];
        s0[k] = m0[k];
        s1[k] = m1[k];
      }
      // advance to the next (tile, chunk) and request it now
      if (++cn == nchunks) {
        cn = 0;
        tile_n = snake_tile(++jn);
      }
      if (tile_n < n_tiles) load(tile_n, cn, n0, n1, m0, m1);
#pragma unroll
      for (int h = 0; h < 2; ++h, ++it) {  // the chunk's two 64-K stages
        const int s = it % kQAStages;
        const long long tw = clock64();
        if (it >= kQAStages && !mbar_wait(&a_empty[s], ((it / kQAStages) - 1) & 1, p.st, 83)) {
          ok = false;
          break;
        }
        t_wait += clock64() - tw;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t r[16];
#pragma unroll
          for (int gl = 0; gl < 2; ++gl) {
            const int gg = 2 * h + gl;
            uint32_t sc0, sc1;
            if constexpr (kFp4) {
              sc0 = (fp4_lane_scales(s0[k], cl) >> (8 * gg)) & 0xffu;
              sc1 = (fp4_lane_scales(s1[k], cl) >> (8 * gg)) & 0xffu;
            } else {
              sc0 = ((gg < 2 ? s0[k].x : s0[k].y) >> (16 * (gg & 1))) & 0xffffu;
              sc1 = ((gg < 2 ? s1[k].x : s1[k].y) >> (16 * (gg & 1))) & 0xffffu;
            }
            uint32_t o0[4], o1[4];
            dq_word<kFp4>(word_at(w0[k], gg), sc0, o0);
            dq_word<kFp4>(word_at(w1[k], gg), sc1, o1);
#pragma unroll
            for (int jh = 0; jh < 2; ++jh) {
              const int i = 2 * gl + jh;  // repetition: columns 8i .. 8i+7 of the stage
              r[4 * i + 0] = o0[2 * jh];
              r[4 * i + 1] = o0[2 * jh + 1];
              r[4 * i + 2] = o1[2 * jh];
              r[4 * i + 3] = o1[2 * jh + 1];
            }
          }
          tmem_st16x256b_x4(tmem_base + ((uint32_t)(32 * q + 16 * k) << 16) + a_col(s, t), r);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&a_full[s]);
      }
      (void)c;
    }
    if (warp == kQWarpDq0 && lane == 0) {
      ptrace(p, 6, t_wait);
      ptrace(p, 7, clock64() - t_start);
    }
  } else if (warp == kQWarpMMA) {
    // ---------------- MMA issuer (one thread): D_t += A_t (TMEM) x B (shared memory)
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      long long t_d = 0, t_f = 0, n_sum = 0;
      const long long t_start = clock64();
      const uint64_t bdesc0 = umma_smem_desc(smem_u32(bst));
      for (int j = 0, tile = snake_tile(0); tile < n_tiles && ok; tile = snake_tile(++j), ++lt) {
        const TileInfo ti = tinfo(j, tile);
        const int N = (ti.nval + 15) & ~15;
        const uint32_t idesc = umma_idesc_f16(kPM, N);
        n_sum += N;
        const long long w0 = clock64();
        if (lt >= 1 && !mbar_wait(d_empty, (lt - 1) & 1, p.st, 84)) break;
        t_d += clock64() - w0;
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int sbq = it % kQBStages, saq = sbq;
          const long long w1 = clock64();
          if (!mbar_wait(&b_full[sbq], (it / kQBStages) & 1, p.st, 85)) {
            ok = false;
            break;
          }
          t_f += clock64() - w1;
          tc_fence_after();
          // stage sbq's descriptor is the first stage's plus its offset in 16-byte units; a 16-K
          // step is 32 bytes further, +2 in the address field
          const uint64_t bdesc = bdesc0 + (uint64_t)(sbq * (kQBBytes >> 4));
          const uint32_t acol0 = tmem_base + a_col(saq, 0), acol1 = tmem_base + a_col(saq, 1);
#pragma unroll
          for (int ks = 0; ks < kPK / 16; ++ks) {
            const uint32_t acc = (kb > 0 || ks > 0) ? 1u : 0u;
            umma_f16_ta(tmem_base, acol0 + (uint32_t)(8 * ks), bdesc + (uint64_t)(2 * ks), idesc, acc);
            umma_f16_ta(tmem_base + 128u, acol1 + (uint32_t)(8 * ks), bdesc + (uint64_t)(2 * ks), idesc, acc);
          }
          umma_commit(&b_empty[sbq]);  // B and A stages are free once these MMAs have read them
        }
        if (!ok) break;
        umma_commit(d_full);
      }
      umma_commit(drain);  // every MMA issued has finished before TMEM is released
      mbar_wait(drain, 0, p.st, 87);
      ptrace(p, 2, t_d);
      ptrace(p, 3, clock64() - t_start);
      ptrace(p, 4, t_f);
      ptrace(p, 11, lt);
      ptrace(p, 12, n_sum);
    }
  } else if (warp >= kQWarpEpi0) {
    // ---------------- epilogue: thread = one TMEM lane = weight row 32q + lane of both M tiles;
    // columns = the tile's routed rows
    const int q = warp & 3, row = 32 * q + lane;
    int lt = 0;
    bool dead = false;
    long long t_wait = 0;
    const long long t_start = clock64();
    for (int j = 0, tile = snake_tile(0); tile < n_tiles; tile = snake_tile(++j), ++lt) {
      const long long w0 = clock64();
      const bool got = !dead && __all_sync(0xffffffffu, mbar_wait(d_full, lt & 1, p.st, 88));
      t_wait += clock64() - w0;
      dead = !got;
      if (dead) break;
      tc_fence_after();
      const TileInfo ti = tinfo(j, tile);
      const float ta = kFp4 ? p.tsa[ti.e] : 1.f, tb = (kFp4 && p.mode == 1) ? p.tsb[ti.e] : 1.f;
      const uint32_t tq = tmem_base + ((uint32_t)(32 * q) << 16);
      // The warp copies its 32 rows of both accumulators into shared memory, already
      // turned around (one routed row's 32 values contiguous) and converted, and releases
      // the accumulators at once; the stores to global memory (16 bytes each) then run
      // under the next tile's MMAs.  Staging per warp: [M tile][routed row][32 values].
      const bool f32out = p.mode == 2 && p.y16 == nullptr;
      unsigned char* stg = epi_stage + (size_t)q * kQStageWarp;
      const int pos = (p.mode == 1) ? kperm(row) - 32 * q : lane;  // this thread's column in the 32
      for (int n0 = 0; n0 < ti.nval; n0 += 16) {
        uint32_t d0[16], d1[16];
        tmem_ld16(tq + (uint32_t)n0, d0);
        tmem_ld16(tq + (uint32_t)(128 + n0), d1);
        tmem_ld_wait();
        if (p.mode == 1) {  // h = silu(gate) * up of feature f, in the K order GEMM 2 reads
          __half* hs = reinterpret_cast<__half*>(stg);
          bool over = false;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float h = silu_mul_fast(__uint_as_float(d0[i]) * ta, __uint_as_float(d1[i]) * tb);
            over |= !(fabsf(h) < kF16Overflow);
            hs[(n0 + i) * 32 + pos] = __float2half_rn(h);
          }
          if (over) record_status(p.st, kStatusCheck, 90, ti.p0 + n0);
        } else if (!f32out) {
          __half* ys = reinterpret_cast<__half*>(stg);
          bool over = false;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float y0 = __uint_as_float(d0[i]) * ta, y1 = __uint_as_float(d1[i]) * ta;
            over |= !(fabsf(y0) < kF16Overflow && fabsf(y1) < kF16Overflow);
            ys[(n0 + i) * 32 + pos] = __float2half_rn(y0);
            ys[(128 + n0 + i) * 32 + pos] = __float2half_rn(y1);
          }
          if (over) record_status(p.st, kStatusCheck, 91, ti.p0 + n0);
        } else {
          float* ys = reinterpret_cast<float*>(stg);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            ys[(n0 + i) * 32 + pos] = __uint_as_float(d0[i]) * ta;
            ys[(128 + n0 + i) * 32 + pos] = __uint_as_float(d1[i]) * ta;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(d_empty);  // the MMAs of the next tile may overwrite D now
      if (p.mode == 1) {  // h rows: 32 features (64 bytes, 4 x 16) per routed row
        const __half* hs = reinterpret_cast<const __half*>(stg);
        const int f0 = ti.f * 128 + 32 * q;
        for (int v = lane; v < ti.nval * 4; v += 32) {
          const int r = v >> 2, c16 = v & 3;
          *reinterpret_cast<uint4*>(p.hout + (size_t)(ti.p0 + r) * p.I + f0 + 8 * c16) =
              *reinterpret_cast<const uint4*>(hs + r * 32 + 8 * c16);
        }
      } else {  // y rows: W_down rows f*256 + 32q + lane (M tile 0) and + 128 (M tile 1)
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
          const int c0 = ti.f * kPN + 128 * t2 + 32 * q;
          if (!f32out) {  // 32 columns (64 bytes, 4 x 16) per routed row
            const __half* ys = reinterpret_cast<const __half*>(stg) + 128 * 32 * t2;
            for (int v = lane; v < ti.nval * 4; v += 32) {
              const int r = v >> 2, c16 = v & 3;
              *reinterpret_cast<uint4*>(p.y16 + (size_t)(ti.p0 + r) * p.d + c0 + 8 * c16) =
                  *reinterpret_cast<const uint4*>(ys + r * 32 + 8 * c16);
            }
          } else {  // fp32: 128 bytes (8 x 16) per routed row
            const float* ys = reinterpret_cast<const float*>(stg) + 128 * 32 * t2;
            for (int v = lane; v < ti.nval * 8; v += 32) {
              const int r = v >> 3, c16 = v & 7;
              *reinterpret_cast<uint4*>(p.yout + (size_t)(ti.p0 + r) * p.d + c0 + 4 * c16) =
                  *reinterpret_cast<const uint4*>(ys + r * 32 + 4 * c16);
            }
          }
        }
      }
      __syncwarp();  // the staging is read before the next tile's copy overwrites it
    }
    if (warp == kQWarpEpi0 && lane == 0) {
      ptrace(p, 9, t_wait);
      ptrace(p, 10, clock64() - t_start);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kQWarpMMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kQTmemCols) : "memory");
  }
}

// pre[e] = sum over e' < e of ceil(n_e' / 128) (pre[E] = the number of 128-row expert
// blocks), and list = those blocks ordered by width, widest first.  One CTA of 1024
// threads, one expert per thread (E <= 1024).
__global__ void __launch_bounds__(1024) block_list_kernel(const int32_t* __restrict__ offsets, int E,
                                                          int32_t* __restrict__ pre, int32_t* __restrict__ list) {
  pdl_enter();
  __shared__ int scan[1024];
  __shared__ int cnt[17], fill[17];
  const int e = threadIdx.x;
  const int n = e < E ? offsets[e + 1] - offsets[e] : 0;
  const int nb = (n + kRowsPerBlock - 1) / kRowsPerBlock;
  scan[e] = nb;
  if (e < 17) cnt[e] = fill[e] = 0;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan
    const int v = e >= o ? scan[e - o] : 0;
    __syncthreads();
    scan[e] += v;
    __syncthreads();
  }
  const int first = scan[e] - nb;
  if (e < E) pre[e] = first;
  if (e == 1023) pre[E] = scan[1023];
  // bucket 0 = 256 rows wide, bucket 15 = 16 rows wide (blocks are at most kRowsPerBlock wide)
  for (int j = 0; j < nb; ++j) {
    const int w = min(kRowsPerBlock, n - j * kRowsPerBlock);
    atomicAdd(&cnt[16 - (w + 15) / 16], 1);
  }
  __syncthreads();
  if (e == 0) {
    int run = 0;
    for (int b = 0; b < 16; ++b) {
      const int c = cnt[b];
      cnt[b] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int j = 0; j < nb; ++j) {
    const int w = min(kRowsPerBlock, n - j * kRowsPerBlock);
    const int b = 16 - (w + 15) / 16;
    list[cnt[b] + atomicAdd(&fill[b], 1)] = first + j;
  }
}

// The same gather with every 32-element group of a row in the K order of the weights
// in tensor memory (kperm): the octet 8c .. 8c+7 of a group lands as two runs of four,
// at 4c and at 4c + 16.
__global__ void gather_f16_perm_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_rows,
                                       int R, int k, int d, __half* __restrict__ xs) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < R; pos += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(sorted_rows[pos] / k) * d);
    uint2* dst = reinterpret_cast<uint2*>(xs + (size_t)pos * d);  // 4 fp16 per uint2
    for (int i = lane; i < d / 8; i += 32) {
      const uint4 v = src[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __half2 h2 = __floats2half2_rn(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
        o[q] = *reinterpret_cast<uint32_t*>(&h2);
      }
      const int grp = i >> 2, c = i & 3;  // 32-element group, octet inside it
      dst[grp * 8 + c] = make_uint2(o[0], o[1]);
      dst[grp * 8 + c + 4] = make_uint2(o[2], o[3]);
    }
  }
}

int sm_count_prefill() {
  static int cnt[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (cnt[dev] == 0) cudaDeviceGetAttribute(&cnt[dev], cudaDevAttrMultiProcessorCount, dev);
  return cnt[dev] > 0 ? cnt[dev] : 148;
}

}  // namespace

bool prefill_eligible(int d, int I) { return d % 256 == 0 && I % 128 == 0 && d >= 256 && I >= 128; }

cudaError_t launch_prefill_ffn(const FfnArgs& a, int32_t* nb_prefix, __half* xs, __half* y16, cudaStream_t s) {
  const int R = a.T * a.k;
  if (R == 0) return cudaSuccess;
  if (!prefill_eligible(a.d, a.I)) return cudaErrorNotSupported;
  PrefillArgs p1 = {};
  cudaError_t err = encode_rows_map(&p1.tmap_a, xs, R, a.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kPK, kBoxRows);
  if (err != cudaSuccess) return err;
  PrefillArgs p2 = {};
  err = encode_rows_map(&p2.tmap_a, a.h_hi, R, a.I, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kPK, kBoxRows);
  if (err != cudaSuccess) return err;
  int32_t* pair_list = nb_prefix + a.E + 1;  // [R/128 + E] entries after the prefix
  if (cudaError_t e_ = launch_pdl(block_list_kernel, dim3(1), dim3(1024), 0, s, a.offsets, a.E, nb_prefix,
                                  pair_list)) return e_;
  const int gw = (R + 7) / 8;  // blocks of 8 warps
  if (cudaError_t e_ = launch_pdl(gather_f16_perm_kernel, dim3(gw < 148 * 8 ? gw : 148 * 8), dim3(256), 0, s, a.x,
                                  a.sorted_rows, R, a.k, a.d, xs)) return e_;
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const bool fp4 = a.gate_ts != nullptr;
  static int attr1[64] = {}, attr_fp4[64] = {};
  if ((err = fp4 ? ensure_smem_attr(prefill_wa_kernel<true>, kQSmem, attr_fp4)
                 : ensure_smem_attr(prefill_wa_kernel<false>, kQSmem, attr1)) != cudaSuccess)
    return err;
  auto kern = fp4 ? prefill_wa_kernel<true> : prefill_wa_kernel<false>;
  const int G = sm_count_prefill();
  // upper bound on the 128-row expert blocks, for the grid size
  const long blocks = (long)R / kRowsPerBlock + (R < a.E ? R : a.E) + 1;
  const size_t need = (size_t)2 * G * 16 * sizeof(unsigned long long);
  unsigned long long* tr = (g_trace_buf && g_trace_bytes >= need) ? static_cast<unsigned long long*>(g_trace_buf) : nullptr;

  p1.mode = 1;
  p1.T = a.T;
  p1.d = a.d;
  p1.I = a.I;
  p1.E = a.E;
  p1.k = a.k;
  p1.Kdim = a.d;
  p1.FB = a.I / 128;
  p1.wa = a.gate;
  p1.wb = a.up;
  p1.tsa = a.gate_ts;
  p1.tsb = a.up_ts;
  p1.wrows = a.I;
  p1.offsets = a.offsets;
  p1.nb_prefix = nb_prefix;
  p1.pair_list = pair_list;
  p1.hout = a.h_hi;  // fp16 h, [R, I]
  p1.st = a.st;
  p1.trace = tr;
  const long g1 = blocks * p1.FB;
  if (cudaError_t e_ = launch_pdl(kern, dim3((int)(g1 < G ? g1 : G)), dim3(kQThreads), kQSmem, s, p1)) return e_;
  if ((err = cudaGetLastError()) != cudaSuccess) return err;

  p2.mode = 2;
  p2.T = a.T;
  p2.d = a.d;
  p2.I = a.I;
  p2.E = a.E;
  p2.k = a.k;
  p2.Kdim = a.I;
  p2.FB = a.d / kPN;
  p2.wa = a.down;
  p2.wb = nullptr;
  p2.tsa = a.down_ts;
  p2.tsb = nullptr;
  p2.wrows = a.d;
  p2.offsets = a.offsets;
  p2.nb_prefix = nb_prefix;
  p2.pair_list = pair_list;
  p2.hout = nullptr;
  p2.yout = a.y_rows;
  p2.y16 = y16;
  p2.st = a.st;
  p2.trace = tr ? tr + (size_t)G * 16 : nullptr;
  const long g2 = blocks * p2.FB;
  if (cudaError_t e_ = launch_pdl(kern, dim3((int)(g2 < G ? g2 : G)), dim3(kQThreads), kQSmem, s, p2)) return e_;
  return cudaGetLastError();
}

}  // namespace bitmoe
