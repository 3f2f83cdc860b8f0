// Token -> expert grouping: a stable counting sort of the R = T*k routed rows.
//
// Row r = t*k + j goes to position offsets[e] + (number of rows r' < r with the
// same expert e), so the result is unique and matches the plain definition
// (experts ascending, rows ascending inside an expert).  The rank inside a
// chunk of 1024 rows comes from warp match masks plus per-warp counts, never
// from atomics, so it does not depend on scheduling.
//
// "Flint 40B : Best Mid Sized LLM", transcript 06:11 (mixture-of-experts
// routing kernels); "Recursive abre o Flint ...", section "O papel da
// quantizacao e dos kernels no lancamento" (operacoes MoE).
#include "kernels.h"

namespace bitmoe {
namespace {

constexpr int kPermThreads = 1024;

// Exclusive scan over the block (1024 threads) of one int per thread.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = warp_tot[lane];
    int winc = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, winc, off);
      if (lane >= off) winc += o;
    }
    warp_tot[lane] = winc - wv;
    if (lane == 31) *total = winc;
  }
  __syncthreads();
  const int r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Places one chunk of up to 1024 rows [base, base + 1024) given cursor[e] =
// first free position of expert e for this chunk; advances cursor.  cnt is a
// [32][E] uint16 scratch in shared memory.
__device__ void place_chunk(const int32_t* __restrict__ ids, int R, int E, int base, int* cursor, uint16_t* cnt,
                            int32_t* __restrict__ sorted_rows, int32_t* __restrict__ inv, DevStatus* st) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < 32 * E; i += kPermThreads) cnt[i] = 0;
  __syncthreads();
  const int r = base + tid;
  int e = -1;
  if (r < R) {
    e = ids[r];
    if (e < 0 || e >= E) {
      record_status(st, kStatusCheck, 3, r);
      inv[r] = -1;
      e = -1;
    }
  }
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const bool leader = (__ffs(peers) - 1) == lane;
  if (e >= 0 && leader) cnt[warp * E + e] = (uint16_t)__popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += kPermThreads) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt[w * E + x];
      cnt[w * E + x] = (uint16_t)run;
      run += c;
    }
    // stash this chunk's total for expert x in the (now unused) top of run
    cursor[E + x] = run;
  }
  __syncthreads();
  if (e >= 0) {
    const int pos = cursor[e] + cnt[warp * E + e] + rank;
    sorted_rows[pos] = r;
    inv[r] = pos;
  }
  __syncthreads();
  for (int x = tid; x < E; x += kPermThreads) cursor[x] += cursor[E + x];
  __syncthreads();
}

// One CTA does everything: histogram, offsets, token-block prefix, placement.
__global__ void __launch_bounds__(kPermThreads) permute_single_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                                      int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ sorted_rows,
                                                                      int32_t* __restrict__ inv,
                                                                      int32_t* __restrict__ blk_prefix,
                                                                      DevStatus* st) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  int* cursor = reinterpret_cast<int*>(smem);           // [2E]
  int* hist = cursor + 2 * E;                           // [E]
  int* warp_tot = hist + E;                             // [32] + total
  uint16_t* cnt = reinterpret_cast<uint16_t*>(warp_tot + 34);  // [32][E]
  const int tid = threadIdx.x;
  for (int x = tid; x < E; x += kPermThreads) hist[x] = 0;
  __syncthreads();
  for (int r = tid; r < R; r += kPermThreads) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  // E <= 1024: one expert per thread
  const int c = tid < E ? hist[tid] : 0;
  const int off = block_exclusive_scan(c, warp_tot, warp_tot + 32);
  if (tid < E) {
    offsets[tid] = off;
    cursor[tid] = off;
  }
  if (tid == 0) offsets[E] = warp_tot[32];
  const int nb = tid < E ? ceil_div(c, kTokBlock) : 0;
  const int bp = block_exclusive_scan(nb, warp_tot, warp_tot + 32);
  if (tid < E) blk_prefix[tid] = bp;
  if (tid == 0) blk_prefix[E] = warp_tot[32];
  __syncthreads();
  for (int base = 0; base < R; base += kPermThreads)
    place_chunk(ids, R, E, base, cursor, cnt, sorted_rows, inv, st);
}

// Multi-CTA path: per-chunk histograms, one scan CTA, per-chunk placement.
__global__ void __launch_bounds__(kPermThreads) permute_hist_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                                    int32_t* __restrict__ chunk_hist) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  int* hist = reinterpret_cast<int*>(smem);
  const int tid = threadIdx.x;
  for (int x = tid; x < E; x += kPermThreads) hist[x] = 0;
  __syncthreads();
  const int r = blockIdx.x * kPermChunk + tid;
  if (r < R) {
    const int e = ids[r];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int x = tid; x < E; x += kPermThreads) chunk_hist[(size_t)blockIdx.x * E + x] = hist[x];
}

__global__ void __launch_bounds__(kPermThreads) permute_scan_kernel(int32_t* __restrict__ chunk_hist, int nchunks,
                                                                    int E, int32_t* __restrict__ offsets,
                                                                    int32_t* __restrict__ blk_prefix) {
  pdl_enter();
  __shared__ int warp_tot[34];
  const int tid = threadIdx.x;
  int tot = 0;
  if (tid < E)
    for (int c = 0; c < nchunks; ++c) tot += chunk_hist[(size_t)c * E + tid];
  const int off = block_exclusive_scan(tot, warp_tot, warp_tot + 32);
  if (tid < E) {
    offsets[tid] = off;
    int run = off;
    for (int c = 0; c < nchunks; ++c) {  // chunk_hist becomes the chunk's first free position
      const int h = chunk_hist[(size_t)c * E + tid];
      chunk_hist[(size_t)c * E + tid] = run;
      run += h;
    }
  }
  if (tid == 0) offsets[E] = warp_tot[32];
  const int nb = tid < E ? ceil_div(tot, kTokBlock) : 0;
  const int bp = block_exclusive_scan(nb, warp_tot, warp_tot + 32);
  if (tid < E) blk_prefix[tid] = bp;
  if (tid == 0) blk_prefix[E] = warp_tot[32];
}

__global__ void __launch_bounds__(kPermThreads) permute_place_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                                     const int32_t* __restrict__ chunk_base,
                                                                     int32_t* __restrict__ sorted_rows,
                                                                     int32_t* __restrict__ inv, DevStatus* st) {
  pdl_enter();
  extern __shared__ __align__(16) unsigned char smem[];
  int* cursor = reinterpret_cast<int*>(smem);                 // [2E]
  uint16_t* cnt = reinterpret_cast<uint16_t*>(cursor + 2 * E);  // [32][E]
  for (int x = threadIdx.x; x < E; x += kPermThreads) cursor[x] = chunk_base[(size_t)blockIdx.x * E + x];
  __syncthreads();
  place_chunk(ids, R, E, blockIdx.x * kPermChunk, cursor, cnt, sorted_rows, inv, st);
}

__global__ void blk_prefix_kernel(const int32_t* __restrict__ offsets, int E, int32_t* __restrict__ blk_prefix) {
  pdl_enter();
  __shared__ int warp_tot[34];
  const int tid = threadIdx.x;
  const int nb = tid < E ? ceil_div(offsets[tid + 1] - offsets[tid], kTokBlock) : 0;
  const int bp = block_exclusive_scan(nb, warp_tot, warp_tot + 32);
  if (tid < E) blk_prefix[tid] = bp;
  if (tid == 0) blk_prefix[E] = warp_tot[32];
}

constexpr int kSingleMaxRows = 4096;

size_t single_smem(int E) { return (size_t)(3 * E + 34) * 4 + (size_t)32 * E * 2; }
size_t place_smem(int E) { return (size_t)2 * E * 4 + (size_t)32 * E * 2; }

}  // namespace

size_t permute_scratch_bytes(int64_t R, int E) {
  if (R <= kSingleMaxRows) return 0;
  return (size_t)ceil_div<int64_t>(R, kPermChunk) * E * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* ids, int R, int E, int32_t* offsets, int32_t* sorted_rows, int32_t* inv,
                           int32_t* blk_prefix, void* scratch, DevStatus* st, cudaStream_t s) {
  if (R <= kSingleMaxRows) {
    const size_t sm = single_smem(E);
    static int attr_set[64] = {};
    cudaError_t err = ensure_smem_attr(permute_single_kernel, sm, attr_set);
    if (err != cudaSuccess) return err;
    if (cudaError_t e_ = launch_pdl(permute_single_kernel, dim3(1), dim3(kPermThreads), sm, s, ids, R, E, offsets,
                                    sorted_rows, inv, blk_prefix, st)) return e_;
    return cudaGetLastError();
  }
  const int nchunks = ceil_div(R, kPermChunk);
  int32_t* chunk_hist = static_cast<int32_t*>(scratch);
  if (cudaError_t e_ = launch_pdl(permute_hist_kernel, dim3(nchunks), dim3(kPermThreads), (size_t)E * 4, s, ids, R, E,
                                  chunk_hist)) return e_;
  if (cudaError_t e_ = launch_pdl(permute_scan_kernel, dim3(1), dim3(kPermThreads), 0, s, chunk_hist, nchunks, E,
                                  offsets, blk_prefix)) return e_;
  const size_t sm = place_smem(E);
  static int attr_set[64] = {};
  cudaError_t err = ensure_smem_attr(permute_place_kernel, sm, attr_set);
  if (err != cudaSuccess) return err;
  if (cudaError_t e_ = launch_pdl(permute_place_kernel, dim3(nchunks), dim3(kPermThreads), sm, s, ids, R, E, chunk_hist,
                                  sorted_rows, inv, st)) return e_;
  return cudaGetLastError();
}

cudaError_t launch_blk_prefix(const int32_t* offsets, int E, int32_t* blk_prefix, cudaStream_t s) {
  if (cudaError_t e_ = launch_pdl(blk_prefix_kernel, dim3(1), dim3(kPermThreads), 0, s, offsets, E,
                                  blk_prefix)) return e_;
  return cudaGetLastError();
}

}  // namespace bitmoe
