// Device helpers shared by the bitmoe kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/bitmoe.h"

namespace bitmoe {

// ---------------------------------------------------------------- constants

constexpr int kGroup = 32;          // int4 scale group along the reduction dim
constexpr int kTileRows = 16;       // rows per packed tile (one mma M)
constexpr int kChunkK = 128;        // columns per packed chunk (four groups)
constexpr int kChunkQBytes = 1024;  // 16 rows x 128 cols x 4 bits
constexpr int kChunkSBytes = 128;   // 16 rows x 4 groups x fp16
constexpr int kChunkBytes = kChunkQBytes + kChunkSBytes;
constexpr int kTokBlock = 16;       // tokens per unit of the streaming FFN kernels
constexpr int kSmemRowPad = 64;     // bytes of padding per staged activation row (bank spread)
constexpr int kPermChunk = 1024;    // rows per permutation chunk
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;

// Device status word values (see bitmoe_get_device_status).
constexpr int kStatusTimeout = BITMOE_ERR_TIMEOUT;
constexpr int kStatusCheck = BITMOE_ERR_DEVICE_CHECK;

// fp16 range: a value of this magnitude or more rounds to infinity (round to nearest).
// The expert intermediates h that the projections carry in fp16 (hi + lo pairs on the
// exact paths, one fp16 on the grouped-GEMM path, which also keeps y in fp16) must stay
// below it; a larger one, or a NaN, records kStatusCheck instead of passing silently.
constexpr float kF16Overflow = 65520.0f;

// A bounded wait gives up after this long and records kStatusTimeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__host__ __device__ constexpr int64_t tile_bytes(int64_t K) { return (K / kChunkK) * kChunkBytes; }

// ---------------------------------------------------------------- status word

struct DevStatus {
  int code;        // first error code recorded (0 = none)
  int where;       // site id of the first error
  int detail;      // extra (e.g. offending index)
  int pad;
};

__device__ __forceinline__ void record_status(DevStatus* st, int code, int where, int detail) {
  if (st == nullptr) return;
  if (atomicCAS(&st->code, 0, code) == 0) {
    st->where = where;
    st->detail = detail;
  }
}

// ---------------------------------------------------------------- PTX: timers, smem, mbarrier, bulk copy

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false (and a recorded timeout) if it
// does not complete within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, DevStatus* st, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_status(st, kStatusTimeout, where, 0);
      return false;
    }
  }
  return true;
}

// Bulk copy global -> shared (TMA, non-tensor), completion counted on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 prefetch of a global range (bulk, no completion tracking).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
//
// Every kernel of the layer's multi-kernel paths is launched with programmatic
// stream serialization: it may be scheduled while the previous kernel on the stream
// drains, and its first statement waits (griddepcontrol.wait) until that kernel has
// completed and its writes are visible, then lets the next kernel be scheduled in
// turn.  Results are those of plain stream order; the launch gaps overlap.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mma.sync m16n8k16

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                        const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// ---------------------------------------------------------------- int4 -> 16-bit pairs
//
// A packed word holds the 8 nibbles one thread feeds to two k16 mma steps:
// pair p (p = 0..3) sits at bits [4p, 4p+4) (first element) and
// [16+4p, 20+4p) (second element).  Masking puts two nibbles in each 16-bit
// half; XOR with 8 turns the two's-complement nibble n into q + 8, and the
// fp16 exponent pattern of 1024 (whose spacing is 1) makes each half the
// float 1024 + q + 8.  Subtracting 1032 leaves q exactly.

// (a & b) ^ c in one LOP3 (truth table 0x6A for the operand order a, b, c).
// The compiler otherwise splits a mask-and-flip into two logic instructions;
// the constants stay in registers.
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// All four fp16 pairs of a word, p = 0..3, with one shift instead of three:
// an odd pair (nibbles at bits 4..7 of each half) is read in place as
// 1024 + 16 (q + 8), which fits fp16's 10-bit mantissa, and one fused
// multiply-add by 1/16 minus 72 leaves q (every step exact).  The f16x2
// constants are bit patterns held in registers (1032 = 0x6408, 1/16 = 0x2C00,
// -72 = 0xD480), so each step is a single instruction: per 8 weights one
// shift, four logic ops, two subtracts and two fused multiply-adds.
__device__ __forceinline__ void nib_pairs4_f16(uint32_t w, uint32_t (&o)[4]) {
  const uint32_t m_lo = 0x000F000Fu, m_hi = 0x00F000F0u, x_lo = 0x64086408u, x_hi = 0x64806480u;
  const uint32_t off = 0x64086408u, sixteenth = 0x2C002C00u, off_hi = 0xD480D480u;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t v = b ? (w >> 8) : w;
    const uint32_t te = and_xor(v, m_lo, x_lo);  // 1032 + q
    const uint32_t to = and_xor(v, m_hi, x_hi);  // 1024 + 16 (q + 8)
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o[2 * b]) : "r"(te), "r"(off));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(o[2 * b + 1]) : "r"(to), "r"(sixteenth), "r"(off_hi));
  }
}

// 2^s as a float, exactly, for |s| <= 126.
__device__ __forceinline__ float pow2i(int s) { return __int_as_float((s + 127) << 23); }

// Exponent s that puts a bf16 row's largest magnitude (bits m, sign cleared)
// in [2^14, 2^15): multiplying the row by 2^s makes every element an exact
// fp16 value (bf16 carries 8 significant bits, fp16 11; only elements below
// 2^-24 of the largest would round).  0 for an all-zero or subnormal-only row.
__device__ __forceinline__ int f16_row_exponent(uint32_t m) {
  const int ef = (int)(m >> 7);
  return (ef == 0) ? 0 : min(126, max(-126, 14 - (ef - 127)));
}

// ---------------------------------------------------------------- NVFP4

// NVFP4 weights: FP4 E2M1 codes, one FP8 E4M3 scale per 16 consecutive
// weights of a row, one fp32 scale per matrix (the "four-bit NVFP" builds of
// "Flint 40B : Best Mid Sized LLM", transcript 07:15).  The packed layout has
// the int4 layout's geometry: a 128-column chunk of a 16-row tile holds the
// 16 x 128 codes (1024 bytes, each 32-bit word the 8 codes of one lane's
// fragment, byte j the pair that fragment register j takes, low nibble first)
// and then 16 rows x 8 block scales (128 bytes).
constexpr int kFp4Block = 16;

// Block scale s (an E4M3 byte) as the fp16 pair (s, s), exactly (E4M3 is a
// subset of fp16).
__device__ __forceinline__ uint32_t e4m3_pair_f16(uint32_t byte) {
  uint32_t d;
  const uint16_t v = (uint16_t)(byte * 0x0101u);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}

// The eight E2M1 codes of a packed word as four fp16 pairs (hardware
// conversion), each multiplied by the block scale pair sc.  Exact: a code has
// at most 2 significant bits and a scale 4, so every product is an fp16 value
// (|product| between 2^-10 and 2688, never below fp16's subnormal step).
__device__ __forceinline__ void e2m1x8_f16_scaled(uint32_t w, uint32_t sc, uint32_t (&o)[4]) {
  uint32_t c0, c1, c2, c3;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(c0), "=r"(c1), "=r"(c2), "=r"(c3)
      : "r"(w));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[0]) : "r"(c0), "r"(sc));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[1]) : "r"(c1), "r"(sc));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[2]) : "r"(c2), "r"(sc));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[3]) : "r"(c3), "r"(sc));
}

// The four block-scale bytes a lane needs from one row's 8 scales of a chunk
// (lane quarter c covers columns 8c .. 8c+7 of every 32-column group, which
// lie in block 2 gg + c / 2 of the chunk for group gg): byte gg of the result
// is the scale of group gg.
__device__ __forceinline__ uint32_t fp4_lane_scales(uint2 s8, int c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(s8.x), "r"(s8.y), "r"((c >> 1) ? 0x7531u : 0x6420u));
  return d;
}

// D = A B (no accumulator input) for one m16n8k16 fp16 step.
__device__ __forceinline__ void mma_f16_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// ---------------------------------------------------------------- misc

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float silu_mul(float a, float u) { return a / (1.0f + expf(-a)) * u; }

// The same with the hardware exponential and an approximate division, for the
// paths whose h is rounded to fp16 right after (a few fp32 ulps of difference).
__device__ __forceinline__ float silu_mul_fast(float a, float u) { return __fdividef(a * u, 1.0f + __expf(-a)); }

// Order-preserving map of a float onto uint32 (for packed argmax keys).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sets a kernel's dynamic shared-memory limit once per device (the call is
// host-side state only, so later launches -- including ones being captured
// into a CUDA graph -- issue nothing but the launch itself).
template <typename F>
inline cudaError_t ensure_smem_attr(F* kernel, size_t bytes, int* max_set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_set[dev] >= (int)bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) max_set[dev] = (int)bytes;
  return e;
}

// Launch with programmatic stream serialization (the kernel must start with pdl_enter()).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename T>
__host__ __device__ constexpr T ceil_div(T a, T b) {
  return (a + b - 1) / b;
}

}  // namespace bitmoe
