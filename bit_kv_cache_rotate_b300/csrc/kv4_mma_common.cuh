// kv4_mma_common.cuh -- device helpers shared by the tensor-core decode
// kernels: mbarrier waits, 1-D bulk copies, the f16 warp MMA, operand
// conversions and the f16 hi/lo split of softmax weights.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kv4 {
namespace mma {

constexpr int kSpinLimit = 1 << 16;     // try_wait rounds, each suspending up to kSuspendNs
constexpr uint32_t kSuspendNs = 20000;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Bounded wait for the phase with the given parity; false on timeout.  The
// suspend hint lets a waiting warp sleep instead of spinning on issue slots.
// `limit` is the number of tries (a limit of 0 gives up at once: the
// KV4_DIAG_EXPIRE_FIRST_WAIT test control).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int limit = kSpinLimit) {
  const uint32_t addr = smem_u32(bar);
  for (int i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA on bf16 operands: bf16 has the exponent range of fp32, so
// operands that span more binades than f16 holds keep their value.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// f16x2 -> bf16x2 through fp32; exact for the E2M1 code values (two
// significant bits).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  uint32_t d;
  asm("{\n\t.reg .b16 l, u;\n\t.reg .f32 fl, fu;\n\tmov.b32 {l, u}, %1;\n\t"
      "cvt.f32.f16 fl, l;\n\tcvt.f32.f16 fu, u;\n\tcvt.rn.bf16x2.f32 %0, fu, fl;\n\t}"
      : "=r"(d)
      : "r"(h));
  return d;
}

// A pair x (fp32) as bf16 hi parts and the bf16-rounded remainders: about 16
// significant bits of x over the whole fp32 exponent range.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(x0, x1);
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
  lo = pack_bf16x2(x0 - h0, x1 - h1);
}

// 2^(byte - e) as fp32 for a UE8M0 byte and a reference exponent byte e, the
// exponent field clamped to [0, 254] (0 gives 0.0: a factor below 2^-126).
__device__ __forceinline__ float pow2_diff(uint32_t byte, int e) {
  const int ex = min(254, max(0, 127 + (int)byte - e));
  return __uint_as_float((uint32_t)ex << 23);
}

// Nonzero when some byte of x is zero.
__device__ __forceinline__ uint32_t has_zero_byte(uint32_t x) {
  return (x - 0x01010101u) & ~x & 0x80808080u;
}

// One byte of two E2M1 codes -> f16x2 (low nibble -> low half), exact.  The
// word is split into .b8 registers so the conversion reads the byte lane in
// place (a shift per byte otherwise); `byte` is a compile-time constant.
#define KV4_CVT_BYTE(B)                                                              \
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\t"         \
      "cvt.rn.f16x2.e2m1x2 %0, b" #B ";\n\t}"                                      \
      : "=r"(out)                                                                    \
      : "r"(word))
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t word, int byte) {
  uint32_t out;
  switch (byte) {
    case 0: KV4_CVT_BYTE(0); break;
    case 1: KV4_CVT_BYTE(1); break;
    case 2: KV4_CVT_BYTE(2); break;
    default: KV4_CVT_BYTE(3); break;
  }
  return out;
}
#undef KV4_CVT_BYTE

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Split a pair x >= 0 into f16-exact hi parts (11 significant bits, Veltkamp)
// and the remainders.  Packed fp32x2 ops with explicit rounding: no step can
// be contracted into an FMA, which would break the split.
__device__ __forceinline__ void split_hi_lo2(float2 x, float2& hi, float2& lo) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const float2 c = __fmul2_rn(x, make_float2(8193.0f, 8193.0f));
  const float2 t = __ffma2_rn(x, m1, c);   // c - x
  hi = __ffma2_rn(t, m1, c);               // c - (c - x)
  lo = __ffma2_rn(hi, m1, x);              // x - hi (exact)
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two E4M3 bytes (half `half` of the word) -> f16x2, exact (E4M3 is a subset
// of f16).  As above, the word is split so the conversion reads the lane in
// place; `half` is a compile-time constant.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t word, int half) {
  uint32_t out;
  if (half == 0)
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h0;\n\t}"
        : "=r"(out) : "r"(word));
  else
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h1;\n\t}"
        : "=r"(out) : "r"(word));
  return out;
}

// Sequence served by grid row z.  CTAs start roughly in launch order (x
// fastest, then y, then z), and with ragged contexts a sequence's CTAs take
// time in proportion to its length; so row z takes the z-th longest sequence
// (ties by index), the long sequences start in the first wave and the short
// ones fill the tail of the last.  Equal lengths give z itself.  Each warp
// ranks the lengths on its own (lane i holds sequences i and i + 32): no
// shared memory, no block barrier; every lane of a full warp must call it.
// Batches above kOrderMaxBatch keep the launch order.
constexpr int kOrderMaxBatch = 64;

__device__ __forceinline__ int longest_first(const int32_t* __restrict__ lens, int B, int z) {
  if (B > kOrderMaxBatch) return z;
  const int lane = threadIdx.x & 31;
  const int i1 = lane + 32;
  const int L0 = lane < B ? lens[lane] : 0;
  const int L1 = i1 < B ? lens[i1] : 0;
  int r0 = 0, r1 = 0;
  for (int j = 0; j < B; ++j) {
    const int Lj = __shfl_sync(0xffffffffu, j < 32 ? L0 : L1, j & 31);
    r0 += (Lj > L0) | ((Lj == L0) & (j < lane));
    r1 += (Lj > L1) | ((Lj == L1) & (j < i1));
  }
  const uint32_t m0 = __ballot_sync(0xffffffffu, lane < B && r0 == z);
  const uint32_t m1 = __ballot_sync(0xffffffffu, i1 < B && r1 == z);
  return m0 ? __ffs(m0) - 1 : (m1 ? 31 + __ffs(m1) : z);
}

}  // namespace mma
}  // namespace kv4
