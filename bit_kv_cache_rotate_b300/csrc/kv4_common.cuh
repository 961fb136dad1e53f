// kv4_common.cuh -- device helpers shared by the libkv4 kernels (sm_103a).
//
// Nothing here is shared with the CPU oracle; the two agree only through
// their documented inputs and outputs.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "kv4.h"

namespace kv4 {

constexpr int kPage = 16;  // tokens per page (the only page size implemented)

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// 2^e as an fp32 value for a UE8M0 byte (e + 127).  Byte 0 (e = -127) is the
// subnormal 2^-127.
__device__ __forceinline__ float ue8m0_to_float(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// Exact fp32 value of an E2M1 code (sign | 2 exponent bits | 1 mantissa bit),
// built from the bit fields: magnitude index 0 -> 0, 1 -> 0.5 (subnormal),
// i >= 2 -> 2^(i/2 - 1) * (1 + (i&1)/2).
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
  const uint32_t mag = c & 7u;
  const uint32_t bits = mag >= 2u ? (((126u + (mag >> 1)) << 23) | ((mag & 1u) << 22))
                                  : (mag ? 0x3F000000u : 0u);
  return __uint_as_float(bits | ((c & 8u) << 28));
}

// Two fp32 values -> two E2M1 codes in one byte (lo in bits 3:0, hi in 7:4),
// round-to-nearest-even, saturating at +-6.  The sign bit of each input is
// forced into its code so that values rounding to zero keep their sign.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  out |= (__float_as_uint(lo) >> 28) & 0x8u;
  out |= (__float_as_uint(hi) >> 24) & 0x80u;
  return out;
}

// Two fp32 values -> two E4M3 bytes (lo in bits 7:0, hi in 15:8), RNE, satfinite.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
  return out;
}

// Two E4M3 bytes (lo in bits 7:0) -> two fp32 values (exact).
// Byte offset of (token t, channel d) in a K code plane: tiles of 8 tokens x
// 32 channels, 128 bytes each, tile (t/8, d/32) at ((t/8)*(D/32) + d/32)*128,
// token t%8 at +16*(t%8), channel d in byte (d%32)/2 (low nibble even).
__host__ __device__ __forceinline__ int k_code_offset(int D, int t, int d) {
  return ((t >> 3) * (D >> 5) + (d >> 5)) * 128 + (t & 7) * 16 + ((d & 31) >> 1);
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
  float2 r;
  asm("cvt.f32.f16 %0, %1;" : "=f"(r.x) : "h"((uint16_t)(h2 & 0xFFFFu)));
  asm("cvt.f32.f16 %0, %1;" : "=f"(r.y) : "h"((uint16_t)(h2 >> 16)));
  return r;
}

// In-register Walsh-Hadamard butterfly (unnormalised, Sylvester natural
// order) over D = 32*E values held by a full warp, lane l holding elements
// [l*E, l*E + E).  Result: x <- H_pm1 x.
template <int E, typename T>
__device__ __forceinline__ void fwht_warp(T (&x)[E]) {
#pragma unroll
  for (int s = 1; s < E; s <<= 1) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      if (!(i & s)) {
        const T a = x[i], b = x[i + s];
        x[i] = a + b;
        x[i + s] = a - b;
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const T o = __shfl_xor_sync(0xffffffffu, x[i], d);
      x[i] = upper ? (o - x[i]) : (x[i] + o);
    }
  }
}

// Raises a kernel's dynamic shared-memory limit on the current device, once
// per device (the attribute is per device); safe to call from several host
// threads (the call is idempotent).
template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

__device__ __forceinline__ void flag_error(int32_t* dev_error, int bit) {
  if (dev_error) atomicOr(dev_error, bit);
}

}  // namespace kv4
