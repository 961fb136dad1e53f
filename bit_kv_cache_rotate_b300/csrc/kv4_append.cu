// kv4_append.cu -- quantise-on-append kernels.
//
// 4-bit path ("UltraQuant on AMD Instinct", section "What is UltraQuant"):
// one warp per (token, kv head, K|V) vector.  The Walsh-Hadamard rotation is
// an fp64 butterfly over warp shuffles: for bf16 inputs inside the exact
// domain every partial sum is exact, so the result equals the exact matrix
// product; it is then scaled by RN64(1/sqrt(D)) in fp64 and rounded once to
// fp32.  Group maxima are shuffle reductions over the lanes of a 32-channel
// group; the UE8M0 exponent is read off the fp32 exponent field; codes come
// from the hardware RNE/satfinite E2M1 conversion.
//
// FP8 comparator: same warp mapping, E4M3 of fp32(x * inv_scale[h]).
#include "kv4_common.cuh"

namespace kv4 {

template <int D>
__global__ void __launch_bounds__(256) append_fp4_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int num_tokens, int Hkv,
    const int32_t* __restrict__ slots, uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
    int num_pages, double inv_sqrt_d, int32_t* dev_error) {
  constexpr int E = D / 32;              // channels per lane
  constexpr int LANES_PER_GROUP = 32 / E;
  constexpr int CODE_BYTES = kPage * D / 2;
  constexpr int BLOCK = CODE_BYTES + kPage * D / 32;

  const int nvec = v ? 2 : 1;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (long long)num_tokens * Hkv * nvec) return;
  const int which = (int)(warp % nvec);
  const long long th = warp / nvec;
  const int h = (int)(th % Hkv);
  const long long tok = th / Hkv;

  const int slot = slots[tok];
  if (slot < 0) return;
  const int page = slot / kPage, off = slot % kPage;
  if (page >= num_pages) {
    if (lane == 0) flag_error(dev_error, KV4_DEVERR_SLOT);
    return;
  }

  // Load E consecutive bf16 channels.
  const uint16_t* src = (which ? v : k) + ((size_t)tok * Hkv + h) * D + lane * E;
  double x[E];
  if constexpr (E == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    x[0] = (double)bf16_bits_to_float(w & 0xFFFFu);
    x[1] = (double)bf16_bits_to_float(w >> 16);
  } else {
#pragma unroll
    for (int i = 0; i < E; i += 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(src + i);
      x[i + 0] = (double)bf16_bits_to_float(w.x & 0xFFFFu);
      x[i + 1] = (double)bf16_bits_to_float(w.x >> 16);
      x[i + 2] = (double)bf16_bits_to_float(w.y & 0xFFFFu);
      x[i + 3] = (double)bf16_bits_to_float(w.y >> 16);
    }
  }

  fwht_warp<E, double>(x);

  float y[E];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    // + 0.0 turns an exact zero sum into +0: a butterfly over negative zeros
    // yields -0 where the exact matrix product has a plain 0 (code 0, not 8).
    y[i] = (float)(x[i] * inv_sqrt_d + 0.0);
    amax = fmaxf(amax, fabsf(y[i]));
  }
#pragma unroll
  for (int d = 1; d < LANES_PER_GROUP; d <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));

  // e = floor(log2 amax) - 2, clamped to [-127, 127]; subnormal or zero amax -> -127.
  const int ef = (int)(__float_as_uint(amax) >> 23);
  const int e = ef == 0 ? -127 : max(ef - 127 - 2, -127);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e, normal for e <= 126

  uint8_t* blk = (which ? v_cache : k_cache) + ((size_t)page * Hkv + h) * BLOCK;
  uint32_t byte[E / 2];
#pragma unroll
  for (int i = 0; i < E; i += 2) byte[i / 2] = f32x2_to_e2m1x2(y[i] * inv, y[i + 1] * inv);

  if (which == 0) {
    // K: 8-token x 32-channel tiles; the lane's E channels (E <= 16, aligned)
    // stay inside one tile row, E/2 consecutive bytes.
    uint8_t* dst = blk + k_code_offset(D, off, lane * E);
    if constexpr (E == 2) {
      dst[0] = (uint8_t)byte[0];
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(byte[0] | (byte[1] << 8));
    } else {
#pragma unroll
      for (int i = 0; i < E / 2; i += 4)
        *reinterpret_cast<uint32_t*>(dst + i) =
            byte[i] | (byte[i + 1] << 8) | (byte[i + 2] << 16) | (byte[i + 3] << 24);
    }
  } else {
    // V: channel-major codes; token `off` owns one nibble of byte (d, off/2),
    // the other nibble belongs to token off^1, which may be appended
    // concurrently -> clear and set the nibble with 32-bit atomics.
    const int shift = ((off >> 1) & 3) * 8 + (off & 1) * 4;
    const uint32_t clear = ~(0xFu << shift);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int d = lane * E + i;
      const uint32_t code = (byte[i / 2] >> ((i & 1) * 4)) & 0xFu;
      uint32_t* word = reinterpret_cast<uint32_t*>(blk + d * (kPage / 2) + ((off >> 1) & ~3));
      atomicAnd(word, clear);
      atomicOr(word, code << shift);
    }
  }
  if ((lane % LANES_PER_GROUP) == 0)
    blk[CODE_BYTES + off * (D / 32) + lane / LANES_PER_GROUP] = (uint8_t)(e + 127);
}

template <int D>
__global__ void __launch_bounds__(256) append_fp8_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int num_tokens, int Hkv,
    const int32_t* __restrict__ slots, const float* __restrict__ k_inv, const float* __restrict__ v_inv,
    uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache, int num_pages, int32_t* dev_error) {
  constexpr int E = D / 32;
  constexpr int BLOCK = kPage * D;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (long long)num_tokens * Hkv * 2) return;
  const int which = (int)(warp & 1);
  const long long th = warp >> 1;
  const int h = (int)(th % Hkv);
  const long long tok = th / Hkv;
  const int slot = slots[tok];
  if (slot < 0) return;
  const int page = slot / kPage, off = slot % kPage;
  if (page >= num_pages) {
    if (lane == 0) flag_error(dev_error, KV4_DEVERR_SLOT);
    return;
  }
  const uint16_t* src = (which ? v : k) + ((size_t)tok * Hkv + h) * D + lane * E;
  const float inv = which ? v_inv[h] : k_inv[h];
  uint8_t* blk = (which ? v_cache : k_cache) + ((size_t)page * Hkv + h) * BLOCK;
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src + i);
    const float a = bf16_bits_to_float(w & 0xFFFFu) * inv;
    const float b = bf16_bits_to_float(w >> 16) * inv;
    const uint32_t two = f32x2_to_e4m3x2(a, b);
    const int d = lane * E + i;
    if (which == 0) {
      *reinterpret_cast<uint16_t*>(blk + off * D + d) = (uint16_t)two;
    } else {
      blk[d * kPage + off] = (uint8_t)(two & 0xFFu);
      blk[(d + 1) * kPage + off] = (uint8_t)(two >> 8);
    }
  }
}

// ---------------------------------------------------------------- launchers
static inline unsigned blocks_for_warps(long long warps) {
  return (unsigned)((warps * 32 + 255) / 256);
}

cudaError_t launch_append_fp4(const void* k, const void* v, int n, int Hkv, int D,
                              const int32_t* slots, uint8_t* kc, uint8_t* vc, int num_pages,
                              double inv_sqrt_d, int32_t* err, cudaStream_t st) {
  const long long warps = (long long)n * Hkv * (v ? 2 : 1);
  if (warps == 0) return cudaSuccess;
  const dim3 grid(blocks_for_warps(warps)), block(256);
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  switch (D) {
    case 64: append_fp4_kernel<64><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kc, vc, num_pages, inv_sqrt_d, err); break;
    case 128: append_fp4_kernel<128><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kc, vc, num_pages, inv_sqrt_d, err); break;
    case 256: append_fp4_kernel<256><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kc, vc, num_pages, inv_sqrt_d, err); break;
    case 512: append_fp4_kernel<512><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kc, vc, num_pages, inv_sqrt_d, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_append_fp8(const void* k, const void* v, int n, int Hkv, int D,
                              const int32_t* slots, const float* kinv, const float* vinv,
                              uint8_t* kc, uint8_t* vc, int num_pages, int32_t* err,
                              cudaStream_t st) {
  const long long warps = (long long)n * Hkv * 2;
  if (warps == 0) return cudaSuccess;
  const dim3 grid(blocks_for_warps(warps)), block(256);
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  const uint16_t* vv = static_cast<const uint16_t*>(v);
  switch (D) {
    case 64: append_fp8_kernel<64><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kinv, vinv, kc, vc, num_pages, err); break;
    case 128: append_fp8_kernel<128><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kinv, vinv, kc, vc, num_pages, err); break;
    case 256: append_fp8_kernel<256><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kinv, vinv, kc, vc, num_pages, err); break;
    case 512: append_fp8_kernel<512><<<grid, block, 0, st>>>(kk, vv, n, Hkv, slots, kinv, vinv, kc, vc, num_pages, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kv4
