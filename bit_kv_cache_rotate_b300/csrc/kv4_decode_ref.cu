// kv4_decode_ref.cu -- generic split-K paged decode attention on CUDA cores,
// plus the log-sum-exp split combine.
//
// This path covers every supported shape (head_dim 64..512, any GQA group,
// T-position causal verify, latent K = V) for both the 4-bit cache and the
// FP8 comparator.  The tensor-core path for the headline shapes lives in
// kv4_decode_mma.cu; this one is the general fallback.
//
// One CTA per (split, kv head, sequence).  Per page of 16 tokens the CTA
// stages the K and V blocks in shared memory, decodes the codes to fp32
// (code value from its bit fields times 2^e from the UE8M0 byte: exact),
// computes the R = T*G scores per token, updates an online softmax per query
// row, and accumulates P.V.  It writes the split's normalised partial output
// and log-sum-exp.  q is rotated by the same Walsh-Hadamard transform as the
// cache ("What is UltraQuant"), so scores equal those of the unrotated
// vectors; the output stays in the rotated space until the combine.
#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_ref_unit.cuh"

namespace kv4 {



template <int D, bool FP8, int RMAX>
__global__ void __launch_bounds__(kRefThreads) decode_ref_kernel(DecodeArgs a) {
  extern __shared__ float smem[];
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.context_lens[b];
  if (L < (a.causal ? a.T : 0) || L > a.max_pages * kPage) {
    if (threadIdx.x == 0 && s == 0 && h == 0) flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
    const int G = a.Hq / a.Hkv, R = a.T * G, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < R; r += kRefThreads / 32) {
      const size_t rr = (((size_t)b * a.T + r / G) * a.Hq + h * G + r % G) * a.S + s;
      for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = 0.0f;
      if (lane == 0) a.part_lse[rr] = -INFINITY;
    }
    return;
  }
  ref_unit<D, FP8, RMAX>(a, s, h, b, 0, a.T, L, smem);
}

// ---------------------------------------------------------------- combine
// One warp per output row (b, j, hq).  rotate != 0 applies H_D (normalised)
// to undo the rotation of V.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      int rows, int S, int rotate, float inv_sqrt_d,
                                                      float* __restrict__ out) {
  constexpr int E = D / 32;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* lse = part_lse + (size_t)row * S;
  float m = -INFINITY;
  for (int s = 0; s < S; ++s) m = fmaxf(m, lse[s]);
  float x[E];
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float l = lse[s];
      if (l == -INFINITY) continue;
      const float w = __expf(l - m);
      wsum += w;
      const float* po = part_o + ((size_t)row * S + s) * D + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i) x[i] = fmaf(w, po[i], x[i]);
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int i = 0; i < E; ++i) x[i] *= inv;
  if (rotate) {
    fwht_warp<E, float>(x);
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] *= inv_sqrt_d;
  }
  float* o = out + (size_t)row * D + lane * E;
#pragma unroll
  for (int i = 0; i < E; ++i) o[i] = x[i];
}

// ---------------------------------------------------------------- launchers
template <int D, bool FP8, int RMAX>
static cudaError_t launch_ref_t(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = ref_unit_smem<D, RMAX>();
  auto kern = decode_ref_kernel<D, FP8, RMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S, a.Hkv, a.B);
  kern<<<grid, kRefThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <bool FP8>
static cudaError_t launch_ref_d(int D, int R, const DecodeArgs& a, cudaStream_t st) {
  switch (D) {
    case 64: return R <= 32 ? launch_ref_t<64, FP8, 32>(a, st) : launch_ref_t<64, FP8, 64>(a, st);
    case 128: return R <= 8 ? launch_ref_t<128, FP8, 8>(a, st)
                            : (R <= 32 ? launch_ref_t<128, FP8, 32>(a, st) : launch_ref_t<128, FP8, 64>(a, st));
    case 256: return R <= 16 ? launch_ref_t<256, FP8, 16>(a, st) : launch_ref_t<256, FP8, 32>(a, st);
    case 512: return launch_ref_t<512, FP8, 16>(a, st);
  }
  return cudaErrorInvalidValue;
}

int ref_max_rows(int D) { return D == 512 ? 16 : (D == 256 ? 32 : 64); }

cudaError_t launch_decode_ref(bool fp8, int D, const DecodeArgs& a, cudaStream_t st) {
  const int R = a.T * (a.Hq / a.Hkv);
  return fp8 ? launch_ref_d<true>(D, R, a, st) : launch_ref_d<false>(D, R, a, st);
}

cudaError_t launch_combine(const float* po, const float* pl, int rows, int S, int D, int rotate,
                           float inv_sqrt_d, float* out, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const dim3 grid((rows + 3) / 4), block(128);
  switch (D) {
    case 64: combine_kernel<64><<<grid, block, 0, st>>>(po, pl, rows, S, rotate, inv_sqrt_d, out); break;
    case 128: combine_kernel<128><<<grid, block, 0, st>>>(po, pl, rows, S, rotate, inv_sqrt_d, out); break;
    case 256: combine_kernel<256><<<grid, block, 0, st>>>(po, pl, rows, S, rotate, inv_sqrt_d, out); break;
    case 512: combine_kernel<512><<<grid, block, 0, st>>>(po, pl, rows, S, rotate, inv_sqrt_d, out); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kv4
