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

namespace kv4 {

constexpr int kRefThreads = 128;



template <int D, bool FP8, int RMAX>
__global__ void __launch_bounds__(kRefThreads) decode_ref_kernel(DecodeArgs a) {
  constexpr int DP = D + 1;                    // padded row (bank spread)
  constexpr int PER_T = D / kRefThreads > 0 ? D / kRefThreads : 1;
  extern __shared__ float smem[];
  const int R = a.T * (a.Hq / a.Hkv);
  float* qs = smem;                            // [R][D]
  float* ks = qs + RMAX * D;                   // [16][DP]
  float* vs = ks + kPage * DP;                 // [16][DP]
  float* ps = vs + kPage * DP;                 // [R][16]
  float* alpha = ps + RMAX * kPage;            // [R]

  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.Hq / a.Hkv;
  const int L = a.context_lens[b];
  const size_t row0 = ((size_t)b * a.T) * a.Hq;  // (b, j=0, hq=0)

  auto write_empty = [&]() {
    for (int r = warp; r < R; r += kRefThreads / 32) {
      const int j = r / G, g = r % G;
      const size_t rr = (row0 + (size_t)j * a.Hq + h * G + g) * a.S + s;
      for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = 0.0f;
      if (lane == 0) a.part_lse[rr] = -INFINITY;
    }
  };
  if (L < (a.causal ? a.T : 0) || L > a.max_pages * kPage) {
    if (tid == 0 && s == 0 && h == 0) flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
    write_empty();
    return;
  }
  const int n_pages = (L + kPage - 1) / kPage;
  const int per = (n_pages + a.S - 1) / a.S;
  const int p0 = s * per, p1 = min(n_pages, p0 + per);
  if (p0 >= p1) {
    write_empty();
    return;
  }

  // q rows for this kv head: r = j*G + g -> q[b][j][h*G+g]; rotate (4-bit only).
  for (int r = warp; r < R; r += kRefThreads / 32) {
    const int j = r / G, g = r % G;
    const uint16_t* src = a.q + (row0 + (size_t)j * a.Hq + h * G + g) * D;
    constexpr int E = D / 32;
    float x[E];
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = bf16_bits_to_float(src[lane * E + i]);
    if constexpr (!FP8) fwht_warp<E, float>(x);
#pragma unroll
    for (int i = 0; i < E; ++i) qs[r * D + lane * E + i] = x[i] * a.qscale;
  }

  // per-row online softmax state, replicated in the 16 lanes that own a row
  float m_run = -INFINITY, l_run = 0.0f;
  float acc[RMAX][PER_T];
#pragma unroll
  for (int r = 0; r < RMAX; ++r)
#pragma unroll
    for (int i = 0; i < PER_T; ++i) acc[r][i] = 0.0f;

  const int BLK = FP8 ? kPage * D : kPage * D / 2 + kPage * D / 32;
  const float ksc = FP8 ? a.k_scale[h] : 1.0f;
  const float vsc = FP8 ? a.v_scale[h] : 1.0f;
  __syncthreads();

  for (int p = p0; p < p1; ++p) {
    int page = a.block_tables[(size_t)b * a.max_pages + p];
    const bool bad = page < 0 || page >= a.num_pages;
    if (bad) {
      if (tid == 0) flag_error(a.dev_error, KV4_DEVERR_PAGE);
      page = 0;
    }
    const uint8_t* kb = a.k_cache + ((size_t)page * a.Hkv + h) * BLK;
    const uint8_t* vb = a.v_cache + ((size_t)page * a.Hkv + h) * BLK;
    // ---- decode the page to fp32 (rotated space for the 4-bit cache).
    // Slots past the context were never written and may hold any bytes (a
    // UE8M0 0xFF is 2^128, an E4M3 0xFF a NaN); their values are taken as 0,
    // since a zero softmax weight times an infinite or NaN value is NaN.
    for (int idx = tid; idx < kPage * D; idx += kRefThreads) {
      const int t = idx / D, d = idx % D;
      float kv = 0.0f, vv = 0.0f;
      if (bad || p * kPage + t >= L) {
      } else if constexpr (FP8) {
        kv = e4m3x2_to_f32x2(kb[t * D + d]).x * ksc;
        vv = e4m3x2_to_f32x2(vb[d * kPage + t]).x * vsc;
      } else {
        const uint8_t* ksb = kb + kPage * D / 2;
        const uint32_t kc = (kb[k_code_offset(D, t, d)] >> ((d & 1) * 4)) & 0xFu;
        kv = e2m1_to_float(kc) * ue8m0_to_float(ksb[t * (D / 32) + d / 32]);
        if (a.latent) {
          vv = kv;
        } else {
          const uint8_t* vsb = vb + kPage * D / 2;
          const uint32_t vc = (vb[d * (kPage / 2) + t / 2] >> ((t & 1) * 4)) & 0xFu;
          vv = e2m1_to_float(vc) * ue8m0_to_float(vsb[t * (D / 32) + d / 32]);
        }
      }
      ks[t * DP + d] = kv;
      vs[t * DP + d] = vv;
    }
    __syncthreads();

    // ---- scores: thread (r, t) for r in [0, R), t in [0, 16): 16 lanes per row
    for (int base = 0; base < R * kPage; base += kRefThreads) {
      const int pr = base + tid;
      const int r = pr / kPage, t = pr % kPage;
      float sc = -INFINITY;
      if (r < R) {
        const int j = r / G;
        const int pos = p * kPage + t;
        const int limit = a.causal ? L - a.T + 1 + j : L;
        if (pos < limit && !bad) {
          float acc_s = 0.0f;
          const float* qr = qs + r * D;
          const float* kr = ks + t * DP;
#pragma unroll 8
          for (int d = 0; d < D; ++d) acc_s = fmaf(qr[d], kr[d], acc_s);
          sc = acc_s;
        }
      }
      // row max over the 16 lanes holding this row (rows never straddle a half-warp)
      float mx = sc;
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (r < R) {
        // running state for row r lives in ps/alpha via the t==0 lane below
        ps[r * kPage + t] = sc;
        if (t == 0) alpha[r] = mx;
      }
    }
    __syncthreads();
    // per-row softmax update: one thread per row
    if (tid < R) {
      const int r = tid;
      // m_run/l_run for row r are kept by thread r
      const float mx = alpha[r];
      const float m_new = fmaxf(m_run, mx);
      float al, lsum = 0.0f;
      if (m_new == -INFINITY) {
        al = 1.0f;
        for (int t = 0; t < kPage; ++t) ps[r * kPage + t] = 0.0f;
      } else {
        al = exp2f(m_run - m_new);
        for (int t = 0; t < kPage; ++t) {
          const float pv = exp2f(ps[r * kPage + t] - m_new);
          ps[r * kPage + t] = pv;
          lsum += pv;
        }
      }
      l_run = l_run * al + lsum;
      m_run = m_new;
      alpha[r] = al;
    }
    __syncthreads();
    // ---- P.V: thread owns channels d = tid + 128*i for all rows
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const float al = alpha[r];
#pragma unroll
        for (int i = 0; i < PER_T; ++i) acc[r][i] *= al;
      }
    }
    for (int t = 0; t < kPage; ++t) {
#pragma unroll
      for (int i = 0; i < PER_T; ++i) {
        const int d = tid + kRefThreads * i;
        if (d < D) {
          const float vv = vs[t * DP + d];
#pragma unroll
          for (int r = 0; r < RMAX; ++r)
            if (r < R) acc[r][i] = fmaf(ps[r * kPage + t], vv, acc[r][i]);
        }
      }
    }
    __syncthreads();
  }

  // ---- write partials: l and m of row r live in thread r; share through smem
  if (tid < R) {
    ps[tid * kPage + 0] = m_run;
    ps[tid * kPage + 1] = l_run;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < R) {
      const int j = r / G, g = r % G;
      const size_t rr = (row0 + (size_t)j * a.Hq + h * G + g) * a.S + s;
      const float m = ps[r * kPage + 0], l = ps[r * kPage + 1];
      const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
      for (int i = 0; i < PER_T; ++i) {
        const int d = tid + kRefThreads * i;
        if (d < D) a.part_o[rr * D + d] = acc[r][i] * inv_l;
      }
      if (tid == 0) a.part_lse[rr] = l > 0.0f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
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
  constexpr int DP = D + 1;
  const size_t smem = sizeof(float) * ((size_t)RMAX * D + 2 * kPage * DP + RMAX * kPage + RMAX);
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
