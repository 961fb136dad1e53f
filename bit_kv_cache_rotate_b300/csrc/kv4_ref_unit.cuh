// kv4_ref_unit.cuh -- exact CUDA-core decode attention of one work unit (one
// split of one kv head of one sequence, for a run of query positions), as a
// device routine.
//
// It is the body of the general decode kernel and the exact fallback of the
// tensor-core kernels: per page of 16 tokens the 128 threads stage the K and V
// blocks in shared memory, decode each code to fp32 (code value from its bit
// fields times 2^e from the UE8M0 byte: exact), form the scores, update an
// online softmax per query row and accumulate P.V in fp32.  Every value keeps
// its own scale, so the result is exact up to fp32 rounding over the whole
// range of per-token scales ("UltraQuant on AMD Instinct", section "What is
// UltraQuant": one power-of-two scale per 32 channels of each token).
#pragma once

#include "kv4_common.cuh"
#include "kv4_decode.h"

namespace kv4 {

constexpr int kRefThreads = 128;

// Shared memory the routine uses: q rows, K and V pages, P, alpha.
template <int D, int RMAX>
__host__ __device__ constexpr size_t ref_unit_smem() {
  return sizeof(float) * ((size_t)RMAX * D + 2 * kPage * (D + 1) + RMAX * kPage + RMAX);
}

// Work unit (split s, kv head h, sequence b, positions j0 .. j0 + Tc - 1):
// rows r = 0 .. Tc*G - 1 are position j0 + r / G of query head h*G + r % G,
// at most RMAX.  Position j sees the first L_seq - T + 1 + j tokens (every
// token when the call is not causal).  The split's pages are those of the
// first L_unit tokens (the tokens the unit's last position sees), cut into
// a.S splits as the tensor-core kernels cut them.  Writes the unit's partial
// outputs (normalised) and log-sum-exps.  All kRefThreads threads of the CTA
// call it; smem holds ref_unit_smem<D, RMAX>() bytes.
template <int D, bool FP8, int RMAX>
__device__ void ref_unit(const DecodeArgs& a, int s, int h, int b, int j0, int Tc, int L_unit, float* smem) {
  constexpr int DP = D + 1;                    // padded row (bank spread)
  constexpr int PER_T = D / kRefThreads > 0 ? D / kRefThreads : 1;
  const int G = a.Hq / a.Hkv;
  const int R = Tc * G;
  float* qs = smem;                            // [R][D]
  float* ks = qs + RMAX * D;                   // [16][DP]
  float* vs = ks + kPage * DP;                 // [16][DP]
  float* ps = vs + kPage * DP;                 // [R][16]
  float* alpha = ps + RMAX * kPage;            // [R]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L_seq = a.context_lens[b];
  const size_t row0 = ((size_t)b * a.T + j0) * a.Hq;  // (b, j0, hq=0)

  const int n_pages = (L_unit + kPage - 1) / kPage;
  const int per = (n_pages + a.S - 1) / a.S;
  const int p0 = s * per, p1 = min(n_pages, p0 + per);
  if (p0 >= p1) {
    for (int r = warp; r < R; r += kRefThreads / 32) {
      const size_t rr = (row0 + (size_t)(r / G) * a.Hq + h * G + r % G) * a.S + s;
      for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = 0.0f;
      if (lane == 0) a.part_lse[rr] = -INFINITY;
    }
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
      if (bad || p * kPage + t >= L_unit) {
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
        const int limit = a.causal ? L_seq - a.T + 1 + j0 + j : L_seq;
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

}  // namespace kv4
