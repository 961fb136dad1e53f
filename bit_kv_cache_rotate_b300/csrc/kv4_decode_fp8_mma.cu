// kv4_decode_fp8_mma.cu -- tensor-core split decode over the FP8 (E4M3,
// per-KV-head scale) comparator cache, head_dim 128 (sm_103a).
//
// "UltraQuant on AMD Instinct", section "Why UltraQuant beats 8-bit KV": the
// 4-bit cache is measured against an FP8 cache holding one byte per value.
// This kernel gives that comparator the same machinery as the 4-bit decode so
// the two differ only in what the format costs: the same split/warp layout,
// the same bulk-copy streaming, f16 MMAs and online softmax.
//
//   Q.K^T   f16 MMA (m16n8k16).  Two E4M3 bytes widen to an f16x2 pair in one
//           exact conversion.  q (not rotated: the FP8 cache stores the plain
//           vectors) is split into f16 hi (row g) + lo (row g+8) as in the
//           4-bit kernel.  One accumulator spans all 128 channels; the K scale
//           of the head multiplies the row constant.
//   P.V     f16 MMA, swap-AB: O^T += V^T P^T with V^T read straight from the
//           channel-major V block (16 token bytes per channel).  P is split
//           into f16 hi + lo.  The V scale of the head multiplies O at the end.
//
// Cache blocks per (page, head): K [16 tokens][128] bytes, V [128][16] bytes.
#include <cuda_fp16.h>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace fp8fast {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kPagesPerChunk = 4;
constexpr int kBlk = kPage * D;        // 2048 bytes per (page, head) block
constexpr int kKStride = kBlk;         // staged K blocks, back to back
constexpr int kVStride = kBlk + 32;    // staged V blocks: +2 16-byte units so the four pages of a quad
                                       // land on distinct banks
constexpr int kStageBytes = kPagesPerChunk * (kKStride + kVStride);
constexpr int kQBytes = 8 * 2 * D * 2;  // f16 q [8 rows][hi, lo][128 ch]
// q A-fragments [k-step][lane] uint4, read per use (registers would spill)
constexpr int kOffQFrag = kWarps * kStageBytes + kQBytes + 8 * kWarps;
constexpr int kSmem = kOffQFrag + 8 * 32 * 16;
static_assert(kWarps * kStageBytes >= kWarps * 8 * D * 4 + 2 * kWarps * 8 * 4, "merge area must fit");

__global__ void __launch_bounds__(kThreads, 3) decode_fp8_mma_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // With pos_split (more query rows than one CTA holds) a CTA serves the
  // pos_tile query positions j0 .. j0 + Tc - 1 of the sequence; position j
  // attends to the first L - T + 1 + j tokens (causal verify or extend), so
  // the tile is a decode of Tc positions over the prefix its last position
  // sees.  The tiles of one (split, head, sequence) are neighbours in launch
  // order (x = split * tiles + tile): they read the same pages, so all but
  // the first read are mostly served by L2.
  const int n_tiles = a.pos_split ? (a.T + a.pos_tile - 1) / a.pos_tile : 1;
  const int s = (int)blockIdx.x / n_tiles;
  const int h = blockIdx.y, b = mma::longest_first(a.context_lens, a.B, blockIdx.z);
  const int j0 = a.pos_split ? ((int)blockIdx.x % n_tiles) * a.pos_tile : 0;
  const int Tc = a.pos_split ? min(a.pos_tile, a.T - j0) : a.T;  // query positions in this CTA
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int R = Tc * G;
  const int L_seq = a.context_lens[b];
  const int L = a.causal ? L_seq - (a.T - Tc) + j0 : L_seq;  // tokens visible to this CTA's last position
  const size_t row0 = ((size_t)b * a.T + j0) * a.Hq;
  uint8_t* stage = smem_raw + w * kStageBytes;
  uint16_t* qt = reinterpret_cast<uint16_t*>(smem_raw + kWarps * kStageBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + kWarps * kStageBytes + kQBytes) + w;

  auto row_index = [&](int r) -> size_t { return row0 + (size_t)(r / G) * a.Hq + h * G + (r % G); };
  auto write_empty = [&]() {
    for (int r = w; r < R; r += kWarps) {
      const size_t rr = row_index(r) * a.S + s;
      for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = 0.0f;
      if (lane == 0) a.part_lse[rr] = -INFINITY;
    }
  };
  if (L_seq < (a.causal ? a.T : 0) || L_seq > a.max_pages * kPage) {
    if (tid == 0 && s == 0 && h == 0) flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
    write_empty();
    return;
  }
  const int n_pages = (L + kPage - 1) / kPage;
  const int per = (n_pages + a.S - 1) / a.S;
  const int p0 = s * per;
  const int p1 = min(n_pages, p0 + per);
  if (p0 >= p1) {
    write_empty();
    return;
  }
  const int n_chunks = (p1 - p0 + kPagesPerChunk - 1) / kPagesPerChunk;
  const int32_t* table = a.block_tables + (size_t)b * a.max_pages;

  if (lane == 0) mbar_init(bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

  auto chunk_page = [&](int c) -> int {
    const int pg = p0 + c * kPagesPerChunk;
    int page = 0;
    if (lane < kPagesPerChunk && pg + lane < p1) {
      page = table[pg + lane];
      if (page < 0 || page >= a.num_pages) {
        flag_error(a.dev_error, KV4_DEVERR_PAGE);
        page = 0;
      }
    }
    return page;
  };
  auto issue = [&](int c, int page) {
    const int nv = min(kPagesPerChunk, p1 - (p0 + c * kPagesPerChunk));
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)(nv * 2 * kBlk));
    __syncwarp();
    if (lane < nv) {
      const size_t blk = ((size_t)page * a.Hkv + h) * kBlk;
      bulk_g2s(stage + lane * kKStride, a.k_cache + blk, kBlk, bar);
      bulk_g2s(stage + kPagesPerChunk * kKStride + lane * kVStride, a.v_cache + blk, kBlk, bar);
    }
  };

  __syncthreads();
  fence_proxy_async();
  if (w < n_chunks) issue(w, chunk_page(w));

  // ---- q prologue: scale row by 2^sigma, split into f16 hi + lo (no rotation)
  __shared__ float row_c[8];
  __shared__ int row_limit[8];
  for (int r = w; r < 8; r += kWarps) {
    float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (r < R) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.q + row_index(r) * D + lane * 4);
      x[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      x[1] = bf16_bits_to_float(raw.x >> 16);
      x[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      x[3] = bf16_bits_to_float(raw.y >> 16);
    }
    float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int sigma = 0;
    if (mx > 0.0f) sigma = max(-113, min(126, 141 - (int)((__float_as_uint(mx) >> 23) & 0xFF)));
    const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float v0 = x[2 * i] * sc, v1 = x[2 * i + 1] * sc;
      const uint32_t hh = pack_f16x2(v0, v1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hh));
      hw[i] = hh;
      lw[i] = pack_f16x2(v0 - hf.x, v1 - hf.y);
    }
    *reinterpret_cast<uint2*>(qt + (r * 2) * D + lane * 4) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(qt + (r * 2 + 1) * D + lane * 4) = make_uint2(lw[0], lw[1]);
    if (lane == 0) {
      // score*log2e = (q*2^sigma . k_e4m3) * 2^-sigma * k_scale * softmax_scale*log2e
      row_c[r] = a.qscale * a.k_scale[h] * __uint_as_float((uint32_t)(127 - sigma) << 23);
      row_limit[r] = r < R ? (a.causal ? L - Tc + 1 + r / G : L) : 0x7fffffff;
    }
  }
  __syncthreads();

  // A fragments for the eight k16 steps j: thread t covers channels 32t .. 32t+31;
  // k index 2t+i of step j is channel 32t + 4j + i, 2t+8+i is 32t + 4j + 2 + i,
  // matching the K words (4 channels per 32-bit word) read below.
  uint4* qfrag = reinterpret_cast<uint4*>(smem_raw + kOffQFrag);
  if (w == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint2 hi = *reinterpret_cast<const uint2*>(qt + (g * 2) * D + 32 * t + 4 * j);
      const uint2 lo = *reinterpret_cast<const uint2*>(qt + (g * 2 + 1) * D + 32 * t + 4 * j);
      qfrag[j * 32 + lane] = make_uint4(hi.x, lo.x, hi.y, lo.y);
    }
  }
  __syncthreads();
  const uint32_t qfrag_addr = smem_u32(qfrag) + lane * 16;
  const float my_c = row_c[g];
  const int my_limit = row_limit[g];
  int min_limit = row_limit[0];
#pragma unroll
  for (int r = 1; r < 8; ++r) min_limit = min(min_limit, row_limit[r]);

  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
  float m_run = -INFINITY;
  float2 l2 = make_float2(0.0f, 0.0f);
  bool timed_out = false;
  int it_fail = 0;

  for (int c = w, it = 0; c < n_chunks; c += kWarps, ++it) {
    const int cn = c + kWarps;
    const int next_page = cn < n_chunks ? chunk_page(cn) : 0;
    if (!mbar_wait(bar, (uint32_t)(it & 1))) {
      timed_out = true;
      it_fail = it;
      break;
    }
    const int pg = p0 + c * kPagesPerChunk;
    const int nv = min(kPagesPerChunk, p1 - pg);
    const bool edge = nv < kPagesPerChunk || (pg + kPagesPerChunk) * kPage > min_limit;

    // ---- Q.K^T: n8 tile n covers token pair n of each page (col 2t'+i -> page t', token 2n+i)
    float2 sc[8];
#pragma unroll
    for (int n = 0; n < 8; n += 2) {
      float acc[2][2][4];  // [tile][even/odd k step]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int e = 0; e < 2; ++e) acc[u][e][0] = acc[u][e][1] = acc[u][e][2] = acc[u][e][3] = 0.0f;
      uint4 kw[2][2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint8_t* krow = stage + (g >> 1) * kKStride + (2 * (n + u) + (g & 1)) * D + 32 * t;
        kw[u][0] = *reinterpret_cast<const uint4*>(krow);
        kw[u][1] = *reinterpret_cast<const uint4*>(krow + 16);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t q0, q1, q2, q3;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                     : "r"(qfrag_addr + j * 512));
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint4& q4 = kw[u][j >> 2];
          const uint32_t word = (j & 3) == 0 ? q4.x : (j & 3) == 1 ? q4.y : (j & 3) == 2 ? q4.z : q4.w;
          mma_f16(acc[u][j & 1], q0, q1, q2, q3, e4m3x2_to_f16x2(word, 0), e4m3x2_to_f16x2(word, 1));
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float2 e0 = __fadd2_rn(make_float2(acc[u][0][0], acc[u][0][1]), make_float2(acc[u][0][2], acc[u][0][3]));
        const float2 e1 = __fadd2_rn(make_float2(acc[u][1][0], acc[u][1][1]), make_float2(acc[u][1][2], acc[u][1][3]));
        float2 v = __fmul2_rn(__fadd2_rn(e0, e1), make_float2(my_c, my_c));
        if (edge) {
          const int posb = (pg + t) * kPage + 2 * (n + u);
          const bool ok = t < nv;
          if (!(ok && posb < my_limit)) v.x = -INFINITY;
          if (!(ok && posb + 1 < my_limit)) v.y = -INFINITY;
        }
        sc[n + u] = v;
      }
    }

    // ---- online softmax (lazy maximum, as in the 4-bit kernel)
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(sc[i].x, sc[i].y);
#pragma unroll
    for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
      for (int i = 0; i < w2; ++i) mx8[i] = fmaxf(mx8[i], mx8[i + w2]);
    float cmx = mx8[0];
    cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 1));
    cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 2));
    const float m_new = cmx > m_run + 8.0f ? cmx : m_run;
    float alpha = 1.0f;
    float2 p[8];
    if (m_new == -INFINITY) {
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = make_float2(0.0f, 0.0f);
    } else {
      alpha = ex2(m_run - m_new);
      const float2 nm = make_float2(-m_new, -m_new);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 d2 = __fadd2_rn(sc[i], nm);
        p[i] = make_float2(ex2(d2.x), ex2(d2.y));
      }
      const float2 ls = __fadd2_rn(__fadd2_rn(__fadd2_rn(p[0], p[1]), __fadd2_rn(p[2], p[3])),
                                   __fadd2_rn(__fadd2_rn(p[4], p[5]), __fadd2_rn(p[6], p[7])));
      l2 = __ffma2_rn(l2, make_float2(alpha, alpha), ls);
    }
    m_run = m_new;
    const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
    const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
    if (__any_sync(0xffffffffu, a0 != 1.0f || a1 != 1.0f)) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        o[j][0] *= a0;
        o[j][1] *= a1;
        o[j][2] *= a0;
        o[j][3] *= a1;
      }
    }

    // ---- P fragments (hi + lo f16), lo MMAs only where some p > 2^-8
    uint32_t ph[4][2], pl[4][2];
    bool need_lo[4];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      float2 h0, l0, h1, l1;
      split_hi_lo2(p[2 * c4], h0, l0);
      split_hi_lo2(p[2 * c4 + 1], h1, l1);
      ph[c4][0] = pack_f16x2(h0.x, h0.y);
      ph[c4][1] = pack_f16x2(h1.x, h1.y);
      pl[c4][0] = pack_f16x2(l0.x, l0.y);
      pl[c4][1] = pack_f16x2(l1.x, l1.y);
      const float pm = fmaxf(fmaxf(p[2 * c4].x, p[2 * c4].y), fmaxf(p[2 * c4 + 1].x, p[2 * c4 + 1].y));
      need_lo[c4] = __any_sync(0xffffffffu, pm > 0.00390625f);
    }

    // ---- P.V: m-tile jt = channels 16jt..16jt+15 of page t's V block; word c4 of a
    // channel row holds tokens 4c4..4c4+3 (k 2t,2t+1 -> low pair, 2t+8,2t+9 -> high pair).
    // In an edge chunk, V bytes of tokens past the context (or of pages the chunk
    // does not hold) are stale stage memory; E4M3 has NaN encodings and p = 0
    // does not cancel a NaN in the MMA, so those bytes are zeroed first.
    const uint8_t* vbase = stage + kPagesPerChunk * kKStride + t * kVStride;
    uint32_t vmask[4] = {~0u, ~0u, ~0u, ~0u};
    if (edge) {
      const int base = (pg + t) * kPage;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int nok = t < nv ? min(4, max(0, L - (base + 4 * c4))) : 0;
        vmask[c4] = nok >= 4 ? ~0u : ((1u << (8 * nok)) - 1u);
      }
    }
#pragma unroll
    for (int jt = 0; jt < 8; jt += 2) {
      uint4 ra[2], rb[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        ra[u] = *reinterpret_cast<const uint4*>(vbase + (16 * (jt + u) + g) * kPage);
        rb[u] = *reinterpret_cast<const uint4*>(vbase + (16 * (jt + u) + g + 8) * kPage);
        if (edge) {
          ra[u].x &= vmask[0]; ra[u].y &= vmask[1]; ra[u].z &= vmask[2]; ra[u].w &= vmask[3];
          rb[u].x &= vmask[0]; rb[u].y &= vmask[1]; rb[u].z &= vmask[2]; rb[u].w &= vmask[3];
        }
      }
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t wa = c4 == 0 ? ra[u].x : c4 == 1 ? ra[u].y : c4 == 2 ? ra[u].z : ra[u].w;
          const uint32_t wb = c4 == 0 ? rb[u].x : c4 == 1 ? rb[u].y : c4 == 2 ? rb[u].z : rb[u].w;
          const uint32_t x0 = e4m3x2_to_f16x2(wa, 0), x1 = e4m3x2_to_f16x2(wb, 0);
          const uint32_t x2 = e4m3x2_to_f16x2(wa, 1), x3 = e4m3x2_to_f16x2(wb, 1);
          mma_f16(o[jt + u], x0, x1, x2, x3, ph[c4][0], ph[c4][1]);
          if (need_lo[c4]) mma_f16(o[jt + u], x0, x1, x2, x3, pl[c4][0], pl[c4][1]);
        }
      }
    }
    __syncwarp();
    if (cn < n_chunks) {
      fence_proxy_async();
      issue(cn, next_page);
    }
  }

  if (timed_out) {
    // Stop streaming, but let the copy this warp issued last land before the
    // shared memory is reused (the wait is bounded again).
    if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
    (void)mbar_wait(bar, (uint32_t)(it_fail & 1));
  }

  // ---- merge the 4 warps (V scale of the head applied here)
  float l_row = l2.x + l2.y;
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
  l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
  __syncthreads();
  float* mo = reinterpret_cast<float*>(smem_raw);  // [kWarps][8 rows][D]
  float* mm = mo + kWarps * 8 * D;
  float* ml = mm + kWarps * 8;
  if (t == 0) {
    mm[w * 8 + g] = m_run;
    ml[w * 8 + g] = l_row;
  }
  const float vs = a.v_scale[h];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    mo[(w * 8 + 2 * t) * D + 16 * j + g] = o[j][0] * vs;
    mo[(w * 8 + 2 * t + 1) * D + 16 * j + g] = o[j][1] * vs;
    mo[(w * 8 + 2 * t) * D + 16 * j + g + 8] = o[j][2] * vs;
    mo[(w * 8 + 2 * t + 1) * D + 16 * j + g + 8] = o[j][3] * vs;
  }
  __syncthreads();
  for (int r = w; r < 8; r += kWarps) {
    if (r >= R) continue;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, mm[ww * 8 + r]);
    float wsum = 0.0f, wt[kWarps];
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      wt[ww] = (M == -INFINITY || mm[ww * 8 + r] == -INFINITY) ? 0.0f : exp2f(mm[ww * 8 + r] - M);
      wsum += wt[ww] * ml[ww * 8 + r];
    }
    const size_t rr = row_index(r) * a.S + s;
    const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
    for (int d = lane; d < D; d += 32) {
      float acc = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) acc = fmaf(wt[ww], mo[(ww * 8 + r) * D + d], acc);
      a.part_o[rr * D + d] = acc * inv;
    }
    if (lane == 0) a.part_lse[rr] = wsum > 0.0f ? (M + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
  }
}

}  // namespace fp8fast

bool fp8_fast_path_supported(int D, int G, int T) {
  (void)T;  // T * G > 8 runs one CTA per query position (pos_split)
  return D == 128 && G <= 8;
}

cudaError_t launch_decode_fp8_fast(const DecodeArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(fp8fast::decode_fp8_mma_kernel, fp8fast::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S * (a.pos_split ? (a.T + a.pos_tile - 1) / a.pos_tile : 1), a.Hkv, a.B);
  fp8fast::decode_fp8_mma_kernel<<<grid, fp8fast::kThreads, fp8fast::kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
