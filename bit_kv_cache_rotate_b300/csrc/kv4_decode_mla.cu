// kv4_decode_mla.cu -- tensor-core split decode over a 4-bit latent cache
// (K = V = one 512-value latent row per token, up to 16 query rows per
// latent head), sm_103a.
//
// "GLM-5.3-Flash on MI300X": the 512-value latent row without a RoPE half is
// the MLA workload; "UltraQuant on AMD Instinct", section "What is UltraQuant":
// the latent row is quantised like any K/V vector (Walsh-Hadamard rotation,
// E2M1 codes, one UE8M0 scale per 32 channels).
//
// Work split: one CTA per (split, latent head, sequence), 4 warps; warp w owns
// latent channels 128w .. 128w+127.  Per chunk of 32 tokens (2 pages):
//   Q.K^T  each warp forms the partial scores of all 32 tokens over its 128
//          channels (f16 MMA m16n8k16, q as f16 hi + lo MMAs into one
//          accumulator, the K scale applied per 32-channel group); the four
//          partials meet in shared memory and every warp sums the same full
//          scores, so every warp runs the identical online softmax.
//   P.V    each warp accumulates O^T for its own 128 channels over all tokens:
//          V is the same codes as K, so the widened K fragments (one token,
//          two channels per register) are transposed in registers with
//          movmatrix into V^T fragments (one channel, two tokens); the V scale
//          is folded into P per group as in the 4-bit kernel.
// No cross-warp merge: each warp writes its own channels of the partial output.
#include <cuda_fp16.h>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace mla {

using namespace kv4::mma;

constexpr int D = 512;
constexpr int kWarps = 4;
constexpr int kThreads = 128;
constexpr int kRows = 16;
constexpr int kChunkPages = 2;                     // 32 tokens
constexpr int kCodeBytes = kPage * D / 2;          // 4096
constexpr int kBlk = kCodeBytes + kPage * D / 32;  // 4352
constexpr int kStages = 3;
constexpr int kStageBytes = kChunkPages * kBlk;
constexpr int kQRow = D * 2 + 16;                  // f16 row + pad (bank spread)
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kStages * kStageBytes;      // [hi, lo][16 rows][kQRow]
constexpr int kOffPart = kOffQ + 2 * kRows * kQRow;           // [2][4 warps][32 lanes][16 floats]
constexpr int kOffKTab = kOffPart + 2 * kWarps * 32 * 64;     // [4 warps][4 groups][32 tokens] float
constexpr int kOffVTab = kOffKTab + kWarps * 512;             // [4 warps][16 pairs][4 groups] f16x2
constexpr int kOffBar = kOffVTab + kWarps * 256;
constexpr int kSmem = kOffBar + 8 * kStages;

__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// P.V of one chunk whose V scales span more binades than the f16 factors hold
// (a V scale more than 14 binades below the group reference): the scale is
// folded into P in fp32, x = p * 2^(e - E_G) with E_G the chunk's largest
// exponent of the group, and x and the codes go through bf16 MMAs, which keep
// fp32's exponent range.  Same fragment layout as the f16 path; p[nn][k] holds
// tokens 8nn + 2t + (k & 1) of rows g (k < 2) and g + 8.
__device__ __forceinline__ void pv_bf16(float (&o)[8][2][4], const float (&p)[4][4], const uint8_t* stage,
                                        uint32_t eref, int w, int g, int t) {
#pragma unroll
  for (int G4 = 0; G4 < 4; ++G4) {
    const int E = (int)((eref >> (8 * G4)) & 0xFFu);
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      // B fragments: [rows 0-7 | 8-15][b0: tokens 16kk + 2t (+1), b1: 16kk + 8 + 2t (+1)]
      uint32_t bh[2][2], bl[2][2];
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int tok = 16 * kk + 8 * bb + 2 * t;
        const uint8_t* sp = stage + (tok >> 4) * kBlk + kCodeBytes + (tok & 15) * 16 + 4 * w + G4;
        const float f0 = pow2_diff(sp[0], E), f1 = pow2_diff(sp[16], E);
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
          split_bf16x2(p[2 * kk + bb][2 * hr] * f0, p[2 * kk + bb][2 * hr + 1] * f1, bh[hr][bb], bl[hr][bb]);
      }
      uint32_t wv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nn = 2 * kk + u;
        wv[u] = *reinterpret_cast<const uint32_t*>(stage + (nn >> 1) * kBlk + (((nn & 1) * 16 + 4 * w + G4) * 128) +
                                                   g * 16 + 4 * t);
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t a0 = movtrans(f16x2_to_bf16x2(e2m1x2_to_f16x2(wv[0], 2 * j)));
        const uint32_t a1 = movtrans(f16x2_to_bf16x2(e2m1x2_to_f16x2(wv[0], 2 * j + 1)));
        const uint32_t a2 = movtrans(f16x2_to_bf16x2(e2m1x2_to_f16x2(wv[1], 2 * j)));
        const uint32_t a3 = movtrans(f16x2_to_bf16x2(e2m1x2_to_f16x2(wv[1], 2 * j + 1)));
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          mma_bf16(o[2 * G4 + j][hr], a0, a1, a2, a3, bh[hr][0], bh[hr][1]);
          mma_bf16(o[2 * G4 + j][hr], a0, a1, a2, a3, bl[hr][0], bl[hr][1]);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 2) decode_mla_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float row_c[kRows];
  __shared__ int row_limit[kRows];
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int R = a.T * G;
  const int L = a.context_lens[b];
  const size_t row0 = (size_t)b * a.T * a.Hq;

  auto row_index = [&](int r) -> size_t { return row0 + (size_t)(r / G) * a.Hq + h * G + (r % G); };
  auto write_empty = [&]() {
    for (int r = w; r < R; r += kWarps) {
      const size_t rr = row_index(r) * a.S + s;
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
  const int p0 = s * per;
  const int p1 = min(n_pages, p0 + per);
  if (p0 >= p1) {
    write_empty();
    return;
  }
  const int n_chunks = (p1 - p0 + kChunkPages - 1) / kChunkPages;
  const int32_t* table = a.block_tables + (size_t)b * a.max_pages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBar);

  if (tid == 0)
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  // chunk c -> stage c % 3 (warp 0: lane i < 2 copies page i of the chunk)
  auto issue = [&](int c) {
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
    const int st = c % kStages;
    if (lane == 0) mbar_expect_tx(&full[st], (uint32_t)(nv * kBlk));
    __syncwarp();
    if (lane < nv) {
      int page = table[pg + lane];
      if (page < 0 || page >= a.num_pages) {
        flag_error(a.dev_error, KV4_DEVERR_PAGE);
        page = 0;
      }
      bulk_g2s(smem + kOffStage + st * kStageBytes + lane * kBlk, a.k_cache + ((size_t)page * a.Hkv + h) * kBlk,
               kBlk, &full[st]);
    }
  };
  __syncthreads();
  fence_proxy_async();
  int issued = 0;
  if (w == 0) {
    for (int c = 0; c < min(n_chunks, kStages - 1); ++c) issue(c);
  }
  issued = min(n_chunks, kStages - 1);

  // ---- q prologue: rotate (fp32 butterfly over 512), scale the row by 2^sigma,
  // split into f16 hi + lo rows in shared memory
  for (int r = w; r < kRows; r += kWarps) {
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.0f;
    if (r < R) {
      const uint4* src = reinterpret_cast<const uint4*>(a.q + row_index(r) * D + lane * 16);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 raw = src[i];
        const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[8 * i + 2 * k] = bf16_bits_to_float(wv[k] & 0xFFFFu);
          x[8 * i + 2 * k + 1] = bf16_bits_to_float(wv[k] >> 16);
        }
      }
      fwht_warp<16, float>(x);
    }
    float mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    int sigma = 0;
    if (mx > 0.0f) sigma = max(-113, min(126, 141 - (int)((__float_as_uint(mx) >> 23) & 0xFF)));
    const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
    uint32_t hw[8], lw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float v0 = x[2 * i] * sc, v1 = x[2 * i + 1] * sc;
      const uint32_t hh = pack_f16x2(v0, v1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hh));
      hw[i] = hh;
      lw[i] = pack_f16x2(v0 - hf.x, v1 - hf.y);
    }
    uint4* qh = reinterpret_cast<uint4*>(smem + kOffQ + r * kQRow + lane * 32);
    uint4* ql = reinterpret_cast<uint4*>(smem + kOffQ + (kRows + r) * kQRow + lane * 32);
    qh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    qh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    ql[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    ql[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
    if (lane == 0) {
      // score*log2e = (q*2^sigma . code * 2^e) * 2^-sigma * softmax_scale*log2e/sqrt(D)
      row_c[r] = a.qscale * __uint_as_float((uint32_t)(127 - sigma) << 23);
      row_limit[r] = r < R ? (a.causal ? L - a.T + 1 + r / G : L) : 0x7fffffff;
    }
  }
  __syncthreads();
  const float rc0 = row_c[g], rc1 = row_c[g + 8];
  const int lim0 = row_limit[g], lim1 = row_limit[g + 8];
  int min_limit = row_limit[0];
#pragma unroll
  for (int r = 1; r < kRows; ++r) min_limit = min(min_limit, row_limit[r]);

  const int cb = 128 * w;  // this warp's latent channels
  float o[8][2][4];        // [m-tile 2*G4 + j][rows 0-7 | 8-15][frag]
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int n = 0; n < 2; ++n) o[m][n][0] = o[m][n][1] = o[m][n][2] = o[m][n][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
  uint32_t eref = 0;
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;
  bool timed_out = false;
  int waited = 0;
  float* ktab = reinterpret_cast<float*>(smem + kOffKTab + w * 512);        // [4 groups][32 tokens]
  uint32_t* vtab = reinterpret_cast<uint32_t*>(smem + kOffVTab + w * 256);  // [16 pairs][4 groups]

#pragma unroll 1
  for (int c = 0; c < n_chunks; ++c) {
    const int st = c % kStages;
    if (!mbar_wait(&full[st], (uint32_t)((c / kStages) & 1), c == 0 ? first_limit : kSpinLimit)) timed_out = true;
    if (__syncthreads_or(timed_out)) {
      timed_out = true;
      break;
    }
    ++waited;
    const uint8_t* stage = smem + kOffStage + st * kStageBytes;
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
    const bool edge = nv < kChunkPages || (pg + kChunkPages) * kPage > min_limit;

    // ---- scale tables of this warp's 4 groups: lane = token (page lane>>4)
    uint32_t eold, enew = 0;
    bool slow;
    {
      const int pi = lane >> 4, tk = lane & 15;
      const bool ok = pi < nv && (pg + pi) * kPage + tk < L;
      const uint32_t word = ok ? *reinterpret_cast<const uint32_t*>(stage + pi * kBlk + kCodeBytes + tk * 16 + 4 * w) : 0u;
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) ktab[G4 * 32 + lane] = __uint_as_float(((word >> (8 * G4)) & 0xFFu) << 23);
      // V reference exponents per group (Eref), as in the 4-bit kernel: fixed from
      // the first chunk, raised when a chunk exceeds it by more than 7.
      eold = eref;
      uint32_t lim = __vaddus4(eref, 0x07070707u);
      const bool over = __vcmpgtu4(word, lim) != 0u;
      if (c == 0 || __any_sync(0xffffffffu, over)) {
        uint32_t cm = word;
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
        eref = __vmaxu4(eref, cm);
        lim = __vaddus4(eref, 0x07070707u);
      }
      // f16 exponent fields (tokens past the context take lim's in-window field)
      const uint32_t av = __vsubus4(0x16161616u, __vsubus4(lim, ok ? word : lim));
      const uint32_t an = __shfl_down_sync(0xffffffffu, av, 1);          // token 2p+1
      // A zero field: a V scale more than 14 binades below the reference (or
      // an all-zero group).  Such a chunk takes the bf16 path with the
      // reference re-taken from the chunk (as in the 4-bit decode kernel).
      slow = __any_sync(0xffffffffu, has_zero_byte(av) != 0u);
      if (slow) {
        uint32_t cm = word;
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
        const uint32_t none = __vcmpeq4(cm, 0u);
        enew = (__vmaxu4(cm, __vsubus4(eold, 0x5A5A5A5Au)) & ~none) | (eold & none);
      } else if ((lane & 1) == 0) {
        uint4 vp;
        vp.x = __byte_perm(__byte_perm(av, an, 0x0040), 0, 0x5140) << 10;
        vp.y = __byte_perm(__byte_perm(av, an, 0x0051), 0, 0x5140) << 10;
        vp.z = __byte_perm(__byte_perm(av, an, 0x0062), 0, 0x5140) << 10;
        vp.w = __byte_perm(__byte_perm(av, an, 0x0073), 0, 0x5140) << 10;
        *reinterpret_cast<uint4*>(vtab + (lane >> 1) * 4) = vp;
      }
      __syncwarp();
    }

    // ---- partial Q.K^T over this warp's channels: n-tile nn = tokens 8nn..8nn+7
    // (B column g -> token 8nn + g); group G4 -> channels cb + 32G4 + ...; the k
    // index 2t+i of step j is channel 8t + 4j + i of the group, 2t+8+i is 8t + 4j + 2 + i.
    float sp[4][4];
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) sp[nn][0] = sp[nn][1] = sp[nn][2] = sp[nn][3] = 0.0f;
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      uint32_t qa[2][2][4];  // [j][hi, lo][a0..a3]
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int hl = 0; hl < 2; ++hl) {
          const int ch = cb + 32 * G4 + 8 * t + 4 * j;
          const uint2 r0 = *reinterpret_cast<const uint2*>(smem + kOffQ + (hl * kRows + g) * kQRow + ch * 2);
          const uint2 r1 = *reinterpret_cast<const uint2*>(smem + kOffQ + (hl * kRows + g + 8) * kQRow + ch * 2);
          qa[j][hl][0] = r0.x;
          qa[j][hl][1] = r1.x;
          qa[j][hl][2] = r0.y;
          qa[j][hl][3] = r1.y;
        }
      float acc[4][4];
#pragma unroll
      for (int nn = 0; nn < 4; ++nn) {
        acc[nn][0] = acc[nn][1] = acc[nn][2] = acc[nn][3] = 0.0f;
        const uint32_t word = *reinterpret_cast<const uint32_t*>(
            stage + (nn >> 1) * kBlk + (((nn & 1) * 16 + 4 * w + G4) * 128) + g * 16 + 4 * t);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t b0 = e2m1x2_to_f16x2(word, 2 * j), b1 = e2m1x2_to_f16x2(word, 2 * j + 1);
          mma_f16(acc[nn], qa[j][0][0], qa[j][0][1], qa[j][0][2], qa[j][0][3], b0, b1);
          mma_f16(acc[nn], qa[j][1][0], qa[j][1][1], qa[j][1][2], qa[j][1][3], b0, b1);
        }
      }
#pragma unroll
      for (int nn = 0; nn < 4; ++nn) {
        const float2 ks = *reinterpret_cast<const float2*>(ktab + G4 * 32 + 8 * nn + 2 * t);
        sp[nn][0] = fmaf(ks.x, acc[nn][0], sp[nn][0]);
        sp[nn][1] = fmaf(ks.y, acc[nn][1], sp[nn][1]);
        sp[nn][2] = fmaf(ks.x, acc[nn][2], sp[nn][2]);
        sp[nn][3] = fmaf(ks.y, acc[nn][3], sp[nn][3]);
      }
    }
    float4* part = reinterpret_cast<float4*>(smem + kOffPart + ((c & 1) * kWarps * 32 * 64));
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) part[(w * 32 + lane) * 4 + nn] = make_float4(sp[nn][0], sp[nn][1], sp[nn][2], sp[nn][3]);
    __syncthreads();
    // every warp is done with chunk c-1: stream chunk c+2 into its stage
    if (w == 0 && issued < n_chunks && issued == c + kStages - 1) {
      fence_proxy_async();
      issue(issued);
    }
    if (issued < n_chunks && issued == c + kStages - 1) ++issued;

    // ---- full scores at this thread's fragment positions (rows g, g+8; tokens 8nn + 2t + i)
    float sc[4][4];
#pragma unroll
    for (int nn = 0; nn < 4; ++nn) {
      float4 v = part[lane * 4 + nn];
#pragma unroll
      for (int ww = 1; ww < kWarps; ++ww) {
        const float4 u = part[(ww * 32 + lane) * 4 + nn];
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
      }
      sc[nn][0] = v.x * rc0;
      sc[nn][1] = v.y * rc0;
      sc[nn][2] = v.z * rc1;
      sc[nn][3] = v.w * rc1;
      if (edge) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tok = 8 * nn + 2 * t + (k & 1);
          const int pos = pg * kPage + tok;
          const bool ok = (tok >> 4) < nv && pos < ((k >> 1) ? lim1 : lim0);
          if (!ok) sc[nn][k] = -INFINITY;
        }
      }
    }
    // ---- online softmax, lazy maximum (moves only when exceeded by more than 8)
    float alpha[2] = {1.0f, 1.0f};
    float p[4][4];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float cm = fmaxf(fmaxf(sc[0][2 * hr], sc[0][2 * hr + 1]), fmaxf(sc[1][2 * hr], sc[1][2 * hr + 1]));
      cm = fmaxf(cm, fmaxf(fmaxf(sc[2][2 * hr], sc[2][2 * hr + 1]), fmaxf(sc[3][2 * hr], sc[3][2 * hr + 1])));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
      if (cm > m_run[hr] + 8.0f) {
        alpha[hr] = ex2(m_run[hr] - cm);
        m_run[hr] = cm;
        l_run[hr] *= alpha[hr];
      }
      float ls = 0.0f;
#pragma unroll
      for (int nn = 0; nn < 4; ++nn)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float pv = m_run[hr] == -INFINITY ? 0.0f : ex2(sc[nn][2 * hr + i] - m_run[hr]);
          p[nn][2 * hr + i] = pv;
          ls += pv;
        }
      l_run[hr] += ls;
    }
    // O^T columns are rows: rows 2t, 2t+1 (+8 for the second n-tile) own alphas
    // held by lanes 8t and 8t + 4
    const float a00 = __shfl_sync(0xffffffffu, alpha[0], 8 * t), a01 = __shfl_sync(0xffffffffu, alpha[0], 8 * t + 4);
    const float a10 = __shfl_sync(0xffffffffu, alpha[1], 8 * t), a11 = __shfl_sync(0xffffffffu, alpha[1], 8 * t + 4);
    if (slow || __any_sync(0xffffffffu, a00 != 1.0f || a01 != 1.0f || a10 != 1.0f || a11 != 1.0f || eold != eref)) {
      const uint32_t dl = __vsubus4(eref, eold);
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) {
        const int ex = 127 - (int)((dl >> (8 * G4)) & 0xFFu);
        // slow chunks: the reference moves to enew, up or down
        const float f = slow ? pow2_diff((eold >> (8 * G4)) & 0xFFu, (int)((enew >> (8 * G4)) & 0xFFu))
                             : (ex > 0 ? __uint_as_float((uint32_t)ex << 23) : 0.0f);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float (&o0)[4] = o[2 * G4 + j][0];
          float (&o1)[4] = o[2 * G4 + j][1];
          o0[0] *= f * a00;
          o0[1] *= f * a01;
          o0[2] *= f * a00;
          o0[3] *= f * a01;
          o1[0] *= f * a10;
          o1[1] *= f * a11;
          o1[2] *= f * a10;
          o1[3] *= f * a11;
        }
      }
    }
    if (slow) eref = enew;
    if (slow) {
      pv_bf16(o, p, stage, eref, w, g, t);
    } else {
    // ---- P fragments: k-step kk = tokens 16kk..16kk+15 = n-tiles 2kk, 2kk+1;
    // b0 = tokens 16kk + 2t (+1), b1 = 16kk + 8 + 2t (+1); [kk][rows 0-7 | 8-15][b0, b1]
    uint32_t ph[2][2][2], pl[2][2][2];
    bool need_lo[2];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      float pm = 0.0f;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const float2 v = make_float2(p[2 * kk + bb][2 * hr], p[2 * kk + bb][2 * hr + 1]);
          float2 hi, lo;
          split_hi_lo2(v, hi, lo);
          ph[kk][hr][bb] = pack_f16x2(hi.x, hi.y);
          pl[kk][hr][bb] = pack_f16x2(lo.x, lo.y);
          pm = fmaxf(pm, fmaxf(v.x, v.y));
        }
      need_lo[kk] = __any_sync(0xffffffffu, pm > 0.00390625f);
    }
    // ---- P.V over this warp's channels.  m-tile (G4, j): rows 0-7 are channels
    // 8(g>>1) + 4j + (g&1) of the group, rows 8-15 the same + 2 (the transposed B
    // fragments of the Q.K^T step); columns are tokens.
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      uint32_t pgh[2][2][2], pgl[2][2][2];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t s0 = vtab[(8 * kk + t) * 4 + G4], s1 = vtab[(8 * kk + 4 + t) * 4 + G4];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          pgh[kk][hr][0] = hmul2(ph[kk][hr][0], s0);
          pgh[kk][hr][1] = hmul2(ph[kk][hr][1], s1);
          pgl[kk][hr][0] = hmul2(pl[kk][hr][0], s0);
          pgl[kk][hr][1] = hmul2(pl[kk][hr][1], s1);
        }
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t wv[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int nn = 2 * kk + u;
          wv[u] = *reinterpret_cast<const uint32_t*>(stage + (nn >> 1) * kBlk + (((nn & 1) * 16 + 4 * w + G4) * 128) +
                                                     g * 16 + 4 * t);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t a0 = movtrans(e2m1x2_to_f16x2(wv[0], 2 * j));
          const uint32_t a1 = movtrans(e2m1x2_to_f16x2(wv[0], 2 * j + 1));
          const uint32_t a2 = movtrans(e2m1x2_to_f16x2(wv[1], 2 * j));
          const uint32_t a3 = movtrans(e2m1x2_to_f16x2(wv[1], 2 * j + 1));
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            mma_f16(o[2 * G4 + j][hr], a0, a1, a2, a3, pgh[kk][hr][0], pgh[kk][hr][1]);
            if (need_lo[kk]) mma_f16(o[2 * G4 + j][hr], a0, a1, a2, a3, pgl[kk][hr][0], pgl[kk][hr][1]);
          }
        }
      }
    }
    }  // fast path
  }

  if (timed_out) {
    if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
    for (; waited < issued; ++waited) (void)mbar_wait(&full[waited % kStages], (uint32_t)((waited / kStages) & 1));
  }
  __syncthreads();

  // ---- row sums over the quad, then each warp writes its own channels
  float l_row[2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    float v = l_run[hr];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    l_row[hr] = v;
  }
  // O^T column j of n-tile hr is row 8hr + 2t + (j&1): its l and m come from lane 8t (+4)
  float inv[2][2], mrow[2][2], lrow[2][2];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      lrow[hr][e] = __shfl_sync(0xffffffffu, l_row[hr], 8 * t + 4 * e);
      mrow[hr][e] = __shfl_sync(0xffffffffu, m_run[hr], 8 * t + 4 * e);
      inv[hr][e] = lrow[hr][e] > 0.0f ? 1.0f / lrow[hr][e] : 0.0f;
    }
#pragma unroll
  for (int G4 = 0; G4 < 4; ++G4) {
    const float eg = __uint_as_float(((eref >> (8 * G4)) & 0xFFu) << 23);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int d0 = cb + 32 * G4 + 8 * (g >> 1) + 4 * j + (g & 1);  // fragment row g
      const int d1 = d0 + 2;                                           // fragment row g + 8
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 8 * hr + 2 * t + e;
          if (r >= R) continue;
          const size_t rr = row_index(r) * a.S + s;
          a.part_o[rr * D + d0] = o[2 * G4 + j][hr][e] * eg * inv[hr][e];
          a.part_o[rr * D + d1] = o[2 * G4 + j][hr][2 + e] * eg * inv[hr][e];
        }
    }
  }
  if (w == 0 && g == 0) {
    // lanes 0..3 (t): rows 2t, 2t+1 and 8 + 2t, 8 + 2t + 1
#pragma unroll
    for (int hr = 0; hr < 2; ++hr)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int r = 8 * hr + 2 * t + e;
        if (r >= R) continue;
        const size_t rr = row_index(r) * a.S + s;
        a.part_lse[rr] = lrow[hr][e] > 0.0f ? (mrow[hr][e] + log2f(lrow[hr][e])) * 0.69314718055994531f : -INFINITY;
      }
  }
}

}  // namespace mla

bool mla_path_supported(int D, int G, int T, bool latent) { return D == 512 && latent && T * G <= 16; }

cudaError_t launch_decode_mla(const DecodeArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(mla::decode_mla_kernel, mla::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S, a.Hkv, a.B);
  mla::decode_mla_kernel<<<grid, mla::kThreads, mla::kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
