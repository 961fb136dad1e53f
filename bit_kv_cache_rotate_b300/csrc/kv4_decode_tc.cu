// kv4_decode_tc.cu -- split decode over the 4-bit cache with Q.K^T on the
// block-scaled tcgen05 tensor core (sm_103a), head_dim 128.
//
// "UltraQuant on AMD Instinct", section "What is UltraQuant": the FP4 codes and
// their power-of-two scales go straight into the matrix units, no lookup
// table.  On B300 that is tcgen05.mma kind::mxf4 with UE8M0 block scales, one
// scale per 32 elements along the reduction dimension -- exactly the cache's
// K format (E2M1 codes, one UE8M0 byte per token and 32 channels):
//
//   Q.K^T  D[token][row] = sum_k K[token][k] * Q[row][k], one MMA tile of
//          M = 128 tokens (8 pages) x N = 32 (4 of the 8 q terms side by side
//          for the 8 query rows), K = 64 channels per instruction.  A = the K codes as the cache
//          stores them (8-token x 32-channel tiles are the MMA's core
//          matrices), scale A = the cache's scale bytes, written into tensor
//          memory per token.  B = q (rotated, times the softmax scale and
//          log2 e) as 8 E2M1 terms, each with its own UE8M0 scale per 32
//          channels; terms i and i+4 accumulate in column 8i + row and the
//          four columns of a row are summed after the load, so the logit (in
//          log2 units) carries about 2^-16 of each 32-channel block's largest
//          q element.  Four wide MMAs per chunk: an N = 16 MMA was measured
//          at about the cost of an N = 32 one.
//   softmax one thread per token: the warp's 32 tokens x 8 rows come out of
//          tensor memory with one load; online softmax with a lazy maximum.
//   P.V    f16 warp MMA (m16n8k16), swap-AB as in the warp-MMA kernel: V codes
//          widened by the hardware E2M1->f16 conversion, the V scale folded
//          into the P fragments, P as f16 hi + lo, the fragments read from
//          shared memory with ldmatrix.trans.
//
// Pipeline (one CTA per (split, kv head, sequence), 4 warps): chunk c = 8
// pages.  K codes + scales of chunk c+2 stream into a double-buffered stage
// by 1-D bulk copies as soon as MMA(c) has completed; each warp streams the V
// of its 2 pages into its own double-buffered stage.  Iteration c writes the
// scale factors of chunk c, syncs the CTA, issues MMA(c) (thread 0, committed
// to an mbarrier), then processes chunk c-1 while MMA(c) runs.  Every wait is
// bounded; a timeout is agreed at the CTA barrier, flagged, and drained.
#include <cuda_fp16.h>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace tc {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 128;
constexpr int kChunkPages = 8;                 // 128 tokens: the MMA's M
constexpr int kCodeBytes = kPage * D / 2;      // 1024
constexpr int kBlk = kCodeBytes + kPage * D / 32;  // 1088
constexpr int kTerms = 8;
constexpr int kTermsN = 4;                     // terms side by side along N
constexpr int kN = 8 * kTermsN;                // MMA N = 32: column 8i + row holds term (4j + i) of the row
constexpr int kTermGroups = kTerms / kTermsN;  // term groups accumulate along K (j = 0, 1)

// shared memory map (bytes)
constexpr int kKCodes = kChunkPages * kCodeBytes;          // 8192 per buffer
constexpr int kKScales = kChunkPages * 64;                  // 512 per buffer
constexpr int kKBufs = 3;                                   // K runs two chunks ahead
constexpr int kOffKCodes = 0;                               // [3][8192]
constexpr int kOffKScales = kOffKCodes + kKBufs * kKCodes;  // [3][512]
constexpr int kVStage = 2 * kBlk;                           // a warp's 2 pages (stride 1088: conflict-free)
constexpr int kOffV = kOffKScales + kKBufs * kKScales;      // [4 warps][2][2176]
constexpr int kQGroup = kN * 64;                            // one term group: 32 B-rows x 64 B
constexpr int kOffQ = kOffV + kWarps * 2 * kVStage;         // [2 term groups][kQGroup]
constexpr int kOffP = kOffQ + kTermGroups * kQGroup;        // [4 warps][hi, lo][32 tokens][16 B]
constexpr int kOffVTab = kOffP + kWarps * 2 * 32 * 16;      // [4 warps][16 pairs][4 groups] f16x2
constexpr int kOffSfb = kOffVTab + kWarps * 16 * 16;        // [8 terms][16 rows][4] bytes
constexpr int kOffBar = kOffSfb + kTerms * 8 * 4;           // mbarriers
constexpr int kNumBars = kKBufs + 2 + 2 * kWarps;           // kfull[3], sdone[2], vfull[4][2]
constexpr int kSmem = kOffBar + 8 * kNumBars + 16;
static_assert(kOffQ % 1024 == 0 || kOffQ % 128 == 0, "operand tiles need 128-byte alignment");
static_assert(kSmem <= 57 * 1024, "four CTAs per SM");
static_assert(kSmem > 228 * 1024 / 5, "at most four CTAs per SM (tensor memory is split four ways)");
static_assert(kOffV >= kWarps * 8 * D * 4 + 2 * kWarps * 8 * 4, "the merge reuses the K stages");

// tensor memory columns (128 allocated)
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColD = 0;      // [2][32]
constexpr uint32_t kColSfa = 64;   // [2 buffers][2 k-steps][4]
constexpr uint32_t kColSfb = 80;   // [2 term groups][2 k-steps][4]

// ---------------------------------------------------------------- tcgen05 helpers
// K-major, no swizzle: core matrices of 8 rows x 16 B; LBO (next 32 elements
// along K) = 128 B, SBO (next 8 rows) = sbo; version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// kind::mxf4, A = B = E2M1, UE8M0 scales, D fp32, both K-major, M = 128, N = 32.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(sfa), "r"(sfb), "r"(accumulate));
}

__device__ __forceinline__ void tmem_st4(uint32_t addr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(v));
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Bounded mbarrier wait agreed by the whole warp (the instructions that
// follow are warp-collective).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ float f16_lo(uint32_t h2) { return __low2float(*reinterpret_cast<const __half2*>(&h2)); }
__device__ __forceinline__ float f16_hi(uint32_t h2) { return __high2float(*reinterpret_cast<const __half2*>(&h2)); }

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 4) decode_fp4_tc_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tmem_base_s;
  __shared__ int row_limit_s[8];
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
  if (L < a.T || L > a.max_pages * kPage) {
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
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kfull = bars;                  // [3], one arrival per warp
  uint64_t* sdone = bars + kKBufs;         // [2]
  uint64_t* vfull = bars + kKBufs + 2 + 2 * w;  // this warp's [2]

  if (tid == 0)
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], i < kKBufs ? kWarps : 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // zero the q operand (unused rows stay zero)
  for (int i = tid; i < kTermGroups * kQGroup / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_lane = tmem + ((uint32_t)(32 * w) << 16);

  // page id of page i of chunk c (0 past the split; bad ids flagged and read as 0)
  auto page_id = [&](int c, int i) -> int {
    const int pg = p0 + c * kChunkPages + i;
    if (pg >= p1) return 0;
    int page = table[pg];
    if (page < 0 || page >= a.num_pages) {
      flag_error(a.dev_error, KV4_DEVERR_PAGE);
      page = 0;
    }
    return page;
  };
  // K of chunk c -> buffer c % 3: each warp copies the codes and scales of its
  // own 2 pages (lane i < 2 -> page 2w + i) and arrives once.
  auto issue_k = [&](int c) {
    const int nv = min(kChunkPages, p1 - (p0 + c * kChunkPages));
    const int nw = max(0, min(2, nv - 2 * w));
    const int buf = c % kKBufs;
    if (lane == 0) mbar_expect_tx(&kfull[buf], (uint32_t)(nw * kBlk));
    __syncwarp();
    if (lane < nw) {
      const int pi = 2 * w + lane;
      const uint8_t* src = a.k_cache + ((size_t)page_id(c, pi) * a.Hkv + h) * kBlk;
      bulk_g2s(smem + kOffKCodes + buf * kKCodes + pi * kCodeBytes, src, kCodeBytes, &kfull[buf]);
      bulk_g2s(smem + kOffKScales + buf * kKScales + pi * 64, src + kCodeBytes, 64, &kfull[buf]);
    }
  };
  // V of this warp's 2 pages of chunk c -> its buffer c&1
  auto issue_v = [&](int c) {
    const int nv = min(kChunkPages, p1 - (p0 + c * kChunkPages));
    const int nw = max(0, min(2, nv - 2 * w));
    const int buf = c & 1;
    if (lane == 0) mbar_expect_tx(&vfull[buf], (uint32_t)(nw * kBlk));
    __syncwarp();
    if (lane < nw) {
      const uint8_t* src = a.v_cache + ((size_t)page_id(c, 2 * w + lane) * a.Hkv + h) * kBlk;
      bulk_g2s(smem + kOffV + (w * 2 + buf) * kVStage + lane * kBlk, src, kBlk, &vfull[buf]);
    }
  };
  // Every expect_tx above is one arrival; a warp with no V pages in a chunk
  // still arrives (zero bytes), so every phase completes.
  fence_proxy_async();
  int k_issued = 0, v_issued = 0;
  for (int c0 = 0; c0 < min(n_chunks, kKBufs); ++c0) issue_k(c0);
  k_issued = min(n_chunks, kKBufs);
  issue_v(0);
  if (n_chunks > 1) issue_v(1);
  v_issued = min(n_chunks, 2);

  // ---- q prologue: rotate (fp32 butterfly), times softmax_scale*log2e/sqrt(D),
  // then 8 E2M1 terms with one UE8M0 scale per 32 channels each.
  uint8_t* sfb_s = smem + kOffSfb;  // [term][8 rows][block]
  for (int r = w; r < 8; r += kWarps) {
    float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (r < R) {
      const uint2 raw = *reinterpret_cast<const uint2*>(a.q + row_index(r) * D + lane * 4);
      x[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      x[1] = bf16_bits_to_float(raw.x >> 16);
      x[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      x[3] = bf16_bits_to_float(raw.y >> 16);
      fwht_warp<4, float>(x);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= a.qscale;
    }
#pragma unroll 1
    for (int term = 0; term < kTerms; ++term) {
      float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
      // block exponent: the smallest e with am <= 6 * 2^e (no saturation)
      int e = -125;
      const uint32_t ab = __float_as_uint(am);
      if (am >= 1.0e-30f) {
        const int e0 = (int)(ab >> 23) - 127;
        e = (ab & 0x7FFFFFu) <= 0x400000u ? e0 - 2 : e0 - 1;
        e = max(-125, min(125, e));
      }
      const float down = __uint_as_float((uint32_t)(127 - e) << 23);
      const float up = __uint_as_float((uint32_t)(127 + e) << 23);
      const uint32_t c01 = f32x2_to_e2m1x2(x[0] * down, x[1] * down);
      const uint32_t c23 = f32x2_to_e2m1x2(x[2] * down, x[3] * down);
      const uint32_t h01 = e2m1x2_to_f16x2(c01, 0), h23 = e2m1x2_to_f16x2(c23, 0);
      x[0] -= f16_lo(h01) * up;
      x[1] -= f16_hi(h01) * up;
      x[2] -= f16_lo(h23) * up;
      x[3] -= f16_hi(h23) * up;
      // term (4j + i) of row r is B-row 8i + r of term group j: core-matrix row
      // group i, channel chunk lane/8, byte 2*(lane%8)
      const int tj = term / kTermsN, ti = term % kTermsN;
      uint8_t* dst = smem + kOffQ + tj * kQGroup + (ti * 4 + (lane >> 3)) * 128 + r * 16 + 2 * (lane & 7);
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(c01 | (c23 << 8));
      if ((lane & 7) == 0) sfb_s[(term * 8 + r) * 4 + (lane >> 3)] = (uint8_t)(e + 127);
    }
    if (lane == 0) row_limit_s[r] = r < R ? L - a.T + 1 + r / G : 0x7fffffff;
  }
  __syncthreads();
  // scale factors of B into tensor memory: each warp writes its lane quadrant
  // (B-row n = 8i + r at lane n), all four columns of each (group, k-step) set
  {
    const int ti = lane >> 3, r = lane & 7;
#pragma unroll
    for (int tj = 0; tj < kTermGroups; ++tj)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint8_t* sb = sfb_s + ((tj * kTermsN + ti) * 8 + r) * 4 + 2 * ks;
        const uint32_t word = (uint32_t)sb[0] | ((uint32_t)sb[1] << 8) | 0x7F7F0000u;
        tmem_st4(tmem_lane + kColSfb + (tj * 2 + ks) * 4, word);
      }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();  // q operand written by ordinary stores, read by the MMA
  int min_limit = row_limit_s[0];
#pragma unroll
  for (int r = 1; r < 8; ++r) min_limit = min(min_limit, row_limit_s[r]);
  int row_lim[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) row_lim[r] = row_limit_s[r];

  // ---- per-warp running state
  float o[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
  float m_run[8], l_run[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.0f;
  }
  uint32_t eref = 0;
  bool timed_out = false;
  int k_waited = 0, s_issued = 0, s_waited = 0, v_waited = 0;
  uint8_t* pbuf = smem + kOffP + w * 2 * 32 * 16;  // [hi, lo][32 tokens][16 B]
  uint32_t* vtab = reinterpret_cast<uint32_t*>(smem + kOffVTab + w * 256);  // [16 pairs][4 groups]
  // ldmatrix row address of this lane: matrix mi = lane/8 -> (kstep mi>>1, half mi&1),
  // row r = lane%8 -> token 8*(r>>1) + 4*kstep + 2*half + (r&1)
  const int lm_mi = lane >> 3, lm_r = lane & 7;
  const int lm_tok = 8 * (lm_r >> 1) + 4 * (lm_mi >> 1) + 2 * (lm_mi & 1) + (lm_r & 1);
  const uint32_t lm_addr_hi = smem_u32(pbuf) + lm_tok * 16;
  const uint32_t lm_addr_lo = lm_addr_hi + 32 * 16;

#pragma unroll 1
  for (int c = 0; c <= n_chunks; ++c) {
    // ---------------- issue MMA(c)
    if (c < n_chunks) {
      const int buf = c & 1, kb = c % kKBufs;
      if (!wait_warp(&kfull[kb], (uint32_t)((c / kKBufs) & 1))) timed_out = true;
      else ++k_waited;
      // scale factors of A for this warp's 32 tokens (lane = token of pages 2w, 2w+1)
      const int pi = 2 * w + (lane >> 4), tok = lane & 15;
      const int pos = (p0 + c * kChunkPages + pi) * kPage + tok;
      uint32_t sw = 0;
      if (!timed_out && p0 + c * kChunkPages + pi < p1 && pos < L)
        sw = *reinterpret_cast<const uint32_t*>(smem + kOffKScales + kb * kKScales + pi * 64 + tok * 4);
      tmem_st4(tmem_lane + kColSfa + buf * 8 + 0, sw & 0xFFFFu);
      tmem_st4(tmem_lane + kColSfa + buf * 8 + 4, sw >> 16);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      if (__syncthreads_or(timed_out)) {
        timed_out = true;
        break;
      }
      if (tid == 32 * (c & 3)) {  // the issuing warp rotates
        fence_after_sync();
        const uint32_t a_base = sbase + kOffKCodes + kb * kKCodes;
        const uint32_t b_base = sbase + kOffQ;
#pragma unroll
        for (int tj = 0; tj < kTermGroups; ++tj)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_mxf4(tmem + kColD + kN * buf, smem_desc(a_base + ks * 256, 512),
                     smem_desc(b_base + tj * kQGroup + ks * 256, 512), tmem + kColSfa + buf * 8 + ks * 4,
                     tmem + kColSfb + (tj * 2 + ks) * 4, (tj | ks) != 0);
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&sdone[buf]))
                     : "memory");
      }
      ++s_issued;
    }
    // ---------------- process chunk c-1 while MMA(c) runs
    if (c == 0) continue;
    const int cc = c - 1, bb = cc & 1;
    if (!wait_warp(&sdone[bb], (uint32_t)((cc >> 1) & 1))) {
      timed_out = true;
      continue;  // agreed at the next barrier
    }
    ++s_waited;
    fence_after_sync();
    // K buffer of chunk cc is free: stream chunk cc+3 into it
    if (cc + kKBufs < n_chunks) {
      fence_proxy_async();
      issue_k(cc + kKBufs);
      ++k_issued;
    }
    // logits of this warp's tokens: column 8i + r holds terms (i, i + 4) of row r
    uint32_t dq[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(dq[0]), "=r"(dq[1]), "=r"(dq[2]), "=r"(dq[3]), "=r"(dq[4]), "=r"(dq[5]), "=r"(dq[6]), "=r"(dq[7]),
          "=r"(dq[8]), "=r"(dq[9]), "=r"(dq[10]), "=r"(dq[11]), "=r"(dq[12]), "=r"(dq[13]), "=r"(dq[14]),
          "=r"(dq[15]), "=r"(dq[16]), "=r"(dq[17]), "=r"(dq[18]), "=r"(dq[19]), "=r"(dq[20]), "=r"(dq[21]),
          "=r"(dq[22]), "=r"(dq[23]), "=r"(dq[24]), "=r"(dq[25]), "=r"(dq[26]), "=r"(dq[27]), "=r"(dq[28]),
          "=r"(dq[29]), "=r"(dq[30]), "=r"(dq[31])
        : "r"(tmem_lane + kColD + kN * bb));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    fence_before_sync();
    float dr[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      dr[r] = (__uint_as_float(dq[r]) + __uint_as_float(dq[8 + r])) +
              (__uint_as_float(dq[16 + r]) + __uint_as_float(dq[24 + r]));
    const int pg0 = p0 + cc * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg0);
    const int pi = 2 * w + (lane >> 4), tok = lane & 15;
    const int pos = (pg0 + pi) * kPage + tok;
    const bool valid = pi < nv && pos < L;
    float sc[8];
    if (a.T == 1) {
#pragma unroll
      for (int r = 0; r < 8; ++r) sc[r] = valid ? dr[r] : -INFINITY;
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) sc[r] = (valid && pos < row_lim[r]) ? dr[r] : -INFINITY;
    }
    // lazy maximum: move a row's reference only when a logit exceeds it by > 8
    bool over = false;
#pragma unroll
    for (int r = 0; r < 8; ++r) over |= sc[r] > m_run[r] + 8.0f;
    float alpha[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) alpha[r] = 1.0f;
    bool rescale = false;
    if (__any_sync(0xffffffffu, over)) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float cm = sc[r];
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
        if (cm > m_run[r] + 8.0f) {
          alpha[r] = ex2(m_run[r] - cm);
          m_run[r] = cm;
          l_run[r] *= alpha[r];
          rescale = true;
        }
      }
    }
    float p[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      p[r] = m_run[r] == -INFINITY ? 0.0f : ex2(sc[r] - m_run[r]);
      l_run[r] += p[r];
    }
    // P rows of this token as f16 hi + lo: [token][8 rows]
    {
      float2 hh[4], ll[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) split_hi_lo2(make_float2(p[2 * i], p[2 * i + 1]), hh[i], ll[i]);
      uint4 ph, pl;
      ph.x = pack_f16x2(hh[0].x, hh[0].y);
      ph.y = pack_f16x2(hh[1].x, hh[1].y);
      ph.z = pack_f16x2(hh[2].x, hh[2].y);
      ph.w = pack_f16x2(hh[3].x, hh[3].y);
      pl.x = pack_f16x2(ll[0].x, ll[0].y);
      pl.y = pack_f16x2(ll[1].x, ll[1].y);
      pl.z = pack_f16x2(ll[2].x, ll[2].y);
      pl.w = pack_f16x2(ll[3].x, ll[3].y);
      *reinterpret_cast<uint4*>(pbuf + lane * 16) = ph;
      *reinterpret_cast<uint4*>(pbuf + 32 * 16 + lane * 16) = pl;
    }
    const float pmax = fmaxf(fmaxf(fmaxf(p[0], p[1]), fmaxf(p[2], p[3])), fmaxf(fmaxf(p[4], p[5]), fmaxf(p[6], p[7])));
    const uint32_t bigm = __ballot_sync(0xffffffffu, pmax > 0.00390625f);
    const bool need_lo0 = (bigm & 0x0F0F0F0Fu) != 0u, need_lo1 = (bigm & 0xF0F0F0F0u) != 0u;

    // ---- V of this warp's 2 pages
    if (!wait_warp(&vfull[bb], (uint32_t)((cc >> 1) & 1))) {
      timed_out = true;
      continue;
    }
    ++v_waited;
    const uint8_t* vst = smem + kOffV + (w * 2 + bb) * kVStage;
    uint32_t eold;
    {
      // lanes 0..15: token pair l (tokens 2l, 2l+1 of the warp's 32)
      uint32_t v0 = 0, v1 = 0;
      if (lane < 16) {
        const int tk = 2 * lane, pj = tk >> 4, tt = tk & 15;
        const int ps = (pg0 + 2 * w + pj) * kPage + tt;
        if (2 * w + pj < nv) {
          const uint2 vv = *reinterpret_cast<const uint2*>(vst + pj * kBlk + kCodeBytes + tt * 4);
          if (ps < L) v0 = vv.x;
          if (ps + 1 < L) v1 = vv.y;
        }
      }
      // V reference exponent per group (Eref), fixed from the warp's first
      // chunk and raised only when a chunk exceeds it by more than 7; the f16
      // factors 2^(e_v - Eref) then lie in [2^-14, 2^7] and p * factor < 2^15.
      eold = eref;
      uint32_t lim = __vaddus4(eref, 0x07070707u);
      const bool vover = (__vcmpgtu4(v0, lim) | __vcmpgtu4(v1, lim)) != 0u;
      if (cc == 0 || __any_sync(0xffffffffu, vover)) {
        uint32_t cm = __vmaxu4(v0, v1);
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
        eref = __vmaxu4(eref, cm);
        lim = __vaddus4(eref, 0x07070707u);
      }
      if (lane < 16) {
        const uint32_t a0 = __vsubus4(0x16161616u, __vsubus4(lim, v0));
        const uint32_t a1 = __vsubus4(0x16161616u, __vsubus4(lim, v1));
        uint4 vp;
        vp.x = __byte_perm(__byte_perm(a0, a1, 0x0040), 0, 0x5140) << 10;
        vp.y = __byte_perm(__byte_perm(a0, a1, 0x0051), 0, 0x5140) << 10;
        vp.z = __byte_perm(__byte_perm(a0, a1, 0x0062), 0, 0x5140) << 10;
        vp.w = __byte_perm(__byte_perm(a0, a1, 0x0073), 0, 0x5140) << 10;
        *reinterpret_cast<uint4*>(vtab + lane * 4) = vp;
      }
      __syncwarp();
    }
    // ---- rescale O: columns 2t, 2t+1 are rows 2t, 2t+1; group factor 2^(Eold - Enew)
    if (rescale || eold != eref) {
      const uint32_t dl = __vsubus4(eref, eold);
      const float a0 = alpha[2 * t], a1 = alpha[2 * t + 1];
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) {
        const int ex = 127 - (int)((dl >> (8 * G4)) & 0xFFu);
        const float f = ex > 0 ? __uint_as_float((uint32_t)ex << 23) : 0.0f;
        const float f0 = f * a0, f1 = f * a1;
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          o[2 * G4 + jj][0] *= f0;
          o[2 * G4 + jj][1] *= f1;
          o[2 * G4 + jj][2] *= f0;
          o[2 * G4 + jj][3] *= f1;
        }
      }
    }
    // ---- P.V: B fragments (P^T) by ldmatrix.trans; k index 2t+i of k-step kk is
    // token 8t + 4kk + i of the warp, 2t+8+i is 8t + 4kk + 2 + i.
    uint32_t bh[4], bl[4];
    ldsm_x4_trans(bh, lm_addr_hi);  // {kk0 b0, kk0 b1, kk1 b0, kk1 b1}
    ldsm_x4_trans(bl, lm_addr_lo);
    const uint4 vs00 = *reinterpret_cast<const uint4*>(vtab + (4 * t + 0) * 4);  // kk0 b0 pair, groups 0..3
    const uint4 vs01 = *reinterpret_cast<const uint4*>(vtab + (4 * t + 1) * 4);  // kk0 b1
    const uint4 vs10 = *reinterpret_cast<const uint4*>(vtab + (4 * t + 2) * 4);  // kk1 b0
    const uint4 vs11 = *reinterpret_cast<const uint4*>(vtab + (4 * t + 3) * 4);  // kk1 b1
    const uint32_t vsc[2][2][4] = {{{vs00.x, vs00.y, vs00.z, vs00.w}, {vs01.x, vs01.y, vs01.z, vs01.w}},
                                   {{vs10.x, vs10.y, vs10.z, vs10.w}, {vs11.x, vs11.y, vs11.z, vs11.w}}};
    // A fragments: thread t reads word (t&1) of channel rows of page (t>>1): tokens 8(t&1)..+7
    const uint8_t* vrow = vst + (t >> 1) * kBlk + 4 * (t & 1);
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      uint32_t wg[2], wg8[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        wg[u] = *reinterpret_cast<const uint32_t*>(vrow + (32 * G4 + 16 * u + g) * 8);
        wg8[u] = *reinterpret_cast<const uint32_t*>(vrow + (32 * G4 + 16 * u + g + 8) * 8);
      }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t h0 = hmul2(bh[2 * kk], vsc[kk][0][G4]), h1 = hmul2(bh[2 * kk + 1], vsc[kk][1][G4]);
        uint32_t x[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          x[u][0] = e2m1x2_to_f16x2(wg[u], 2 * kk);
          x[u][1] = e2m1x2_to_f16x2(wg8[u], 2 * kk);
          x[u][2] = e2m1x2_to_f16x2(wg[u], 2 * kk + 1);
          x[u][3] = e2m1x2_to_f16x2(wg8[u], 2 * kk + 1);
          mma_f16(o[2 * G4 + u], x[u][0], x[u][1], x[u][2], x[u][3], h0, h1);
        }
        if (kk == 0 ? need_lo0 : need_lo1) {
          const uint32_t l0 = hmul2(bl[2 * kk], vsc[kk][0][G4]), l1 = hmul2(bl[2 * kk + 1], vsc[kk][1][G4]);
#pragma unroll
          for (int u = 0; u < 2; ++u) mma_f16(o[2 * G4 + u], x[u][0], x[u][1], x[u][2], x[u][3], l0, l1);
        }
      }
    }
    __syncwarp();
    if (cc + 2 < n_chunks) {
      fence_proxy_async();
      issue_v(cc + 2);
      ++v_issued;
    }
  }

  if (timed_out) {
    // Flag, then let every copy and MMA this CTA issued land (bounded waits)
    // before shared and tensor memory are reused or freed.
    if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
    for (; s_waited < s_issued; ++s_waited) (void)mbar_wait(&sdone[s_waited & 1], (uint32_t)((s_waited >> 1) & 1));
    for (; k_waited < k_issued; ++k_waited)
      (void)mbar_wait(&kfull[k_waited % kKBufs], (uint32_t)((k_waited / kKBufs) & 1));
    for (; v_waited < v_issued; ++v_waited) (void)mbar_wait(&vfull[v_waited & 1], (uint32_t)((v_waited >> 1) & 1));
  }

  // ---- merge the 4 warps: row sums over the warp's tokens, then O scaled by 2^Eref_G
  float l_row[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float v = l_run[r];
#pragma unroll
    for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
    l_row[r] = v;
  }
  fence_before_sync();
  __syncthreads();
  if (w == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  float* mo = reinterpret_cast<float*>(smem);  // [kWarps][8 rows][D]
  float* mm = mo + kWarps * 8 * D;
  float* ml = mm + kWarps * 8;
  if (lane < 8) {
    float mv = m_run[0], lv = l_row[0];
#pragma unroll
    for (int r = 1; r < 8; ++r)
      if (lane == r) {
        mv = m_run[r];
        lv = l_row[r];
      }
    mm[w * 8 + lane] = mv;
    ml[w * 8 + lane] = lv;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float eg = __uint_as_float(((eref >> (8 * (j >> 1))) & 0xFFu) << 23);
    mo[(w * 8 + 2 * t) * D + 16 * j + g] = o[j][0] * eg;
    mo[(w * 8 + 2 * t + 1) * D + 16 * j + g] = o[j][1] * eg;
    mo[(w * 8 + 2 * t) * D + 16 * j + g + 8] = o[j][2] * eg;
    mo[(w * 8 + 2 * t + 1) * D + 16 * j + g + 8] = o[j][3] * eg;
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

}  // namespace tc

bool tc_path_supported(int D, int G, int T, bool latent) { return D == 128 && !latent && T * G <= 8; }

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(tc::decode_fp4_tc_kernel, tc::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S, a.Hkv, a.B);
  tc::decode_fp4_tc_kernel<<<grid, tc::kThreads, tc::kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
