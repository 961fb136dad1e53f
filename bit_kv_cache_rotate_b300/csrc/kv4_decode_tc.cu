// kv4_decode_tc.cu -- warp-specialised split decode over the 4-bit cache with
// Q.K^T on the block-scaled tcgen05 tensor core (sm_103a): head_dim 128, up to
// 8 query rows per kv head (a decode step of up to 8 query heads per kv head).
//
// "UltraQuant on AMD Instinct", section "What is UltraQuant": the FP4 codes and
// their power-of-two scales go straight into the matrix units, no lookup
// table.  On B300 that is tcgen05.mma kind::mxf4 with UE8M0 block scales, one
// scale per 32 elements along the reduction dimension -- the cache's K format:
//
//   Q.K^T  S[token][col] over M = 128 tokens (8 pages), N = 32, K = 64 channels
//          per instruction.  A = the K codes as cached (8-token x 32-channel
//          tiles are the MMA's core matrices), scale A = the cache's scale
//          bytes, placed in tensor memory per token.  B = q (rotated, times
//          the softmax scale and log2 e) as 8 E2M1 terms with their own UE8M0
//          scale per 32 channels: terms i and i+4 accumulate in column 8i + r
//          (row r), so four MMAs per chunk; the four columns of a row are
//          summed after the load.
//   P.V    f16 warp MMA (m16n8k16), swap-AB: O^T[dims x rows] += V^T P^T.  V
//          codes widened by the hardware E2M1->f16 conversion, the V scale
//          folded into the P fragments (a bf16 path for chunks whose V scales
//          span more binades than f16 factors hold), P as f16 hi + lo read
//          with ldmatrix.trans.
//
// Warp roles (one CTA per (split, kv head, sequence), 5 warps):
//   warp 4      producer: tensor gathers of chunk c (K codes, K scales and V
//               blocks of 8 pages) into stage c % 3, three chunks ahead, and
//               the Q.K^T MMAs of chunk c into S buffer c % 2 (one lane issues);
//   warps 0..3  consumers, warp w = tensor-memory lanes 32w..32w+31 = tokens
//               32w..32w+31 of every chunk (pages 2w, 2w+1): each places its
//               tokens' K scales in tensor memory, loads its tokens' logits,
//               runs its own online softmax and its own P.V, and the four
//               merge once at the end.
// Hand-over is by mbarriers only: full (copies landed), empty (the consumers
// are done with a stage), sfa (scales of A placed), sfull (Q.K^T done) and
// sempty (logits loaded) -- no CTA-wide barrier per chunk.  Every wait is
// bounded and also gives up when another warp has given up (a flag in shared
// memory); a timeout sets KV4_DEVERR_TIMEOUT, the producer waits (bounded) for
// every copy and MMA it issued, and the kernel frees its tensor memory and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace tc {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kConsumers = 4;
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kProducer = kConsumers;            // warp index
constexpr int kChunkPages = 8;                   // 128 tokens: the MMA's M
constexpr int kCodeBytes = kPage * D / 2;        // 1024
constexpr int kBlk = kCodeBytes + kPage * D / 32;  // 1088
constexpr int kStages = 3;
constexpr int kTerms = 8;
constexpr int kTermsN = 4;                       // terms side by side along N
constexpr int kN = 8 * kTermsN;                  // MMA N = 32: column 8i + r holds term (4j + i) of row r
constexpr int kTermGroups = kTerms / kTermsN;    // term groups accumulate along K (j = 0, 1)

// stage: K codes [8 pages][1024] | K scales [8][64] | V blocks [8][1088]
constexpr int kOffSK = 0;
constexpr int kOffSS = kChunkPages * kCodeBytes;
constexpr int kOffSV = kOffSS + kChunkPages * 64;
constexpr int kStageBytes = kOffSV + kChunkPages * kBlk;
constexpr int kOffQ = kStages * kStageBytes;                 // [2 term groups][32 B-rows x 64 B]
constexpr int kQGroup = kN * 64;
constexpr int kOffP = kOffQ + kTermGroups * kQGroup;         // [4 warps][hi, lo][32 tokens][16 B]
constexpr int kOffVTab = kOffP + kConsumers * 1024;          // [4 warps][16 pairs][4 groups] f16x2
constexpr int kOffSfb = kOffVTab + kConsumers * 256;         // [8 terms][8 rows][4] bytes
constexpr int kOffLim = kOffSfb + kTerms * 8 * 4;            // [8] row limits
constexpr int kOffBar = kOffLim + 8 * 4;
constexpr int kNumBars = 2 * kStages + 7;                    // full[3] empty[3] sfa[2] sfull[2] sempty[2] drain
constexpr int kOffFlag = kOffBar + 8 * kNumBars;             // abort flag
constexpr int kSmem = kOffFlag + 16;
static_assert(kStageBytes % 128 == 0 && kOffSS % 128 == 0 && kOffSV % 128 == 0 && kOffQ % 128 == 0,
              "tensor copies land on 128-byte boundaries; MMA operands are 16-byte aligned");
static_assert(kOffBar % 8 == 0, "mbarrier alignment");
static_assert(kSmem <= 227 * 1024 / 3, "three CTAs per SM");
static_assert(kConsumers * 8 * D * 4 + 2 * kConsumers * 8 * 4 <= kOffQ, "the merge reuses the stages");

// tensor memory (128 columns)
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColS = 0;      // [2 buffers][32]
constexpr uint32_t kColSfa = 64;   // [2 buffers][2 k-steps][4]
constexpr uint32_t kColSfb = 80;   // [2 term groups][2 k-steps][4]

// K-major, no swizzle: core matrices of 8 rows x 16 B; LBO (next 32 elements
// along K) = 128 B, SBO (next 8 rows) = sbo; descriptor version 1.
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

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t addr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(v));
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                            int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

// Bounded wait that also gives up as soon as another warp has set the abort
// flag (so one timeout stops every role quickly).  Warp-uniform result.
// Between tries the warp sleeps (32 ns doubling to 256 ns) instead of spinning:
// a spinning warp takes issue slots from the warps that have work.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                              int limit = kSpinLimit) {
  const uint32_t addr = smem_u32(bar);
  bool ok = false;
  uint32_t ns = 32;
  for (int i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) {
      ok = true;
      break;
    }
    if (*abort) break;
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return __all_sync(0xffffffffu, ok);
}

struct Maps {
  CUtensorMap kcodes;  // K blocks, first 1024 bytes of each (128 eight-byte elements)
  CUtensorMap kscale;  // K blocks, the 64 scale bytes (elements 128..135)
  CUtensorMap vblock;  // V blocks, whole (136 elements)
};

// P.V over this warp's 32 tokens for a chunk whose V scales span more binades
// than the f16 factors hold: x = p * 2^(e_v - E_G) in fp32, split as bf16 hi +
// lo, bf16 MMAs (fp32's exponent range).  pf: fp32 P [32 tokens][8 rows];
// vst: the warp's two staged V blocks.  Fragment mapping as in the f16 path:
// k index 2t+i of k-step kk is token 8t + 4kk + i, 2t+8+i is 8t + 4kk + 2 + i.
__device__ __forceinline__ void pv_bf16(float (&o)[8][4], const float* pf, const uint8_t* vst, uint32_t eref,
                                        int g, int t) {
  const uint8_t* vrow = vst + (t >> 1) * kBlk + 4 * (t & 1);
  const uint8_t* vsb = vst + (t >> 1) * kBlk + kCodeBytes;  // scale bytes [16 tokens][4 groups] of page t >> 1
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    float pv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pv[i] = pf[(8 * t + 4 * kk + i) * 8 + g];
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      const int E = (int)((eref >> (8 * G4)) & 0xFFu);
      float x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = pv[i] * pow2_diff(vsb[(8 * (t & 1) + 4 * kk + i) * 4 + G4], E);
      uint32_t h0, l0, h1, l1;
      split_bf16x2(x[0], x[1], h0, l0);
      split_bf16x2(x[2], x[3], h1, l1);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t wg = *reinterpret_cast<const uint32_t*>(vrow + (32 * G4 + 16 * u + g) * 8);
        const uint32_t wg8 = *reinterpret_cast<const uint32_t*>(vrow + (32 * G4 + 16 * u + g + 8) * 8);
        const uint32_t a0 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wg, 2 * kk));
        const uint32_t a1 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wg8, 2 * kk));
        const uint32_t a2 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wg, 2 * kk + 1));
        const uint32_t a3 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wg8, 2 * kk + 1));
        mma_bf16(o[2 * G4 + u], a0, a1, a2, a3, h0, h1);
        mma_bf16(o[2 * G4 + u], a0, a1, a2, a3, l0, l1);
      }
    }
  }
}

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 3)
    decode_fp4_tc_kernel(DecodeArgs a, const __grid_constant__ Maps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tmem_base_s;
  const int s = blockIdx.x, h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = mma::longest_first(a.context_lens, a.B, blockIdx.z);
  const int g = lane >> 2, t = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int R = a.T * G;
  const int L = a.context_lens[b];
  const size_t row0 = (size_t)b * a.T * a.Hq;

  auto row_index = [&](int r) -> size_t { return row0 + (size_t)(r / G) * a.Hq + h * G + (r % G); };
  auto write_empty = [&]() {
    for (int r = w; r < R; r += kConsumers + 1) {
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
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;                    // [3] copies of a chunk landed (1 arrival + bytes)
  uint64_t* empty = bars + kStages;         // [3] the consumers are done with a stage (4 arrivals)
  uint64_t* sfa = bars + 2 * kStages;       // [2] scales of A of a chunk placed (4 arrivals)
  uint64_t* sfull = sfa + 2;                // [2] Q.K^T of a chunk done (commit)
  uint64_t* sempty = sfull + 2;             // [2] logits of a chunk loaded (4 arrivals)
  uint64_t* drain = sempty + 2;             // every MMA issued done (after an abort)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffFlag);
  int* row_lim_s = reinterpret_cast<int*>(smem + kOffLim);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfa[i], kConsumers);
      mbar_init(&sfull[i], 1);
      mbar_init(&sempty[i], kConsumers);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // zero the q operand (rows past R stay zero)
  for (int i = tid; i < kTermGroups * kQGroup / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;
  int n_done = n_chunks;  // chunks the consumers finished (less after an abort)

  if (w == kProducer) {
    // ================================================================ producer
    fence_proxy_async();  // this warp's share of the zeroed q operand, read by the MMA
    int tma_issued = 0, mma_issued = 0;
    // chunk c -> stage c % 3: lanes 0..7 read the page ids, lane 0 issues six
    // tensor gathers (K codes and K scales of the 8 pages by two gathers each,
    // V blocks by two); pages past the split re-read the chunk's first page
    // (their tokens are masked).
    // The page ids (lane i: page i) are loaded one refill ahead by load_page and
    // only checked when the copies are issued, so the load's latency is spent
    // while the producer waits for the MMAs' inputs.
    auto load_page = [&](int c) -> int {
      const int pg = p0 + c * kChunkPages;
      return (c < n_chunks && lane < min(kChunkPages, p1 - pg)) ? table[pg + lane] : 0;
    };
    auto issue_tma = [&](int c, int page) {
      const int pg = p0 + c * kChunkPages;
      const int nv = min(kChunkPages, p1 - pg);
      if (lane < nv && (page < 0 || page >= a.num_pages)) {
        flag_error(a.dev_error, KV4_DEVERR_PAGE);
        page = 0;
      }
      const int row = page * a.Hkv + h;
      const int r0 = __shfl_sync(0xffffffffu, row, 0);
      int r[kChunkPages];
#pragma unroll
      for (int i = 0; i < kChunkPages; ++i) {
        const int ri = __shfl_sync(0xffffffffu, row, i);
        r[i] = i < nv ? ri : r0;
      }
      if (lane == 0) {
        const int st = c % kStages;
        const uint32_t base = sbase + st * kStageBytes;
        mbar_expect_tx(&full[st], (uint32_t)(kChunkPages * (kCodeBytes + 64 + kBlk)));
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          tma_gather4(base + kOffSK + q * 4 * kCodeBytes, &maps.kcodes, 0, r[4 * q], r[4 * q + 1], r[4 * q + 2],
                      r[4 * q + 3], &full[st]);
          tma_gather4(base + kOffSS + q * 4 * 64, &maps.kscale, kCodeBytes / 8, r[4 * q], r[4 * q + 1], r[4 * q + 2],
                      r[4 * q + 3], &full[st]);
          tma_gather4(base + kOffSV + q * 4 * kBlk, &maps.vblock, 0, r[4 * q], r[4 * q + 1], r[4 * q + 2],
                      r[4 * q + 3], &full[st]);
        }
      }
      __syncwarp();
    };
    bool ok = true;
    for (int c = 0; c < min(n_chunks, kStages); ++c) issue_tma(c, load_page(c));
    tma_issued = min(n_chunks, kStages);
    int next_page = load_page(kStages);  // the page ids of the first refill
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int st = c % kStages, bb = c & 1;
      // ---- Q.K^T of chunk c into S buffer c % 2
      ok = wait_or_abort(&full[st], (uint32_t)((c / kStages) & 1), abort_flag) &&
           wait_or_abort(&sfa[bb], (uint32_t)((c >> 1) & 1), abort_flag) &&
           (c < 2 || wait_or_abort(&sempty[bb], (uint32_t)(((c >> 1) + 1) & 1), abort_flag));
      if (!ok) break;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t a_base = sbase + st * kStageBytes + kOffSK;
        const uint32_t b_base = sbase + kOffQ;
#pragma unroll
        for (int tj = 0; tj < kTermGroups; ++tj)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_mxf4(tmem + kColS + kN * bb, smem_desc(a_base + ks * 256, 512),
                     smem_desc(b_base + tj * kQGroup + ks * 256, 512), tmem + kColSfa + bb * 8 + ks * 4,
                     tmem + kColSfb + (tj * 2 + ks) * 4, (tj | ks) != 0);
        commit(&sfull[bb]);
      }
      ++mma_issued;
      __syncwarp();
      // ---- refill the stage of chunk c - 1 once the consumers are done with it
      const int cn = c - 1 + kStages;
      if (c >= 1 && cn < n_chunks) {
        ok = wait_or_abort(&empty[(c - 1) % kStages], (uint32_t)(((c - 1) / kStages) & 1), abort_flag);
        if (!ok) break;
        fence_proxy_async();
        issue_tma(cn, next_page);
        tma_issued = cn + 1;
        next_page = load_page(cn + 1);
      }
    }
    if (!ok) {
      if (lane == 0) {
        *abort_flag = 1;
        flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
      }
    }
    __syncthreads();  // (1) every role has left its loop
    if (*abort_flag) {
      // let every copy and MMA issued land before shared and tensor memory go
      // (bounded; each stage's latest phase is the last chunk issued into it)
      for (int c = max(0, tma_issued - kStages); c < tma_issued; ++c)
        (void)mbar_wait(&full[c % kStages], (uint32_t)((c / kStages) & 1));
      if (lane == 0 && mma_issued > 0) {
        commit(drain);
        (void)mbar_wait(drain, 0u);
      }
      __syncwarp();
    }
    fence_before_sync();
    __syncthreads();  // (2) drained
  } else {
    // ================================================================ consumers
    const uint32_t tmem_lane = tmem + ((uint32_t)(32 * w) << 16);
    // ---- q prologue (rows w, w + 4): rotate (fp32 butterfly), times
    // softmax_scale*log2e/sqrt(D), then 8 E2M1 terms with one UE8M0 scale per
    // 32 channels each; term (4j + i) of row r is B-row 8i + r of term group j
    uint8_t* sfb_s = smem + kOffSfb;  // [term][8 rows][block]
    for (int r = w; r < 8; r += kConsumers) {
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
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        x[0] -= f01.x * up;
        x[1] -= f01.y * up;
        x[2] -= f23.x * up;
        x[3] -= f23.y * up;
        const int tj = term / kTermsN, ti = term % kTermsN;
        uint8_t* dst = smem + kOffQ + tj * kQGroup + (ti * 4 + (lane >> 3)) * 128 + r * 16 + 2 * (lane & 7);
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(c01 | (c23 << 8));
        if ((lane & 7) == 0) sfb_s[(term * 8 + r) * 4 + (lane >> 3)] = (uint8_t)(e + 127);
      }
      if (lane == 0)
        row_lim_s[r] = r < R ? (a.causal ? L - a.T + 1 + r / G : L) : 0x7fffffff;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");  // the four consumer warps
    // scale factors of B into tensor memory, this warp's lane quadrant (B-row
    // n = 8i + r at lane n), all four columns of each (term group, k-step) set
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
    }
    fence_proxy_async();  // q operand written by ordinary stores, read by the MMA
    int row_lim[8];
    int min_limit = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      row_lim[r] = row_lim_s[r];
      min_limit = min(min_limit, row_lim[r]);
    }

    // Scales of A of chunk cc (token 32w + lane) into tensor memory buffer cc % 2
    // after its copies landed; neutral scales past the split or the context.
    auto place_sfa = [&](int cc, int limit) -> bool {
      const int st = cc % kStages;
      if (!wait_or_abort(&full[st], (uint32_t)((cc / kStages) & 1), abort_flag, limit)) return false;
      const int pi = 2 * w + (lane >> 4), tok = lane & 15;
      const int pg = p0 + cc * kChunkPages + pi;
      uint32_t sw = 0x7F7F7F7Fu;
      if (pg < p1 && pg * kPage + tok < L)
        sw = *reinterpret_cast<const uint32_t*>(smem + st * kStageBytes + kOffSS + pi * 64 + tok * 4);
      tmem_st4(tmem_lane + kColSfa + (cc & 1) * 8 + 0, (sw & 0xFFFFu) | 0x7F7F0000u);
      tmem_st4(tmem_lane + kColSfa + (cc & 1) * 8 + 4, (sw >> 16) | 0x7F7F0000u);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfa[cc & 1]);
      return true;
    };

    // ---- per-warp running state
    float o[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
    float m_run[8], l_run[8];
#pragma unroll
    // A finite start for the maximum: the first visible logit of a row always
    // moves it (lazy test below), and p = 2^(s - m) needs no test for an unset m.
    for (int r = 0; r < 8; ++r) {
      m_run[r] = -1.0e30f;
      l_run[r] = 0.0f;
    }
    uint32_t eref = 0;
    uint8_t* pbuf = smem + kOffP + w * 1024;                                  // [hi, lo][32 tokens][16 B]
    uint32_t* vtab = reinterpret_cast<uint32_t*>(smem + kOffVTab + w * 256);  // [16 pairs][4 groups]
    // ldmatrix row address of this lane: matrix mi = lane/8 -> (kstep mi>>1, half mi&1),
    // row r = lane%8 -> token 8*(r>>1) + 4*kstep + 2*half + (r&1)
    const int lm_mi = lane >> 3, lm_r = lane & 7;
    const int lm_tok = 8 * (lm_r >> 1) + 4 * (lm_mi >> 1) + 2 * (lm_mi & 1) + (lm_r & 1);
    const uint32_t lm_addr_hi = smem_u32(pbuf) + lm_tok * 16;
    const uint32_t lm_addr_lo = lm_addr_hi + 32 * 16;

    bool ok = place_sfa(0, first_limit);
    int c = 0;
    for (; c < n_chunks && ok; ++c) {
      const int st = c % kStages, bb = c & 1;
      if (c + 1 < n_chunks && !place_sfa(c + 1, kSpinLimit)) {
        ok = false;
        break;
      }
      // ---- logits of this warp's tokens: column 8i + r holds terms (i, i + 4) of row r
      if (!wait_or_abort(&sfull[bb], (uint32_t)((c >> 1) & 1), abort_flag)) {
        ok = false;
        break;
      }
      fence_after_sync();
      uint32_t dq[32];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
          "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
          : "=r"(dq[0]), "=r"(dq[1]), "=r"(dq[2]), "=r"(dq[3]), "=r"(dq[4]), "=r"(dq[5]), "=r"(dq[6]), "=r"(dq[7]),
            "=r"(dq[8]), "=r"(dq[9]), "=r"(dq[10]), "=r"(dq[11]), "=r"(dq[12]), "=r"(dq[13]), "=r"(dq[14]),
            "=r"(dq[15]), "=r"(dq[16]), "=r"(dq[17]), "=r"(dq[18]), "=r"(dq[19]), "=r"(dq[20]), "=r"(dq[21]),
            "=r"(dq[22]), "=r"(dq[23]), "=r"(dq[24]), "=r"(dq[25]), "=r"(dq[26]), "=r"(dq[27]), "=r"(dq[28]),
            "=r"(dq[29]), "=r"(dq[30]), "=r"(dq[31])
          : "r"(tmem_lane + kColS + kN * bb));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[bb]);
      float sc[8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
        sc[r] = (__uint_as_float(dq[r]) + __uint_as_float(dq[8 + r])) +
                (__uint_as_float(dq[16 + r]) + __uint_as_float(dq[24 + r]));
      const int pg0 = p0 + c * kChunkPages;
      const int nv = min(kChunkPages, p1 - pg0);
      const uint8_t* vst = smem + st * kStageBytes + kOffSV + 2 * w * kBlk;  // this warp's 2 V blocks
      {
        const int pi = 2 * w + (lane >> 4), tok = lane & 15;
        const int pos = (pg0 + pi) * kPage + tok;
        const bool valid = pi < nv && pos < L;
        if ((pg0 + kChunkPages) * kPage > min_limit || nv < kChunkPages) {
#pragma unroll
          for (int r = 0; r < 8; ++r)
            if (!(valid && pos < row_lim[r])) sc[r] = -INFINITY;
        }
      }
      // ---- online softmax, lazy maximum (a row's reference moves only when a
      // logit exceeds it by more than 8, log2 units)
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
        p[r] = ex2(sc[r] - m_run[r]);
        l_run[r] += p[r];
      }

      // ---- V scale table: lane = token of the warp (page lane >> 4), pairs joined
      // by the even lane: vtab[pair][group] = f16x2 2^(e_v - Eref_G) of tokens 2l, 2l+1
      uint32_t eold, enew = 0;
      bool slow;
      {
        const int pj = lane >> 4, tt = lane & 15;
        const bool okv = 2 * w + pj < nv && (pg0 + 2 * w + pj) * kPage + tt < L;
        const uint32_t v = okv ? *reinterpret_cast<const uint32_t*>(vst + pj * kBlk + kCodeBytes + tt * 4) : 0u;
        // V reference exponent per group (Eref), raised only when a chunk exceeds
        // it by more than 7; the f16 factors 2^(e_v - Eref) then lie in
        // [2^-14, 2^7] and p * factor < 2^15.
        eold = eref;
        uint32_t lim = __vaddus4(eref, 0x07070707u);
        if (c == 0 || __any_sync(0xffffffffu, __vcmpgtu4(v, lim) != 0u)) {
          uint32_t cm = v;
#pragma unroll
          for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
          eref = __vmaxu4(eref, cm);
          lim = __vaddus4(eref, 0x07070707u);
        }
        // f16 exponent fields 15 + e_v - Eref (tokens past the context: lim's field)
        const uint32_t av = __vsubus4(0x16161616u, __vsubus4(lim, okv ? v : lim));
        // a zero field: a V scale more than 14 binades below the reference (or an
        // all-zero group): the chunk takes the bf16 path, the reference re-taken
        // from the chunk (each group's largest exponent, at most 90 below the old)
        slow = __any_sync(0xffffffffu, has_zero_byte(av) != 0u);
        if (slow) {
          uint32_t cm = v;
#pragma unroll
          for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
          const uint32_t none = __vcmpeq4(cm, 0u);
          enew = (__vmaxu4(cm, __vsubus4(eold, 0x5A5A5A5Au)) & ~none) | (eold & none);
        } else {
          const uint32_t an = __shfl_down_sync(0xffffffffu, av, 1);  // token 2l + 1
          if ((lane & 1) == 0) {
            uint4 vp;
            vp.x = __byte_perm(__byte_perm(av, an, 0x0040), 0, 0x5140) << 10;
            vp.y = __byte_perm(__byte_perm(av, an, 0x0051), 0, 0x5140) << 10;
            vp.z = __byte_perm(__byte_perm(av, an, 0x0062), 0, 0x5140) << 10;
            vp.w = __byte_perm(__byte_perm(av, an, 0x0073), 0, 0x5140) << 10;
            *reinterpret_cast<uint4*>(vtab + (lane >> 1) * 4) = vp;
          }
        }
      }

      // ---- P rows of this token: f16 hi + lo [token][8 rows] (fp32 on the bf16 path)
      bool need_lo0 = true, need_lo1 = true;
      if (!slow) {
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
        const float pmax =
            fmaxf(fmaxf(fmaxf(p[0], p[1]), fmaxf(p[2], p[3])), fmaxf(fmaxf(p[4], p[5]), fmaxf(p[6], p[7])));
        const uint32_t bigm = __ballot_sync(0xffffffffu, pmax > 0.00390625f);
        need_lo0 = (bigm & 0x0F0F0F0Fu) != 0u;
        need_lo1 = (bigm & 0xF0F0F0F0u) != 0u;
      } else {
        float4* pf = reinterpret_cast<float4*>(pbuf + lane * 32);
        pf[0] = make_float4(p[0], p[1], p[2], p[3]);
        pf[1] = make_float4(p[4], p[5], p[6], p[7]);
      }
      __syncwarp();

      // ---- rescale O: columns 2t, 2t+1 are rows 2t, 2t+1; group factor 2^(Eold - Enew)
      const uint32_t enext = slow ? enew : eref;
      if (__any_sync(0xffffffffu, rescale || eold != enext)) {
        // every lane holds every row's alpha (the warp-wide maximum moved it)
        float al0 = 1.0f, al1 = 1.0f;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (2 * t == r) al0 = alpha[r];
          if (2 * t + 1 == r) al1 = alpha[r];
        }
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) {
          const float f = pow2_diff((eold >> (8 * G4)) & 0xFFu, (int)((enext >> (8 * G4)) & 0xFFu));
          const float f0 = f * al0, f1 = f * al1;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            o[2 * G4 + jj][0] *= f0;
            o[2 * G4 + jj][1] *= f1;
            o[2 * G4 + jj][2] *= f0;
            o[2 * G4 + jj][3] *= f1;
          }
        }
        eref = enext;
      }

      if (slow) {
        pv_bf16(o, reinterpret_cast<const float*>(pbuf), vst, eref, g, t);
      } else {
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
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) {
      if (lane == 0) {
        *abort_flag = 1;
        flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
      }
    }
    n_done = c;
    __syncthreads();  // (1) every role has left its loop
    fence_before_sync();
    __syncthreads();  // (2) the producer drained

    // ---- merge the 4 warps: row sums over the warp's tokens, then O scaled by 2^Eref_G
    float l_row[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v = l_run[r];
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
      l_row[r] = v;
    }
    float* mo = reinterpret_cast<float*>(smem);  // [4 warps][8 rows][D] (the stages are idle now)
    float* mm = mo + kConsumers * 8 * D;
    float* ml = mm + kConsumers * 8;
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
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
    const bool aborted = *abort_flag != 0 || n_done < n_chunks;
    for (int r = w; r < 8; r += kConsumers) {
      if (r >= R) continue;
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) M = fmaxf(M, mm[ww * 8 + r]);
      float wsum = 0.0f, wt[kConsumers];
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) {
        wt[ww] = (M == -INFINITY || mm[ww * 8 + r] == -INFINITY) ? 0.0f : exp2f(mm[ww * 8 + r] - M);
        wsum += wt[ww] * ml[ww * 8 + r];
      }
      if (aborted) wsum = 0.0f;  // a timed-out split contributes nothing
      const size_t rr = row_index(r) * a.S + s;
      const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
      for (int d = lane; d < D; d += 32) {
        float acc = 0.0f;
#pragma unroll
        for (int ww = 0; ww < kConsumers; ++ww) acc = fmaf(wt[ww], mo[(ww * 8 + r) * D + d], acc);
        a.part_o[rr * D + d] = acc * inv;
      }
      if (lane == 0) a.part_lse[rr] = wsum > 0.0f ? (M + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
    }
  }
  fence_after_sync();
  if (w == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace tc

bool tc_path_supported(int D, int G, int T, bool latent) { return D == 128 && !latent && T * G <= 8; }

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) return cudaErrorNotSupported;
  // Each cache as a 2-D tensor of (page, head) blocks: 136 eight-byte elements
  // per row, row stride 1088 bytes; boxes of one row (gather4).  The maps of
  // the caches a host thread used last are kept (address and sizes only).
  struct MapCache {
    const void* k = nullptr;
    const void* v = nullptr;
    cuuint64_t rows = 0;
    tc::Maps maps;
  };
  thread_local MapCache mc;
  const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv;
  if (mc.k != a.k_cache || mc.v != a.v_cache || mc.rows != rows) {
    mc.k = nullptr;
    const cuuint64_t dims[2] = {(cuuint64_t)tc::kBlk / 8, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)tc::kBlk};
    const cuuint32_t estr[2] = {1, 1};
    struct {
      CUtensorMap* map;
      const uint8_t* base;
      cuuint32_t box0;
    } spec[3] = {{&mc.maps.kcodes, a.k_cache, tc::kCodeBytes / 8},
                 {&mc.maps.kscale, a.k_cache, 8},
                 {&mc.maps.vblock, a.v_cache, tc::kBlk / 8}};
    for (auto& sp : spec) {
      const cuuint32_t box[2] = {sp.box0, 1};
      if (encode(sp.map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t*>(sp.base), dims, strides, box,
                 estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    mc.k = a.k_cache;
    mc.v = a.v_cache;
    mc.rows = rows;
  }
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(tc::decode_fp4_tc_kernel, tc::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S, a.Hkv, a.B);
  tc::decode_fp4_tc_kernel<<<grid, tc::kThreads, tc::kSmem, st>>>(a, mc.maps);
  return cudaGetLastError();
}

}  // namespace kv4
