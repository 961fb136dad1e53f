// kv4_decode_mla_tc.cu -- split decode over a 4-bit latent cache on the
// tcgen05 tensor cores (sm_103a): K = V = one 512-value latent row per token,
// up to 16 query rows per latent head.
//
// "GLM-5.3-Flash on MI300X": the 512-value latent row without a RoPE half is
// the MLA workload, and every query head of a sequence reads the same latent
// rows, so each byte of the cache feeds 16 query rows in both products.
// "UltraQuant on AMD Instinct", section "What is UltraQuant": the latent row is
// quantised like any K/V vector (Walsh-Hadamard rotation, E2M1 codes, one
// UE8M0 scale per 32 channels) and the FP4 codes with their power-of-two
// scales go straight into the matrix units.  Per chunk of 128 tokens (8 pages):
//
//   Q.K^T  S[token][col], M = 128 tokens, N = 32, K = 64 channels per MMA,
//          kind::mxf4 block-scaled: A = the cached codes as stored (their
//          8-token x 32-channel tiles are the MMA's core matrices), scale A =
//          the cached UE8M0 bytes, placed in tensor memory per token.  B = q
//          (rotated, times softmax scale and log2 e) as 8 E2M1 terms with one
//          UE8M0 scale per 32 channels each, two terms side by side (column
//          16i + r is term 2p + i of row r) and four passes p accumulating in
//          the same columns: 32 MMAs per chunk.
//   P.V    O^T[channel][row] = V'^T P^T, M = 128 channels (four blocks), N =
//          16 rows, K = 16 tokens per MMA, kind::f16.  A = V' = code * 2^(e -
//          E_c), E_c the chunk's largest exponent of the channel group, widened
//          once per chunk by the converter warps (exact in f16 from 23 binades
//          below E_c; a chunk whose scales span more takes bf16 V' and P);
//          B = P as f16 hi + remainder (two MMAs per k-step).  Each chunk's O^T
//          starts afresh in tensor memory and is added into the running O
//          (registers, fp32) with the softmax and group-reference factors.
//
// Warp roles, one CTA per (split, latent head, sequence), 10 warps, one CTA
// per SM (all of tensor memory):
//   warps 0-3  softmax: thread = token 32w + lane of the chunk; places the
//              chunk's scales of A, loads its logits, runs the online softmax
//              (a lazy maximum shared by the four warps), writes P^T, computes
//              the chunk's V factors, and folds O^T (channels 32w + lane of
//              each block) into registers; at the end writes its channels.
//   warps 4-7  converters: V' of the chunk, 32 tokens at a time, into two
//              alternating tiles (E2M1 -> f16 conversion times the factor,
//              stored token by token: the tile is MN-major).
//   warp 8     copies: 8 pages per chunk (codes and scale bytes separately)
//              into a ring of three stages.
//   warp 9     MMAs (one lane): Q.K^T of chunk c, then P.V of chunk c - 1.
// Hand-over is by mbarriers; every wait is bounded and also gives up when
// another warp has given up (a flag in shared memory).  A timeout sets
// KV4_DEVERR_TIMEOUT; the copy warp waits (bounded) for the copies it issued,
// the MMA warp for its MMAs, and the kernel frees its tensor memory and
// returns without writing its partial.
#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace mlatc {

using namespace kv4::mma;

constexpr int D = 512;
constexpr int kRows = 16;                          // query rows per CTA (MMA N of P.V)
constexpr int kChunkPages = 8;
constexpr int kChunk = kChunkPages * kPage;        // 128 tokens: M of Q.K^T, K of P.V
constexpr int kCodeBytes = kPage * D / 2;          // 4096 per page
constexpr int kScaleBytes = kPage * D / 32;        // 256 per page
constexpr int kBlk = kCodeBytes + kScaleBytes;     // 4352: one (page, head) block
constexpr int kGroups = D / 32;                    // 16 channel groups
constexpr int kStages = 3;
constexpr int kTerms = 8;
constexpr int kPasses = 4;                         // two terms side by side per pass
constexpr int kN = 2 * kRows;                      // Q.K^T N = 32
constexpr int kKSteps = D / 64;                    // 8 MMAs of K = 64 per pass
constexpr int kSub = 32;                           // tokens per V' tile
constexpr int kSubs = kChunk / kSub;               // 4 tiles per chunk

constexpr int kSmWarps = 4;
constexpr int kCvWarps = 4;
constexpr int kCopyWarp = 8;
constexpr int kMmaWarp = 9;                        // Q.K^T issue
constexpr int kPvWarp = 10;                        // P.V issue
constexpr int kStatWarp = 11;                      // chunk scale statistics
constexpr int kThreads = 12 * 32;

// ---- shared memory (bytes)
// stage: codes [8 pages][4096] (the Q.K^T A operand: token octet o at
// o * 2048, channel block k at k * 128) | scale bytes [8 pages][16 tokens][16]
constexpr int kStageCodes = kChunkPages * kCodeBytes;            // 32768
constexpr int kStageBytes = kStageCodes + kChunkPages * kScaleBytes;  // 34816
constexpr int kOffStage = 0;
// q terms, the Q.K^T B operand: pass p = [4 row octets][16 channel blocks][128 B]
constexpr int kQPass = kN * D / 2;                               // 8192
constexpr int kOffQ = kOffStage + kStages * kStageBytes;         // 104448
// V' tiles, the P.V A operand, MN-major (a token's channels contiguous):
// [4 token octets][64 channel octets][8 tokens][8 channels]; channel octets
// (M) 128 B apart, token octets (K) 8 KB apart
constexpr int kVpLbo = (D / 8) * 128;                            // 8192
constexpr int kVpBytes = (kSub / 8) * kVpLbo;                    // 32768
constexpr int kOffVp = kOffQ + kPasses * kQPass;                 // 137216
// P^T, the P.V B operand, MN-major (a token's rows contiguous): [hi, lo]
// [16 token octets][2 row octets][8 tokens][8 rows]; row octets (N) 128 B
// apart, token octets (K) 256 B apart
constexpr int kPLbo = (kRows / 8) * 128;                         // 256
constexpr int kPHalf = (kChunk / 8) * kPLbo;                     // 4096
constexpr int kPBuf = 2 * kPHalf;                                // 8192
constexpr int kOffP = kOffVp + 2 * kVpBytes;                     // 202752
// V factors of a chunk, 2^(e - E_g) as f16 (bf16 when wide) bits:
// [2 chunks][128 tokens][16 groups]
constexpr int kFacBytes = kChunk * kGroups * 2;                  // 4096
constexpr int kOffFac = kOffP + 2 * kPBuf;
// chunk references: [4 chunks][4 words of group exponents E, flags (bit 0:
// wide), 3 spare]
constexpr int kRefRing = 4;
constexpr int kOffRef = kOffFac + 2 * kFacBytes;
// softmax warps' exchange words: [4 warps][16] group bytes and masks, [4
// warps][16] row maxima or sums, [3 chunks][16] the rows' softmax factors
constexpr int kXchWords = 2 * kSmWarps * 16 + 3 * kRows;
constexpr int kOffXch = kOffRef + kRefRing * 8 * 4;
constexpr int kOffBar = kOffXch + kXchWords * 4;
constexpr int kNumBars = 38;
constexpr int kOffAbort = kOffBar + 8 * kNumBars;
constexpr int kSmem = kOffAbort + 16;
// the q-term scale bytes of the prologue [8 terms][16 rows][16 blocks] sit in
// the V' tiles, unused until the first chunk
constexpr int kOffQScale = kOffVp;
static_assert(kStageBytes % 128 == 0 && kOffQ % 1024 == 0 && kOffVp % 128 == 0 && kOffP % 16 == 0 &&
                  kOffRef % 16 == 0 && kOffBar % 8 == 0,
              "operand and copy alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kSmem > 227 * 1024 / 2, "one CTA per SM: the kernel takes all 512 tensor-memory columns");

// ---- tensor memory (512 columns)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // S: [2 buffers][32]
constexpr uint32_t kColSfa = 64;   // scales of A: [2 buffers][8 k-steps][4]
constexpr uint32_t kColSfb = 128;  // scales of B: [4 passes][8 k-steps][4]
constexpr uint32_t kColO = 256;    // O^T of a chunk: [3 buffers][4 channel blocks][16 rows]
constexpr int kOBufs = 3;

// barriers
constexpr int kBarFull = 0;        // [3] a chunk's copies landed (expect_tx)
constexpr int kBarStageEmpty = 3;  // [3] softmax and converter warps done with a stage (8)
constexpr int kBarSfa = 6;         // [2] scales of A placed (4)
constexpr int kBarSFull = 8;       // [2] Q.K^T done (commit)
constexpr int kBarSEmpty = 10;     // [2] logits loaded (4)
constexpr int kBarRefReady = 12;   // [4] a chunk's references published (4)
constexpr int kBarP = 16;          // [2] P^T written (4)
constexpr int kBarVpFull = 18;     // [2] a V' tile written (4)
constexpr int kBarVpEmpty = 20;    // [2] the MMAs reading a V' tile done (commit)
constexpr int kBarPv = 22;         // [3] P.V of a chunk done (commit)
constexpr int kBarOEmpty = 25;     // [3] O^T of a chunk loaded (4)
constexpr int kBarCvDone = 28;     // [4] converter warps done with a chunk (4)
constexpr int kBarDrain = 32;      // [2] every MMA a warp issued done (after a timeout)
constexpr int kBarRefStats = 34;   // [4] a chunk's group references and wide flag written (1)

// No swizzle: core matrices of 8 x 16 B; lbo = next core matrix along K, sbo
// = next core matrix along M (N); descriptor version 1.  K-major: a core
// matrix row is 16 B along K; MN-major: 16 B along M (N), rows along K.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// kind::mxf4 (A = B = E2M1, UE8M0 scales, D fp32), M = 128, N = 32, both K-major.
constexpr uint32_t kIdescQK = (1u << 7) | (1u << 10) | ((uint32_t)(kN >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
// kind::f16 (f16 operands, D fp32), M = 128, N = 16, both MN-major (bits 15,
// 16); the bf16 form (A and B formats 1) for wide chunks.
constexpr uint32_t kIdescPV =
    (1u << 4) | (1u << 15) | (1u << 16) | ((uint32_t)(kRows >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t kIdescPVbf16 = kIdescPV | (1u << 7) | (1u << 10);

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescQK), "r"(sfa), "r"(sfb), "r"(accumulate));
}

__device__ __forceinline__ void mma_pv(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 32 consecutive columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
}

__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(addr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Barrier among the `n` threads of named barrier `id` that also ORs a flag
// over them (warp-aligned: every thread of a taking part warp executes it).
__device__ __forceinline__ bool bar_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// Bounded wait that also gives up as soon as another warp has set the abort
// flag.  Each try suspends the thread until the phase completes or about 1 us
// passes (the hardware wakes it at completion), then looks at the flag.
// Warp-uniform result.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                              int limit = kSpinLimit) {
  const uint32_t addr = smem_u32(bar);
  bool ok = false;
  for (int i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr), "r"(parity), "r"(1000u)
        : "memory");
    if (done) {
      ok = true;
      break;
    }
    if (*abort) break;
  }
  return __all_sync(0xffffffffu, ok);
}

// f16 bits of 2^k for k <= 0 (subnormal below 2^-14, 0 below 2^-24)
__device__ __forceinline__ uint32_t f16_pow2(int k) {
  return k >= -14 ? (uint32_t)(15 + k) << 10 : (k >= -24 ? 1u << (k + 24) : 0u);
}
// bf16 bits of 2^k for k <= 0 (subnormal below 2^-126, 0 below 2^-133)
__device__ __forceinline__ uint32_t bf16_pow2(int k) {
  return k >= -126 ? (uint32_t)(127 + k) << 7 : (k >= -133 ? 1u << (k + 133) : 0u);
}

// One V' tile (tokens 32 j .. 32 j + 31 of the chunk) of converter warp wc.
// Lane l: token 8 o + l % 8 of each token octet o of the tile, 8-channel block
// x = l / 8 of each of the warp's groups 4 wc .. 4 wc + 3: four bytes of codes
// widen to f16, times the token's factor (bf16 for a wide chunk), one 16-byte
// row of V' (the eight lanes of a store phase write one core matrix).
template <bool kWide>
__device__ __forceinline__ void convert_tile(const uint8_t* codes, const uint16_t* fac, uint8_t* vp, int j, int wc,
                                             int lane) {
  // every load of the tile first (the stores below may not be moved above
  // them), then the conversions and the stores
  uint32_t cw[kSub / 8][4];
  uint2 f4[kSub / 8];
#pragma unroll
  for (int ol = 0; ol < kSub / 8; ++ol) {
    const int t = 8 * (kSub / 8 * j + ol) + (lane & 7);  // token of the chunk
    f4[ol] = *reinterpret_cast<const uint2*>(fac + t * kGroups + 4 * wc);
    const uint8_t* cb =
        codes + (t >> 4) * kCodeBytes + ((t >> 3) & 1) * 2048 + (4 * wc) * 128 + (t & 7) * 16 + 4 * (lane >> 3);
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) cw[ol][gi] = *reinterpret_cast<const uint32_t*>(cb + gi * 128);
  }
#pragma unroll
  for (int ol = 0; ol < kSub / 8; ++ol) {
    uint8_t* db = vp + ol * kVpLbo + (16 * wc + (lane >> 3)) * 128 + (lane & 7) * 16;
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      const uint32_t f = __byte_perm(gi < 2 ? f4[ol].x : f4[ol].y, 0u, (gi & 1) ? 0x3232 : 0x1010);
      const uint32_t w = cw[ol][gi];
      uint4 out;
      if (!kWide) {
        out.x = hmul2(e2m1x2_to_f16x2(w, 0), f);
        out.y = hmul2(e2m1x2_to_f16x2(w, 1), f);
        out.z = hmul2(e2m1x2_to_f16x2(w, 2), f);
        out.w = hmul2(e2m1x2_to_f16x2(w, 3), f);
      } else {
        out.x = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(w, 0)), f);
        out.y = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(w, 1)), f);
        out.z = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(w, 2)), f);
        out.w = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(w, 3)), f);
      }
      *reinterpret_cast<uint4*>(db + gi * 4 * 128) = out;
    }
  }
}

// ---------------------------------------------------------------- kernel
__global__ void __launch_bounds__(kThreads, 1) decode_mla_tc_kernel(DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tmem_base_s;
  __shared__ int row_lim_s[kRows];
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int G = a.Hq / a.Hkv;
  const int R = a.T * G;
  const int L = a.context_lens[b];
  const size_t row0 = (size_t)b * a.T * a.Hq;

  auto row_index = [&](int r) -> size_t { return row0 + (size_t)(r / G) * a.Hq + h * G + (r % G); };
  auto write_empty = [&]() {
    for (int r = w; r < R; r += kThreads / 32) {
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
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  uint32_t* ref_s = reinterpret_cast<uint32_t*>(smem + kOffRef);  // [4][8]

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars[kBarFull + i], 1);
      mbar_init(&bars[kBarStageEmpty + i], kSmWarps + kCvWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarSfa + i], kSmWarps);
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarSEmpty + i], kSmWarps);
      mbar_init(&bars[kBarP + i], kSmWarps);
      mbar_init(&bars[kBarVpFull + i], kCvWarps);
      mbar_init(&bars[kBarVpEmpty + i], 1);
      mbar_init(&bars[kBarDrain + i], 1);
    }
    for (int i = 0; i < kOBufs; ++i) {
      mbar_init(&bars[kBarPv + i], 1);
      mbar_init(&bars[kBarOEmpty + i], kSmWarps);
    }
    for (int i = 0; i < kRefRing; ++i) {
      mbar_init(&bars[kBarRefReady + i], kSmWarps);
      mbar_init(&bars[kBarCvDone + i], kCvWarps);
      mbar_init(&bars[kBarRefStats + i], 1);
    }
    *abort_flag = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // zero the q operand (rows past R stay zero)
  for (int i = tid; i < kPasses * kQPass / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;

  // ---- copies: chunk c -> stage c % 3, lane i < 8 copies page i's codes and
  // scale bytes (pages past the split re-read the chunk's first page; their
  // tokens are masked)
  int tma_issued = 0;
  auto issue_copies = [&](int c) {
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
    int page = 0;
    if (lane < nv) {
      page = table[pg + lane];
      if (page < 0 || page >= a.num_pages) {
        flag_error(a.dev_error, KV4_DEVERR_PAGE);
        page = 0;
      }
    }
    const int page0 = __shfl_sync(0xffffffffu, page, 0);
    if (lane >= nv) page = page0;
    const int st = c % kStages;
    uint64_t* bar = &bars[kBarFull + st];
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)(kChunkPages * kBlk));
    __syncwarp();
    if (lane < kChunkPages) {
      const uint8_t* src = a.k_cache + ((size_t)page * a.Hkv + h) * kBlk;
      uint8_t* dst = smem + kOffStage + st * kStageBytes;
      bulk_g2s(dst + lane * kCodeBytes, src, kCodeBytes, bar);
      bulk_g2s(dst + kStageCodes + lane * kScaleBytes, src + kCodeBytes, kScaleBytes, bar);
    }
    __syncwarp();
  };
  if (w == kCopyWarp) {
    fence_proxy_async();
    for (int c = 0; c < min(n_chunks, kStages); ++c) issue_copies(c);
    tma_issued = min(n_chunks, kStages);
  }

  // ---- q prologue (softmax and converter warps, two rows each): rotate
  // (fp32 butterfly over 512), times softmax_scale * log2 e, then 8 E2M1
  // terms with one UE8M0 scale per 32 channels each.  Term t of row r is
  // B-row n = 16 (t & 1) + r of pass t >> 1.  Lane l holds channels
  // 16l .. 16l + 15: half l & 1 of channel block l >> 1.
  uint8_t* qsc = smem + kOffQScale;  // [term][row][block] scale bytes
  if (w < kSmWarps + kCvWarps) {
    for (int r = w; r < kRows; r += kSmWarps + kCvWarps) {
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
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] *= a.qscale;
      }
#pragma unroll 1
      for (int term = 0; term < kTerms; ++term) {
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(x[i]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
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
        uint32_t c8[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t cc = f32x2_to_e2m1x2(x[2 * i] * down, x[2 * i + 1] * down);
          const uint32_t hh = e2m1x2_to_f16x2(cc, 0);
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hh));
          x[2 * i] -= f.x * up;
          x[2 * i + 1] -= f.y * up;
          c8[i >> 2] |= cc << (8 * (i & 3));
        }
        const int n = 16 * (term & 1) + r, blk = lane >> 1;
        uint8_t* dst = smem + kOffQ + (term >> 1) * kQPass + (n >> 3) * (kGroups * 128) + blk * 128 + (n & 7) * 16 +
                       8 * (lane & 1);
        *reinterpret_cast<uint2*>(dst) = make_uint2(c8[0], c8[1]);
        if ((lane & 1) == 0) qsc[(term * kRows + r) * kGroups + blk] = (uint8_t)(e + 127);
      }
      if (lane == 0) row_lim_s[r] = r < R ? (a.causal ? L - a.T + 1 + r / G : L) : 0;
    }
  }
  fence_proxy_async();  // q terms written by ordinary stores, read by the MMA
  __syncthreads();
  // scales of B into tensor memory: B-row n = lane of pass p, k-step k at
  // column kColSfb + 4 (8p + k) (four copies; the MMA reads row n at column
  // + n / 32).  Every softmax warp fills its own lane quadrant.
  if (w < kSmWarps) {
    const int n = lane, r = n & 15, t2 = n >> 4;
#pragma unroll 1
    for (int half = 0; half < 4; ++half) {  // passes 2 half .. : 8 (pass, k-step) pairs per store of 32 columns
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int idx = 8 * half + i, p = idx >> 3, k = idx & 7;
        const int term = 2 * p + t2;
        const uint8_t* sb = qsc + (term * kRows + r) * kGroups + 2 * k;
        const uint32_t word = r < R ? ((uint32_t)sb[0] | ((uint32_t)sb[1] << 8) | 0x7F7F0000u) : 0x7F7F7F7Fu;
        v[4 * i] = v[4 * i + 1] = v[4 * i + 2] = v[4 * i + 3] = word;
      }
      tmem_st32(tmem + ((uint32_t)(32 * w) << 16) + kColSfb + 32 * half, v);
    }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();  // the prologue's scale bytes are dead: the V' tiles may be written
  fence_after_sync();

  int qk_issued = 0, pv_issued = 0;  // for the drain after a timeout
  if (w == kCopyWarp) {
    // ================================================================ copies
    bool ok = true;
    for (int c = kStages; c < n_chunks && ok; ++c) {
      const int st = c % kStages;
      ok = wait_or_abort(&bars[kBarStageEmpty + st], (uint32_t)(((c - kStages) / kStages) & 1), abort_flag);
      if (!ok) break;
      fence_proxy_async();
      issue_copies(c);
      tma_issued = c + 1;
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (w == kMmaWarp) {
    // ================================================================ Q.K^T
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int st = c % kStages, bb = c & 1;
      ok = wait_or_abort(&bars[kBarFull + st], (uint32_t)((c / kStages) & 1), abort_flag,
                         c == 0 ? first_limit : kSpinLimit) &&
           wait_or_abort(&bars[kBarSfa + bb], (uint32_t)((c >> 1) & 1), abort_flag) &&
           (c < 2 || wait_or_abort(&bars[kBarSEmpty + bb], (uint32_t)(((c - 2) >> 1) & 1), abort_flag));
      if (!ok) break;
      fence_after_sync();
      if (lane == 0) {
        const uint32_t a_base = sbase + kOffStage + st * kStageBytes;
#pragma unroll 1
        for (int p = 0; p < kPasses; ++p)
#pragma unroll
          for (int k = 0; k < kKSteps; ++k)
            mma_mxf4(tmem + kColS + kN * bb, smem_desc(a_base + k * 256, 128, 2048),
                     smem_desc(sbase + kOffQ + p * kQPass + k * 256, 128, kGroups * 128),
                     tmem + kColSfa + bb * 32 + 4 * k, tmem + kColSfb + 4 * (8 * p + k), (p | k) != 0);
        commit(&bars[kBarSFull + bb]);
      }
      __syncwarp();
      qk_issued = c + 1;
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (w == kPvWarp) {
    // ================================================================ P.V
    bool ok = true;
    for (int x = 0; x < n_chunks && ok; ++x) {
      const int bx = x & 1, ob = x % kOBufs;
      ok = wait_or_abort(&bars[kBarP + bx], (uint32_t)((x >> 1) & 1), abort_flag, x == 0 ? first_limit : kSpinLimit) &&
           (x < kOBufs || wait_or_abort(&bars[kBarOEmpty + ob], (uint32_t)(((x - kOBufs) / kOBufs) & 1), abort_flag));
      if (!ok) break;
      const bool wide = (ref_s[(x % kRefRing) * 8 + 4] & 1u) != 0u;
      const uint32_t idesc = wide ? kIdescPVbf16 : kIdescPV;
      for (int j = 0; j < kSubs; ++j) {
        const int gj = kSubs * x + j, vb = gj & 1;
        if (!wait_or_abort(&bars[kBarVpFull + vb], (uint32_t)((gj >> 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        fence_after_sync();
        if (lane == 0) {
          const uint32_t vbase = sbase + kOffVp + vb * kVpBytes;
          const uint32_t pbase = sbase + kOffP + bx * kPBuf;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb)
#pragma unroll
            for (int ks = 0; ks < 2; ++ks)
#pragma unroll
              for (int hl = 0; hl < 2; ++hl) {
                const uint64_t da = smem_desc(vbase + (2 * ks) * kVpLbo + (16 * mb) * 128, kVpLbo, 128);
                const uint64_t db = smem_desc(pbase + hl * kPHalf + (4 * j + 2 * ks) * kPLbo, kPLbo, 128);
                mma_pv(tmem + kColO + ob * 64 + mb * 16, da, db, idesc, (j | ks | hl) != 0);
              }
          commit(&bars[kBarVpEmpty + vb]);
          if (j == kSubs - 1) commit(&bars[kBarPv + ob]);
        }
        __syncwarp();
        pv_issued = 1;
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (w == kStatWarp) {
    // ================================================================ statistics
    // Chunk c's group references E (each group's largest visible exponent)
    // and its wide flag (a visible nonzero exponent more than 23 binades below
    // its group's maximum) into reference slot c % 4, once slot c % 4's last
    // reader, the fold of chunk c - 4, is done.  Lane l: tokens 4l .. 4l + 3.
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int st = c % kStages, rx = c % kRefRing;
      ok = wait_or_abort(&bars[kBarFull + st], (uint32_t)((c / kStages) & 1), abort_flag,
                         c == 0 ? first_limit : kSpinLimit) &&
           (c < kRefRing ||
            wait_or_abort(&bars[kBarOEmpty + (c - kRefRing) % kOBufs], (uint32_t)(((c - kRefRing) / kOBufs) & 1),
                          abort_flag));
      if (!ok) break;
      const int pg = p0 + c * kChunkPages;
      uint32_t mx[4] = {0u, 0u, 0u, 0u}, mn[4] = {~0u, ~0u, ~0u, ~0u};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * lane + i, pi = t >> 4, tk = t & 15;
        if (pg + pi < p1 && (pg + pi) * kPage + tk < L) {
          const uint4 sw = *reinterpret_cast<const uint4*>(smem + kOffStage + st * kStageBytes + kStageCodes +
                                                           pi * kScaleBytes + tk * 16);
          const uint32_t sws[4] = {sw.x, sw.y, sw.z, sw.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            mx[q] = __vmaxu4(mx[q], sws[q]);
            mn[q] = __vminu4(mn[q], sws[q] | __vcmpeq4(sws[q], 0u));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) {
          mx[q] = __vmaxu4(mx[q], __shfl_xor_sync(0xffffffffu, mx[q], o2));
          mn[q] = __vminu4(mn[q], __shfl_xor_sync(0xffffffffu, mn[q], o2));
        }
      if (lane == 0) {
        uint32_t wd = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ref_s[rx * 8 + q] = mx[q];
          wd |= __vcmpgtu4(__vsubus4(mx[q], mn[q]), 0x17171717u);
        }
        ref_s[rx * 8 + 4] = wd != 0u ? 1u : 0u;
        mbar_arrive(&bars[kBarRefStats + rx]);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else if (w >= kSmWarps) {
    // ================================================================ converters
    const int wc = w - kSmWarps;
    bool ok = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int st = c % kStages, rx = c % kRefRing;
      ok = wait_or_abort(&bars[kBarFull + st], (uint32_t)((c / kStages) & 1), abort_flag,
                         c == 0 ? first_limit : kSpinLimit) &&
           wait_or_abort(&bars[kBarRefReady + rx], (uint32_t)((c / kRefRing) & 1), abort_flag);
      if (!ok) break;
      const bool wide = (ref_s[rx * 8 + 4] & 1u) != 0u;
      const uint8_t* codes = smem + kOffStage + st * kStageBytes;
      const uint16_t* fac = reinterpret_cast<const uint16_t*>(smem + kOffFac + (c & 1) * kFacBytes);
      for (int j = 0; j < kSubs && ok; ++j) {
        const int gj = kSubs * c + j, vb = gj & 1;
        if (gj >= 2) {
          ok = wait_or_abort(&bars[kBarVpEmpty + vb], (uint32_t)(((gj - 2) >> 1) & 1), abort_flag);
          if (!ok) break;
        }
        uint8_t* vp = smem + kOffVp + vb * kVpBytes;
        if (!wide)
          convert_tile<false>(codes, fac, vp, j, wc, lane);
        else
          convert_tile<true>(codes, fac, vp, j, wc, lane);
        fence_proxy_async();  // V' written by ordinary stores, read by the MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarVpFull + vb]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kBarCvDone + rx]);
        mbar_arrive(&bars[kBarStageEmpty + st]);
      }
    }
    if (!ok && lane == 0) *abort_flag = 1;
  } else {
    // ================================================================ softmax
    const uint32_t tmem_lane = tmem + ((uint32_t)(32 * w) << 16);
    const int m = 32 * w + lane;  // token of the chunk
    uint32_t* xchu = reinterpret_cast<uint32_t*>(smem + kOffXch);         // [4 warps][16]
    float* xch = reinterpret_cast<float*>(smem + kOffXch) + kSmWarps * 16;  // [4 warps][16]
    float* alpha_s = xch + kSmWarps * 16;                                  // [3][16]
    bool ok = true;

    // Chunk x's scale bytes (this thread's token) as the scales of A, into
    // tensor memory buffer x % 2.  Per warp; false when a wait failed.
    auto place_sfa = [&](int x, bool good) -> bool {
      const int st = x % kStages, bx = x & 1;
      if (good)
        good = wait_or_abort(&bars[kBarFull + st], (uint32_t)((x / kStages) & 1), abort_flag,
                             x == 0 ? first_limit : kSpinLimit);
      if (!good) {
        if (lane == 0) *abort_flag = 1;
        return false;
      }
      const int pg = p0 + x * kChunkPages;
      const int pi = m >> 4, tk = m & 15;
      const bool vis = pg + pi < p1 && (pg + pi) * kPage + tk < L;
      uint4 sw = make_uint4(0u, 0u, 0u, 0u);
      if (vis)
        sw = *reinterpret_cast<const uint4*>(smem + kOffStage + st * kStageBytes + kStageCodes + pi * kScaleBytes +
                                             tk * 16);
      const uint32_t sws[4] = {sw.x, sw.y, sw.z, sw.w};
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < kKSteps; ++k) {
        const uint32_t two = vis ? ((sws[k >> 1] >> (16 * (k & 1))) & 0xFFFFu) : 0x7F7Fu;
        v[4 * k] = v[4 * k + 1] = v[4 * k + 2] = v[4 * k + 3] = two | 0x7F7F0000u;
      }
      tmem_st32(tmem_lane + kColSfa + bx * 32, v);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarSfa + bx]);
      return true;
    };

    // This token's V factors of chunk x, 2^(e - E_g) as f16 bits (bf16 when
    // the chunk is wide; 0 if the token is invisible), from the chunk's
    // references (statistics warp) into factor buffer x % 2, once the
    // converters are done with chunk x - 2.  Per warp; false when a wait
    // failed.
    auto publish_ref = [&](int x, bool good) -> bool {
      const int st = x % kStages, rx = x % kRefRing;
      if (good)
        good = wait_or_abort(&bars[kBarRefStats + rx], (uint32_t)((x / kRefRing) & 1), abort_flag);
      if (good && x >= 2)
        good = wait_or_abort(&bars[kBarCvDone + (x - 2) % kRefRing], (uint32_t)(((x - 2) / kRefRing) & 1), abort_flag);
      if (!good) {
        if (lane == 0) *abort_flag = 1;
        return false;
      }
      const int pg = p0 + x * kChunkPages;
      const int pi = m >> 4, tk = m & 15;
      const bool vis = pg + pi < p1 && (pg + pi) * kPage + tk < L;
      uint32_t fw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (vis) {
        const uint4 sw = *reinterpret_cast<const uint4*>(smem + kOffStage + st * kStageBytes + kStageCodes +
                                                         pi * kScaleBytes + tk * 16);
        const uint32_t sws[4] = {sw.x, sw.y, sw.z, sw.w};
        const bool wd = (ref_s[rx * 8 + 4] & 1u) != 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t Eq = ref_s[rx * 8 + q];
          const uint32_t d = __vsubus4(Eq, sws[q]);  // E_g - e >= 0 per group
          // exponent field of 2^-d: 15 - d (f16) or 127 - d (bf16), four groups
          // at once; a factor below the normal range (d > 14 f16, d > 126
          // bf16: rare) takes the scalar form
          const uint32_t top = wd ? 0x7E7E7E7Eu : 0x0E0E0E0Eu;
          if (__vcmpgtu4(d, top) == 0u) {
            const uint32_t fld = __vsubus4(wd ? 0x7F7F7F7Fu : 0x0F0F0F0Fu, d);
            const int sh = wd ? 7 : 10;
            fw[2 * q] = __byte_perm(fld, 0u, 0x5140) << sh;      // groups 4q, 4q + 1
            fw[2 * q + 1] = __byte_perm(fld, 0u, 0x5342) << sh;  // groups 4q + 2, 4q + 3
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = -(int)((d >> (8 * u)) & 0xFFu);
              const uint32_t bits = wd ? bf16_pow2(k) : f16_pow2(k);
              fw[2 * q + (u >> 1)] |= bits << (16 * (u & 1));
            }
          }
        }
      }
      uint4* fd = reinterpret_cast<uint4*>(smem + kOffFac + (x & 1) * kFacBytes + m * kGroups * 2);
      fd[0] = make_uint4(fw[0], fw[1], fw[2], fw[3]);
      fd[1] = make_uint4(fw[4], fw[5], fw[6], fw[7]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarRefReady + rx]);
      return true;
    };

    // running state: lazy row maxima (shared by all four warps), this
    // thread's share of the row sums, O for channels 32w + lane of each block
    float m_run[kRows], l_part[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      m_run[r] = -1.0e30f;
      l_part[r] = 0.0f;
    }
    float o[4][kRows];
#pragma unroll
    for (int mb = 0; mb < 4; ++mb)
#pragma unroll
      for (int r = 0; r < kRows; ++r) o[mb][r] = 0.0f;
    int Rg[4] = {0, 0, 0, 0};  // running reference exponent of group 4 mb + w

    // Fold O^T of chunk x (its references in slot x % 4, its softmax
    // factors in alpha_s[x % 3]) into the running O.
    auto fold = [&](int x) -> bool {
      const int ob = x % kOBufs;
      const float* al = alpha_s + ob * kRows;
      const uint32_t* Ex = ref_s + (x % kRefRing) * 8;
      if (!wait_or_abort(&bars[kBarPv + ob], (uint32_t)((x / kOBufs) & 1), abort_flag)) return false;
      fence_after_sync();
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {  // channel blocks 2hb, 2hb + 1 (32 columns)
        uint32_t v[32];
        tmem_ld32(tmem_lane + kColO + ob * 64 + 32 * hb, v);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int mb = 2 * hb + i, g = 4 * mb + w;
          const int ex = (int)((Ex[g >> 2] >> (8 * (g & 3))) & 0xFFu);
          float gf = 1.0f, cf = 1.0f;
          if (ex > Rg[mb]) {
            gf = pow2_diff((uint32_t)Rg[mb], ex);
            Rg[mb] = ex;
          } else {
            cf = pow2_diff((uint32_t)ex, Rg[mb]);
          }
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            o[mb][r] = fmaf(o[mb][r], al[r] * gf, __uint_as_float(v[16 * i + r]) * cf);
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarOEmpty + ob]);
      return true;
    };

    // A failed wait sets `good` false; the warp then skips the chunk's work
    // (the abort flag ends every other wait at once) and the next barrier,
    // where all four warps take part, turns it into a common exit.
    ok = place_sfa(0, true);
    ok = publish_ref(0, ok);
    ok = !bar_or(1, kSmWarps * 32, !ok);
    bool good = true;
    for (int c = 0; c < n_chunks && ok; ++c) {
      const int st = c % kStages, bb = c & 1;
      // ---- scales of A for chunk c + 1 (its Q.K^T runs while this chunk's softmax does)
      if (c + 1 < n_chunks) good = place_sfa(c + 1, good);
      // ---- logits of this token: column 16i + r holds term pairs (2p + i) of row r
      good = good && wait_or_abort(&bars[kBarSFull + bb], (uint32_t)((c >> 1) & 1), abort_flag);
      if (!good && lane == 0) *abort_flag = 1;
      float sc[kRows];
      if (good) {
        fence_after_sync();
        uint32_t dq[32];
        tmem_ld32(tmem_lane + kColS + kN * bb, dq);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kBarSEmpty + bb]);
          mbar_arrive(&bars[kBarStageEmpty + st]);
        }
        const int pg = p0 + c * kChunkPages;
        const int pos = pg * kPage + m;
        const bool in_split = pg + (m >> 4) < p1;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          sc[r] = __uint_as_float(dq[r]) + __uint_as_float(dq[16 + r]);
          if (!(in_split && pos < row_lim_s[r])) sc[r] = -INFINITY;
        }
      } else {
#pragma unroll
        for (int r = 0; r < kRows; ++r) sc[r] = -INFINITY;
      }
      // ---- lazy maximum, shared by the four warps: a row's reference moves
      // (to the chunk maximum) only when a logit exceeds it by more than 8
      uint32_t over = 0u;
#pragma unroll
      for (int r = 0; r < kRows; ++r) over |= (sc[r] > m_run[r] + 8.0f ? 1u : 0u) << r;
      over = __reduce_or_sync(0xffffffffu, over);
      if (lane == 0) xchu[w * 16 + 8] = over;
      if (bar_or(1, kSmWarps * 32, !good)) {
        ok = false;
        break;
      }
      // from here to the next barrier a failed wait only skips work
      over = xchu[8] | xchu[16 + 8] | xchu[32 + 8] | xchu[48 + 8];
      // this chunk's factors 2^(m_old - m_new), the same in every thread: one
      // thread keeps them for the fold (read after the next barrier)
      const int ab = c % kOBufs;
      if (m == 0)
#pragma unroll
        for (int r = 0; r < kRows; ++r) alpha_s[ab * kRows + r] = 1.0f;
      if (over != 0u) {
        // chunk maxima of the rows that moved (rare: the first chunks and
        // jumps of more than 8)
        float cm[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          cm[r] = sc[r];
#pragma unroll
          for (int o2 = 16; o2 >= 1; o2 >>= 1) cm[r] = fmaxf(cm[r], __shfl_xor_sync(0xffffffffu, cm[r], o2));
        }
        // the exchange words of the previous use are read by now (barrier above)
        if (lane == 0)
#pragma unroll
          for (int r = 0; r < kRows; ++r) xch[w * 16 + r] = cm[r];
        bar_or(1, kSmWarps * 32, false);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (!((over >> r) & 1u)) continue;
          float M = xch[r];
#pragma unroll
          for (int ww = 1; ww < kSmWarps; ++ww) M = fmaxf(M, xch[ww * 16 + r]);
          const float al = ex2(m_run[r] - M);
          m_run[r] = M;
          l_part[r] *= al;
          if (m == 0) alpha_s[ab * kRows + r] = al;
        }
        bar_or(1, kSmWarps * 32, false);  // the maxima are read before the next chunk's writes
      }
      float p[kRows];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        p[r] = ex2(sc[r] - m_run[r]);
        l_part[r] += p[r];
      }
      // ---- P^T of the chunk (buffer c % 2, free once P.V of chunk c - 2 ran):
      // B-row r, token m: row octet r / 8, token octet m / 8
      if (c >= 2) good = good && wait_or_abort(&bars[kBarPv + (c - 2) % kOBufs], (uint32_t)(((c - 2) / kOBufs) & 1),
                                               abort_flag);
      if (!good && lane == 0) *abort_flag = 1;
      const bool wide_c = (ref_s[(c % kRefRing) * 8 + 4] & 1u) != 0u;
      if (good) {
        // token m's 16 rows: row octets 0 and 1 of token octet m / 8, row m % 8
        uint8_t* pb = smem + kOffP + bb * kPBuf + (m >> 3) * kPLbo + (m & 7) * 16;
        uint32_t hw[8], lw[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (!wide_c) {
            float2 hh, ll;
            split_hi_lo2(make_float2(p[2 * i], p[2 * i + 1]), hh, ll);
            hw[i] = pack_f16x2(hh.x, hh.y);
            lw[i] = pack_f16x2(ll.x, ll.y);
          } else {
            split_bf16x2(p[2 * i], p[2 * i + 1], hw[i], lw[i]);
          }
        }
        *reinterpret_cast<uint4*>(pb) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(pb + 128) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        *reinterpret_cast<uint4*>(pb + kPHalf) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        *reinterpret_cast<uint4*>(pb + kPHalf + 128) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
      }
      fence_proxy_async();
      __syncwarp();
      if (good && lane == 0) mbar_arrive(&bars[kBarP + bb]);
      // ---- V factors of chunk c + 1 (the converters start on it)
      if (c + 1 < n_chunks) good = publish_ref(c + 1, good);
      // ---- fold chunk c - 2 (its P.V finished before P^T of chunk c went in)
      if (good && c >= 2) good = fold(c - 2);
      if (!good && lane == 0) *abort_flag = 1;
    }
    ok = ok && good;
    // the last chunk's softmax factors (one thread wrote them) are read after
    // this barrier; then the row sums over the 128 tokens and this thread's
    // channels
    if (!bar_or(1, kSmWarps * 32, !ok)) {
      if (n_chunks >= 2) ok = fold(n_chunks - 2);
      ok = ok && fold(n_chunks - 1);
      if (!ok && lane == 0) *abort_flag = 1;
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        float v = l_part[r];
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
        l_part[r] = v;
      }
      if (lane == 0)
#pragma unroll
        for (int r = 0; r < kRows; ++r) xch[w * 16 + r] = l_part[r];
      if (!bar_or(1, kSmWarps * 32, !ok)) {
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          if (r >= R) continue;
          float l = 0.0f;
#pragma unroll
          for (int ww = 0; ww < kSmWarps; ++ww) l += xch[ww * 16 + r];
          const size_t rr = row_index(r) * a.S + s;
          const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
            const float eg = __uint_as_float((uint32_t)max(Rg[mb], 1) << 23) * (Rg[mb] == 0 ? 0.5f : 1.0f);
            a.part_o[rr * D + 128 * mb + m] = o[mb][r] * eg * inv;
          }
          if (m == 0) a.part_lse[rr] = l > 0.0f ? (m_run[r] + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
      }
    }
  }

  __syncthreads();  // (1) every role has left its loop
  if (*abort_flag) {
    if (tid == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
    // let every copy and MMA issued land before shared and tensor memory go
    if (w == kCopyWarp) {
      for (int c = max(0, tma_issued - kStages); c < tma_issued; ++c)
        (void)mbar_wait(&bars[kBarFull + c % kStages], (uint32_t)((c / kStages) & 1));
    }
    if (w == kMmaWarp && lane == 0 && qk_issued > 0) {
      commit(&bars[kBarDrain]);
      (void)mbar_wait(&bars[kBarDrain], 0u);
    }
    if (w == kPvWarp && lane == 0 && pv_issued > 0) {
      commit(&bars[kBarDrain + 1]);
      (void)mbar_wait(&bars[kBarDrain + 1], 0u);
    }
    __syncwarp();
  }
  fence_before_sync();
  __syncthreads();  // (2) drained
  if (w == 0) {
    fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace mlatc

bool mla_tc_path_supported(int D, int G, int T, bool latent) { return D == 512 && latent && T * G <= 16; }

cudaError_t launch_decode_mla_tc(const DecodeArgs& a, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(mlatc::decode_mla_tc_kernel, mlatc::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S, a.Hkv, a.B);
  mlatc::decode_mla_tc_kernel<<<grid, mlatc::kThreads, mlatc::kSmem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kv4
