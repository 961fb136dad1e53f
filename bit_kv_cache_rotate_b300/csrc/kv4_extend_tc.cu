// kv4_extend_tc.cu -- extend attention over the 4-bit cache on the tcgen05
// tensor cores (sm_103a), head_dim 128, 1, 2, 4 or 8 query heads per kv head.
//
// An extend step is a chunk of new prompt tokens per sequence: T query
// positions attend to the cached prefix and causally to each other ("Agentic
// serving": long shared prefixes, short new turns; the time to first token of
// "Key results").  With 128 query rows per CTA (128 / G positions of G query
// heads each) both products are real tiles, so they go to tcgen05.mma with the
// accumulators in tensor memory:
//
//   Q.K^T  S[row][token] (M = 128 rows, N = 128 tokens = 8 pages, K = 128
//          channels), kind::mxf4 block-scaled ("What is UltraQuant": FP4 codes
//          and power-of-two scales straight into the matrix units).  B = the
//          cache's K codes as stored (its 8-token x 32-channel tiles are the
//          MMA's core matrices, brought in by tensor gathers), scale B = the
//          cache's UE8M0 bytes.  A = q, rotated and times softmax scale and
//          log2 e, as 8 E2M1 terms with one UE8M0 scale per 32 channels each
//          (each term codes the remainder of the ones before it, a factor of
//          at least 4 smaller); the terms accumulate into the same S, 16 MMAs
//          per chunk, and carry q to about 2^-16 of each 32-channel block's
//          largest element (11 terms measured no smaller output error).
//   softmax one thread per row: S comes out of tensor memory row by row; online
//          softmax with a lazy maximum (the reference moves only when a logit
//          exceeds it by more than 8, log2 units).
//   P.V    O[row][dim] (M = 128, N = 128 dims, K = 16 tokens per MMA),
//          kind::f16.  B = V widened to f16 once per chunk by the CUDA cores
//          (hardware E2M1->f16 conversion times 2^(e - E_c), E_c the chunk's
//          largest V scale exponent, so the f16 values are exact from 2^-22 of
//          the chunk maximum up); A = P' = p * 2^(E_c - E_ref) as f16 hi +
//          f16 remainder (lo), two MMAs per k-step, so P carries about 22 bits.
//          E_ref moves (and O is rescaled in tensor memory) only when a chunk's
//          E_c exceeds it by more than 4, or with the softmax reference.
//
// One CTA per (split, position tile, kv head, sequence), 8 warps; 216 KB of
// shared memory and all 512 tensor-memory columns, so one CTA per SM.  The K
// and V pages stream in by tensor gathers three chunks ahead.  The tensor core
// runs the Q.K^T of chunk c + 1 (S is double-buffered in tensor memory) and the
// P.V of chunk c - 1 while the CUDA cores widen V and run the softmax of chunk
// c.  Every wait is bounded; a timeout is agreed at a CTA barrier, flagged as
// KV4_DEVERR_TIMEOUT, and the kernel drains its copies and MMAs, frees its
// tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace ext {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
// single threads that issue the MMAs and the copies: lane 0 of warps 7 and 6,
// which have no scale-factor work in the chunk's serial part
constexpr int kMmaThread = kThreads - 32;
constexpr int kCopyThread = kThreads - 64;
constexpr int kRows = 128;                            // query rows per CTA (MMA M)
constexpr int kChunkPages = 8;
constexpr int kChunk = kChunkPages * kPage;           // 128 tokens (Q.K^T N, P.V K)
constexpr int kTerms = 8;                             // q terms (E2M1 + UE8M0 each)
constexpr int kCodeBytes = kPage * D / 2;             // 1024
constexpr int kBlk = kCodeBytes + kPage * D / 32;     // 1088

// shared memory map (bytes; operand tiles 128-byte aligned)
constexpr int kQTerm = kRows * D / 2;                 // one q term: 128 rows x 64 B
constexpr int kOffQ = 0;                              // [kTerms]
constexpr int kRaw = 3;                               // chunk buffers: copies run 2 chunks ahead of Q.K^T
constexpr int kKC = kChunkPages * kCodeBytes;         // K codes of a chunk
constexpr int kOffKC = kOffQ + kTerms * kQTerm;       // [kRaw]
constexpr int kKS = kChunkPages * 64;                 // K scales of a chunk [8 pages][16 tokens][4]
constexpr int kOffKS = kOffKC + kRaw * kKC;           // [kRaw]
constexpr int kVR = kChunkPages * kBlk;               // V blocks of a chunk, as cached
constexpr int kOffVR = kOffKS + kRaw * kKS;           // [kRaw]
constexpr int kVF = D * kChunk * 2;                   // V' f16, 128 dims x 128 tokens
constexpr int kOffVF = kOffVR + kRaw * kVR;
constexpr int kPF = kRows * kChunk * 2;               // P' f16, 128 rows x 128 tokens
constexpr int kOffP = kOffVF + kVF;                   // [hi, lo]
constexpr int kOffFac = kOffP + 2 * kPF;              // f16 [4 groups][128 tokens] V factors
constexpr int kOffSfa = kOffFac + 4 * kChunk * 2;     // [kTerms][128 rows][4 groups] q scale bytes
constexpr int kOffMisc = kOffSfa + kTerms * kRows * 4;  // [4] per-warp maxima, [4] minima
constexpr int kOffBar = kOffMisc + 64;                // full[kRaw], sdone[2], pvdone, drain
constexpr int kNumBars = kRaw + 4;
constexpr int kSmem = kOffBar + 8 * kNumBars;
static_assert(kOffKC % 1024 == 0 && kOffKS % 128 == 0 && kOffVR % 128 == 0 && kVR % 128 == 0 &&
                  kOffVF % 128 == 0 && kOffP % 128 == 0 && kOffFac % 16 == 0 && kOffBar % 8 == 0,
              "operand and copy alignment");
static_assert(kSmem <= 227 * 1024 && kSmem > 227 * 1024 / 2, "one CTA per SM (all 512 tensor-memory columns)");

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;      // S: [2 buffers][128 columns (tokens)]
constexpr uint32_t kColO = 256;    // O of the current segment of chunks: 128 columns (dims)
constexpr uint32_t kColSfa = 384;  // [kTerms][2 k-steps][4]
constexpr uint32_t kColSfb = 448;  // [kRaw][2 k-steps][4]
static_assert(kColSfa + kTerms * 8 <= kColSfb && kColSfb + kRaw * 8 <= kTmemCols, "tensor memory map");
// The tensor core's own accumulation of O is kept to kFold chunks (kFold * 16
// MMAs): a segment is then added into the running O, held in registers (64
// values per thread), by the CUDA cores (fp32, round to nearest).  One
// accumulator over a 32K context (4096 MMAs) gave sampled output errors up to
// 6e-4 and about 2e-3 over a whole step; with a fold every 8 chunks they stay
// below 5e-5.
constexpr int kFold = 8;

// kind::mxf4 (A = B = E2M1, UE8M0 scales), M = 128, N = 128; kind::f16 (f16
// operands, fp32 accumulate), M = 128, N = 128.  Both K-major.
constexpr uint32_t kIdescQK =
    (1u << 7) | (1u << 10) | ((uint32_t)(kChunk >> 3) << 17) | (1u << 23) | ((uint32_t)(kRows >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | ((uint32_t)(D >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

// K-major, no swizzle: core matrices of 8 rows x 16 B; LBO (next core matrix
// along K) 128 B, SBO (next 8 rows) sbo; descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa, uint32_t sfb,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdescQK), "r"(sfa), "r"(sfb), "r"(accumulate));
}

// The same P.V on bf16 operands (A and B formats 1): chunks whose V exponents
// span more binades than f16 holds.
constexpr uint32_t kIdescPVbf16 = kIdescPV | (1u << 7) | (1u << 10);

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate,
                                        uint32_t idesc = kIdescPV) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_st4(uint32_t addr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3));
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

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int r0, int r1, int r2,
                                            int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

struct Maps {
  CUtensorMap kcodes;  // K blocks, first 1024 bytes of each (128 eight-byte elements)
  CUtensorMap kscale;  // K blocks, the 64 scale bytes (elements 128..135)
  CUtensorMap vblock;  // V blocks, whole (136 elements)
};

// ---------------------------------------------------------------- kernel
// Warp w serves the 32 rows of lane quadrant w % 4 (the tensor-memory lanes it
// may access) and half w / 4 of the columns: tokens 64h .. 64h + 63 of S and
// dims 64h .. 64h + 63 of O.  The two warps of a quadrant exchange their row
// maxima and sums through shared memory.
__global__ void __launch_bounds__(kThreads, 1)
    extend_fp4_tc_kernel(DecodeArgs a, const __grid_constant__ Maps maps) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint32_t tmem_base_s;
  __shared__ float xch_s[2][kRows];
  const int G = a.Hq / a.Hkv;
  const int PT = kRows / G;  // positions per tile
  const int n_tiles = (a.T + PT - 1) / PT;
  const int s = (int)blockIdx.x / n_tiles;
  const int j0 = ((int)blockIdx.x % n_tiles) * PT;
  const int h = blockIdx.y, b = blockIdx.z;
  const int Tc = min(PT, a.T - j0);
  const int R = Tc * G;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int qd = w & 3, hf = w >> 2;
  const int L_seq = a.context_lens[b];
  // tokens visible to the tile's last position; row r (position j0 + r / G)
  // sees the first L - Tc + 1 + r / G of them
  const int L = a.causal ? L_seq - (a.T - Tc) + j0 : L_seq;
  const size_t row0 = ((size_t)b * a.T + j0) * a.Hq;
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
  const int n_chunks = (p1 - p0 + kChunkPages - 1) / kChunkPages;
  const int32_t* table = a.block_tables + (size_t)b * a.max_pages;
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;              // [kRaw]: one chunk's K codes, K scales and V blocks
  uint64_t* sdone = bars + kRaw;      // [2]: Q.K^T into S buffer 0 / 1 complete
  uint64_t* pvdone = bars + kRaw + 2; // P.V of a chunk complete
  uint64_t* drain = bars + kRaw + 3;  // every MMA issued so far complete (after a timeout)
  int* wmax = reinterpret_cast<int*>(smem + kOffMisc);
  int* wmin = wmax + 4;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (w == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_s)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_s;
  const uint32_t tmem_lane = tmem + ((uint32_t)(32 * qd) << 16);

  // chunk c -> buffer c % kRaw: four tensor gathers for K (codes, scales of 8
  // pages), two for V; pages past the split re-read the chunk's first page
  // (masked like tokens past the context).  Issued by thread 0.
  auto load_rows = [&](int c, int (&rows)[kChunkPages]) {
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
#pragma unroll
    for (int i = 0; i < kChunkPages; ++i) {
      int page = 0;
      if (i < nv) {
        page = table[pg + i];
        if (page < 0 || page >= a.num_pages) {
          flag_error(a.dev_error, KV4_DEVERR_PAGE);
          page = 0;
        }
      }
      rows[i] = i < nv ? page * a.Hkv + h : rows[0];
    }
  };
  auto issue = [&](int c, const int (&rows)[kChunkPages]) {
    const int buf = c % kRaw;
    uint64_t* bar = &full[buf];
    mbar_expect_tx(bar, (uint32_t)(kChunkPages * (kCodeBytes + 64 + kBlk)));
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int* r4 = rows + 4 * q;
      tma_gather4(sbase + kOffKC + buf * kKC + q * 4 * kCodeBytes, &maps.kcodes, 0, r4[0], r4[1], r4[2], r4[3], bar);
      tma_gather4(sbase + kOffKS + buf * kKS + q * 4 * 64, &maps.kscale, kCodeBytes / 8, r4[0], r4[1], r4[2], r4[3],
                  bar);
      tma_gather4(sbase + kOffVR + buf * kVR + q * 4 * kBlk, &maps.vblock, 0, r4[0], r4[1], r4[2], r4[3], bar);
    }
  };
  // copies (kCopyThread) and MMAs (kMmaThread) issued, for the drain after a
  // timeout; the copy thread holds the page rows of chunk c + 3 from the start
  // of iteration c, so their loads are long done when the copies go out
  int issued = 0, qk_issued = 0;
  int next_rows[kChunkPages];
  if (tid == kCopyThread) {
    fence_proxy_async();
    for (int c = 0; c < min(n_chunks, kRaw); ++c) {
      load_rows(c, next_rows);
      issue(c, next_rows);
    }
    issued = min(n_chunks, kRaw);
  }

  // ---- q prologue: rotate (fp32 butterfly), times softmax_scale*log2e/sqrt(D),
  // then kTerms E2M1 terms with one UE8M0 scale per 32 channels each.  Row r
  // of term j: core-matrix row group r/8, channel block lane/8, bytes 2*(lane%8).
  uint8_t* sfa_s = smem + kOffSfa;  // [term][row][block]
  for (int r = w; r < kRows; r += kWarps) {
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
      uint8_t* dst = smem + kOffQ + term * kQTerm + ((r >> 3) * 4 + (lane >> 3)) * 128 + (r & 7) * 16 + 2 * (lane & 7);
      *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(c01 | (c23 << 8));
      if ((lane & 7) == 0) sfa_s[(term * kRows + r) * 4 + (lane >> 3)] = (uint8_t)(e + 127);
    }
  }
  __syncthreads();
  // q scale factors into tensor memory, replicated in every lane quadrant:
  // column c0 + i of lane l holds row 32i + l (the MMA reads row m at lane m,
  // column c0 + m/32).
  if (hf == 0) {
#pragma unroll 1
    for (int term = 0; term < kTerms; ++term)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint8_t* sb = sfa_s + (term * kRows + 32 * i + lane) * 4 + 2 * ks;
          v[i] = (uint32_t)sb[0] | ((uint32_t)sb[1] << 8) | 0x7F7F0000u;
        }
        tmem_st4(tmem_lane + kColSfa + (term * 2 + ks) * 4, v[0], v[1], v[2], v[3]);
      }
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  }
  fence_proxy_async();  // q terms written by ordinary stores, read by the MMA

  // this thread's row and column half
  const int my_r = 32 * qd + lane;
  const int my_limit = my_r < R ? (a.causal ? L - Tc + 1 + my_r / G : L) : 0;
  float m_run = -INFINITY;
  float l_half = 0.0f;  // this half's share of the row sum
  float om[64];         // running O of this row's half, summed segments
#pragma unroll
  for (int i = 0; i < 64; ++i) om[i] = 0.0f;
  int e_ref = 0;        // V scale reference (UE8M0 byte value)
  bool timed_out = false;
  int waited_full = 0;
  __half* fac = reinterpret_cast<__half*>(smem + kOffFac);  // [4][128]

  // Wait for chunk c's pages; the warps of half 0 write its K scales into
  // tensor memory (token 32i + lane at column c0 + i of every quadrant).
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;
  auto stage_k = [&](int c) {
    const int rb = c % kRaw;
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
    if (!mbar_wait(&full[rb], (uint32_t)((c / kRaw) & 1), c == 0 ? first_limit : kSpinLimit)) timed_out = true;
    if (hf == 0 && __all_sync(0xffffffffu, !timed_out)) {
      uint32_t v0[4], v1[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int n = 32 * i + lane, pi = n >> 4, tk = n & 15;
        const bool ok = pi < nv && (pg + pi) * kPage + tk < L;
        const uint32_t sw = ok ? *reinterpret_cast<const uint32_t*>(smem + kOffKS + rb * kKS + pi * 64 + tk * 4)
                               : 0x7F7F7F7Fu;
        v0[i] = (sw & 0xFFFFu) | 0x7F7F0000u;
        v1[i] = (sw >> 16) | 0x7F7F0000u;
      }
      tmem_st4(tmem_lane + kColSfb + rb * 8 + 0, v0[0], v0[1], v0[2], v0[3]);
      tmem_st4(tmem_lane + kColSfb + rb * 8 + 4, v1[0], v1[1], v1[2], v1[3]);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
  };
  // Q.K^T of chunk c into S buffer c & 1 (one thread, after a CTA barrier)
  auto issue_qk = [&](int c) {
    const int rb = c % kRaw;
    const uint32_t kb = sbase + kOffKC + rb * kKC;
#pragma unroll
    for (int term = 0; term < kTerms; ++term)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
        mma_mxf4(tmem + kColS + (c & 1) * kChunk, smem_desc(sbase + kOffQ + term * kQTerm + ks * 256, 512),
                 smem_desc(kb + ks * 256, 512), tmem + kColSfa + (term * 2 + ks) * 4,
                 tmem + kColSfb + rb * 8 + ks * 4, (term | ks) != 0);
    commit(&sdone[c & 1]);
    ++qk_issued;
  };

  // chunk 0's Q.K^T goes out before the loop; inside, chunk c + 1's is issued
  // before chunk c's softmax, so the tensor core works while the CUDA cores do
  stage_k(0);
  fence_before_sync();
  if (__syncthreads_or(timed_out)) timed_out = true;
  fence_after_sync();
  // after a timeout the drain waits for chunk 0's copies again (a wait on a
  // completed phase returns at once)
  waited_full = timed_out ? 0 : 1;
  if (!timed_out && tid == kMmaThread) issue_qk(0);

#pragma unroll 1
  for (int c = 0; c < n_chunks && !timed_out; ++c) {
    const int rb = c % kRaw;
    const int pg = p0 + c * kChunkPages;
    const int nv = min(kChunkPages, p1 - pg);
    // ---- next chunk's K; this chunk's V scale bytes (token tid % 128)
    if (c + 1 < n_chunks) stage_k(c + 1);
    if (tid == kCopyThread && c + kRaw < n_chunks) load_rows(c + kRaw, next_rows);
    const int vt = tid & (kChunk - 1);
    const int vpi = vt >> 4, vtk = vt & 15;
    const bool vok = vpi < nv && (pg + vpi) * kPage + vtk < L;
    const uint32_t vsw = vok ? *reinterpret_cast<const uint32_t*>(smem + kOffVR + rb * kVR + vpi * kBlk +
                                                                  kCodeBytes + vtk * 4)
                             : 0u;
    if (hf == 0) {
      uint32_t m4 = __vmaxu4(vsw, vsw >> 16);
      m4 = max(m4 & 0xFFu, (m4 >> 8) & 0xFFu);
      m4 = __reduce_max_sync(0xffffffffu, m4);
      // smallest nonzero exponent (zero bytes: invisible tokens, all-zero groups)
      const uint32_t nz = vsw | __vcmpeq4(vsw, 0u);
      uint32_t n4 = __vminu4(nz, nz >> 16);
      n4 = min(n4 & 0xFFu, (n4 >> 8) & 0xFFu);
      n4 = __reduce_min_sync(0xffffffffu, n4);
      if (lane == 0) {
        wmax[w] = (int)m4;
        wmin[w] = (int)n4;
      }
    }
    fence_before_sync();
    if (__syncthreads_or(timed_out)) {
      timed_out = true;
      break;
    }
    fence_after_sync();
    waited_full = min(n_chunks, c + 2);
    if (tid == kMmaThread && c + 1 < n_chunks) issue_qk(c + 1);
    const int e_c = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
    const int e_lo = min(min(wmin[0], wmin[1]), min(wmin[2], wmin[3]));
    // V reference: set by the first chunk, moved to the chunk's largest
    // exponent when that differs from it by more than 4 either way (at most 90
    // binades down at once, so the rescaled O stays finite; a chunk with no
    // visible nonzero scale leaves it).  Moving down matters after a chunk with
    // a few large values: p' = p * 2^(E_x - E_ref) keeps its precision.
    float o_fac = 1.0f;
    if (c == 0) {
      e_ref = e_c;
    } else if (e_c > e_ref + 4 || (e_c > 0 && e_c < e_ref - 4)) {
      const int e_new = max(e_c, e_ref - 90);
      o_fac = pow2_diff((uint32_t)e_ref, e_new);
      e_ref = e_new;
    }
    // exponent of the chunk's V' (E_x = e_c unless the chunk lies more than 90
    // binades below the reference)
    const int e_x = max(e_c, e_ref - 90);
    // V' holds code * 2^(e - E_x).  As f16 that is exact down to 23 binades
    // below E_x; a chunk whose visible exponents span more ("wide") widens V'
    // and writes P' as bf16 instead (fp32's exponent range) and its P.V runs
    // on bf16 operands.
    const bool wide = e_c - e_lo > 23;
    // V factors 2^(e - E_x) as f16 or bf16 bits (0 for tokens past the split or context)
    if (hf == 0) {
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const int e = (int)((vsw >> (8 * g4)) & 0xFFu) - e_x;  // <= 0
        const float f = (vok && e >= -126) ? __uint_as_float((uint32_t)(127 + e) << 23) : 0.0f;
        if (wide)
          reinterpret_cast<uint16_t*>(fac)[g4 * kChunk + vt] = (uint16_t)(__float_as_uint(f) >> 16);
        else
          fac[g4 * kChunk + vt] = __float2half_rn(f);
      }
    }
    __syncthreads();  // factors visible
    // V' and P' of the previous chunk are read by its P.V, which ran meanwhile
    if (c > 0) {
      if (!mbar_wait(pvdone, (uint32_t)((c - 1) & 1))) timed_out = true;
      fence_after_sync();
    }
    // ---- V' (dim tid % 128, pages 4h .. 4h + 3 of the chunk) -> canonical K-major tile
    // (the f16 and bf16 forms as separate loops: one branch per chunk)
    auto widen_v = [&](auto wide_t) {
      constexpr bool kWide = decltype(wide_t)::value;
      const int d = tid & (D - 1), g4 = d >> 5;
      const uint8_t* vr = smem + kOffVR + rb * kVR + d * 8;
      const uint4* fr = reinterpret_cast<const uint4*>(fac + g4 * kChunk);
#pragma unroll 2
      for (int pp = 0; pp < kChunkPages / 2; ++pp) {
        const int pi = hf * (kChunkPages / 2) + pp;
        const uint2 wv = *reinterpret_cast<const uint2*>(vr + pi * kBlk);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t word = hh ? wv.y : wv.x;
          const uint4 f = fr[pi * 2 + hh];
          uint4 o;
          if (!kWide) {
            o.x = hmul2(e2m1x2_to_f16x2(word, 0), f.x);
            o.y = hmul2(e2m1x2_to_f16x2(word, 1), f.y);
            o.z = hmul2(e2m1x2_to_f16x2(word, 2), f.z);
            o.w = hmul2(e2m1x2_to_f16x2(word, 3), f.w);
          } else {
            o.x = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(word, 0)), f.x);
            o.y = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(word, 1)), f.y);
            o.z = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(word, 2)), f.z);
            o.w = bmul2(f16x2_to_bf16x2(e2m1x2_to_f16x2(word, 3)), f.w);
          }
          *reinterpret_cast<uint4*>(smem + kOffVF + ((d >> 3) * 16 + pi * 2 + hh) * 128 + (d & 7) * 16) = o;
        }
      }
    };
    if (!timed_out) {
      if (wide) widen_v(std::true_type{});
      else widen_v(std::false_type{});
    }
    // ---- S of the chunk
    if (!mbar_wait(&sdone[c & 1], (uint32_t)((c >> 1) & 1))) timed_out = true;
    if (__any_sync(0xffffffffu, timed_out)) timed_out = true;
    fence_after_sync();
    // tokens 0 .. nvr-1 of the chunk are visible to this row (the chunk's
    // positions are consecutive); whole warps with every token visible skip the
    // per-token test
    const int nvr = max(0, min(nv * kPage, my_limit - pg * kPage));
    const bool all_full = __all_sync(0xffffffffu, nvr == kChunk);
    const int lim0 = nvr - 64 * hf;  // visible tokens among this half's columns
    const uint32_t s_addr = tmem_lane + kColS + (c & 1) * kChunk + 64 * hf;
    float cmx = -INFINITY;
    auto row_max = [&](auto masked) {
      constexpr bool M = decltype(masked)::value;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        tmem_ld32(s_addr + 32 * q, sv);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int lim = lim0 - 32 * q;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = __uint_as_float(sv[i]);
          m4[i & 3] = fmaxf(m4[i & 3], (!M || i < lim) ? x : -INFINITY);
        }
        cmx = fmaxf(cmx, fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])));
      }
    };
    if (!timed_out) {
      if (all_full) row_max(std::false_type{});
      else row_max(std::true_type{});
    }
    xch_s[hf][my_r] = cmx;
    if (__syncthreads_or(timed_out)) {
      timed_out = true;
      break;
    }
    cmx = fmaxf(xch_s[0][my_r], xch_s[1][my_r]);
    const float m_new = cmx > m_run + 8.0f ? cmx : m_run;
    const float alpha = m_new == m_run ? 1.0f : ex2(m_run - m_new);
    m_run = m_new;
    // p' = 2^(s - m + E_x - E_ref): the V factor folded into the exponent (a
    // row with nothing visible yet gets p' = 0)
    const float shift = m_new == -INFINITY ? -INFINITY : (float)(e_x - e_ref) - m_new;
    const float2 sh2 = make_float2(shift, shift);
    float2 ls2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
    auto write_p = [&](auto masked, auto wide_t) {
      constexpr bool M = decltype(masked)::value;
      constexpr bool kWide = decltype(wide_t)::value;
#pragma unroll 1
      for (int q = 0; q < 2; ++q) {
        uint32_t sv[32];
        tmem_ld32(s_addr + 32 * q, sv);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int lim = lim0 - 32 * q;
#pragma unroll
        for (int o8 = 0; o8 < 4; ++o8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            const int i = o8 * 8 + i2 * 2;
            float2 x = make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
            if (M) {
              x.x = i < lim ? x.x : -INFINITY;
              x.y = i + 1 < lim ? x.y : -INFINITY;
            }
            const float2 t = __fadd2_rn(x, sh2);
            const float2 pp = make_float2(ex2(t.x), ex2(t.y));
            ls2[i2 & 1] = __fadd2_rn(ls2[i2 & 1], pp);
            if (!kWide) {
              hw[i2] = pack_f16x2(pp.x, pp.y);
              const float2 hf2 = __half22float2(*reinterpret_cast<const __half2*>(&hw[i2]));
              const float2 lo = __fadd2_rn(pp, make_float2(-hf2.x, -hf2.y));
              lw[i2] = pack_f16x2(lo.x, lo.y);
            } else {
              split_bf16x2(pp.x, pp.y, hw[i2], lw[i2]);
            }
          }
          const int k8 = hf * 8 + q * 4 + o8;  // token octet
          const int off = ((my_r >> 3) * 16 + k8) * 128 + (my_r & 7) * 16;
          *reinterpret_cast<uint4*>(smem + kOffP + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(smem + kOffP + kPF + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    };
    if (!timed_out) {
      if (!wide) {
        if (all_full) write_p(std::false_type{}, std::false_type{});
        else write_p(std::true_type{}, std::false_type{});
      } else {
        if (all_full) write_p(std::false_type{}, std::true_type{});
        else write_p(std::true_type{}, std::true_type{});
      }
    }
    const float lsum = (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
    // l in the units of p (not p'): p = p' * 2^(E_ref - E_x), E_ref - E_x in [-4, 30]
    l_half = l_half * alpha + lsum * __uint_as_float((uint32_t)(127 + e_ref - e_x) << 23);
    // ---- fold the segment into the running O (this half's dims): at the end
    // of a segment, and whenever the softmax or V reference moved (the fold
    // applies the factor)
    const float f_row = alpha * o_fac;
    if (c > 0 && !timed_out && __any_sync(0xffffffffu, f_row != 1.0f || c % kFold == 0)) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t ov[32];
        tmem_ld32(tmem_lane + kColO + 64 * hf + 32 * q, ov);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          om[32 * q + i] = (om[32 * q + i] + __uint_as_float(ov[i])) * f_row;
          ov[i] = 0u;
        }
        tmem_st32(tmem_lane + kColO + 64 * hf + 32 * q, ov);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    fence_proxy_async();  // P' and V' written by ordinary stores, read by the MMA
    fence_before_sync();
    if (__syncthreads_or(timed_out)) {
      timed_out = true;
      break;
    }
    fence_after_sync();
    // ---- P.V of the chunk; the chunk's buffers are refilled with chunk c + kRaw
    if (tid == kMmaThread) {
#pragma unroll
      for (int ks = 0; ks < kChunk / 16; ++ks) {
        const uint64_t vd = smem_desc(sbase + kOffVF + ks * 256, 2048);
        const uint32_t idesc = wide ? kIdescPVbf16 : kIdescPV;
        mma_f16(tmem + kColO, smem_desc(sbase + kOffP + ks * 256, 2048), vd, (c | ks) != 0, idesc);
        mma_f16(tmem + kColO, smem_desc(sbase + kOffP + kPF + ks * 256, 2048), vd, 1, idesc);
      }
      commit(pvdone);
    }
    if (tid == kCopyThread && c + kRaw < n_chunks) {
      fence_proxy_async();
      issue(c + kRaw, next_rows);
      issued = c + kRaw + 1;
    }
  }
  // the last P.V
  if (!timed_out) {
    const bool ok = mbar_wait(pvdone, (uint32_t)((n_chunks - 1) & 1));
    fence_after_sync();
    if (__syncthreads_or(!ok)) timed_out = true;
  }

  if (timed_out) {
    // Stop, but let every copy and MMA this CTA issued finish before the
    // shared and tensor memory are released (each wait again bounded): the
    // copies by their own barriers, the MMAs by one more commit.
    if (tid == kCopyThread) {
      flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
      for (int c = waited_full; c < issued; ++c) (void)mbar_wait(&full[c % kRaw], (uint32_t)((c / kRaw) & 1));
    }
    if (tid == kMmaThread && qk_issued > 0) {
      commit(drain);
      (void)mbar_wait(drain, 0u);
    }
    fence_before_sync();
    __syncthreads();
  } else {
    // ---- this split's output of row my_r, dims 64h .. 64h + 63:
    // O * 2^(E_ref - 127) / l (rotated space); the loads are warp-collective,
    // rows past R only skip the stores
    xch_s[hf][my_r] = l_half;
    __syncthreads();
    const float l_row = xch_s[0][my_r] + xch_s[1][my_r];
    const bool valid_row = my_r < R;
    const size_t rr = valid_row ? row_index(my_r) * a.S + s : 0;
    float* dst = a.part_o + rr * D + 64 * hf;
    const bool any = l_row > 0.0f;
    const float sc = any ? __uint_as_float((uint32_t)e_ref << 23) / l_row : 0.0f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t ov[32];
      tmem_ld32(tmem_lane + kColO + 64 * hf + 32 * q, ov);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (valid_row) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 o4;
          o4.x = (om[32 * q + i] + __uint_as_float(ov[i])) * sc;
          o4.y = (om[32 * q + i + 1] + __uint_as_float(ov[i + 1])) * sc;
          o4.z = (om[32 * q + i + 2] + __uint_as_float(ov[i + 2])) * sc;
          o4.w = (om[32 * q + i + 3] + __uint_as_float(ov[i + 3])) * sc;
          *reinterpret_cast<float4*>(dst + 32 * q + i) = o4;
        }
      }
    }
    if (valid_row && hf == 0) a.part_lse[rr] = any ? (m_run + log2f(l_row)) * 0.69314718055994531f : -INFINITY;
    fence_before_sync();
    __syncthreads();
  }
  if (w == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace ext

bool extend_tc_supported(int D, int G, int T, bool latent) {
  return D == 128 && !latent && (G == 1 || G == 2 || G == 4 || G == 8) && T * G > kTileRows;
}

cudaError_t launch_extend_tc(const DecodeArgs& a, cudaStream_t st) {
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
  // per row, row stride 1088 bytes.  Boxes of one row (gather4).  As in the
  // decode launcher, the maps of the caches a host thread used last are kept.
  struct MapCache {
    const void* k = nullptr;
    const void* v = nullptr;
    cuuint64_t rows = 0;
    ext::Maps maps;
  };
  thread_local MapCache mc;
  const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv;
  if (mc.k != a.k_cache || mc.v != a.v_cache || mc.rows != rows) {
    mc.k = nullptr;
    const cuuint64_t dims[2] = {(cuuint64_t)ext::kBlk / 8, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ext::kBlk};
    const cuuint32_t estr[2] = {1, 1};
    struct {
      CUtensorMap* map;
      const uint8_t* base;
      cuuint32_t box0;
    } spec[3] = {{&mc.maps.kcodes, a.k_cache, ext::kCodeBytes / 8},
                 {&mc.maps.kscale, a.k_cache, 8},
                 {&mc.maps.vblock, a.v_cache, ext::kBlk / 8}};
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
  const ext::Maps& maps = mc.maps;
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(ext::extend_fp4_tc_kernel, ext::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const int G = a.Hq / a.Hkv;
  const int PT = ext::kRows / G;
  const dim3 grid(a.S * ((a.T + PT - 1) / PT), a.Hkv, a.B);
  ext::extend_fp4_tc_kernel<<<grid, ext::kThreads, ext::kSmem, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace kv4
