// kv4_decode_mma.cu -- tensor-core split decode over the 4-bit cache (sm_103a).
//
// "UltraQuant on AMD Instinct", section "What is UltraQuant": the codes stay
// FP4 until the matrix units; the power-of-two scale is applied as part of
// the multiply, no lookup table.  On B300 the warp-level tensor instructions
// take f16 (or e4m3, measured at two f16 MMAs plus operand conversions and
// adds each), so the codes are widened to f16 on the fly by the hardware
// E2M1->f16 conversion, which is exact:
//
//   Q.K^T   f16 MMA (m16n8k16).  A K byte (two codes) becomes an f16x2 pair
//           of the code values in one conversion.  q (rotated in fp32,
//           scaled per row by a power of two) is split into an f16 hi part
//           (MMA row g) and the f16-rounded remainder (row g+8), so the two
//           rows' sum resolves q to about 2^-22 of its largest element.
//           Each 32-channel group accumulates separately and is multiplied by
//           its UE8M0 scale 2^e (a float built from the scale byte).
//   P.V     f16 MMA (m16n8k16), swap-AB: O^T[dims x rows] += V^T P^T.  V codes
//           are widened the same way; the V scale enters as 2^(e_v - Eref_G)
//           multiplied into the P fragments of group G, Eref_G being a per-
//           warp reference exponent (O rows of the group are rescaled when it
//           rises).  P is split into f16 hi + lo parts (p rounded to f16
//           and the rounded remainder), so P.V carries about 22 bits of P.
//
// Work split: one CTA per (split, kv head, sequence); 4 consumer warps each
// own every 4th chunk of 4 pages (64 tokens) of the split, with their own
// online-softmax state, and merge at the end.  Each warp streams its chunks
// with two tensor gathers (TMA cp.async.bulk.tensor tile::gather4: the 4 K and
// the 4 V page blocks of a chunk, each block one row of a 2-D tensor map) into
// a private shared-memory stage completed through an mbarrier, refilling the
// stage as soon as it is consumed.
// Four CTAs share an SM (registers capped at 128 per thread), so sixteen
// warps' copies and math overlap; one stage per warp measured faster than
// two stages at two CTAs per SM.  Every wait is bounded: on timeout the
// kernel flags KV4_DEVERR_TIMEOUT and stops.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <mutex>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace fast {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kPagesPerChunk = 4;
constexpr int kBlk = kPage * D / 2 + kPage * D / 32;  // 1088 bytes per (page, head) block
constexpr int kCodeBytes = kPage * D / 2;            // 1024
constexpr int kBlkStride = 1088;                     // smem stride between staged K blocks
constexpr int kVStride = 1088;                       // smem stride between staged V blocks (gathered rows are contiguous)
// K blocks then V blocks; a multiple of 128 bytes (tensor copies land on 128-byte boundaries)
constexpr int kStageBytes = (kPagesPerChunk * (kBlkStride + kVStride) + 127) / 128 * 128;
constexpr int kStages = 1;
// Scale tables, rows padded so the four t-lanes of a quad hit distinct banks.
constexpr int kKTabPage = 272;                     // fp32 [8 token pairs][4 groups][2 tokens] + pad
constexpr int kVTabPage = 160;                     // f16x2 [4 groups][8 token pairs] + pad
constexpr int kKTab = kPagesPerChunk * kKTabPage;
constexpr int kVTab = kPagesPerChunk * kVTabPage;
constexpr int kTabBytes = kKTab + kVTab;
constexpr int kQBytes = 8 * 2 * D * 2;             // f16 q per 8-row block [8 rows][hi, lo][128 ch]
// The q terms (prologue only) alias the scale tables; with several row blocks
// the shared area grows to hold them.
__host__ __device__ constexpr int tab_area(int RB) {
  return kWarps * kTabBytes > RB * kQBytes ? kWarps * kTabBytes : RB * kQBytes;
}
// q A-fragments, [row block][group][k-step][lane] uint4, read per use:
// keeping them in registers (32 per thread per block) spilled at the
// 128-register cap of four CTAs/SM.
__host__ __device__ constexpr int qfrag_off(int RB) {
  return kWarps * kStages * kStageBytes + tab_area(RB) + 8 * kWarps * kStages;
}
__host__ __device__ constexpr int smem_bytes(int RB) { return qfrag_off(RB) + RB * 4 * 2 * 32 * 16; }

template <int RB>
struct Smem {
  uint8_t* base;
  __device__ uint8_t* stage(int w, int s) const { return base + (w * kStages + s) * kStageBytes; }
  __device__ uint8_t* tabs(int w) const { return base + kWarps * kStages * kStageBytes + w * kTabBytes; }
  __device__ float* ktab(int w) const { return reinterpret_cast<float*>(tabs(w)); }
  __device__ uint32_t* vtab(int w) const { return reinterpret_cast<uint32_t*>(tabs(w) + kKTab); }
  __device__ uint8_t* qterms() const { return tabs(0); }  // prologue only
  __device__ uint64_t* bars() const {
    return reinterpret_cast<uint64_t*>(base + kWarps * kStages * kStageBytes + tab_area(RB));
  }
};

// P.V of one chunk for chunks whose V scales span more binades than the f16
// factors hold (a V scale more than 14 binades below the group reference).
// The scale is folded into P in fp32, x = p * 2^(e_v - E_G) with E_G the
// group's reference (the chunk's largest V exponent), and x and the V codes
// go through bf16 MMAs: bf16 keeps fp32's exponent range, so every token's
// value survives down to 2^-126 of the reference; x carries about 16
// significant bits as bf16 hi + lo.  vbase: the staged V block of page t
// (thread quad index); same fragment layout as the f16 path.
template <int RB>
__device__ __forceinline__ void pv_bf16(float (&o)[RB][8][4], const float2 (&p)[RB][8], const uint8_t* vbase,
                                        uint32_t eref, int g) {
  uint32_t sw[16];  // the V scale words of the page's 16 tokens, 4 groups each
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 x = *reinterpret_cast<const uint4*>(vbase + kCodeBytes + 16 * i);
    sw[4 * i] = x.x;
    sw[4 * i + 1] = x.y;
    sw[4 * i + 2] = x.z;
    sw[4 * i + 3] = x.w;
  }
#pragma unroll
  for (int G4 = 0; G4 < 4; ++G4) {
    const int E = (int)((eref >> (8 * G4)) & 0xFFu);
    const uint2 rA0 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + g) * (kPage / 2));
    const uint2 rB0 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + g + 8) * (kPage / 2));
    const uint2 rA1 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + 16 + g) * (kPage / 2));
    const uint2 rB1 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + 16 + g + 8) * (kPage / 2));
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int b0 = (2 * c4) & 3, b1 = (2 * c4 + 1) & 3;
      const uint32_t wA0 = c4 < 2 ? rA0.x : rA0.y, wB0 = c4 < 2 ? rB0.x : rB0.y;
      const uint32_t wA1 = c4 < 2 ? rA1.x : rA1.y, wB1 = c4 < 2 ? rB1.x : rB1.y;
      const uint32_t x00 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wA0, b0)), x01 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wB0, b0));
      const uint32_t x02 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wA0, b1)), x03 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wB0, b1));
      const uint32_t x10 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wA1, b0)), x11 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wB1, b0));
      const uint32_t x12 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wA1, b1)), x13 = f16x2_to_bf16x2(e2m1x2_to_f16x2(wB1, b1));
      float f[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = pow2_diff((sw[4 * c4 + i] >> (8 * G4)) & 0xFFu, E);
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        uint32_t h01, l01, h23, l23;
        split_bf16x2(p[rb][2 * c4].x * f[0], p[rb][2 * c4].y * f[1], h01, l01);
        split_bf16x2(p[rb][2 * c4 + 1].x * f[2], p[rb][2 * c4 + 1].y * f[3], h23, l23);
        mma_bf16(o[rb][2 * G4], x00, x01, x02, x03, h01, h23);
        mma_bf16(o[rb][2 * G4 + 1], x10, x11, x12, x13, h01, h23);
        mma_bf16(o[rb][2 * G4], x00, x01, x02, x03, l01, l23);
        mma_bf16(o[rb][2 * G4 + 1], x10, x11, x12, x13, l01, l23);
      }
    }
  }
}

// Share of a row's running sum above which a token keeps the lo part of P:
// 2^-4 while every V group reference is at most 2^1 (|v| < 12), a quarter of
// that per binade above, so the error the other tokens' f16 rounding leaves
// (about 2^-11 |v| sqrt(share)) stays the same for any V magnitude.
__device__ __forceinline__ float lo_share_of(uint32_t eref) {
  uint32_t em = __vmaxu4(eref, eref >> 16);
  em = max(em & 0xFFu, (em >> 8) & 0xFFu);
  const int k = min(120, 4 + 2 * max(0, (int)em - 128));
  return __uint_as_float((uint32_t)(127 - k) << 23);
}

// ---------------------------------------------------------------- kernel
// Rows: the R = T*G query rows of one kv head, R <= 8 * RB (row r -> position
// r / G, query head h*G + r % G), in RB blocks of 8 MMA rows; unused rows
// carry zero q and are never written.  Each K and V fragment is widened once
// and used by every row block (a T = 3 verify step shares the decode work of
// its three positions).
template <int RB, bool FLAT>
__global__ void __launch_bounds__(kThreads, RB == 1 ? 4 : 2)
    decode_fp4_mma_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<RB> sm{smem_raw};
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.Hq / a.Hkv;
  uint64_t* bars = sm.bars();  // [kWarps][kStages]

  // ---- barriers, once: a warp's k-th chunk (over all its units) uses stage
  // k % kStages with phase (k / kStages) & 1
  if (lane == 0)
    for (int i = 0; i < kStages; ++i) mbar_init(&bars[w * kStages + i], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  int it_base = 0;  // this warp's chunks in earlier units
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;

  // ---- flat mode: CTA i takes the i-th equal part of the flat range of 4-page
  // chunks in (sequence, kv head, chunk) order and runs each (sequence, kv
  // head) run of it as one unit, writing that unit's partial in slot (CTA -
  // the unit's first CTA).  The part size keeps every (sequence, kv head)
  // within S CTAs; the CTA holding its last chunk writes the unused slots as
  // empty partials, so the combine merges them like the split form's.
  __shared__ long long fl_cur, fl_hi, fl_per;
  __shared__ int fl_unit[6];  // b, h, first chunk, end chunk, slot, first empty slot
  __shared__ int fl_stop;
  auto fl_valid = [&](int Ls) { return Ls >= a.T && Ls <= a.max_pages * kPage; };
  auto fl_chunks = [&](int Ls) { return ((Ls + kPage - 1) / kPage + kPagesPerChunk - 1) / kPagesPerChunk; };
  if constexpr (FLAT) {
    if (w == 0) {
      long long C = 0;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int bq = b0 + lane;
        const int Ls = bq < a.B ? a.context_lens[bq] : 0;
        const int nc = bq < a.B && fl_valid(Ls) ? fl_chunks(Ls) : 0;
        C += (long long)__reduce_add_sync(0xffffffffu, (unsigned)nc) * a.Hkv;
      }
      if (lane == 0) {
        const long long nc_max = (a.max_pages + kPagesPerChunk - 1) / kPagesPerChunk;
        const long long even = (C + gridDim.x - 1) / gridDim.x;
        const long long bound = (nc_max + a.S - 2) / (a.S - 1);
        const long long per = even > bound ? even : bound;
        fl_per = per > 0 ? per : 1;
        fl_cur = (long long)blockIdx.x * fl_per;
        fl_hi = fl_cur + fl_per < C ? fl_cur + fl_per : C;
        fl_stop = 0;
      }
    }
    // CTA 0: sequences whose context is out of range get empty partials
    if (blockIdx.x == 0) {
      const int R0 = a.T * G;
      for (int bq = w; bq < a.B; bq += kWarps) {
        if (fl_valid(a.context_lens[bq])) continue;
        if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
        for (int hh = 0; hh < a.Hkv; ++hh)
          for (int r = 0; r < R0; ++r) {
            const size_t row = ((size_t)bq * a.T + r / G) * a.Hq + hh * G + (r % G);
            for (int sl = 0; sl < a.S; ++sl) {
              for (int d = lane; d < D; d += 32) a.part_o[(row * a.S + sl) * D + d] = 0.0f;
              if (lane == 0) a.part_lse[row * a.S + sl] = -INFINITY;
            }
          }
      }
    }
    __syncthreads();
  }

  for (;;) {  // units: one in the split form, the runs of this CTA's part in flat mode
  int b, h, s, c_first = 0, c_end = 0, empty_from = 0;
  if constexpr (FLAT) {
    if (fl_cur >= fl_hi || fl_stop) break;
    // the (sequence, kv head) holding chunk fl_cur
    if (w == 0) {
      const long long cur = fl_cur, hi = fl_hi, per = fl_per;
      long long base = 0;
      bool found = false;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int bq = b0 + lane;
        const int Ls = bq < a.B ? a.context_lens[bq] : 0;
        const int nc = bq < a.B && fl_valid(Ls) ? fl_chunks(Ls) : 0;
        int incl = nc;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o2);
          if (lane >= o2) incl += y;
        }
        const long long bb = base + (long long)(incl - nc) * a.Hkv;  // sequence bq's first chunk
        const bool mine = nc > 0 && cur >= bb && cur < bb + (long long)nc * a.Hkv;
        const uint32_t m = __ballot_sync(0xffffffffu, mine);
        if (mine) {
          const int hh = (int)((cur - bb) / nc);
          const long long ps = bb + (long long)hh * nc, pe = ps + nc;
          const long long e1 = hi < pe ? hi : pe;
          const long long first_cta = ps / per, last_cta = (pe - 1) / per;
          fl_unit[0] = bq;
          fl_unit[1] = hh;
          fl_unit[2] = (int)(cur - ps);
          fl_unit[3] = (int)(e1 - ps);
          fl_unit[4] = (int)((long long)blockIdx.x - first_cta);
          fl_unit[5] = (long long)blockIdx.x == last_cta ? (int)(last_cta - first_cta + 1) : a.S;
        }
        if (m) {
          found = true;
          break;
        }
        base += (long long)__shfl_sync(0xffffffffu, incl, 31) * a.Hkv;
      }
      if (!found && lane == 0) {  // context lengths changed under the launch
        flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
        fl_stop = 1;
      }
    }
    __syncthreads();
    if (fl_stop) break;
    b = fl_unit[0];
    h = fl_unit[1];
    c_first = fl_unit[2];
    c_end = fl_unit[3];
    s = fl_unit[4];
    empty_from = fl_unit[5];
  } else {
    s = 0;
    h = blockIdx.y;
    b = mma::longest_first(a.context_lens, a.B, blockIdx.z);
  }
  do {  // one unit; early exits leave by break
  // With pos_split (more query rows than one CTA holds) a CTA serves the
  // pos_tile query positions j0 .. j0 + Tc - 1 of the sequence; position j
  // attends to the first L - T + 1 + j tokens (causal verify or extend), so
  // the tile is a decode of Tc positions over the prefix its last position
  // sees.  The tiles of one (split, head, sequence) are neighbours in launch
  // order (x = split * tiles + tile): they read the same pages, so all but
  // the first read are mostly served by L2.
  const int n_tiles = a.pos_split ? (a.T + a.pos_tile - 1) / a.pos_tile : 1;
  if (!FLAT) s = (int)blockIdx.x / n_tiles;
  const int j0 = a.pos_split ? ((int)blockIdx.x % n_tiles) * a.pos_tile : 0;
  const int Tc = a.pos_split ? min(a.pos_tile, a.T - j0) : a.T;  // query positions in this CTA
  const int R = Tc * G;
  const int L_seq = a.context_lens[b];
  const int L = a.causal ? L_seq - (a.T - Tc) + j0 : L_seq;  // tokens visible to this CTA's last position
  const size_t row0 = ((size_t)b * a.T + j0) * a.Hq;

  auto row_index = [&](int r) -> size_t {  // flat (b, j, hq) row of query row r
    return row0 + (size_t)(r / G) * a.Hq + h * G + (r % G);
  };
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
    break;
  }
  const int n_pages = (L + kPage - 1) / kPage;
  int p0, p1;
  if constexpr (FLAT) {
    p0 = c_first * kPagesPerChunk;
    p1 = min(n_pages, c_end * kPagesPerChunk);
  } else {
    const int per = (n_pages + a.S - 1) / a.S;
    p0 = s * per;
    p1 = min(n_pages, p0 + per);
  }
  if (p0 >= p1) {
    write_empty();
    break;
  }
  const int n_chunks = (p1 - p0 + kPagesPerChunk - 1) / kPagesPerChunk;
  const int32_t* table = a.block_tables + (size_t)b * a.max_pages;

  // Page ids of chunk c for lanes 0..3 (page 0 for lanes past the split; a
  // bad id is flagged and read as page 0).
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
  // Issue chunk c into stage st: lane i < nv copies page i's K and V blocks.
  auto issue = [&](int c, int st, int page) {
    const int nv = min(kPagesPerChunk, p1 - (p0 + c * kPagesPerChunk));
    uint8_t* dst = sm.stage(w, st);
    uint64_t* bar = &bars[w * kStages + st];
    // K and V: the 4 page blocks of each in one tensor gather (tile::gather4,
    // one 1088-byte row per page block); rows past the split re-read the
    // chunk's first block and are masked like any token past the context.
    const int row = page * a.Hkv + h;
    const int r0 = __shfl_sync(0xffffffffu, row, 0);
    const int r1 = nv > 1 ? __shfl_sync(0xffffffffu, row, 1) : r0;
    const int r2 = nv > 2 ? __shfl_sync(0xffffffffu, row, 2) : r0;
    const int r3 = nv > 3 ? __shfl_sync(0xffffffffu, row, 3) : r0;
    if (lane == 0) {
      mbar_expect_tx(bar, (uint32_t)(2 * kPagesPerChunk * kBlk));
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
          "%4, %5, %6}], [%7];" ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(&kmap)), "r"(0), "r"(r0), "r"(r1),
          "r"(r2), "r"(r3), "r"(smem_u32(bar))
          : "memory");
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
          "%4, %5, %6}], [%7];" ::"r"(smem_u32(dst + kPagesPerChunk * kBlkStride)), "l"(reinterpret_cast<uint64_t>(&vmap)), "r"(0), "r"(r0), "r"(r1),
          "r"(r2), "r"(r3), "r"(smem_u32(bar))
          : "memory");
    }
    __syncwarp();
  };

  // Start streaming before the q prologue so the first loads overlap it.
  __syncthreads();
  fence_proxy_async();
  for (int i = 0; i < kStages; ++i) {
    const int c = w + kWarps * i;
    if (c < n_chunks) issue(c, (it_base + i) % kStages, chunk_page(c));
  }

  // ---- q prologue: rotate (fp32 butterfly), scale row by 2^sigma, split into f16 hi + lo
  uint16_t* qt = reinterpret_cast<uint16_t*>(sm.qterms());  // [8 * RB rows][hi, lo][128]
  __shared__ float row_c[8 * RB];
  __shared__ int row_limit[8 * RB];
  for (int r = w; r < 8 * RB; r += kWarps) {
    float x[4];
    if (r < R) {
      const uint16_t* src = a.q + row_index(r) * D + lane * 4;
      const uint2 raw = *reinterpret_cast<const uint2*>(src);
      x[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
      x[1] = bf16_bits_to_float(raw.x >> 16);
      x[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
      x[3] = bf16_bits_to_float(raw.y >> 16);
      fwht_warp<4, float>(x);
    } else {
      x[0] = x[1] = x[2] = x[3] = 0.0f;
    }
    float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    // sigma puts the row maximum in [2^14, 2^15) (f16 range, lo parts far
    // above the f16 subnormal floor); x * 2^sigma is exact.
    int sigma = 0;
    if (mx > 0.0f) sigma = max(-113, min(126, 141 - (int)((__float_as_uint(mx) >> 23) & 0xFF)));
    const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float v0 = x[2 * i] * sc, v1 = x[2 * i + 1] * sc;
      const uint32_t h = pack_f16x2(v0, v1);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&h));
      hw[i] = h;
      lw[i] = pack_f16x2(v0 - hf.x, v1 - hf.y);  // exact remainders, rounded to f16
    }
    *reinterpret_cast<uint2*>(qt + (r * 2) * D + lane * 4) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(qt + (r * 2 + 1) * D + lane * 4) = make_uint2(lw[0], lw[1]);
    if (lane == 0) {
      // score*log2e = (q*2^sigma . code * 2^e) * 2^-sigma * softmax_scale*log2e/sqrt(D)
      row_c[r] = a.qscale * __uint_as_float((uint32_t)(127 - sigma) << 23);
      row_limit[r] = r < R ? (a.causal ? L - Tc + 1 + r / G : L) : 0x7fffffff;
    }
  }
  __syncthreads();

  // A fragments, per 32-channel group two k16 steps.  Row g holds hi, row g+8
  // lo.  Step j's k index 2t+i maps to channel 32G + 8t + 4j + i and 2t+8+i to
  // 32G + 8t + 4j + 2 + i, matching the K B-fragments built from one 32-bit
  // word of codes per thread (bytes 4t .. 4t+3 of the group).
  uint4* qfrag = reinterpret_cast<uint4*>(smem_raw + qfrag_off(RB));
  for (int rb = w; rb < RB; rb += kWarps) {
    const uint16_t* qb = qt + (8 * rb) * 2 * D;
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      const uint4 hi = *reinterpret_cast<const uint4*>(qb + (g * 2) * D + 32 * G4 + 8 * t);
      const uint4 lo = *reinterpret_cast<const uint4*>(qb + (g * 2 + 1) * D + 32 * G4 + 8 * t);
      qfrag[((rb * 4 + G4) * 2 + 0) * 32 + lane] = make_uint4(hi.x, lo.x, hi.y, lo.y);
      qfrag[((rb * 4 + G4) * 2 + 1) * 32 + lane] = make_uint4(hi.z, lo.z, hi.w, lo.w);
    }
  }
  const uint32_t qfrag_addr = smem_u32(qfrag) + lane * 16;
  float my_c[RB];
  int my_limit[RB];
#pragma unroll
  for (int rb = 0; rb < RB; ++rb) {
    my_c[rb] = row_c[8 * rb + g];
    my_limit[rb] = row_limit[8 * rb + g];
  }
  int min_limit = row_limit[0];
#pragma unroll
  for (int r = 1; r < 8 * RB; ++r) min_limit = min(min_limit, row_limit[r]);
  __syncthreads();  // the q terms share memory with the scale tables

  // ---- per-warp running state
  float o[RB][8][4];
#pragma unroll
  for (int rb = 0; rb < RB; ++rb)
#pragma unroll
    for (int j = 0; j < 8; ++j) o[rb][j][0] = o[rb][j][1] = o[rb][j][2] = o[rb][j][3] = 0.0f;
  float m_run[RB];
  float2 l2[RB];
#pragma unroll
  for (int rb = 0; rb < RB; ++rb) {
    m_run[rb] = -INFINITY;
    l2[rb] = make_float2(0.0f, 0.0f);
  }
  uint32_t eref = 0;  // 4 UE8M0 bytes: running max of V exponents per group
  float lo_share = 0.0625f;  // the lo part of P's share threshold for this eref

  float* ktab = sm.ktab(w);
  uint32_t* vtab = sm.vtab(w);
  bool timed_out = false;
  int it_fail = 0;

  for (int c = w, it = 0; c < n_chunks; c += kWarps, ++it) {
    const int st = (it_base + it) % kStages;
    const uint32_t parity = (uint32_t)(((it_base + it) / kStages) & 1);
    // page ids for the refill of this stage, loaded now to hide their latency
    const int cn = c + kWarps * kStages;
    const int next_page = cn < n_chunks ? chunk_page(cn) : 0;
    if (!mbar_wait(&bars[w * kStages + st], parity, it_base + it == 0 ? first_limit : kSpinLimit)) {
      timed_out = true;
      it_fail = it;
      break;
    }
    const uint8_t* stg = sm.stage(w, st);
    const int pg = p0 + c * kPagesPerChunk;
    const int nv = min(kPagesPerChunk, p1 - pg);
    const bool edge = nv < kPagesPerChunk || (pg + kPagesPerChunk) * kPage > min_limit;

    // ---- scale tables: lane -> page lane>>3, token pair lane&7
    uint32_t eold;
    bool under;  // this lane holds a visible V scale below the f16 window
    {
      const int pp = lane >> 3, pr = lane & 7, tk = 2 * pr;
      const int pos = (pg + pp) * kPage + tk;
      uint32_t k0 = 0, k1 = 0, v0 = 0, v1 = 0;
      const bool ok0 = pp < nv && pos < L, ok1 = pp < nv && pos + 1 < L;
      if (pp < nv) {
        const uint8_t* kb = stg + pp * kBlkStride + kCodeBytes;
        const uint8_t* vb = stg + kPagesPerChunk * kBlkStride + pp * kVStride + kCodeBytes;
        const uint2 kk = *reinterpret_cast<const uint2*>(kb + tk * 4);
        const uint2 vv = *reinterpret_cast<const uint2*>(vb + tk * 4);
        if (ok0) { k0 = kk.x; v0 = vv.x; }
        if (ok1) { k1 = kk.y; v1 = vv.y; }
      }
      // V reference exponent per group (Eref): fixed from the warp's first
      // chunk, so the usual chunk needs no reduction.  The f16 scale factors
      // 2^(e_v - Eref) hold exponents from -14 to +7; a chunk with an exponent
      // more than 7 above Eref (a rare jump) raises Eref to the chunk maximum
      // and the accumulators are rescaled below.  With p <= 2^8 (lazy softmax
      // maximum) the scaled P stays below 2^15, inside the f16 range.
      eold = eref;
      uint32_t lim = __vaddus4(eref, 0x07070707u);
      const bool over = (__vcmpgtu4(v0, lim) | __vcmpgtu4(v1, lim)) != 0u;
      if (it == 0 || __any_sync(0xffffffffu, over)) {
        uint32_t cm = __vmaxu4(v0, v1);
#pragma unroll
        for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
        eref = __vmaxu4(eref, cm);
        lo_share = lo_share_of(eref);
        lim = __vaddus4(eref, 0x07070707u);
      }
      // K scale pairs: {2^e(tk,G), 2^e(tk+1,G)} for G = 0..3 (byte 0 -> 0.0)
      float4 f01, f23;
      f01.x = __uint_as_float((k0 << 23) & 0x7F800000u);
      f01.y = __uint_as_float((k1 << 23) & 0x7F800000u);
      f01.z = __uint_as_float((k0 << 15) & 0x7F800000u);
      f01.w = __uint_as_float((k1 << 15) & 0x7F800000u);
      f23.x = __uint_as_float((k0 << 7) & 0x7F800000u);
      f23.y = __uint_as_float((k1 << 7) & 0x7F800000u);
      f23.z = __uint_as_float((k0 >> 1) & 0x7F800000u);
      f23.w = __uint_as_float((k1 >> 1) & 0x7F800000u);
      float4* kt = reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(ktab) + pp * kKTabPage + pr * 32);
      kt[0] = f01;
      kt[1] = f23;
      // V scale pairs 2^(e_v - Eref_G) as f16x2 (token tk low half, tk+1 high half):
      // f16 exponent field 15 + e_v - Eref per byte, in [0, 22] here (as
      // 22 - (Eref + 7 - e_v), both differences non-negative).  Tokens past
      // the context take the in-window field of `lim` (their p is 0).
      const uint32_t a0 = __vsubus4(0x16161616u, __vsubus4(lim, ok0 ? v0 : lim));
      const uint32_t a1 = __vsubus4(0x16161616u, __vsubus4(lim, ok1 ? v1 : lim));
      // A zero field is a V scale more than 14 binades below the reference
      // (or a zero byte: an all-zero group): f16 cannot carry that factor, and
      // the chunk's P.V takes the bf16 path below (the vote waits until then).
      under = (has_zero_byte(a0) | has_zero_byte(a1)) != 0u;
      uint4 vp;
      vp.x = __byte_perm(__byte_perm(a0, a1, 0x0040), 0, 0x5140) << 10;
      vp.y = __byte_perm(__byte_perm(a0, a1, 0x0051), 0, 0x5140) << 10;
      vp.z = __byte_perm(__byte_perm(a0, a1, 0x0062), 0, 0x5140) << 10;
      vp.w = __byte_perm(__byte_perm(a0, a1, 0x0073), 0, 0x5140) << 10;
      uint32_t* vt = vtab + pp * (kVTabPage / 4) + pr;
      vt[0] = vp.x;
      vt[8] = vp.y;
      vt[16] = vp.z;
      vt[24] = vp.w;
      __syncwarp();
    }

    // ---- Q.K^T, group-major: per 32-channel group G the q fragments are read
    // once for NB n-tiles (tile n: token pair n of each page, col 2t'+i -> page
    // t', token 2n+i); each tile's group result (hi row + lo row) is multiplied
    // by that group's K scale and accumulated over the groups.  The row factor
    // (softmax scale, log2 e, 2^-sigma) is applied in the softmax below.
    constexpr int NB = RB == 1 ? 4 : 2;
    float2 sc[RB][8];  // row 8rb + g, tokens (2n, 2n+1) of page t
    const uint8_t* ktb = reinterpret_cast<const uint8_t*>(ktab) + t * kKTabPage;
#pragma unroll
    for (int n0 = 0; n0 < 8; n0 += NB) {
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) {
        uint32_t kb[NB][4];
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const uint32_t x = *reinterpret_cast<const uint32_t*>(
              stg + (g >> 1) * kBlkStride + k_code_offset(D, 2 * (n0 + u) + (g & 1), 8 * t) + 128 * G4);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) kb[u][bb] = e2m1x2_to_f16x2(x, bb);
        }
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          float acc[NB][4];
#pragma unroll
          for (int u = 0; u < NB; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.0f;
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            uint32_t q0, q1, q2, q3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                         : "r"(qfrag_addr + ((rb * 4 + G4) * 2 + j2) * 512));
#pragma unroll
            for (int u = 0; u < NB; ++u) mma_f16(acc[u], q0, q1, q2, q3, kb[u][2 * j2], kb[u][2 * j2 + 1]);
          }
#pragma unroll
          for (int u = 0; u < NB; ++u) {
            const float2 ks = *reinterpret_cast<const float2*>(ktb + (n0 + u) * 32 + G4 * 8);
            const float2 tt = __fadd2_rn(make_float2(acc[u][0], acc[u][1]), make_float2(acc[u][2], acc[u][3]));
            sc[rb][n0 + u] = G4 == 0 ? __fmul2_rn(ks, tt) : __ffma2_rn(ks, tt, sc[rb][n0 + u]);
          }
        }
      }
    }

    // tokens past the split's pages, the context or a row's causal limit
    if (edge) {
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int posb = (pg + t) * kPage + 2 * n;
          const bool ok = t < nv;
          if (!(ok && posb < my_limit[rb])) sc[rb][n].x = -INFINITY;
          if (!(ok && posb + 1 < my_limit[rb])) sc[rb][n].y = -INFINITY;
        }
    }

    // ---- online softmax per row block (row 8rb + g; the quad t = 0..3 holds the row)
    float alpha[RB];
    float2 p[RB][8];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(sc[rb][i].x, sc[rb][i].y);
#pragma unroll
      for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) mx8[i] = fmaxf(mx8[i], mx8[i + w2]);
      float cmx = mx8[0];
      cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 1));
      cmx = fmaxf(cmx, __shfl_xor_sync(0xffffffffu, cmx, 2));
      // to log2 units: the row factor is positive (the softmax scale is checked
      // at the API), so the maximum of the scaled logits is the scaled maximum
      cmx *= my_c[rb];
      // Lazy maximum: the row's reference moves only when the chunk maximum
      // exceeds it by more than 8 (log2 units), so p <= 2^8 and O is rarely
      // rescaled.  Any reference gives the same (O, l) up to that common factor.
      const float m_new = cmx > m_run[rb] + 8.0f ? cmx : m_run[rb];
      alpha[rb] = 1.0f;
      if (m_new == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 8; ++i) p[rb][i] = make_float2(0.0f, 0.0f);
      } else {
        alpha[rb] = ex2(m_run[rb] - m_new);
        const float2 nm = make_float2(-m_new, -m_new);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 d2 = __ffma2_rn(sc[rb][i], make_float2(my_c[rb], my_c[rb]), nm);
          p[rb][i] = make_float2(ex2(d2.x), ex2(d2.y));
        }
        const float2 ls =
            __fadd2_rn(__fadd2_rn(__fadd2_rn(p[rb][0], p[rb][1]), __fadd2_rn(p[rb][2], p[rb][3])),
                       __fadd2_rn(__fadd2_rn(p[rb][4], p[rb][5]), __fadd2_rn(p[rb][6], p[rb][7])));
        l2[rb] = __ffma2_rn(l2[rb], make_float2(alpha[rb], alpha[rb]), ls);
      }
      m_run[rb] = m_new;
    }

    // ---- rescale O: columns 2t, 2t+1 are rows 8rb + 2t, 8rb + 2t + 1; group factor 2^(Eold - Enew)
    {
      float a0[RB], a1[RB];
      bool any_a = false;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        a0[rb] = __shfl_sync(0xffffffffu, alpha[rb], 8 * t);
        a1[rb] = __shfl_sync(0xffffffffu, alpha[rb], 8 * t + 4);
        any_a |= a0[rb] != 1.0f || a1[rb] != 1.0f;
      }
      if (__any_sync(0xffffffffu, eold != eref || any_a)) {
        const uint32_t dl = __vsubus4(eref, eold);  // Enew - Eold per group
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) {
          const int ex = 127 - (int)((dl >> (8 * G4)) & 0xFFu);
          const float f = ex > 0 ? __uint_as_float((uint32_t)ex << 23) : 0.0f;
#pragma unroll
          for (int rb = 0; rb < RB; ++rb) {
            const float f0 = f * a0[rb], f1 = f * a1[rb];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              o[rb][2 * G4 + jj][0] *= f0;
              o[rb][2 * G4 + jj][1] *= f1;
              o[rb][2 * G4 + jj][2] *= f0;
              o[rb][2 * G4 + jj][3] *= f1;
            }
          }
        }
      }
    }

    // ---- P fragments (hi + lo f16): k-step c4 uses tokens 4c4..4c4+3 of page t.
    // hi is p rounded to f16, lo the exact fp32 remainder p - hi rounded to f16.
    // The lo part matters only for a token that carries a noticeable share of
    // its row: its MMAs run for a k-step only when some p of the step (any row,
    // any page) exceeds tau times its row's running sum in this warp.  Every
    // other token keeps p rounded to f16 (relative error at most 2^-11); those
    // errors enter the output weighted by p / l, each weight below tau, and
    // add up like independent roundings: about 2^-11 |v| times the root of the
    // sum of the squared weights, at most sqrt(tau).  tau = 2^-4 while |v| <
    // 12 (largest V group reference 2^1) puts that near 2^-11 * 12 / 4 = 1.5e-3
    // in the worst case and measures 1e-4 to 5e-4 on the workloads and stress
    // cases; tau falls by 4 per binade of larger V (lo_share_of) so the bound
    // holds for any V magnitude.  In a long context every token's weight is
    // far below tau and the lo MMAs are skipped; a short one keeps them.
    const uint8_t* vbase = stg + kPagesPerChunk * kBlkStride + t * kVStride;
    if (__any_sync(0xffffffffu, under)) {
      // The reference is re-taken from the chunk itself: each group's largest
      // visible V exponent (at most 90 binades below the current one, so the
      // rescaled O stays finite; groups with no visible token keep theirs).
      // It moves up or down, and O is rescaled by 2^(Eref - Enew).
      const int pp = lane >> 3, tk = 2 * (lane & 7);
      const int pos = (pg + pp) * kPage + tk;
      uint32_t v0 = 0, v1 = 0;
      if (pp < nv) {
        const uint2 vv =
            *reinterpret_cast<const uint2*>(stg + kPagesPerChunk * kBlkStride + pp * kVStride + kCodeBytes + tk * 4);
        if (pos < L) v0 = vv.x;
        if (pos + 1 < L) v1 = vv.y;
      }
      uint32_t cm = __vmaxu4(v0, v1);
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
      const uint32_t none = __vcmpeq4(cm, 0u);
      const uint32_t enew = (__vmaxu4(cm, __vsubus4(eref, 0x5A5A5A5Au)) & ~none) | (eref & none);
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) {
        const float f = pow2_diff((eref >> (8 * G4)) & 0xFFu, (int)((enew >> (8 * G4)) & 0xFFu));
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
#pragma unroll
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) o[rb][2 * G4 + jj][k4] *= f;
      }
      eref = enew;
      lo_share = lo_share_of(eref);
      pv_bf16<RB>(o, p, vbase, eref, g);
    } else {
    uint32_t ph[RB][4][2], pl[RB][4][2];
    bool need_lo[4];
    // lo matters for a token above a share (lo_share) of its row's running
    // sum in this warp, this chunk included
    float lo_thr[RB];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      float lr = l2[rb].x + l2[rb].y;
      lr += __shfl_xor_sync(0xffffffffu, lr, 1);
      lr += __shfl_xor_sync(0xffffffffu, lr, 2);
      lo_thr[rb] = lo_share * lr;
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      bool big = false;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
        ph[rb][c4][0] = pack_f16x2(p[rb][2 * c4].x, p[rb][2 * c4].y);
        ph[rb][c4][1] = pack_f16x2(p[rb][2 * c4 + 1].x, p[rb][2 * c4 + 1].y);
        const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&ph[rb][c4][0]));
        const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&ph[rb][c4][1]));
        const float2 l0 = __fadd2_rn(p[rb][2 * c4], make_float2(-h0.x, -h0.y));
        const float2 l1 = __fadd2_rn(p[rb][2 * c4 + 1], make_float2(-h1.x, -h1.y));
        pl[rb][c4][0] = pack_f16x2(l0.x, l0.y);
        pl[rb][c4][1] = pack_f16x2(l1.x, l1.y);
        const float pm = fmaxf(fmaxf(p[rb][2 * c4].x, p[rb][2 * c4].y), fmaxf(p[rb][2 * c4 + 1].x, p[rb][2 * c4 + 1].y));
        big |= pm > lo_thr[rb];
      }
      need_lo[c4] = __any_sync(0xffffffffu, big);
    }

    // ---- P.V: m-tile j = dims 16j..16j+15 (group j/2); rows g, g+8 -> dims 16j+g, 16j+g+8.
    // V codes widen exactly to f16; the V scale 2^(e_v - Eref_G) multiplies the
    // P fragments of group G instead (two tokens per f16x2, as in the A fragment).
    const uint32_t* vrow = vtab + t * (kVTabPage / 4);
#pragma unroll
    for (int G4 = 0; G4 < 4; ++G4) {
      const uint2 rA0 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + g) * (kPage / 2));
      const uint2 rB0 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + g + 8) * (kPage / 2));
      const uint2 rA1 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + 16 + g) * (kPage / 2));
      const uint2 rB1 = *reinterpret_cast<const uint2*>(vbase + (32 * G4 + 16 + g + 8) * (kPage / 2));
      const uint4 vs0 = *reinterpret_cast<const uint4*>(vrow + G4 * 8);
      const uint4 vs1 = *reinterpret_cast<const uint4*>(vrow + G4 * 8 + 4);
      const uint32_t vsc[8] = {vs0.x, vs0.y, vs0.z, vs0.w, vs1.x, vs1.y, vs1.z, vs1.w};
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        const int b0 = (2 * c4) & 3, b1 = (2 * c4 + 1) & 3;
        const uint32_t wA0 = c4 < 2 ? rA0.x : rA0.y, wB0 = c4 < 2 ? rB0.x : rB0.y;
        const uint32_t wA1 = c4 < 2 ? rA1.x : rA1.y, wB1 = c4 < 2 ? rB1.x : rB1.y;
        const uint32_t x00 = e2m1x2_to_f16x2(wA0, b0), x01 = e2m1x2_to_f16x2(wB0, b0);
        const uint32_t x02 = e2m1x2_to_f16x2(wA0, b1), x03 = e2m1x2_to_f16x2(wB0, b1);
        const uint32_t x10 = e2m1x2_to_f16x2(wA1, b0), x11 = e2m1x2_to_f16x2(wB1, b0);
        const uint32_t x12 = e2m1x2_to_f16x2(wA1, b1), x13 = e2m1x2_to_f16x2(wB1, b1);
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          const uint32_t ph0 = hmul2(ph[rb][c4][0], vsc[2 * c4]), ph1 = hmul2(ph[rb][c4][1], vsc[2 * c4 + 1]);
          mma_f16(o[rb][2 * G4], x00, x01, x02, x03, ph0, ph1);
          mma_f16(o[rb][2 * G4 + 1], x10, x11, x12, x13, ph0, ph1);
          if (need_lo[c4]) {
            const uint32_t pl0 = hmul2(pl[rb][c4][0], vsc[2 * c4]), pl1 = hmul2(pl[rb][c4][1], vsc[2 * c4 + 1]);
            mma_f16(o[rb][2 * G4], x00, x01, x02, x03, pl0, pl1);
            mma_f16(o[rb][2 * G4 + 1], x10, x11, x12, x13, pl0, pl1);
          }
        }
      }
    }
    }  // fast path
    __syncwarp();
    // refill this stage with the warp's chunk kStages ahead
    if (cn < n_chunks) {
      fence_proxy_async();
      issue(cn, st, next_page);
    }
  }

  if (timed_out) {
    // Stop streaming, but let every copy this warp issued land before the
    // shared memory is reused: iterations it_fail .. it_fail + kStages - 1 were
    // issued and not yet waited on (each wait again bounded).
    if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
    for (int it = it_fail; it < it_fail + kStages; ++it)
      if (w + kWarps * it < n_chunks)
        (void)mbar_wait(&bars[w * kStages + (it_base + it) % kStages], (uint32_t)(((it_base + it) / kStages) & 1));
  }

  // ---- merge the 4 warps, one row block at a time: row l sums, then O scaled
  // by 2^Eref_G and exp2(m_w - M)
  float* mo = reinterpret_cast<float*>(smem_raw);  // [kWarps][8 rows][D]
  float* mm = mo + kWarps * 8 * D;                  // [kWarps][8]
  float* ml = mm + kWarps * 8;                      // [kWarps][8]
#pragma unroll
  for (int rb = 0; rb < RB; ++rb) {
    float l_row = l2[rb].x + l2[rb].y;
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
    l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
    __syncthreads();  // stages (first block) or the previous block's merge are done with
    if (t == 0) {
      mm[w * 8 + g] = m_run[rb];
      ml[w * 8 + g] = l_row;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float eg = __uint_as_float(((eref >> (8 * (j >> 1))) & 0xFFu) << 23);
      mo[(w * 8 + 2 * t) * D + 16 * j + g] = o[rb][j][0] * eg;
      mo[(w * 8 + 2 * t + 1) * D + 16 * j + g] = o[rb][j][1] * eg;
      mo[(w * 8 + 2 * t) * D + 16 * j + g + 8] = o[rb][j][2] * eg;
      mo[(w * 8 + 2 * t + 1) * D + 16 * j + g + 8] = o[rb][j][3] * eg;
    }
    __syncthreads();
    // warp w finalises rows w and w+4 of the block
    for (int r = w; r < 8; r += kWarps) {
      const int rr_row = 8 * rb + r;
      if (rr_row >= R) continue;
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) M = fmaxf(M, mm[ww * 8 + r]);
      float wsum = 0.0f, wt[kWarps];
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        wt[ww] = (M == -INFINITY || mm[ww * 8 + r] == -INFINITY) ? 0.0f : exp2f(mm[ww * 8 + r] - M);
        wsum += wt[ww] * ml[ww * 8 + r];
      }
      const size_t rr = row_index(rr_row) * a.S + s;
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
  if constexpr (FLAT) {
    // the unit's unused slots, by the CTA holding its last chunk
    for (int r = w; r < R; r += kWarps)
      for (int sl = empty_from; sl < a.S; ++sl) {
        const size_t rr = row_index(r) * a.S + sl;
        for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = 0.0f;
        if (lane == 0) a.part_lse[rr] = -INFINITY;
      }
    if (timed_out) fl_stop = 1;
  }
  it_base += n_chunks > w ? (n_chunks - w + kWarps - 1) / kWarps : 0;
  } while (0);
  if constexpr (!FLAT) break;
  // the next unit of this CTA's part, once every thread is done with the
  // merge area (the stages) and this unit's shared values
  fence_proxy_async();
  __syncthreads();
  if (tid == 0) fl_cur += fl_unit[3] - fl_unit[2];
  __syncthreads();
  }  // units
}

}  // namespace fast

bool fast_path_supported(int D, int G, int T, bool latent) {
  (void)T;  // more than 24 rows are tiled over CTAs by query position (pos_split)
  return D == 128 && !latent && G <= 8;
}

namespace {

// Rows per CTA when the query positions are tiled: whole positions of G rows.
constexpr int kSplitRows = 24;

template <int RB>
cudaError_t launch_rb(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(fast::decode_fp4_mma_kernel<RB, false>, fast::smem_bytes(RB), smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(a.S * (a.pos_split ? (a.T + a.pos_tile - 1) / a.pos_tile : 1), a.Hkv, a.B);
  fast::decode_fp4_mma_kernel<RB, false><<<grid, fast::kThreads, fast::smem_bytes(RB), st>>>(a, kmap, vmap);
  return cudaGetLastError();
}

// Flat mode: one wave of CTAs (every resident slot of every SM), each an equal
// part of the step's chunks.
template <int RB>
cudaError_t launch_flat(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap, cudaStream_t st) {
  static std::atomic<unsigned long long> smem_set{0};
  auto* kern = fast::decode_fp4_mma_kernel<RB, true>;
  const cudaError_t e = set_smem_limit_once(kern, fast::smem_bytes(RB), smem_set);
  if (e != cudaSuccess) return e;
  const int grid = flat_grid_size(8 * RB);
  if (grid < 1) return cudaErrorUnknown;
  kern<<<grid, fast::kThreads, fast::smem_bytes(RB), st>>>(a, kmap, vmap);
  return cudaGetLastError();
}

template <int RB>
int flat_grid_of() {
  static int grid = 0;
  if (grid == 0) {
    int dev = 0, sms = 0, per_sm = 0;
    auto* kern = fast::decode_fp4_mma_kernel<RB, true>;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, fast::smem_bytes(RB)) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, fast::kThreads, fast::smem_bytes(RB)) != cudaSuccess)
      return 0;
    grid = sms * (per_sm > 0 ? per_sm : 1);
  }
  return grid;
}

}  // namespace

// Up to 24 query rows per kv head (T * G <= 24, e.g. a T = 3 verify step with
// G = 8) run in one CTA as 1-3 row blocks; more rows (longer verify blocks,
// extend steps) are tiled over CTAs of kSplitRows rows' worth of whole
// positions each (pos_split).
cudaError_t launch_decode_fast(int D, const DecodeArgs& a_in, cudaStream_t st, bool flat) {
  if (D != 128) return cudaErrorNotSupported;
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
  // Each cache as a 2-D tensor of rows, one (page, head) block per row: 136
  // eight-byte elements, row stride 1088 bytes.  A map holds only the address
  // and the sizes, so the maps of the caches a host thread used last are kept
  // and re-encoded only when the cache or its size changes (a serving loop
  // decodes the same caches step after step).
  struct MapCache {
    const void* k = nullptr;
    const void* v = nullptr;
    cuuint64_t rows = 0;
    CUtensorMap kmap, vmap;
  };
  thread_local MapCache mc;
  const cuuint64_t rows = (cuuint64_t)a_in.num_pages * a_in.Hkv;
  if (mc.k != a_in.k_cache || mc.v != a_in.v_cache || mc.rows != rows) {
    mc.k = nullptr;
    const cuuint64_t dims[2] = {(cuuint64_t)fast::kBlk / 8, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)fast::kBlk};
    const cuuint32_t box[2] = {(cuuint32_t)fast::kBlk / 8, 1};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 2; ++i) {
      if (encode(i ? &mc.vmap : &mc.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2,
                 const_cast<uint8_t*>(i ? a_in.v_cache : a_in.k_cache), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    mc.k = a_in.k_cache;
    mc.v = a_in.v_cache;
    mc.rows = rows;
  }
  const CUtensorMap& kmap = mc.kmap;
  const CUtensorMap& vmap = mc.vmap;
  DecodeArgs a = a_in;
  const int G = a.Hq / a.Hkv;
  int R = a.T * G;
  a.pos_split = R > kTileRows ? 1 : 0;
  if (a.pos_split) {
    a.pos_tile = kSplitRows / G > 0 ? kSplitRows / G : 1;
    R = a.pos_tile * G;
  }
  if (flat) {
    if (a.pos_split || a.S < 2 || !a.causal) return cudaErrorNotSupported;
    if (R <= 8) return launch_flat<1>(a, kmap, vmap, st);
    return R <= 16 ? launch_flat<2>(a, kmap, vmap, st) : launch_flat<3>(a, kmap, vmap, st);
  }
  if (R <= 8) return launch_rb<1>(a, kmap, vmap, st);
  return R <= 16 ? launch_rb<2>(a, kmap, vmap, st) : launch_rb<3>(a, kmap, vmap, st);
}

bool flat_path_supported(int D, int G, int T, bool latent, int S) {
  return D == 128 && !latent && T * G <= kTileRows && S >= 2;
}

int flat_grid_size(int rows) {
  if (rows <= 8) return flat_grid_of<1>();
  return rows <= 16 ? flat_grid_of<2>() : flat_grid_of<3>();
}

}  // namespace kv4
