// kv4_decode_flat.cu -- balanced split decode over the 4-bit cache (sm_103a):
// head_dim 128, up to 8 query rows per kv head (a decode step of up to 8 query
// heads per kv head, or a short causal block).
//
// "UltraQuant on AMD Instinct", section "Why UltraQuant beats 8-bit KV": every
// decode step re-reads the whole cache, so the step is a stream over
// (sequence, kv head, page) and its speed is the memory system's.  The
// warp-MMA split kernel runs one CTA per (split, kv head, sequence); with four
// such CTAs per SM they progress unevenly (the warp scheduler favours the
// older ones) and the last wave leaves SMs with fewer CTAs.  Here the whole
// step is one flat range of 4-page chunks, in (sequence, kv head, chunk)
// order; CTA i of one per SM takes the i-th equal part, and its 16 warps pull
// chunks from that part through a shared-memory counter, so the SM works at
// its full rate until its part is done, whichever warps run faster.
//
// A CTA's part crosses (sequence, kv head) boundaries: each run of chunks of
// one (sequence, kv head) is a segment.  A warp keeps one online-softmax state
// (the arithmetic of the warp-MMA kernel, one 8-row block) and merges it into
// the segment's accumulator in shared memory when its next chunk belongs to
// another segment; at the end the CTA writes one split partial per segment,
// in slot (CTA - first CTA of the (sequence, kv head)).  The part size keeps
// every (sequence, kv head) within num_splits CTAs; the CTA holding a
// (sequence, kv head)'s last chunk writes its unused slots as empty partials,
// so kv4_split_combine merges them like the split kernel's.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "kv4_common.cuh"
#include "kv4_decode.h"
#include "kv4_mma_common.cuh"

namespace kv4 {
namespace flat {

using namespace kv4::mma;

constexpr int D = 128;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPagesPerChunk = 4;
constexpr int kBlk = kPage * D / 2 + kPage * D / 32;  // 1088 bytes per (page, head) block
constexpr int kCodeBytes = kPage * D / 2;            // 1024
constexpr int kBlkStride = 1088;
constexpr int kVStride = 1088;
constexpr int kStageBytes = (kPagesPerChunk * (kBlkStride + kVStride) + 127) / 128 * 128;  // 8704
constexpr int kKTabPage = 272;  // fp32 [8 token pairs][4 groups][2 tokens] + pad
constexpr int kVTabPage = 160;  // f16x2 [4 groups][8 token pairs] + pad
constexpr int kKTab = kPagesPerChunk * kKTabPage;
constexpr int kVTab = kPagesPerChunk * kVTabPage;
constexpr int kTabBytes = kKTab + kVTab;
constexpr int kMaxSeg = 4;                    // segments per round
constexpr int kQFragBytes = 4 * 2 * 32 * 16;  // q A-fragments [group][k-step][lane] uint4
constexpr int kQTermBytes = 8 * 2 * D * 2;    // f16 q [8 rows][hi, lo][128]
constexpr int kAccBytes = 8 * D * 4 + 2 * 8 * 4;  // o[8][128], m[8], l[8]

struct SegInfo {
  int b, h, L;     // sequence, kv head, context length
  int c_lo, c_hi;  // chunks of the (sequence, kv head) in this round
  int kbase;       // first index of the segment in the round's chunk order
  int slot;        // split slot of this CTA's partial
  int empty_from;  // this CTA holds the last chunk: slots empty_from .. S-1 are empty (else S)
};

struct Misc {
  uint64_t bars[kWarps];
  SegInfo seg[kMaxSeg];
  int nseg, nk, next, abort;
  int lock[kMaxSeg];
  long long lo, hi, per, cur, cur_next;
  float row_c[kMaxSeg][8];
  int row_limit[kMaxSeg][8];
};

// shared memory: stages | scale tables (q terms in the prologue) | q fragments
// [kMaxSeg] | segment accumulators [kMaxSeg] | misc
constexpr int kOffStage = 0;
constexpr int kOffTab = kWarps * kStageBytes;
constexpr int kOffQFrag = kOffTab + kWarps * kTabBytes;
constexpr int kOffAcc = kOffQFrag + kMaxSeg * kQFragBytes;
constexpr int kOffMisc = kOffAcc + kMaxSeg * kAccBytes;
constexpr int kSmem = kOffMisc + (int)sizeof(Misc);
static_assert(kMaxSeg * kQTermBytes <= kWarps * kTabBytes, "q terms of a round fit in the scale tables");
static_assert(kOffTab % 128 == 0 && kOffQFrag % 16 == 0 && kOffAcc % 16 == 0 && kOffMisc % 8 == 0, "alignment");
static_assert(kSmem <= 227 * 1024, "shared memory");

// Chunks of a sequence of context L: 4-page chunks of its ceil(L / 16) pages.
__device__ __forceinline__ int chunks_of(int L) { return ((L + kPage - 1) / kPage + kPagesPerChunk - 1) / kPagesPerChunk; }

__global__ void __launch_bounds__(kThreads, 1)
    decode_fp4_flat_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap) {
  extern __shared__ __align__(128) uint8_t smem[];
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.Hq / a.Hkv;
  const int R = a.T * G;  // <= 8
  const int S = a.S;      // >= 2
  const int nc_max = (a.max_pages + kPagesPerChunk - 1) / kPagesPerChunk;
  auto valid_len = [&](int L) { return L >= a.T && L <= a.max_pages * kPage; };

  // ---- this CTA's part of the flat chunk range
  if (w == 0) {
    long long C = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int nc = 0;
      if (b < a.B) {
        const int L = a.context_lens[b];
        nc = valid_len(L) ? chunks_of(L) : 0;
      }
      C += (long long)__reduce_add_sync(0xffffffffu, (unsigned)nc) * a.Hkv;
    }
    if (lane == 0) {
      const long long even = (C + gridDim.x - 1) / gridDim.x;
      const long long bound = (nc_max + S - 2) / (S - 1);  // a (sequence, kv head) spans <= S CTAs
      const long long per = even > bound ? even : bound;
      ms.per = per > 0 ? per : 1;
      ms.lo = (long long)blockIdx.x * ms.per;
      ms.hi = ms.lo + ms.per < C ? ms.lo + ms.per : C;
      ms.cur = ms.lo;
      ms.abort = 0;
    }
  }
  // CTA 0: sequences whose context is out of range get empty partials
  if (blockIdx.x == 0) {
    for (int b = w; b < a.B; b += kWarps) {
      const int L = a.context_lens[b];
      if (valid_len(L)) continue;
      if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_CONTEXT);
      for (int hh = 0; hh < a.Hkv; ++hh)
        for (int r = 0; r < R; ++r) {
          const size_t row = ((size_t)b * a.T + r / G) * a.Hq + hh * G + (r % G);
          for (int sl = 0; sl < S; ++sl) {
            for (int d = lane; d < D; d += 32) a.part_o[(row * S + sl) * D + d] = 0.0f;
            if (lane == 0) a.part_lse[row * S + sl] = -INFINITY;
          }
        }
    }
  }
  if (lane == 0) mbar_init(&ms.bars[w], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncthreads();
  const int first_limit = (a.diag & KV4_DIAG_EXPIRE_FIRST_WAIT) ? 0 : kSpinLimit;
  int it = 0;  // this warp's chunks so far (stage phase)
  bool first_wait = true;

  float* ktab = reinterpret_cast<float*>(smem + kOffTab + w * kTabBytes);
  uint32_t* vtab = reinterpret_cast<uint32_t*>(smem + kOffTab + w * kTabBytes + kKTab);
  uint8_t* stg_w = smem + kOffStage + w * kStageBytes;

  while (ms.cur < ms.hi) {
    // ---- the round's segments: runs of one (sequence, kv head) from cur, at most kMaxSeg
    if (w == 0) {
      const long long cur = ms.cur, hi = ms.hi, per = ms.per;
      long long base = 0;  // flat index of sequence b0's first chunk
      int found = 0;
      long long round_end = cur;
      for (int b0 = 0; b0 < a.B && found < kMaxSeg; b0 += 32) {
        const int b = b0 + lane;
        int nc = 0, L = 0;
        if (b < a.B) {
          L = a.context_lens[b];
          nc = valid_len(L) ? chunks_of(L) : 0;
        }
        // inclusive scan of this block's chunk counts
        int incl = nc;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o2);
          if (lane >= o2) incl += y;
        }
        const long long bb = base + (long long)(incl - nc) * a.Hkv;  // sequence b's first chunk
        // kv heads of sequence b whose chunks meet [cur, hi)
        int h_lo = 0, h_hi = 0;
        if (nc > 0) {
          const long long s0 = cur > bb ? (cur - bb) / nc : 0;
          const long long e0 = hi > bb ? (hi - bb + nc - 1) / nc : 0;
          h_lo = (int)(s0 < a.Hkv ? s0 : a.Hkv);
          h_hi = (int)(e0 < a.Hkv ? e0 : a.Hkv);
          if (h_hi < h_lo) h_hi = h_lo;
        }
        const int cnt = h_hi - h_lo;
        int before = cnt;
#pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, before, o2);
          if (lane >= o2) before += y;
        }
        before -= cnt;  // segments of earlier lanes in this block
        for (int i = 0; i < cnt; ++i) {
          const int idx = found + before + i;
          if (idx >= kMaxSeg) break;
          const int hh = h_lo + i;
          const long long ps = bb + (long long)hh * nc, pe = ps + nc;  // the pair's chunks
          const long long s1 = cur > ps ? cur : ps, e1 = hi < pe ? hi : pe;
          SegInfo& sg = ms.seg[idx];
          sg.b = b;
          sg.h = hh;
          sg.L = L;
          sg.c_lo = (int)(s1 - ps);
          sg.c_hi = (int)(e1 - ps);
          const long long first_cta = ps / per, last_cta = (pe - 1) / per;
          sg.slot = (int)((long long)blockIdx.x - first_cta);
          sg.empty_from = (long long)blockIdx.x == last_cta ? (int)(last_cta - first_cta + 1) : S;
        }
        const int tot = __reduce_add_sync(0xffffffffu, (unsigned)cnt);
        found += tot;
        base += (long long)__shfl_sync(0xffffffffu, incl, 31) * a.Hkv;
      }
      if (found > kMaxSeg) found = kMaxSeg;
      if (lane == 0) {
        int kb = 0;
        for (int i = 0; i < found; ++i) {
          ms.seg[i].kbase = kb;
          kb += ms.seg[i].c_hi - ms.seg[i].c_lo;
        }
        ms.nseg = found;
        ms.nk = kb;
        ms.next = 0;
        // the round ends after its last segment
        if (found > 0) {
          const SegInfo& sl = ms.seg[found - 1];
          round_end = cur + kb;
          (void)sl;
        }
        ms.cur_next = found > 0 ? round_end : hi;
        for (int i = 0; i < kMaxSeg; ++i) ms.lock[i] = 0;
      }
    }
    __syncthreads();
    const int nseg = ms.nseg, nk = ms.nk;

    // ---- q prologue of the round's segments: rotate (fp32 butterfly), scale
    // each row by 2^sigma, split into f16 hi + lo; then the MMA A-fragments
    uint16_t* qt_all = reinterpret_cast<uint16_t*>(smem + kOffTab);  // [seg][8 rows][hi, lo][128]
    for (int sr = w; sr < nseg * 8; sr += kWarps) {
      const int si = sr >> 3, r = sr & 7;
      const SegInfo& sg = ms.seg[si];
      uint16_t* qt = qt_all + si * (kQTermBytes / 2);
      float x[4];
      if (r < R) {
        const size_t row = ((size_t)sg.b * a.T + r / G) * a.Hq + sg.h * G + (r % G);
        const uint2 raw = *reinterpret_cast<const uint2*>(a.q + row * D + lane * 4);
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
      int sigma = 0;
      if (mx > 0.0f) sigma = max(-113, min(126, 141 - (int)((__float_as_uint(mx) >> 23) & 0xFF)));
      const float sc = __uint_as_float((uint32_t)(127 + sigma) << 23);
      uint32_t hw[2], lw[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float v0 = x[2 * i] * sc, v1 = x[2 * i + 1] * sc;
        const uint32_t hv = pack_f16x2(v0, v1);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hv));
        hw[i] = hv;
        lw[i] = pack_f16x2(v0 - hf.x, v1 - hf.y);
      }
      *reinterpret_cast<uint2*>(qt + (r * 2) * D + lane * 4) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(qt + (r * 2 + 1) * D + lane * 4) = make_uint2(lw[0], lw[1]);
      if (lane == 0) {
        ms.row_c[si][r] = a.qscale * __uint_as_float((uint32_t)(127 - sigma) << 23);
        ms.row_limit[si][r] = r < R ? sg.L - a.T + 1 + r / G : 0x7fffffff;
      }
    }
    // segment accumulators start empty
    for (int i = tid; i < nseg * (kAccBytes / 4); i += kThreads) {
      const int si = i / (kAccBytes / 4), e = i % (kAccBytes / 4);
      float* acc = reinterpret_cast<float*>(smem + kOffAcc + si * kAccBytes);
      acc[e] = e >= 8 * D && e < 8 * D + 8 ? -INFINITY : 0.0f;  // m = -inf, o = l = 0
    }
    __syncthreads();
    for (int si = w; si < nseg; si += kWarps) {
      const uint16_t* qb = qt_all + si * (kQTermBytes / 2);
      uint4* qfrag = reinterpret_cast<uint4*>(smem + kOffQFrag + si * kQFragBytes);
#pragma unroll
      for (int G4 = 0; G4 < 4; ++G4) {
        const uint4 hi = *reinterpret_cast<const uint4*>(qb + (g * 2) * D + 32 * G4 + 8 * t);
        const uint4 lo = *reinterpret_cast<const uint4*>(qb + (g * 2 + 1) * D + 32 * G4 + 8 * t);
        qfrag[(G4 * 2 + 0) * 32 + lane] = make_uint4(hi.x, lo.x, hi.y, lo.y);
        qfrag[(G4 * 2 + 1) * 32 + lane] = make_uint4(hi.z, lo.z, hi.w, lo.w);
      }
    }
    __syncthreads();  // the q terms share memory with the scale tables

    // ---- the warps pull chunks k of the round: segment si, chunk c of its
    // (sequence, kv head)
    auto locate = [&](int k, int& si, int& pg) {
      si = 0;
#pragma unroll
      for (int i = 1; i < kMaxSeg; ++i)
        if (i < nseg && k >= ms.seg[i].kbase) si = i;
      pg = (ms.seg[si].c_lo + (k - ms.seg[si].kbase)) * kPagesPerChunk;
    };
    auto grab = [&]() -> int {
      int k = 0;
      if (lane == 0) k = *reinterpret_cast<volatile int*>(&ms.abort) ? nk : atomicAdd(&ms.next, 1);
      return __shfl_sync(0xffffffffu, k, 0);
    };
    // page ids of chunk (si, pg) for lanes 0..3 (a bad id is flagged and read as page 0)
    auto chunk_page = [&](int si, int pg) -> int {
      const SegInfo& sg = ms.seg[si];
      const int n_pages = (sg.L + kPage - 1) / kPage;
      int page = 0;
      if (lane < kPagesPerChunk && pg + lane < n_pages) {
        page = a.block_tables[(size_t)sg.b * a.max_pages + pg + lane];
        if (page < 0 || page >= a.num_pages) {
          flag_error(a.dev_error, KV4_DEVERR_PAGE);
          page = 0;
        }
      }
      return page;
    };
    auto issue = [&](int si, int pg, int page) {
      const SegInfo& sg = ms.seg[si];
      const int n_pages = (sg.L + kPage - 1) / kPage;
      const int nv = min(kPagesPerChunk, n_pages - pg);
      uint64_t* bar = &ms.bars[w];
      const int row = page * a.Hkv + sg.h;
      const int r0 = __shfl_sync(0xffffffffu, row, 0);
      const int r1 = nv > 1 ? __shfl_sync(0xffffffffu, row, 1) : r0;
      const int r2 = nv > 2 ? __shfl_sync(0xffffffffu, row, 2) : r0;
      const int r3 = nv > 3 ? __shfl_sync(0xffffffffu, row, 3) : r0;
      if (lane == 0) {
        mbar_expect_tx(bar, (uint32_t)(2 * kPagesPerChunk * kBlk));
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3, %4, %5, %6}], [%7];" ::"r"(smem_u32(stg_w)),
            "l"(reinterpret_cast<uint64_t>(&kmap)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
            : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
            "%3, %4, %5, %6}], [%7];" ::"r"(smem_u32(stg_w + kPagesPerChunk * kBlkStride)),
            "l"(reinterpret_cast<uint64_t>(&vmap)), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
            : "memory");
      }
      __syncwarp();
    };

    // per-warp softmax state of its current segment
    float o[8][4];
    float m_run = -INFINITY;
    float2 l2 = make_float2(0.0f, 0.0f);
    uint32_t eref = 0;
    int cur_seg = -1;
    bool first_in_seg = false;  // the warp's first chunk of its segment (warp-uniform)
    float my_c = 0.0f;
    int my_limit = 0, min_limit = 0;
    uint32_t qfrag_addr = 0;
    bool timed_out = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;

    // Merge this warp's state into its segment's accumulator (under the
    // segment's lock) and clear it.
    auto flush = [&]() {
      if (cur_seg < 0) return;
      float* acc = reinterpret_cast<float*>(smem + kOffAcc + cur_seg * kAccBytes);
      float* am = acc + 8 * D;
      float* al = am + 8;
      // row sums of this warp: row g over the quad
      float l_row = l2.x + l2.y;
      l_row += __shfl_xor_sync(0xffffffffu, l_row, 1);
      l_row += __shfl_xor_sync(0xffffffffu, l_row, 2);
      bool got = false;
      if (lane == 0) {
        for (int i = 0; i < kSpinLimit && !got; ++i) {
          got = atomicCAS(&ms.lock[cur_seg], 0, 1) == 0;
          if (!got) __nanosleep(64);
        }
      }
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) {
        if (lane == 0) flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
        return;
      }
      __threadfence_block();
      // row g: old accumulator (m_a, l_a) and this warp's (m_run, l_row)
      const float m_a = am[g];
      const float M = fmaxf(m_a, m_run);
      const float fa = M == -INFINITY || m_a == -INFINITY ? 0.0f : exp2f(m_a - M);
      const float fw = M == -INFINITY || m_run == -INFINITY ? 0.0f : exp2f(m_run - M);
      __syncwarp();
      if (t == 0) {
        am[g] = M;
        al[g] = al[g] * fa + l_row * fw;
      }
      // O^T fragment columns 2t, 2t+1 are rows 2t, 2t+1: their factors from lanes 8t, 8t+4
      const float fa0 = __shfl_sync(0xffffffffu, fa, 8 * t), fa1 = __shfl_sync(0xffffffffu, fa, 8 * t + 4);
      const float fw0 = __shfl_sync(0xffffffffu, fw, 8 * t), fw1 = __shfl_sync(0xffffffffu, fw, 8 * t + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float eg = __uint_as_float(((eref >> (8 * (j >> 1))) & 0xFFu) << 23);
        float* r0p = acc + (2 * t) * D + 16 * j + g;
        float* r1p = acc + (2 * t + 1) * D + 16 * j + g;
        r0p[0] = r0p[0] * fa0 + o[j][0] * eg * fw0;
        r1p[0] = r1p[0] * fa1 + o[j][1] * eg * fw1;
        r0p[8] = r0p[8] * fa0 + o[j][2] * eg * fw0;
        r1p[8] = r1p[8] * fa1 + o[j][3] * eg * fw1;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) atomicExch(&ms.lock[cur_seg], 0);
      cur_seg = -1;
    };
    auto enter = [&](int si) {
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.0f;
      m_run = -INFINITY;
      l2 = make_float2(0.0f, 0.0f);
      eref = 0;
      cur_seg = si;
      first_in_seg = true;
      my_c = ms.row_c[si][g];
      my_limit = ms.row_limit[si][g];
      min_limit = ms.row_limit[si][0];
#pragma unroll
      for (int r = 1; r < 8; ++r) min_limit = min(min_limit, ms.row_limit[si][r]);
      qfrag_addr = smem_u32(smem + kOffQFrag + si * kQFragBytes) + lane * 16;
    };

    int k_cur = grab();
    int si_cur = 0, pg_cur = 0;
    if (k_cur < nk) {
      locate(k_cur, si_cur, pg_cur);
      fence_proxy_async();
      issue(si_cur, pg_cur, chunk_page(si_cur, pg_cur));
    }
    while (k_cur < nk) {
      const int k_next = grab();
      int si_next = 0, pg_next = 0, page_next = 0;
      if (k_next < nk) {
        locate(k_next, si_next, pg_next);
        page_next = chunk_page(si_next, pg_next);
      }
      if (!mbar_wait(&ms.bars[w], (uint32_t)(it & 1), first_wait ? first_limit : kSpinLimit)) {
        timed_out = true;
        break;
      }
      first_wait = false;
      ++it;
      if (si_cur != cur_seg) {
        flush();
        enter(si_cur);
      }
      const SegInfo& sg = ms.seg[si_cur];
      const int L = sg.L;
      const int n_pages = (L + kPage - 1) / kPage;
      const uint8_t* stg = stg_w;
      const int pg = pg_cur;
      const int nv = min(kPagesPerChunk, n_pages - pg);
      const bool edge = nv < kPagesPerChunk || (pg + kPagesPerChunk) * kPage > min_limit;

      // ---- scale tables: lane -> page lane>>3, token pair lane&7
      uint32_t eold;
      bool under;
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
          if (ok0) {
            k0 = kk.x;
            v0 = vv.x;
          }
          if (ok1) {
            k1 = kk.y;
            v1 = vv.y;
          }
        }
        // V reference exponent per group: set by the segment's first chunk,
        // raised when a chunk exceeds it by more than 7 (O rescaled below)
        eold = eref;
        uint32_t lim = __vaddus4(eref, 0x07070707u);
        const bool over = (__vcmpgtu4(v0, lim) | __vcmpgtu4(v1, lim)) != 0u;
        if (first_in_seg || __any_sync(0xffffffffu, over)) {
          uint32_t cm = __vmaxu4(v0, v1);
#pragma unroll
          for (int o2 = 16; o2 >= 1; o2 >>= 1) cm = __vmaxu4(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
          eref = __vmaxu4(eref, cm);
          lim = __vaddus4(eref, 0x07070707u);
        }
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
        // V factors 2^(e_v - Eref) as f16 exponent fields 22 - (Eref + 7 - e_v)
        const uint32_t a0 = __vsubus4(0x16161616u, __vsubus4(lim, ok0 ? v0 : lim));
        const uint32_t a1 = __vsubus4(0x16161616u, __vsubus4(lim, ok1 ? v1 : lim));
        // a zero field: a V scale more than 14 binades below the reference
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

      first_in_seg = false;
      // ---- Q.K^T, group-major (see the warp-MMA kernel): tile n = token pair n of each page
      float2 sc[8];
      const uint8_t* ktb = reinterpret_cast<const uint8_t*>(ktab) + t * kKTabPage;
#pragma unroll
      for (int n0 = 0; n0 < 8; n0 += 4) {
#pragma unroll
        for (int G4 = 0; G4 < 4; ++G4) {
          uint32_t kb[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t x = *reinterpret_cast<const uint32_t*>(
                stg + (g >> 1) * kBlkStride + k_code_offset(D, 2 * (n0 + u) + (g & 1), 8 * t) + 128 * G4);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) kb[u][bb] = e2m1x2_to_f16x2(x, bb);
          }
          float acc[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.0f;
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            uint32_t q0, q1, q2, q3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(q0), "=r"(q1), "=r"(q2), "=r"(q3)
                         : "r"(qfrag_addr + (G4 * 2 + j2) * 512));
#pragma unroll
            for (int u = 0; u < 4; ++u) mma_f16(acc[u], q0, q1, q2, q3, kb[u][2 * j2], kb[u][2 * j2 + 1]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 ks = *reinterpret_cast<const float2*>(ktb + (n0 + u) * 32 + G4 * 8);
            const float2 tt = __fadd2_rn(make_float2(acc[u][0], acc[u][1]), make_float2(acc[u][2], acc[u][3]));
            sc[n0 + u] = G4 == 0 ? __fmul2_rn(ks, tt) : __ffma2_rn(ks, tt, sc[n0 + u]);
          }
        }
      }
      if (edge) {
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int posb = (pg + t) * kPage + 2 * n;
          const bool okp = t < nv;
          if (!(okp && posb < my_limit)) sc[n].x = -INFINITY;
          if (!(okp && posb + 1 < my_limit)) sc[n].y = -INFINITY;
        }
      }

      // ---- online softmax (row g; the quad t holds the row), lazy maximum
      float alpha;
      float2 p[8];
      {
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
        cmx *= my_c;
        const float m_new = cmx > m_run + 8.0f ? cmx : m_run;
        alpha = 1.0f;
        if (m_new == -INFINITY) {
#pragma unroll
          for (int i = 0; i < 8; ++i) p[i] = make_float2(0.0f, 0.0f);
        } else {
          alpha = ex2(m_run - m_new);
          const float2 nm = make_float2(-m_new, -m_new);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 d2 = __ffma2_rn(sc[i], make_float2(my_c, my_c), nm);
            p[i] = make_float2(ex2(d2.x), ex2(d2.y));
          }
          const float2 ls = __fadd2_rn(__fadd2_rn(__fadd2_rn(p[0], p[1]), __fadd2_rn(p[2], p[3])),
                                       __fadd2_rn(__fadd2_rn(p[4], p[5]), __fadd2_rn(p[6], p[7])));
          l2 = __ffma2_rn(l2, make_float2(alpha, alpha), ls);
        }
        m_run = m_new;
      }
      // ---- rescale O: columns 2t, 2t+1 are rows 2t, 2t+1; group factor 2^(Eold - Enew)
      {
        const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
        const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
        const bool any_a = a0 != 1.0f || a1 != 1.0f;
        if (__any_sync(0xffffffffu, eold != eref || any_a)) {
          const uint32_t dl = __vsubus4(eref, eold);
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
      }
      // ---- P.V (f16 window, or the bf16 path when a V scale lies below it)
      const uint8_t* vbase = stg + kPagesPerChunk * kBlkStride + t * kVStride;
      if (__any_sync(0xffffffffu, under)) {
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
          for (int jj = 0; jj < 2; ++jj)
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) o[2 * G4 + jj][k4] *= f;
        }
        eref = enew;
        // bf16 P.V: x = p * 2^(e_v - E_G) in fp32 as bf16 hi + lo
        uint32_t sw[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 xw = *reinterpret_cast<const uint4*>(vbase + kCodeBytes + 16 * i);
          sw[4 * i] = xw.x;
          sw[4 * i + 1] = xw.y;
          sw[4 * i + 2] = xw.z;
          sw[4 * i + 3] = xw.w;
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
            uint32_t h01, l01, h23, l23;
            split_bf16x2(p[2 * c4].x * f[0], p[2 * c4].y * f[1], h01, l01);
            split_bf16x2(p[2 * c4 + 1].x * f[2], p[2 * c4 + 1].y * f[3], h23, l23);
            mma_bf16(o[2 * G4], x00, x01, x02, x03, h01, h23);
            mma_bf16(o[2 * G4 + 1], x10, x11, x12, x13, h01, h23);
            mma_bf16(o[2 * G4], x00, x01, x02, x03, l01, l23);
            mma_bf16(o[2 * G4 + 1], x10, x11, x12, x13, l01, l23);
          }
        }
      } else {
        uint32_t ph[4][2], pl[4][2];
        bool need_lo[4];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          ph[c4][0] = pack_f16x2(p[2 * c4].x, p[2 * c4].y);
          ph[c4][1] = pack_f16x2(p[2 * c4 + 1].x, p[2 * c4 + 1].y);
          const float2 h0 = __half22float2(*reinterpret_cast<const __half2*>(&ph[c4][0]));
          const float2 h1 = __half22float2(*reinterpret_cast<const __half2*>(&ph[c4][1]));
          const float2 l0 = __fadd2_rn(p[2 * c4], make_float2(-h0.x, -h0.y));
          const float2 l1 = __fadd2_rn(p[2 * c4 + 1], make_float2(-h1.x, -h1.y));
          pl[c4][0] = pack_f16x2(l0.x, l0.y);
          pl[c4][1] = pack_f16x2(l1.x, l1.y);
          const float pm = fmaxf(fmaxf(p[2 * c4].x, p[2 * c4].y), fmaxf(p[2 * c4 + 1].x, p[2 * c4 + 1].y));
          need_lo[c4] = __any_sync(0xffffffffu, pm > 0.00390625f);
        }
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
            const uint32_t ph0 = hmul2(ph[c4][0], vsc[2 * c4]), ph1 = hmul2(ph[c4][1], vsc[2 * c4 + 1]);
            mma_f16(o[2 * G4], x00, x01, x02, x03, ph0, ph1);
            mma_f16(o[2 * G4 + 1], x10, x11, x12, x13, ph0, ph1);
            if (need_lo[c4]) {
              const uint32_t pl0 = hmul2(pl[c4][0], vsc[2 * c4]), pl1 = hmul2(pl[c4][1], vsc[2 * c4 + 1]);
              mma_f16(o[2 * G4], x00, x01, x02, x03, pl0, pl1);
              mma_f16(o[2 * G4 + 1], x10, x11, x12, x13, pl0, pl1);
            }
          }
        }
      }
      __syncwarp();
      // refill the stage with the chunk grabbed next
      if (k_next < nk) {
        fence_proxy_async();
        issue(si_next, pg_next, page_next);
      }
      k_cur = k_next;
      si_cur = si_next;
      pg_cur = pg_next;
    }
    if (timed_out) {
      // let the copy in flight land before the stage is reused, then stop every warp
      if (lane == 0) {
        flag_error(a.dev_error, KV4_DEVERR_TIMEOUT);
        ms.abort = 1;
      }
      (void)mbar_wait(&ms.bars[w], (uint32_t)(it & 1));
      ++it;
      cur_seg = -1;
    }
    flush();
    __syncthreads();

    // ---- one split partial per segment of the round (empty slots by the
    // CTA holding a (sequence, kv head)'s last chunk)
    for (int sr = w; sr < nseg * 8; sr += kWarps) {
      const int si = sr >> 3, r = sr & 7;
      if (r >= R) continue;
      const SegInfo& sg = ms.seg[si];
      const float* acc = reinterpret_cast<const float*>(smem + kOffAcc + si * kAccBytes);
      const float m_a = acc[8 * D + r], l_a = acc[8 * D + 8 + r];
      const size_t row = ((size_t)sg.b * a.T + r / G) * a.Hq + sg.h * G + (r % G);
      const size_t rr = row * S + sg.slot;
      const float inv = l_a > 0.0f ? 1.0f / l_a : 0.0f;
      for (int d = lane; d < D; d += 32) a.part_o[rr * D + d] = acc[r * D + d] * inv;
      if (lane == 0) a.part_lse[rr] = l_a > 0.0f ? (m_a + log2f(l_a)) * 0.69314718055994531f : -INFINITY;
      for (int sl = sg.empty_from; sl < S; ++sl) {
        for (int d = lane; d < D; d += 32) a.part_o[(row * S + sl) * D + d] = 0.0f;
        if (lane == 0) a.part_lse[row * S + sl] = -INFINITY;
      }
    }
    if (tid == 0) ms.cur = ms.cur_next;
    __syncthreads();
    if (ms.abort) break;
  }
}

}  // namespace flat

bool flat_path_supported(int D, int G, int T, bool latent, int S) { return D == 128 && !latent && T * G <= 8 && S >= 2; }

int flat_grid() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
      n = 1;
  }
  return n;
}

cudaError_t launch_decode_flat(const DecodeArgs& a, cudaStream_t st) {
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
  // the caches as 2-D tensors of (page, head) rows, as the warp-MMA kernel maps
  // them; the maps of the caches a host thread used last are kept
  struct MapCache {
    const void* k = nullptr;
    const void* v = nullptr;
    cuuint64_t rows = 0;
    CUtensorMap kmap, vmap;
  };
  thread_local MapCache mc;
  const cuuint64_t rows = (cuuint64_t)a.num_pages * a.Hkv;
  if (mc.k != a.k_cache || mc.v != a.v_cache || mc.rows != rows) {
    mc.k = nullptr;
    const cuuint64_t dims[2] = {(cuuint64_t)flat::kBlk / 8, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)flat::kBlk};
    const cuuint32_t box[2] = {(cuuint32_t)flat::kBlk / 8, 1};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 2; ++i) {
      if (encode(i ? &mc.vmap : &mc.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2,
                 const_cast<uint8_t*>(i ? a.v_cache : a.k_cache), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    mc.k = a.k_cache;
    mc.v = a.v_cache;
    mc.rows = rows;
  }
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(flat::decode_fp4_flat_kernel, flat::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  flat::decode_fp4_flat_kernel<<<flat_grid(), flat::kThreads, flat::kSmem, st>>>(a, mc.kmap, mc.vmap);
  return cudaGetLastError();
}

}  // namespace kv4
