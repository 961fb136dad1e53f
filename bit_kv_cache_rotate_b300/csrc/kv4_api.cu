// kv4_api.cu -- host side of libkv4: argument validation, split choice and
// kernel dispatch behind the extern "C" entry points declared in kv4.h.
#include <math.h>

#include "kv4_common.cuh"

namespace kv4 {
cudaError_t launch_append_fp4(const void* k, const void* v, int n, int Hkv, int D,
                              const int32_t* slots, uint8_t* kc, uint8_t* vc, int num_pages,
                              double inv_sqrt_d, int32_t* err, cudaStream_t st);
cudaError_t launch_append_fp8(const void* k, const void* v, int n, int Hkv, int D,
                              const int32_t* slots, const float* kinv, const float* vinv,
                              uint8_t* kc, uint8_t* vc, int num_pages, int32_t* err,
                              cudaStream_t st);
cudaError_t launch_combine(const float* po, const float* pl, int rows, int S, int D, int rotate,
                           float inv_sqrt_d, float* out, cudaStream_t st);
int ref_max_rows(int D);
}  // namespace kv4

#include "kv4_decode.h"

namespace {

bool valid_dim(int D) { return D == 64 || D == 128 || D == 256 || D == 512; }

// RN_fp64(1/sqrt(D)): D = 4^k gives an exact power of two; otherwise
// 1/sqrt(D) = (1/sqrt 2) * 2^-(log2(D)-1)/2 and the scaling is exact, so the
// correctly rounded M_SQRT1_2 yields the correctly rounded constant.
double inv_sqrt_dim(int D) {
  int lg = 0;
  while ((1 << lg) < D) ++lg;
  if (lg % 2 == 0) return ldexp(1.0, -lg / 2);
  return ldexp(M_SQRT1_2, -(lg - 1) / 2);
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  }
  return n;
}

kv4_status check_decode_shape(int batch, int T, int Hq, int Hkv, int D, int P, int max_pages,
                              int num_pages) {
  if (batch < 0 || T < 1 || Hq < 1 || Hkv < 1 || max_pages < 1 || num_pages < 1)
    return KV4_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return KV4_ERR_INVALID_ARG;
  if (!valid_dim(D) || P != kv4::kPage || T > KV4_MAX_Q_PER_SEQ) return KV4_ERR_UNSUPPORTED;
  return KV4_OK;
}

}  // namespace

extern "C" {

const char* kv4_status_string(kv4_status s) {
  switch (s) {
    case KV4_OK: return "ok";
    case KV4_ERR_INVALID_ARG: return "invalid argument";
    case KV4_ERR_UNSUPPORTED: return "unsupported shape";
    case KV4_ERR_CUDA: return "CUDA launch error";
    case KV4_ERR_DEVICE_BOUNDS: return "device-side bounds error";
  }
  return "unknown status";
}

size_t kv4_cache_bytes(int num_pages, int num_kv_heads, int page_size, int head_dim) {
  if (num_pages < 0 || num_kv_heads < 0 || page_size <= 0 || head_dim <= 0 || head_dim % 32 ||
      page_size % 2)
    return 0;
  return (size_t)num_pages * num_kv_heads *
         ((size_t)page_size * head_dim / 2 + (size_t)page_size * head_dim / 32);
}

size_t fp8_cache_bytes(int num_pages, int num_kv_heads, int page_size, int head_dim) {
  if (num_pages < 0 || num_kv_heads < 0 || page_size <= 0 || head_dim <= 0) return 0;
  return (size_t)num_pages * num_kv_heads * page_size * head_dim;
}

kv4_status kv4_append_quantize(const void* k, const void* v, int num_tokens, int num_kv_heads,
                               int head_dim, const int32_t* slot_mapping, uint8_t* k_cache,
                               uint8_t* v_cache, int num_pages, int page_size, int32_t* dev_error,
                               kv4_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_pages < 0) return KV4_ERR_INVALID_ARG;
  if (!valid_dim(head_dim) || page_size != kv4::kPage) return KV4_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KV4_OK;
  if (!k || !slot_mapping || !k_cache) return KV4_ERR_INVALID_ARG;
  if ((v == nullptr) != (v_cache == nullptr)) return KV4_ERR_INVALID_ARG;
  if (((uintptr_t)k | (uintptr_t)v) & 7) return KV4_ERR_INVALID_ARG;
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15) return KV4_ERR_INVALID_ARG;
  cudaError_t e = kv4::launch_append_fp4(k, v, num_tokens, num_kv_heads, head_dim, slot_mapping,
                                         k_cache, v_cache, num_pages, inv_sqrt_dim(head_dim),
                                         dev_error, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

kv4_status fp8_append_quantize(const void* k, const void* v, int num_tokens, int num_kv_heads,
                               int head_dim, const int32_t* slot_mapping,
                               const float* k_inv_scale, const float* v_inv_scale,
                               uint8_t* k_cache, uint8_t* v_cache, int num_pages, int page_size,
                               int32_t* dev_error, kv4_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_pages < 0) return KV4_ERR_INVALID_ARG;
  if (!valid_dim(head_dim) || page_size != kv4::kPage) return KV4_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KV4_OK;
  if (!k || !v || !slot_mapping || !k_inv_scale || !v_inv_scale || !k_cache || !v_cache)
    return KV4_ERR_INVALID_ARG;
  if (((uintptr_t)k | (uintptr_t)v) & 7) return KV4_ERR_INVALID_ARG;
  if (((uintptr_t)k_cache | (uintptr_t)v_cache) & 15) return KV4_ERR_INVALID_ARG;
  cudaError_t e = kv4::launch_append_fp8(k, v, num_tokens, num_kv_heads, head_dim, slot_mapping,
                                         k_inv_scale, v_inv_scale, k_cache, v_cache, num_pages,
                                         dev_error, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

int kv4_decode_auto_splits(int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                           int head_dim, int page_size, int max_pages_per_seq) {
  (void)page_size;
  if (batch < 1 || num_kv_heads < 1 || max_pages_per_seq < 1 || q_per_seq < 1 || num_q_heads < 1) return 1;
  // CTAs per split: one per (sequence, kv head) and position tile
  const long long rows = (long long)q_per_seq * (num_q_heads / num_kv_heads > 0 ? num_q_heads / num_kv_heads : 1);
  const long long tiles = rows > kv4::kTileRows ? (rows + kv4::kTileRows - 1) / kv4::kTileRows : 1;
  const long long units = (long long)batch * num_kv_heads * tiles;
  return kv4::choose_splits(units > (1 << 30) ? (1 << 30) : (int)units, max_pages_per_seq, head_dim, sm_count());
}

size_t kv4_decode_workspace_bytes(int batch, int q_per_seq, int num_q_heads, int head_dim,
                                  int num_splits) {
  if (batch < 0 || q_per_seq < 1 || num_q_heads < 1 || head_dim < 1 || num_splits < 1) return 0;
  const size_t rows = (size_t)batch * q_per_seq * num_q_heads;
  const size_t o = rows * num_splits * head_dim * sizeof(float);
  const size_t l = rows * num_splits * sizeof(float);
  return ((o + 255) / 256) * 256 + l;
}

// Automatic kernel choice.  By shape: extend steps (more query rows than the
// warp-MMA kernel holds per CTA) on the tcgen05 extend kernel, the latent
// cache on the tcgen05 latent kernel, head_dim 128 with up to 24 query rows
// per kv head on the warp-MMA kernel, everything else on the general kernel.
// The extend kernel's tile is 128 query rows; a block of a few positions (a
// 6-token verify: 48 rows) leaves most of it idle and runs slower than the
// warp-MMA kernel's position tiles reading the pages once per 24 rows (L2
// serves the repeats), so only blocks above 96 rows (four tiles of 24) go to
// the extend kernel.  Up to 8 rows per kv head, the warp-MMA kernel runs in
// flat mode (one wave of CTAs over equal parts of the step's chunks) when the
// S slots allow a wave's worth of equal parts of sequences of the table's full
// length: (S - 1) x units >= the wave's CTAs; otherwise (few slots for many
// sequences) the split form.  With more rows (a verify block) the flat mode
// measured slower (two CTAs per SM, its parts cross the shared prefix at
// different times) and is an explicit choice only.
static int auto_kernel(bool fp8, int D, int G, int T, bool latent, bool causal, int S, long long units) {
  if (!fp8 && kv4::extend_tc_supported(D, G, T, latent) && T * G > 4 * kv4::kTileRows) return KV4_KERNEL_EXTEND;
  if (!fp8 && kv4::mla_tc_path_supported(D, G, T, latent)) return KV4_KERNEL_LATENT_TC;
  if (!fp8 && causal && T * G <= 8 && kv4::flat_path_supported(D, G, T, latent, S)) {
    const int grid = kv4::flat_grid_size(T * G);
    if (grid > 0 && (long long)(S - 1) * units >= grid) return KV4_KERNEL_BALANCED;
  }
  const bool ok_warp = fp8 ? kv4::fp8_fast_path_supported(D, G, T) : kv4::fast_path_supported(D, G, T, latent);
  return ok_warp ? KV4_KERNEL_WARP_MMA : KV4_KERNEL_GENERAL;
}

int kv4_decode_kernel_choice(int batch, int q_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                             int num_splits, int latent) {
  if (batch < 1 || q_per_seq < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || num_q_heads % num_kv_heads ||
      !valid_dim(head_dim) || num_splits < 1)
    return -1;
  return auto_kernel(false, head_dim, num_q_heads / num_kv_heads, q_per_seq, latent != 0, true, num_splits,
                     (long long)batch * num_kv_heads);
}

static kv4_status decode_common(bool fp8, const void* q, const uint8_t* k_cache,
                                const uint8_t* v_cache, const float* k_scale,
                                const float* v_scale, const int32_t* block_tables,
                                const int32_t* context_lens, int batch, int T, int Hq, int Hkv,
                                int D, int P, int max_pages, int num_pages, float softmax_scale,
                                int num_splits, void* workspace, size_t workspace_bytes,
                                float* out, int32_t* dev_error, cudaStream_t st,
                                bool combine = true, int kernel = KV4_KERNEL_AUTO, int diag = 0,
                                bool causal = true) {
  kv4_status s = check_decode_shape(batch, T, Hq, Hkv, D, P, max_pages, num_pages);
  if (s != KV4_OK) return s;
  if (batch == 0) return KV4_OK;
  if (!q || !k_cache || !block_tables || !context_lens || !workspace || (combine && !out))
    return KV4_ERR_INVALID_ARG;
  if (!combine && num_splits < 1) return KV4_ERR_INVALID_ARG;
  // The kernels take the softmax maximum over unscaled logits; a positive,
  // finite factor keeps that maximum the maximum of the scaled ones.
  if (!(softmax_scale > 0.0f) || !isfinite(softmax_scale)) return KV4_ERR_INVALID_ARG;
  if (fp8 && (!v_cache || !k_scale || !v_scale)) return KV4_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)k_cache & 15) || ((uintptr_t)v_cache & 15) ||
      ((uintptr_t)workspace & 255) || (combine && ((uintptr_t)out & 15)))
    return KV4_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > 4096) return KV4_ERR_INVALID_ARG;
  const int S = num_splits ? num_splits
                           : kv4_decode_auto_splits(batch, T, Hq, Hkv, D, P, max_pages);
  if (workspace_bytes < kv4_decode_workspace_bytes(batch, T, Hq, D, S)) return KV4_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  const bool latent = !fp8 && (v_cache == nullptr || v_cache == k_cache);

  const size_t rows = (size_t)batch * T * Hq;
  float* part_o = static_cast<float*>(workspace);
  const size_t o_bytes = ((rows * S * D * sizeof(float) + 255) / 256) * 256;
  float* part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes);

  kv4::DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k_cache = k_cache;
  a.v_cache = latent ? k_cache : v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.dev_error = dev_error;
  a.B = batch;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.S = S;
  a.latent = latent ? 1 : 0;
  const double log2e = 1.4426950408889634;
  a.qscale = (float)(softmax_scale * log2e * (fp8 ? 1.0 : inv_sqrt_dim(D)));

  a.diag = diag;
  a.causal = causal ? 1 : 0;
  a.pos_split = 0;
  a.pos_tile = 1;

  // An explicit choice (kv4_decode_attention_select) must serve the shape.
  const bool ok_tc = !fp8 && kv4::tc_path_supported(D, G, T, latent);
  const bool ok_ext = !fp8 && kv4::extend_tc_supported(D, G, T, latent);
  const bool ok_mla = !fp8 && kv4::mla_path_supported(D, G, T, latent);
  const bool ok_mla_tc = !fp8 && kv4::mla_tc_path_supported(D, G, T, latent);
  const bool ok_flat = !fp8 && causal && kv4::flat_path_supported(D, G, T, latent, S);
  const bool ok_warp = fp8 ? kv4::fp8_fast_path_supported(D, G, T) : kv4::fast_path_supported(D, G, T, latent);
  const bool ok_gen = T * G <= kv4::ref_max_rows(D);
  const int k = kernel == KV4_KERNEL_AUTO ? auto_kernel(fp8, D, G, T, latent, causal, S, (long long)batch * Hkv)
                                          : kernel;
  cudaError_t e;
  switch (k) {
    case KV4_KERNEL_TCGEN05:
      if (!ok_tc) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_decode_tc(a, st);
      break;
    case KV4_KERNEL_EXTEND:
      if (!ok_ext) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_extend_tc(a, st);
      break;
    case KV4_KERNEL_LATENT:
      if (!ok_mla) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_decode_mla(a, st);
      break;
    case KV4_KERNEL_LATENT_TC:
      if (!ok_mla_tc) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_decode_mla_tc(a, st);
      break;
    case KV4_KERNEL_BALANCED:
      if (!ok_flat) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_decode_fast(D, a, st, true);
      break;
    case KV4_KERNEL_WARP_MMA:
      if (!ok_warp) return KV4_ERR_UNSUPPORTED;
      if (fp8) {
        a.pos_split = T * G > 8 ? 1 : 0;
        e = kv4::launch_decode_fp8_fast(a, st);
      } else {
        e = kv4::launch_decode_fast(D, a, st);  // chooses row blocks or pos_split
      }
      break;
    case KV4_KERNEL_GENERAL:
      if (!ok_gen) return KV4_ERR_UNSUPPORTED;
      e = kv4::launch_decode_ref(fp8, D, a, st);
      break;
    default:
      return KV4_ERR_INVALID_ARG;
  }
  if (e != cudaSuccess) return KV4_ERR_CUDA;
  if (!combine) return KV4_OK;
  e = kv4::launch_combine(part_o, part_lse, (int)rows, S, D, fp8 ? 0 : 1,
                          (float)inv_sqrt_dim(D), out, st);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

kv4_status kv4_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                                float softmax_scale, int num_splits, void* workspace,
                                size_t workspace_bytes, float* out, int32_t* dev_error,
                                kv4_stream_t stream) {
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                       batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                       max_pages_per_seq, num_pages, softmax_scale, num_splits, workspace,
                       workspace_bytes, out, dev_error, (cudaStream_t)stream);
}

kv4_status kv4_decode_attention_select(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                       int head_dim, int page_size, int max_pages_per_seq,
                                       int num_pages, float softmax_scale, int num_splits,
                                       void* workspace, size_t workspace_bytes, float* out,
                                       int32_t* dev_error, int kernel, int diag_flags,
                                       kv4_stream_t stream) {
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                       batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                       max_pages_per_seq, num_pages, softmax_scale, num_splits, workspace,
                       workspace_bytes, out, dev_error, (cudaStream_t)stream, true, kernel, diag_flags);
}

kv4_status kv4_decode_partials(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                               int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                               float softmax_scale, int num_splits, void* workspace,
                               size_t workspace_bytes, int32_t* dev_error, kv4_stream_t stream) {
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                       batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                       max_pages_per_seq, num_pages, softmax_scale, num_splits, workspace,
                       workspace_bytes, nullptr, dev_error, (cudaStream_t)stream, false);
}

kv4_status kv4_decode_partials_prefix(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, int max_pages_per_seq,
                                      int num_pages, float softmax_scale, int num_splits,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_error,
                                      kv4_stream_t stream) {
  return decode_common(false, q, k_cache, v_cache, nullptr, nullptr, block_tables, context_lens,
                       batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                       max_pages_per_seq, num_pages, softmax_scale, num_splits, workspace,
                       workspace_bytes, nullptr, dev_error, (cudaStream_t)stream, false,
                       KV4_KERNEL_AUTO, 0, false);
}

kv4_status fp8_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                                float softmax_scale, int num_splits, void* workspace,
                                size_t workspace_bytes, float* out, int32_t* dev_error,
                                kv4_stream_t stream) {
  return decode_common(true, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                       batch, q_per_seq, num_q_heads, num_kv_heads, head_dim, page_size,
                       max_pages_per_seq, num_pages, softmax_scale, num_splits, workspace,
                       workspace_bytes, out, dev_error, (cudaStream_t)stream);
}

kv4_status kv4_split_combine(const float* partial_o, const float* partial_lse, int batch,
                             int q_per_seq, int num_q_heads, int head_dim, int num_splits,
                             float* out, kv4_stream_t stream) {
  if (batch < 0 || q_per_seq < 1 || num_q_heads < 1 || num_splits < 1) return KV4_ERR_INVALID_ARG;
  if (!valid_dim(head_dim)) return KV4_ERR_UNSUPPORTED;
  if (batch == 0) return KV4_OK;
  if (!partial_o || !partial_lse || !out) return KV4_ERR_INVALID_ARG;
  const int rows = batch * q_per_seq * num_q_heads;
  cudaError_t e = kv4::launch_combine(partial_o, partial_lse, rows, num_splits, head_dim, 1,
                                      (float)inv_sqrt_dim(head_dim), out, (cudaStream_t)stream);
  return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

}  // extern "C"
