// kv4_decode.h -- internal interface between the host API and the decode
// kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kv4 {

struct DecodeArgs {
  const uint16_t* q;       // bf16 [B][T][Hq][D], unrotated
  const uint8_t* k_cache;
  const uint8_t* v_cache;  // latent: == k_cache, read with the K layout
  const float* k_scale;    // fp8 only
  const float* v_scale;    // fp8 only
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;           // [B][T][Hq][S][D]
  float* part_lse;         // [B][T][Hq][S]
  int32_t* dev_error;
  int B, T, Hq, Hkv, max_pages, num_pages, S;
  int latent;
  int pos_split;           // 1: query positions split over CTAs, pos_tile per CTA
  int pos_tile;            //    (grid x = S * ceil(T / pos_tile), split-major)
  float qscale;            // softmax_scale * log2(e), times 1/sqrt(D) for the 4-bit rotation
  int diag;                // KV4_DIAG_* test controls (0 in normal calls)
  int causal;              // 1: the last T cached tokens are the query positions (causal among
                           //    them); 0: every cached token precedes the queries and is
                           //    visible to all of them (a leading share of a sequence split
                           //    across devices); context lengths may then be 0
};

// Splits per sequence: about seven CTAs per SM in all (1.75 waves of the
// 4-bit kernel's four resident CTAs; measured best at batch 32, 32K context,
// where more splits add partial-output traffic and per-CTA set-up), at least
// four pages per split.
// The latent (head_dim 512) tcgen05 kernel holds a whole SM: one wave of at
// most one CTA per SM (measured best at batch 8, 96K context).
// Query rows per CTA above which the positions are tiled over CTAs (the
// warp-MMA kernel's three 8-row blocks).
constexpr int kTileRows = 24;

inline int choose_splits(int units, int max_pages, int head_dim, int sms) {
  int s = head_dim == 512 ? sms / units : (7 * sms + units / 2) / units;
  const int cap = max_pages / 4 > 0 ? max_pages / 4 : 1;
  if (s > cap) s = cap;
  if (s > 256) s = 256;
  return s < 1 ? 1 : s;
}

cudaError_t launch_decode_ref(bool fp8, int D, const DecodeArgs& a, cudaStream_t st);
bool fast_path_supported(int D, int G, int T, bool latent);
// flat: one wave of CTAs over equal parts of the step's chunks (T * G <= 24,
// causal, S >= 2 slots per sequence and kv head); else the split form.
cudaError_t launch_decode_fast(int D, const DecodeArgs& a, cudaStream_t st, bool flat = false);
bool mla_path_supported(int D, int G, int T, bool latent);
cudaError_t launch_decode_mla(const DecodeArgs& a, cudaStream_t st);
bool mla_tc_path_supported(int D, int G, int T, bool latent);
bool flat_path_supported(int D, int G, int T, bool latent, int S);
// CTAs of the flat mode's launch for `rows` query rows per kv head: every
// resident slot of every SM (0 on error).
int flat_grid_size(int rows);
cudaError_t launch_decode_mla_tc(const DecodeArgs& a, cudaStream_t st);
bool tc_path_supported(int D, int G, int T, bool latent);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t st);
bool fp8_fast_path_supported(int D, int G, int T);
cudaError_t launch_decode_fp8_fast(const DecodeArgs& a, cudaStream_t st);
bool extend_tc_supported(int D, int G, int T, bool latent);
cudaError_t launch_extend_tc(const DecodeArgs& a, cudaStream_t st);

}  // namespace kv4
