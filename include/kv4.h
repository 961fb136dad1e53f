/*
 * kv4.h -- C ABI of libkv4: 4-bit rotated KV-cache decode attention on B300.
 *
 * The method is the one described on the "UltraQuant on AMD Instinct" page:
 *   section "What is UltraQuant"  -- every key/value head vector is rotated by
 *     a Walsh-Hadamard transform, then stored as FP4 (E2M1) codes with one
 *     shared power-of-two (UE8M0) scale per 32 channels: 17 bytes per 32
 *     values instead of 32 for an 8-bit cache; the attention kernel consumes
 *     the FP4 codes directly and applies the power-of-two scale as part of the
 *     multiply, with no lookup-table dequantisation;
 *   section "Why UltraQuant beats 8-bit KV" -- each decode step re-reads the
 *     whole cache, so the step time follows the cache bytes;
 *   section "Throughput-latency trade-off" -- MTP verify: several query
 *     positions of one sequence share one paged cache, causal among them.
 *
 * Conventions for every entry point
 *   - Pointers marked "device" are device (HBM) pointers owned by the caller;
 *     the library never allocates, frees or synchronises.  All work is queued
 *     on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Host-side validation runs first and returns KV4_ERR_INVALID_ARG or
 *     KV4_ERR_UNSUPPORTED without launching anything.  A failed launch returns
 *     KV4_ERR_CUDA.  Errors found on the device (a page id outside
 *     [0, num_pages), a context length outside [q_per_seq, max_pages *
 *     page_size], a slot outside the cache) skip the offending work and set
 *     *dev_error to a nonzero KV4_DEVERR_* bit when dev_error is non-NULL; the
 *     caller reads it after synchronising.  No kernel traps or waits on
 *     another block.
 *   - Supported: head_dim in {64, 128, 256, 512}; page_size 16; num_q_heads a
 *     multiple of num_kv_heads; q_per_seq (T) in 1..KV4_MAX_Q_PER_SEQ.  The
 *     query rows per kv head, R = T * num_q_heads / num_kv_heads, are
 *     unlimited for head_dim 128 with at most 8 query heads per kv head
 *     (4-bit cache without the latent mode, and the FP8 cache); every other
 *     shape takes R up to 64 (32 at head_dim 256, 16 at 512) and returns
 *     KV4_ERR_UNSUPPORTED above that.
 *   - Entry points are thread-safe.  Their only process-wide state is set up
 *     once and never changes results: each kernel's raised shared-memory
 *     limit (per device), the driver's tensor-map encoder (looked up once),
 *     per host thread the tensor maps (address and sizes) of the caches that
 *     thread decoded last, re-encoded whenever a cache pointer or size
 *     differs, and for kv4_decode_attention_noalloc the address of its
 *     scratch array (per device; that array's ordering rule is stated there).
 *     Nothing reads the environment; the kernel choice depends on the shape
 *     alone (kv4_decode_attention_select makes it explicit).
 *
 * Cache layout (one block per (page, kv head), blocks page-major:
 * block index = page * num_kv_heads + head, block bytes = P*D/2 + P*D/32):
 *   K block (also the latent cache):
 *     codes  tiles of 8 tokens x 32 channels (128 bytes): tile (t/8, d/32)
 *            starts at byte ((t/8)*(D/32) + d/32)*128; inside it token t%8
 *            takes 16 bytes, byte (d%32)/2 holding channel d (low nibble =
 *            even channel).  This is the 8-row core-matrix order in which
 *            the block-scaled tensor-core MMA reads its K operand.
 *     scales [P][D/32] one UE8M0 byte (exponent + 127) per (token, group)
 *   V block:
 *     codes  [D][P/2]  channel-major: byte (d, j) = token 2j (low nibble),
 *                      token 2j+1 (high nibble) of channel d
 *     scales [P][D/32] as for K
 * Codes are OCP E2M1 nibbles (sign | 2 exponent bits | 1 mantissa bit).
 * Values are stored in the rotated space: y = H_D x with H_D the orthonormal
 * Sylvester Walsh-Hadamard matrix (natural order); q is rotated by the same
 * H_D inside the decode call and the output is rotated back, so callers pass
 * and receive unrotated vectors.
 */
#ifndef KV4_H_
#define KV4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kv4_stream_t; /* same type as cudaStream_t */

typedef enum {
  KV4_OK = 0,
  KV4_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad relation between sizes */
  KV4_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim, page_size, T) */
  KV4_ERR_CUDA = 3,          /* a kernel launch failed */
  KV4_ERR_DEVICE_BOUNDS = 4  /* reserved for callers that fold *dev_error into a status */
} kv4_status;

/* Bits written to *dev_error by kernels. */
/* Largest q_per_seq: decode (1), MTP verify (a few) and extend steps (a
 * chunk of new tokens over a cached prefix) share one entry point. */
#define KV4_MAX_Q_PER_SEQ 4096

#define KV4_DEVERR_PAGE 1      /* block_tables entry outside [0, num_pages) */
#define KV4_DEVERR_CONTEXT 2   /* context_lens[b] outside [q_per_seq, max_pages*page_size]
                                  ([0, ...] for kv4_decode_partials_prefix) */
#define KV4_DEVERR_SLOT 4      /* slot_mapping entry outside the cache */
#define KV4_DEVERR_TIMEOUT 8   /* a bounded wait for streamed cache data gave up */

/* Human-readable name of a status. */
const char* kv4_status_string(kv4_status s);

/* Bytes of one 4-bit cache (K, V or latent): num_pages * num_kv_heads *
 * (page_size*head_dim/2 + page_size*head_dim/32) -- 17 bytes per 32 values
 * ("What is UltraQuant").  Returns 0 for invalid sizes. */
size_t kv4_cache_bytes(int num_pages, int num_kv_heads, int page_size, int head_dim);

/* Quantise-on-append ("What is UltraQuant": rotation, FP4 codes, one
 * power-of-two scale per 32 channels).
 *   k, v          device bf16 [num_tokens][num_kv_heads][head_dim], unrotated.
 *                 v == NULL selects the latent cache (MLA): only k is written,
 *                 into k_cache, and v_cache must be NULL too.
 *   slot_mapping  device int32 [num_tokens]: token i goes to page
 *                 slot/page_size, row slot%page_size; negative slots skip.
 *   k_cache, v_cache  device uint8, kv4_cache_bytes(num_pages, ...) each.
 * Per (token, head): y = fp32(fp64(exact(H+-1 . x)) * RN64(1/sqrt(D))); per
 * 32-channel group e = clamp(floor(log2 max|y|) - 2, -127, 127) (e = -127 for
 * an all-zero group); code = RNE_E2M1_saturating(y / 2^e) with the sign bit
 * kept for nonzero values that round to zero (an exact zero y is +0); the
 * scale byte is e + 127.
 * Codes and scales are bit-exact for vectors whose exact Hadamard sum is
 * representable in binary64 (in-vector dynamic range below about 2^40).
 * Concurrent appends to the two tokens sharing a V byte are safe. */
kv4_status kv4_append_quantize(const void* k, const void* v, int num_tokens, int num_kv_heads,
                               int head_dim, const int32_t* slot_mapping, uint8_t* k_cache,
                               uint8_t* v_cache, int num_pages, int page_size, int32_t* dev_error,
                               kv4_stream_t stream);

/* Number of KV splits the decode uses when called with num_splits = 0. */
int kv4_decode_auto_splits(int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                           int head_dim, int page_size, int max_pages_per_seq);

/* Workspace bytes for kv4_decode_attention / fp8_decode_attention with the
 * given split count: partial outputs fp32 [B][T][Hq][S][D] and log-sum-exp
 * fp32 [B][T][Hq][S]. */
size_t kv4_decode_workspace_bytes(int batch, int q_per_seq, int num_q_heads, int head_dim,
                                  int num_splits);

/* Paged decode attention over the 4-bit cache ("What is UltraQuant", "Why
 * UltraQuant beats 8-bit KV"; T > 1 is the MTP verify block of
 * "Throughput-latency trade-off"; a large T is an extend step, a chunk of
 * new prompt tokens over a long cached prefix, the prefill side of the
 * agentic traffic in "Agentic serving" and of the time to first token in
 * "Key results").
 *   q             device bf16 [batch][q_per_seq][num_q_heads][head_dim], unrotated.
 *                 Query head hq reads kv head hq / (num_q_heads/num_kv_heads).
 *   k_cache       device, layout above.  v_cache: device, or NULL / == k_cache
 *                 for the latent cache (K = V = latent row).
 *   block_tables  device int32 [batch][max_pages_per_seq] physical page ids.
 *   context_lens  device int32 [batch]: tokens in the cache for each sequence,
 *                 counting the q_per_seq new ones.  Query position j attends
 *                 to tokens t < context_lens[b] - q_per_seq + 1 + j.
 *   softmax_scale multiplies q.k before the softmax; finite and > 0, else
 *                 KV4_ERR_INVALID_ARG.
 *   num_splits    KV splits per sequence: partial slots per (sequence, kv
 *                 head), 0 = kv4_decode_auto_splits.  The split form cuts each
 *                 sequence into num_splits equal parts; the flat mode (up to 24
 *                 query rows per kv head) cuts the step's chunks into one
 *                 wave of equal parts, of which a sequence's kv head spans at
 *                 most num_splits.
 *   workspace     device, >= kv4_decode_workspace_bytes(...) bytes.
 *   out           device fp32 [batch][q_per_seq][num_q_heads][head_dim],
 *                 unrotated: out = softmax(s q.k) . v over the dequantised cache.
 * Runs the split decode kernel then kv4_split_combine. */
kv4_status kv4_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                                float softmax_scale, int num_splits, void* workspace,
                                size_t workspace_bytes, float* out, int32_t* dev_error,
                                kv4_stream_t stream);

/* The split stage of kv4_decode_attention alone: writes the per-split
 * partial outputs (rotated space, each normalised by its own softmax sum)
 * and log-sum-exps into `workspace` laid out as described for
 * kv4_split_combine (partial_o at offset 0, partial_lse at offset
 * round_up(B*T*Hq*S*D*4, 256)).  num_splits must be > 0 here (use
 * kv4_decode_auto_splits to pick one).  kv4_decode_attention is this call
 * followed by kv4_split_combine. */
kv4_status kv4_decode_partials(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                               int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                               float softmax_scale, int num_splits, void* workspace,
                               size_t workspace_bytes, int32_t* dev_error, kv4_stream_t stream);

/* The split stage over a leading share of each sequence's cache, for one
 * long context split across devices ("GLM-5.3-Flash on MI300X": sharding the
 * KV cache instead of replicating it is what frees capacity for long
 * contexts).  A sequence's pages are cut into consecutive shares, one per
 * device; the device that holds the newest tokens (the q_per_seq query
 * positions and everything after the other shares) calls
 * kv4_decode_partials on its share, every other device calls this entry point
 * on its own.  Here every cached token precedes the query positions, so all of
 * them are visible to every position (no causal mask); context_lens[b] is the
 * share's token count and may be 0 (an empty share writes empty partials:
 * lse = -inf).  Arguments, layout and errors are those of kv4_decode_partials.
 * The partials of all shares, gathered into one device's memory and
 * concatenated along the split axis (partial_o [B][T][Hq][S_total][D],
 * partial_lse [B][T][Hq][S_total]), merge with kv4_split_combine into the
 * attention over the whole sequence: the log-sum-exp merge is exact whatever
 * the order and grouping of the splits. */
kv4_status kv4_decode_partials_prefix(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                      int head_dim, int page_size, int max_pages_per_seq,
                                      int num_pages, float softmax_scale, int num_splits,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_error,
                                      kv4_stream_t stream);

/* Decode attention for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for callers
 * such as operator plugins that the host framework hands only input and
 * output buffers, or step loops that must not call cudaMalloc (it
 * synchronises the device and can fail once a memory pool owns the GPU).
 * Arguments and results are those of kv4_decode_attention without the
 * workspace: the split partials live in a fixed array of
 * KV4_NOALLOC_SCRATCH_BYTES bytes in device global memory that libkv4
 * declares itself.  The call itself allocates nothing and calls no
 * allocating routine (no cudaMalloc, no memory-pool or library allocator).
 *   - The array is reserved on a device when the CUDA runtime loads the
 *     library's module that holds it there.  Under CUDA's default lazy module
 *     loading that is the first call of this entry point on the device (its
 *     address lookup loads the module), so that first call can fail with
 *     KV4_ERR_CUDA if the device has no 16 MiB left; with
 *     CUDA_MODULE_LOADING=EAGER it is reserved when the context is created.
 *     Make the first call during set-up, before a memory pool takes the
 *     device's free memory; the array then stays reserved until the process
 *     exits and later calls reserve nothing.
 *   - num_splits = 0 picks kv4_decode_auto_splits, lowered if needed to the
 *     largest count whose partials (kv4_decode_workspace_bytes) fit.  An
 *     explicit num_splits whose partials do not fit, or a request that does
 *     not fit even with one split per sequence, returns KV4_ERR_INVALID_ARG
 *     before anything is launched.  batch = 0 is validated like
 *     kv4_decode_attention and launches nothing.
 *   - The first call on each device also looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - All calls share the array, which keeps what the last call wrote.
 *     Nothing in it has to start at zero: the kernels write every partial
 *     they read back.  Calls whose GPU work overlaps (other streams, other
 *     host threads without ordering) race on the array and give wrong
 *     results; order them. */
#define KV4_NOALLOC_SCRATCH_BYTES (16u << 20)
kv4_status kv4_decode_attention_noalloc(const void* q, const uint8_t* k_cache,
                                        const uint8_t* v_cache, const int32_t* block_tables,
                                        const int32_t* context_lens, int batch, int q_per_seq,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int page_size, int max_pages_per_seq, int num_pages,
                                        float softmax_scale, int num_splits, float* out,
                                        int32_t* dev_error, kv4_stream_t stream);

/* ---------------------------------------------------------------------
 * Kernel choice and test controls (diagnostics).
 *
 * kv4_decode_attention picks the split kernel from the shape (and, for the
 * flat mode, from num_splits and the device's SM count).  This
 * entry point is the same call with that choice made explicit, for tests and
 * measurements that compare the kernels on one input.  Every kernel computes
 * the same attention (the results differ by accumulation order, well inside
 * the 2e-3 parity tolerance); a kernel that does not serve the shape returns
 * KV4_ERR_UNSUPPORTED before anything is launched.  No global state: the
 * choice applies to this call only.
 * --------------------------------------------------------------------- */
#define KV4_KERNEL_AUTO 0      /* what kv4_decode_attention picks */
#define KV4_KERNEL_WARP_MMA 1  /* warp-MMA kernel: head_dim 128, <= 8 query heads per kv head;
                                  up to 24 rows per CTA, more rows as position tiles */
#define KV4_KERNEL_EXTEND 2    /* tcgen05 extend kernel: head_dim 128, G in {1,2,4,8}, > 24 rows */
#define KV4_KERNEL_LATENT 3    /* warp-MMA latent (MLA) kernel: head_dim 512, K = V, <= 16 rows */
#define KV4_KERNEL_GENERAL 4   /* CUDA-core kernel: every shape within the documented row limits */
#define KV4_KERNEL_TCGEN05 5   /* warp-specialised tcgen05 decode kernel: head_dim 128, <= 8 rows
                                  (T * num_q_heads / num_kv_heads <= 8) */
#define KV4_KERNEL_LATENT_TC 6 /* warp-specialised tcgen05 latent (MLA) kernel: head_dim 512,
                                  K = V, <= 16 rows; one CTA per SM */
#define KV4_KERNEL_BALANCED 7  /* warp-MMA kernel in flat mode: head_dim 128, <= 24 rows, num_splits >= 2,
                                  not the prefix form; one wave of CTAs, each an equal share of
                                  the step's 64-token chunks in (sequence, kv head) order; a
                                  sequence and kv head spans at most num_splits CTAs (its
                                  partial slots) */

/* Test controls (bits of diag_flags; 0 in normal use).
 * KV4_DIAG_EXPIRE_FIRST_WAIT: the first bounded wait of every warp that streams
 *   cache data gives up without trying, as a wait that ran out would.  The
 *   kernel then sets KV4_DEVERR_TIMEOUT in *dev_error, waits (bounded) for
 *   the copies it issued, and returns; the output is not meaningful.  It
 *   exercises the timeout path without a fault or a hang; kernels without
 *   streamed waits (the general kernel) ignore it. */
#define KV4_DIAG_EXPIRE_FIRST_WAIT 1

kv4_status kv4_decode_attention_select(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                       const int32_t* block_tables, const int32_t* context_lens,
                                       int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                       int head_dim, int page_size, int max_pages_per_seq,
                                       int num_pages, float softmax_scale, int num_splits,
                                       void* workspace, size_t workspace_bytes, float* out,
                                       int32_t* dev_error, int kernel, int diag_flags,
                                       kv4_stream_t stream);

/* The KV4_KERNEL_* id that kv4_decode_attention (4-bit cache, causal form)
 * would run for this shape with num_splits slots (>= 1; pass the value the
 * call would use, e.g. kv4_decode_auto_splits) on the current device; latent
 * != 0 for the latent cache (v_cache NULL or == k_cache).  -1 for an invalid
 * shape.  Host only; it reads the device's SM count and the flat mode's
 * occupancy once. */
int kv4_decode_kernel_choice(int batch, int q_per_seq, int num_q_heads, int num_kv_heads, int head_dim,
                             int num_splits, int latent);

/* Log-sum-exp merge of split partials, then the inverse rotation:
 *   lse = log sum_s exp(lse_s);  O = sum_s exp(lse_s - lse) O_s;  out = H_D O.
 *   partial_o    device fp32 [batch][q_per_seq][num_q_heads][num_splits][head_dim]
 *                (each O_s already normalised by its own softmax sum)
 *   partial_lse  device fp32 [batch][q_per_seq][num_q_heads][num_splits]
 *                (natural log; -inf marks an empty split)
 *   out          device fp32 [batch][q_per_seq][num_q_heads][head_dim].
 * The page does not describe a split or its merge; this is the standard
 * blockwise-softmax merge. */
kv4_status kv4_split_combine(const float* partial_o, const float* partial_lse, int batch,
                             int q_per_seq, int num_q_heads, int head_dim, int num_splits,
                             float* out, kv4_stream_t stream);

/* ---------------------------------------------------------------------
 * FP8 comparator: the 8-bit KV cache the page measures UltraQuant against
 * ("UltraQuant vs 8-bit KV": standard FP8 cache on the AITER backends).
 * E4M3 (OCP) with one fp32 scale per kv head, no rotation.
 * Block per (page, kv head): K [P][D] token-major bytes, V [D][P]
 * channel-major bytes; block bytes = P*D.
 * --------------------------------------------------------------------- */
size_t fp8_cache_bytes(int num_pages, int num_kv_heads, int page_size, int head_dim);

/* code = E4M3_RNE_satfinite(fp32(x * inv_scale[h])).
 *   k_inv_scale, v_inv_scale  device fp32 [num_kv_heads]. */
kv4_status fp8_append_quantize(const void* k, const void* v, int num_tokens, int num_kv_heads,
                               int head_dim, const int32_t* slot_mapping,
                               const float* k_inv_scale, const float* v_inv_scale,
                               uint8_t* k_cache, uint8_t* v_cache, int num_pages, int page_size,
                               int32_t* dev_error, kv4_stream_t stream);

/* As kv4_decode_attention over the FP8 cache; k_scale, v_scale: device fp32
 * [num_kv_heads] (dequantised value = E4M3 value * scale). */
kv4_status fp8_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, const int32_t* context_lens,
                                int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
                                int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                                float softmax_scale, int num_splits, void* workspace,
                                size_t workspace_bytes, float* out, int32_t* dev_error,
                                kv4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KV4_H_ */
