// kv4_noalloc.cu -- decode attention that needs no caller-provided workspace.
//
// kv4_decode_attention writes its split partials into a workspace the caller
// allocates.  Some callers cannot allocate device memory at the point where
// they run attention: an operator plugin that is handed only its input and
// output buffers by the host framework, or a step loop that must not call
// cudaMalloc (it synchronises the device and may fail once a memory pool has
// claimed the GPU).  For them this file keeps the partials in a fixed array
// in device global memory, declared below, and forwards to
// kv4_decode_attention with that array as the workspace.
#include <mutex>

#include "kv4_common.cuh"

namespace {

// The fixed scratch.  It is part of this file's device module: the CUDA
// runtime reserves its bytes on a device when it loads the module there, and
// they stay reserved until the process exits.  Under CUDA's default lazy
// module loading the load happens at the first symbol lookup below, that is
// the first call of the entry point on that device; with eager loading
// (CUDA_MODULE_LOADING=EAGER) it happens when the context is created.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KV4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kv4_status kv4_decode_attention_noalloc(
    const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const int32_t* block_tables,
    const int32_t* context_lens, int batch, int q_per_seq, int num_q_heads, int num_kv_heads,
    int head_dim, int page_size, int max_pages_per_seq, int num_pages, float softmax_scale,
    int num_splits, float* out, int32_t* dev_error, kv4_stream_t stream) {
  if (batch == 0) {
    // nothing to compute: the regular entry point validates the rest of the
    // shape and returns without launching
    return kv4_decode_attention(q, k_cache, v_cache, block_tables, context_lens, batch, q_per_seq,
                                num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                                num_pages, softmax_scale, num_splits, nullptr, 0, out, dev_error, stream);
  }
  if (num_splits < 0) return KV4_ERR_INVALID_ARG;
  int S = num_splits ? num_splits
                     : kv4_decode_auto_splits(batch, q_per_seq, num_q_heads, num_kv_heads, head_dim,
                                              page_size, max_pages_per_seq);
  size_t need = kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, S);
  if (need == 0) {
    // Invalid sizes: let the regular entry point report which one.
    return kv4_decode_attention(q, k_cache, v_cache, block_tables, context_lens, batch, q_per_seq,
                                num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                                num_pages, softmax_scale, S, nullptr, 0, out, dev_error, stream);
  }
  if (need > KV4_NOALLOC_SCRATCH_BYTES) {
    if (num_splits) return KV4_ERR_INVALID_ARG;  // an explicit split count that does not fit
    while (S > 1 && kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, S) >
                        KV4_NOALLOC_SCRATCH_BYTES)
      --S;  // automatic choice: the largest split count whose partials fit
    if (kv4_decode_workspace_bytes(batch, q_per_seq, num_q_heads, head_dim, S) >
        KV4_NOALLOC_SCRATCH_BYTES)
      return KV4_ERR_INVALID_ARG;  // even one split per sequence does not fit
  }
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return KV4_ERR_CUDA;
  return kv4_decode_attention(q, k_cache, v_cache, block_tables, context_lens, batch, q_per_seq,
                              num_q_heads, num_kv_heads, head_dim, page_size, max_pages_per_seq,
                              num_pages, softmax_scale, S, ws, KV4_NOALLOC_SCRATCH_BYTES, out,
                              dev_error, stream);
}
