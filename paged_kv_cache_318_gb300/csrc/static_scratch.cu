// pkv_paged_attention_varlen_static_scratch: the attention entry point for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: plugin hosts and
// serving runtimes that plan every device byte up front and expose no scratch
// to an individual call, and latency-critical loops that must not call
// cudaMalloc/cudaFree, which can block the host and synchronise the whole
// device (stalling work on every other stream).  This entry point takes the
// split-KV scratch from a fixed array that lives in the library's own device
// memory instead, and allocates nothing.
//
// The array is a file-scope __device__ array, so every GPU that loads the
// library holds its kStaticScratchBytes until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it.
#include <stdio.h>


#include "pkv_common.cuh"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char
    g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  Looked up on
// every call (a host-side lookup once the module is loaded, no allocation),
// so that a device reset, which reloads the module, cannot leave a stale
// address behind.
cudaError_t scratch_address(void** out) {
  return cudaGetSymbolAddress(out, g_static_scratch);
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attention_varlen_static_scratch(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], void* out, int64_t o_stride_tok,
    int64_t o_stride_head, const int32_t* cu_seqlens_q,
    const int32_t* seqused_k, int batch, int total_q, int max_seqlen_q,
    int max_seqlen_k, const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, float softmax_scale, int causal,
    int window_left, int window_right, float softcap,
    const float* alibi_slopes, int num_splits, float* softmax_lse,
    pkv_dtype dtype, pkv_stream_t stream) {
  // the scratch must hold what the call requires; the optional prefill
  // tail (item counter, split partials) is used when it fits as well
  const size_t need = pkv::required_workspace_bytes(
      batch, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
      head_size, block_size, causal, window_left, window_right, num_splits);
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  if (need != static_cast<size_t>(-1)) {
    if (need > pkv::kStaticScratchBytes) {
      char msg[256];
      snprintf(msg, sizeof(msg),
               "this call needs %zu bytes of split-KV scratch but the "
               "built-in scratch holds %zu; call pkv_paged_attention_varlen "
               "with a workspace, or use fewer splits or a smaller batch",
               need, pkv::kStaticScratchBytes);
      pkv::set_last_error(msg);
      return PKV_ERR_WORKSPACE_TOO_SMALL;
    }
    cudaError_t e = pkv::scratch_address(&scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static scratch): %s",
               cudaGetErrorString(e));
      pkv::set_last_error(msg);
      return PKV_ERR_CUDA;
    }
    scratch_bytes = pkv::kStaticScratchBytes;
  }
  // (invalid arguments make need == (size_t)-1; the regular entry point
  // then rejects them with its own message)
  return pkv_paged_attention_varlen(
      q, q_stride_tok, q_stride_head, key_cache, value_cache, cache_strides,
      out, o_stride_tok, o_stride_head, cu_seqlens_q, seqused_k, batch,
      total_q, max_seqlen_q, max_seqlen_k, block_table, block_table_stride,
      max_blocks_per_seq, num_heads, num_kv_heads, head_size, block_size,
      num_blocks, softmax_scale, causal, window_left, window_right, softcap,
      alibi_slopes, num_splits, softmax_lse, scratch, scratch_bytes, dtype,
      stream);
}

}  // extern "C"
