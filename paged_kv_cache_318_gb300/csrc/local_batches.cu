// Chunked local attention: split requests into chunk-aligned virtual
// requests (host code; the attention itself runs on the regular kernels).
//
// Source: "vllm.v1.attention.backends.flash_attn" (vLLM v0.9.0.1 docs),
// make_local_attention_virtual_batches and its use in
// FlashAttentionMetadataBuilder.build.  With chunk size C, a request with
// q queries (positions L - q .. L - 1) yields one virtual request per C-wide
// key chunk that holds a query; the virtual request's queries attend
// causally to that chunk's keys only, through the chunk's own slice of the
// block table.
#include <stdio.h>
#include <string.h>

#include "pkv_common.cuh"

extern "C" {

pkv_status pkv_make_local_attention_virtual_batches(
    int attn_chunk_size, const int32_t* query_start_loc,
    const int32_t* seq_lens, int batch, const int32_t* block_table,
    int64_t block_table_stride, int max_blocks_per_seq, int block_size,
    int* num_virtual, int32_t* seqlens_q_local, int32_t* cu_seqlens_q_local,
    int32_t* seqlens_k_local, int32_t* block_table_local, int capacity) {
  char msg[256];
  if (attn_chunk_size <= 0 || block_size <= 0 ||
      attn_chunk_size % block_size != 0) {
    snprintf(msg, sizeof(msg),
             "attn_chunk_size %d must be a positive multiple of block_size %d",
             attn_chunk_size, block_size);
    pkv::set_last_error(msg);
    return PKV_ERR_INVALID_ARG;
  }
  if (batch < 0 || !num_virtual || (batch > 0 && (!query_start_loc ||
                                                  !seq_lens))) {
    pkv::set_last_error("bad batch or NULL host array");
    return PKV_ERR_INVALID_ARG;
  }
  const int C = attn_chunk_size;
  const int pages = C / block_size;
  int64_t v = 0;
  for (int b = 0; b < batch; ++b) {
    const int q = query_start_loc[b + 1] - query_start_loc[b];
    const int L = seq_lens[b];
    if (q <= 0 || L < q) {
      snprintf(msg, sizeof(msg),
               "request %d: need 0 < query_len (%d) <= seq_len (%d)", b, q,
               L);
      pkv::set_last_error(msg);
      return PKV_ERR_INVALID_ARG;
    }
    v += (L - 1) / C - (L - q) / C + 1;
  }
  *num_virtual = static_cast<int>(v);
  if (!seqlens_q_local && !cu_seqlens_q_local && !seqlens_k_local &&
      !block_table_local)
    return PKV_OK;                      // size query
  if (v > capacity || !seqlens_q_local || !cu_seqlens_q_local ||
      !seqlens_k_local || !block_table_local || !block_table ||
      max_blocks_per_seq <= 0 || block_table_stride < max_blocks_per_seq) {
    snprintf(msg, sizeof(msg),
             "need room for %lld virtual requests (capacity %d) and all "
             "output arrays",
             static_cast<long long>(v), capacity);
    pkv::set_last_error(msg);
    return PKV_ERR_INVALID_ARG;
  }
  int i = 0;
  cu_seqlens_q_local[0] = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seq_lens[b];
    const int first = L - (query_start_loc[b + 1] - query_start_loc[b]);
    for (int c = first / C; c <= (L - 1) / C; ++c, ++i) {
      const int lo = c * C, hi = lo + C;
      const int end = hi < L ? hi : L;
      seqlens_q_local[i] = end - (lo > first ? lo : first);
      seqlens_k_local[i] = end - lo;
      cu_seqlens_q_local[i + 1] = cu_seqlens_q_local[i] + seqlens_q_local[i];
      for (int pg = 0; pg < pages; ++pg) {
        int col = lo / block_size + pg;
        if (col > max_blocks_per_seq - 1) col = max_blocks_per_seq - 1;
        block_table_local[static_cast<int64_t>(i) * pages + pg] =
            block_table[static_cast<int64_t>(b) * block_table_stride + col];
      }
    }
  }
  return PKV_OK;
}

}  // extern "C"
