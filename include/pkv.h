/*
 * pkv.h -- C ABI of the paged KV-cache attention library (libpkv.so).
 *
 * Three operations, named and shaped after the calls that the vLLM and
 * Aphrodite attention backends make (sources cited per function, by page
 * title and section):
 *
 *   pkv_reshape_and_cache        -- "reshape_and_cache_flash"
 *   pkv_paged_attention_varlen   -- "flash_attn_varlen_func" with block_table
 *   pkv_merge_attn_states        -- "merge_attn_states"
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates no device memory and keeps no per-call state; scratch
 *     space is the caller's `workspace` buffer.
 *   - All work is enqueued on the caller's stream and is ordered on it.  No
 *     entry point synchronises the host, so calls can be issued inside CUDA
 *     graph capture (except pkv_check_device_errors, which synchronises).
 *   - Element strides are in ELEMENTS, not bytes.  The innermost (head_size)
 *     dimension is always contiguous.  16-byte alignment of every row start
 *     (pointer and strides a multiple of 8 elements for fp16/bf16) is required.
 *   - On failure an entry point returns a non-zero pkv_status, launches
 *     nothing, and leaves a message for pkv_last_error().  Nothing aborts the
 *     process or traps the GPU.
 *   - Thread safety: entry points may be called from several host threads;
 *     the error message is per thread.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

/* Same underlying type as cudaStream_t / CUstream (NULL = legacy stream). */
typedef struct CUstream_st* pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,          /* shape / pointer / value is wrong       */
  PKV_ERR_UNSUPPORTED = 2,          /* valid but not built (dtype, D, fp8 ...) */
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the needed size  */
  PKV_ERR_CUDA = 4,                 /* a CUDA runtime call failed              */
  PKV_ERR_BAD_INDEX = 5,            /* a kernel met an out-of-range block id or
                                       slot and skipped it (see
                                       pkv_check_device_errors)               */
  PKV_ERR_TIMEOUT = 6               /* a kernel's bounded wait for data ran
                                       out; its CTA drained its copies and
                                       stopped without writing (see
                                       pkv_check_device_errors)               */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_F32 = 2 } pkv_dtype;

/*
 * pkv_reshape_and_cache -- scatter new K/V rows into the paged cache.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
 * forward (the reshape_and_cache_flash call and its note that the op takes
 * the token count from slot_mapping, so key/value may carry padded rows);
 * "vllm.v1.attention.backends.flash_attn" (v0.9.0.1 docs),
 * FlashAttentionMetadataBuilder.build (unused slots are filled with -1).
 *
 * For t in [0, num_tokens) with s = slot_mapping[t] >= 0:
 *   key_cache[s / block_size, s % block_size, h, :]   = key[t, h, :]
 *   value_cache[s / block_size, s % block_size, h, :] = value[t, h, :]
 * for every KV head h.  Entries with s < 0 are skipped.  Rows are copied bit
 * for bit.  Slots >= num_blocks * block_size are skipped and flagged
 * (PKV_ERR_BAD_INDEX through pkv_check_device_errors).
 *
 * key, value      : [>= num_tokens, num_kv_heads, head_size] with element
 *                   strides (k_stride_tok, k_stride_head), (v_stride_tok,
 *                   v_stride_head).
 * key_cache,
 * value_cache     : 4-D views [num_blocks, block_size, num_kv_heads,
 *                   head_size] with element strides cache_strides[0..3]
 *                   (host array; cache_strides[3] must be 1).  The usual
 *                   NHD cache [2, NB, BS, Hkv, D] gives strides
 *                   (BS*Hkv*D, Hkv*D, D, 1); an HND cache [2, NB, Hkv, BS, D]
 *                   viewed as NHD gives (Hkv*BS*D, D, BS*D, 1).
 * slot_mapping    : int64 [num_tokens], device.
 * block_size      : multiple of 16 (else PKV_ERR_INVALID_ARG).
 * kv_cache_dtype  : "auto" (the cache has the dtype of key/value), or "fp8"
 *                   / "fp8_e4m3": the cache holds one-byte E4M3 ("fn")
 *                   codes, code = e4m3(x / scale) rounded to nearest (ties
 *                   to even) and saturated at +-448, with cache_strides in
 *                   bytes (key/value rows 16-byte aligned, cache rows 8-byte
 *                   aligned, else PKV_ERR_UNSUPPORTED).  Anything else
 *                   returns PKV_ERR_UNSUPPORTED.
 * k_scale, v_scale: device float scalars for an fp8 cache (required there);
 *                   ignored for "auto" and may be NULL.
 * num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_reshape_and_cache(
    const void* key, const void* value,
    int64_t k_stride_tok, int64_t k_stride_head,
    int64_t v_stride_tok, int64_t v_stride_head,
    void* key_cache, void* value_cache, const int64_t cache_strides[4],
    const int64_t* slot_mapping, int64_t num_tokens,
    int num_kv_heads, int head_size, int block_size, int64_t num_blocks,
    pkv_dtype dtype, const char* kv_cache_dtype,
    const float* k_scale, const float* v_scale,
    pkv_stream_t stream);

/*
 * pkv_paged_attention_varlen -- varlen attention over the paged cache.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py", FlashAttentionImpl.
 * forward (the flash_attn_varlen_func call: cu_seqlens_q, seqused_k,
 * block_table, window_size, softcap, alibi_slopes, num_splits, out) and
 * _forward_with_dcp (return_softmax_lse, LSE laid out [num_heads, tokens]);
 * FlashAttentionMetadata (seq_len = context_len + query_len, the queries are
 * the last query_len positions); FlashAttentionImpl.__init__ (window tuple,
 * soft-cap 0 = none, num_heads / num_kv_heads query heads per KV head).
 *
 * For request b with q_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries and
 * L_b = seqused_k[b] keys, query i (token t = cu_seqlens_q[b] + i) sits at
 * position p = L_b - q_b + i.  Query head h reads KV head h / (Hq / Hkv).
 * Key j (< L_b) lives at key_cache[block_table[b, j / BS], j % BS].
 *   s_j = softmax_scale * <q[t,h], k_j>
 *   if softcap > 0:   s_j = softcap * tanh(s_j / softcap)
 *   if alibi_slopes:  s_j -= alibi_slopes[h] * |p - j|
 *   admissible iff (!causal || j <= p) && (window_left < 0 || j >= p -
 *   window_left) && (window_right < 0 || j <= p + window_right)
 *   out[t,h]  = sum_adm softmax(s)_j * v_j      (rounded to dtype)
 *   lse[h, t] = ln sum_adm exp(s_j)             (float)
 * A row with no admissible key gets out = 0 and lse = -inf.
 *
 * q            : [T, Hq, D], strides (q_stride_tok, q_stride_head).
 * key_cache,
 * value_cache  : 4-D views as in pkv_reshape_and_cache.
 * out          : [T, Hq, D], strides (o_stride_tok, o_stride_head); only
 *                rows [0, T) are written, T = cu_seqlens_q[batch] (which must
 *                not exceed total_q).
 * cu_seqlens_q : int32 [batch+1] device; seqused_k: int32 [batch] device.
 * total_q      : rows of q/out/lse the caller allocated (>= T).
 * max_seqlen_q,
 * max_seqlen_k : host upper bounds of q_b and L_b (they size the grid).
 * block_table  : int32 [batch, >= ceil(L_b / BS)] device, row stride
 *                block_table_stride elements; entries must lie in
 *                [0, num_blocks) (out-of-range ids are not followed: the key
 *                is read as zero and the error is flagged).
 * num_splits   : 0 = choose; 1 = no split; N > 1 = split each request's keys
 *                into N chunks (split-KV), combined by LSE in a second launch.
 * softmax_lse  : float [num_heads, total_q] device, natural log, or NULL.
 * workspace    : device scratch of workspace_bytes >= the value
 *                pkv_paged_attention_workspace_size returns for the same
 *                arguments (may be NULL when that value is 0), 256-byte
 *                aligned.  For calls with prefill-class requests it ends
 *                with an optional tail: 256 bytes for the prefill kernel's
 *                work-item counter (the call zeroes it), then, when the
 *                call has fewer prefill work items than SMs, fp32 split-KV
 *                partials of the prefill kernel.  A workspace short of the
 *                tail (or NULL, when the rest needs none) is accepted: the
 *                items are then dealt in a fixed order, or not split.
 * dtype        : PKV_F16 or PKV_BF16 (q, cache and out share it).
 * head_size    : 64, 128 or 256 (others: PKV_ERR_UNSUPPORTED).
 * Hq % Hkv != 0, block_size % 16 != 0: PKV_ERR_INVALID_ARG.
 */
PKV_API pkv_status pkv_paged_attention_varlen(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4],
    void* out, int64_t o_stride_tok, int64_t o_stride_head,
    const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch,
    int total_q, int max_seqlen_q, int max_seqlen_k,
    const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq,
    int num_heads, int num_kv_heads, int head_size, int block_size,
    int64_t num_blocks,
    float softmax_scale, int causal, int window_left, int window_right,
    float softcap, const float* alibi_slopes,
    int num_splits, float* softmax_lse,
    void* workspace, size_t workspace_bytes,
    pkv_dtype dtype, pkv_stream_t stream);

/*
 * Optional features of the attention call; zero-initialise and set what is
 * used.  A NULL options pointer means all off.
 *
 * sinks: [num_heads] float32 device array of per-head attention-sink
 *   logits, or NULL.  Source: "vllm/v1/attention/backends/flash_attn.py",
 *   FlashAttentionImpl.__init__ (sinks, one per query head) and forward
 *   (s_aux=self.sinks); cascade_attention passes s_aux to the prefix call
 *   only ("incorporated into prefix_lse ... during the final attention
 *   merge").  The sink is one more logit of the row's softmax with no value:
 *   out = sum_j e^{s_j} v_j / (e^{sink_h} + sum_j e^{s_j}) and
 *   lse = ln(e^{sink_h} + sum_j e^{s_j}) (a row without keys gets out = 0,
 *   lse = sink_h).  The sink is neither scaled nor soft-capped.
 */
typedef struct {
  const float* sinks;
  /* kv_cache_fp8 != 0: key_cache/value_cache hold E4M3 ("fn") codes, one
   * byte per element (cache_strides in bytes), and a cached value reads back
   * as code * (*k_scale) or code * (*v_scale) (device float scalars, the
   * same ones given to pkv_reshape_and_cache).  Source: "vllm/v1/attention/
   * backends/flash_attn.py", FlashAttentionImpl.forward (kv_cache_dtype
   * "fp8", k_descale / v_descale = layer._k_scale / _v_scale); the FlashInfer
   * page's _trtllm_prefill_attn_kvfp8_dequant (value = fp8 * scale).
   * Decode-class requests read the fp8 pages directly; prefill-class
   * requests read them through a 16-bit copy in the workspace.  head_size
   * must be a multiple of 16 and cache rows 16-byte aligned. */
  int kv_cache_fp8;
  const float* k_scale;
  const float* v_scale;
  /* cu_seqlens_k != NULL selects non-paged (encoder) attention: the keys of
   * request b are rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of one K/V
   * tensor of total_k rows, passed as key_cache / value_cache.  Its layout
   * is [total_k, num_kv_heads, head_size] under cache_strides = {ignored,
   * row stride, head stride, 1} (elements; 16-byte multiples), so a
   * head-major [num_kv_heads, total_k, head_size] view works too.  The key
   * count of request b is cu_seqlens_k[b+1] - cu_seqlens_k[b]; seqused_k,
   * block_table, max_blocks_per_seq, block_size and num_blocks are ignored
   * (may be NULL / 0).  Causal alignment, windows, softcap, ALiBi and sinks
   * apply as in the paged call; an fp8 cache is rejected
   * (PKV_ERR_UNSUPPORTED).  Rows outside [0, total_k) are never read: a
   * request whose range leaves the tensor is clipped and the device error
   * word records PKV_ERR_BAD_INDEX.  Source: "vllm/v1/attention/backends/
   * flash_attn.py", FlashAttentionImpl._forward_encoder_attention (query,
   * key and value of shape [num_encoder_tokens, heads, head_size];
   * cu_seqlens_k = query_start_loc; bidirectional; no cache; fp8 rejected);
   * the aphrodite-engine flash_attn.py page, prefill without a cache
   * (cu_seqlens_k = seq_start_loc). */
  const int32_t* cu_seqlens_k;
  int total_k;
  /* fixed_split_size > 0: batch-invariant split-KV.  Every decode-class
   * request is cut into key ranges of fixed_split_size keys (rounded up to
   * a multiple of 64) counted from the start of its own key range, whatever
   * the rest of the batch is, and always goes through the split-combine
   * path, so a request's output bits do not depend on the batch it shares
   * a call with.  num_splits must then be 0.  Source: the FlashInfer
   * backend page, FlashInferMetadataBuilder (decode_fixed_split_size 2048
   * and prefill_fixed_split_size 4096 under batch invariance) and the
   * flash_attn.py page (num_splits = 1 under vllm_is_batch_invariant). */
  int fixed_split_size;
  /* q_fp8 != 0: q holds E4M3 codes, one byte per element (q strides in
   * bytes, rows 16-byte aligned), and a query value reads back as
   * code * (*q_scale) (a device float scalar, the scale given to
   * pkv_scaled_fp8_quant).  Needs kv_cache_fp8 (PKV_ERR_UNSUPPORTED
   * otherwise); `dtype` then names the output's type.  The logits are
   * softmax_scale * q_scale * k_scale * sum_d code_q * code_k.  The
   * persistent decode kernel widens the query codes to f16 in registers (as
   * it does the key codes: exact); the other kernels read an exact 16-bit
   * copy of the query codes that the call writes to its workspace.  Source:
   * "vllm/v1/attention/backends/flash_attn.py" (git view and v0.9.0.1 docs),
   * FlashAttentionImpl.forward (with an fp8 cache the query goes through
   * scaled_fp8_quant(query, layer._q_scale) and the call gets
   * q_descale = layer._q_scale); the FlashInfer backend page,
   * get_xqa_bmm1_scale (bmm1 scale = scale * q_scale * k_scale). */
  int q_fp8;
  const float* q_scale;
  /* no_pdl != 0: launch every kernel of the call in plain stream order.
   * By default some launches are programmatic dependent launches: the
   * persistent decode kernel (pkv_set_decode_kernel) depends on the kernel
   * queued before the call and waits for it (griddepcontrol.wait) before
   * it reads or writes anything; in a call with both decode-class and
   * prefill-class requests, the second of the two attention kernels (and
   * the split combine after it) may start while the first still runs, and
   * its grid ends only after the first one's.  The first form is correct
   * when the kernel queued before the call completes only after the work
   * queued before it, which holds for every kernel of this library and for
   * any kernel that is not itself a programmatic dependent launch.
   * (Library plumbing with no counterpart on the pages; the cascade entry
   * point has its own `overlap` switch.) */
  int no_pdl;
} pkv_attention_options;

/* Workspace bytes for pkv_paged_attention_varlen_opts with these options
 * (an fp8 cache with prefill-class requests needs room for 16-bit copies of
 * up to batch * max_blocks_per_seq pages; an fp8 query, for a 16-bit copy
 * of the query codes: total_q * num_heads * head_size * 2 bytes and one
 * scalar).  (size_t)-1 on bad arguments. */
PKV_API size_t pkv_paged_attention_workspace_size_opts(
    int batch, int total_q, int max_seqlen_q, int max_seqlen_k,
    int num_heads, int num_kv_heads, int head_size, int block_size,
    int causal, int window_left, int window_right, int num_splits,
    int max_blocks_per_seq, const pkv_attention_options* opts);

/* pkv_paged_attention_varlen with options (see pkv_attention_options). */
PKV_API pkv_status pkv_paged_attention_varlen_opts(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4],
    void* out, int64_t o_stride_tok, int64_t o_stride_head,
    const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch,
    int total_q, int max_seqlen_q, int max_seqlen_k,
    const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq,
    int num_heads, int num_kv_heads, int head_size, int block_size,
    int64_t num_blocks,
    float softmax_scale, int causal, int window_left, int window_right,
    float softcap, const float* alibi_slopes,
    int num_splits, float* softmax_lse,
    void* workspace, size_t workspace_bytes,
    pkv_dtype dtype, pkv_stream_t stream,
    const pkv_attention_options* opts);

/*
 * pkv_cascade_attention -- shared-prefix ("cascade") attention in one call.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py", cascade_attention:
 * the prefix call (every query over the common_prefix_len keys of the
 * shared blocks, block_table[:1], non-causal, cu_prefix_query_lens =
 * [0, num_tokens], prefix_kv_lens = [common_prefix_len], with s_aux), the
 * suffix call (block_table[:, common_prefix_len // block_size:],
 * suffix_kv_lens, causal) and merge_attn_states(output, prefix_output,
 * prefix_lse, suffix_output, suffix_lse).  Those three steps, with the same
 * meaning for every argument; window and ALiBi are not taken (the page
 * rejects both).  The prefix runs unsplit.  With `overlap` the suffix's
 * decode kernel (16-bit caches) is launched as a programmatic dependent of
 * the prefix kernel: it starts once the prefix's CTAs are resident and
 * takes the SMs they leave free, and its last CTA waits for the prefix grid
 * to end before the merge.  With overlap = 0 the steps run one after the
 * other; both give the same bits.
 *
 * output : [num_tokens, num_heads, head_size] contiguous, `dtype`.
 * query  : as in pkv_paged_attention_varlen (element strides).
 * cu_query_lens [batch+1], suffix_kv_lens [batch], cu_prefix_query_lens
 *          [2], prefix_kv_lens [1]: device int32.  max_kv_len bounds
 *          common_prefix_len + suffix_kv_lens[b].
 * block_table : [batch, >= max_blocks_per_seq] int32; the first
 *          common_prefix_len / block_size entries of row 0 are the shared
 *          blocks (every row holds them first).
 * num_splits : split-KV of the suffix call (0 = the library's plan).
 * opts   : sinks (prefix only), fp8 cache and query; NULL = none.  No
 *          cu_seqlens_k or fixed split (PKV_ERR_INVALID_ARG).
 * workspace : pkv_cascade_attention_workspace_size bytes, 256-byte aligned.
 */
PKV_API size_t pkv_cascade_attention_workspace_size(
    int batch, int num_tokens, int max_query_len, int max_kv_len,
    int common_prefix_len, int num_heads, int num_kv_heads, int head_size,
    int block_size, int max_blocks_per_seq, int num_splits,
    const pkv_attention_options* opts);

PKV_API pkv_status pkv_cascade_attention(
    void* output, const void* query, int64_t q_stride_tok,
    int64_t q_stride_head, const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4], const int32_t* cu_query_lens,
    int max_query_len, const int32_t* cu_prefix_query_lens,
    const int32_t* prefix_kv_lens, const int32_t* suffix_kv_lens,
    int max_kv_len, int batch, int num_tokens, float softmax_scale,
    float logits_soft_cap, const int32_t* block_table,
    int64_t block_table_stride, int max_blocks_per_seq,
    int common_prefix_len, int num_heads, int num_kv_heads, int head_size,
    int block_size, int64_t num_blocks, int num_splits, int overlap,
    void* workspace, size_t workspace_bytes, pkv_dtype dtype,
    pkv_stream_t stream, const pkv_attention_options* opts);

/*
 * pkv_scaled_fp8_quant -- per-tensor E4M3 quantization of a query matrix.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py" (git view and the
 * v0.9.0.1 docs page), FlashAttentionImpl.forward: with an fp8 KV cache the
 * query, viewed as [num_tokens, num_heads * head_size], goes through
 * ops.scaled_fp8_quant(query, layer._q_scale) before the attention call;
 * the FlashInfer backend page, maybe_quant_query (the same call).  The
 * scale is static (given); the pages never call the dynamic form.
 *
 * out[r, c] = RN_satfinite_e4m3(in[r, c] / *scale) for r < rows, c < cols:
 * the quotient in IEEE float32, rounded to the nearest E4M3 value (ties to
 * the even code), saturating at +-448; NaN gives the code 0x7F.
 *
 * in     : [rows, cols] fp16/bf16 (`dtype`), row stride in_row_stride
 *          elements; out: [rows, cols] uint8 codes, row stride
 *          out_row_stride bytes.  cols % 16 == 0; both base pointers and
 *          row strides 16-byte aligned (PKV_ERR_UNSUPPORTED otherwise).
 * scale  : device float32 scalar, > 0.
 * Enqueued on `stream`; no host synchronisation.
 */
PKV_API pkv_status pkv_scaled_fp8_quant(const void* in, int64_t in_row_stride,
                                        void* out, int64_t out_row_stride,
                                        int64_t rows, int cols,
                                        const float* scale, pkv_dtype dtype,
                                        pkv_stream_t stream);

/*
 * Bytes of workspace pkv_paged_attention_varlen needs for these arguments
 * (on the current device: the split plans and the persistent decode grid
 * depend on its SM count), counting the optional tail: the persistent
 * decode kernel's scratch (num_splits = 0), and for calls with
 * prefill-class requests (max_seqlen_q * num_heads / num_kv_heads > 16)
 * the 256-byte item counter and the prefill split-KV partials.  Returns 0
 * when no scratch is needed, and (size_t)-1 for invalid arguments.
 */
PKV_API size_t pkv_paged_attention_workspace_size(
    int batch, int total_q, int max_seqlen_q, int max_seqlen_k,
    int num_heads, int num_kv_heads, int head_size, int block_size,
    int causal, int window_left, int window_right, int num_splits);

/*
 * pkv_paged_attention_varlen_static_scratch -- pkv_paged_attention_varlen
 * for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart of this entry point.
 *
 * Some callers cannot provide the `workspace` the split-KV path needs:
 * plugin hosts and serving runtimes that plan all device memory up front and
 * give an individual call no scratch, and latency-critical loops that must
 * not call cudaMalloc/cudaFree (they can block the host and synchronise the
 * whole device).  This variant takes the same arguments minus
 * workspace/workspace_bytes and computes the same result.  Its scratch is a
 * fixed array of PKV_STATIC_SCRATCH_BYTES inside the library's own device
 * memory, which every GPU that loads the library holds until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - Set-up: every call looks up the array's device address on the current
 *   device (cudaGetSymbolAddress: a host-side lookup once the module is
 *   loaded, so a device reset cannot leave a stale address).  The first
 *   call on a device also raises the kernels' shared-memory limits; make it
 *   before any stream capture.  Later calls can be captured into a CUDA
 *   graph.
 * - Inputs: the same as pkv_paged_attention_varlen, which has no options,
 *   so the cache holds fp16/bf16 values (no fp8 cache, sinks or non-paged
 *   keys through this entry point).
 * - Limit: a call whose decode split plan needs more than
 *   PKV_STATIC_SCRATCH_BYTES is rejected with PKV_ERR_WORKSPACE_TOO_SMALL
 *   and a message; nothing is launched.  The optional tail (see
 *   pkv_paged_attention_workspace_size) is used when it fits in the rest of
 *   the array.
 * - Sharing: all calls on a device share the one array and it keeps the
 *   last call's contents.  Nothing in it needs clearing: every scratch value
 *   a call reads was written earlier in the same call (the prefill item
 *   counter is zeroed by the call).  Calls that overlap on the GPU
 *   (different streams, or several host threads) race on the array and
 *   corrupt each other's results; order them on one stream.
 */
#define PKV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

PKV_API pkv_status pkv_paged_attention_varlen_static_scratch(
    const void* q, int64_t q_stride_tok, int64_t q_stride_head,
    const void* key_cache, const void* value_cache,
    const int64_t cache_strides[4],
    void* out, int64_t o_stride_tok, int64_t o_stride_head,
    const int32_t* cu_seqlens_q, const int32_t* seqused_k, int batch,
    int total_q, int max_seqlen_q, int max_seqlen_k,
    const int32_t* block_table, int64_t block_table_stride,
    int max_blocks_per_seq,
    int num_heads, int num_kv_heads, int head_size, int block_size,
    int64_t num_blocks,
    float softmax_scale, int causal, int window_left, int window_right,
    float softcap, const float* alibi_slopes,
    int num_splits, float* softmax_lse,
    pkv_dtype dtype, pkv_stream_t stream);

/*
 * pkv_merge_attn_states -- combine two partial attentions by their LSEs.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py", cascade_attention (the
 * merge of the shared-prefix and suffix results) and _forward_with_dcp (the
 * merge of context and new-token results); the FlashInfer backend page
 * converts base-2 LSEs to natural log before the same merge, so LSEs here
 * are natural-log.
 *
 * With M = max(l1, l2), w_i = exp(l_i - M):
 *   output = (w1 * prefix_output + w2 * suffix_output) / (w1 + w2)
 *   output_lse = M + ln(w1 + w2)
 * A side with lse = -inf holds no keys and is ignored; if both are -inf the
 * row is 0 with lse -inf.
 *
 * output, prefix_output, suffix_output: contiguous [num_tokens, num_heads,
 *   head_size]; output has out_dtype (PKV_F16/PKV_BF16/PKV_F32), the two
 *   inputs have in_dtype.
 * prefix_lse, suffix_lse: contiguous float [num_heads, num_tokens].
 * output_lse: float [num_heads, num_tokens] or NULL.
 * head_size: multiple of 8, at most 512.
 */
PKV_API pkv_status pkv_merge_attn_states(
    void* output, const void* prefix_output, const float* prefix_lse,
    const void* suffix_output, const float* suffix_lse, float* output_lse,
    int num_tokens, int num_heads, int head_size,
    pkv_dtype out_dtype, pkv_dtype in_dtype, pkv_stream_t stream);

/*
 * pkv_make_local_attention_virtual_batches -- chunked local attention as
 * virtual requests (HOST arrays in and out; no GPU work).
 *
 * Source: "vllm.v1.attention.backends.flash_attn" (vLLM v0.9.0.1 docs),
 * make_local_attention_virtual_batches and FlashAttentionMetadataBuilder.
 * build.  With chunk size C (a multiple of block_size), request b with
 * q_b = query_start_loc[b+1] - query_start_loc[b] > 0 queries and
 * L_b = seq_lens[b] >= q_b keys is split into one virtual request per C-wide
 * key chunk c that holds one of its queries: seqlens_q_local = the queries in
 * chunk c, seqlens_k_local = min(L_b, (c+1)C) - cC, block_table_local row =
 * columns cC/BS .. cC/BS + C/BS - 1 of block-table row b (clipped to the last
 * column).  Running pkv_paged_attention_varlen (causal) on the virtual
 * requests gives chunked local attention: the query at position p sees keys
 * j <= p with j / C == p / C.
 *
 * Pass all four output pointers NULL to get only *num_virtual.  Otherwise
 * capacity must be >= *num_virtual; cu_seqlens_q_local has capacity + 1
 * entries and block_table_local is [capacity, C / block_size].
 * Errors: C not a positive multiple of block_size, q_b <= 0, L_b < q_b, NULL
 * arrays, too little capacity -> PKV_ERR_INVALID_ARG.
 */
PKV_API pkv_status pkv_make_local_attention_virtual_batches(
    int attn_chunk_size, const int32_t* query_start_loc,
    const int32_t* seq_lens, int batch, const int32_t* block_table,
    int64_t block_table_stride, int max_blocks_per_seq, int block_size,
    int* num_virtual, int32_t* seqlens_q_local, int32_t* cu_seqlens_q_local,
    int32_t* seqlens_k_local, int32_t* block_table_local, int capacity);

/*
 * pkv_use_cascade_attention -- host policy: 1 if a batch whose requests share
 * a common_prefix_len-token prefix should run cascade attention, else 0.
 *
 * Source: "vllm/v1/attention/backends/flash_attn.py", use_cascade_attention:
 * off for a prefix < 256 tokens, < 8 requests, ALiBi, sliding window, local
 * attention or DCP (dcp_world_size > 1); on when the plain call would not
 * use split-KV decoding (GQA ratio 1 or any query_lens[i] != 1); otherwise
 * on iff ceil(Hq * ceil(B/128) / SMs) * ceil(P/128) <
 * ceil(B * Hkv * ceil(G/128) * ceil(P/128) / SMs).  query_lens: host int32
 * [num_reqs].  Pure host arithmetic; no GPU work.
 */
PKV_API int pkv_use_cascade_attention(
    int common_prefix_len, const int32_t* query_lens, int num_reqs,
    int num_heads, int num_kv_heads, int use_alibi, int use_sliding_window,
    int use_local_attention, int num_sms, int dcp_world_size);

/*
 * pkv_check_device_errors -- synchronise `stream`, then read and clear the
 * library's device error word (one per device; kernels OR bits into it and
 * never trap).  Returns, by priority:
 *   PKV_ERR_TIMEOUT    a kernel's bounded wait for its data ran out (about
 *                      2 s; the CTA drained its copies, freed what it held
 *                      and returned without writing its outputs);
 *   PKV_ERR_BAD_INDEX  a kernel met an out-of-range block id or slot (the
 *                      access was skipped, never performed), a key range
 *                      past the table row, or a request with more queries
 *                      than the call's max_seqlen_q (not computed);
 *   PKV_ERR_CUDA       an internal launch fault was caught (misaligned
 *                      shared memory);
 *   PKV_OK             nothing since the last check.
 * The message (pkv_last_error) lists every cause seen.  Not for use inside
 * graph capture.
 */
PKV_API pkv_status pkv_check_device_errors(pkv_stream_t stream);

/*
 * Which kernel serves prefill-class requests (more than 16 packed query rows
 * per KV head): the tcgen05/TMEM kernel (for head sizes up to 128 it keeps
 * the softmax output P in tensor memory), the tcgen05 kernel that stages P
 * through shared memory, or the warp-level mma.sync kernel.  A process-wide
 * diagnostic switch for A/B comparison; all give the same result within
 * rounding.  Returns PKV_ERR_INVALID_ARG for other values.
 */
#define PKV_PREFILL_TCGEN05 0
#define PKV_PREFILL_MMA_SYNC 1
#define PKV_PREFILL_TCGEN05_SMEM_P 2
PKV_API pkv_status pkv_set_prefill_kernel(int which);

/*
 * Which kernel serves decode-class requests (at most 16 packed query rows
 * per KV head):
 *   PKV_DECODE_PERSISTENT  one wave of CTAs, each streaming an equal share
 *       of the batch's key tiles (a request's keys may be cut between CTAs;
 *       the pieces are merged by LSE).  Taken by calls that leave the split
 *       to the library (num_splits = 0, no fixed split size) when the
 *       workspace holds its scratch (see pkv_paged_attention_workspace_size);
 *       16-bit caches with head_size 64/128/256 and fp8 caches with
 *       head_size 128/256.  Other calls fall back to the kernels below.
 *   PKV_DECODE_TMA  one CTA per (request, KV head, split), K/V pages moved
 *       by a TMA producer warp (16-bit caches).
 *   PKV_DECODE_CP_ASYNC  one CTA per (request, KV head, split), pages
 *       gathered with 16-byte cp.async (fp8 caches the persistent kernel
 *       does not take use it always).
 *   PKV_DECODE_AUTO (default)  the persistent kernel for fp8 caches and
 *       for calls with at least two waves of long (request, KV head) units
 *       (batch * num_kv_heads >= 2 * 3 * SMs, and a key range of at least
 *       2048 by max_seqlen_k and the window), else PKV_DECODE_TMA.
 * A process-wide switch for A/B comparison; all give the same result
 * within rounding.  Returns PKV_ERR_INVALID_ARG for other values.
 */
#define PKV_DECODE_TMA 0
#define PKV_DECODE_CP_ASYNC 1
#define PKV_DECODE_PERSISTENT 2
#define PKV_DECODE_AUTO 3
PKV_API pkv_status pkv_set_decode_kernel(int which);

/*
 * Limit of the bounded waits of the decode kernels (a consumer waiting for
 * its K/V pages, the producer waiting for a free ring stage), in
 * nanoseconds; the default is PKV_WAIT_LIMIT_DEFAULT_NS (2 s).  A wait that
 * runs out records a timeout in the device error word, the CTA drains the
 * copies it issued (those drains always keep the 2 s limit), frees what it
 * holds and returns without writing its outputs; pkv_check_device_errors
 * then reports PKV_ERR_TIMEOUT and the next call runs normally.  A
 * process-wide diagnostic for testing that path: a small limit makes calls
 * fail.  No counterpart on the source pages.
 */
#define PKV_WAIT_LIMIT_DEFAULT_NS 2000000000ull
PKV_API pkv_status pkv_set_wait_limit_ns(uint64_t ns);

/*
 * Number of kernels this library has launched in this process (all devices,
 * all threads), for accounting of launches per step.
 */
PKV_API uint64_t pkv_launch_count(void);

/* Message for the last non-OK status returned on this host thread. */
PKV_API const char* pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
