// Host policy: should a batch with a shared prefix use cascade attention?
//
// Source: "vllm/v1/attention/backends/flash_attn.py", use_cascade_attention.
// Cascade is off for a short prefix (< 256 tokens), fewer than 8 requests,
// ALiBi, sliding window, local attention or DCP.  It is on outright when the
// plain call would not use split-KV decoding (GQA ratio 1, a window or
// ALiBi, or any query longer than 1).  Otherwise a wave model with 128 x 128
// tiles compares the two:
//   cascade  = ceil(Hq * ceil(B / 128) / SMs) * ceil(P / 128)
//   split-KV = ceil(B * Hkv * ceil(G / 128) * ceil(P / 128) / SMs)
#include "pkv_common.cuh"

extern "C" {

int pkv_use_cascade_attention(int common_prefix_len,
                              const int32_t* query_lens, int num_reqs,
                              int num_heads, int num_kv_heads, int use_alibi,
                              int use_sliding_window, int use_local_attention,
                              int num_sms, int dcp_world_size) {
  auto cdiv = [](int64_t a, int64_t b) { return (a + b - 1) / b; };
  if (common_prefix_len < 256) return 0;
  if (use_alibi || use_sliding_window || use_local_attention) return 0;
  if (num_reqs < 8) return 0;
  if (dcp_world_size > 1) return 0;
  if (num_kv_heads <= 0 || num_sms <= 0 || !query_lens) return 0;
  const int group = num_heads / num_kv_heads;
  bool all_single = true;
  for (int i = 0; i < num_reqs; ++i) all_single &= query_lens[i] == 1;
  const bool flash_decoding = group > 1 && all_single;
  if (!flash_decoding) return 1;
  const int64_t tiles = cdiv(common_prefix_len, 128);
  const int64_t cascade_time =
      cdiv(static_cast<int64_t>(num_heads) * cdiv(num_reqs, 128), num_sms) *
      tiles;
  const int64_t fd_ctas = static_cast<int64_t>(num_reqs) * num_kv_heads *
                          cdiv(group, 128) * tiles;
  return cascade_time < cdiv(fd_ctas, num_sms) ? 1 : 0;
}

}  // extern "C"
