"""Float64 CPU oracle for paged attention over a block-table KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA path: it imports numpy and nothing else.

Every function is the plain definition of what the attention backends on the
source pages compute, written out with numpy in float64 (element copies for the
cache scatter).  Sources, cited by page title and section:

* "vllm/v1/attention/backends/flash_attn.py" (vLLM v1 FlashAttention backend):
  ``FlashAttentionMetadata`` (context/query/seq length note),
  ``FlashAttentionImpl.__init__`` (window tuple, soft-cap 0 = none, GQA ratio),
  ``FlashAttentionImpl.forward`` (cache write, varlen call, LSE return),
  ``FlashAttentionImpl._forward_encoder_attention`` (attention without a
  cache), ``cascade_attention``, ``use_cascade_attention``.
* "vllm.v1.attention.backends.flash_attn" (vLLM v0.9.0.1 API docs):
  ``FlashAttentionMetadataBuilder.build`` (slot_mapping tail filled with -1),
  ``make_local_attention_virtual_batches`` (worked example).
* "flashinfer.py . tduncan/Nvidia-Optimization-Stack-VLLM": end-aligned causal
  mask note, base-2 LSE converted to natural log before merging.
* "aphrodite-engine/aphrodite/attention/backends/flash_attn.py":
  ``FlashAttentionMetadata`` block-table and seq_start_loc examples; the
  cache-free prefill call (``cu_seqlens_k = seq_start_loc``).

Readings taken where the pages are silent:

* slot s addresses block ``s // block_size``, row ``s % block_size``; s < 0 is
  a padding slot and is skipped;
* query i of a request with L keys and q queries sits at position
  ``p = L - q + i`` (bottom-right / end-aligned causal alignment);
* window (left, right) admits keys j with ``p - left <= j <= p + right``, a
  negative side meaning unbounded;
* soft-cap: ``cap * tanh(scale * q.k / cap)``, then the ALiBi bias
  ``-slope_h * |p - j|`` is added, then the mask;
* query head h reads KV head ``h // (Hq // Hkv)``;
* LSE is natural-log, float, laid out ``[Hq, T]``;
* an attention sink (``s_aux``) is one more logit per head in the softmax
  denominator, with no value; the LSE includes it;
* a row with no admissible key gives out = 0 and lse = -inf.

Parity status: every function is pinned by ``tests/test_oracle_*.py`` against
brute-force dense attention (torch's CPU ``scaled_dot_product_attention`` in
float64), closed forms and invariants.  The soft-cap and ALiBi formulas are
pinned by limits and saturation / geometric-series closed forms of the
readings above; the pages print neither formula.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# a2: cache write ("reshape_and_cache_flash")
# ---------------------------------------------------------------------------

def reshape_and_cache_ref(key, value, key_cache, value_cache, slot_mapping):
    """Scatter new K/V rows into the paged cache, in place.

    vLLM v1 ``FlashAttentionImpl.forward``: the op reads ``len(slot_mapping)``
    rows of ``key``/``value`` (extra padded rows are ignored), and the v0.9.0.1
    metadata builder fills unused slots with -1.

    key, value:          [>= T, Hkv, D] arrays (any dtype; copied element-wise,
                         so bf16 bit patterns stored as uint16 stay bit-exact)
    key_cache, value_cache: [NB, BS, Hkv, D] arrays, modified in place
    slot_mapping:        [T] integers
    """
    block_size = key_cache.shape[1]
    for t in range(len(slot_mapping)):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        blk, off = divmod(s, block_size)
        key_cache[blk, off] = key[t]
        value_cache[blk, off] = value[t]


def gather_ref(cache, block_table_row, seq_len):
    """Logical rows 0..seq_len-1 of one request, read through its block table.

    Aphrodite ``FlashAttentionMetadata``: block table entry [b, j] is the
    physical block that holds logical block j of request b.
    Returns [seq_len, Hkv, D].
    """
    block_size = cache.shape[1]
    rows = [cache[int(block_table_row[j // block_size]), j % block_size]
            for j in range(seq_len)]
    if not rows:
        return np.zeros((0,) + cache.shape[2:], dtype=cache.dtype)
    return np.stack(rows)


# ---------------------------------------------------------------------------
# a3-a6: varlen paged attention ("flash_attn_varlen_func" with block_table)
# ---------------------------------------------------------------------------

def admissible_mask(q_len, k_len, causal, window_size):
    """Boolean [q_len, k_len]: which keys each query of one request may see.

    Query i sits at position p = k_len - q_len + i (vLLM v1
    ``FlashAttentionMetadata`` note: seq_len = context_len + query_len, the
    queries are the last query_len tokens; FlashInfer page: end-aligned causal
    mask).  window_size = (left, right), -1 = unbounded (vLLM v1
    ``FlashAttentionImpl.__init__``).
    """
    left, right = window_size
    p = (k_len - q_len + np.arange(q_len))[:, None]
    j = np.arange(k_len)[None, :]
    ok = np.ones((q_len, k_len), dtype=bool)
    if causal:
        ok &= j <= p
    if left >= 0:
        ok &= j >= p - left
    if right >= 0:
        ok &= j <= p + right
    return ok


def attention_logits(q_rows, k_rows, q_len, k_len, softmax_scale, softcap,
                     alibi_slope):
    """Final logits [q_len, k_len] for one (request, query head).

    Scale first, then the soft-cap (0 = none, vLLM v1
    ``FlashAttentionImpl.__init__``), then the ALiBi bias -slope*|p - j|.
    """
    s = softmax_scale * (q_rows @ k_rows.T)
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    if alibi_slope is not None:
        p = (k_len - q_len + np.arange(q_len))[:, None]
        j = np.arange(k_len)[None, :]
        s = s - alibi_slope * np.abs(p - j)
    return s


def add_sink_ref(out, lse, sinks):
    """Fold per-head sink logits into finished attention results.

    vLLM v1 ``FlashAttentionImpl`` passes ``sinks`` [num_heads] float32 as
    ``s_aux``; ``cascade_attention`` notes that the kernel incorporates it
    into the prefix LSE so that it takes effect in the merge.  Reading: the
    sink is one more logit in each row's softmax denominator with no value,
    so lse' = ln(e^lse + e^sink) and out' = out * e^(lse - lse').
    out [T, H, D], lse [H, T], sinks [H].
    """
    sinks = np.asarray(sinks, dtype=np.float64)[:, None]        # [H, 1]
    new_lse = np.logaddexp(lse, sinks)
    w = np.where(np.isfinite(lse), np.exp(lse - new_lse), 0.0)  # [H, T]
    return out * w.T[..., None], new_lse


def paged_attention_ref(q, key_cache, value_cache, cu_seqlens_q, seqused_k,
                        block_table, softmax_scale, causal=True,
                        window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                        sinks=None):
    """Varlen attention of q over the paged cache; returns (out, lse).

    vLLM v1 ``FlashAttentionImpl.forward`` call to ``flash_attn_varlen_func``
    with ``cu_seqlens_q``, ``seqused_k``, ``block_table``, ``window_size``,
    ``softcap``, ``alibi_slopes`` and ``return_softmax_lse`` (LSE in [H, T],
    per ``_forward_with_dcp``'s note).

    q:            [T, Hq, D] float64
    key_cache,
    value_cache:  [NB, BS, Hkv, D] float64
    cu_seqlens_q: [B+1]; seqused_k: [B]; block_table: [B, max_blocks]
    returns out [T, Hq, D] float64, lse [Hq, T] float64 (natural log)
    """
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = key_cache.shape[2]
    assert Hq % Hkv == 0
    group = Hq // Hkv
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.full((Hq, T), -np.inf, dtype=np.float64)
    for b in range(len(seqused_k)):
        t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        q_len, k_len = t1 - t0, int(seqused_k[b])
        if q_len == 0:
            continue
        k_b = gather_ref(key_cache, block_table[b], k_len).astype(np.float64)
        v_b = gather_ref(value_cache, block_table[b], k_len).astype(np.float64)
        _attend_request(q, t0, t1, k_b, v_b, group, softmax_scale, causal,
                        window_size, softcap, alibi_slopes, out, lse)
    if sinks is not None:
        out, lse = add_sink_ref(out, lse, sinks)
    return out, lse


def _attend_request(q, t0, t1, k_b, v_b, group, softmax_scale, causal,
                    window_size, softcap, alibi_slopes, out, lse):
    """Softmax attention of queries t0..t1-1 over one request's key rows
    k_b, v_b [k_len, Hkv, D]; writes out[t0:t1] and lse[:, t0:t1]."""
    q_len, k_len = t1 - t0, k_b.shape[0]
    ok = admissible_mask(q_len, k_len, causal, window_size)
    for h in range(q.shape[1]):
        g = h // group
        slope = None if alibi_slopes is None else float(alibi_slopes[h])
        s = attention_logits(q[t0:t1, h, :], k_b[:, g, :], q_len, k_len,
                             softmax_scale, softcap, slope)
        s = np.where(ok, s, -np.inf)
        m = s.max(axis=1, initial=-np.inf)
        has = np.isfinite(m)
        m_safe = np.where(has, m, 0.0)
        w = np.exp(s - m_safe[:, None])          # masked entries -> 0
        l = w.sum(axis=1)
        row_lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)),
                           -np.inf)
        o = (w @ v_b[:, g, :]) / np.where(has, l, 1.0)[:, None]
        out[t0:t1, h, :] = np.where(has[:, None], o, 0.0)
        lse[h, t0:t1] = row_lse


def varlen_attention_ref(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale,
                         causal=False, window_size=(-1, -1), softcap=0.0,
                         alibi_slopes=None, sinks=None):
    """Varlen attention over plain (non-paged) K/V rows; returns (out, lse).

    vLLM v1 ``FlashAttentionImpl._forward_encoder_attention``: query, key and
    value are [num_tokens, heads, head_size] with no cache, request b's keys
    are rows ``cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1`` (the encoder passes
    ``cu_seqlens_k = query_start_loc`` and ``causal=False``); the aphrodite
    page's cache-free prefill passes ``cu_seqlens_k = seq_start_loc`` with
    ``causal=True``.  Every other rule is that of ``paged_attention_ref``.

    q [T, Hq, D]; k, v [Tk, Hkv, D]; cu_seqlens_q, cu_seqlens_k [B+1].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0
    out = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.full((Hq, T), -np.inf, dtype=np.float64)
    for b in range(len(cu_seqlens_q) - 1):
        t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        k0, k1 = int(cu_seqlens_k[b]), int(cu_seqlens_k[b + 1])
        if t1 == t0:
            continue
        _attend_request(q, t0, t1, k[k0:k1], v[k0:k1], Hq // Hkv,
                        softmax_scale, causal, window_size, softcap,
                        alibi_slopes, out, lse)
    if sinks is not None:
        out, lse = add_sink_ref(out, lse, sinks)
    return out, lse


# ---------------------------------------------------------------------------
# a8: LSE merge ("merge_attn_states") and the N-way split combine
# ---------------------------------------------------------------------------

def merge_attn_states_ref(prefix_output, prefix_lse, suffix_output,
                          suffix_lse):
    """Combine two partial attentions over disjoint key sets by their LSEs.

    Call sites: vLLM v1 ``cascade_attention`` (prefix + suffix) and
    ``_forward_with_dcp`` (context + new tokens).  With M = max(l1, l2),
    w_i = exp(l_i - M): out = (w1 o1 + w2 o2) / (w1 + w2),
    lse = M + ln(w1 + w2).  A side with lse = -inf holds no keys and drops
    out (its output is not read); if both are -inf the row is out = 0,
    lse = -inf.  Non-finite LSEs the pages do not define take the limit of
    the formula: a side with lse = +inf takes all the weight (two such sides
    weigh the same) and the merged lse is +inf; a NaN lse gives a NaN row.

    outputs [T, H, D]; lse [H, T].  Returns (out float64, lse float64).
    """
    o1 = np.asarray(prefix_output, dtype=np.float64)
    o2 = np.asarray(suffix_output, dtype=np.float64)
    l1 = np.asarray(prefix_lse, dtype=np.float64).T      # [T, H]
    l2 = np.asarray(suffix_lse, dtype=np.float64).T
    nan = np.isnan(l1) | np.isnan(l2)
    inf1, inf2 = l1 == np.inf, l2 == np.inf
    pinf = inf1 | inf2
    with np.errstate(invalid="ignore"):
        m = np.maximum(l1, l2)
    finite_m = np.isfinite(m)
    m_safe = np.where(finite_m, m, 0.0)
    with np.errstate(invalid="ignore", over="ignore"):
        w1 = np.where(np.isfinite(l1), np.exp(l1 - m_safe), 0.0)
        w2 = np.where(np.isfinite(l2), np.exp(l2 - m_safe), 0.0)
    w1 = np.where(pinf, inf1.astype(np.float64), w1)
    w2 = np.where(pinf, inf2.astype(np.float64), w2)
    any_keys = finite_m | pinf
    tot = w1 + w2
    tot_safe = np.where(any_keys & (tot > 0), tot, 1.0)
    # a side without weight is not read (its rows may hold anything)
    with np.errstate(invalid="ignore"):
        num = np.where((w1 > 0)[..., None], w1[..., None] * o1, 0.0) + \
            np.where((w2 > 0)[..., None], w2[..., None] * o2, 0.0)
    out = num / tot_safe[..., None]
    out = np.where(any_keys[..., None], out, 0.0)
    lse = np.where(finite_m, m_safe + np.log(tot_safe), -np.inf)
    lse = np.where(pinf, np.inf, lse)
    out = np.where(nan[..., None], np.nan, out)
    lse = np.where(nan, np.nan, lse)
    return out, lse.T.copy()


def merge_many_ref(outputs, lses):
    """N-way LSE combine of split-KV partials: a left fold of the 2-way merge.

    vLLM v1 ``FlashAttentionMetadataBuilder``: num_splits > 1 produces
    [num_splits, ...] intermediates that the kernel combines; the combine is
    the associative fold of ``merge_attn_states_ref``.
    """
    out, lse = outputs[0], lses[0]
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    for o, l in zip(outputs[1:], lses[1:]):
        out, lse = merge_attn_states_ref(out, lse, o, l)
    return out, lse


# ---------------------------------------------------------------------------
# a10: cascade (shared-prefix) attention
# ---------------------------------------------------------------------------

def cascade_ref(q, key_cache, value_cache, cu_seqlens_q, seqused_k,
                block_table, common_prefix_len, softmax_scale, softcap=0.0,
                sinks=None):
    """Shared-prefix attention as vLLM v1 ``cascade_attention`` defines it.

    Prefix: all T queries as one non-causal "sequence" over
    ``block_table[:1]`` with ``common_prefix_len`` keys.  Suffix: causal over
    ``block_table[:, P/BS:]`` with ``seqused_k - P`` keys.  Then merge.  No
    ALiBi and no window (the page asserts both).
    """
    T = q.shape[0]
    block_size = key_cache.shape[1]
    assert common_prefix_len % block_size == 0 and common_prefix_len > 0
    n_common = common_prefix_len // block_size
    cu_prefix = np.array([0, T])
    prefix_lens = np.array([common_prefix_len])
    o_p, l_p = paged_attention_ref(q, key_cache, value_cache, cu_prefix,
                                   prefix_lens, block_table[:1],
                                   softmax_scale, causal=False,
                                   softcap=softcap, sinks=sinks)
    suffix_lens = np.asarray(seqused_k) - common_prefix_len
    o_s, l_s = paged_attention_ref(q, key_cache, value_cache, cu_seqlens_q,
                                   suffix_lens, block_table[:, n_common:],
                                   softmax_scale, causal=True,
                                   softcap=softcap)
    return merge_attn_states_ref(o_p, l_p, o_s, l_s)


# ---------------------------------------------------------------------------
# Host policy: use_cascade_attention (wave model)
# ---------------------------------------------------------------------------

def use_cascade_attention_ref(common_prefix_len, query_lens, num_query_heads,
                              num_kv_heads, use_alibi, use_sliding_window,
                              use_local_attention, num_sms):
    """Cascade-or-not decision of vLLM v1 ``use_cascade_attention``.

    Thresholds: prefix >= 256 tokens, >= 8 requests, no ALiBi / window /
    local attention.  If FlashDecoding would not be used (GQA ratio 1, or any
    query longer than 1) cascade wins outright; otherwise compare the wave
    model with 128 x 128 tiles:
    cascade = ceil(Hq * ceil(B / 128) / SMs) * ceil(P / 128) against
    flash-decoding = ceil(B * Hkv * ceil(G / 128) * ceil(P / 128) / SMs).
    """
    def cdiv(a, b):
        return -(-a // b)

    if common_prefix_len < 256:
        return False
    if use_alibi or use_sliding_window or use_local_attention:
        return False
    query_lens = np.asarray(query_lens)
    num_reqs = len(query_lens)
    if num_reqs < 8:
        return False
    group = num_query_heads // num_kv_heads
    flash_decoding = (group > 1 and not use_sliding_window and not use_alibi
                      and bool(np.all(query_lens == 1)))
    if not flash_decoding:
        return True
    tiles = cdiv(common_prefix_len, 128)
    cascade_time = cdiv(num_query_heads * cdiv(num_reqs, 128), num_sms) * tiles
    fd_ctas = num_reqs * num_kv_heads * cdiv(group, 128) * tiles
    return cascade_time < cdiv(fd_ctas, num_sms)


def lse_log2_to_ln(lse2):
    """FlashInfer page: base-2 LSE times ln 2 gives the natural-log LSE."""
    return np.asarray(lse2, dtype=np.float64) * math.log(2.0)
