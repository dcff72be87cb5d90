"""Glue that feeds a seeded workload to the float64 oracle.

TEST INFRASTRUCTURE ONLY (tests, smoke, the bench's CPU baseline).  It reads
the workload's metadata arrays and drawn rows (converted to float64 on the
host) and calls the oracle functions; it never touches the CUDA path.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import (cascade_ref, paged_attention_ref,
                              reshape_and_cache_ref)


def _f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _bits16(t):
    import torch  # the rows arrive as torch tensors
    return t.detach().cpu().contiguous().view(torch.int16).numpy() \
        .view(np.uint16)


def full_cache_bits(wl, poison_bits):
    """The whole cache after the context and new rows are written, as raw
    16-bit patterns [2, NB, BS, Hkv, D] (bit-exact reference for the cache
    write).  Unwritten rows hold ``poison_bits``, the pattern the cache was
    filled with before any write."""
    shape = wl.cache_shape()
    kc = np.full(shape[1:], poison_bits, dtype=np.uint16)
    vc = np.full(shape[1:], poison_bits, dtype=np.uint16)
    reshape_and_cache_ref(_bits16(wl.k_ctx), _bits16(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_bits16(wl.k_new), _bits16(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    return np.stack([kc, vc])


def full_reference(wl):
    """Oracle out [T, Hq, D] and lse [Hq, T] for the whole workload, going
    through the oracle's own cache scatter (float64 cache, NaN elsewhere)."""
    shape = wl.cache_shape()
    kc = np.full(shape[1:], np.nan)
    vc = np.full(shape[1:], np.nan)
    reshape_and_cache_ref(_f64(wl.k_ctx), _f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_f64(wl.k_new), _f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    q = _f64(wl.q)
    if wl.common_prefix_len > 0:
        return cascade_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                           wl.block_table, wl.common_prefix_len,
                           wl.softmax_scale, softcap=wl.softcap)
    return paged_attention_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                               wl.block_table, wl.softmax_scale,
                               causal=wl.causal, window_size=wl.window_size,
                               softcap=wl.softcap,
                               alibi_slopes=wl.alibi_slopes)


def _ctx_layout(wl):
    """First context position and row offset of each request's context rows
    (shared-prefix rows are stored once, by request 0)."""
    P = wl.common_prefix_len
    first = np.zeros(wl.batch, dtype=np.int64)
    if P:
        first[1:] = P
    n_ctx = (wl.seq_lens - wl.q_lens).astype(np.int64) - first
    n_ctx = np.maximum(n_ctx, 0)
    offs = np.zeros(wl.batch + 1, dtype=np.int64)
    np.cumsum(n_ctx, out=offs[1:])
    return first, offs


def request_rows(wl, b):
    """K and V rows of request b in position order, float64 [L_b, Hkv, D]."""
    first, offs = _ctx_layout(wl)
    L, q = int(wl.seq_lens[b]), int(wl.q_lens[b])
    t0 = int(wl.cu_seqlens_q[b])
    parts_k, parts_v = [], []
    if first[b] > 0:                      # shared prefix lives in request 0
        parts_k.append(wl.k_ctx[0:first[b]])
        parts_v.append(wl.v_ctx[0:first[b]])
    parts_k.append(wl.k_ctx[offs[b]:offs[b + 1]])
    parts_v.append(wl.v_ctx[offs[b]:offs[b + 1]])
    parts_k.append(wl.k_new[t0:t0 + q])
    parts_v.append(wl.v_new[t0:t0 + q])
    import torch
    k = _f64(torch.cat(parts_k))
    v = _f64(torch.cat(parts_v))
    assert k.shape[0] == L, (k.shape, L)
    return k, v


def request_reference(wl, b, last_rows=None, row_range=None):
    """Oracle out [k, Hq, D] and lse [Hq, k] for the last k queries of
    request b (all q_b queries when ``last_rows`` and ``row_range`` are
    None), or for its queries i0 .. i1-1 with ``row_range = (i0, i1)``.

    The request's rows are laid out in a compact cache (its logical blocks
    in order), which the oracle's block-permutation invariance makes
    equivalent to the workload's own table.  The last k queries of a request
    are themselves a request with q_len = k over the same keys (the queries
    are the last q_len positions), so sampling needs no other change.  A
    causal request's queries i0 .. i1-1 see no key past position c + i1 - 1
    (c = context length), so they are the last i1 - i0 queries of the same
    request cut to its first c + i1 keys; row ranges need a causal workload.
    """
    k, v = request_rows(wl, b)
    if row_range is not None:
        if not wl.causal:
            raise ValueError("row_range needs a causal workload")
        i0, i1 = (int(x) for x in row_range)
        q_b = int(wl.q_lens[b])
        assert 0 <= i0 < i1 <= q_b, (i0, i1, q_b)
        cut = int(wl.seq_lens[b]) - q_b + i1
        k, v = k[:cut], v[:cut]
        last_rows = i1 - i0
        t_end = int(wl.cu_seqlens_q[b]) + i1
    else:
        t_end = int(wl.cu_seqlens_q[b + 1])
    BS = wl.block_size
    L = k.shape[0]
    nb = max(-(-L // BS), 1)
    Hkv, D = k.shape[1], k.shape[2]
    kc = np.full((nb, BS, Hkv, D), np.nan)
    vc = np.full((nb, BS, Hkv, D), np.nan)
    kc.reshape(nb * BS, Hkv, D)[:L] = k
    vc.reshape(nb * BS, Hkv, D)[:L] = v
    t0, t1 = int(wl.cu_seqlens_q[b]), t_end
    if last_rows is not None:
        t0 = max(t0, t1 - int(last_rows))
    q = _f64(wl.q[t0:t1])
    table = np.arange(nb, dtype=np.int32)[None, :]
    # (for a shared-prefix workload this is the flat form, which the pinned
    # cascade == flat invariant makes equal to the cascade result)
    out, lse = paged_attention_ref(q, kc, vc, np.array([0, t1 - t0]),
                                   np.array([L]), table, wl.softmax_scale,
                                   causal=wl.causal,
                                   window_size=wl.window_size,
                                   softcap=wl.softcap,
                                   alibi_slopes=wl.alibi_slopes)
    return out, lse
