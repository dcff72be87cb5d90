"""Chunked local attention: oracle for the virtual-batch transform.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Source: "vllm.v1.attention.backends.flash_attn" (vLLM v0.9.0.1 docs),
``make_local_attention_virtual_batches`` and its use in
``FlashAttentionMetadataBuilder.build``: with attention chunk size C, each
request is split into virtual requests, one per C-aligned chunk of its keys
that holds at least one of its queries; the chunk's queries attend causally
to the chunk's keys only.  The page prints a worked example (C = 4,
q_seqlens [4, 10, 5], k_seqlens [6, 17, 9], block_size 2), stored in
tests/golden/local_virtual_batches_example.json.

Two functions:
* ``local_virtual_batches_ref`` -- the transform, written as its plain
  definition (a loop over each request's chunks), pinned by the worked
  example;
* ``local_attention_ref`` -- chunked local attention written directly as a
  mask (query at p sees key j iff j <= p and j // C == p // C), independent of
  the transform; attention over the virtual batches must equal it.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import gather_ref


def local_virtual_batches_ref(attn_chunk_size, query_start_loc, seq_lens,
                              block_table, block_size):
    """Returns (seqlens_q_local, cu_seqlens_q_local, seqlens_k_local,
    block_table_local) as int32 numpy arrays.

    For request b with q_b queries (positions L_b - q_b .. L_b - 1) and
    chunk c (keys c*C .. c*C + C - 1) that holds a query: the virtual
    request has the queries inside chunk c, keys c*C .. min(L_b, (c+1)*C) - 1
    (its seqused_k counts from c*C), and the block-table columns
    c*C/BS .. c*C/BS + C/BS - 1 of row b (clipped to the last column).
    """
    C, BS = int(attn_chunk_size), int(block_size)
    assert C % BS == 0
    pages = C // BS
    block_table = np.asarray(block_table)
    width = block_table.shape[1]
    sq, sk, rows = [], [], []
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        q = int(query_start_loc[b + 1]) - int(query_start_loc[b])
        assert q > 0
        first_pos, last_pos = L - q, L - 1
        for c in range(first_pos // C, last_pos // C + 1):
            lo, hi = c * C, (c + 1) * C
            sq.append(min(hi, L) - max(lo, first_pos))
            sk.append(min(hi, L) - lo)
            cols = [min(lo // BS + i, width - 1) for i in range(pages)]
            rows.append(block_table[b, cols])
    seqlens_q = np.array(sq, dtype=np.int32)
    cu = np.zeros(len(sq) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens_q)
    return (seqlens_q, cu, np.array(sk, dtype=np.int32),
            np.array(rows, dtype=np.int32).reshape(len(rows), pages))


def local_attention_ref(q, key_cache, value_cache, cu_seqlens_q, seqused_k,
                        block_table, softmax_scale, attn_chunk_size):
    """Causal attention restricted to each query's own key chunk.

    q [T, Hq, D] float64; caches [NB, BS, Hkv, D]; returns out [T, Hq, D],
    lse [Hq, T] (natural log).
    """
    C = int(attn_chunk_size)
    T, Hq, D = q.shape
    Hkv = key_cache.shape[2]
    group = Hq // Hkv
    out = np.zeros((T, Hq, D))
    lse = np.full((Hq, T), -np.inf)
    for b in range(len(seqused_k)):
        t0, t1 = int(cu_seqlens_q[b]), int(cu_seqlens_q[b + 1])
        L = int(seqused_k[b])
        k_b = gather_ref(key_cache, block_table[b], L).astype(np.float64)
        v_b = gather_ref(value_cache, block_table[b], L).astype(np.float64)
        p = (L - (t1 - t0) + np.arange(t1 - t0))[:, None]
        j = np.arange(L)[None, :]
        ok = (j <= p) & (j // C == p // C)
        for h in range(Hq):
            s = softmax_scale * (q[t0:t1, h] @ k_b[:, h // group].T)
            s = np.where(ok, s, -np.inf)
            m = s.max(axis=1)
            w = np.exp(s - m[:, None])
            den = w.sum(axis=1)
            out[t0:t1, h] = (w @ v_b[:, h // group]) / den[:, None]
            lse[h, t0:t1] = m + np.log(den)
    return out, lse
