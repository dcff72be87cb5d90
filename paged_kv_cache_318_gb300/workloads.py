"""Seeded synthetic inputs for paged attention (lengths, block pools, rows).

This module draws inputs only: request lengths, block tables taken without
replacement from a shuffled block pool, slot mappings, and N(0,1) rows for
Q/K/V rounded to the working dtype.  It holds none of the attention
arithmetic, so the CUDA path and the float64 oracle can both be fed from it.

Conventions the inputs follow (cited by page title and section):

* cache shape [2, num_blocks, block_size, num_kv_heads, head_size], block
  table [B, max_blocks] int32, slot_mapping int64 with slot =
  block_id * block_size + offset ("vllm/v1/attention/backends/flash_attn.py",
  ``FlashAttentionBackend.get_kv_cache_shape``; Aphrodite
  ``FlashAttentionMetadata`` block-table note);
* cu_seqlens_q is the running sum of the query lengths, e.g. lengths [4, 6]
  give [0, 4, 10] (Aphrodite ``FlashAttentionMetadata.seq_start_loc`` note);
* seqused_k = context + query length; a request's queries are its last
  query_len positions (vLLM v1 ``FlashAttentionMetadata`` note);
* table entries past a request's last block point at an unused "pad" block,
  which tests fill with NaN to catch over-reads.

Values are drawn with ``numpy.random.default_rng`` on the host (float32
N(0,1), rounded to the dtype by torch's round-to-nearest-even cast) or, for
multi-GB caches, with a seeded ``torch.Generator`` on the device.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16}


def cu_seqlens(lengths) -> np.ndarray:
    """Running sum of lengths with a leading zero, int32 [B+1]."""
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=out[1:])
    return out.astype(np.int32)


@dataclasses.dataclass
class PagedWorkload:
    """One batch of paged-attention inputs.

    Metadata are numpy arrays.  Values are torch tensors in ``dtype`` on
    ``device``.  ``k_ctx``/``v_ctx`` are the rows already in the cache before
    the step (written once at set-up); ``k_new``/``v_new`` are the step's new
    rows, in query order.
    """
    name: str
    seed: int
    dtype: str
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    num_blocks: int
    q_lens: np.ndarray          # int32 [B]
    seq_lens: np.ndarray        # int32 [B]   (seqused_k)
    cu_seqlens_q: np.ndarray    # int32 [B+1]
    block_table: np.ndarray     # int32 [B, max_blocks]
    slot_mapping_ctx: np.ndarray  # int64 [N_ctx]
    slot_mapping_new: np.ndarray  # int64 [T]
    pad_block: int
    unused_blocks: np.ndarray   # int64, blocks no request uses
    softmax_scale: float
    causal: bool = True
    window_size: tuple = (-1, -1)
    softcap: float = 0.0
    alibi_slopes: Optional[np.ndarray] = None
    num_splits: int = 0
    common_prefix_len: int = 0
    q: Optional[torch.Tensor] = None        # [T, Hq, D]
    k_new: Optional[torch.Tensor] = None    # [T, Hkv, D]
    v_new: Optional[torch.Tensor] = None
    k_ctx: Optional[torch.Tensor] = None    # [N_ctx, Hkv, D]
    v_ctx: Optional[torch.Tensor] = None

    @property
    def batch(self) -> int:
        return len(self.q_lens)

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max()) if len(self.q_lens) else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seq_lens.max()) if len(self.seq_lens) else 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def cache_shape(self):
        return (2, self.num_blocks, self.block_size, self.num_kv_heads,
                self.head_size)


def _draw_lengths(rng, lo, hi, n):
    return rng.integers(lo, hi, size=n, endpoint=True).astype(np.int32)


def build_workload(name, seed, q_lens, seq_lens, num_heads, num_kv_heads,
                   head_size, block_size, *, dtype="bf16", pool_blocks=None,
                   shared_prefix_len=0, softmax_scale=None, causal=True,
                   window_size=(-1, -1), softcap=0.0, alibi_slopes=None,
                   num_splits=0, device="cpu", values=True) -> PagedWorkload:
    """Assemble a workload from given lengths.

    Blocks come from ``rng.permutation(pool)`` in order, without replacement.
    With ``shared_prefix_len`` P > 0 (a multiple of block_size) every request
    starts with the same P/block_size physical blocks; the prefix rows are
    written once, by request 0.
    """
    rng = np.random.default_rng([seed, 0])
    q_lens = np.asarray(q_lens, dtype=np.int32)
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(q_lens)
    assert np.all(seq_lens >= q_lens)
    assert shared_prefix_len % block_size == 0
    n_shared = shared_prefix_len // block_size
    blocks_per = -(-seq_lens.astype(np.int64) // block_size)
    own = np.maximum(blocks_per - n_shared, 0) if n_shared else blocks_per
    need = int(own.sum()) + n_shared + 1          # + one pad block
    if pool_blocks is None:
        pool_blocks = need + max(8, need // 16)
    assert pool_blocks >= need, (pool_blocks, need)
    perm = rng.permutation(pool_blocks).astype(np.int64)
    max_blocks = int(blocks_per.max()) if B else 1
    max_blocks = max(max_blocks, 1)
    pos = 0
    shared = perm[pos:pos + n_shared]
    pos += n_shared
    table = np.empty((B, max_blocks), dtype=np.int64)
    for b in range(B):
        nb = int(own[b])
        row = np.concatenate([shared, perm[pos:pos + nb]]) if n_shared \
            else perm[pos:pos + nb]
        pos += nb
        table[b, :len(row)] = row
        table[b, len(row):] = -1
    unused = perm[pos:]
    pad_block = int(unused[0])
    table[table < 0] = pad_block

    slots_ctx, slots_new = [], []
    for b in range(B):
        L, q = int(seq_lens[b]), int(q_lens[b])
        first = shared_prefix_len if (n_shared and b > 0) else 0
        j = np.arange(first, L, dtype=np.int64)
        s = table[b, j // block_size] * block_size + j % block_size
        c = L - q
        slots_ctx.append(s[j < c])
        slots_new.append(s[j >= c])
    wl = PagedWorkload(
        name=name, seed=seed, dtype=dtype, num_heads=num_heads,
        num_kv_heads=num_kv_heads, head_size=head_size,
        block_size=block_size, num_blocks=pool_blocks, q_lens=q_lens,
        seq_lens=seq_lens, cu_seqlens_q=cu_seqlens(q_lens),
        block_table=table.astype(np.int32),
        slot_mapping_ctx=np.concatenate(slots_ctx) if B else
        np.zeros(0, np.int64),
        slot_mapping_new=np.concatenate(slots_new) if B else
        np.zeros(0, np.int64),
        pad_block=pad_block, unused_blocks=unused,
        softmax_scale=(1.0 / math.sqrt(head_size) if softmax_scale is None
                       else float(softmax_scale)),
        causal=causal, window_size=tuple(window_size), softcap=float(softcap),
        alibi_slopes=None if alibi_slopes is None else
        np.asarray(alibi_slopes, dtype=np.float32),
        num_splits=num_splits, common_prefix_len=shared_prefix_len)
    if values:
        draw_values(wl, device=device)
    return wl


def draw_values(wl: PagedWorkload, device="cpu"):
    """Draw Q, context K/V and new K/V rows, N(0,1), rounded to wl.dtype."""
    T = wl.num_tokens
    n_ctx = len(wl.slot_mapping_ctx)
    Hq, Hkv, D = wl.num_heads, wl.num_kv_heads, wl.head_size
    shapes = [("q", (T, Hq, D)), ("k_new", (T, Hkv, D)),
              ("v_new", (T, Hkv, D)), ("k_ctx", (n_ctx, Hkv, D)),
              ("v_ctx", (n_ctx, Hkv, D))]
    tdt = wl.torch_dtype
    if str(device) == "cpu":
        rng = np.random.default_rng([wl.seed, 1])
        for key, shp in shapes:
            x = rng.standard_normal(size=shp, dtype=np.float32)
            setattr(wl, key, torch.from_numpy(x).to(tdt))
    else:
        gen = torch.Generator(device=device)
        gen.manual_seed(wl.seed * 7919 + 1)
        for key, shp in shapes:
            x = torch.empty(shp, dtype=tdt, device=device)
            if x.numel():
                x.normal_(generator=gen)
            setattr(wl, key, x)
    return wl


# ---------------------------------------------------------------------------
# The five workloads (and scaled-down variants for fast tests)
# ---------------------------------------------------------------------------

def tiny_decode(seed=318, dtype="bf16", device="cpu"):
    """2 requests, query_len 1, lengths 37 and 50, 4/2 heads, D 64, BS 16,
    8-block pool in a seeded random order, scale 1/8."""
    return build_workload("tiny_decode", seed, [1, 1], [37, 50], 4, 2, 64, 16,
                          dtype=dtype, pool_blocks=8, softmax_scale=1 / 8,
                          device=device)


def batched_decode(seed=319, dtype="bf16", device="cpu", batch=64,
                   lo=512, hi=4096, pool_blocks=20000, values=True):
    """Llama-3-8B attention shape: 64 requests, query_len 1, 32/8 heads,
    D 128, BS 16, lengths U[512, 4096], 20k-block shuffled pool."""
    rng = np.random.default_rng([seed, 2])
    L = _draw_lengths(rng, lo, hi, batch)
    return build_workload("batched_decode", seed, np.ones(batch, np.int32), L,
                          32, 8, 128, 16, dtype=dtype,
                          pool_blocks=pool_blocks, device=device,
                          values=values)


def prefill_with_prefix(seed=320, dtype="bf16", device="cpu", batch=8,
                        q_lo=256, q_hi=2048, c_lo=0, c_hi=1024, values=True):
    """Varlen causal prefill: 8 sequences, new tokens U[256, 2048], cached
    prefix U[0, 1024], 32/8 heads, D 128, BS 16."""
    rng = np.random.default_rng([seed, 2])
    q = _draw_lengths(rng, q_lo, q_hi, batch)
    c = _draw_lengths(rng, c_lo, c_hi, batch)
    return build_workload("prefill_with_prefix", seed, q, q + c, 32, 8, 128,
                          16, dtype=dtype, device=device, values=values)


def mixed_gemma(seed=321, dtype="bf16", device="cpu", n_prefill=4,
                chunk=512, c_hi=8192, n_decode=124, d_lo=1024, d_hi=16384,
                values=True):
    """Chunked prefill + decode, Gemma-like: 4 chunks of 512 (context
    U[0, 8192]) after 124 decodes (context U[1024, 16384]); 16/8 heads,
    D 256, BS 32, window (4095, 0), soft-cap 50; decodes first."""
    rng = np.random.default_rng([seed, 2])
    dec_L = _draw_lengths(rng, d_lo, d_hi, n_decode)
    pre_c = _draw_lengths(rng, 0, c_hi, n_prefill)
    q = np.concatenate([np.ones(n_decode, np.int32),
                        np.full(n_prefill, chunk, np.int32)])
    L = np.concatenate([dec_L, pre_c + chunk]).astype(np.int32)
    return build_workload("mixed_gemma", seed, q, L, 16, 8, 256, 32,
                          dtype=dtype, window_size=(4095, 0), softcap=50.0,
                          device=device, values=values)


def long_decode(seed=322, dtype="bf16", device="cpu", batch=8,
                ctx=131072, num_splits=16, values=True):
    """Long-context split-KV decode: 8 requests x 131072 keys, 64/8 heads,
    D 128, BS 64, 16 splits per request."""
    return build_workload("long_decode", seed, np.ones(batch, np.int32),
                          np.full(batch, ctx, np.int32), 64, 8, 128, 64,
                          dtype=dtype, num_splits=num_splits, device=device,
                          values=values)


def cascade_decode(seed=323, dtype="bf16", device="cpu", batch=256,
                   prefix=8192, unique=512, values=True):
    """Shared-prefix decode: 256 requests over one 8192-token prefix held in
    the same physical blocks, plus 512 own tokens each; 64/8 heads, D 128,
    BS 64."""
    L = np.full(batch, prefix + unique, np.int32)
    return build_workload("cascade_decode", seed, np.ones(batch, np.int32), L,
                          64, 8, 128, 64, dtype=dtype,
                          shared_prefix_len=prefix, device=device,
                          values=values)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "batched_decode": batched_decode,
    "prefill_with_prefix": prefill_with_prefix,
    "mixed_gemma": mixed_gemma,
    "long_decode": long_decode,
    "cascade_decode": cascade_decode,
}


# ---------------------------------------------------------------------------
# Attention without a cache (encoder / cache-free prefill inputs)
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class NonPagedInputs:
    """Q [T, Hq, D] and K/V rows [Tk, Hkv, D] with their cu_seqlens."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens_q: np.ndarray
    cu_seqlens_k: np.ndarray
    dtype: str


def nonpaged_inputs(seed, q_lens, k_lens, num_heads, num_kv_heads, head_size,
                    dtype="bf16"):
    """N(0,1) values rounded to ``dtype`` (CPU tensors), drawn in a fixed
    order from one seeded generator."""
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    rng = np.random.default_rng([seed, 2])
    T, Tk = int(sum(q_lens)), int(sum(k_lens))
    draw = lambda shp: torch.from_numpy(                     # noqa: E731
        rng.standard_normal(size=shp, dtype=np.float32)).to(tdt)
    return NonPagedInputs(
        q=draw((T, num_heads, head_size)),
        k=draw((Tk, num_kv_heads, head_size)),
        v=draw((Tk, num_kv_heads, head_size)),
        cu_seqlens_q=cu_seqlens(q_lens), cu_seqlens_k=cu_seqlens(k_lens),
        dtype=dtype)
