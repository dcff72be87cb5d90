"""One batch of paged attention resident on the GPU, and its step.

A step is the whole hot path for one batch: scatter the new K/V rows into the
cache (``reshape_and_cache_flash``), then varlen paged attention over the
cache (decode and/or prefill kernels, split-KV partials folded by LSE), or,
for a shared-prefix batch, cascade attention (prefix + suffix + LSE merge).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import api


class DeviceBatch:
    """Device tensors for a ``workloads.PagedWorkload``.

    The cache starts filled with NaN (``poison=True``) or uninitialised, so
    any read of a slot that was never written shows up in the output.
    """

    def __init__(self, wl, device="cuda", poison=True, cascade=False):
        self.wl = wl
        self.device = torch.device(device)
        dt = wl.torch_dtype
        shape = wl.cache_shape()
        if poison:
            self.kv_cache = torch.full(shape, math.nan, dtype=dt,
                                       device=self.device)
        else:
            self.kv_cache = torch.empty(shape, dtype=dt, device=self.device)
        self.key_cache, self.value_cache = self.kv_cache.unbind(0)

        def dev(x, dtype):
            return torch.as_tensor(np.ascontiguousarray(x), dtype=dtype) \
                .to(self.device)

        self.cu_seqlens_q = dev(wl.cu_seqlens_q, torch.int32)
        self.seqused_k = dev(wl.seq_lens, torch.int32)
        self.block_table = dev(wl.block_table, torch.int32)
        self.slots_ctx = dev(wl.slot_mapping_ctx, torch.int64)
        self.slots_new = dev(wl.slot_mapping_new, torch.int64)
        self.q = wl.q.to(self.device)
        self.k_new = wl.k_new.to(self.device)
        self.v_new = wl.v_new.to(self.device)
        self.k_ctx = wl.k_ctx.to(self.device)
        self.v_ctx = wl.v_ctx.to(self.device)
        self.out = torch.empty_like(self.q)
        self.alibi = None if wl.alibi_slopes is None else \
            dev(wl.alibi_slopes, torch.float32)
        self.cascade = cascade
        T = wl.num_tokens
        self.workspace = None
        if cascade:
            P = wl.common_prefix_len
            self.cu_prefix = dev([0, T], torch.int32)
            self.prefix_lens = dev([P], torch.int32)
            self.suffix_lens = dev(wl.seq_lens - P, torch.int32)
            n = api.cascade_attention_workspace_size(
                wl.batch, T, wl.max_seqlen_q, wl.max_seqlen_k, P,
                wl.num_heads, wl.num_kv_heads, wl.head_size, wl.block_size,
                wl.block_table.shape[1], wl.num_splits)
        else:
            n = api.paged_attention_workspace_size(
                wl.batch, T, wl.max_seqlen_q, wl.max_seqlen_k, wl.num_heads,
                wl.num_kv_heads, wl.head_size, wl.block_size, wl.causal,
                wl.window_size, wl.num_splits)
        if n > 0:
            self.workspace = torch.empty(n, dtype=torch.uint8,
                                         device=self.device)

    def write_context(self):
        """Set-up: put every context row in the cache (not part of a step)."""
        if self.slots_ctx.numel():
            api.reshape_and_cache_flash(self.k_ctx, self.v_ctx,
                                        self.key_cache, self.value_cache,
                                        self.slots_ctx)

    def write_new(self):
        if self.slots_new.numel():
            api.reshape_and_cache_flash(self.k_new, self.v_new,
                                        self.key_cache, self.value_cache,
                                        self.slots_new)

    def attend(self, return_lse=True):
        wl = self.wl
        if self.cascade:
            api.cascade_attention(
                self.out, self.q, self.key_cache, self.value_cache,
                self.cu_seqlens_q, wl.max_seqlen_q, self.cu_prefix,
                self.prefix_lens, self.suffix_lens, wl.max_seqlen_k,
                wl.softmax_scale, None, (-1, -1), wl.softcap,
                self.block_table, wl.common_prefix_len, wl.num_splits,
                workspace=self.workspace)
            return self.out, None
        return api.flash_attn_varlen_func(
            self.q, self.key_cache, self.value_cache, wl.max_seqlen_q,
            self.cu_seqlens_q, wl.max_seqlen_k, seqused_k=self.seqused_k,
            softmax_scale=wl.softmax_scale, causal=wl.causal,
            window_size=wl.window_size, softcap=wl.softcap,
            alibi_slopes=self.alibi, block_table=self.block_table,
            return_softmax_lse=return_lse, out=self.out,
            num_splits=wl.num_splits, workspace=self.workspace)

    def step(self, return_lse=False):
        """One pass of the hot path: cache write, then attention."""
        self.write_new()
        return self.attend(return_lse=return_lse)
