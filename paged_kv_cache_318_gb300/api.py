"""Python binding of libpkv (ctypes): argument marshalling only.

Every function takes torch tensors that already live on the GPU, reads their
pointers, strides and the current CUDA stream, and calls the C ABI declared in
``include/pkv.h``.  All computation happens in the library's kernels.  A
missing library raises ``RuntimeError``; a non-OK status raises
``ValueError`` (invalid argument), ``NotImplementedError`` (unsupported
configuration) or ``RuntimeError`` (anything else), as the attention backends
on the vLLM pages do.

Names and argument orders follow those pages: ``reshape_and_cache_flash``,
``flash_attn_varlen_func``, ``merge_attn_states`` and ``cascade_attention``
("vllm/v1/attention/backends/flash_attn.py").
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import _build

_lib = None
_lib_lock = threading.Lock()

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_WORKSPACE_TOO_SMALL = 3
PKV_ERR_CUDA = 4
PKV_ERR_BAD_INDEX = 5
PKV_ERR_TIMEOUT = 6

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}

c_i64p = ctypes.POINTER(ctypes.c_int64)
vp = ctypes.c_void_p
i32, i64, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, \
    ctypes.c_size_t


class _Options(ctypes.Structure):
    """pkv_attention_options (include/pkv.h)."""
    _fields_ = [("sinks", ctypes.c_void_p), ("kv_cache_fp8", ctypes.c_int),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("cu_seqlens_k", ctypes.c_void_p), ("total_k", ctypes.c_int),
                ("fixed_split_size", ctypes.c_int), ("q_fp8", ctypes.c_int),
                ("q_scale", ctypes.c_void_p), ("no_pdl", ctypes.c_int)]


_FP8_CACHE = (torch.float8_e4m3fn, torch.uint8)


class PkvError(RuntimeError):
    """A libpkv call returned a CUDA or device-index error."""

    def __init__(self, status, message):
        super().__init__("pkv status %d: %s" % (status, message))
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libpkv.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                "libpkv.so is not built (%s); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
        lib = ctypes.CDLL(path)
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_reshape_and_cache.restype = i32
        lib.pkv_reshape_and_cache.argtypes = [
            vp, vp, i64, i64, i64, i64, vp, vp, c_i64p, vp, i64, i32, i32,
            i32, i64, i32, ctypes.c_char_p, vp, vp, vp]
        lib.pkv_paged_attention_varlen.restype = i32
        lib.pkv_paged_attention_varlen.argtypes = [
            vp, i64, i64, vp, vp, c_i64p, vp, i64, i64, vp, vp, i32, i32,
            i32, i32, vp, i64, i32, i32, i32, i32, i32, i64, f32, i32, i32,
            i32, f32, vp, i32, vp, vp, sz, i32, vp]
        lib.pkv_paged_attention_varlen_opts.restype = i32
        lib.pkv_paged_attention_varlen_opts.argtypes = \
            lib.pkv_paged_attention_varlen.argtypes + [vp]
        lib.pkv_paged_attention_workspace_size_opts.restype = sz
        lib.pkv_paged_attention_workspace_size_opts.argtypes = [i32] * 13 + [
            vp]
        lib.pkv_paged_attention_workspace_size.restype = sz
        lib.pkv_paged_attention_workspace_size.argtypes = [i32] * 12
        lib.pkv_merge_attn_states.restype = i32
        lib.pkv_merge_attn_states.argtypes = [
            vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp]
        lib.pkv_make_local_attention_virtual_batches.restype = i32
        lib.pkv_make_local_attention_virtual_batches.argtypes = [
            i32, vp, vp, i32, vp, i64, i32, i32, ctypes.POINTER(ctypes.c_int),
            vp, vp, vp, vp, i32]
        lib.pkv_use_cascade_attention.restype = i32
        lib.pkv_use_cascade_attention.argtypes = [i32, vp] + [i32] * 8
        lib.pkv_cascade_attention_workspace_size.restype = sz
        lib.pkv_cascade_attention_workspace_size.argtypes = [i32] * 11 + [vp]
        lib.pkv_cascade_attention.restype = i32
        lib.pkv_cascade_attention.argtypes = (
            [vp, vp, i64, i64, vp, vp, c_i64p, vp, i32, vp, vp, vp, i32, i32,
             i32, f32, f32, vp, i64, i32, i32, i32, i32, i32, i32, i64, i32,
             i32, vp, sz, i32, vp, vp])
        lib.pkv_scaled_fp8_quant.restype = i32
        lib.pkv_scaled_fp8_quant.argtypes = [vp, i64, vp, i64, i64, i32, vp,
                                             i32, vp]
        lib.pkv_set_prefill_kernel.restype = i32
        lib.pkv_set_prefill_kernel.argtypes = [i32]
        lib.pkv_set_decode_kernel.restype = i32
        lib.pkv_set_decode_kernel.argtypes = [i32]
        lib.pkv_set_wait_limit_ns.restype = i32
        lib.pkv_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.pkv_launch_count.restype = ctypes.c_uint64
        lib.pkv_launch_count.argtypes = []
        lib.pkv_check_device_errors.restype = i32
        lib.pkv_check_device_errors.argtypes = [vp]
        _lib = lib
    return _lib


def _check(status):
    if status == PKV_OK:
        return
    msg = load_library().pkv_last_error().decode(errors="replace")
    if status == PKV_ERR_INVALID_ARG:
        raise ValueError(msg)
    if status == PKV_ERR_UNSUPPORTED:
        raise NotImplementedError(msg)
    raise PkvError(status, msg)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise NotImplementedError("dtype %s is not supported" % t.dtype)


def _cache_strides(key_cache, value_cache):
    if key_cache.dim() != 4:
        raise ValueError("cache views must be 4-D [num_blocks, block_size, "
                         "num_kv_heads, head_size]")
    if tuple(key_cache.stride()) != tuple(value_cache.stride()) or \
            key_cache.shape != value_cache.shape:
        raise ValueError("key_cache and value_cache must share shape and "
                         "strides")
    return (ctypes.c_int64 * 4)(*key_cache.stride())


PREFILL_TCGEN05 = 0
PREFILL_MMA_SYNC = 1
PREFILL_TCGEN05_SMEM_P = 2


def set_prefill_kernel(which: int):
    """Choose the prefill kernel (PREFILL_TCGEN05, PREFILL_TCGEN05_SMEM_P
    or PREFILL_MMA_SYNC)."""
    _check(load_library().pkv_set_prefill_kernel(int(which)))


DECODE_TMA = 0
DECODE_CP_ASYNC = 1
DECODE_PERSISTENT = 2
DECODE_AUTO = 3


def set_decode_kernel(which: int):
    """Choose the decode kernel: DECODE_AUTO (default), DECODE_PERSISTENT,
    DECODE_TMA or DECODE_CP_ASYNC."""
    _check(load_library().pkv_set_decode_kernel(int(which)))


WAIT_LIMIT_DEFAULT_NS = 2_000_000_000


def set_wait_limit_ns(ns: int = WAIT_LIMIT_DEFAULT_NS):
    """Limit of the decode kernels' bounded waits (diagnostic; a small limit
    makes calls stop with PKV_ERR_TIMEOUT)."""
    _check(load_library().pkv_set_wait_limit_ns(int(ns)))


def launch_count() -> int:
    """Kernels libpkv has launched in this process so far."""
    return int(load_library().pkv_launch_count())


def check_device_errors(device=None):
    """Synchronise the current stream and raise if a kernel skipped an
    out-of-range block id or slot since the last check."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    s = torch.cuda.current_stream(dev).cuda_stream
    _check(load_library().pkv_check_device_errors(ctypes.c_void_p(s)))


# ------------------------------------------------------------------ cache write

def reshape_and_cache_flash(key, value, key_cache, value_cache, slot_mapping,
                            kv_cache_dtype: str = "auto", k_scale=None,
                            v_scale=None):
    """Scatter key/value [>= T, Hkv, D] into the paged cache at slot_mapping.

    T = len(slot_mapping); padded rows of key/value are ignored and slots < 0
    are skipped.  key_cache/value_cache are [num_blocks, block_size, Hkv, D]
    views (e.g. ``kv_cache.unbind(0)``), any strides with D contiguous.
    """
    lib = load_library()
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if key.stride(-1) != 1 or value.stride(-1) != 1:
        raise ValueError("key/value head_size dim must be contiguous")
    if key.dtype != key_cache.dtype and kv_cache_dtype == "auto":
        raise ValueError("cache dtype must match key dtype for 'auto'")
    if kv_cache_dtype.startswith("fp8"):
        if key_cache.dtype not in _FP8_CACHE:
            raise ValueError("an fp8 cache must be float8_e4m3fn or uint8")
        if k_scale is None or v_scale is None or \
                k_scale.dtype != torch.float32 or \
                v_scale.dtype != torch.float32:
            raise ValueError("fp8 cache needs float32 k_scale and v_scale")
    NB, BS, H, D = key_cache.shape
    cs = _cache_strides(key_cache, value_cache)
    _check(lib.pkv_reshape_and_cache(
        _ptr(key), _ptr(value), key.stride(0), key.stride(1), value.stride(0),
        value.stride(1), _ptr(key_cache), _ptr(value_cache), cs,
        _ptr(slot_mapping), slot_mapping.shape[0], H, D, BS, NB,
        _dtype(key), kv_cache_dtype.encode(), _ptr(k_scale), _ptr(v_scale),
        _stream(key)))


def scaled_fp8_quant(input, scale, out=None):
    """Static per-tensor E4M3 quantization: codes of ``input / scale``.

    input [rows, cols] (or [tokens, heads, head_size], taken as [tokens,
    heads * head_size]) fp16/bf16 with contiguous rows; scale a float32
    device tensor of one element.  Returns (codes, scale), codes a
    float8_e4m3fn tensor of input's shape, as the vLLM FA backend's
    ``ops.scaled_fp8_quant(query, layer._q_scale)`` does
    ("vllm/v1/attention/backends/flash_attn.py").
    """
    lib = load_library()
    if scale is None or scale.dtype != torch.float32 or scale.numel() < 1:
        raise ValueError("scale must be a float32 tensor (static scale)")
    shape = input.shape
    x = input.reshape(shape[0], -1) if input.dim() == 3 else input
    if x.dim() != 2 or x.stride(-1) != 1:
        raise ValueError("input must be [rows, cols] with contiguous rows")
    if out is None:
        out = torch.empty(shape, dtype=torch.float8_e4m3fn,
                          device=input.device)
    elif out.dtype not in _FP8_CACHE or out.shape != shape:
        raise ValueError("out must be float8_e4m3fn/uint8 of input's shape")
    o = out.reshape(shape[0], -1) if out.dim() == 3 else out
    if o.stride(-1) != 1:
        raise ValueError("out rows must be contiguous")
    _check(lib.pkv_scaled_fp8_quant(
        _ptr(x), x.stride(0), _ptr(o), o.stride(0), x.shape[0], x.shape[1],
        _ptr(scale), _dtype(x), _stream(x)))
    return out, scale


# --------------------------------------------------------------- attention

def paged_attention_workspace_size(batch, total_q, max_seqlen_q, max_seqlen_k,
                                   num_heads, num_kv_heads, head_size,
                                   block_size, causal=True,
                                   window_size=(-1, -1), num_splits=0) -> int:
    n = load_library().pkv_paged_attention_workspace_size(
        batch, total_q, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
        head_size, block_size, int(bool(causal)), int(window_size[0]),
        int(window_size[1]), num_splits)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError(load_library().pkv_last_error().decode())
    return n


def flash_attn_varlen_func(q, k, v, max_seqlen_q, cu_seqlens_q, max_seqlen_k,
                           seqused_k=None, softmax_scale=None, causal=False,
                           window_size=(-1, -1), softcap=0.0,
                           alibi_slopes=None, block_table=None,
                           return_softmax_lse=False, out=None, num_splits=0,
                           cu_seqlens_k=None, workspace=None, s_aux=None,
                           k_descale=None, v_descale=None,
                           fixed_split_size=0, q_descale=None,
                           enable_pdl=True):
    """Varlen attention over a paged KV cache, or over plain K/V rows.

    q [T, Hq, D].  Paged: k, v are cache views [num_blocks, block_size, Hkv,
    D] with seqused_k int32 [B] and block_table int32 [B, max_blocks].
    Non-paged (encoder / cache-free prefill): k, v are [Tk, Hkv, D] and
    cu_seqlens_k int32 [B+1] gives each request's rows.  cu_seqlens_q int32
    [B+1].  fixed_split_size > 0 makes decode split-KV batch-invariant.
    An fp8 (E4M3) q, from ``scaled_fp8_quant``, needs an fp8 cache, its
    scale as ``q_descale`` and ``out`` (which names the output type).
    ``enable_pdl=False`` launches every kernel in plain stream order
    (``no_pdl`` in pkv_attention_options).
    Returns out (and lse [Hq, T] float32 when return_softmax_lse).
    """
    lib = load_library()
    nonpaged = cu_seqlens_k is not None
    if q.stride(-1) != 1:
        raise ValueError("q head_size dim must be contiguous")
    T, Hq, D = q.shape
    if nonpaged:
        if k.dim() != 3 or v.shape != k.shape:
            raise ValueError("non-paged k and v must both be [Tk, Hkv, D]")
        Tk, Hkv, Dk = k.shape
        NB, BS = 1, 16
        if cu_seqlens_k.dtype != torch.int32:
            raise ValueError("cu_seqlens_k must be int32")
        batch = cu_seqlens_k.shape[0] - 1
        if cu_seqlens_q.shape[0] != batch + 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k lengths differ")
        if k.stride(1) != v.stride(1) or k.stride(0) != v.stride(0) or \
                k.stride(2) != 1 or v.stride(2) != 1:
            raise ValueError("k and v need the same strides, D contiguous")
        cs = (ctypes.c_int64 * 4)(0, k.stride(0), k.stride(1), 1)
        max_blocks, bt_stride = 0, 0
    else:
        if block_table is None or seqused_k is None:
            raise ValueError("block_table and seqused_k are required")
        NB, BS, Hkv, Dk = k.shape
        if seqused_k.dtype != torch.int32 or block_table.dtype != torch.int32:
            raise ValueError("seqused_k and block_table must be int32")
        if block_table.stride(-1) != 1:
            raise ValueError("block_table rows must be contiguous")
        batch = seqused_k.shape[0]
        cs = _cache_strides(k, v)
        max_blocks, bt_stride = block_table.shape[1], block_table.stride(0)
    if Dk != D:
        raise ValueError("q and k head_size differ")
    kv8 = k.dtype in _FP8_CACHE
    q8 = q.dtype in _FP8_CACHE
    if q8:
        if not kv8:
            raise NotImplementedError("an fp8 query needs an fp8 cache")
        if q_descale is None or q_descale.dtype != torch.float32 or \
                q_descale.numel() < 1:
            raise ValueError("an fp8 query needs a float32 q_descale")
        if out is None:
            raise ValueError("an fp8 query needs `out` (the output type)")
    if kv8:
        if nonpaged:
            raise NotImplementedError("fp8 K/V needs the paged cache")
        if v.dtype not in _FP8_CACHE or k_descale is None or \
                v_descale is None:
            raise ValueError("an fp8 cache needs k_descale and v_descale")
    elif k.dtype != q.dtype or v.dtype != q.dtype:
        raise NotImplementedError("q and cache dtypes must match")
    if cu_seqlens_q.dtype != torch.int32:
        raise ValueError("cu_seqlens_q must be int32")
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    elif not q8 and out.dtype != q.dtype:
        raise ValueError("out must have q's dtype")
    lse = None
    if return_softmax_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    opts = _Options()
    if s_aux is not None:
        if s_aux.dtype != torch.float32 or s_aux.shape != (Hq,):
            raise ValueError("s_aux (sinks) must be float32 [num_heads]")
        opts.sinks = s_aux.data_ptr()
    if kv8:
        for t in (k_descale, v_descale):
            if t.dtype != torch.float32 or t.numel() < 1:
                raise ValueError("k_descale/v_descale must be float32")
        opts.kv_cache_fp8 = 1
        opts.k_scale = k_descale.data_ptr()
        opts.v_scale = v_descale.data_ptr()
    if q8:
        opts.q_fp8 = 1
        opts.q_scale = q_descale.data_ptr()
    if nonpaged:
        opts.cu_seqlens_k = cu_seqlens_k.data_ptr()
        opts.total_k = k.shape[0]
    opts.fixed_split_size = int(fixed_split_size)
    opts.no_pdl = 0 if enable_pdl else 1
    ws_need = lib.pkv_paged_attention_workspace_size_opts(
        batch, T, max_seqlen_q, max_seqlen_k, Hq, Hkv, D, BS,
        int(bool(causal)), int(window_size[0]), int(window_size[1]),
        num_splits, max_blocks, ctypes.byref(opts))
    if ws_need == ctypes.c_size_t(-1).value:
        raise ValueError(lib.pkv_last_error().decode())
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * \
        workspace.element_size()
    if alibi_slopes is not None and alibi_slopes.dtype != torch.float32:
        raise ValueError("alibi_slopes must be float32")
    _check(lib.pkv_paged_attention_varlen_opts(
        _ptr(q), q.stride(0), q.stride(1), _ptr(k), _ptr(v), cs, _ptr(out),
        out.stride(0), out.stride(1), _ptr(cu_seqlens_q), _ptr(seqused_k),
        batch, T, int(max_seqlen_q), int(max_seqlen_k), _ptr(block_table),
        bt_stride, max_blocks, Hq, Hkv, D, BS, NB,
        float(softmax_scale), int(bool(causal)), int(window_size[0]),
        int(window_size[1]), float(softcap or 0.0), _ptr(alibi_slopes),
        int(num_splits), _ptr(lse), _ptr(workspace), ws_bytes, _dtype(out),
        _stream(q), ctypes.byref(opts)))
    if return_softmax_lse:
        return out, lse
    return out


def make_local_attention_virtual_batches(attn_chunk_size, query_start_loc,
                                         seq_lens, block_table, block_size):
    """Chunked local attention as virtual requests (host numpy in/out).

    Returns (seqlens_q_local, cu_seqlens_q_local, seqlens_k_local,
    block_table_local) as int32 numpy arrays, as the vLLM v0.9.0.1 backend's
    ``make_local_attention_virtual_batches`` does.
    """
    import numpy as np
    lib = load_library()
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    batch = len(sl)
    n = ctypes.c_int(0)
    P = ctypes.c_void_p
    _check(lib.pkv_make_local_attention_virtual_batches(
        attn_chunk_size, qsl.ctypes.data_as(P), sl.ctypes.data_as(P), batch,
        bt.ctypes.data_as(P), bt.shape[1], bt.shape[1], block_size,
        ctypes.byref(n), None, None, None, None, 0))
    V, pages = n.value, attn_chunk_size // block_size
    sq = np.empty(V, np.int32)
    cu = np.empty(V + 1, np.int32)
    sk = np.empty(V, np.int32)
    btl = np.empty((V, pages), np.int32)
    _check(lib.pkv_make_local_attention_virtual_batches(
        attn_chunk_size, qsl.ctypes.data_as(P), sl.ctypes.data_as(P), batch,
        bt.ctypes.data_as(P), bt.shape[1], bt.shape[1], block_size,
        ctypes.byref(n), sq.ctypes.data_as(P), cu.ctypes.data_as(P),
        sk.ctypes.data_as(P), btl.ctypes.data_as(P), V))
    return sq, cu, sk, btl


def use_cascade_attention(common_prefix_len, query_lens, num_query_heads,
                          num_kv_heads, use_alibi, use_sliding_window,
                          use_local_attention, num_sms, dcp_world_size=1):
    """vLLM v1 ``use_cascade_attention`` policy (host, native)."""
    import numpy as np
    ql = np.ascontiguousarray(query_lens, dtype=np.int32)
    return bool(load_library().pkv_use_cascade_attention(
        int(common_prefix_len), ql.ctypes.data_as(ctypes.c_void_p), len(ql),
        num_query_heads, num_kv_heads, int(bool(use_alibi)),
        int(bool(use_sliding_window)), int(bool(use_local_attention)),
        int(num_sms), int(dcp_world_size)))


def merge_attn_states(output, prefix_output, prefix_lse, suffix_output,
                      suffix_lse, output_lse=None):
    """output = LSE-weighted combination of two partial attentions.

    outputs [T, H, D] contiguous; LSEs float32 [H, T] contiguous.
    """
    lib = load_library()
    for t in (output, prefix_output, suffix_output, prefix_lse, suffix_lse):
        if not t.is_contiguous():
            raise ValueError("merge_attn_states needs contiguous tensors")
    if prefix_output.dtype != suffix_output.dtype:
        raise ValueError("prefix and suffix outputs must share a dtype")
    T, H, D = output.shape
    if prefix_lse.shape != (H, T) or suffix_lse.shape != (H, T):
        raise ValueError("LSE shape must be [num_heads, num_tokens]")
    _check(lib.pkv_merge_attn_states(
        _ptr(output), _ptr(prefix_output), _ptr(prefix_lse),
        _ptr(suffix_output), _ptr(suffix_lse), _ptr(output_lse), T, H, D,
        _dtype(output), _dtype(prefix_output), _stream(output)))
    return output


_SIDE_STREAMS = {}


def cascade_attention_workspace_size(batch, num_tokens, max_query_len,
                                     max_kv_len, common_prefix_len,
                                     num_heads, num_kv_heads, head_size,
                                     block_size, max_blocks_per_seq,
                                     num_splits=0) -> int:
    """Workspace bytes of ``cascade_attention`` (16-bit cache and query)."""
    n = load_library().pkv_cascade_attention_workspace_size(
        batch, num_tokens, max_query_len, max_kv_len, common_prefix_len,
        num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
        num_splits, None)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid cascade shapes")
    return n


def cascade_attention(output, query, key_cache, value_cache, cu_query_lens,
                      max_query_len, cu_prefix_query_lens, prefix_kv_lens,
                      suffix_kv_lens, max_kv_len, softmax_scale,
                      alibi_slopes, sliding_window, logits_soft_cap,
                      block_table, common_prefix_len, max_num_splits=0,
                      workspace=None, s_aux=None, overlap=True,
                      k_descale=None, v_descale=None, q_descale=None):
    """Shared-prefix attention: prefix (non-causal, block_table[:1], with the
    sinks) + suffix (causal, block_table[:, P/BS:]) merged by LSE, as in
    vLLM v1's ``cascade_attention``, in one library call.

    With ``overlap`` the suffix's decode kernel starts beside the prefix
    kernel on the SMs it leaves free (same bits as ``overlap=False``).
    ``max_num_splits`` is the suffix's split-KV; the prefix runs unsplit.
    ``output`` must be contiguous [num_tokens, num_heads, head_size]."""
    lib = load_library()
    if alibi_slopes is not None:
        raise ValueError("Cascade attention does not support ALiBi.")
    if tuple(sliding_window) != (-1, -1):
        raise ValueError("Cascade attention does not support sliding window.")
    T, Hq, D = query.shape
    NB, BS, Hkv, Dk = key_cache.shape
    if common_prefix_len % BS != 0:
        raise ValueError("common_prefix_len must be a multiple of block_size")
    if common_prefix_len <= 0:
        raise ValueError("common_prefix_len must be > 0")
    if not output.is_contiguous() or output.shape != query.shape[:2] + (D,):
        raise ValueError("output must be contiguous [T, Hq, D]")
    if query.stride(-1) != 1:
        raise ValueError("query head_size dim must be contiguous")
    for t in (cu_query_lens, cu_prefix_query_lens, prefix_kv_lens,
              suffix_kv_lens, block_table):
        if t.dtype != torch.int32:
            raise ValueError("lengths and block_table must be int32")
    opts = _Options()
    if s_aux is not None:
        if s_aux.dtype != torch.float32 or s_aux.shape != (Hq,):
            raise ValueError("s_aux (sinks) must be float32 [num_heads]")
        opts.sinks = s_aux.data_ptr()
    kv8 = key_cache.dtype in _FP8_CACHE
    q8 = query.dtype in _FP8_CACHE
    if kv8:
        if k_descale is None or v_descale is None:
            raise ValueError("an fp8 cache needs k_descale and v_descale")
        opts.kv_cache_fp8 = 1
        opts.k_scale = k_descale.data_ptr()
        opts.v_scale = v_descale.data_ptr()
    elif key_cache.dtype != query.dtype:
        raise NotImplementedError("q and cache dtypes must match")
    if q8:
        if q_descale is None:
            raise ValueError("an fp8 query needs q_descale")
        opts.q_fp8 = 1
        opts.q_scale = q_descale.data_ptr()
    batch = suffix_kv_lens.shape[0]
    max_blocks = block_table.shape[1]
    need = lib.pkv_cascade_attention_workspace_size(
        batch, T, int(max_query_len), int(max_kv_len),
        int(common_prefix_len), Hq, Hkv, D, BS, max_blocks,
        int(max_num_splits), ctypes.byref(opts))
    if need == ctypes.c_size_t(-1).value:
        raise ValueError("invalid cascade shapes")
    if workspace is None or workspace.numel() * workspace.element_size() < \
            need:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    cs = _cache_strides(key_cache, value_cache)
    _check(lib.pkv_cascade_attention(
        _ptr(output), _ptr(query), query.stride(0), query.stride(1),
        _ptr(key_cache), _ptr(value_cache), cs, _ptr(cu_query_lens),
        int(max_query_len), _ptr(cu_prefix_query_lens), _ptr(prefix_kv_lens),
        _ptr(suffix_kv_lens), int(max_kv_len), batch, T,
        float(softmax_scale), float(logits_soft_cap or 0.0),
        _ptr(block_table), block_table.stride(0), max_blocks,
        int(common_prefix_len), Hq, Hkv, D, BS, NB, int(max_num_splits),
        int(bool(overlap)), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _dtype(output),
        _stream(query), ctypes.byref(opts)))
    return output
