"""The allocation-free attention entry point.

``pkv_paged_attention_varlen_static_scratch`` serves callers that cannot
allocate device memory (runtimes that plan every device byte up front and
give a call no scratch, loops that must not call cudaMalloc/cudaFree because
those can block and synchronise the device).  It takes its split-KV scratch
from a fixed array inside the library.  Here it is called through the C ABI
twice in a row, on different inputs.  Each result must equal the regular
workspace entry point's bit for bit (the two run the same plan and kernels;
only where the scratch lives differs) and match the float64 oracle within
the parity tolerance of the other tests.  A call that needs more scratch
than the array holds must be rejected.

This file sorts last so that a run stopping at the first failure has run
every other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle.harness import request_reference
from paged_kv_cache_318_gb300 import api, workloads
from paged_kv_cache_318_gb300.batch import DeviceBatch

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f16": 4e-3}
LSE_TOL = 1e-3
STATIC_SCRATCH_BYTES = 16 << 20     # PKV_STATIC_SCRATCH_BYTES in pkv.h


def _entry(lib):
    fn = lib.pkv_paged_attention_varlen_static_scratch
    vp, i32, i64, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                         ctypes.c_float)
    fn.restype = i32
    fn.argtypes = [vp, i64, i64, vp, vp, ctypes.POINTER(ctypes.c_int64), vp,
                   i64, i64, vp, vp, i32, i32, i32, i32, vp, i64, i32, i32,
                   i32, i32, i32, i64, f32, i32, i32, i32, f32, vp, i32, vp,
                   i32, vp]
    return fn


def _call_static(fn, b, out, lse, num_splits, max_seqlen_k=None):
    wl = b.wl
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa
    cs = (ctypes.c_int64 * 4)(*b.key_cache.stride())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(p(b.q), b.q.stride(0), b.q.stride(1), p(b.key_cache),
              p(b.value_cache), cs, p(out), out.stride(0), out.stride(1),
              p(b.cu_seqlens_q), p(b.seqused_k), wl.batch, wl.num_tokens,
              wl.max_seqlen_q,
              wl.max_seqlen_k if max_seqlen_k is None else max_seqlen_k,
              p(b.block_table), b.block_table.stride(0),
              b.block_table.shape[1], wl.num_heads, wl.num_kv_heads,
              wl.head_size, wl.block_size, wl.num_blocks,
              float(wl.softmax_scale), int(wl.causal), wl.window_size[0],
              wl.window_size[1], float(wl.softcap), None, num_splits, p(lse),
              1 if wl.dtype == "bf16" else 0, stream)


def _assert_oracle(wl, out, lse):
    """Every request of wl against the float64 oracle."""
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    for b in range(wl.batch):
        t0, t1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
        ref_o, ref_l = request_reference(wl, b)
        err = np.abs(o[t0:t1] - ref_o).max()
        lerr = np.abs(ls[:, t0:t1] - ref_l).max()
        assert err <= TOL[wl.dtype], (b, err)
        assert lerr <= LSE_TOL, (b, lerr)


@pytest.fixture(scope="module")
def lib(cuda_device):
    from paged_kv_cache_318_gb300 import _build
    _build.build()
    return api.load_library()


def test_static_scratch_matches_workspace_entry(cuda_device, lib):
    fn = _entry(lib)
    cases = [
        (workloads.batched_decode(batch=16, lo=300, hi=3000,
                                  pool_blocks=4000, device=cuda_device), 4),
        (workloads.long_decode(batch=3, ctx=9000, num_splits=16,
                               dtype="f16", device=cuda_device), 16),
    ]
    batches = []
    for wl, splits in cases:
        wl.num_splits = splits
        b = DeviceBatch(wl, cuda_device)
        b.write_context()
        b.write_new()
        need = api.paged_attention_workspace_size(
            wl.batch, wl.num_tokens, wl.max_seqlen_q, wl.max_seqlen_k,
            wl.num_heads, wl.num_kv_heads, wl.head_size, wl.block_size,
            wl.causal, wl.window_size, splits)
        assert 0 < need <= STATIC_SCRATCH_BYTES   # the scratch is used
        ref_out, ref_lse = b.attend()             # regular entry point
        batches.append((b, ref_out.clone(), ref_lse.clone(), splits))
    # two calls in a row of the allocation-free entry point
    for b, ref_out, ref_lse, splits in batches:
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _call_static(fn, b, out, lse, splits)
        assert st == 0, lib.pkv_last_error()
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        _assert_oracle(b.wl, out, lse)


def test_static_scratch_rejects_oversized_plans(cuda_device, lib):
    fn = _entry(lib)
    wl = workloads.batched_decode(batch=64, lo=500, hi=600, pool_blocks=3000,
                                  device=cuda_device)
    b = DeviceBatch(wl, cuda_device)
    out = torch.empty_like(b.q)
    # 64 splits over a (claimed) 2M-key range: far beyond 16 MiB of scratch
    need = api.paged_attention_workspace_size(
        wl.batch, wl.num_tokens, 1, 1 << 21, wl.num_heads, wl.num_kv_heads,
        wl.head_size, wl.block_size, True, (-1, -1), 64)
    assert need > STATIC_SCRATCH_BYTES
    st = _call_static(fn, b, out, None, 64, max_seqlen_k=1 << 21)
    assert st == api.PKV_ERR_WORKSPACE_TOO_SMALL
    assert b"built-in scratch" in lib.pkv_last_error()


def test_static_scratch_prefill_uses_the_optional_tail(cuda_device, lib):
    """Prefill-class calls: the required scratch is zero, and the optional
    tail (the prefill item counter and, with few work items, its split-KV
    partials) comes from the built-in array when it fits.  The results equal
    the workspace entry point's bit for bit, with and without a split."""
    fn = _entry(lib)
    cases = [
        # few items: the prefill kernel splits its keys
        workloads.build_workload("ss_split", 970, [200], [6000], 32, 8, 128,
                                 16, device=cuda_device),
        # many items: no split, items dealt at run time
        workloads.prefill_with_prefix(device=cuda_device),
    ]
    for wl in cases:
        b = DeviceBatch(wl, cuda_device)
        b.write_context()
        b.write_new()
        need = api.paged_attention_workspace_size(
            wl.batch, wl.num_tokens, wl.max_seqlen_q, wl.max_seqlen_k,
            wl.num_heads, wl.num_kv_heads, wl.head_size, wl.block_size,
            wl.causal, wl.window_size, 0)
        assert 256 <= need <= STATIC_SCRATCH_BYTES   # the tail fits
        ref_out, ref_lse = b.attend()
        ref_out, ref_lse = ref_out.clone(), ref_lse.clone()
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _call_static(fn, b, out, lse, 0)
        assert st == 0, lib.pkv_last_error()
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
        if wl.batch == 1:       # (the oracle runs the small case only)
            _assert_oracle(wl, out, lse)


def test_static_scratch_call_captured_in_cuda_graph(cuda_device, lib):
    """After a first call (which sets the kernels' shared-memory limits),
    a call of the allocation-free entry point can be captured into a CUDA
    graph: a device allocation or a synchronising call inside it would fail
    the capture.  Replays equal the eager call bit for bit."""
    fn = _entry(lib)
    wl = workloads.batched_decode(batch=16, lo=300, hi=3000,
                                  pool_blocks=4000, device=cuda_device)
    wl.num_splits = 4
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    ref_out = torch.empty_like(b.q)
    ref_lse = torch.empty((wl.num_heads, wl.num_tokens), dtype=torch.float32,
                          device=cuda_device)
    assert _call_static(fn, b, ref_out, ref_lse, 4) == 0, lib.pkv_last_error()
    torch.cuda.synchronize()
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        st = _call_static(fn, b, out, lse, 4)
    assert st == 0, lib.pkv_last_error()
    for _ in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    _assert_oracle(b.wl, out, lse)
