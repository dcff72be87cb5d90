"""The C-ABI library builds, loads, exports what include/pkv.h declares,
and rejects invalid arguments on the host (no GPU needed: validation runs
before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_318_gb300 import _build, api
    _build.build()
    return api.load_library()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(",
                                    text))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"pkv_reshape_and_cache", "pkv_paged_attention_varlen",
            "pkv_merge_attn_states", "pkv_last_error"} <= names
    for n in names:
        assert hasattr(lib, n), n


def _attn_call(lib, **kw):
    args = dict(q=None, qst=0, qsh=0, kc=None, vc=None,
                cs=(ctypes.c_int64 * 4)(2048, 128, 16, 1), out=None, ost=0,
                osh=0, cu=None, su=None, batch=1, total_q=1, max_q=1,
                max_k=16, bt=None, bts=1, maxb=1, Hq=4, Hkv=2, D=64, BS=16,
                NB=8, scale=0.125, causal=1, wl=-1, wr=-1, softcap=0.0,
                alibi=None, splits=0, lse=None, ws=None, wsb=0, dtype=1,
                stream=None)
    args.update(kw)
    return lib.pkv_paged_attention_varlen(*args.values())


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), 1),            # Hq % Hkv != 0
    (dict(BS=24), 1),                   # block_size % 16 != 0
    (dict(D=100), 2),                   # head size not supported
    (dict(D=96), 2),                    # valid for the pages, not built here
    (dict(dtype=2), 2),                 # fp32 attention
    (dict(softcap=-1.0), 1),
    (dict(splits=-2), 1),
    (dict(scale=float("inf")), 1),
])
def test_attention_rejects_bad_arguments(lib, kw, status):
    assert _attn_call(lib, **kw) == status
    assert lib.pkv_last_error()


def test_attention_empty_batch_is_noop(lib):
    assert _attn_call(lib, batch=0) == 0


def test_cache_write_rejects_bad_kv_dtype_and_block_size(lib):
    cs = (ctypes.c_int64 * 4)(2048, 128, 16, 1)
    common = [None, None, 0, 0, 0, 0, None, None, cs, None, 4, 2, 64]
    st = lib.pkv_reshape_and_cache(*common, 16, 8, 1, b"fp8_e5m2", None,
                                   None, None)
    assert st == 2 and b"fp8_e5m2" in lib.pkv_last_error()
    # fp8 (E4M3) is supported but needs its scales
    st = lib.pkv_reshape_and_cache(*common, 16, 8, 1, b"fp8", None, None,
                                   None)
    assert st == 1 and b"scale" in lib.pkv_last_error()
    st = lib.pkv_reshape_and_cache(*common, 20, 8, 1, b"auto", None, None,
                                   None)
    assert st == 1
    # zero tokens: nothing to do, no pointer needed
    zero = [None, None, 0, 0, 0, 0, None, None, cs, None, 0, 2, 64]
    assert lib.pkv_reshape_and_cache(*zero, 16, 8, 1, b"auto", None, None,
                                     None) == 0


def test_scaled_fp8_quant_rejects_bad_arguments(lib):
    q = lib.pkv_scaled_fp8_quant
    # (in, in_stride, out, out_stride, rows, cols, scale, dtype, stream)
    assert q(None, 64, None, 64, 4, 24, None, 1, None) == 2   # cols % 16
    assert q(None, 64, None, 64, 4, 64, None, 2, None) == 2   # fp32 input
    assert q(None, 64, None, 64, -1, 64, None, 1, None) == 1
    assert q(None, 64, None, 64, 4, 64, None, 1, None) == 1   # NULL
    assert b"NULL" in lib.pkv_last_error()
    assert q(None, 64, None, 64, 0, 64, None, 1, None) == 0   # nothing to do
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    one = ctypes.c_float(1.0)
    assert q(base, 32, base, 64, 4, 64, ctypes.byref(one), 1, None) == 1
    assert q(base + 8, 64, base, 64, 4, 64, ctypes.byref(one), 1,
             None) == 2                                        # unaligned


def test_attention_rejects_fp8_query_without_fp8_cache(lib):
    from paged_kv_cache_318_gb300.api import _Options
    o = _Options()
    o.q_fp8 = 1
    args = dict(q=None, qst=0, qsh=0, kc=None, vc=None,
                cs=(ctypes.c_int64 * 4)(2048, 128, 16, 1), out=None, ost=0,
                osh=0, cu=None, su=None, batch=1, total_q=1, max_q=1,
                max_k=16, bt=None, bts=1, maxb=1, Hq=4, Hkv=2, D=64, BS=16,
                NB=8, scale=0.125, causal=1, wl=-1, wr=-1, softcap=0.0,
                alibi=None, splits=0, lse=None, ws=None, wsb=0, dtype=1,
                stream=None)
    dummy = ctypes.create_string_buffer(64)
    for k in ("q", "kc", "vc", "out", "cu", "su", "bt"):
        args[k] = ctypes.addressof(dummy)
    st = lib.pkv_paged_attention_varlen_opts(*args.values(),
                                             ctypes.byref(o))
    assert st == 2 and b"fp8 cache" in lib.pkv_last_error()
    o.kv_cache_fp8 = 1
    one = ctypes.c_float(1.0)
    o.k_scale = o.v_scale = ctypes.addressof(one)
    st = lib.pkv_paged_attention_varlen_opts(*args.values(),
                                             ctypes.byref(o))
    assert st == 1 and b"q_scale" in lib.pkv_last_error()


def test_cascade_rejects_bad_prefix(lib):
    cs = (ctypes.c_int64 * 4)(2048, 128, 16, 1)
    dummy = ctypes.create_string_buffer(64)
    ptr = ctypes.addressof(dummy)

    def call(P, max_kv=300, max_blocks=8):
        return lib.pkv_cascade_attention(
            ptr, ptr, 256, 64, ptr, ptr, cs, ptr, 1, ptr, ptr, ptr, max_kv,
            2, 2, 0.125, 0.0, ptr, max_blocks, max_blocks, P, 4, 2, 64, 16,
            8, 0, 1, None, 0, 1, None, None)
    assert call(40) == 1            # not a multiple of block_size
    assert call(0) == 1
    assert call(320) == 1           # longer than max_kv_len
    assert call(160, 300, 8) == 1   # longer than the table row
    assert lib.pkv_last_error()
    assert lib.pkv_cascade_attention_workspace_size(
        2, 2, 1, 300, 40, 4, 2, 64, 16, 8, 0, None) == \
        ctypes.c_size_t(-1).value


def test_merge_rejects_mixed_half_types(lib):
    st = lib.pkv_merge_attn_states(None, None, None, None, None, None, 4, 2,
                                   64, 0, 1, None)
    assert st == 2


def test_native_cascade_policy_matches_oracle(lib):
    import numpy as np
    from oracle import use_cascade_attention_ref
    from paged_kv_cache_318_gb300 import api
    rng = np.random.default_rng(0)
    for trial in range(400):
        n = int(rng.integers(1, 300))
        ql = np.ones(n, np.int32) if rng.random() < 0.7 else \
            rng.integers(1, 4, size=n).astype(np.int32)
        P = int(rng.choice([0, 100, 255, 256, 1024, 8192, 65536]))
        hkv = int(rng.choice([1, 2, 8]))
        hq = hkv * int(rng.choice([1, 2, 4, 8, 16]))
        flags = [bool(rng.random() < 0.15) for _ in range(3)]
        sms = int(rng.choice([132, 148, 152]))
        want = use_cascade_attention_ref(P, ql, hq, hkv, *flags, sms)
        got = api.use_cascade_attention(P, ql, hq, hkv, *flags, sms)
        assert got == want, (trial, P, n, hq, hkv, flags, sms)
    # DCP disables cascade
    assert not api.use_cascade_attention(8192, np.ones(256), 64, 8, False,
                                         False, False, 152, dcp_world_size=2)
