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
