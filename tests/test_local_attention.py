"""Chunked local attention (virtual batches): oracle pins, the native
host transform against the oracle, and (GPU) attention over the virtual
batches against the direct masked definition."""
import json
import os

import numpy as np
import pytest

from oracle import paged_attention_ref
from oracle.local_attention import (local_attention_ref,
                                    local_virtual_batches_ref)
from _util import random_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "local_virtual_batches_example.json")


def golden_inputs():
    g = json.load(open(GOLDEN))
    cu = np.concatenate([[0], np.cumsum(g["q_seqlens"])]).astype(np.int32)
    return g, cu, np.array(g["k_seqlens"], np.int32), \
        np.array(g["block_table"], np.int32)


def test_oracle_reproduces_printed_example():
    g, cu, sk, bt = golden_inputs()
    sq_l, cu_l, sk_l, bt_l = local_virtual_batches_ref(
        g["attn_chunk_size"], cu, sk, bt, g["block_size"])
    assert sq_l.tolist() == g["seqlens_q_local"]
    assert sk_l.tolist() == g["seqlens_k_local"]
    assert bt_l.tolist() == g["block_table_local"]
    assert cu_l.tolist() == [0] + np.cumsum(g["seqlens_q_local"]).tolist()
    # intermediate quantities the page prints
    C = g["attn_chunk_size"]
    q = np.diff(cu)
    first = [min(C - (int(L) - int(n)) % C, int(n)) for L, n in zip(sk, q)]
    assert first == g["q_tokens_in_first_block"]
    counts = [(int(L) - 1) // C - (int(L) - int(n)) // C + 1
              for L, n in zip(sk, q)]
    assert counts == g["local_blocks"]
    # k start of each virtual request = first column * block_size, row-local
    starts = [int(np.where(np.asarray(g["block_table"][b]) == r[0])[0][0])
              * g["block_size"] for b, r in zip(
                  np.repeat(np.arange(3), g["local_blocks"]), bt_l)]
    assert starts == g["k_seqstarts_absolute"]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_318_gb300 import _build, api
    _build.build()
    return api


def test_native_transform_matches_oracle(lib):
    g, cu, sk, bt = golden_inputs()
    got = lib.make_local_attention_virtual_batches(
        g["attn_chunk_size"], cu, sk, bt, g["block_size"])
    ref = local_virtual_batches_ref(g["attn_chunk_size"], cu, sk, bt,
                                    g["block_size"])
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)
    rng = np.random.default_rng(0)
    for trial in range(50):
        B = int(rng.integers(1, 7))
        BS = int(rng.choice([16, 32]))
        C = BS * int(rng.integers(1, 5))
        q = rng.integers(1, 300, size=B)
        L = q + rng.integers(0, 500, size=B)
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        width = int(-(-L.max() // BS)) + int(rng.integers(0, 3))
        bt = rng.integers(0, 10000, size=(B, width)).astype(np.int32)
        got = lib.make_local_attention_virtual_batches(C, cu, L, bt, BS)
        ref = local_virtual_batches_ref(C, cu, L, bt, BS)
        for a, b in zip(got, ref):
            assert np.array_equal(a, b), trial


def test_native_transform_rejects_bad_arguments(lib):
    cu = np.array([0, 4], np.int32)
    with pytest.raises(ValueError):
        lib.make_local_attention_virtual_batches(6, cu, [10], [[0, 1]], 4)
    with pytest.raises(ValueError):     # query longer than the sequence
        lib.make_local_attention_virtual_batches(4, cu, [3], [[0, 1]], 2)


@pytest.mark.parametrize("C", [4, 8, 16])
def test_virtual_batches_equal_masked_local_attention(C):
    """Attention over the virtual requests == the direct chunk mask."""
    rng = np.random.default_rng(C)
    q_lens, k_lens = [5, 13, 1, 20], [9, 40, 7, 20]
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, q_lens, k_lens, 4,
                                                   2, 8, block_size=4)
    sq_l, cu_l, sk_l, bt_l = local_virtual_batches_ref(C, cu, su, table, 4)
    o1, l1 = paged_attention_ref(q, kc, vc, cu_l, sk_l, bt_l, 0.5,
                                 causal=True)
    o2, l2 = local_attention_ref(q, kc, vc, cu, su, table, 0.5, C)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_gpu_local_attention(cuda_device, lib, dtype):
    import torch
    from paged_kv_cache_318_gb300 import workloads
    from paged_kv_cache_318_gb300.batch import DeviceBatch
    from oracle.harness import _f64
    from oracle import reshape_and_cache_ref
    wl = workloads.build_workload("local", 41, [1, 300, 77, 1], [900, 1000,
                                                                77, 33],
                                  16, 4, 128, 16, dtype=dtype)
    C = 128
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    sq_l, cu_l, sk_l, bt_l = lib.make_local_attention_virtual_batches(
        C, wl.cu_seqlens_q, wl.seq_lens, wl.block_table, wl.block_size)
    dev = cuda_device
    out, lse = lib.flash_attn_varlen_func(
        b.q, b.key_cache, b.value_cache, int(sq_l.max()),
        torch.from_numpy(cu_l).to(dev), int(sk_l.max()),
        seqused_k=torch.from_numpy(sk_l).to(dev), softmax_scale=wl.softmax_scale,
        causal=True, block_table=torch.from_numpy(bt_l).to(dev),
        return_softmax_lse=True)
    torch.cuda.synchronize()
    kc = np.full(wl.cache_shape()[1:], np.nan)
    vc = np.full(wl.cache_shape()[1:], np.nan)
    reshape_and_cache_ref(_f64(wl.k_ctx), _f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_f64(wl.k_new), _f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    ro, rl = local_attention_ref(_f64(wl.q), kc, vc, wl.cu_seqlens_q,
                                 wl.seq_lens, wl.block_table,
                                 wl.softmax_scale, C)
    tol = 2e-2 if dtype == "bf16" else 4e-3
    assert np.abs(out.float().cpu().numpy() - ro).max() <= tol
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
