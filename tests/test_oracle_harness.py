"""Pins of the oracle's per-request helpers (oracle/harness.py).

``request_rows`` / ``request_reference`` rebuild one request's K/V rows from
the generator's storage order and run the oracle on that request alone; the
full-size sampled parity tests take their expected values from them.
``full_reference`` instead scatters every row through the workload's own
slot mapping into the workload's own block tables and runs the oracle on the
whole batch.  The two routes share only the oracle's attention function, so
a slip in the row reconstruction (wrong context offsets, shared-prefix rows
taken twice or from the wrong request, new rows out of place) shows up as a
mismatch here.
"""
import numpy as np
import pytest

from oracle.harness import full_reference, request_reference, request_rows
from paged_kv_cache_318_gb300 import workloads


def _small_cascade():
    # shared 128-token prefix (two 64-row blocks) + 40 own tokens each
    return workloads.cascade_decode(batch=9, prefix=128, unique=40)


def _small_mixed():
    return workloads.mixed_gemma(n_prefill=2, chunk=24, c_hi=90, n_decode=5,
                                 d_lo=40, d_hi=130)


def _small_prefill():
    return workloads.prefill_with_prefix(batch=3, q_lo=20, q_hi=50, c_lo=0,
                                         c_hi=40)


def _windowed():
    # window, soft-cap and ALiBi all active, ragged blocks
    return workloads.build_workload(
        "windowed", 77, [1, 9, 3, 17], [30, 41, 3, 17], 4, 2, 64, 16,
        window_size=(11, 0), softcap=5.0,
        alibi_slopes=[0.5, 0.25, 0.125, 0.0625])


CASES = {"cascade": _small_cascade, "mixed": _small_mixed,
         "prefill": _small_prefill, "windowed": _windowed}


@pytest.mark.parametrize("name", sorted(CASES))
def test_request_reference_matches_full_reference(name):
    wl = CASES[name]()
    out, lse = full_reference(wl)
    for b in range(wl.batch):
        t0, t1 = int(wl.cu_seqlens_q[b]), int(wl.cu_seqlens_q[b + 1])
        o_b, l_b = request_reference(wl, b)
        assert o_b.shape == (t1 - t0, wl.num_heads, wl.head_size)
        np.testing.assert_allclose(o_b, out[t0:t1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_b, lse[:, t0:t1], rtol=0, atol=1e-12)
        # the last k queries alone
        k = max(1, (t1 - t0) // 2)
        o_k, l_k = request_reference(wl, b, last_rows=k)
        np.testing.assert_allclose(o_k, out[t1 - k:t1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l_k, lse[:, t1 - k:t1], rtol=0,
                                   atol=1e-12)


@pytest.mark.parametrize("name", sorted(CASES))
def test_request_rows_match_cache_through_table(name):
    """Row j of request b is what the workload's block table and slot
    mapping put at key position j (the gather of the written cache)."""
    from oracle.harness import _f64
    from oracle.paged_attention import reshape_and_cache_ref
    wl = CASES[name]()
    shape = wl.cache_shape()
    kc = np.full(shape[1:], np.nan)
    vc = np.full(shape[1:], np.nan)
    reshape_and_cache_ref(_f64(wl.k_ctx), _f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_f64(wl.k_new), _f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    BS = wl.block_size
    for b in range(wl.batch):
        k, v = request_rows(wl, b)
        L = int(wl.seq_lens[b])
        j = np.arange(L)
        blk = wl.block_table[b, j // BS]
        assert np.array_equal(k, kc[blk, j % BS])
        assert np.array_equal(v, vc[blk, j % BS])
        assert not np.isnan(k).any()


def test_shared_prefix_rows_are_request_zeros():
    wl = _small_cascade()
    k0, v0 = request_rows(wl, 0)
    P = wl.common_prefix_len
    for b in range(1, wl.batch):
        kb, vb = request_rows(wl, b)
        assert np.array_equal(kb[:P], k0[:P])
        assert np.array_equal(vb[:P], v0[:P])
        # own rows differ from request 0's
        assert not np.array_equal(kb[P:], k0[P:])


@pytest.mark.parametrize("name", ["mixed", "prefill", "windowed"])
def test_request_reference_row_ranges(name):
    """Queries i0 .. i1-1 of a causal request (first rows, a middle run)
    against the whole-batch oracle."""
    wl = CASES[name]()
    out, lse = full_reference(wl)
    for b in range(wl.batch):
        q = int(wl.q_lens[b])
        t0 = int(wl.cu_seqlens_q[b])
        for i0, i1 in ((0, min(3, q)), (q // 3, max(q // 3 + 1, 2 * q // 3)),
                       (0, q)):
            if i1 <= i0:
                continue
            o, l = request_reference(wl, b, row_range=(i0, i1))
            np.testing.assert_allclose(o, out[t0 + i0:t0 + i1], rtol=0,
                                       atol=1e-12)
            np.testing.assert_allclose(l, lse[:, t0 + i0:t0 + i1], rtol=0,
                                       atol=1e-12)
