"""Pins for the oracle's LSE merge, split combine and cascade (CPU only)."""
import math

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle import (cascade_ref, lse_log2_to_ln, merge_attn_states_ref,
                    merge_many_ref, paged_attention_ref,
                    use_cascade_attention_ref)
from paged_kv_cache_318_gb300 import workloads
from _util import random_case


def test_merge_closed_forms():
    rng = np.random.default_rng(0)
    T, H, D = 3, 2, 4
    o1, o2 = rng.standard_normal((2, T, H, D))
    l1 = rng.standard_normal((H, T))
    # equal LSEs -> plain average, lse + ln 2
    o, l = merge_attn_states_ref(o1, l1, o2, l1)
    np.testing.assert_allclose(o, (o1 + o2) / 2, atol=1e-15)
    np.testing.assert_allclose(l, l1 + math.log(2), atol=1e-15)
    # one side empty (-inf) -> the other side unchanged
    ninf = np.full((H, T), -np.inf)
    o, l = merge_attn_states_ref(o1, l1, o2, ninf)
    np.testing.assert_allclose(o, o1, atol=0)
    np.testing.assert_allclose(l, l1, atol=0)
    o, l = merge_attn_states_ref(o1, ninf, o2, l1)
    np.testing.assert_allclose(o, o2, atol=0)
    # both empty -> zero, -inf
    o, l = merge_attn_states_ref(o1, ninf, o2, ninf)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # lse of the merge is logsumexp of the two lses
    l2 = rng.standard_normal((H, T)) * 3
    _, l = merge_attn_states_ref(o1, l1, o2, l2)
    np.testing.assert_allclose(l, logsumexp(np.stack([l1, l2]), axis=0),
                               atol=1e-14)


def test_merge_two_key_halves_equals_whole():
    """Attention over keys [0, L1) merged with [L1, L) equals all keys."""
    rng = np.random.default_rng(1)
    BS = 4
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [3, 2], [16, 12], 4,
                                                   2, 8, block_size=BS)
    whole = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=False)
    L1 = 8                                   # a block boundary
    first = paged_attention_ref(q, kc, vc, cu, np.minimum(su, L1), table,
                                0.5, causal=False)
    second = paged_attention_ref(q, kc, vc, cu, su - L1, table[:, L1 // BS:],
                                 0.5, causal=False)
    o, l = merge_attn_states_ref(*first, *second)
    np.testing.assert_allclose(o, whole[0], atol=1e-13)
    np.testing.assert_allclose(l, whole[1], atol=1e-13)


def test_merge_many_split_decode_equals_whole_any_order():
    rng = np.random.default_rng(2)
    BS = 4
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [1, 1], [23, 9], 8, 2,
                                                   8, block_size=BS)
    whole = paged_attention_ref(q, kc, vc, cu, su, table, 0.5)
    parts = []
    for start in range(0, 24, 8):           # 3 splits of 8 keys
        lens = np.clip(su - start, 0, 8)
        parts.append(paged_attention_ref(q, kc, vc, cu, lens,
                                         table[:, start // BS:], 0.5,
                                         causal=False))
    for order in ([0, 1, 2], [2, 0, 1]):
        o, l = merge_many_ref([parts[i][0] for i in order],
                              [parts[i][1] for i in order])
        np.testing.assert_allclose(o, whole[0], atol=1e-13)
        np.testing.assert_allclose(l, whole[1], atol=1e-13)


@pytest.mark.parametrize("q_lens", [[1] * 9, [1, 3, 1, 2, 1, 1, 4, 1, 2]])
def test_cascade_equals_flat(q_lens):
    n = len(q_lens)
    wl = workloads.build_workload("casc", 7, q_lens, [12 + 3 * i for i in
                                                      range(n)],
                                  4, 2, 8, 4, shared_prefix_len=8)
    kc = np.full(wl.cache_shape()[1:], np.nan)
    vc = np.full(wl.cache_shape()[1:], np.nan)
    from oracle import reshape_and_cache_ref
    f64 = lambda t: t.double().numpy()      # noqa: E731
    reshape_and_cache_ref(f64(wl.k_ctx), f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(f64(wl.k_new), f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    q = f64(wl.q)
    flat = paged_attention_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                               wl.block_table, 0.4)
    casc = cascade_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                       wl.block_table, 8, 0.4)
    np.testing.assert_allclose(casc[0], flat[0], atol=1e-13)
    np.testing.assert_allclose(casc[1], flat[1], atol=1e-13)
    # every request really shares the first two physical blocks
    assert (wl.block_table[:, :2] == wl.block_table[0, :2]).all()


def test_use_cascade_policy_hand_evaluated():
    """Wave model with 128x128 tiles, evaluated by hand for 152 SMs.

    256 decodes, P = 8192, Hq 64 / Hkv 8: cascade = ceil(64*2/152)*64 = 64,
    flash-decoding = ceil(256*8*1*64/152) = 863 -> cascade.
    8 decodes, same heads: cascade = ceil(64/152)*64 = 64, flash-decoding =
    ceil(8*8*64/152) = 27 -> no cascade.
    """
    ones = lambda n: np.ones(n, np.int64)     # noqa: E731
    assert use_cascade_attention_ref(8192, ones(256), 64, 8, False, False,
                                     False, 152) is True
    assert use_cascade_attention_ref(8192, ones(8), 64, 8, False, False,
                                     False, 152) is False
    # thresholds: prefix < 256, fewer than 8 requests, window / ALiBi
    assert not use_cascade_attention_ref(255, ones(256), 64, 8, False, False,
                                         False, 152)
    assert not use_cascade_attention_ref(8192, ones(7), 32, 32, False, False,
                                         False, 152)
    assert not use_cascade_attention_ref(8192, ones(64), 64, 8, True, False,
                                         False, 152)
    assert not use_cascade_attention_ref(8192, ones(64), 64, 8, False, True,
                                         False, 152)
    # no flash-decoding (MHA, or a prefill in the batch) -> cascade
    assert use_cascade_attention_ref(1024, ones(8), 32, 32, False, False,
                                     False, 152)
    q = ones(8)
    q[3] = 5
    assert use_cascade_attention_ref(1024, q, 32, 8, False, False, False, 152)


def test_log2_lse_conversion():
    x = np.random.default_rng(3).standard_normal(17) * 4
    lse2 = np.log2(np.sum(np.exp2(x * math.log2(math.e))))
    assert lse_log2_to_ln(lse2) == pytest.approx(logsumexp(x), abs=1e-12)


def test_cascade_with_sinks_on_prefix_equals_flat_with_sinks():
    """vLLM v1 cascade_attention passes s_aux to the prefix call only; its
    effect reaches the output through the merged LSE."""
    n = 9
    wl = workloads.build_workload("cs", 11, [1] * n, [12 + i for i in
                                                     range(n)], 4, 2, 8, 4,
                                  shared_prefix_len=8)
    from oracle import reshape_and_cache_ref
    kc = np.full(wl.cache_shape()[1:], np.nan)
    vc = np.full(wl.cache_shape()[1:], np.nan)
    f64 = lambda t: t.double().numpy()      # noqa: E731
    reshape_and_cache_ref(f64(wl.k_ctx), f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(f64(wl.k_new), f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    sinks = np.array([0.3, -0.2, 1.5, 0.0])
    q = f64(wl.q)
    flat = paged_attention_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                               wl.block_table, 0.4, sinks=sinks)
    casc = cascade_ref(q, kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                       wl.block_table, 8, 0.4, sinks=sinks)
    np.testing.assert_allclose(casc[0], flat[0], atol=1e-13)
    np.testing.assert_allclose(casc[1], flat[1], atol=1e-13)


def test_merge_non_finite_lse_edges():
    """-inf drops a side (its output is not read, even NaN); +inf takes all
    the weight (two +inf sides weigh the same) with merged lse +inf; NaN
    propagates.  Limits of the merge formula, evaluated by hand."""
    inf, nan = np.inf, np.nan
    o1 = np.array([[[1.0, 2.0]], [[1.0, 2.0]], [[nan, nan]], [[1.0, 2.0]],
                   [[1.0, 2.0]], [[3.0, 5.0]]])           # [T=6, H=1, D=2]
    o2 = np.array([[[5.0, 6.0]], [[5.0, 6.0]], [[5.0, 6.0]], [[5.0, 6.0]],
                   [[nan, 0.0]], [[7.0, 9.0]]])
    l1 = np.array([[inf, 0.3, -inf, nan, inf, inf]])       # [H=1, T=6]
    l2 = np.array([[2.0, inf, 1.5, 0.0, -inf, inf]])
    out, lse = merge_attn_states_ref(o1, l1, o2, l2)
    np.testing.assert_array_equal(out[0, 0], [1.0, 2.0])   # +inf left
    np.testing.assert_array_equal(out[1, 0], [5.0, 6.0])   # +inf right
    np.testing.assert_array_equal(out[2, 0], [5.0, 6.0])   # -inf, NaN rows
    assert np.isnan(out[3]).all() and np.isnan(lse[0, 3])  # NaN lse
    np.testing.assert_array_equal(out[4, 0], [1.0, 2.0])   # +inf vs -inf
    np.testing.assert_array_equal(out[5, 0], [5.0, 7.0])   # both +inf: mean
    assert lse[0, 0] == inf and lse[0, 1] == inf and lse[0, 4] == inf
    assert lse[0, 5] == inf and lse[0, 2] == 1.5
