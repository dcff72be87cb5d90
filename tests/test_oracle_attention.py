"""Pins for the oracle's paged attention (CPU only).

Brute force: torch's CPU scaled_dot_product_attention in float64 on the
contiguous (un-paged) rows, with masks built by tril/triu; closed forms;
invariants.  A plausible slip in the oracle (dropped scale, wrong GQA
mapping, top-left instead of bottom-right causal alignment, window
off-by-one, soft-cap before scale, ALiBi sign) fails one of these.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import paged_attention_ref
from _util import paged_from_contiguous, random_case


def sdpa_reference(q, ks, vs, cu, scale, causal, window=(-1, -1), G=1,
                   bias_fn=None):
    """Dense per-request attention with torch SDPA (float64) + logsumexp."""
    outs, lses = [], []
    for b in range(len(ks)):
        qb = torch.from_numpy(q[cu[b]:cu[b + 1]]).transpose(0, 1)  # [H,q,D]
        kb = torch.from_numpy(ks[b]).transpose(0, 1).repeat_interleave(G, 0)
        vb = torch.from_numpy(vs[b]).transpose(0, 1).repeat_interleave(G, 0)
        nq, nk = qb.shape[1], kb.shape[1]
        allowed = torch.ones(nq, nk, dtype=torch.bool)
        if causal:                      # bottom-right aligned
            allowed &= torch.ones(nq, nk, dtype=torch.bool).tril(nk - nq)
        if window[0] >= 0:
            allowed &= torch.ones(nq, nk, dtype=torch.bool).triu(
                nk - nq - window[0])
        if window[1] >= 0:
            allowed &= torch.ones(nq, nk, dtype=torch.bool).tril(
                nk - nq + window[1])
        logits = scale * (qb @ kb.transpose(1, 2))
        mask = torch.where(allowed, 0.0, -math.inf).to(torch.float64)
        if bias_fn is not None:
            mask = mask + bias_fn(nq, nk)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask,
                                           scale=scale)
        lse = torch.logsumexp(logits + mask, dim=-1)
        outs.append(o.transpose(0, 1).numpy())
        lses.append(lse.numpy())
    return np.concatenate(outs), np.concatenate(lses, axis=1)


CASES = [
    # q_lens, k_lens, Hq, Hkv, D, causal, window
    ([1, 1, 1], [5, 13, 1], 4, 2, 16, True, (-1, -1)),
    ([3, 7, 1], [3, 20, 9], 4, 1, 16, True, (-1, -1)),
    ([4, 6], [10, 6], 2, 2, 8, False, (-1, -1)),
    ([5, 2], [17, 12], 6, 3, 8, True, (3, 0)),
    ([5, 8], [17, 12], 4, 4, 8, False, (2, 1)),
    ([9], [9], 8, 2, 32, True, (0, 0)),
]


@pytest.mark.parametrize("case", CASES)
def test_matches_torch_sdpa(case):
    q_lens, k_lens, Hq, Hkv, D, causal, window = case
    rng = np.random.default_rng(hash(str(case)) % 2**32)
    q, ks, vs, kc, vc, table, cu, seqused = random_case(rng, q_lens, k_lens,
                                                        Hq, Hkv, D)
    scale = 0.37
    out, lse = paged_attention_ref(q, kc, vc, cu, seqused, table, scale,
                                   causal=causal, window_size=window)
    ro, rl = sdpa_reference(q, ks, vs, cu, scale, causal, window,
                            G=Hq // Hkv)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ro, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, rl, atol=1e-12, rtol=0)


def test_alibi_matches_sdpa_with_float_bias():
    rng = np.random.default_rng(11)
    q, ks, vs, kc, vc, table, cu, seqused = random_case(
        rng, [2, 3], [9, 14], 4, 2, 8)
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])

    def bias(nq, nk):
        p = torch.arange(nq)[:, None] + (nk - nq)
        j = torch.arange(nk)[None, :]
        return -torch.from_numpy(slopes)[:, None, None] * (p - j).abs()

    out, lse = paged_attention_ref(q, kc, vc, cu, seqused, table, 0.3,
                                   causal=True, alibi_slopes=slopes)
    ro, rl = sdpa_reference(q, ks, vs, cu, 0.3, True, G=2, bias_fn=bias)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def _identical_keys_case(q_len, k_len, D=4, BS=4, seed=0):
    rng = np.random.default_rng(seed)
    k_row = rng.standard_normal((1, 1, D))
    ks = [np.repeat(k_row, k_len, axis=0)]
    vs = [np.arange(k_len, dtype=np.float64)[:, None, None]
          * np.ones((1, 1, D))]
    q = rng.standard_normal((q_len, 1, D))
    kc, vc, table = paged_from_contiguous(ks, vs, BS, rng)
    cu = np.array([0, q_len], np.int32)
    return q, k_row, kc, vc, table, cu, np.array([k_len], np.int32)


@pytest.mark.parametrize("window", [(-1, -1), (2, 0), (0, 0), (5, 0)])
def test_identical_keys_mean_and_count(window):
    """Identical keys: out = mean of admissible V, lse = s + ln(count).

    With L = 10 keys and 3 queries, query i is at position 7 + i (end
    aligned), so causal admits keys 0..7+i; window (left, 0) keeps the last
    left+1 of those.
    """
    q, k_row, kc, vc, table, cu, seqused = _identical_keys_case(3, 10)
    scale = 0.5
    out, lse = paged_attention_ref(q, kc, vc, cu, seqused, table, scale,
                                   causal=True, window_size=window)
    for i in range(3):
        p = 7 + i
        lo = 0 if window[0] < 0 else max(0, p - window[0])
        keys = np.arange(lo, p + 1)
        s = scale * float(q[i, 0] @ k_row[0, 0])
        assert out[i, 0, 0] == pytest.approx(keys.mean(), abs=1e-12)
        assert lse[0, i] == pytest.approx(s + math.log(len(keys)), abs=1e-12)


def test_single_admissible_key_gives_that_row():
    rng = np.random.default_rng(4)
    q, ks, vs, kc, vc, table, cu, seqused = random_case(rng, [4], [11], 2, 1,
                                                        8)
    out, lse = paged_attention_ref(q, kc, vc, cu, seqused, table, 0.7,
                                   causal=True, window_size=(0, 0))
    for i in range(4):
        p = 7 + i
        for h in range(2):
            np.testing.assert_allclose(out[i, h], vs[0][p, 0], atol=1e-14)
            assert lse[h, i] == pytest.approx(
                0.7 * float(q[i, h] @ ks[0][p, 0]), abs=1e-12)


def test_empty_rows_are_zero_and_minus_inf():
    """A request with zero keys, and causal rows that see no key."""
    rng = np.random.default_rng(5)
    q, ks, vs, kc, vc, table, cu, seqused = random_case(rng, [2, 3], [0, 2],
                                                        2, 2, 8)
    out, lse = paged_attention_ref(q, kc, vc, cu, seqused, table, 1.0,
                                   causal=True)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:, :2]))
    # request 1: q=3 > L=2, query 0 sits at p = -1 -> nothing admissible
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[:, 2]))
    assert np.isfinite(lse[:, 3:]).all()


def test_rows_sum_to_one():
    """V = 1 everywhere -> out = 1 for every row that sees a key."""
    rng = np.random.default_rng(6)
    q, ks, vs, kc, vc, table, cu, seqused = random_case(rng, [3, 1], [8, 5],
                                                        4, 2, 8)
    ones = [np.ones_like(v) for v in vs]
    kc2, vc2, table2 = paged_from_contiguous(ks, ones, 4,
                                             np.random.default_rng(0))
    out, _ = paged_attention_ref(q, kc2, vc2, cu, seqused, table2, 0.9,
                                 causal=True, window_size=(3, 0))
    np.testing.assert_allclose(out, 1.0, atol=1e-13)


def test_softcap_saturation_scale_first():
    """Huge logits saturate at +cap: out = mean V and lse = cap + ln n.

    Applying the cap before the scale would give scale*cap + ln n instead.
    """
    rng = np.random.default_rng(7)
    D, L, cap, scale = 8, 6, 5.0, 0.25
    q = np.ones((1, 1, D)) * 100.0
    ks = [np.abs(rng.standard_normal((L, 1, D))) * 50 + 10]
    vs = [rng.standard_normal((L, 1, D))]
    kc, vc, table = paged_from_contiguous(ks, vs, 4, rng)
    cu, su = np.array([0, 1]), np.array([L])
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, scale,
                                   causal=True, softcap=cap)
    np.testing.assert_allclose(out[0, 0], vs[0][:, 0].mean(axis=0),
                               atol=1e-12)
    assert lse[0, 0] == pytest.approx(cap + math.log(L), abs=1e-12)
    # without the cap the largest logit dominates completely
    out2, _ = paged_attention_ref(q, kc, vc, cu, su, table, scale,
                                  causal=True)
    best = int(np.argmax(ks[0][:, 0] @ q[0, 0]))
    np.testing.assert_allclose(out2[0, 0], vs[0][best, 0], atol=1e-9)


def test_softcap_limits():
    """cap = 0 means no cap (vLLM v1 FlashAttentionImpl); cap -> inf too."""
    rng = np.random.default_rng(8)
    args = random_case(rng, [2, 1], [7, 9], 4, 2, 8)
    q, ks, vs, kc, vc, table, cu, su = args
    base = paged_attention_ref(q, kc, vc, cu, su, table, 0.4)
    for cap in (0.0, 1e30):
        o, l = paged_attention_ref(q, kc, vc, cu, su, table, 0.4, softcap=cap)
        np.testing.assert_allclose(o, base[0], atol=1e-13)
        np.testing.assert_allclose(l, base[1], atol=1e-13)
    o, _ = paged_attention_ref(q, kc, vc, cu, su, table, 0.4, softcap=1.0)
    assert np.abs(o - base[0]).max() > 1e-3


def test_alibi_geometric_closed_form():
    """Identical keys, V_j = j, slope a: weights r^(p-j), r = e^-a.

    E[p - j] over n = p+1 keys is r/(1-r) - n r^n / (1 - r^n), and
    lse = s + ln((1 - r^n)/(1 - r)); a positive slope favours near keys.
    """
    L, a = 12, 0.3
    q, k_row, kc, vc, table, cu, su = _identical_keys_case(1, L, seed=3)
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, 0.5,
                                   causal=True, alibi_slopes=np.array([a]))
    r, n, p = math.exp(-a), L, L - 1
    mean_d = r / (1 - r) - n * r ** n / (1 - r ** n)
    assert out[0, 0, 0] == pytest.approx(p - mean_d, abs=1e-12)
    s = 0.5 * float(q[0, 0] @ k_row[0, 0])
    assert lse[0, 0] == pytest.approx(
        s + math.log((1 - r ** n) / (1 - r)), abs=1e-12)
    o0, _ = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=True,
                                alibi_slopes=np.array([0.0]))
    assert o0[0, 0, 0] == pytest.approx((L - 1) / 2, abs=1e-12)


# ------------------------------------------------------------------ invariants

def test_block_permutation_invariance():
    rng = np.random.default_rng(9)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [3, 2], [13, 6], 4,
                                                   2, 8)
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, 0.5,
                                   window_size=(4, 0))
    perm = rng.permutation(kc.shape[0])          # new position of block i
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    out2, lse2 = paged_attention_ref(q, kc2, vc2, cu, su, perm[table], 0.5,
                                     window_size=(4, 0))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_paged_equals_contiguous():
    """Block size 4 vs one block holding the whole request."""
    rng = np.random.default_rng(10)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [2, 5], [9, 16], 4, 2,
                                                   8)
    big_kc, big_vc, big_table = paged_from_contiguous(ks, vs, 16, rng)
    a = paged_attention_ref(q, kc, vc, cu, su, table, 0.5)
    b = paged_attention_ref(q, big_kc, big_vc, cu, su, big_table, 0.5)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_gqa_equals_replicated_mha():
    rng = np.random.default_rng(12)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [3], [10], 8, 2, 8)
    ks4 = [np.repeat(k, 4, axis=1) for k in ks]
    vs4 = [np.repeat(v, 4, axis=1) for v in vs]
    kc4, vc4, t4 = paged_from_contiguous(ks4, vs4, 4, rng)
    a = paged_attention_ref(q, kc, vc, cu, su, table, 0.5)
    b = paged_attention_ref(q, kc4, vc4, cu, su, t4, 0.5)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_decode_causal_equals_noncausal_and_wide_window_is_none():
    rng = np.random.default_rng(13)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [1, 1], [7, 12], 4,
                                                   1, 8)
    a = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=True)
    b = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=False)
    c = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=True,
                            window_size=(12, 0))
    for x in (b, c):
        np.testing.assert_allclose(a[0], x[0], atol=1e-14)
        np.testing.assert_allclose(a[1], x[1], atol=1e-14)
    d = paged_attention_ref(q, kc, vc, cu, su, table, 0.5, causal=True,
                            window_size=(3, 0))
    assert np.abs(d[0] - a[0]).max() > 1e-3


def test_poison_never_reaches_output():
    """Unused blocks and padding rows are NaN; outputs stay finite."""
    rng = np.random.default_rng(14)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [2, 1, 3], [5, 17, 3],
                                                   4, 2, 8)
    assert np.isnan(kc).any()
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, 0.5)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ------------------------------------------------------------ attention sinks

def test_sink_closed_form_identical_keys():
    """n identical keys with logit s and a sink z: out = n e^s v / (n e^s +
    e^z), lse = ln(n e^s + e^z)."""
    q, k_row, kc, vc, table, cu, su = _identical_keys_case(1, 6)
    out0, lse0 = paged_attention_ref(q, kc, vc, cu, su, table, 0.5)
    z = 0.7
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, 0.5,
                                   sinks=np.array([z]))
    s = 0.5 * float(q[0, 0] @ k_row[0, 0])
    n = 6
    assert lse[0, 0] == pytest.approx(math.log(n * math.exp(s) + math.exp(z)),
                                      abs=1e-12)
    frac = n * math.exp(s) / (n * math.exp(s) + math.exp(z))
    np.testing.assert_allclose(out[0, 0], frac * out0[0, 0], atol=1e-13)


def test_sink_limits_and_empty_rows():
    rng = np.random.default_rng(21)
    q, ks, vs, kc, vc, table, cu, su = random_case(rng, [2, 3], [0, 9], 4, 2,
                                                   8)
    base = paged_attention_ref(q, kc, vc, cu, su, table, 0.4)
    off = paged_attention_ref(q, kc, vc, cu, su, table, 0.4,
                              sinks=np.full(4, -1e300))
    np.testing.assert_allclose(off[0], base[0], atol=1e-14)
    np.testing.assert_allclose(off[1][:, 2:], base[1][:, 2:], atol=1e-14)
    sinks = np.array([0.5, -1.0, 2.0, 0.0])
    out, lse = paged_attention_ref(q, kc, vc, cu, su, table, 0.4,
                                   sinks=sinks)
    # request 0 has no keys: out 0, lse = the sink
    assert np.all(out[:2] == 0)
    np.testing.assert_allclose(lse[:, :2], np.repeat(sinks[:, None], 2, 1))
    # a huge sink swallows the whole row
    big = paged_attention_ref(q, kc, vc, cu, su, table, 0.4,
                              sinks=np.full(4, 1e3))
    assert np.abs(big[0]).max() < 1e-300


# --------------------------------------------------------------- non-paged

NONPAGED_CASES = [
    # q_lens, k_lens, Hq, Hkv, D, causal, window
    ([4, 9, 1], [4, 9, 1], 4, 2, 8, False, (-1, -1)),   # encoder: cu_k = cu_q
    ([4, 9, 3], [4, 9, 3], 4, 4, 8, True, (-1, -1)),    # cache-free prefill
    ([2, 5], [11, 7], 6, 2, 16, True, (3, 1)),          # more keys than queries
    ([6, 1], [3, 0], 2, 1, 8, False, (-1, -1)),         # fewer / no keys
]


@pytest.mark.parametrize("case", NONPAGED_CASES)
def test_nonpaged_matches_torch_sdpa(case):
    from oracle import varlen_attention_ref
    q_lens, k_lens, Hq, Hkv, D, causal, window = case
    rng = np.random.default_rng(len(str(case)) + sum(k_lens))
    q = rng.standard_normal((sum(q_lens), Hq, D))
    ks = [rng.standard_normal((L, Hkv, D)) for L in k_lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in k_lens]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)])
    cu_k = np.concatenate([[0], np.cumsum(k_lens)])
    k = np.concatenate(ks) if sum(k_lens) else np.zeros((0, Hkv, D))
    v = np.concatenate(vs) if sum(k_lens) else np.zeros((0, Hkv, D))
    out, lse = varlen_attention_ref(q, k, v, cu_q, cu_k, 0.41, causal=causal,
                                    window_size=window)
    keep = [b for b in range(len(k_lens)) if k_lens[b] > 0]
    ro, rl = sdpa_reference(q[np.concatenate([np.arange(cu_q[b], cu_q[b + 1])
                                              for b in keep])],
                            [ks[b] for b in keep], [vs[b] for b in keep],
                            np.concatenate([[0], np.cumsum([q_lens[b]
                                                            for b in keep])]),
                            0.41, causal, window, G=Hq // Hkv)
    rows = np.concatenate([np.arange(cu_q[b], cu_q[b + 1]) for b in keep])
    np.testing.assert_allclose(out[rows], ro, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse[:, rows], rl, atol=1e-12, rtol=0)
    for b in range(len(k_lens)):               # requests without keys
        if k_lens[b] == 0:
            sl = slice(cu_q[b], cu_q[b + 1])
            assert (out[sl] == 0).all() and np.isneginf(lse[:, sl]).all()


def test_nonpaged_reads_only_its_own_rows_and_is_order_free():
    """Changing another request's rows changes nothing; without a causal
    mask or window, permuting a request's (key, value) rows changes
    nothing either (the softmax is a sum over keys)."""
    from oracle import varlen_attention_ref
    rng = np.random.default_rng(5)
    q = rng.standard_normal((7, 4, 8))
    k = rng.standard_normal((12, 2, 8))
    v = rng.standard_normal((12, 2, 8))
    cu_q, cu_k = np.array([0, 3, 7]), np.array([0, 5, 12])
    base = varlen_attention_ref(q, k, v, cu_q, cu_k, 0.3)
    k2, v2 = k.copy(), v.copy()
    k2[5:] = rng.standard_normal((7, 2, 8))
    v2[5:] = rng.standard_normal((7, 2, 8))
    other = varlen_attention_ref(q, k2, v2, cu_q, cu_k, 0.3)
    np.testing.assert_array_equal(other[0][:3], base[0][:3])
    np.testing.assert_array_equal(other[1][:, :3], base[1][:, :3])
    perm = np.concatenate([rng.permutation(5), 5 + rng.permutation(7)])
    shuffled = varlen_attention_ref(q, k[perm], v[perm], cu_q, cu_k, 0.3)
    np.testing.assert_allclose(shuffled[0], base[0], atol=1e-13)
    np.testing.assert_allclose(shuffled[1], base[1], atol=1e-13)
