"""Pins for the oracle's cache scatter and block-table gather (CPU only)."""
import json
import os

import numpy as np

from oracle import gather_ref, reshape_and_cache_ref
from paged_kv_cache_318_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_cu_seqlens_golden():
    g = json.load(open(os.path.join(GOLDEN, "cu_seqlens_example.json")))
    assert workloads.cu_seqlens(g["lengths"]).tolist() == g["cu_seqlens"]


def test_block_table_golden():
    """Table row [0, 1, 2]: logical block j lives in physical block j."""
    g = json.load(open(os.path.join(GOLDEN, "block_table_example.json")))
    NB, BS, H, D = 5, 4, 1, 2
    cache = np.zeros((NB, BS, H, D))
    for blk in range(NB):
        for off in range(BS):
            cache[blk, off, 0] = (blk, off)
    rows = gather_ref(cache, np.array(g["block_table_row"]), 3 * BS)
    got_blocks = rows[::BS, 0, 0].astype(int).tolist()
    assert got_blocks == g["blocks_holding_tokens_in_order"]
    assert rows[:, 0, 1].astype(int).tolist() == list(range(BS)) * 3


def _random_problem(rng, NB=12, BS=4, H=3, D=8, T=20):
    key = rng.integers(0, 2**16, size=(T + 3, H, D), dtype=np.uint16)
    value = rng.integers(0, 2**16, size=(T + 3, H, D), dtype=np.uint16)
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    return key, value, slots


def test_scatter_matches_flat_slot_indexing():
    """Slot s is row s of the cache flattened over (block, offset)."""
    rng = np.random.default_rng(0)
    NB, BS, H, D = 12, 4, 3, 8
    key, value, slots = _random_problem(rng, NB, BS, H, D)
    kc = rng.integers(0, 2**16, size=(NB, BS, H, D), dtype=np.uint16)
    vc = kc.copy()
    kc_exp = kc.reshape(NB * BS, H, D).copy()
    vc_exp = vc.reshape(NB * BS, H, D).copy()
    for t, s in enumerate(slots):
        kc_exp[s] = key[t]
        vc_exp[s] = value[t]
    reshape_and_cache_ref(key, value, kc, vc, slots)
    assert np.array_equal(kc.reshape(NB * BS, H, D), kc_exp)
    assert np.array_equal(vc.reshape(NB * BS, H, D), vc_exp)


def test_scatter_skips_negative_and_ignores_extra_rows():
    rng = np.random.default_rng(1)
    NB, BS, H, D = 6, 4, 2, 4
    key, value, slots = _random_problem(rng, NB, BS, H, D, T=10)
    slots[[2, 5]] = -1
    kc = np.zeros((NB, BS, H, D), np.uint16)
    vc = np.zeros((NB, BS, H, D), np.uint16)
    reshape_and_cache_ref(key, value, kc, vc, slots)
    written = set(int(s) for s in slots if s >= 0)
    flat = kc.reshape(NB * BS, H, D)
    for s in range(NB * BS):
        if s not in written:
            assert not flat[s].any()
    # rows key[10:] (padding past len(slot_mapping)) never land anywhere
    for extra in key[10:]:
        assert not any(np.array_equal(extra, flat[s]) for s in written)


def test_scatter_into_hnd_view_equals_nhd():
    """A [NB, Hkv, BS, D] physical cache viewed as [NB, BS, Hkv, D]."""
    rng = np.random.default_rng(2)
    NB, BS, H, D = 8, 4, 3, 8
    key, value, slots = _random_problem(rng, NB, BS, H, D)
    kc = np.zeros((NB, BS, H, D), np.uint16)
    vc = np.zeros((NB, BS, H, D), np.uint16)
    reshape_and_cache_ref(key, value, kc, vc, slots)
    kh = np.zeros((NB, H, BS, D), np.uint16)
    vh = np.zeros((NB, H, BS, D), np.uint16)
    reshape_and_cache_ref(key, value, kh.transpose(0, 2, 1, 3),
                          vh.transpose(0, 2, 1, 3), slots)
    assert np.array_equal(kh.transpose(0, 2, 1, 3), kc)
    assert np.array_equal(vh.transpose(0, 2, 1, 3), vc)


def test_round_trip_through_workload_tables():
    """gather(scatter(rows)) == rows for every request of a workload."""
    wl = workloads.build_workload("rt", 5, [3, 1, 7], [9, 30, 7], 4, 2, 8, 4,
                                  pool_blocks=40)
    H, D = 2, 8
    n_ctx, T = len(wl.slot_mapping_ctx), wl.num_tokens
    rng = np.random.default_rng(3)
    k_ctx = rng.integers(0, 2**16, (n_ctx, H, D), dtype=np.uint16)
    k_new = rng.integers(0, 2**16, (T, H, D), dtype=np.uint16)
    kc = np.zeros((wl.num_blocks, 4, H, D), np.uint16)
    vc = np.zeros_like(kc)
    reshape_and_cache_ref(k_ctx, k_ctx, kc, vc, wl.slot_mapping_ctx)
    reshape_and_cache_ref(k_new, k_new, kc, vc, wl.slot_mapping_new)
    ctx_pos, new_pos = 0, 0
    for b in range(wl.batch):
        L, q = int(wl.seq_lens[b]), int(wl.q_lens[b])
        rows = gather_ref(kc, wl.block_table[b], L)
        assert np.array_equal(rows[:L - q], k_ctx[ctx_pos:ctx_pos + L - q])
        assert np.array_equal(rows[L - q:], k_new[new_pos:new_pos + q])
        ctx_pos += L - q
        new_pos += q
    # every used block is distinct, the pad block is unused
    used = [int(x) for b in range(wl.batch)
            for x in wl.block_table[b, :-(-int(wl.seq_lens[b]) // 4)]]
    assert len(used) == len(set(used))
    assert wl.pad_block not in used


def test_nan_payload_bits_copied_exactly():
    key = np.array([[[0x7FC1, 0xFF80, 0x0001, 0x8000]]], np.uint16)
    kc = np.zeros((1, 2, 1, 4), np.uint16)
    vc = np.zeros_like(kc)
    reshape_and_cache_ref(key, key, kc, vc, np.array([1]))
    assert kc[0, 1, 0].tolist() == [0x7FC1, 0xFF80, 0x0001, 0x8000]
