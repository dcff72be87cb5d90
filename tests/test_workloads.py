"""The seeded workloads the bench and the tests run: their sizes, length
ranges and tables, and the bench's algorithmic byte and FLOP counts for
them (geometry only, no values drawn)."""
import numpy as np

import bench
from paged_kv_cache_318_gb300 import workloads


def _tables_ok(wl):
    """Every request's blocks are distinct from every other request's,
    except a shared prefix; the pad block is in no request's range."""
    BS, P = wl.block_size, wl.common_prefix_len
    seen = set()
    for b in range(wl.batch):
        nb = -(-int(wl.seq_lens[b]) // BS)
        row = [int(x) for x in wl.block_table[b, :nb]]
        own = row[P // BS:] if (P and b > 0) else row
        assert wl.pad_block not in row
        assert 0 <= min(row) and max(row) < wl.num_blocks
        assert not (set(own) & seen), b
        seen.update(own)


def test_batched_decode_recipe():
    wl = workloads.batched_decode(values=False)
    assert wl.batch == 64 and np.all(wl.q_lens == 1)
    assert (wl.num_heads, wl.num_kv_heads, wl.head_size, wl.block_size) == \
        (32, 8, 128, 16)
    assert wl.num_blocks == 20000
    assert 512 <= wl.seq_lens.min() and wl.seq_lens.max() <= 4096
    assert int(wl.seq_lens.sum()) == 158295
    acct = bench.decode_bytes(wl)
    assert acct["kv"] == 158295 * 2 * 8 * 128 * 2 == 648376320
    assert acct["attention"] == 649465108
    _tables_ok(wl)


def test_prefill_with_prefix_recipe():
    wl = workloads.prefill_with_prefix(values=False)
    assert wl.batch == 8 and wl.num_tokens == 11207
    ctx = wl.seq_lens - wl.q_lens
    assert 256 <= wl.q_lens.min() and wl.q_lens.max() <= 2048
    assert 0 <= ctx.min() and ctx.max() <= 1024
    assert bench.prefill_flops(wl) == 227367075840.0
    # the causal pair count, in closed form per request
    pairs = sum(int(q) * int(c) + int(q) * (int(q) + 1) // 2
                for q, c in zip(wl.q_lens, ctx))
    assert bench.prefill_flops(wl) == 4.0 * 128 * 32 * pairs
    _tables_ok(wl)


def test_other_recipes():
    ld = workloads.long_decode(values=False)
    assert ld.batch == 8 and np.all(ld.seq_lens == 131072)
    assert (ld.num_heads, ld.num_kv_heads, ld.block_size, ld.num_splits) == \
        (64, 8, 64, 16)
    _tables_ok(ld)
    cd = workloads.cascade_decode(values=False)
    assert cd.batch == 256 and np.all(cd.seq_lens == 8192 + 512)
    assert cd.common_prefix_len == 8192
    assert np.all(cd.block_table[:, :128] == cd.block_table[0, :128])
    _tables_ok(cd)
    mg = workloads.mixed_gemma(values=False)
    assert mg.batch == 128
    assert np.all(mg.q_lens[:124] == 1) and np.all(mg.q_lens[124:] == 512)
    assert (mg.num_heads, mg.num_kv_heads, mg.head_size, mg.block_size) == \
        (16, 8, 256, 32)
    assert mg.window_size == (4095, 0) and mg.softcap == 50.0
    _tables_ok(mg)
