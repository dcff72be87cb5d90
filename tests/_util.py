"""Test helpers: build small paged caches from contiguous rows, compare."""
import numpy as np


def paged_from_contiguous(ks, vs, block_size, rng, spare_blocks=2,
                          poison=np.nan):
    """Lay per-request K/V rows [L_b, Hkv, D] out in a shuffled paged cache.

    Returns key_cache, value_cache [NB, BS, Hkv, D] float64, block_table
    [B, max_blocks] int32.  Unused blocks and padding rows hold ``poison``;
    table padding points at an unused (poisoned) block.
    """
    H, D = ks[0].shape[1], ks[0].shape[2]
    nblk = [-(-len(k) // block_size) for k in ks]
    NB = sum(nblk) + spare_blocks
    perm = rng.permutation(NB)
    kc = np.full((NB, block_size, H, D), poison)
    vc = np.full((NB, block_size, H, D), poison)
    maxb = max(max(nblk), 1)
    table = np.full((len(ks), maxb), perm[-1], dtype=np.int32)
    pos = 0
    for b, (k, v) in enumerate(zip(ks, vs)):
        for j in range(len(k)):
            blk = perm[pos + j // block_size]
            kc[blk, j % block_size] = k[j]
            vc[blk, j % block_size] = v[j]
        table[b, :nblk[b]] = perm[pos:pos + nblk[b]]
        pos += nblk[b]
    return kc, vc, table


def random_case(rng, q_lens, k_lens, Hq, Hkv, D, block_size=4):
    q_lens = np.asarray(q_lens)
    T = int(q_lens.sum())
    q = rng.standard_normal((T, Hq, D))
    ks = [rng.standard_normal((L, Hkv, D)) for L in k_lens]
    vs = [rng.standard_normal((L, Hkv, D)) for L in k_lens]
    kc, vc, table = paged_from_contiguous(ks, vs, block_size, rng)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return q, ks, vs, kc, vc, table, cu, np.asarray(k_lens, np.int32)
