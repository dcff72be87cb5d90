"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerances (stated in the task's correctness bar): attention outputs within
max-abs 2e-2 (bf16) / 4e-3 (fp16) of the oracle, LSE within 1e-3, the cache
write bit-exact.
"""
import math

import numpy as np
import pytest
import torch

from oracle import add_sink_ref, merge_attn_states_ref, paged_attention_ref
from oracle.harness import (full_cache_bits, full_reference,
                            request_reference)
from paged_kv_cache_318_gb300 import api, workloads
from paged_kv_cache_318_gb300.batch import DeviceBatch

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f16": 4e-3}
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    from paged_kv_cache_318_gb300 import _build
    _build.build()
    api.load_library()


def nan_bits(dtype):
    """The 16-bit pattern torch uses for NaN in ``dtype`` (the cache's
    initial fill)."""
    t = torch.tensor(float("nan"), dtype=dtype)
    return int(t.view(torch.int16).item()) & 0xFFFF


def run_batch(wl, dev, cascade=False):
    b = DeviceBatch(wl, dev, cascade=cascade)
    b.write_context()
    res = b.step(return_lse=not cascade)
    torch.cuda.synchronize(dev)
    api.check_device_errors(dev)
    out, lse = res if isinstance(res, tuple) else (res, None)
    return b, out.float().cpu().numpy(), \
        None if lse is None else lse.cpu().numpy()


def assert_close(wl, out, lse, ref_out, ref_lse, what=""):
    assert np.isfinite(out).all(), what + ": non-finite output"
    err = np.abs(out - ref_out).max() if out.size else 0.0
    assert err <= TOL[wl.dtype], "%s out err %g" % (what, err)
    if lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin), what + ": lse -inf set"
        lerr = np.abs(lse[fin] - ref_lse[fin]).max() if fin.any() else 0.0
        assert lerr <= LSE_TOL, "%s lse err %g" % (what, lerr)


# ----------------------------------------------------------- small, full
def small_cases():
    return {
        "tiny_decode": lambda dt: workloads.tiny_decode(dtype=dt),
        "batched_decode_s": lambda dt: workloads.batched_decode(
            dtype=dt, batch=9, lo=20, hi=700, pool_blocks=600),
        "prefill_s": lambda dt: workloads.prefill_with_prefix(
            dtype=dt, batch=3, q_lo=17, q_hi=200, c_lo=0, c_hi=150),
        "mixed_s": lambda dt: workloads.mixed_gemma(
            dtype=dt, n_prefill=2, chunk=40, c_hi=300, n_decode=6, d_lo=50,
            d_hi=600),
        "long_decode_s": lambda dt: workloads.long_decode(
            dtype=dt, batch=2, ctx=3000, num_splits=16),
    }


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("name", list(small_cases()))
def test_small_workloads_full_outputs(cuda_device, name, dtype):
    wl = small_cases()[name](dtype)
    batch, out, lse = run_batch(wl, cuda_device)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out, lse, ref_out, ref_lse, name)
    bits = batch.kv_cache.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits, full_cache_bits(wl, nan_bits(wl.torch_dtype))), \
        name + ": cache bits"


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_cascade_small(cuda_device, dtype):
    wl = workloads.cascade_decode(dtype=dtype, batch=9, prefix=128,
                                  unique=70)
    _, out, _ = run_batch(wl, cuda_device, cascade=True)
    ref_out, _ = full_reference(wl)
    assert_close(wl, out, None, ref_out, None, "cascade")


CASCADE_OVERLAP_CASES = {
    "decode": lambda: workloads.cascade_decode(batch=9, prefix=128,
                                               unique=70),
    # suffix with decode-class and prefill-class requests: the suffix call
    # launches its decode kernel beside the prefix, then its prefill kernel
    "mixed_suffix": lambda: workloads.build_workload(
        "casc_mixed", 71, [1, 37, 1, 90, 2], [200, 177, 129, 260, 300], 16,
        4, 128, 64, shared_prefix_len=128),
    "bf16_256": lambda: workloads.build_workload(
        "casc_d256", 72, [1] * 20, list(range(300, 340, 2)), 16, 8, 256, 32,
        shared_prefix_len=256),
    "f16": lambda: workloads.build_workload(
        "casc_f16", 73, [1] * 40, list(range(700, 740)), 32, 8, 128, 16,
        shared_prefix_len=512, dtype="f16"),
}


@pytest.mark.parametrize("name", sorted(CASCADE_OVERLAP_CASES))
def test_cascade_overlap_equals_serial(cuda_device, name):
    """The suffix's decode kernel launched beside the prefix kernel (as its
    programmatic dependent) gives the same bits as the steps one after the
    other, and both match the oracle."""
    wl = CASCADE_OVERLAP_CASES[name]()
    b = DeviceBatch(wl, cuda_device, cascade=True)
    b.write_context()
    b.write_new()
    outs = []
    for ov in (True, False):
        api.cascade_attention(
            b.out, b.q, b.key_cache, b.value_cache, b.cu_seqlens_q,
            wl.max_seqlen_q, b.cu_prefix, b.prefix_lens, b.suffix_lens,
            wl.max_seqlen_k, wl.softmax_scale, None, (-1, -1), 0.0,
            b.block_table, wl.common_prefix_len, 0, overlap=ov)
        torch.cuda.synchronize()
        outs.append(b.out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    api.check_device_errors(cuda_device)
    ref_out, _ = full_reference(wl)
    assert_close(wl, outs[0].float().cpu().numpy(), None, ref_out, None,
                 "cascade overlap %s" % name)


# ------------------------------------------------------ feature matrix
FEATURES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, kwargs
    ([1, 1, 1], [1, 17, 300], 8, 8, 64, 16, dict()),
    ([1, 1], [100, 513], 8, 1, 128, 32, dict(num_splits=4)),
    ([1, 2, 3], [60, 61, 62], 16, 2, 128, 16, dict(num_splits=1)),
    ([5, 1, 70], [90, 33, 70], 4, 2, 64, 16, dict(causal=False)),
    ([33, 1], [200, 129], 8, 4, 128, 64, dict(window_size=(31, 0))),
    ([20, 3], [70, 100], 4, 4, 64, 16, dict(window_size=(10, 5),
                                            causal=False)),
    ([1, 40], [500, 90], 4, 2, 256, 32, dict(softcap=5.0)),
    ([3, 1, 19], [50, 77, 19], 8, 2, 128, 16,
     dict(alibi_slopes=[0.5, 0.25, 0.125, 0.0625, 0.03, 0.01, 0.3, 0.2])),
    ([0, 4, 0], [10, 9, 0], 4, 2, 64, 16, dict()),      # empty requests
    ([1] * 5, [4100] * 5, 16, 2, 256, 32, dict(window_size=(1000, 0),
                                                 softcap=50.0)),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("idx", range(len(FEATURES)))
def test_feature_matrix(cuda_device, idx, dtype):
    q_lens, seq_lens, Hq, Hkv, D, BS, kw = FEATURES[idx]
    wl = workloads.build_workload("feat%d" % idx, 500 + idx, q_lens,
                                  seq_lens, Hq, Hkv, D, BS, dtype=dtype, **kw)
    _, out, lse = run_batch(wl, cuda_device)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out, lse, ref_out, ref_lse, "feature %d" % idx)


PREFILL_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, kwargs  (all prefill-class)
    ([40], [200], 4, 2, 128, 16, dict()),
    ([70, 33], [300, 40], 8, 2, 64, 16, dict()),
    ([50, 130], [333, 130], 4, 2, 256, 32, dict()),
    ([60, 20], [90, 200], 4, 4, 128, 16, dict(causal=False)),
    ([90, 300], [700, 900], 8, 2, 128, 64, dict(window_size=(100, 0),
                                                softcap=20.0)),
    ([33], [100], 4, 2, 128, 16, dict(alibi_slopes=[0.1, 0.2, 0.05, 0.3])),
    ([64, 129], [64, 400], 8, 1, 128, 16, dict(dtype="f16")),
    ([257, 17], [1000, 517], 16, 8, 128, 16, dict()),
    ([20, 31], [2000, 31], 32, 8, 128, 16, dict(window_size=(7, 3))),
    # two-tile CTAs: B tile partly filled, windowed key ranges of A and B
    # that differ, non-causal, and an fp16 D = 64 case
    ([100, 70], [3000, 900], 32, 8, 128, 16, dict(window_size=(200, 0))),
    ([65, 300], [65, 700], 8, 2, 128, 32, dict(causal=False)),
    ([129, 200], [500, 1200], 16, 4, 64, 16, dict(dtype="f16")),
    # head size 256 (two softmax warps per row): window and soft-cap, ALiBi
    # in fp16, non-causal
    ([200, 77], [1300, 300], 8, 4, 256, 32, dict(window_size=(150, 0),
                                                 softcap=30.0)),
    ([129, 64], [500, 64], 4, 2, 256, 16,
     dict(alibi_slopes=[0.05, 0.1, 0.2, 0.4], dtype="f16")),
    ([100, 40], [260, 700], 8, 2, 256, 32, dict(causal=False)),
    # 240 short requests: 480 items dealt at run time, one item per request
    # and KV head
    ([9 + (i * 7) % 32 for i in range(240)],
     [9 + (i * 7) % 32 + (i * 37) % 150 for i in range(240)], 4, 2, 128, 16,
     dict()),
]


@pytest.mark.parametrize("kernel", ["tcgen05", "tcgen05_smem_p",
                                    "mma_sync"])
@pytest.mark.parametrize("idx", range(len(PREFILL_CASES)))
def test_prefill_kernels(cuda_device, idx, kernel):
    q_lens, seq_lens, Hq, Hkv, D, BS, kw = PREFILL_CASES[idx]
    wl = workloads.build_workload("pre%d" % idx, 900 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, **kw)
    which = {"tcgen05": api.PREFILL_TCGEN05,
             "tcgen05_smem_p": api.PREFILL_TCGEN05_SMEM_P,
             "mma_sync": api.PREFILL_MMA_SYNC}[kernel]
    api.set_prefill_kernel(which)
    try:
        _, out, lse = run_batch(wl, cuda_device)
    finally:
        api.set_prefill_kernel(api.PREFILL_TCGEN05)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out, lse, ref_out, ref_lse, "%s %d" % (kernel, idx))


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("view", ["hnd", "padded_blocks"])
def test_prefill_cache_views(cuda_device, view, D):
    """Prefill over other cache views: an HND physical cache seen through an
    NHD view and blocks with 8 padding rows each (block stride !=
    block_size x row stride).  At D = 256 the first takes the row-group
    boxes over the page x head axis and the second the per-column-block
    boxes; at D = 128 both take the persistent kernel's per-column-block
    boxes."""
    wl = workloads.build_workload("v%d" % D, 1234, [130, 60], [700, 260], 8,
                                  4, D, 32, window_size=(300, 0),
                                  softcap=30.0)
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    NB, BS, H, D = b.key_cache.shape
    dt, dev = b.key_cache.dtype, b.key_cache.device
    if view == "hnd":
        phys = torch.full((2, NB, H, BS, D), math.nan, dtype=dt, device=dev)
        kc, vc = phys.permute(0, 1, 3, 2, 4).unbind(0)
    else:
        phys = torch.full((2, NB, BS + 8, H, D), math.nan, dtype=dt,
                          device=dev)
        kc, vc = phys[:, :, :BS].unbind(0)
    kc.copy_(b.key_cache)
    vc.copy_(b.value_cache)
    b.key_cache, b.value_cache = kc, vc
    out, lse = b.attend(return_lse=True)
    torch.cuda.synchronize(dev)
    api.check_device_errors(dev)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ref_out,
                 ref_lse, view)


@pytest.mark.parametrize("BS", [16, 48])
@pytest.mark.parametrize("view", ["hnd", "padded_blocks"])
def test_decode_tma_cache_views(cuda_device, view, BS):
    """The TMA decode kernel over an HND physical cache seen through an NHD
    view (row-group boxes over the page x head axis) and over blocks with 8
    padding rows (per-column-block boxes), at block sizes 16 and 48."""
    wl = workloads.build_workload("dv%d" % BS, 1300 + BS, [1, 1, 2],
                                  [900, 333, 1500], 16, 4, 128, BS,
                                  window_size=(700, 0))
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    NB, BS_, H, D = b.key_cache.shape
    dt, dev = b.key_cache.dtype, b.key_cache.device
    if view == "hnd":
        phys = torch.full((2, NB, H, BS_, D), math.nan, dtype=dt, device=dev)
        kc, vc = phys.permute(0, 1, 3, 2, 4).unbind(0)
    else:
        phys = torch.full((2, NB, BS_ + 8, H, D), math.nan, dtype=dt,
                          device=dev)
        kc, vc = phys[:, :, :BS_].unbind(0)
    kc.copy_(b.key_cache)
    vc.copy_(b.value_cache)
    b.key_cache, b.value_cache = kc, vc
    api.set_decode_kernel(api.DECODE_TMA)
    try:
        out, lse = b.attend(return_lse=True)
        torch.cuda.synchronize(dev)
    finally:
        api.set_decode_kernel(api.DECODE_AUTO)
    api.check_device_errors(dev)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ref_out,
                 ref_lse, view)


DECODE_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, kwargs  (all decode-class)
    ([1, 1, 1, 1], [1, 15, 16, 17], 8, 2, 128, 16, dict()),
    ([1, 2, 1], [700, 1500, 90], 8, 4, 128, 16, dict(num_splits=5)),
    ([1] * 6, [64, 65, 127, 128, 129, 4000], 32, 8, 128, 64, dict()),
    ([1, 1], [3000, 2999], 16, 8, 256, 32, dict(window_size=(1000, 0),
                                               softcap=30.0)),
    ([1, 1, 4], [333, 1030, 77], 8, 2, 64, 16, dict(window_size=(100, 0),
                                                    num_splits=3)),
    ([2, 1], [500, 2049], 8, 8, 128, 48, dict()),        # block_size 48
    ([3, 1], [30, 260], 4, 1, 64, 128, dict(causal=False)),
    ([1, 1], [900, 901], 16, 2, 128, 16, dict(
        alibi_slopes=[0.01 * (i + 1) for i in range(16)], dtype="f16")),
    ([1], [131], 4, 4, 256, 16, dict(window_size=(20, 0))),
]


@pytest.mark.parametrize("kernel", ["persistent", "tma", "cp_async"])
@pytest.mark.parametrize("idx", range(len(DECODE_CASES)))
def test_decode_kernels(cuda_device, idx, kernel):
    """Every decode kernel over page sizes 16-128 (and a non-power-of-two
    48), window starts off the tile grid, split counts, poisoned page tails
    and every head size.  The persistent kernel serves calls that leave the
    split to the library, so its runs use num_splits = 0."""
    q_lens, seq_lens, Hq, Hkv, D, BS, kw = DECODE_CASES[idx]
    if kernel == "persistent":
        kw = dict(kw, num_splits=0)
    wl = workloads.build_workload("dec%d" % idx, 950 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, **kw)
    which = {"persistent": api.DECODE_PERSISTENT, "tma": api.DECODE_TMA,
             "cp_async": api.DECODE_CP_ASYNC}[kernel]
    api.set_decode_kernel(which)
    try:
        _, out, lse = run_batch(wl, cuda_device)
    finally:
        api.set_decode_kernel(api.DECODE_AUTO)
    ref_out, ref_lse = full_reference(wl)
    assert_close(wl, out, lse, ref_out, ref_lse, "%s %d" % (kernel, idx))


def test_rows_without_keys(cuda_device):
    """seqused_k below the query count: early rows see no key (out 0,
    lse -inf); a request with no keys at all likewise."""
    import dataclasses
    dev = cuda_device
    wl = workloads.build_workload("empty", 9, [3, 1, 2], [10, 5, 40], 4, 2,
                                  64, 16)
    b = DeviceBatch(wl, dev)
    b.write_context()
    b.write_new()
    short = np.array([2, 0, 40], dtype=np.int32)
    b.seqused_k.copy_(torch.from_numpy(short))
    out, lse = b.attend()
    torch.cuda.synchronize(dev)
    ref_out, ref_lse = full_reference(dataclasses.replace(wl,
                                                          seq_lens=short))
    assert_close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ref_out,
                 ref_lse, "rows without keys")
    assert np.isneginf(ref_lse[:, 0]).all()


def test_split_counts_agree(cuda_device):
    """Every explicit split count gives the same answer within tolerance."""
    wl = workloads.build_workload("splits", 77, [1] * 4, [3000, 64, 1, 2047],
                                  32, 8, 128, 16)
    ref_out, ref_lse = full_reference(wl)
    for s in (0, 1, 2, 3, 7, 16, 64):
        wl.num_splits = s
        _, out, lse = run_batch(wl, cuda_device)
        assert_close(wl, out, lse, ref_out, ref_lse, "splits=%d" % s)


# --------------------------------------------------------- cache write
def test_cache_write_hnd_view_and_padding(cuda_device):
    """HND physical cache seen through an NHD view; padded key rows past
    len(slot_mapping); -1 slots skipped; bit-exact."""
    dev = cuda_device
    NB, BS, H, D = 12, 16, 4, 128
    rng = np.random.default_rng(1)
    T = 40
    slots = rng.permutation(NB * BS)[:T].astype(np.int64)
    slots[[3, 17]] = -1
    key = torch.randn(T + 5, H, D, dtype=torch.bfloat16, device=dev)
    val = torch.randn(T + 5, H, D, dtype=torch.bfloat16, device=dev)
    hnd = torch.full((2, NB, H, BS, D), math.nan, dtype=torch.bfloat16,
                     device=dev)
    kc, vc = hnd.permute(0, 1, 3, 2, 4).unbind(0)
    api.reshape_and_cache_flash(key, val, kc, vc,
                                torch.from_numpy(slots).to(dev))
    torch.cuda.synchronize(dev)
    from oracle import reshape_and_cache_ref
    kb = key.cpu().view(torch.int16).numpy().view(np.uint16)
    vb = val.cpu().view(torch.int16).numpy().view(np.uint16)
    ek = np.full((NB, BS, H, D), nan_bits(torch.bfloat16), np.uint16)
    ev = ek.copy()
    reshape_and_cache_ref(kb, vb, ek, ev, slots)
    got = hnd.permute(0, 1, 3, 2, 4).cpu().contiguous().view(torch.int16) \
        .numpy().view(np.uint16)
    assert np.array_equal(got[0], ek) and np.array_equal(got[1], ev)


def test_cache_write_strided_key_rows(cuda_device):
    """key/value as slices of a fused qkv tensor (token stride > Hkv*D)."""
    dev = cuda_device
    NB, BS, H, D = 6, 16, 2, 64
    qkv = torch.randn(30, 4 * H * D, dtype=torch.float16, device=dev)
    key = qkv[:, H * D:2 * H * D].view(30, H, D)
    val = qkv[:, 2 * H * D:3 * H * D].view(30, H, D)
    cache = torch.zeros(2, NB, BS, H, D, dtype=torch.float16, device=dev)
    slots = torch.arange(30, dtype=torch.int64, device=dev) * 3
    api.reshape_and_cache_flash(key, val, cache[0], cache[1], slots)
    torch.cuda.synchronize(dev)
    flat = cache.view(2, NB * BS, H, D)
    assert torch.equal(flat[0, slots], key) and torch.equal(flat[1, slots],
                                                            val)


def test_out_of_range_indices_are_skipped_and_flagged(cuda_device):
    """A block id >= num_blocks and a slot past the cache: the kernels skip
    them (no access), the error word reports PKV_ERR_BAD_INDEX."""
    dev = cuda_device
    wl = workloads.build_workload("bad", 3, [1, 1], [20, 40], 4, 2, 64, 16)
    b = DeviceBatch(wl, dev)
    b.write_context()
    api.check_device_errors(dev)
    b.block_table[1, 1] = wl.num_blocks + 5
    b.step()
    with pytest.raises(api.PkvError) as ei:
        api.check_device_errors(dev)
    assert ei.value.status == api.PKV_ERR_BAD_INDEX
    assert torch.isfinite(b.out).all()
    bad = torch.tensor([wl.num_blocks * wl.block_size + 7], dtype=torch.int64,
                       device=dev)
    api.reshape_and_cache_flash(b.k_new[:1], b.v_new[:1], b.key_cache,
                                b.value_cache, bad)
    with pytest.raises(api.PkvError):
        api.check_device_errors(dev)
    api.check_device_errors(dev)   # cleared


# ---------------------------------------------------------------- merge
@pytest.mark.parametrize("dts", [("bf16", "bf16"), ("f16", "f16"),
                                 ("f32", "f32"), ("bf16", "f32")])
def test_merge_attn_states(cuda_device, dts):
    dev = cuda_device
    tmap = {"bf16": torch.bfloat16, "f16": torch.float16,
            "f32": torch.float32}
    out_dt, in_dt = tmap[dts[0]], tmap[dts[1]]
    T, H, D = 37, 6, 128
    g = torch.Generator(device="cpu").manual_seed(5)
    o1 = torch.randn(T, H, D, generator=g).to(in_dt)
    o2 = torch.randn(T, H, D, generator=g).to(in_dt)
    l1 = torch.randn(H, T, generator=g) * 3
    l2 = torch.randn(H, T, generator=g) * 3
    l1[0, :5] = -math.inf
    l2[1, 3:9] = -math.inf
    l1[2, 7] = l2[2, 7] = -math.inf
    out = torch.empty(T, H, D, dtype=out_dt, device=dev)
    lse = torch.empty(H, T, dtype=torch.float32, device=dev)
    api.merge_attn_states(out, o1.to(dev), l1.to(dev), o2.to(dev), l2.to(dev),
                          output_lse=lse)
    torch.cuda.synchronize(dev)
    ro, rl = merge_attn_states_ref(o1.double().numpy(), l1.double().numpy(),
                                   o2.double().numpy(), l2.double().numpy())
    tol = {torch.bfloat16: 2e-2, torch.float16: 4e-3, torch.float32: 1e-5}
    assert np.abs(out.float().cpu().numpy() - ro).max() <= tol[out_dt]
    got_l = lse.cpu().numpy()
    assert np.array_equal(np.isfinite(got_l), np.isfinite(rl))
    fin = np.isfinite(rl)
    assert np.abs(got_l[fin] - rl[fin]).max() <= LSE_TOL


def test_merge_non_finite_lse(cuda_device):
    """LSE +inf takes all the weight, -inf drops a side (even a NaN output),
    NaN propagates; the kernel against the oracle's reading."""
    dev = cuda_device
    inf, nan = math.inf, math.nan
    T, H, D = 6, 2, 64
    g = torch.Generator(device="cpu").manual_seed(11)
    o1 = torch.randn(T, H, D, generator=g)
    o2 = torch.randn(T, H, D, generator=g)
    o1[2] = nan                      # a side without keys may hold anything
    l1 = torch.tensor([[inf, 0.3, -inf, nan, inf, inf]] * H)
    l2 = torch.tensor([[2.0, inf, 1.5, 0.0, -inf, inf]] * H)
    out = torch.empty(T, H, D, dtype=torch.float32, device=dev)
    lse = torch.empty(H, T, dtype=torch.float32, device=dev)
    api.merge_attn_states(out, o1.to(dev), l1.to(dev), o2.to(dev),
                          l2.to(dev), output_lse=lse)
    torch.cuda.synchronize(dev)
    ro, rl = merge_attn_states_ref(o1.double().numpy(), l1.double().numpy(),
                                   o2.double().numpy(), l2.double().numpy())
    got, gl = out.cpu().numpy(), lse.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ro))
    fin = ~np.isnan(ro)
    assert np.abs(got[fin] - ro[fin]).max() <= 1e-5
    assert np.array_equal(np.isnan(gl), np.isnan(rl))
    assert np.array_equal(gl[~np.isnan(rl)], rl[~np.isnan(rl)]
                          .astype(np.float32))


# -------------------------------------------- full sizes, sampled outputs
def _sampled(wl, dev, reqs, last_rows=None, cascade=False):
    b, out, lse = run_batch(wl, dev, cascade=cascade)
    for r in reqs:
        t0, t1 = int(wl.cu_seqlens_q[r]), int(wl.cu_seqlens_q[r + 1])
        k = t1 - t0 if last_rows is None else min(last_rows, t1 - t0)
        ref_o, ref_l = request_reference(wl, r, last_rows=k)
        got_l = None if lse is None else lse[:, t1 - k:t1]
        assert_close(wl, out[t1 - k:t1], got_l, ref_o, ref_l,
                     "%s req %d" % (wl.name, r))
    # the cache rows of sampled slots are bit-exact copies of the inputs
    slots = wl.slot_mapping_new
    kbits = b.key_cache.view(torch.int16).reshape(
        -1, wl.num_kv_heads, wl.head_size)
    idx = torch.from_numpy(slots[:: max(1, len(slots) // 64)]).to(dev)
    src = torch.arange(0, len(slots), max(1, len(slots) // 64), device=dev)
    assert torch.equal(kbits[idx], b.k_new.view(torch.int16)[src])
    return b


def test_full_batched_decode_sampled(cuda_device):
    wl = workloads.batched_decode(device=cuda_device)
    _sampled(wl, cuda_device, [0, 17, 63])


def _row_slices(wl, b, out, lse, tile=128):
    """The first `tile` rows, a middle run of `tile` rows and the last 96
    rows of prefill-class request b against the oracle."""
    q = int(wl.q_lens[b])
    t0 = int(wl.cu_seqlens_q[b])
    mid = max(0, q // 2 - tile // 2)
    for i0, i1 in ((0, min(tile, q)), (mid, min(q, mid + tile)),
                   (max(0, q - 96), q)):
        ref_o, ref_l = request_reference(wl, b, row_range=(i0, i1))
        assert_close(wl, out[t0 + i0:t0 + i1], lse[:, t0 + i0:t0 + i1],
                     ref_o, ref_l, "%s req %d rows %d-%d" % (wl.name, b, i0,
                                                             i1))


def test_full_prefill_sampled(cuda_device):
    """Every request of the varlen prefill workload at full size: its first
    128 packed rows (prefix-only key tiles and the first causal diagonal),
    a middle tile and its last rows."""
    wl = workloads.prefill_with_prefix(device=cuda_device)
    _, out, lse = run_batch(wl, cuda_device)
    for b in range(wl.batch):
        _row_slices(wl, b, out, lse)


def test_full_mixed_sampled(cuda_device):
    wl = workloads.mixed_gemma(device=cuda_device)
    _, out, lse = run_batch(wl, cuda_device)
    for b in (0, 61, 123):                       # decode-class
        t0 = int(wl.cu_seqlens_q[b])
        ref_o, ref_l = request_reference(wl, b)
        assert_close(wl, out[t0:t0 + 1], lse[:, t0:t0 + 1], ref_o, ref_l,
                     "mixed req %d" % b)
    for b in range(124, wl.batch):               # the prefill chunks
        _row_slices(wl, b, out, lse)


def test_full_long_decode_sampled(cuda_device):
    wl = workloads.long_decode(device=cuda_device)
    _sampled(wl, cuda_device, [0, 7])


def test_full_cascade_sampled(cuda_device):
    wl = workloads.cascade_decode(device=cuda_device)
    _sampled(wl, cuda_device, [0, 100, 255], cascade=True)


# -------------------------------------------------------- attention sinks
SINK_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, num_splits, prefill kernel
    ([1, 1, 1], [500, 3000, 7], 16, 4, 128, 16, 0, "tcgen05"),
    ([1, 1], [5000, 64], 8, 2, 128, 64, 4, "tcgen05"),
    ([1, 2], [900, 33], 8, 4, 64, 16, 1, "tcgen05"),
    ([150, 60], [700, 60], 16, 4, 128, 16, 0, "tcgen05"),
    ([150, 60], [700, 60], 16, 4, 128, 16, 0, "mma_sync"),
    ([90, 1], [400, 2000], 8, 4, 256, 32, 0, "tcgen05"),
    ([2, 3], [1, 2], 4, 2, 64, 16, 0, "tcgen05"),     # rows without keys
]


@pytest.mark.parametrize("idx", range(len(SINK_CASES)))
def test_sinks(cuda_device, idx):
    import dataclasses
    from oracle.harness import _f64
    from oracle import reshape_and_cache_ref
    q_lens, seq_lens, Hq, Hkv, D, BS, splits, kern = SINK_CASES[idx]
    ok_lens = [max(L, q) for q, L in zip(q_lens, seq_lens)]
    wl = workloads.build_workload("sink%d" % idx, 700 + idx, q_lens, ok_lens,
                                  Hq, Hkv, D, BS, num_splits=splits)
    dev = cuda_device
    b = DeviceBatch(wl, dev)
    b.write_context()
    b.write_new()
    lens = np.array(seq_lens, np.int32)          # may be below q_len
    b.seqused_k.copy_(torch.from_numpy(lens))
    sinks = torch.linspace(-1.0, 2.0, Hq, dtype=torch.float32)
    api.set_prefill_kernel(api.PREFILL_TCGEN05 if kern == "tcgen05"
                           else api.PREFILL_MMA_SYNC)
    try:
        out, lse = api.flash_attn_varlen_func(
            b.q, b.key_cache, b.value_cache, wl.max_seqlen_q, b.cu_seqlens_q,
            wl.max_seqlen_k, seqused_k=b.seqused_k,
            softmax_scale=wl.softmax_scale, causal=True,
            block_table=b.block_table, return_softmax_lse=True,
            num_splits=splits, s_aux=sinks.to(dev))
        torch.cuda.synchronize()
    finally:
        api.set_prefill_kernel(api.PREFILL_TCGEN05)
    wl2 = dataclasses.replace(wl, seq_lens=lens)
    kc = np.full(wl.cache_shape()[1:], np.nan)
    vc = np.full(wl.cache_shape()[1:], np.nan)
    reshape_and_cache_ref(_f64(wl.k_ctx), _f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_f64(wl.k_new), _f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    ro, rl = paged_attention_ref(_f64(wl.q), kc, vc, wl2.cu_seqlens_q,
                                 lens, wl.block_table, wl.softmax_scale,
                                 sinks=sinks.double().numpy())
    assert_close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl,
                 "sinks %d" % idx)


def test_cascade_with_sinks(cuda_device):
    from oracle import cascade_ref
    wl = workloads.cascade_decode(batch=9, prefix=128, unique=70)
    dev = cuda_device
    b = DeviceBatch(wl, dev, cascade=True)
    b.write_context()
    b.write_new()
    sinks = torch.linspace(0.5, -0.5, wl.num_heads, dtype=torch.float32)
    api.cascade_attention(
        b.out, b.q, b.key_cache, b.value_cache, b.cu_seqlens_q,
        wl.max_seqlen_q, b.cu_prefix, b.prefix_lens, b.suffix_lens,
        wl.max_seqlen_k, wl.softmax_scale, None, (-1, -1), 0.0,
        b.block_table, wl.common_prefix_len, 0, s_aux=sinks.to(dev))
    torch.cuda.synchronize()
    from oracle.harness import _f64
    from oracle import reshape_and_cache_ref
    kc = np.full(wl.cache_shape()[1:], np.nan)
    vc = np.full(wl.cache_shape()[1:], np.nan)
    reshape_and_cache_ref(_f64(wl.k_ctx), _f64(wl.v_ctx), kc, vc,
                          wl.slot_mapping_ctx)
    reshape_and_cache_ref(_f64(wl.k_new), _f64(wl.v_new), kc, vc,
                          wl.slot_mapping_new)
    ro, _ = cascade_ref(_f64(wl.q), kc, vc, wl.cu_seqlens_q, wl.seq_lens,
                        wl.block_table, wl.common_prefix_len,
                        wl.softmax_scale, sinks=sinks.double().numpy())
    assert_close(wl, b.out.float().cpu().numpy(), None, ro, None,
                 "cascade sinks")


def test_many_requests_prefill_and_decode(cuda_device):
    """2100 requests, a mix of decode-class and prefill-class ones: more than
    the prefill kernel caches per CTA (its request metadata is then read from
    global memory), many work items per CTA, and a decode grid over
    thousands of (request, KV head) pairs."""
    rng = np.random.default_rng(77)
    n = 2100
    q_lens = np.where(rng.random(n) < 0.5, 1, rng.integers(5, 40, n))
    seq_lens = q_lens + rng.integers(0, 300, n)
    wl = workloads.build_workload("many", 78, q_lens.tolist(),
                                  seq_lens.tolist(), 8, 2, 128, 16,
                                  device=cuda_device)
    _sampled(wl, cuda_device, [0, 1, 777, 1500, 2098, 2099])


@pytest.mark.parametrize("name", ["prefill_with_prefix", "many"])
def test_prefill_item_order_leaves_bits_unchanged(cuda_device, name):
    """The persistent prefill kernel deals its work items at run time when
    the workspace holds its counter, and in a fixed order when it does not.
    Which SM computes an item must not change a bit of the output or LSE."""
    if name == "many":
        rng = np.random.default_rng(79)
        n = 700
        q_lens = np.where(rng.random(n) < 0.3, 1, rng.integers(5, 200, n))
        seq_lens = q_lens + rng.integers(0, 900, n)
        wl = workloads.build_workload("many_order", 80, q_lens.tolist(),
                                      seq_lens.tolist(), 16, 4, 128, 16,
                                      device=cuda_device)
    else:
        wl = workloads.prefill_with_prefix(device=cuda_device)
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    full = b.workspace
    assert full is not None and full.numel() >= 256
    out_dyn, lse_dyn = [t.clone() for t in b.attend()]
    # the same call with the counter's 256 bytes left out of the workspace
    b.workspace = full[:full.numel() - 256]
    out_fix, lse_fix = [t.clone() for t in b.attend()]
    b.workspace = full
    torch.cuda.synchronize()
    api.check_device_errors(cuda_device)
    assert torch.equal(out_dyn.view(torch.int16), out_fix.view(torch.int16))
    assert torch.equal(lse_dyn.view(torch.int32), lse_fix.view(torch.int32))
    # and both are right: the last rows of a few requests against the oracle
    o = out_dyn.float().cpu().numpy()
    lse = lse_dyn.cpu().numpy()
    for r in (0, wl.batch // 2, wl.batch - 1):
        t1 = int(wl.cu_seqlens_q[r + 1])
        k = min(8, t1 - int(wl.cu_seqlens_q[r]))
        ref_o, ref_l = request_reference(wl, r, last_rows=k)
        assert_close(wl, o[t1 - k:t1], lse[:, t1 - k:t1], ref_o, ref_l,
                     "%s req %d" % (name, r))


def _a256(x):
    return (x + 255) // 256 * 256


def _prefill_splits(wl, sms):
    """The key splits the library plans for the persistent prefill kernel
    (restated from its rule: an upper bound of the work items must leave half
    the SMs idle; one wave; >= 4 key tiles of 128 per split; <= 16)."""
    G = wl.num_heads // wl.num_kv_heads
    items = (-(-wl.num_tokens * G // 256) + wl.batch) * wl.num_kv_heads
    if wl.head_size > 128 or items * 2 > sms:
        return 1
    s = min(sms // items, int(wl.max_seqlen_k) // 512, 16)
    return s if s >= 2 else 1


SPLIT_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, kwargs
    ([300], [6000], 32, 8, 128, 16, dict()),                    # causal
    ([200, 40], [3000, 2500], 16, 4, 128, 32, dict(causal=False)),
    ([130, 17, 64], [4100, 1000, 64], 8, 2, 64, 16,
     dict(window_size=(700, 0))),                               # empty splits
    ([256], [8192], 64, 8, 128, 64, dict(causal=False)),        # cascade prefix
    ([100, 70], [3000, 900], 32, 8, 128, 16, dict(softcap=30.0, dtype="f16")),
]


@pytest.mark.parametrize("idx", range(len(SPLIT_CASES)))
def test_prefill_split_kv(cuda_device, idx):
    """Calls with few prefill work items split each item's keys across
    more SMs and fold the partials by LSE.  Split and unsplit runs (the
    workspace without the split partials) both match the oracle."""
    q_lens, seq_lens, Hq, Hkv, D, BS, kw = SPLIT_CASES[idx]
    wl = workloads.build_workload("split%d" % idx, 950 + idx, q_lens,
                                  seq_lens, Hq, Hkv, D, BS, **kw)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    S = _prefill_splits(wl, sms)
    assert S >= 2, "case %d does not exercise the split path" % idx
    ref_out, ref_lse = full_reference(wl)
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    full = b.workspace
    T = wl.num_tokens
    split_bytes = _a256(S * T * Hq * D * 4) + _a256(S * Hq * T * 4)
    assert full.numel() >= split_bytes + 256
    for ws in (full, full[:full.numel() - split_bytes]):
        b.workspace = ws
        out, lse = b.attend()
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        assert_close(wl, out.float().cpu().numpy(), lse.cpu().numpy(),
                     ref_out, ref_lse,
                     "split case %d ws %d" % (idx, ws.numel()))
    b.workspace = full


def test_prefill_split_kv_with_sinks(cuda_device):
    wl = workloads.build_workload("split_sink", 960, [120, 3], [5000, 900],
                                  16, 4, 128, 16)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    assert _prefill_splits(wl, sms) >= 2
    rng = np.random.default_rng(961)
    sinks = torch.from_numpy(rng.uniform(-1, 3, 16).astype(np.float32))
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    out, lse = api.flash_attn_varlen_func(
        b.q, b.key_cache, b.value_cache, wl.max_seqlen_q, b.cu_seqlens_q,
        wl.max_seqlen_k, seqused_k=b.seqused_k,
        softmax_scale=wl.softmax_scale, causal=True,
        block_table=b.block_table, return_softmax_lse=True,
        s_aux=sinks.to(cuda_device))
    torch.cuda.synchronize()
    api.check_device_errors(cuda_device)
    for r in range(wl.batch):
        t1 = int(wl.cu_seqlens_q[r + 1])
        k = min(16, t1 - int(wl.cu_seqlens_q[r]))
        ro, rl = request_reference(wl, r, last_rows=k)
        # the sink is one more logit of the softmax denominator
        ro, rl = add_sink_ref(ro, rl, sinks.double().numpy())
        assert_close(wl, out[t1 - k:t1].float().cpu().numpy(),
                     lse[:, t1 - k:t1].cpu().numpy(), ro, rl,
                     "sinks req %d" % r)


GRAPH_CASES = [
    # decode-class and prefill-class requests in one call (the prefill
    # kernel launched first, the decode kernel and the split combine as
    # programmatic dependents, the item counter zeroed by a memset)
    ("mixed", dict(q_lens=[1, 300, 1, 1, 90], seq_lens=[700, 900, 40, 3000,
                                                       400])),
    # the cascade (prefix kernel, suffix decode beside it, merge)
    ("cascade", None),
]


@pytest.mark.parametrize("idx", range(len(GRAPH_CASES)))
def test_call_captured_in_cuda_graph(cuda_device, idx):
    """The attention calls queue only stream-ordered work (kernels, with
    programmatic dependent launches, and memsets), so a call can be
    captured into a CUDA graph: replays equal the eager call bit for bit,
    and the eager call matches the oracle."""
    name, kw = GRAPH_CASES[idx]
    if name == "cascade":
        wl = workloads.build_workload("gcas", 77, [1] * 12, [800] * 12, 16, 4,
                                      128, 16, shared_prefix_len=512)
        cascade = True
    else:
        wl = workloads.build_workload("gmix", 78, kw["q_lens"],
                                      kw["seq_lens"], 32, 8, 128, 16)
        cascade = False
    b = DeviceBatch(wl, cuda_device, cascade=cascade)
    b.write_context()
    b.write_new()
    res = b.attend(return_lse=not cascade)
    torch.cuda.synchronize()
    api.check_device_errors(cuda_device)
    out_e, lse_e = res if isinstance(res, tuple) else (res, None)
    ref_out = out_e.clone()
    ref_lse = None if lse_e is None else lse_e.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res_g = b.attend(return_lse=not cascade)
    out_g, lse_g = res_g if isinstance(res_g, tuple) else (res_g, None)
    for _ in range(2):
        out_g.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        assert torch.equal(out_g.view(torch.int16), ref_out.view(torch.int16))
        if ref_lse is not None:
            assert torch.equal(lse_g.view(torch.int32),
                               ref_lse.view(torch.int32))
    o_ref, l_ref = full_reference(wl)
    assert_close(wl, ref_out.float().cpu().numpy(),
                 None if ref_lse is None else ref_lse.cpu().numpy(),
                 o_ref, l_ref, name)


def test_mixed_call_without_dependent_launches(cuda_device):
    """A call with decode-class and prefill-class requests launches the
    prefill kernel first and the decode kernel as its programmatic
    dependent; with the dependent launches off (``enable_pdl=False``) the
    decode kernel runs first, in plain stream order.  The two orders write
    the same bits, which match the oracle."""
    wl = workloads.build_workload("nopdl", 79, [1, 300, 1, 1, 90, 1],
                                  [700, 900, 40, 3000, 400, 2500], 32, 8,
                                  128, 16)
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    outs = []
    for pdl in (True, False):
        out, lse = api.flash_attn_varlen_func(
            b.q, b.key_cache, b.value_cache, wl.max_seqlen_q,
            b.cu_seqlens_q, wl.max_seqlen_k, seqused_k=b.seqused_k,
            softmax_scale=wl.softmax_scale, causal=True,
            block_table=b.block_table, return_softmax_lse=True,
            enable_pdl=pdl)
        torch.cuda.synchronize()
        api.check_device_errors(cuda_device)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))
    o_ref, l_ref = full_reference(wl)
    assert_close(wl, outs[0][0].float().cpu().numpy(), outs[0][1].cpu().numpy(),
                 o_ref, l_ref, "no-pdl")
