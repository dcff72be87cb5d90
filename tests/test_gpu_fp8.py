"""FP8 (E4M3) KV cache on the GPU: the quantizing cache write is bit-exact
against the oracle's codes, and attention over an fp8 cache matches the
float64 oracle on the dequantized values (code * scale) within the bf16 /
fp16 output tolerances."""
import numpy as np
import pytest
import torch

from oracle import paged_attention_ref
from oracle.fp8 import e4m3_decode, reshape_and_cache_fp8_ref
from paged_kv_cache_318_gb300 import api, workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f16": 4e-3}


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    from paged_kv_cache_318_gb300 import _build
    _build.build()
    api.load_library()


def f32(t):
    return t.detach().float().cpu().numpy()


def fp8_batch(wl, dev, k_scale, v_scale):
    """Device fp8 cache filled through the library's cache write."""
    cache = torch.zeros(wl.cache_shape(), dtype=torch.uint8, device=dev)
    kc, vc = cache.unbind(0)
    ks = torch.tensor([k_scale], dtype=torch.float32, device=dev)
    vs = torch.tensor([v_scale], dtype=torch.float32, device=dev)
    for rows_k, rows_v, slots in ((wl.k_ctx, wl.v_ctx, wl.slot_mapping_ctx),
                                  (wl.k_new, wl.v_new, wl.slot_mapping_new)):
        if len(slots):
            api.reshape_and_cache_flash(
                rows_k.to(dev), rows_v.to(dev), kc, vc,
                torch.from_numpy(slots).to(dev), "fp8", ks, vs)
    torch.cuda.synchronize()
    return cache, kc, vc, ks, vs


def oracle_codes(wl, k_scale, v_scale):
    shape = wl.cache_shape()[1:]
    kc = np.zeros(shape, np.uint8)
    vc = np.zeros(shape, np.uint8)
    reshape_and_cache_fp8_ref(f32(wl.k_ctx), f32(wl.v_ctx), kc, vc,
                              wl.slot_mapping_ctx, k_scale, v_scale)
    reshape_and_cache_fp8_ref(f32(wl.k_new), f32(wl.v_new), kc, vc,
                              wl.slot_mapping_new, k_scale, v_scale)
    return kc, vc


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fp8_cache_write_bit_exact(cuda_device, dtype):
    wl = workloads.build_workload("w8", 3, [1, 5, 40], [300, 77, 40], 8, 2,
                                  128, 16, dtype=dtype)
    cache, *_ = fp8_batch(wl, cuda_device, 0.013, 0.021)
    kc, vc = oracle_codes(wl, 0.013, 0.021)
    got = cache.cpu().numpy()
    assert np.array_equal(got[0], kc) and np.array_equal(got[1], vc)


CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, num_splits, dtype, prefill kernel
    ([1, 1, 1], [700, 3000, 9], 32, 8, 128, 16, 0, "bf16", "tcgen05"),
    ([1, 1], [4000, 64], 16, 2, 128, 64, 4, "bf16", "tcgen05"),
    ([1, 2], [500, 70], 8, 2, 64, 16, 1, "f16", "tcgen05"),
    ([200, 1, 90], [900, 2000, 90], 32, 8, 128, 16, 0, "bf16", "tcgen05"),
    ([200, 90], [900, 90], 32, 8, 128, 16, 0, "bf16", "mma_sync"),
    ([70, 1], [600, 1200], 16, 8, 256, 32, 0, "bf16", "tcgen05"),
    ([130, 1], [400, 800], 16, 4, 64, 16, 0, "f16", "tcgen05"),
    ([1, 3, 1], [33, 2049, 4100], 16, 8, 256, 32, 3, "f16", "tcgen05"),
    ([1, 1], [1, 129], 8, 4, 128, 128, 0, "bf16", "tcgen05"),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_fp8_attention(cuda_device, idx):
    q_lens, seq_lens, Hq, Hkv, D, BS, splits, dtype, kern = CASES[idx]
    wl = workloads.build_workload("a8_%d" % idx, 40 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, dtype=dtype,
                                  num_splits=splits)
    dev = cuda_device
    ksc, vsc = 0.011, 0.017
    cache, kc, vc, ks, vs = fp8_batch(wl, dev, ksc, vsc)
    q = wl.q.to(dev)
    api.set_prefill_kernel(api.PREFILL_TCGEN05 if kern == "tcgen05"
                           else api.PREFILL_MMA_SYNC)
    try:
        out, lse = api.flash_attn_varlen_func(
            q, kc, vc, wl.max_seqlen_q,
            torch.from_numpy(wl.cu_seqlens_q).to(dev), wl.max_seqlen_k,
            seqused_k=torch.from_numpy(wl.seq_lens).to(dev),
            softmax_scale=wl.softmax_scale, causal=True,
            block_table=torch.from_numpy(wl.block_table).to(dev),
            return_softmax_lse=True, num_splits=splits, k_descale=ks,
            v_descale=vs)
        torch.cuda.synchronize()
    finally:
        api.set_prefill_kernel(api.PREFILL_TCGEN05)
    api.check_device_errors(dev)
    kcodes, vcodes = oracle_codes(wl, ksc, vsc)
    kref = e4m3_decode(kcodes) * np.float64(np.float32(ksc))
    vref = e4m3_decode(vcodes) * np.float64(np.float32(vsc))
    ro, rl = paged_attention_ref(f32(wl.q).astype(np.float64), kref, vref,
                                 wl.cu_seqlens_q, wl.seq_lens,
                                 wl.block_table, wl.softmax_scale)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    assert np.abs(o - ro).max() <= TOL[dtype], np.abs(o - ro).max()
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3
