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


@pytest.mark.parametrize("dkern", ["auto", "tma"])
@pytest.mark.parametrize("idx", range(len(CASES)))
def test_fp8_attention(cuda_device, idx, dkern):
    """E4M3 cache against the float64 oracle on code * scale values; the
    decode-class requests through the automatic choice and, at D = 128,
    through the one-CTA-per-unit TMA kernel (codes in 128-byte boxes)."""
    q_lens, seq_lens, Hq, Hkv, D, BS, splits, dtype, kern = CASES[idx]
    if dkern == "tma" and D != 128:
        pytest.skip("the TMA decode kernel reads E4M3 codes at D = 128")
    wl = workloads.build_workload("a8_%d" % idx, 40 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, dtype=dtype,
                                  num_splits=splits)
    dev = cuda_device
    ksc, vsc = 0.011, 0.017
    cache, kc, vc, ks, vs = fp8_batch(wl, dev, ksc, vsc)
    q = wl.q.to(dev)
    api.set_prefill_kernel(api.PREFILL_TCGEN05 if kern == "tcgen05"
                           else api.PREFILL_MMA_SYNC)
    api.set_decode_kernel(api.DECODE_TMA if dkern == "tma"
                          else api.DECODE_AUTO)
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
        api.set_decode_kernel(api.DECODE_AUTO)
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


# ------------------------------------------------------------ fp8 queries

@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_scaled_fp8_quant_bit_exact(cuda_device, dtype):
    """The query quantization against the oracle's codes: every element of
    a [tokens, heads * head_size] matrix, with saturating, zero and NaN
    inputs among them."""
    from oracle.fp8 import scaled_fp8_quant_ref
    dev = cuda_device
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(37, 8, 128, generator=g) *
         torch.tensor([0.01, 1.0, 30.0, 900.0]).repeat(2)[None, :, None])
    x = x.to(tdt)
    x[3, 2, :5] = 0.0
    x[4, 1, 7] = float("nan")
    scale = torch.tensor([0.37], dtype=torch.float32, device=dev)
    codes, s = api.scaled_fp8_quant(x.to(dev), scale)
    torch.cuda.synchronize()
    assert s is scale and codes.dtype == torch.float8_e4m3fn
    got = codes.view(torch.uint8).cpu().numpy()
    ref = scaled_fp8_quant_ref(f32(x), np.float32(0.37))
    nan = np.isnan(f32(x))
    assert np.array_equal(got[~nan], ref[~nan])
    assert ((got[nan] & 0x7F) == 0x7F).all()
    # strided rows in, strided rows out
    xs = torch.zeros(37, 8 * 128 + 64, dtype=tdt, device=dev)
    xs[:, :1024] = x.reshape(37, 1024).to(dev)
    out = torch.zeros(37, 1024 + 32, dtype=torch.uint8, device=dev)
    api.scaled_fp8_quant(xs[:, :1024], scale, out=out[:, :1024])
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.array_equal(o[:, :1024].reshape(37, 8, 128)[~nan], ref[~nan])
    assert not o[:, 1024:].any()


Q8_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, num_splits, dtype, decode kernel
    ([1, 1, 1, 1], [700, 3000, 9, 1], 32, 8, 128, 16, 0, "bf16", "auto"),
    ([1, 1, 1], [1200, 77, 4100], 32, 8, 128, 16, 0, "f16", "auto"),
    ([2, 1], [900, 3000], 16, 8, 256, 32, 0, "bf16", "auto"),
    ([1, 3, 1], [33, 2049, 4100], 16, 8, 256, 32, 0, "f16", "auto"),
    ([1, 1], [4000, 64], 16, 2, 128, 64, 4, "bf16", "auto"),
    ([1, 1, 1], [500, 1500, 40], 32, 8, 128, 16, 0, "bf16", "cp_async"),
    ([1, 1, 1, 1], [700, 3000, 9, 1], 32, 8, 128, 16, 0, "bf16", "tma"),
    ([1, 1, 1], [1200, 77, 4100], 32, 8, 128, 16, 0, "f16", "tma"),
    ([1, 1], [4000, 64], 16, 2, 128, 64, 4, "bf16", "tma"),
    ([1, 2], [500, 70], 8, 2, 64, 16, 0, "f16", "auto"),
    ([200, 1, 90], [900, 2000, 90], 32, 8, 128, 16, 0, "bf16", "auto"),
    ([70, 1], [600, 1200], 16, 8, 256, 32, 0, "bf16", "auto"),
]


@pytest.mark.parametrize("idx", range(len(Q8_CASES)))
def test_fp8_query_attention(cuda_device, idx):
    """E4M3 query codes (the library's scaled_fp8_quant, checked against
    the oracle's codes) over an E4M3 cache: the persistent decode kernel's
    E4M3 tensor-core path, and the 16-bit copy of the codes that the other
    kernels read, against the float64 oracle on code * scale values."""
    from oracle.fp8 import dequantize_ref, scaled_fp8_quant_ref
    q_lens, seq_lens, Hq, Hkv, D, BS, splits, dtype, kern = Q8_CASES[idx]
    wl = workloads.build_workload("q8_%d" % idx, 90 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, dtype=dtype,
                                  num_splits=splits)
    dev = cuda_device
    ksc, vsc, qsc = 0.011, 0.017, 0.023
    cache, kc, vc, ks, vs = fp8_batch(wl, dev, ksc, vsc)
    qs = torch.tensor([qsc], dtype=torch.float32, device=dev)
    q8, _ = api.scaled_fp8_quant(wl.q.to(dev), qs)
    qcodes = scaled_fp8_quant_ref(f32(wl.q), np.float32(qsc))
    assert np.array_equal(q8.view(torch.uint8).cpu().numpy(), qcodes)
    out = torch.empty(wl.q.shape, dtype=wl.q.dtype, device=dev)
    api.set_decode_kernel({"cp_async": api.DECODE_CP_ASYNC,
                           "tma": api.DECODE_TMA}.get(kern, api.DECODE_AUTO))
    try:
        _, lse = api.flash_attn_varlen_func(
            q8, kc, vc, wl.max_seqlen_q,
            torch.from_numpy(wl.cu_seqlens_q).to(dev), wl.max_seqlen_k,
            seqused_k=torch.from_numpy(wl.seq_lens).to(dev),
            softmax_scale=wl.softmax_scale, causal=True,
            block_table=torch.from_numpy(wl.block_table).to(dev),
            return_softmax_lse=True, num_splits=splits, k_descale=ks,
            v_descale=vs, q_descale=qs, out=out)
        torch.cuda.synchronize()
    finally:
        api.set_decode_kernel(api.DECODE_AUTO)
    api.check_device_errors(dev)
    kcodes, vcodes = oracle_codes(wl, ksc, vsc)
    ro, rl = paged_attention_ref(dequantize_ref(qcodes, qsc),
                                 dequantize_ref(kcodes, ksc),
                                 dequantize_ref(vcodes, vsc),
                                 wl.cu_seqlens_q, wl.seq_lens,
                                 wl.block_table, wl.softmax_scale)
    o = out.float().cpu().numpy()
    assert np.isfinite(o).all()
    assert np.abs(o - ro).max() <= TOL[dtype], np.abs(o - ro).max()
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


def test_fp8_query_rejected_without_fp8_cache(cuda_device):
    wl = workloads.build_workload("q8r", 5, [1], [40], 8, 2, 128, 16)
    dev = cuda_device
    qs = torch.tensor([0.02], dtype=torch.float32, device=dev)
    q8, _ = api.scaled_fp8_quant(wl.q.to(dev), qs)
    cache = torch.zeros(wl.cache_shape(), dtype=wl.q.dtype, device=dev)
    kc, vc = cache.unbind(0)
    with pytest.raises(NotImplementedError):
        api.flash_attn_varlen_func(
            q8, kc, vc, 1, torch.from_numpy(wl.cu_seqlens_q).to(dev), 40,
            seqused_k=torch.from_numpy(wl.seq_lens).to(dev),
            block_table=torch.from_numpy(wl.block_table).to(dev),
            q_descale=qs, out=torch.empty(wl.q.shape, dtype=wl.q.dtype,
                                          device=dev))


def test_dependent_launch_after_cache_write(cuda_device):
    """The persistent decode kernel launches as a programmatic dependent of
    the kernel before it.  Queued right behind cache writes that change the
    rows it reads (no synchronisation between), every call must read the
    written values: bit-equal to the same call in plain stream order after
    a device sync, and within tolerance of the oracle at the end."""
    wl = workloads.build_workload("pdl8", 61, [1] * 24,
                                  [int(x) for x in np.linspace(40, 6000, 24)],
                                  32, 8, 128, 16)
    dev = cuda_device
    ksc, vsc = 0.011, 0.017
    cache, kc, vc, ks, vs = fp8_batch(wl, dev, ksc, vsc)
    q = wl.q.to(dev)
    cu = torch.from_numpy(wl.cu_seqlens_q).to(dev)
    used = torch.from_numpy(wl.seq_lens).to(dev)
    bt = torch.from_numpy(wl.block_table).to(dev)
    slots = torch.from_numpy(wl.slot_mapping_new).to(dev)
    gen = torch.Generator().manual_seed(62)

    def call(enable_pdl):
        return api.flash_attn_varlen_func(
            q, kc, vc, 1, cu, wl.max_seqlen_k, seqused_k=used,
            softmax_scale=wl.softmax_scale, causal=True, block_table=bt,
            k_descale=ks, v_descale=vs, enable_pdl=enable_pdl)

    k_rows = v_rows = None
    for rep in range(4):
        # every request's last row changes, then the call reads it at once
        k_rows = (torch.randn(wl.k_new.shape, generator=gen) * 3).to(
            wl.k_new.dtype)
        v_rows = (torch.randn(wl.v_new.shape, generator=gen) * 3).to(
            wl.v_new.dtype)
        api.reshape_and_cache_flash(k_rows.to(dev), v_rows.to(dev), kc, vc,
                                    slots, "fp8", ks, vs)
        got = call(True)
        torch.cuda.synchronize()
        want = call(False)
        torch.cuda.synchronize()
        assert torch.equal(got, want), rep
    api.check_device_errors(dev)
    shape = wl.cache_shape()[1:]
    kcodes = np.zeros(shape, np.uint8)
    vcodes = np.zeros(shape, np.uint8)
    reshape_and_cache_fp8_ref(f32(wl.k_ctx), f32(wl.v_ctx), kcodes, vcodes,
                              wl.slot_mapping_ctx, ksc, vsc)
    reshape_and_cache_fp8_ref(f32(k_rows), f32(v_rows), kcodes, vcodes,
                              wl.slot_mapping_new, ksc, vsc)
    kref = e4m3_decode(kcodes) * np.float64(np.float32(ksc))
    vref = e4m3_decode(vcodes) * np.float64(np.float32(vsc))
    ro, _ = paged_attention_ref(f32(wl.q).astype(np.float64), kref, vref,
                                wl.cu_seqlens_q, wl.seq_lens, wl.block_table,
                                wl.softmax_scale)
    o = got.float().cpu().numpy()
    assert np.abs(o - ro).max() <= TOL["bf16"], np.abs(o - ro).max()
