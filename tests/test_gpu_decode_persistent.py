"""The persistent decode kernel against the float64 oracle.

Every CTA of this kernel streams an equal share of the batch's key tiles, so
one request's keys may be cut between several CTAs; the pieces are merged by
LSE in a second launch.  These cases aim at that bookkeeping: units cut many
times (one very long request), units of every length next to each other,
prefill-class requests between decode-class ones (skipped by the walk),
requests with no keys, sinks added once after the merge, a workspace without
the kernel's scratch (the fallback kernels), and E4M3 caches with queries
far from unit scale (the per-unit power-of-two scaling) and NaN codes in
unused rows.
"""
import numpy as np
import pytest
import torch

from oracle import add_sink_ref, paged_attention_ref
from oracle.fp8 import e4m3_decode, reshape_and_cache_fp8_ref
from oracle.harness import full_reference, request_reference
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
    api.set_decode_kernel(api.DECODE_PERSISTENT)
    yield
    api.set_decode_kernel(api.DECODE_AUTO)


def _close(wl, out, lse, ref_out, ref_lse, what):
    assert np.isfinite(out).all(), what + ": non-finite output"
    err = np.abs(out - ref_out).max() if out.size else 0.0
    assert err <= TOL[wl.dtype], "%s out err %g" % (what, err)
    if lse is not None:
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lse), fin), what + ": -inf rows"
        if fin.any():
            lerr = np.abs(lse[fin] - ref_lse[fin]).max()
            assert lerr <= LSE_TOL, "%s lse err %g" % (what, lerr)


def _run(wl, dev, sinks=None, workspace=None):
    b = DeviceBatch(wl, dev)
    b.write_context()
    b.write_new()
    if workspace is not None:
        b.workspace = workspace(b.workspace)
    out, lse = api.flash_attn_varlen_func(
        b.q, b.key_cache, b.value_cache, wl.max_seqlen_q, b.cu_seqlens_q,
        wl.max_seqlen_k, seqused_k=b.seqused_k,
        softmax_scale=wl.softmax_scale, causal=wl.causal,
        window_size=wl.window_size, softcap=wl.softcap,
        alibi_slopes=b.alibi, block_table=b.block_table,
        return_softmax_lse=True, workspace=b.workspace, s_aux=sinks)
    torch.cuda.synchronize(dev)
    api.check_device_errors(dev)
    return b, out.float().cpu().numpy(), lse.cpu().numpy()


CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, kwargs
    # one request far longer than a CTA's share: cut into many pieces
    ([1], [60000], 8, 2, 128, 16, dict()),
    # lengths spanning 1 .. 9000 keys, many per CTA and many cut
    ([1] * 40, [1, 2, 63, 64, 65, 100, 200, 300, 500, 900] * 3 +
     [1000, 2000, 3000, 4000, 5000, 6000, 7000, 8000, 9000, 17], 32, 8, 128,
     16, dict()),
    # prefill-class requests between decode-class ones
    ([1, 300, 1, 2, 40, 1], [5000, 700, 3, 4000, 90, 2500], 8, 4, 128, 32,
     dict()),
    # D 64 and D 256, window and soft-cap
    ([1, 1, 1, 3], [9000, 40, 5000, 700], 8, 2, 64, 16,
     dict(window_size=(3000, 0))),
    ([1, 1, 1], [12000, 300, 4100], 16, 8, 256, 32,
     dict(window_size=(4095, 0), softcap=50.0)),
    # fp16, ALiBi, non-causal, block size 64
    ([1, 2, 1], [3000, 2500, 65], 8, 2, 128, 64,
     dict(dtype="f16", causal=False,
          alibi_slopes=[0.001 * (i + 1) for i in range(8)])),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_persistent_decode(cuda_device, idx):
    q_lens, seq_lens, Hq, Hkv, D, BS, kw = CASES[idx]
    wl = workloads.build_workload("sk%d" % idx, 1200 + idx, q_lens, seq_lens,
                                  Hq, Hkv, D, BS, **kw)
    _, out, lse = _run(wl, cuda_device)
    ref_out, ref_lse = full_reference(wl)
    _close(wl, out, lse, ref_out, ref_lse, "case %d" % idx)


def test_persistent_decode_with_sinks(cuda_device):
    """A sink logit enters once per row, after the pieces are merged."""
    wl = workloads.build_workload("sk_sink", 1300, [1, 1, 1, 2],
                                  [40000, 7, 3000, 900], 16, 4, 128, 16)
    sinks = torch.linspace(-2.0, 3.0, 16, dtype=torch.float32)
    _, out, lse = _run(wl, cuda_device, sinks=sinks.to(cuda_device))
    ref_out, ref_lse = full_reference(wl)
    ro, rl = add_sink_ref(ref_out, ref_lse, sinks.double().numpy())
    _close(wl, out, lse, ro, rl, "sinks")


def test_persistent_decode_rows_without_keys(cuda_device):
    """Requests whose rows see no key take one pseudo-tile of the sequence
    and write out 0, lse -inf."""
    import dataclasses
    wl = workloads.build_workload("sk_empty", 1301, [1, 1, 3, 1],
                                  [3000, 5, 10, 2000], 8, 2, 64, 16)
    dev = cuda_device
    b = DeviceBatch(wl, dev)
    b.write_context()
    b.write_new()
    short = np.array([3000, 0, 1, 2000], dtype=np.int32)
    b.seqused_k.copy_(torch.from_numpy(short))
    out, lse = b.attend()
    torch.cuda.synchronize(dev)
    ref_out, ref_lse = full_reference(dataclasses.replace(wl,
                                                          seq_lens=short))
    _close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ref_out,
           ref_lse, "rows without keys")
    assert np.isneginf(ref_lse[:, 1]).all()


def test_workspace_without_scratch_falls_back(cuda_device):
    """The kernel's scratch is part of the optional workspace tail: without
    it the call runs one CTA per (request, KV head) and is still right."""
    wl = workloads.batched_decode(batch=24, lo=100, hi=5000,
                                  pool_blocks=9000)
    ref_out, ref_lse = full_reference(wl)
    _, out_sk, lse_sk = _run(wl, cuda_device)
    _close(wl, out_sk, lse_sk, ref_out, ref_lse, "persistent")
    # one byte short of the tail: only the required part remains usable
    _, out_fb, lse_fb = _run(wl, cuda_device,
                             workspace=lambda w: w[:w.numel() - 1])
    _close(wl, out_fb, lse_fb, ref_out, ref_lse, "fallback")


def test_full_batched_decode_every_request(cuda_device):
    """The bench's batched decode workload at full size: every request of
    the persistent kernel's output against the oracle."""
    wl = workloads.batched_decode(device=cuda_device)
    b = DeviceBatch(wl, cuda_device, poison=True)
    b.write_context()
    out, lse = b.step(return_lse=True)
    torch.cuda.synchronize()
    api.check_device_errors(cuda_device)
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    for r in range(wl.batch):
        ref_o, ref_l = request_reference(wl, r)
        _close(wl, o[r:r + 1], ls[:, r:r + 1], ref_o, ref_l, "req %d" % r)


# ------------------------------------------------------------ E4M3 caches
def _fp8_cache(wl, dev, ksc, vsc, nan_fill):
    fill = 0x7F if nan_fill else 0
    cache = torch.full(wl.cache_shape(), fill, dtype=torch.uint8, device=dev)
    kc, vc = cache.unbind(0)
    ks = torch.tensor([ksc], dtype=torch.float32, device=dev)
    vs = torch.tensor([vsc], dtype=torch.float32, device=dev)
    for rk, rv, sl in ((wl.k_ctx, wl.v_ctx, wl.slot_mapping_ctx),
                       (wl.k_new, wl.v_new, wl.slot_mapping_new)):
        if len(sl):
            api.reshape_and_cache_flash(rk.to(dev), rv.to(dev), kc, vc,
                                        torch.from_numpy(sl).to(dev), "fp8",
                                        ks, vs)
    return kc, vc, ks, vs


FP8_CASES = [
    # q_lens, seq_lens, Hq, Hkv, D, BS, dtype, q multiplier, NaN fill
    ([1, 1, 1], [9000, 33, 2500], 32, 8, 128, 16, "bf16", 1.0, True),
    ([1, 2, 1], [4000, 600, 70], 16, 2, 128, 64, "bf16", 300.0, True),
    ([1, 1], [3000, 129], 8, 4, 128, 16, "bf16", 1e-3, False),
    ([1, 1, 1], [5000, 200, 31], 16, 8, 256, 32, "bf16", 1.0, True),
    ([1, 3], [2000, 900], 8, 2, 128, 16, "f16", 1.0, True),
    ([1, 1], [7000, 64], 16, 8, 256, 32, "f16", 0.5, False),
]


@pytest.mark.parametrize("idx", range(len(FP8_CASES)))
def test_persistent_decode_fp8(cuda_device, idx):
    q_lens, seq_lens, Hq, Hkv, D, BS, dtype, qmul, nan_fill = FP8_CASES[idx]
    wl = workloads.build_workload("sk8_%d" % idx, 1400 + idx, q_lens,
                                  seq_lens, Hq, Hkv, D, BS, dtype=dtype)
    wl.q = (wl.q.float() * qmul).to(wl.torch_dtype)
    dev = cuda_device
    ksc, vsc = 0.013, 0.019
    kc, vc, ks, vs = _fp8_cache(wl, dev, ksc, vsc, nan_fill)
    out, lse = api.flash_attn_varlen_func(
        wl.q.to(dev), kc, vc, wl.max_seqlen_q,
        torch.from_numpy(wl.cu_seqlens_q).to(dev), wl.max_seqlen_k,
        seqused_k=torch.from_numpy(wl.seq_lens).to(dev),
        softmax_scale=wl.softmax_scale, causal=True,
        block_table=torch.from_numpy(wl.block_table).to(dev),
        return_softmax_lse=True, k_descale=ks, v_descale=vs)
    torch.cuda.synchronize()
    api.check_device_errors(dev)
    shape = wl.cache_shape()[1:]
    kcode = np.zeros(shape, np.uint8)
    vcode = np.zeros(shape, np.uint8)
    f32 = lambda t: t.float().numpy()                        # noqa: E731
    reshape_and_cache_fp8_ref(f32(wl.k_ctx), f32(wl.v_ctx), kcode, vcode,
                              wl.slot_mapping_ctx, ksc, vsc)
    reshape_and_cache_fp8_ref(f32(wl.k_new), f32(wl.v_new), kcode, vcode,
                              wl.slot_mapping_new, ksc, vsc)
    kref = e4m3_decode(kcode) * np.float64(np.float32(ksc))
    vref = e4m3_decode(vcode) * np.float64(np.float32(vsc))
    ro, rl = paged_attention_ref(f32(wl.q).astype(np.float64), kref, vref,
                                 wl.cu_seqlens_q, wl.seq_lens,
                                 wl.block_table, wl.softmax_scale)
    _close(wl, out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl,
           "fp8 case %d" % idx)
