"""GPU parity for attention without a cache, and batch-invariant splits.

Non-paged ("encoder") attention: K/V are plain [Tk, Hkv, D] rows selected
per request by cu_seqlens_k, as vLLM v1's ``_forward_encoder_attention``
(bidirectional, cu_seqlens_k = query_start_loc) and aphrodite's cache-free
prefill (causal, cu_seqlens_k = seq_start_loc) call flash attention.  The
CUDA path is compared with the float64 oracle ``varlen_attention_ref``:
outputs within max-abs 2e-2 (bf16) / 4e-3 (fp16), LSE within 1e-3.

Batch invariance: with a fixed split size, a request's output and LSE bits
must not change when the rest of its batch changes.
"""
import numpy as np
import pytest
import torch

from oracle import varlen_attention_ref
from oracle.harness import request_reference
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


CASES = [
    # q_lens, k_lens, Hq, Hkv, D, kwargs
    ([37, 200, 1, 129], [37, 200, 1, 129], 8, 8, 64, dict()),     # encoder
    ([300, 17, 64, 2], [300, 17, 64, 2], 16, 2, 128, dict()),     # GQA
    ([150, 3, 260], [150, 3, 260], 8, 2, 128, dict(causal=True)),
    ([1, 2, 40], [700, 1500, 90], 8, 4, 128, dict(causal=True)),
    ([1, 2], [2100, 900], 8, 8, 64, dict(causal=True, num_splits=3)),
    ([1, 70], [3000, 70], 8, 2, 256, dict(causal=True, softcap=20.0,
                                          window_size=(100, 0))),
    ([130, 9], [130, 9], 4, 4, 256, dict()),
    ([5, 64], [80, 64], 4, 2, 64, dict(causal=True, alibi=True, sinks=True)),
    ([20, 3], [45, 3], 4, 4, 64, dict(window_size=(10, 5))),
    ([0, 3, 2, 40], [5, 0, 7, 0], 4, 2, 64, dict()),     # empty q / empty k
]


def _run(inp, dev, head_major=False, **kw):
    q = inp.q.to(dev)
    k, v = inp.k.to(dev), inp.v.to(dev)
    if head_major:
        # physical [Hkv, Tk, D], viewed as [Tk, Hkv, D]
        k = k.transpose(0, 1).contiguous().transpose(0, 1)
        v = v.transpose(0, 1).contiguous().transpose(0, 1)
    cu_q = torch.as_tensor(inp.cu_seqlens_q, dtype=torch.int32, device=dev)
    cu_k = torch.as_tensor(inp.cu_seqlens_k, dtype=torch.int32, device=dev)
    mq = int(np.diff(inp.cu_seqlens_q).max())
    mk = int(np.diff(inp.cu_seqlens_k).max())
    out, lse = api.flash_attn_varlen_func(
        q, k, v, mq, cu_q, mk, cu_seqlens_k=cu_k, return_softmax_lse=True,
        **kw)
    torch.cuda.synchronize(dev)
    api.check_device_errors(dev)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _check(inp, out, lse, ref_out, ref_lse, what):
    assert np.isfinite(out).all(), what
    err = np.abs(out - ref_out).max() if out.size else 0.0
    assert err <= TOL[inp.dtype], "%s out err %g" % (what, err)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), what + ": lse -inf set"
    if fin.any():
        lerr = np.abs(lse[fin] - ref_lse[fin]).max()
        assert lerr <= LSE_TOL, "%s lse err %g" % (what, lerr)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("idx", range(len(CASES)))
def test_nonpaged_matches_oracle(cuda_device, idx, dtype):
    q_lens, k_lens, Hq, Hkv, D, kw = CASES[idx]
    kw = dict(kw)
    inp = workloads.nonpaged_inputs(400 + idx, q_lens, k_lens, Hq, Hkv, D,
                                    dtype)
    scale = D ** -0.5
    rng = np.random.default_rng(idx)
    alibi = sinks = None
    if kw.pop("alibi", False):
        alibi = rng.uniform(0.01, 0.5, Hq).astype(np.float32)
        kw["alibi_slopes"] = torch.from_numpy(alibi).to(cuda_device)
    if kw.pop("sinks", False):
        sinks = rng.uniform(-1, 2, Hq).astype(np.float32)
        kw["s_aux"] = torch.from_numpy(sinks).to(cuda_device)
    causal = kw.get("causal", False)
    ref_out, ref_lse = varlen_attention_ref(
        inp.q.double().numpy(), inp.k.double().numpy(),
        inp.v.double().numpy(), inp.cu_seqlens_q, inp.cu_seqlens_k, scale,
        causal=causal, window_size=kw.get("window_size", (-1, -1)),
        softcap=kw.get("softcap", 0.0), alibi_slopes=alibi, sinks=sinks)
    for head_major in (False, True):
        out, lse = _run(inp, cuda_device, head_major=head_major,
                        softmax_scale=scale, **kw)
        _check(inp, out, lse, ref_out, ref_lse,
               "case %d head_major=%s" % (idx, head_major))


def test_nonpaged_rows_past_the_tensor_are_flagged(cuda_device):
    """cu_seqlens_k running past total_k: nothing outside the K/V rows is
    read, the clipped requests are reported through the device error
    word, and the in-range requests still match the oracle."""
    inp = workloads.nonpaged_inputs(450, [1, 40, 3], [30, 40, 20], 4, 2, 64)
    cu_k = inp.cu_seqlens_k.copy()
    cu_k[-1] += 25                       # request 2 claims 25 rows too many
    dev = cuda_device
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cq = torch.as_tensor(inp.cu_seqlens_q, dtype=torch.int32, device=dev)
    ck = torch.as_tensor(cu_k, dtype=torch.int32, device=dev)
    out, lse = api.flash_attn_varlen_func(q, k, v, 40, cq, 45,
                                          cu_seqlens_k=ck,
                                          return_softmax_lse=True)
    with pytest.raises(api.PkvError):
        api.check_device_errors(dev)
    ref_out, ref_lse = varlen_attention_ref(
        inp.q.double().numpy(), inp.k.double().numpy(),
        inp.v.double().numpy(), inp.cu_seqlens_q, inp.cu_seqlens_k,
        64 ** -0.5)
    rows = slice(0, 41)                  # requests 0 and 1
    o = out.float().cpu().numpy()[rows]
    assert np.abs(o - ref_out[rows]).max() <= TOL["bf16"]
    assert np.abs(lse.cpu().numpy()[:, rows] - ref_lse[:, rows]).max() \
        <= LSE_TOL
    api.check_device_errors(dev)         # the word was cleared


def test_nonpaged_rejects_fp8_and_bad_options(cuda_device):
    inp = workloads.nonpaged_inputs(451, [2], [9], 4, 2, 64)
    dev = cuda_device
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cq = torch.as_tensor(inp.cu_seqlens_q, dtype=torch.int32, device=dev)
    ck = torch.as_tensor(inp.cu_seqlens_k, dtype=torch.int32, device=dev)
    k8 = k.to(torch.float8_e4m3fn)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    with pytest.raises(NotImplementedError):
        api.flash_attn_varlen_func(q, k8, k8, 2, cq, 9, cu_seqlens_k=ck,
                                   k_descale=one, v_descale=one)
    with pytest.raises(ValueError):
        api.flash_attn_varlen_func(q, k, v, 2, cq, 9, cu_seqlens_k=ck,
                                   num_splits=2, fixed_split_size=256)


# ------------------------------------------------------- batch invariance
def _sub_batch_call(b, idx, **kw):
    """Attention for requests ``idx`` of DeviceBatch ``b`` alone."""
    wl, dev = b.wl, b.device
    cu = wl.cu_seqlens_q
    rows = np.concatenate([np.arange(cu[i], cu[i + 1]) for i in idx])
    q_lens = [int(cu[i + 1] - cu[i]) for i in idx]
    q = b.q[torch.as_tensor(rows, device=dev)]
    cu_sub = torch.as_tensor(workloads.cu_seqlens(q_lens), dtype=torch.int32,
                             device=dev)
    su = b.seqused_k[torch.as_tensor(idx, device=dev)]
    bt = b.block_table[torch.as_tensor(idx, device=dev)].contiguous()
    out, lse = api.flash_attn_varlen_func(
        q, b.key_cache, b.value_cache, max(q_lens), cu_sub,
        int(wl.seq_lens[idx].max()), seqused_k=su,
        softmax_scale=wl.softmax_scale, causal=True, block_table=bt,
        window_size=wl.window_size, softcap=wl.softcap,
        return_softmax_lse=True, **kw)
    return rows, out, lse


def _mixed_d128(dtype):
    """40 decodes (L ~ U[100, 9000]) then 3 chunks of 90 tokens (context
    ~ U[0, 2000]), 32/8 heads, D 128: sub-batches that hold a chunk have few
    prefill work items, where a free plan would split the chunk's keys."""
    rng = np.random.default_rng([326, 2])
    dec = rng.integers(100, 9001, 40)
    ctx = rng.integers(0, 2001, 3)
    q = [1] * 40 + [90] * 3
    L = list(dec) + list(ctx + 90)
    return workloads.build_workload("mixed_d128", 326, q, L, 32, 8, 128, 16,
                                    dtype=dtype)


@pytest.mark.parametrize("kind", ["gemma_d256", "llama_d128"])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("mode", [dict(fixed_split_size=2048),
                                  dict(fixed_split_size=100),
                                  dict(num_splits=1)])
def test_fixed_splits_are_batch_invariant(cuda_device, mode, dtype, kind):
    if kind == "gemma_d256":
        wl = workloads.mixed_gemma(dtype=dtype, n_prefill=3, chunk=90,
                                   c_hi=2000, n_decode=40, d_lo=100,
                                   d_hi=9000)
    else:
        wl = _mixed_d128(dtype)
    wl.num_splits = 0
    b = DeviceBatch(wl, cuda_device)
    b.write_context()
    b.write_new()
    full_out, full_lse = api.flash_attn_varlen_func(
        b.q, b.key_cache, b.value_cache, wl.max_seqlen_q, b.cu_seqlens_q,
        wl.max_seqlen_k, seqused_k=b.seqused_k,
        softmax_scale=wl.softmax_scale, causal=True,
        block_table=b.block_table, window_size=wl.window_size,
        softcap=wl.softcap, return_softmax_lse=True, **mode)
    torch.cuda.synchronize()
    api.check_device_errors(cuda_device)
    longest = int(np.argmax(wl.seq_lens))
    for idx in ([longest], [5, longest, 0], [1, 7, 12, 30, 41],
                list(range(wl.batch))[::-1]):
        rows, out, lse = _sub_batch_call(b, np.asarray(idx), **mode)
        torch.cuda.synchronize()
        r = torch.as_tensor(rows, device=cuda_device)
        assert torch.equal(out.view(torch.int16),
                           full_out[r].view(torch.int16)), idx
        assert torch.equal(lse.view(torch.int32),
                           full_lse[:, r].view(torch.int32)), idx
    # and the invariant result is still the right one
    for i in (0, longest, wl.batch - 1):
        ro, rl = request_reference(wl, i, last_rows=4)
        t1 = int(wl.cu_seqlens_q[i + 1])
        t0 = max(int(wl.cu_seqlens_q[i]), t1 - 4)
        o = full_out[t0:t1].float().cpu().numpy()
        assert np.abs(o - ro).max() <= TOL[dtype]
        assert np.abs(full_lse[:, t0:t1].cpu().numpy() - rl).max() <= LSE_TOL
