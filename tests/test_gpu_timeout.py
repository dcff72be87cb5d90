"""A bounded device wait that runs out, and the status the host reads.

Every mbarrier wait of the decode kernels is bounded.  With the limit set to
0 (pkv_set_wait_limit_ns), a consumer gives up at the first poll that does
not find its K/V stage complete, and the producer at the first poll that
does not find a free stage; on the 600 MB batched decode some of those polls
must miss.  The CTA records a timeout in the device error word, drains the
copies it issued (the drains keep the full limit, so nothing is in flight
when it exits) and returns.  The host then reads PKV_ERR_TIMEOUT, and the
next call, with the default limit, runs clean and matches the oracle.  No
GPU fault, trap or hang is involved: the failure is a wait that the kernel
itself stops.
"""
import numpy as np
import pytest
import torch

from oracle.harness import request_reference
from paged_kv_cache_318_gb300 import api, workloads
from paged_kv_cache_318_gb300.batch import DeviceBatch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built(cuda_device):
    from paged_kv_cache_318_gb300 import _build
    _build.build()
    api.load_library()
    yield
    api.set_wait_limit_ns(api.WAIT_LIMIT_DEFAULT_NS)
    api.set_decode_kernel(api.DECODE_AUTO)


@pytest.mark.parametrize("kernel", ["tma", "persistent"])
def test_wait_limit_runs_out_then_next_call_is_clean(cuda_device, kernel):
    dev = cuda_device
    wl = workloads.batched_decode(device=dev)
    b = DeviceBatch(wl, dev, poison=False)
    b.write_context()
    b.write_new()
    torch.cuda.synchronize()
    api.check_device_errors(dev)
    api.set_decode_kernel(api.DECODE_TMA if kernel == "tma"
                          else api.DECODE_PERSISTENT)
    try:
        api.set_wait_limit_ns(0)
        status = None
        for _ in range(3):
            b.attend(return_lse=False)
            try:
                api.check_device_errors(dev)
            except api.PkvError as e:
                status = e.status
                msg = str(e)
                break
        assert status == api.PKV_ERR_TIMEOUT, status
        assert "bounded wait" in msg
        # the error word was read and cleared
        api.check_device_errors(dev)
    finally:
        api.set_wait_limit_ns(api.WAIT_LIMIT_DEFAULT_NS)
    try:
        out, lse = b.attend(return_lse=True)
        torch.cuda.synchronize()
        api.check_device_errors(dev)
    finally:
        api.set_decode_kernel(api.DECODE_AUTO)
    o = out.float().cpu().numpy()
    ls = lse.cpu().numpy()
    for r in (0, 31, 63):
        ref_o, ref_l = request_reference(wl, r)
        assert np.abs(o[r:r + 1] - ref_o).max() <= 2e-2
        assert np.abs(ls[:, r:r + 1] - ref_l).max() <= 1e-3
