"""Failure detection on the GPU without a fault: bounded waits give up.

Each case makes a device-side wait run out on purpose (an mbarrier nobody
arrives on; a grid barrier expecting one block too many).  The kernel must
record NVFP4_ERR_TIMEOUT and return, and the context must stay usable for
the next real computation.
"""
import numpy as np
import pytest
import torch

from nvfp4_weight_only_02_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_reports_timeout_and_context_survives(nv, orc, which):
    ws = nv.new_workspace(256)
    nv.nvfp4_wait_selftest(ws, which)
    assert nv.nvfp4_get_device_status(ws) == nv.ERR_TIMEOUT
    assert nv.nvfp4_get_device_status(ws) == nv.OK
    # the context still works: a real quantisation is bit-exact afterwards
    bits = synth.normal_weight((64, 256), 0.02, 1)
    w = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    q = nv.quantize(w, workspace=ws)
    torch.cuda.synchronize()
    rc, codes, scales, st = orc.quantize(bits)
    assert np.array_equal(q.codes.cpu().numpy(), codes)
    assert nv.nvfp4_get_device_status(ws) == nv.OK


def test_timeout_with_tile_counters_leaves_workspace_reusable(nv, orc):
    """A wait that gives up after a kernel has counted arrivals at output
    tiles leaves those counters non-zero; nvfp4_get_device_status reports the
    timeout and sets them (and every counter and flag word) back to zero, so
    the same workspace then serves a decode GEMM that matches the oracle."""
    c = synth.small_case(8, 700, 2048, 16, seed=12)
    M, K = c.x.shape
    N = c.w.shape[0]
    ws = nv.new_workspace(nv.nvfp4_workspace_bytes(M, N, K, 16))
    nv.nvfp4_wait_selftest(ws, 2)
    torch.cuda.synchronize()
    words = ws[:256 + 4 * 8192].view(torch.int32).cpu().numpy()
    assert (words[64:] != 0).sum() == 4          # four tile counters left counted
    assert nv.nvfp4_get_device_status(ws) == nv.ERR_TIMEOUT
    words = ws[:256 + 4 * 8192].view(torch.int32).cpu().numpy()
    assert not words.any()                        # control block and counters all zero again
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    q = nv.quantize(dev(c.w))
    y = nv.gemm(dev(c.x), q, dev(c.a), dev(c.b), c.lora_scale, torch.from_numpy(c.z).cuda(), workspace=ws)
    assert nv.nvfp4_get_device_status(ws) == nv.OK
    rc, codes, scales, st = orc.quantize(c.w)
    ref = orc.gemm(c.x, codes, scales, st, c.a, c.b, c.lora_scale, c.z)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max() and err.sum() <= 1e-3 * np.abs(ref).sum()
