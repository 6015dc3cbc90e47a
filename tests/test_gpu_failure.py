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
