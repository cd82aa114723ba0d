"""Failure detection on the GPU without a fault: the library's bounded
mbarrier wait runs out (a barrier nothing arrives on, 1 ms limit), the kernel
sets the timeout bit and returns, the host reads the bit, and the context
stays usable for the next call."""

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu

XP_DEVERR_TIMEOUT = 2


def test_bounded_wait_gives_up_and_reports(orc):
    ws = xpress.workspace(xpress.add_argmax_workspace_size(6, 1000))
    xpress.selftest_wait_timeout(ws, limit_us=1000)
    torch.cuda.synchronize()
    assert xpress.read_error(ws) == XP_DEVERR_TIMEOUT
    assert xpress.read_error(ws) == 0  # read and cleared
    # the context is usable: an ordinary call right after gives the right answer
    a = synth.argmax_inputs(6, 1000, 2, 4, seed=5, tie_frac=0.0)
    blk = dev(a["blk"].copy())
    xpress.add_argmax(dev_bf16(a["base"]), dev_bf16(a["bias"]), blk, ws)
    torch.cuda.synchronize()
    assert xpress.read_error(ws) == 0
    want = a["blk"].copy()
    orc.add_argmax(a["base"], a["bias"], want)
    np.testing.assert_array_equal(blk.cpu().numpy(), want)


def test_limit_is_checked_on_the_host():
    ws = xpress.workspace(256)
    with pytest.raises(xpress.XpressError):
        xpress.selftest_wait_timeout(ws, limit_us=0)
    with pytest.raises(xpress.XpressError):
        xpress.selftest_wait_timeout(ws, limit_us=3_000_000)
