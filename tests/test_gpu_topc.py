"""GPU parity of xp_topc_argmax (argmax over a slot's C gathered candidates,
written back as a vocab id) against the oracle: bit-exact.

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels --
fused_topc_argmax_to_blk / _xpress_topc_argmax_to_blk_kernel (the sum is
rounded to bf16 before the compare; ties go to the lowest candidate
position)."""

import numpy as np
import pytest

from gpu_util import dev, dev_bf16
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu


def _case(N, B, C, seed, tie_frac=0.1):
    rows = N * (B - 1)
    base = synth.normal_bf16(seed, 1, (rows, C), 3.0)
    bias = synth.normal_bf16(seed, 2, (rows, C), 1.0)
    if C > 1:
        synth.plant_ties(base, bias, tie_frac, seed)
    rng = np.random.default_rng(seed)
    cand = rng.integers(0, 152064, (rows, C), dtype=np.int64)
    blk = synth.tokens(seed, 3, (N, B), 152064)
    return base, bias, cand, blk


@pytest.mark.parametrize("N,B,C", [(2, 4, 1), (2, 4, 7), (3, 5, 32), (32, 16, 64), (5, 9, 100),
                                   (4, 16, 1000), (1, 2, 4097)])
def test_topc_bit_exact(orc, N, B, C):
    base, bias, cand, blk = _case(N, B, C, seed=N * 131 + C)
    tb = dev(blk.copy())
    xpress.topc_argmax(dev_bf16(base), dev_bf16(bias), dev(cand), tb)
    want = blk.copy()
    orc.topc_argmax(base, bias, cand, want)
    got = tb.cpu().numpy()
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got[:, 0], blk[:, 0])  # slot 0 untouched


def test_topc_signed_zero_and_ties(orc):
    """+0 and -0 tie (the lower position wins); equal maxima pick the lowest
    position; all-negative rows."""
    N, B, C = 1, 4, 40
    rows = N * (B - 1)
    base = np.zeros((rows, C), np.uint16)
    bias = np.zeros((rows, C), np.uint16)
    # row 0: -0 at position 3, +0 everywhere else (all other sums 0) -> position 0
    base[0, 3] = 0x8000
    bias[0, 3] = 0x8000
    # row 1: every value -1 except two equal maxima -0.5 at 33 and 17 -> 17
    base[1, :] = 0xBF80
    base[1, 33] = 0xBF00
    base[1, 17] = 0xBF00
    # row 2: strictly decreasing; the first position wins
    base[2, :] = synth.to_bf16_bits(-np.arange(C, dtype=np.float32) / 8.0)
    cand = np.arange(rows * C, dtype=np.int64).reshape(rows, C) * 7 + 1
    blk = np.full((N, B), -5, np.int64)
    tb = dev(blk.copy())
    xpress.topc_argmax(dev_bf16(base), dev_bf16(bias), dev(cand), tb)
    want = blk.copy()
    orc.topc_argmax(base, bias, cand, want)
    got = tb.cpu().numpy()
    np.testing.assert_array_equal(got, want)
    assert got[0, 1] == cand[0, 0] and got[0, 2] == cand[1, 17] and got[0, 3] == cand[2, 0]


def test_topc_empty_and_errors():
    import torch

    blk = torch.zeros((0, 4), dtype=torch.int64, device="cuda")
    z = torch.zeros((0, 3, 8), dtype=torch.bfloat16, device="cuda")
    xpress.topc_argmax(z, z, torch.zeros((0, 3, 8), dtype=torch.int64, device="cuda"), blk)  # N = 0: no-op
    blk = torch.zeros((2, 4), dtype=torch.int64, device="cuda")
    bad = torch.zeros((5, 8), dtype=torch.bfloat16, device="cuda")  # rows != N*(B-1)
    with pytest.raises(xpress.XpressError) as e:
        xpress.topc_argmax(bad, bad, torch.zeros((5, 8), dtype=torch.int64, device="cuda"), blk)
    assert e.value.status == xpress.XP_ERR_SHAPE
