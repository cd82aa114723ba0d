"""Pins of the oracle's add-argmax and top-C argmax (CPU only).

Definition (vLLM docs, ``vllm.v1.worker.gpu.spec_decode.xpress.kernels``,
``fused_add_argmax_to_blk`` and its two stage kernels): for row
r = n*(B-1)+b, blk[n, 1+b] = the lowest v maximising bf16(base[r,v]+bias[r,v]);
slot 0 is never written."""

import json
import os

import numpy as np
import pytest
import torch

from exact import argmax_lowest, bf16_sum
from speculative_decoding_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(x):
    return synth.to_bf16_bits(np.asarray(x, np.float32))


def test_golden_hand_rows(orc):
    g = json.load(open(os.path.join(HERE, "golden", "add_argmax_hand.json")))
    base = _bits(g["base"])
    bias = _bits(g["bias"])
    # the fixture's -0.0 entries must survive as negative zero
    assert base[3, 2] == 0x8000 and bias[3, 2] == 0x8000
    blk = np.array(g["blk_before"], np.int64)
    orc.add_argmax(base, bias, blk)
    assert blk.tolist() == g["blk_after"]


def test_bruteforce_fractions_tiny(orc):
    """Exact rational brute force on the tiny workload's rows (6 x 1000)."""
    d = synth.argmax_inputs(6, 1000, 2, 4, seed=0, tie_frac=0.05)
    blk = d["blk"].copy()
    before = blk.copy()
    orc.add_argmax(d["base"], d["bias"], blk)
    for r in range(6):
        sums = [bf16_sum(int(a), int(b)) for a, b in zip(d["base"][r], d["bias"][r])]
        n, b = divmod(r, 3)
        assert blk[n, 1 + b] == argmax_lowest(sums)
    np.testing.assert_array_equal(blk[:, 0], before[:, 0])


@pytest.mark.parametrize("rows,V", [(6, 1000), (30, 4097), (15, 7), (3, 1), (45, 65536 + 13)])
def test_matches_torch_bf16_add_argmax(orc, rows, V):
    """Library pin: torch adds two bf16 tensors with one rounding and
    torch.argmax returns the first maximal index."""
    B = 4 if rows % 3 == 0 else 16
    N = rows // (B - 1)
    d = synth.argmax_inputs(rows, V, N, B, seed=rows + V, tie_frac=0.1)
    blk = d["blk"].copy()
    orc.add_argmax(d["base"], d["bias"], blk)
    tb = torch.from_numpy(d["base"].view(np.int16)).view(torch.bfloat16)
    tc = torch.from_numpy(d["bias"].view(np.int16)).view(torch.bfloat16)
    want = torch.argmax((tb + tc).float(), dim=1).numpy()
    got = blk[:, 1:].reshape(-1)
    np.testing.assert_array_equal(got, want)


def test_planted_ties_lowest_position(orc):
    d = synth.argmax_inputs(480, 20000, 32, 16, seed=3, tie_frac=0.01)
    assert len(d["planted"]) == 5
    blk = d["blk"].copy()
    orc.add_argmax(d["base"], d["bias"], blk)
    for r, pos in d["planted"].items():
        n, b = divmod(r, 15)
        assert blk[n, 1 + b] == min(pos)


def test_signed_zero_tie(orc):
    base = _bits([[-1.0, -0.0, 0.0, -0.0, -2.0]])
    bias = _bits([[0.0, -0.0, 0.0, 0.0, 0.0]])
    assert base[0, 1] == 0x8000 and bias[0, 1] == 0x8000
    blk = np.zeros((1, 2), np.int64)
    orc.add_argmax(base, bias, blk)
    assert blk[0, 1] == 1        # -0 at v=1 ties +0 at v=2 and -0+0 at v=3
    base = _bits([[-1.0, 0.0, -0.0]])
    bias = _bits([[0.0, 0.0, -0.0]])
    orc.add_argmax(base, bias, blk)
    assert blk[0, 1] == 1


def test_overflow_to_inf_is_a_value(orc):
    big = 3.3e38
    base = _bits([[1.0, big, big, 2.0]])
    bias = _bits([[0.0, 0.0, big, 0.0]])
    blk = np.zeros((1, 2), np.int64)
    orc.add_argmax(base, bias, blk)
    assert blk[0, 1] == 2        # big + big rounds to +inf


def test_errors(orc):
    base = _bits(np.zeros((4, 8)))
    blk = np.zeros((2, 3), np.int64)
    with pytest.raises(orc.OracleError):
        orc.add_argmax(base, base, np.zeros((2, 4), np.int64))   # rows != N*(B-1)
    with pytest.raises(orc.OracleError):
        orc.add_argmax(base, base, np.zeros((4, 1), np.int64))   # B < 2
    bad = base.copy()
    bad[1, 3] = 0x7F80
    with pytest.raises(orc.OracleError):
        orc.add_argmax(bad, base, blk)
    orc.add_argmax(base, base, blk)
    assert (blk[:, 1:] == 0).all()


def test_topc_bruteforce(orc):
    rng = np.random.default_rng(11)
    N, B, C = 3, 5, 37
    rows = N * (B - 1)
    base_c = _bits(rng.normal(0, 3, (rows, C)))
    bias_c = _bits(rng.normal(0, 1, (rows, C)))
    base_c[2, 30] = base_c[2, 4] = _bits([40.0])[0]
    bias_c[2, 30] = bias_c[2, 4] = 0
    cand = rng.integers(0, 152064, (rows, C), dtype=np.int64)
    blk = rng.integers(0, 152064, (N, B), dtype=np.int64)
    before = blk.copy()
    orc.topc_argmax(base_c, bias_c, cand, blk)
    for r in range(rows):
        sums = [bf16_sum(int(a), int(b)) for a, b in zip(base_c[r], bias_c[r])]
        n, b = divmod(r, B - 1)
        assert blk[n, 1 + b] == cand[r, argmax_lowest(sums)]
    assert blk[0, 3] == cand[2, 4]
    np.testing.assert_array_equal(blk[:, 0], before[:, 0])
