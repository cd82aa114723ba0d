"""GPU parity of xp_readout_argmax (tcgen05 readout with the add + argmax
fused into its epilogue) against the oracle.

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels -- module
docstring (readout logits = base + x @ W2, argmax written to blk) and
fused_add_argmax_to_blk (sum rounded to bf16 before the argmax).

Two kinds of check:
  * exact-arithmetic inputs (small integers times powers of two) make every
    fp32 partial sum exact, so the bias is identical on both sides and blk
    must match bit for bit -- this pins the MMA operand layouts;
  * random inputs: the fp32 accumulation order may move the bias by one bf16
    step near a rounding boundary, so the rule is the pass tolerance: the
    chosen token's oracle logit lies within 0.0625 of the oracle row maximum
    (and nearly all tokens are equal)."""

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu


def _bits(x):
    return synth.to_bf16_bits(np.asarray(x, np.float32))


def _run(lat, W2, base, blk, ld=None):
    rows, R = lat.shape
    V = W2.shape[1]
    tb = dev_bf16(base) if ld is None else None
    if ld is not None:
        full = np.zeros((rows, ld), np.uint16)
        full[:, :V] = base
        tb = dev_bf16(full)[:, :V]
    tblk = dev(blk.copy())
    changed = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = xpress.workspace(xpress.readout_workspace_size(rows, V))
    # the library takes the readout weight vocabulary-major: W2t = W2.T, [V, R]
    xpress.readout_argmax(dev_bf16(lat), dev_bf16(np.ascontiguousarray(W2.T)), tb, tblk, ws, changed=changed)
    torch.cuda.synchronize()
    assert xpress.read_error(ws) == 0
    assert int(ws[256:].count_nonzero().item()) == 0, "workspace not left clean"
    return tblk.cpu().numpy(), int(changed.item())


def _exact_inputs(rows, V, R, seed):
    rng = np.random.default_rng(seed)
    lat = _bits(rng.integers(-3, 4, (rows, R)).astype(np.float32))
    W2 = _bits(rng.integers(-4, 5, (R, V)).astype(np.float32) / 16.0)
    base = synth.normal_bf16(seed, 1, (rows, V), 3.0)
    return lat, W2, base


@pytest.mark.parametrize("N,B,V,R", [(2, 4, 1000, 32), (1, 16, 4096, 64), (32, 16, 152064, 512),
                                     (10, 21, 2056, 128), (5, 27, 520, 512), (9, 16, 768, 256),
                                     (64, 16, 8192, 512)])
def test_exact_inputs_bit_exact(orc, N, B, V, R):
    rows = N * (B - 1)
    lat, W2, base = _exact_inputs(rows, V, R, seed=V + R)
    blk = synth.tokens(5, 5, (N, B), V)
    got, changed = _run(lat, W2, base, blk)
    bias = orc.readout_bias(lat, W2)
    want = blk.copy()
    orc.add_argmax(base, bias, want)
    np.testing.assert_array_equal(got, want)
    assert changed == int((want != blk).sum())


@pytest.mark.parametrize("N,B,V,R", [(3, 5, 1001, 64), (2, 3, 33, 32), (4, 9, 4097, 128)])
def test_odd_vocab_all_negative(orc, N, B, V, R):
    """V odd, and V < 64 (a whole 32-column chunk of the first tile lies past
    V): the padding past V reads as zero on the device, which would beat
    every real logit here (all negative); it must never win.  The base rows
    need a leading dimension that is a multiple of 8."""
    rows = N * (B - 1)
    lat, W2, base = _exact_inputs(rows, V, R, seed=V)
    base = _bits(synth._f32(base) - 64.0)
    blk = synth.tokens(8, 8, (N, B), V)
    got, changed = _run(lat, W2, base, blk, ld=(V + 7) // 8 * 8)
    bias = orc.readout_bias(lat, W2)
    want = blk.copy()
    orc.add_argmax(base, bias, want)
    np.testing.assert_array_equal(got, want)
    assert changed == int((want != blk).sum())


def test_exact_inputs_strided_base(orc):
    N, B, V, R = 3, 5, 1000, 64
    rows = N * (B - 1)
    lat, W2, base = _exact_inputs(rows, V, R, seed=3)
    blk = synth.tokens(6, 6, (N, B), V)
    got, _ = _run(lat, W2, base, blk, ld=1064)
    bias = orc.readout_bias(lat, W2)
    want = blk.copy()
    orc.add_argmax(base, bias, want)
    np.testing.assert_array_equal(got, want)


def _check_tolerance(orc, lat, W2, base, got, sample_rows, B):
    exact = 0
    for r in sample_rows:
        s = orc.row_logits(lat[r], W2, base[r])
        n, j = divmod(r, B - 1)
        tok = got[n, 1 + j]
        assert s[tok] >= s.max() - 0.0625, (r, tok, s[tok], s.max())
        exact += int(tok == int(np.argmax(s)))
    return exact


@pytest.mark.parametrize("N,B,V,R", [(2, 4, 1000, 32), (8, 16, 20000, 512)])
def test_random_inputs_tolerance(orc, N, B, V, R):
    rows = N * (B - 1)
    rng = np.random.default_rng(R)
    lat = _bits(rng.normal(0, 1, (rows, R)).astype(np.float32))
    W2 = synth.normal_bf16(9, 9, (R, V), 1.0 / np.sqrt(R))
    base = synth.normal_bf16(9, 10, (rows, V), 3.0)
    blk = synth.tokens(7, 7, (N, B), V)
    got, _ = _run(lat, W2, base, blk)
    exact = _check_tolerance(orc, lat, W2, base, got, range(rows), B)
    assert exact >= rows - max(1, rows // 50)


def test_full_size_random_sampled(orc):
    """rows = 480 (N=32, B=16), V = 152064, R = 512 with the pass's weight
    scale; 24 sampled rows checked against the oracle's row logits."""
    N, B, V, R = 32, 16, 152064, 512
    rows = N * (B - 1)
    rng = np.random.default_rng(0)
    lat = _bits(rng.normal(0, 1, (rows, R)).astype(np.float32))
    W2 = synth.normal_bf16(2, 6, (R, V), 1.0 / np.sqrt(R))
    base = synth.normal_bf16(2, 9, (rows, V), 3.0)
    blk = synth.tokens(2, 12, (N, B), V)
    got, _ = _run(lat, W2, base, blk)
    sample = sorted(set([0, 1, 127, 128, 255, 256, 383, 384, 479] + rng.choice(rows, 15, replace=False).tolist()))
    exact = _check_tolerance(orc, lat, W2, base, got, sample, B)
    assert exact >= len(sample) - 1
    np.testing.assert_array_equal(got[:, 0], blk[:, 0])
