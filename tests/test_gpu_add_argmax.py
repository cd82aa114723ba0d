"""GPU parity of xp_add_argmax against the oracle, bit-exact (indices are
integers decided by bf16 comparisons on both sides).

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
fused_add_argmax_to_blk -- blk[n, 1+j] = lowest argmax_v bf16(base + bias)."""

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16, host_bits, padded_bf16
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu


def _run(base_bits, bias_bits, blk, ld=None, guard=4):
    """Run xp_add_argmax; blk lives inside a buffer with canaries on both sides."""
    rows, V = base_bits.shape
    N, B = blk.shape
    if ld is None or ld == V:
        tb, tc = dev_bf16(base_bits), dev_bf16(bias_bits)
    else:
        tb, tc = padded_bf16(base_bits, ld), padded_bf16(bias_bits, ld)
    canary = np.int64(-7777)
    buf = np.full(N * B + 2 * guard, canary, np.int64)
    buf[guard:guard + N * B] = blk.reshape(-1)
    tbuf = dev(buf)
    tblk = tbuf[guard:guard + N * B].view(N, B)
    ws = xpress.workspace(xpress.add_argmax_workspace_size(rows, V))
    xpress.add_argmax(tb, tc, tblk, ws)
    torch.cuda.synchronize()
    out = tbuf.cpu().numpy()
    assert (out[:guard] == canary).all() and (out[guard + N * B:] == canary).all(), "wrote outside blk"
    assert int(ws[:256].view(torch.int32)[0].item()) == 0
    # the call must leave the workspace's reduction state zero
    assert int(ws[256:].count_nonzero().item()) == 0
    return out[guard:guard + N * B].reshape(N, B)


def _oracle(orc, base, bias, blk):
    want = blk.copy()
    orc.add_argmax(base, bias, want)
    return want


@pytest.mark.parametrize("rows,V,B,ld", [(6, 1000, 4, None), (15, 7, 16, 8), (3, 1, 4, 8), (30, 4097, 4, 4104),
                                         (45, 8192, 16, None), (60, 8193, 4, 8200), (30, 65536 + 13, 16, 65552),
                                         (16, 20000, 17, 20000 + 64)])
def test_parity_shapes(orc, rows, V, B, ld):
    N = rows // (B - 1)
    d = synth.argmax_inputs(rows, V, N, B, seed=rows * 7 + V, tie_frac=0.1)
    got = _run(d["base"], d["bias"], d["blk"], ld=ld)
    want = _oracle(orc, d["base"], d["bias"], d["blk"])
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got[:, 0], d["blk"][:, 0])
    for r, pos in d["planted"].items():
        n, j = divmod(r, B - 1)
        assert got[n, 1 + j] == min(pos)


def test_parity_full_size_480x152064(orc):
    """The standalone add-argmax workload: 480 rows x 152064, 1% planted ties;
    every row checked."""
    d = synth.argmax_inputs(synth.ARGMAX_ROWS, synth.ARGMAX_V, 32, 16, seed=synth.ARGMAX_SEED, tie_frac=0.01)
    assert len(d["planted"]) == 5
    got = _run(d["base"], d["bias"], d["blk"])
    want = _oracle(orc, d["base"], d["bias"], d["blk"])
    np.testing.assert_array_equal(got, want)
    # run again on the same (self-cleaning) workspace path
    got2 = _run(d["base"], d["bias"], d["blk"])
    np.testing.assert_array_equal(got2, want)


def _bits(x):
    return synth.to_bf16_bits(np.asarray(x, np.float32))


def test_edge_values(orc):
    """Signed zeros tie; subnormal sums round like the oracle; overflow to
    +inf is a value; planted ties across vector and CTA boundaries."""
    V = 9000
    rows = 6
    base = np.full((rows, V), _bits([-5.0])[0], np.uint16)
    bias = np.zeros((rows, V), np.uint16)
    # row 0: -0 + -0 at 8191 (CTA 0's last element) ties +0 at 8192 (CTA 1)
    base[0, 8191] = 0x8000; bias[0, 8191] = 0x8000
    base[0, 8192] = 0x0000
    # row 1: subnormals: 2^-133 + 2^-133 vs 3*2^-134 ... exact bf16 subnormal arithmetic
    base[1, :] = 0x0001; bias[1, :] = 0x0000
    base[1, 7000] = 0x0001; bias[1, 7000] = 0x0001        # 2 * min subnormal
    base[1, 100] = 0x0002; bias[1, 100] = 0x0000          # the same value, earlier
    # row 2: overflow to +inf
    big = _bits([3.3e38])[0]
    base[2, 5] = big; base[2, 6000] = big; bias[2, 6000] = big
    # row 3: a tie inside one 16-byte vector (positions 3 and 5)
    base[3, 3] = base[3, 5] = _bits([9.0])[0]
    # row 4: all equal -> index 0
    base[4, :] = _bits([1.5])[0]
    # row 5: maximum only at the last element
    base[5, V - 1] = _bits([2.0])[0]
    blk = np.arange(2 * 4, dtype=np.int64).reshape(2, 4)
    got = _run(base, bias, blk)
    want = _oracle(orc, base, bias, blk)
    np.testing.assert_array_equal(got, want)
    assert got[0, 1] == 8191 and got[0, 2] == 100 and got[0, 3] == 6000
    assert got[1, 1] == 3 and got[1, 2] == 0 and got[1, 3] == V - 1


def test_empty_is_noop():
    ws = xpress.workspace(256)
    blk = torch.zeros((0, 4), dtype=torch.int64, device="cuda")
    base = torch.zeros((0, 8), dtype=torch.bfloat16, device="cuda")
    xpress.add_argmax(base, base, blk, ws)


def test_misaligned_rejected():
    base = torch.zeros((3, 1000 + 8), dtype=torch.bfloat16, device="cuda")
    blk = torch.zeros((1, 4), dtype=torch.int64, device="cuda")
    ws = xpress.workspace(xpress.add_argmax_workspace_size(3, 1000))
    with pytest.raises(xpress.XpressError) as e:
        xpress.add_argmax(base[:, 1:1001], base[:, :1000], blk, ws)
    assert e.value.status == xpress.XP_ERR_ALIGN
