"""GPU parity of xp_latent_pass against the oracle.

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
_xpress_latent_kernel (gather of the previous slot's embedding, hidden cache,
W_lat projection, folded causal mixer, SwiGLU MLP with the residual on u).
Tolerance: max |gpu - oracle| <= 2e-2 * max |oracle| over all outputs (fp32
accumulation order and bf16 roundings of intermediate values differ from the
oracle's double accumulation)."""

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16, host_bits
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_latent(d, shape):
    N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    lat = torch.zeros((N, B - 1, R), dtype=torch.bfloat16, device="cuda")
    ws = xpress.workspace(xpress.latent_workspace_size(N, B, D, R, H))
    xpress.latent_pass(dev(d["blk"]), dev(d["am1"]), dev_bf16(d["hcache"]), dev_bf16(d["E"]), dev_bf16(d["W_lat"]),
                       dev(d["L"]), dev_bf16(d["Wg"]), dev_bf16(d["Wu"]), dev_bf16(d["Wd"]), lat, ws)
    torch.cuda.synchronize()
    return host_bits(lat), xpress.read_error(ws)


def oracle_latent(orc, d):
    return orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])


SHAPES = [
    synth.TINY,
    synth.PassShape("t1", 3, 5, 500, 192, 64, 128, 11),
    synth.PassShape("t2", 8, 16, 4096, 512, 128, 256, 12),
    synth.PassShape("t3", 5, 7, 3000, 200, 256, 192, 13),
    synth.PassShape("t4", 17, 16, 2048, 1024, 512, 512, 14),
    synth.PassShape("t5", 1, 2, 100, 64, 16, 64, 15),
    # D = R: the pages' own layout (embedding already at the latent width)
    synth.PassShape("dr", 6, 16, 3000, 512, 512, 256, 16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_latent_parity(orc, shape):
    d = synth.pass_inputs(shape)
    got, err = run_latent(d, shape)
    assert err == 0
    want = oracle_latent(orc, d)
    g, w = _f(got).astype(np.float64), _f(want).astype(np.float64)
    tol = 2e-2 * np.abs(w).max()
    assert np.abs(g - w).max() <= tol, (np.abs(g - w).max(), tol)
    # almost every element agrees to one bf16 step
    assert np.mean(np.abs(g - w) <= np.abs(w) * 2**-7 + 1e-6) > 0.97


# exact-arithmetic inputs (synth.exact_pass_inputs): every sum is exact in
# fp32 whatever its order, so the latent must equal the oracle's bit for bit
EXACT_SHAPES = [
    synth.PassShape("e1", 4, 8, 1000, 64, 64, 64, 5),          # D = 64: the projection's D sum is not split
    synth.PassShape("e2", 160, 16, 1000, 256, 512, 512, 6),    # 80 output tiles: not split either (64-channel tiles)
    synth.PassShape("e3", 9, 16, 3000, 256, 128, 256, 7),
    synth.PassShape("e4", 32, 16, 4096, 3584, 512, 1536, 8),   # the serving dims (E's vocab reduced)
    synth.PassShape("e5", 1, 16, 4096, 3584, 512, 1536, 9),    # one block at the serving dims
    synth.PassShape("e6", 96, 16, 1000, 256, 512, 512, 10),    # 12 M tiles: a 2-way D split would not fit, unsplit
    synth.PassShape("e7", 64, 16, 1000, 256, 512, 1536, 11),   # MLP grids of 192 and 256 CTAs: two CTAs per SM
]


@pytest.mark.parametrize("shape", EXACT_SHAPES, ids=[s.name for s in EXACT_SHAPES])
def test_latent_exact_arithmetic_bit_exact(orc, shape):
    d = synth.exact_pass_inputs(shape)
    got, err = run_latent(d, shape)
    assert err == 0
    want = oracle_latent(orc, d)
    bad = np.argwhere(got != want)
    assert len(bad) == 0, (len(bad), bad[:8].tolist())


def test_identity_path_exact(orc):
    """W_lat = 0, L = I, Wd = 0: lat[n, b-1] = hcache[n, b] bit for bit."""
    shape = synth.PassShape("id", 4, 6, 300, 128, 64, 64, 21)
    d = synth.pass_inputs(shape)
    d["W_lat"][:] = 0
    d["Wd"][:] = 0
    L = np.zeros((shape.B, shape.B, shape.R), np.float32)
    for b in range(shape.B):
        L[b, b, :] = 1.0
    d["L"] = L
    got, _ = run_latent(d, shape)
    np.testing.assert_array_equal(got, d["hcache"][:, 1:, :])


def test_full_size_latent(orc):
    """N=32, B=16, D=3584, R=512, H=1536 (the serving workload's latent)."""
    shape = synth.SERVE
    d = synth.pass_inputs(shape)
    got, err = run_latent(d, shape)
    assert err == 0
    want = oracle_latent(orc, d)
    g, w = _f(got).astype(np.float64), _f(want).astype(np.float64)
    assert np.abs(g - w).max() <= 2e-2 * np.abs(w).max()


def test_bad_token_flags_error():
    shape = synth.PassShape("bad", 2, 4, 100, 64, 32, 64, 3)
    d = synth.pass_inputs(shape)
    d["blk"][1, 1] = 100     # == V
    _, err = run_latent(d, shape)
    assert err & xpress.XP_DEVERR_TOKEN
