"""GPU parity of the GEMM-MLP schedule (xp_latent_pass_ex / xp_jacobi_pass_ex
with do_mlp = 0) against the oracle.

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
xpress_latent_pass with do_mlp False: the kernel hands back bf16(u), then
u @ wgu_t (bf16), silu_and_mul, u.addmm_(m, wd_t) on the bf16 u.  Tolerances
as for the in-kernel schedule (latent: max |gpu - oracle| <= 2e-2 max |oracle|;
pass: the chosen token's oracle logit within 0.0625 of the row maximum); the
two closed forms that separate the schedules are checked bit for bit."""

import math

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16, host_bits
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu
TOL = 0.0625


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits(values):
    return synth.to_bf16_bits(np.asarray(values, np.float32))


def run_latent(d, shape, do_mlp):
    N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    lat = torch.zeros((N, B - 1, R), dtype=torch.bfloat16, device="cuda")
    ws = xpress.workspace(xpress.latent_workspace_size(N, B, D, R, H))
    xpress.latent_pass(dev(d["blk"]), dev(d["am1"]), dev_bf16(d["hcache"]), dev_bf16(d["E"]), dev_bf16(d["W_lat"]),
                       dev(d["L"]), dev_bf16(d["Wg"]), dev_bf16(d["Wu"]), dev_bf16(d["Wd"]), lat, ws, do_mlp=do_mlp)
    torch.cuda.synchronize()
    assert xpress.read_error(ws) == 0
    return host_bits(lat)


SHAPES = [
    synth.TINY,
    synth.PassShape("g1", 3, 5, 500, 192, 64, 128, 41),
    synth.PassShape("g2", 8, 16, 4096, 512, 128, 256, 42),
    synth.PassShape("g3", 17, 16, 2048, 1024, 512, 512, 43),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_latent_gemm_schedule_parity(orc, shape):
    d = synth.pass_inputs(shape)
    got = _f(run_latent(d, shape, do_mlp=False))
    want = _f(orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"],
                         do_mlp=False))
    diff = np.abs(got - want)
    assert diff.max() <= 2e-2 * np.abs(want).max(), diff.max()
    assert np.mean(diff <= np.abs(want) * 2.0**-7 + 1e-6) > 0.97


def _small(R=16, H=64, B=2):
    shape = synth.PassShape("c", 1, B, 4, 8, R, H, 44)
    d = dict(blk=np.zeros((1, B), np.int64), am1=np.zeros(1, np.int64), E=np.zeros((4, 8), np.uint16),
             W_lat=np.zeros((8, R), np.uint16), hcache=np.zeros((1, B, R), np.uint16),
             L=np.zeros((B, B, R), np.float32), Wg=np.zeros((R, H), np.uint16), Wu=np.zeros((R, H), np.uint16),
             Wd=np.zeros((H, R), np.uint16))
    return shape, d


def test_residual_is_the_bf16_u():
    """Channel 0: u = 1 + 2^-9 (hcache slots 0 and 1 mixed), m @ Wd = 2^-8
    (g = 16, v = 2^-12).  In-kernel: bf16(1 + 2^-9 + 2^-8) = 1 + 2^-7; GEMM
    schedule: bf16(bf16(u) + 2^-8) = bf16(1 + 2^-8), a tie, = 1."""
    shape, d = _small()
    d["hcache"][0, 0, 0], d["hcache"][0, 1, 0] = _bits([1.0, 2.0**-9])
    d["L"][0, 0, :] = 1.0
    d["L"][1, 0, 0] = d["L"][1, 1, :] = 1.0
    d["Wg"][0, 0], d["Wu"][0, 0], d["Wd"][0, 0] = _bits([16.0, 2.0**-12, 1.0])
    assert _f(run_latent(d, shape, do_mlp=True)[0, 0, 0]) == 1.0 + 2.0**-7
    assert _f(run_latent(d, shape, do_mlp=False)[0, 0, 0]) == 1.0


def test_gate_and_up_are_rounded_to_bf16():
    """ub = [1, 2^-9, 0, ...], Wg[:, 0] = [1, 1, 0, ...], Wu[:, 0] = e_0:
    g = 1 + 2^-9, v = 1.  The GEMM schedule rounds g to 1 first, so
    m = bf16(silu(1)); the in-kernel MLP gives bf16(silu(1 + 2^-9)), one bf16
    step higher.  Wd copies m into channel 2 (residual 0)."""
    shape, d = _small()
    d["hcache"][0, 1, :2] = _bits([1.0, 2.0**-9])
    d["L"][0, 0, :] = d["L"][1, 1, :] = 1.0
    d["Wg"][0, 0] = d["Wg"][1, 0] = _bits([1.0])[0]
    d["Wu"][0, 0] = _bits([1.0])[0]
    d["Wd"][0, 2] = _bits([1.0])[0]
    silu = lambda g: g / (1.0 + math.exp(-g))
    m_gemm = _f(_bits([silu(1.0)])[0])
    m_fused = _f(_bits([silu(1.0 + 2.0**-9)])[0])
    assert m_gemm != m_fused
    assert _f(run_latent(d, shape, do_mlp=False)[0, 0, 2]) == m_gemm
    assert _f(run_latent(d, shape, do_mlp=True)[0, 0, 2]) == m_fused


@pytest.mark.parametrize("shape", [synth.TINY, synth.PassShape("gp", 9, 16, 3000, 256, 128, 256, 45)],
                         ids=["tiny", "gp"])
def test_pass_gemm_schedule_parity(orc, shape):
    d = synth.pass_inputs(shape)
    N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
    t = {k: dev_bf16(d[k]) for k in ("hcache", "E", "W_lat", "Wg", "Wu", "Wd", "base")}
    W2t = dev_bf16(np.ascontiguousarray(d["W2"].T))
    ws = xpress.workspace(xpress.jacobi_workspace_size(N, B, V, D, R, H))
    blk = dev(d["blk"].copy())
    xpress.jacobi_pass(blk, dev(d["am1"]), t["hcache"], t["E"], t["W_lat"], dev(d["L"]), t["Wg"], t["Wu"], t["Wd"],
                       W2t, t["base"], ws, do_mlp=False)
    torch.cuda.synchronize()
    assert xpress.read_error(ws) == 0
    out = blk.cpu().numpy()
    np.testing.assert_array_equal(out[:, 0], d["blk"][:, 0])
    lat = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"],
                     do_mlp=False).reshape(-1, R)
    exact = 0
    for r in range(shape.rows):
        s = orc.row_logits(lat[r], d["W2"], d["base"][r])
        n, j = divmod(r, B - 1)
        tok = out[n, 1 + j]
        assert s[tok] >= s.max() - TOL, (r, tok, s[tok], s.max())
        exact += int(tok == int(np.argmax(s)))
    assert exact >= shape.rows - max(1, shape.rows // 50)
    # the oracle's own pass in the same schedule agrees on the exact tokens
    ob = d["blk"].copy()
    orc.jacobi_pass(ob, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"], d["W2"],
                    d["base"], do_mlp=False)
    assert np.mean(ob == out) >= 1 - max(1, shape.rows // 50) / shape.rows


def test_bad_do_mlp_is_a_shape_error():
    shape, d = _small()
    lat = torch.zeros((1, 1, 16), dtype=torch.bfloat16, device="cuda")
    ws = xpress.workspace(xpress.latent_workspace_size(1, 2, 8, 16, 64))
    lib = xpress.lib()
    p = lambda a: a.data_ptr()
    tens = [dev(d["blk"]), dev(d["am1"]), dev_bf16(d["hcache"]), dev_bf16(d["E"]), dev_bf16(d["W_lat"]), dev(d["L"]),
            dev_bf16(d["Wg"]), dev_bf16(d["Wu"]), dev_bf16(d["Wd"]), lat]
    st = lib.xp_latent_pass_ex(*[p(x) for x in tens], 1, 2, 4, 8, 16, 64, 2, p(ws), ws.numel(), None)
    assert st == xpress.XP_ERR_SHAPE
