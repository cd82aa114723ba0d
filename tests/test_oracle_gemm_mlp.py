"""Pins of the oracle's GEMM-MLP schedule (CPU only).

Method (vLLM docs, ``vllm.v1.worker.gpu.spec_decode.xpress.kernels``,
``xpress_latent_pass`` with ``do_mlp`` False): the latent kernel stops after
the mixer and hands back bf16(u) for slots 1..B-1; the caller then runs the
SwiGLU as GEMMs on the bf16 tensor: ``gu = u @ wgu_t`` (Wg and Wu side by
side, a bf16 matmul), ``m = silu_and_mul(gu)`` and ``u.addmm_(m, wd_t)``.
So g and v are rounded to bf16 before the SiLU, and the residual is the bf16
u, where the in-kernel MLP keeps both in fp32.

Two exact closed forms separate the schedules on the roundings they differ
in; a third test checks the whole schedule against torch's own CPU ops for
the three calls (library routines) on random data."""

import math
from fractions import Fraction

import numpy as np
import torch

from exact import round_bf16
from speculative_decoding_gb300 import synth


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bits(values):
    return synth.to_bf16_bits(np.asarray(values, np.float32))


def _tiny(B, R, H, V=4, D=8):
    """Inputs with E = W_lat = 0 (so x = hcache) and all-zero tokens."""
    return dict(blk=np.zeros((1, B), np.int64), am1=np.zeros(1, np.int64),
                E=np.zeros((V, D), np.uint16), W_lat=np.zeros((D, R), np.uint16))


def _silu_bf16(g, v):
    return float(round_bf16(Fraction(g / (1.0 + math.exp(-g)) * v)))


def test_residual_is_the_bf16_u(orc):
    """u = 1 + 2^-9 (the mixer adds hcache slots 0 and 1), m @ Wd = 2^-8.
    In-kernel: bf16(1 + 2^-9 + 2^-8) = 1 + 2^-7.  GEMM schedule: the residual
    is bf16(u) = 1, and bf16(1 + 2^-8) is a tie that rounds to even: 1."""
    d = _tiny(B=2, R=1, H=1)
    hc = np.zeros((1, 2, 1), np.uint16)
    hc[0, 0, 0], hc[0, 1, 0] = _bits([1.0, 2.0**-9])
    L = np.zeros((2, 2, 1), np.float32)
    L[0, 0, 0] = 1.0
    L[1, 0, 0] = L[1, 1, 0] = 1.0
    Wg, Wu, Wd = _bits([[16.0]]), _bits([[2.0**-12]]), _bits([[1.0]])
    # both schedules feed ub = bf16(u) = 1 to the MLP: g = 16, v = 2^-12, and
    # silu(16) * 2^-12 rounds to exactly 2^-8
    assert _silu_bf16(16.0, 2.0**-12) == 2.0**-8
    args = (d["blk"], d["am1"], hc, d["E"], d["W_lat"], L, Wg, Wu, Wd)
    fused = orc.latent(*args)
    gemm = orc.latent(*args, do_mlp=False)
    assert _f(fused[0, 0, 0]) == 1.0 + 2.0**-7
    assert _f(gemm[0, 0, 0]) == 1.0


def test_gate_and_up_are_rounded_to_bf16(orc):
    """ub = [1, 2^-9, 0] (bf16 already), Wg = [1, 1, 0], Wu = [1, 0, 0]:
    g = 1 + 2^-9, v = 1.  GEMM schedule: bf16(g) = 1, so m = bf16(silu(1));
    in-kernel: m = bf16(silu(1 + 2^-9)), one bf16 step higher.  Wd copies m
    into channel 2, whose residual is 0, so lat[.., 2] = m exactly."""
    d = _tiny(B=2, R=3, H=1)
    hc = np.zeros((1, 2, 3), np.uint16)
    hc[0, 1, :] = _bits([1.0, 2.0**-9, 0.0])
    L = np.zeros((2, 2, 3), np.float32)
    L[0, 0, :] = L[1, 1, :] = 1.0
    Wg = _bits([[1.0], [1.0], [0.0]])
    Wu = _bits([[1.0], [0.0], [0.0]])
    Wd = _bits([[0.0, 0.0, 1.0]])
    args = (d["blk"], d["am1"], hc, d["E"], d["W_lat"], L, Wg, Wu, Wd)
    m_gemm, m_fused = _silu_bf16(1.0, 1.0), _silu_bf16(1.0 + 2.0**-9, 1.0)
    assert m_gemm != m_fused  # the two schedules must differ here
    fused = orc.latent(*args)
    gemm = orc.latent(*args, do_mlp=False)
    assert _f(gemm[0, 0, 2]) == m_gemm
    assert _f(fused[0, 0, 2]) == m_fused
    # the other channels: residual only (Wd is zero there)
    assert _f(gemm[0, 0, 0]) == 1.0 and _f(gemm[0, 0, 1]) == 2.0**-9


def test_gemm_schedule_matches_torch_ops(orc):
    """Random data: the oracle's GEMM schedule against torch's CPU bf16 ops
    for the pages' three calls (``u @ wgu_t``; SiLU(gate) * up rounded once;
    ``addmm_`` into the bf16 u).  torch accumulates in fp32 where the oracle
    uses double, so a result may sit one bf16 step away."""
    sh = synth.PassShape("g", 3, 5, 300, 64, 48, 96, 31)
    d = synth.pass_inputs(sh)
    args = (d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
    _, u = orc.latent(*args, want_u=True)
    got = _f(orc.latent(*args, do_mlp=False))
    bf = torch.bfloat16
    ub = torch.from_numpy(orc.bf16_from_double(u[:, 1:, :]).reshape(-1, sh.R).view(np.int16)).view(bf)
    t = lambda a: torch.from_numpy(a.view(np.int16)).view(bf)
    wgu = torch.cat([t(d["Wg"]), t(d["Wu"])], dim=1)
    gu = ub @ wgu
    m = (torch.nn.functional.silu(gu[:, : sh.H].float()) * gu[:, sh.H:].float()).to(bf)
    want = torch.addmm(ub, m, t(d["Wd"])).float().numpy().astype(np.float64).reshape(got.shape)
    diff = np.abs(got - want)
    assert diff.max() <= 2e-2 * np.abs(want).max(), diff.max()
    assert np.mean(diff <= np.abs(want) * 2.0**-7 + 1e-9) > 0.97


def test_schedules_agree_without_mlp_and_share_the_mixer(orc):
    """Wg = 0: m = 0 in both schedules, so both give bf16(u); and the mixer
    output u never depends on the schedule."""
    sh = synth.PassShape("z", 2, 4, 100, 32, 16, 64, 32)
    d = synth.pass_inputs(sh)
    d["Wg"][:] = 0
    args = (d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
    lat1, u1 = orc.latent(*args, want_u=True)
    lat0, u0 = orc.latent(*args, want_u=True, do_mlp=False)
    np.testing.assert_array_equal(u0, u1)
    np.testing.assert_array_equal(lat0, lat1)
    np.testing.assert_array_equal(lat0, orc.bf16_from_double(u0[:, 1:, :]))
