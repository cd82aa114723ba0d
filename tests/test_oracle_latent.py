"""Pins of the oracle's latent stage (CPU only), by special cases whose
answer is known without the oracle.

Definition (vLLM docs, ``vllm.v1.worker.gpu.spec_decode.xpress.kernels``,
``_xpress_latent_kernel``): slot b gathers E[blk[n, b-1]] (slot 0: E[am1[n]]),
x = hcache + e @ W_lat, u[b] = sum_{j<=b} L[b,j] * x[j] per channel,
ub = bf16(u), m = bf16(silu(ub@Wg) * (ub@Wu)), lat[n, b-1] = bf16(u + m@Wd)
for b = 1..B-1."""

import math

import numpy as np
import torch

from speculative_decoding_gb300 import synth


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _case(seed=0, N=3, B=5, V=50, D=24, R=16, H=20):
    sh = synth.PassShape("t", N, B, V, D, R, H, seed)
    d = synth.pass_inputs(sh)
    return d, sh


def _eye_mixer(B, R):
    L = np.zeros((B, B, R), np.float32)
    for b in range(B):
        L[b, b, :] = 1.0
    return L


def test_identity_path_returns_hcache_exactly(orc):
    """W_lat = 0, L = I, Wd = 0: lat[n, b-1] = hcache[n, b] bit for bit
    (also pins the slot -> output row mapping)."""
    d, sh = _case()
    d["W_lat"][:] = 0
    d["Wd"][:] = 0
    L = _eye_mixer(sh.B, sh.R)
    lat = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], L, d["Wg"], d["Wu"], d["Wd"])
    np.testing.assert_array_equal(lat, d["hcache"][:, 1:, :])


def test_gather_selects_previous_token(orc):
    """One-hot embedding (E = I, D = V) and W_lat with distinct rows: slot b
    must see row blk[n, b-1] of W_lat, slot 0 row am1[n]."""
    N, B, V, R, H = 2, 4, 12, 8, 8
    sh = synth.PassShape("t", N, B, V, V, R, H, 1)
    d = synth.pass_inputs(sh)
    E = synth.to_bf16_bits(np.eye(V, dtype=np.float32))
    W_lat = synth.to_bf16_bits(np.arange(V * R, dtype=np.float32).reshape(V, R) / 8.0)
    hc = np.zeros_like(d["hcache"])
    d["Wd"][:] = 0
    L = _eye_mixer(B, R)
    lat, u = orc.latent(d["blk"], d["am1"], hc, E, W_lat, L, d["Wg"], d["Wu"], d["Wd"], want_u=True)
    Wf = _f(W_lat)
    for n in range(N):
        for b in range(B):
            prev = d["am1"][n] if b == 0 else d["blk"][n, b - 1]
            np.testing.assert_array_equal(u[n, b], Wf[prev])


def test_projection_matches_library_matmul(orc):
    """L = I, Wd = 0: lat = bf16(hcache + E[prev] @ W_lat); the product is
    checked against torch's float64 matmul (a library pin), to within one bf16
    rounding decision."""
    d, sh = _case(seed=2, N=4, B=6, V=300, D=96, R=32, H=16)
    d["Wd"][:] = 0
    L = _eye_mixer(sh.B, sh.R)
    lat, u = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], L, d["Wg"], d["Wu"],
                        d["Wd"], want_u=True)
    prev = np.concatenate([d["am1"][:, None], d["blk"][:, :-1]], axis=1)
    e = torch.from_numpy(_f(d["E"])[prev])
    x = torch.from_numpy(_f(d["hcache"])) + e @ torch.from_numpy(_f(d["W_lat"]))
    np.testing.assert_allclose(u, x.numpy(), rtol=0, atol=1e-12)
    want = torch.from_numpy(x.numpy()[:, 1:, :].astype(np.float32)).to(torch.bfloat16).float().numpy()
    got = _f(lat).astype(np.float32)
    # identical except where x sits within float rounding of a bf16 tie
    assert np.mean(got != want) < 1e-3
    np.testing.assert_allclose(got, want, rtol=2**-7, atol=0)


def test_mixer_cumulative_mean(orc):
    """W_lat = 0, L[b, j] = 1/(b+1) for j <= b: u[b] = mean(hcache[0..b]) --
    the closed form of an averaging causal mixer."""
    d, sh = _case(seed=3)
    d["W_lat"][:] = 0
    B, R = sh.B, sh.R
    L = np.zeros((B, B, R), np.float32)
    for b in range(B):
        L[b, : b + 1, :] = np.float32(1.0 / (b + 1))
    _, u = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], L, d["Wg"], d["Wu"],
                      d["Wd"], want_u=True)
    hc = _f(d["hcache"])
    for b in range(B):
        want = np.float64(np.float32(1.0 / (b + 1))) * hc[:, : b + 1, :].sum(axis=1)
        np.testing.assert_allclose(u[:, b, :], want, rtol=1e-12, atol=1e-12)


def test_mixer_channel_varying_selector(orc):
    """W_lat = 0 and a mixer that differs per channel: L[b, j, r] = 1 when
    j == r mod (b+1), else 0, so u[n, b, r] = hcache[n, r mod (b+1), r].  Each
    channel r of slot b picks a different earlier slot, so a mixer that lost
    the channel index (L[b, j, 0] for every r), or read L[j, b] instead of
    L[b, j], gives another answer."""
    d, sh = _case(seed=7, N=3, B=7, R=32)
    d["W_lat"][:] = 0
    B, R = sh.B, sh.R
    L = np.zeros((B, B, R), np.float32)
    for b in range(B):
        for r in range(R):
            L[b, r % (b + 1), r] = 1.0
    _, u = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], L, d["Wg"], d["Wu"],
                      d["Wd"], want_u=True)
    hc = _f(d["hcache"])
    for b in range(B):
        for r in range(R):
            np.testing.assert_array_equal(u[:, b, r], hc[:, r % (b + 1), r], err_msg=f"b={b} r={r}")
    # the selector is not symmetric in (b, j) and not constant over r
    assert not np.array_equal(L, L.transpose(1, 0, 2))
    assert not np.array_equal(L[:, :, 0:1].repeat(R, axis=2), L)


def test_mixer_is_causal(orc):
    """Changing slot j's inputs never changes u[b] for b < j."""
    d, sh = _case(seed=4, N=2, B=6)
    args = lambda hc: (d["blk"], d["am1"], hc, d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
    lat0, u0 = orc.latent(*args(d["hcache"]), want_u=True)
    hc = d["hcache"].copy()
    hc[:, 4, :] = synth.to_bf16_bits(np.full((sh.N, sh.R), 5.0, np.float32))
    lat1, u1 = orc.latent(*args(hc), want_u=True)
    np.testing.assert_array_equal(u0[:, :4], u1[:, :4])
    np.testing.assert_array_equal(lat0[:, :3], lat1[:, :3])
    assert not np.array_equal(lat0[:, 3], lat1[:, 3])


def test_mlp_closed_form_diagonal(orc):
    """R = H, Wg = a*I, Wu = c*I, Wd = s*I, W_lat = 0, L = I: per channel
    y = u + s * bf16(silu(a*ub) * c*ub), ub = bf16(u) -- a scalar closed form
    evaluated here with math.exp and exact bf16 rounding in Fractions."""
    from fractions import Fraction
    from exact import round_bf16

    N, B, R = 2, 3, 8
    sh = synth.PassShape("t", N, B, 40, 8, R, R, 5)
    d = synth.pass_inputs(sh)
    a, c, s = 0.75, -1.5, 0.5
    I = np.eye(R, dtype=np.float32)
    Wg, Wu, Wd = (synth.to_bf16_bits(k * I) for k in (a, c, s))
    d["W_lat"][:] = 0
    L = _eye_mixer(B, R)
    lat = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], L, Wg, Wu, Wd)
    hc = _f(d["hcache"])
    for n in range(N):
        for b in range(1, B):
            for r in range(R):
                ub = hc[n, b, r]                       # u = hcache here, already bf16
                g, v = a * ub, c * ub
                m = float(round_bf16(Fraction(g / (1.0 + math.exp(-g)) * v)))
                y = float(round_bf16(Fraction(ub + s * m)))
                assert _f(lat[n, b - 1, r]) == y, (n, b, r)


def test_zero_gate_gives_rounded_u(orc):
    """Wg = 0: silu(0) = 0 so m = 0 and lat = bf16(u)."""
    d, sh = _case(seed=6)
    d["Wg"][:] = 0
    lat, u = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"],
                        d["Wd"], want_u=True)
    np.testing.assert_array_equal(lat, orc.bf16_from_double(u[:, 1:, :]))


def test_token_out_of_range_is_an_error(orc):
    d, sh = _case()
    blk = d["blk"].copy()
    blk[1, 2] = sh.V
    import pytest

    with pytest.raises(orc.OracleError):
        orc.latent(blk, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
