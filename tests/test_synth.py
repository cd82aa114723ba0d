"""The seeded input generators (CPU): the same seed gives the same values
whatever the thread count, the distributions have the stated moments, the
mixer is lower-triangular with rows summing to 1, and planted ties make the
lowest planted position the row's unique first maximum."""

import numpy as np
import pytest

from speculative_decoding_gb300 import synth


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_normals_do_not_depend_on_the_thread_count(monkeypatch):
    n = 3 * (1 << 22) + 12345  # several chunks and a ragged tail
    a = synth._normal_f32(7, 3, n, 1.0)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    b = synth._normal_f32(7, 3, n, 1.0)
    np.testing.assert_array_equal(a, b)
    assert not np.array_equal(a[:1000], synth._normal_f32(8, 3, 1000, 1.0))   # another seed
    assert not np.array_equal(a[:1000], synth._normal_f32(7, 4, 1000, 1.0))   # another stream


@pytest.mark.parametrize("std", [0.02, 1.0, 3.0])
def test_normal_moments(std):
    x = _f(synth.normal_bf16(1, 9, (1 << 20,), std))
    assert abs(x.mean()) < 5 * std / 1024          # 5 standard errors
    assert abs(x.std() / std - 1.0) < 0.01


def test_tokens_in_range_and_seeded():
    t = synth.tokens(3, 12, (64, 16), 152064)
    assert t.dtype == np.int64 and t.min() >= 0 and t.max() < 152064
    np.testing.assert_array_equal(t, synth.tokens(3, 12, (64, 16), 152064))


def test_mixer_is_folded_lower_triangular():
    L = synth.mixer(5, 16, 64)
    assert L.dtype == np.float32
    upper = np.triu(np.ones((16, 16), bool), 1)
    assert np.all(L[upper] == 0)
    assert np.all(L[~upper] > 0)
    np.testing.assert_allclose(L.astype(np.float64).sum(axis=1), 1.0, rtol=1e-6)


def test_planted_ties_make_the_lowest_position_the_answer():
    a = synth.argmax_inputs(40, 3000, 8, 6, seed=11, tie_frac=0.25)
    assert len(a["planted"]) == 10
    for r, pos in a["planted"].items():
        assert 2 <= len(pos) <= 4 and pos == sorted(pos)
        s = _f(a["base"][r]) + _f(a["bias"][r])   # exact in double for these magnitudes
        top = s.max()
        assert list(np.flatnonzero(s == top)) == pos


def test_pass_inputs_shapes_and_dtypes():
    sh = synth.PassShape("t", 3, 5, 500, 64, 32, 64, 9)
    d = synth.pass_inputs(sh)
    want = dict(E=(500, 64), W_lat=(64, 32), Wg=(32, 64), Wu=(32, 64), Wd=(64, 32), W2=(32, 500),
                hcache=(3, 5, 32), base=(12, 500), am1=(3,), blk=(3, 5), L=(5, 5, 32))
    for k, shp in want.items():
        assert d[k].shape == shp, k
    for k in ("E", "W_lat", "Wg", "Wu", "Wd", "W2", "hcache", "base"):
        assert d[k].dtype == np.uint16, k
    assert d["am1"].dtype == np.int64 and d["L"].dtype == np.float32
    # the activations alone match the full draw
    act = synth.pass_activations(sh)
    for k in ("hcache", "base", "am1", "blk"):
        np.testing.assert_array_equal(act[k], d[k])


@pytest.mark.parametrize("dims", [(4, 8, 1000, 64, 64, 64), (160, 16, 1000, 256, 512, 512),
                                  (32, 16, 4096, 3584, 512, 1536)])
def test_exact_inputs_keep_every_sum_exact(orc, dims):
    """The bounds synth.exact_pass_inputs states, checked on the oracle's own
    values: u (and so lat) on the 2^-7 grid with at most 24 significant bits,
    and every partial sum of lat @ W2 on the 2^-11 grid below 2^13, so fp32
    represents every intermediate exactly."""
    shape = synth.PassShape("exact", *dims, 5)
    d = synth.exact_pass_inputs(shape)
    lat, u = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"],
                        want_u=True)
    assert np.all(u * 2**7 == np.round(u * 2**7)) and np.abs(u).max() < 2**17
    lf = orc.bf16_to_float(lat).astype(np.float64)
    # m = 0 (Wg = 0): lat = bf16(u), which stays on the 2^-7 grid
    np.testing.assert_array_equal(lat, orc.bf16_from_double(u[:, 1:, :]))
    assert np.all(lf * 2**7 == np.round(lf * 2**7))
    W2 = orc.bf16_to_float(d["W2"]).astype(np.float64)
    assert np.all(W2 * 16 == np.round(W2 * 16))
    assert (np.abs(lf.reshape(-1, shape.R)) @ np.abs(W2)).max() < 2**13
    L = d["L"].astype(np.float64)
    np.testing.assert_array_equal(L.sum(axis=1), 1.0)
    assert np.all(np.triu(np.ones((shape.B, shape.B)), 1)[:, :, None] * L == 0)
