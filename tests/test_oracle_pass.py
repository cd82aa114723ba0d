"""Pins of the oracle's readout and full pass (CPU only).

The pass (vLLM docs, ``vllm.v1.worker.gpu.spec_decode.xpress.kernels``, module
docstring): latent -> readout logits = base + x @ W2 -> blk = argmax_v logits,
with the bias x @ W2 produced in bf16 by the caller's matmul
(``xpress_latent_pass`` docstring) and the sum rounded to bf16 before the
argmax.  Repeated passes read blk in place (``_xpress_add_argmax_reduce_to_blk_kernel``)."""

import numpy as np
import torch

from speculative_decoding_gb300 import synth


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _tiny():
    return synth.pass_inputs(synth.TINY)


def test_readout_matches_library_matmul(orc):
    d = _tiny()
    rng = np.random.default_rng(0)
    lat = synth.to_bf16_bits(rng.normal(0, 1, (6, 32)).astype(np.float32))
    bias = orc.readout_bias(lat, d["W2"])
    ref = (torch.from_numpy(_f(lat)) @ torch.from_numpy(_f(d["W2"]))).numpy()
    want = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    got = _f(bias).astype(np.float32)
    assert np.mean(got != want) < 1e-3
    np.testing.assert_allclose(got, want, rtol=2**-7)


def test_row_logits_is_readout_plus_base(orc):
    d = _tiny()
    rng = np.random.default_rng(1)
    lat = synth.to_bf16_bits(rng.normal(0, 1, (2, 32)).astype(np.float32))
    bias = orc.readout_bias(lat, d["W2"])
    for r in range(2):
        s = orc.row_logits(lat[r], d["W2"], d["base"][r])
        want = [orc.bf16_add(int(a), int(b)) for a, b in zip(d["base"][r], bias[r])]
        np.testing.assert_array_equal(s, _f(np.array(want, np.uint16)))


def test_zero_readout_reduces_to_argmax_of_base(orc):
    """W2 = 0: the bias is 0 and the pass writes torch.argmax(base) per row."""
    d = _tiny()
    d["W2"][:] = 0
    blk = d["blk"].copy()
    orc.jacobi_pass(blk, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"],
                    d["W2"], d["base"])
    want = torch.argmax(torch.from_numpy(_f(d["base"])), dim=1).numpy()
    np.testing.assert_array_equal(blk[:, 1:].reshape(-1), want)
    np.testing.assert_array_equal(blk[:, 0], d["blk"][:, 0])


def test_pass_is_latent_then_readout_then_argmax(orc):
    d = _tiny()
    blk = d["blk"].copy()
    changed = orc.jacobi_pass(blk, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"],
                              d["Wd"], d["W2"], d["base"])
    lat = orc.latent(d["blk"], d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
    bias = orc.readout_bias(lat.reshape(-1, lat.shape[-1]), d["W2"])
    blk2 = d["blk"].copy()
    orc.add_argmax(d["base"], bias, blk2)
    np.testing.assert_array_equal(blk, blk2)
    assert changed == int((blk[:, 1:] != d["blk"][:, 1:]).sum())


def test_multipass_causal_fixpoint(orc):
    """Slot s's token depends only on tokens at slots < s, so after pass p
    slots 1..p are final; a fixpoint is reached within B passes."""
    sh = synth.PassShape("t", 3, 6, 300, 32, 16, 24, 9)
    d = synth.pass_inputs(sh)
    # shrink base so the readout matters and tokens move between passes
    d["base"] = synth.to_bf16_bits(_f(d["base"]).astype(np.float32) * np.float32(0.05))
    d["W2"] = synth.to_bf16_bits(_f(d["W2"]).astype(np.float32) * np.float32(8.0))
    blk = d["blk"].copy()
    history = [blk.copy()]
    args = (d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"], d["W2"], d["base"])
    counts = []
    for _ in range(sh.B):
        counts.append(orc.jacobi_pass(blk, *args))
        history.append(blk.copy())
        if counts[-1] == 0:
            break
    assert counts[-1] == 0 and len(counts) <= sh.B
    assert counts[0] > 0
    for p in range(1, len(history)):
        for q in range(p, len(history)):
            np.testing.assert_array_equal(history[q][:, 1:p + 1], history[p][:, 1:p + 1])
    passes, cnt = orc.jacobi_to_fixpoint(d["blk"].copy(), *args, max_passes=sh.B)
    assert passes == len(counts) and cnt == counts
