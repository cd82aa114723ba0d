"""GPU parity of xp_jacobi_pass (latent -> tcgen05 readout with the fused
add + argmax) against the oracle.

Method: vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels, module
docstring (one pass: latent, readout, argmax into blk[n, 1+b], blk read in
place by the next pass).  Rule for tokens: equal to the oracle's, or the
oracle logit of the chosen token lies within 0.0625 of the oracle's row
maximum (floating-point accumulation order may move a bias by one bf16 step
near a tie).  Multi-pass runs are teacher-forced: before every pass the oracle
gets the GPU's blk, so one near-tie cannot cascade."""

import numpy as np
import pytest
import torch

from gpu_util import dev, dev_bf16
from speculative_decoding_gb300 import synth, xpress

pytestmark = pytest.mark.gpu
TOL = 0.0625


class Pass:
    def __init__(self, d, shape):
        self.d, self.shape = d, shape
        N, B, V, D, R, H = shape.N, shape.B, shape.V, shape.D, shape.R, shape.H
        self.t = {k: dev_bf16(d[k]) for k in ("hcache", "E", "W_lat", "Wg", "Wu", "Wd", "base")}
        self.t["W2t"] = dev_bf16(np.ascontiguousarray(d["W2"].T))  # the library's vocabulary-major layout
        self.am1 = dev(d["am1"])
        self.L = dev(d["L"])
        self.ws = xpress.workspace(xpress.jacobi_workspace_size(N, B, V, D, R, H))
        self.changed = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self, blk_np):
        blk = dev(blk_np.copy())
        self.changed.zero_()
        t = self.t
        xpress.jacobi_pass(blk, self.am1, t["hcache"], t["E"], t["W_lat"], self.L, t["Wg"], t["Wu"], t["Wd"],
                           t["W2t"], t["base"], self.ws, changed=self.changed)
        torch.cuda.synchronize()
        assert xpress.read_error(self.ws) == 0
        return blk.cpu().numpy(), int(self.changed.item())


def check_rows(orc, d, blk_in, blk_out, rows):
    """The token rule on the given rows: each token equals the oracle's, or
    its oracle logit lies within 0.0625 of the oracle row maximum.  Returns
    how many tokens were exactly the oracle's."""
    lat = orc.latent(blk_in, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"])
    B = blk_in.shape[1]
    R = lat.shape[-1]
    flat = lat.reshape(-1, R)
    exact = 0
    for r in rows:
        s = orc.row_logits(flat[r], d["W2"], d["base"][r])
        n, j = divmod(r, B - 1)
        tok = blk_out[n, 1 + j]
        assert s[tok] >= s.max() - TOL, (r, tok, s[tok], s.max())
        exact += int(tok == int(np.argmax(s)))
    return exact


def oracle_pass(orc, d, blk_in):
    """The oracle's own pass on a copy of blk_in."""
    o = blk_in.copy()
    orc.jacobi_pass(o, d["am1"], d["hcache"], d["E"], d["W_lat"], d["L"], d["Wg"], d["Wu"], d["Wd"], d["W2"],
                    d["base"])
    return o


def check_all_rows(orc, d, blk_in, blk_out):
    """Every row of one GPU pass against the oracle run on the same input
    (teacher forcing): slot 0 untouched; each token equal to the oracle's, or
    (a near-tie) its oracle logit within 0.0625 of the row maximum.  Returns
    the oracle's blk and the rows whose token differs from the oracle's."""
    np.testing.assert_array_equal(blk_out[:, 0], blk_in[:, 0])
    o = oracle_pass(orc, d, blk_in)
    B = blk_in.shape[1]
    diff = [int(n) * (B - 1) + int(j) for n, j in np.argwhere(o[:, 1:] != blk_out[:, 1:])]
    if diff:
        assert check_rows(orc, d, blk_in, blk_out, diff) == 0
    return o, diff


SHAPES = [synth.TINY, synth.PassShape("p1", 9, 16, 3000, 256, 128, 256, 31),
          synth.PassShape("p2", 4, 5, 1000, 128, 64, 128, 32),
          synth.PassShape("pdr", 5, 16, 2000, 256, 256, 256, 33),  # D = R, the pages' layout
          synth.PassShape("n200", 200, 16, 4096, 512, 512, 256, 34),  # 3000 rows: D sum unsplit, 12 readout pair rows
          synth.PassShape("n96", 96, 16, 4096, 512, 512, 1536, 35)]  # 12 M tiles; MLP grids above the SM count


@pytest.mark.parametrize("shape", SHAPES, ids=[s.name for s in SHAPES])
def test_pass_parity(orc, shape):
    d = synth.pass_inputs(shape)
    p = Pass(d, shape)
    out, changed = p.run(d["blk"])
    assert changed == int((out != d["blk"]).sum())
    _, diff = check_all_rows(orc, d, d["blk"], out)
    assert len(diff) <= max(1, shape.rows // 50)


def _f(h):
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _trajectory(p, blk0, cap):
    """Host loop of single GPU passes: [blk0, after pass 1, ...], stopping
    after the first pass that changed nothing or after cap passes; plus each
    pass's changed count."""
    hist, counts = [blk0.copy()], []
    while len(counts) < cap:
        out, changed = p.run(hist[-1])
        assert changed == int((out != hist[-1]).sum())
        hist.append(out)
        counts.append(changed)
        if changed == 0:
            break
    return hist, counts


def _exact_pass_inputs(N=4, B=8, V=1000, D=64, R=64, H=64, seed=5):
    """A pass whose every floating-point result is exact on both sides, so the
    GPU's tokens are the oracle's bit for bit and a multi-pass trajectory
    cannot drift (the inputs come from synth.exact_pass_inputs, which states
    the bounds; tests/test_synth.py checks them on the oracle's values)."""
    return synth.exact_pass_inputs(synth.PassShape("exact", N, B, V, D, R, H, seed))


def test_multipass_exact_arithmetic_matches_oracle_trajectory(orc):
    """Jacobi passes to the fixpoint on exact-arithmetic inputs: every pass's
    blk, the per-pass change counts and the pass count equal the oracle's own
    untouched run (no near-tie can move either side), for the host loop of
    single passes and for xp_jacobi_fixpoint."""
    N, B, V, D, R, H = 4, 8, 1000, 64, 64, 64
    shape = synth.PassShape("exact", N, B, V, D, R, H, 5)
    d = _exact_pass_inputs(N, B, V, D, R, H)
    cap = 2 * B
    p = Pass(d, shape)
    hist, counts = _trajectory(p, d["blk"], cap)
    ohist, ocounts = [d["blk"].copy()], []
    while len(ocounts) < cap:
        o = oracle_pass(orc, d, ohist[-1])
        ocounts.append(int((o != ohist[-1]).sum()))
        ohist.append(o)
        if ocounts[-1] == 0:
            break
    assert counts == ocounts
    for q, (g, o) in enumerate(zip(hist, ohist)):
        np.testing.assert_array_equal(g, o, err_msg=f"after pass {q}")
    assert 2 < len(counts) <= B  # the input moves tokens for several passes, and converges (causal mixer)
    got, passes, changed = _fixpoint_run(p, d["blk"], cap)
    assert passes == len(ocounts) and changed == sum(ocounts)
    np.testing.assert_array_equal(got, ohist[-1])
    for got, passes, changed in _fixpoint_graph_runs(p, d["blk"], cap):
        assert passes == len(ocounts) and changed == sum(ocounts)
        np.testing.assert_array_equal(got, ohist[-1])


def test_multipass_teacher_forced_and_fixpoint(orc):
    """Jacobi iteration to a fixpoint on random inputs (base scaled down so
    the readout moves tokens): every row of every pass checked against the
    oracle on the GPU's own input; the per-pass change count equals the
    oracle's on that input up to the near-tie rows of that pass (each can move
    the count by one); the causal invariant (slots 1..p final after pass p)
    holds on the GPU."""
    shape = synth.PassShape("fp", 6, 8, 2000, 128, 64, 128, 41)
    d = synth.pass_inputs(shape)
    d["base"] = synth.to_bf16_bits(_f(d["base"]) * np.float32(0.05))
    d["W2"] = synth.to_bf16_bits(_f(d["W2"]) * np.float32(8.0))
    p = Pass(d, shape)
    hist, counts = _trajectory(p, d["blk"], shape.B + 1)
    assert counts[-1] == 0 and len(counts) <= shape.B
    for q in range(1, len(hist)):
        o, diff = check_all_rows(orc, d, hist[q - 1], hist[q])
        oc = int((o != hist[q - 1]).sum())
        assert abs(oc - counts[q - 1]) <= len(diff), (q, oc, counts[q - 1], diff)
    for q in range(1, len(hist)):
        for r in range(q, len(hist)):
            np.testing.assert_array_equal(hist[r][:, 1:q + 1], hist[q][:, 1:q + 1])


def test_full_size_pass_all_rows(orc):
    """N=32, B=16, V=152064, D=3584, R=512, H=1536: every one of the 480 rows
    against the oracle's pass on the same input."""
    shape = synth.SERVE
    d = synth.pass_inputs(shape)
    p = Pass(d, shape)
    out, changed = p.run(d["blk"])
    assert changed == int((out != d["blk"]).sum())
    _, diff = check_all_rows(orc, d, d["blk"], out)
    print(f"\nfull-size pass: {shape.rows - len(diff)}/{shape.rows} tokens equal to the oracle's; "
          f"near-tie rows {diff}")
    assert len(diff) <= shape.rows // 50


def test_latency_floor_pass_direct_and_graph_replay(orc):
    """N=1 at the serving dims (V=152064, D=3584, R=512, H=1536): one readout
    pair whose second CTA holds only padding rows.  The pass called directly
    and the same pass captured in a CUDA graph, replayed twice from the same
    input, give the oracle's tokens (rule above) and each other's bit for bit
    (the kernels are deterministic)."""
    shape = synth.FLOOR
    d = synth.pass_inputs(shape)
    p = Pass(d, shape)
    out, changed = p.run(d["blk"])
    _, diff = check_all_rows(orc, d, d["blk"], out)
    assert len(diff) <= 1
    t = p.t
    blk = dev(d["blk"].copy())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        xpress.jacobi_pass(blk, p.am1, t["hcache"], t["E"], t["W_lat"], p.L, t["Wg"], t["Wu"], t["Wd"], t["W2t"],
                           t["base"], p.ws, changed=p.changed)
    blk0 = dev(d["blk"].copy())
    for rep in range(2):
        blk.copy_(blk0)
        p.changed.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(blk.cpu().numpy(), out, err_msg=f"replay {rep}")
        assert int(p.changed.item()) == changed
    assert xpress.read_error(p.ws) == 0


def _fixpoint_run(p, blk_np, max_passes):
    blk = dev(blk_np.copy())
    passes = torch.zeros(1, dtype=torch.int32, device="cuda")
    changed = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = p.t
    xpress.jacobi_fixpoint(blk, p.am1, t["hcache"], t["E"], t["W_lat"], p.L, t["Wg"], t["Wu"], t["Wd"], t["W2t"],
                           t["base"], p.ws, passes, max_passes=max_passes, changed=changed)
    torch.cuda.synchronize()
    assert xpress.read_error(p.ws) == 0
    return blk.cpu().numpy(), int(passes.item()), int(changed.item())


def _fixpoint_graph_runs(p, blk_np, max_passes, replays=2):
    """xp_jacobi_fixpoint captured in a CUDA graph (a conditional while node
    whose body is one pass), replayed from blk_np several times: the list of
    (blk, passes, changed) of each replay."""
    blk = dev(blk_np.copy())
    blk0 = dev(blk_np.copy())
    passes = torch.zeros(1, dtype=torch.int32, device="cuda")
    changed = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = p.t
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        xpress.jacobi_fixpoint(blk, p.am1, t["hcache"], t["E"], t["W_lat"], p.L, t["Wg"], t["Wu"], t["Wd"],
                               t["W2t"], t["base"], p.ws, passes, max_passes=max_passes, changed=changed)
    out = []
    for _ in range(replays):
        blk.copy_(blk0)
        changed.zero_()
        passes.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        out.append((blk.cpu().numpy(), int(passes.item()), int(changed.item())))
    assert xpress.read_error(p.ws) == 0
    return out


@pytest.mark.parametrize("cap", [3, 16])
def test_fixpoint_driver_matches_pass_loop(cap):
    """xp_jacobi_fixpoint (all passes enqueued, no host round trip) against the
    host loop of xp_jacobi_pass that stops after the first pass that changed
    nothing: same final blk, same pass count (the kernels are deterministic),
    and the passes after the fixpoint leave blk alone."""
    shape = synth.PassShape("fp", 6, 8, 2000, 128, 64, 128, 41)
    d = synth.pass_inputs(shape)
    d["base"] = synth.to_bf16_bits(_f(d["base"]) * np.float32(0.05))
    d["W2"] = synth.to_bf16_bits(_f(d["W2"]) * np.float32(8.0))
    p = Pass(d, shape)
    hist, counts = _trajectory(p, d["blk"], cap)
    got, passes, changed = _fixpoint_run(p, d["blk"], cap)
    np.testing.assert_array_equal(got, hist[-1])
    assert passes == len(counts) and changed == sum(counts)
    if cap == 16:
        assert len(counts) < cap  # this input converges within B passes


@pytest.mark.parametrize("cap", [1, 3, 16])
def test_fixpoint_captured_while_node_matches_pass_loop(cap):
    """xp_jacobi_fixpoint captured in a CUDA graph runs a conditional while
    node (one pass per iteration, stopped by the readout's last CTA): every
    replay gives the host pass loop's final blk, pass count and change count,
    also when max_passes stops it before the fixpoint (cap 1 and 3)."""
    shape = synth.PassShape("fp", 6, 8, 2000, 128, 64, 128, 41)
    d = synth.pass_inputs(shape)
    d["base"] = synth.to_bf16_bits(_f(d["base"]) * np.float32(0.05))
    d["W2"] = synth.to_bf16_bits(_f(d["W2"]) * np.float32(8.0))
    p = Pass(d, shape)
    hist, counts = _trajectory(p, d["blk"], cap)
    for got, passes, changed in _fixpoint_graph_runs(p, d["blk"], cap, replays=3):
        np.testing.assert_array_equal(got, hist[-1])
        assert passes == len(counts) and changed == sum(counts)


def test_fixpoint_multipass_workload_vs_oracle(orc):
    """The multi-pass workload: N=64, B=16, V=152064, D=3584, R=512, H=1536,
    at most 8 passes.
      * xp_jacobi_fixpoint gives the host pass loop's blk and pass count;
      * every row of every GPU pass is checked against the oracle on the
        GPU's own input (teacher forcing), and each pass's change count equals
        the oracle's on that input up to that pass's near-tie rows;
      * the oracle's own untouched run to its fixpoint: its pass count and
        final blk equal the GPU's whenever no near-tie moved the GPU's
        trajectory; a near-tie that did is shown by the 0.0625 rule above."""
    shape = synth.FIXPOINT
    cap = 8
    d = synth.pass_inputs(shape)
    p = Pass(d, shape)
    hist, counts = _trajectory(p, d["blk"], cap)
    got, passes, _ = _fixpoint_run(p, d["blk"], cap)
    np.testing.assert_array_equal(got, hist[-1])
    assert passes == len(counts)
    for got, passes, changed in _fixpoint_graph_runs(p, d["blk"], cap):
        np.testing.assert_array_equal(got, hist[-1])
        assert passes == len(counts) and changed == sum(counts)
    near = []
    ohist, ocounts = [d["blk"].copy()], []
    for q in range(1, len(hist)):
        o, diff = check_all_rows(orc, d, hist[q - 1], hist[q])
        oc = int((o != hist[q - 1]).sum())
        assert abs(oc - counts[q - 1]) <= len(diff), (q, oc, counts[q - 1], diff)
        near += [(q, r) for r in diff]
        if np.array_equal(ohist[-1], hist[q - 1]) and len(ocounts) == q - 1 and (not ocounts or ocounts[-1]):
            ohist.append(o)  # the untouched oracle had the GPU's input: same pass
            ocounts.append(oc)
    while len(ocounts) < cap and ocounts[-1] != 0:  # the oracle's run past a divergence
        o = oracle_pass(orc, d, ohist[-1])
        ocounts.append(int((o != ohist[-1]).sum()))
        ohist.append(o)
    print(f"\nmulti-pass workload: GPU {len(counts)} passes {counts}; oracle {len(ocounts)} passes {ocounts}; "
          f"near-tie (pass, row) {near}")
    if not near:
        assert ocounts == counts
        np.testing.assert_array_equal(ohist[-1], hist[-1])
