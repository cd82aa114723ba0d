"""xp_add_argmax_noalloc: the add-argmax on the library's fixed scratch.

Collected last on purpose: it must give the workspace entry point's answer
whether it runs alone or after every other test has used the device.
"""
import ctypes

import pytest
import torch

from gpu_util import padded_bf16
from speculative_decoding_gb300 import synth
from speculative_decoding_gb300 import xpress as X


def test_noalloc_limit_declared_and_enforced():
    # the Python constant mirrors the header's limit
    text = open(X.HEADER).read()
    assert f"#define XP_ADD_ARGMAX_NOALLOC_MAX_ROWS {X.NOALLOC_MAX_ROWS}" in text
    L = X.lib()
    fake = ctypes.c_void_p(1 << 20)
    B = 2
    N = X.NOALLOC_MAX_ROWS + 1  # rows = N*(B-1) one above the limit
    st = L.xp_add_argmax_noalloc(fake, 4096, fake, 4096, N * (B - 1), 4096, fake, N, B, None)
    assert st == X.XP_ERR_SHAPE
    # empty input is a no-op that touches nothing
    assert L.xp_add_argmax_noalloc(None, 8, None, 8, 0, 8, None, 0, 2, None) == X.XP_OK


def _inputs(N, B, V, seed):
    # rows padded to a multiple of 8 elements (the entry points' stride
    # rule), so a ragged V is a strided view
    rows = N * (B - 1)
    d = synth.argmax_inputs(rows, V, N, B, seed=seed, tie_frac=0.1)
    ld = (V + 7) // 8 * 8
    return rows, padded_bf16(d["base"], ld), padded_bf16(d["bias"], ld)


@pytest.mark.gpu
@pytest.mark.parametrize("N,B,V", [(3, 5, 1000), (32, 16, 152064), (546, 16, 32003)])
def test_noalloc_matches_workspace_entry(N, B, V):
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    rows, base, bias = _inputs(N, B, V, seed=7 + N)
    blk_ref = torch.full((N, B), -1, dtype=torch.int64, device=dev)
    ws = X.workspace(X.add_argmax_workspace_size(rows, V), dev)
    X.add_argmax(base, bias, blk_ref, ws)
    for call in range(2):  # two calls in a row: the scratch must be clean for the second
        blk = torch.full((N, B), -1, dtype=torch.int64, device=dev)
        X.add_argmax_noalloc(base, bias, blk)
        torch.cuda.synchronize()
        assert torch.equal(blk, blk_ref), f"call {call}"
    assert (blk_ref[:, 0] == -1).all()  # column 0 is never written


@pytest.mark.gpu
def test_noalloc_second_call_after_different_shape():
    # a large call followed by a small one reuses the same scratch rows
    dev = torch.device("cuda:0")
    for (N, B, V, seed) in [(500, 16, 4099, 11), (2, 3, 300, 12), (500, 16, 4099, 13)]:
        rows, base, bias = _inputs(N, B, V, seed)
        ws = X.workspace(X.add_argmax_workspace_size(rows, V), dev)
        blk_ref = torch.zeros((N, B), dtype=torch.int64, device=dev)
        X.add_argmax(base, bias, blk_ref, ws)
        blk = torch.zeros((N, B), dtype=torch.int64, device=dev)
        X.add_argmax_noalloc(base, bias, blk)
        torch.cuda.synchronize()
        assert torch.equal(blk, blk_ref)
