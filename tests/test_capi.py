"""The C-ABI library without a GPU: it loads, exports every symbol
include/xpress.h declares, and rejects bad arguments on the host before any
CUDA call (so these checks run on a CPU-only machine)."""

import ctypes
import re

import pytest

from speculative_decoding_gb300 import build, xpress


@pytest.fixture(scope="module")
def L():
    build.build()
    return xpress.lib()


def test_exports_every_declared_symbol(L):
    names = xpress.declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(xpress._SIGS), "binding signatures cover exactly the header"


def test_status_strings(L):
    for st in range(7):
        assert xpress.status_string(st).startswith("XP_")
    assert "unknown" in xpress.status_string(99)
    assert L.xp_version() >= 100


def test_workspace_sizes_monotone(L):
    a = xpress.add_argmax_workspace_size(480, 152064)
    assert a >= 256 + 480 * 12 and a % 256 == 0
    assert xpress.add_argmax_workspace_size(960, 152064) > a


FAKE = 1 << 20   # a non-null, 256-aligned dummy address; never dereferenced


def _aa(rows=6, V=1000, N=2, B=4, ld=1000, base=FAKE, bias=FAKE, blk=FAKE, ws=FAKE, nbytes=1 << 20):
    return xpress.lib().xp_add_argmax(base, ld, bias, ld, rows, V, blk, N, B, ws, nbytes, None)


def test_add_argmax_host_validation(L):
    assert _aa(rows=5) == xpress.XP_ERR_SHAPE                 # rows != N*(B-1)
    assert _aa(B=1, rows=0) == xpress.XP_ERR_SHAPE
    assert _aa(V=0) == xpress.XP_ERR_SHAPE
    assert _aa(ld=999) == xpress.XP_ERR_SHAPE                 # ld < V
    assert _aa(N=0, rows=0) == xpress.XP_OK                   # empty: no-op
    assert _aa(base=0) == xpress.XP_ERR_NULL
    assert _aa(ws=0) == xpress.XP_ERR_NULL
    assert _aa(base=FAKE + 8) == xpress.XP_ERR_ALIGN
    assert _aa(ld=1004) == xpress.XP_ERR_ALIGN
    assert _aa(ws=FAKE + 16) == xpress.XP_ERR_WORKSPACE
    assert _aa(nbytes=64) == xpress.XP_ERR_WORKSPACE


def test_read_error_validation(L):
    bits = ctypes.c_uint32()
    assert L.xp_read_error(None, None, ctypes.byref(bits)) == xpress.XP_ERR_NULL
    assert L.xp_read_error(FAKE + 1, None, ctypes.byref(bits)) == xpress.XP_ERR_WORKSPACE


def _lp(L, do_mlp=0, N=2, B=4, V=1000, D=64, R=32, H=64, lat=FAKE, ws=FAKE, nbytes=1 << 24, ptr=FAKE):
    return L.xp_latent_pass_ex(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, lat, N, B, V, D, R, H, do_mlp, ws,
                               nbytes, None)


def _jp(L, do_mlp=0, N=2, B=4, V=1000, D=64, R=32, H=64, ld=1000, ws=FAKE, nbytes=1 << 24, ptr=FAKE):
    return L.xp_jacobi_pass_ex(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ld, N, B, V, D, R, H, do_mlp,
                               None, ws, nbytes, None)


def test_schedule_entry_points_host_validation(L):
    """The do_mlp entry points reject bad arguments before any CUDA call.
    (No call here passes every check: on a GPU machine that would launch
    kernels on the dummy addresses.)"""
    for f in (_lp, _jp):
        assert f(L, do_mlp=2) == xpress.XP_ERR_SHAPE
        assert f(L, do_mlp=-1) == xpress.XP_ERR_SHAPE
        assert f(L, B=1) == xpress.XP_ERR_SHAPE
        assert f(L, B=17) == xpress.XP_ERR_SHAPE
        assert f(L, R=24) == xpress.XP_ERR_ALIGN        # R a multiple of 16
        assert f(L, H=96) == xpress.XP_ERR_ALIGN        # H a multiple of 64
        assert f(L, ptr=0) == xpress.XP_ERR_NULL
        assert f(L, ws=FAKE + 16) == xpress.XP_ERR_WORKSPACE
        assert f(L, nbytes=64) == xpress.XP_ERR_WORKSPACE
    assert _lp(L, lat=0) == xpress.XP_ERR_NULL
    assert _lp(L, lat=FAKE + 8) == xpress.XP_ERR_ALIGN
    assert _jp(L, ld=999) == xpress.XP_ERR_SHAPE        # ld_base < V
    assert _jp(L, ld=1004) == xpress.XP_ERR_ALIGN       # ld_base a multiple of 8
    assert _lp(L, N=0) == xpress.XP_OK                  # empty: no-op


def test_readout_weight_parameter_is_named_transposed():
    """The readout weight crosses the boundary vocabulary-major ([V, R], the
    pages' W2 [R, V] transposed).  A raw pointer carries no shape, so the
    parameter's name is what tells a caller: every declaration that takes it
    must call it d_W2t, and its comment must state the [V,R] layout."""
    text = open(xpress.HEADER).read()
    decls = re.findall(r"XP_API[^;]*?\b(xp_\w+)\s*\(([^;]*?)\);", text, flags=re.S)
    takers = {}
    for name, params in decls:
        w2 = re.findall(r"\b(d_W2\w*)\b", params)
        if w2:
            takers[name] = w2
    assert {"xp_readout_argmax", "xp_jacobi_pass", "xp_jacobi_pass_ex", "xp_jacobi_fixpoint"} <= set(takers)
    for name, params in takers.items():
        assert params == ["d_W2t"], (name, params)
        # the comment block right above the declaration names the layout
        head = text[:text.index(f"{name}(")]
        block = head[head.rindex("/*"):]
        assert "d_W2t" in block and "[V,R]" in block, name
