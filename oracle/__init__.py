"""CPU oracle for one XPress Jacobi draft pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
product path (``speculative_decoding_gb300``) never imports it, and the two
share no code: the oracle is the plain definition in ``xp_oracle.c``, accumulated
in double, with bf16 rounding exactly where the vLLM ``xpress.kernels`` pages
round (module docstring; ``_xpress_add_argmax_partial_kernel``;
``_xpress_latent_kernel``; ``fused_topc_argmax_to_blk``).

Arrays are numpy: bf16 tensors travel as ``uint16`` bit patterns, tokens as
``int64``, the mixer ``L`` as ``float32``.  Every function checks shapes and
returns/raises on the oracle's status codes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "xp_oracle.c")
_LIB = os.path.join(_HERE, "libxp_oracle.so")

_ERRORS = {-1: "bad argument", -2: "token out of range", -3: "non-finite input"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile ``xp_oracle.c`` into ``libxp_oracle.so`` next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_bf16_from_float.restype = ctypes.c_uint16
        L.orc_bf16_from_float.argtypes = [ctypes.c_float]
        L.orc_double_from_bf16.restype = ctypes.c_double
        L.orc_double_from_bf16.argtypes = [ctypes.c_uint16]
        L.orc_bf16_add.restype = ctypes.c_uint16
        L.orc_bf16_add.argtypes = [ctypes.c_uint16, ctypes.c_uint16]
        L.orc_bf16_from_float_array.argtypes = [_f32p, _u16p, _i64]
        L.orc_bf16_from_double_array.argtypes = [_f64p, _u16p, _i64]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_add_argmax.argtypes = [_u16p, _i64, _u16p, _i64, _i64, _i64, _i64p, _i64, _i64]
        L.orc_topc_argmax.argtypes = [_u16p, _u16p, _i64p, _i64, _i64, _i64p, _i64, _i64]
        L.orc_latent.argtypes = [_i64p, _i64p, _u16p, _u16p, _u16p, _f32p, _u16p, _u16p, _u16p, _u16p,
                                 _i64, _i64, _i64, _i64, _i64, _i64, _f64p, _i64, _i64]
        L.orc_row_logits.argtypes = [_u16p, _u16p, _u16p, _i64, _i64, _f64p]
        L.orc_readout_bias.argtypes = [_u16p, _u16p, _i64, _i64, _i64, _u16p]
        L.orc_jacobi_pass.argtypes = [_i64p, _i64p, _u16p, _u16p, _u16p, _f32p, _u16p, _u16p, _u16p,
                                      _u16p, _u16p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64p]
        L.orc_latent_ex.argtypes = [_i64p, _i64p, _u16p, _u16p, _u16p, _f32p, _u16p, _u16p, _u16p, _u16p,
                                    _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f64p, _i64, _i64]
        L.orc_jacobi_pass_ex.argtypes = [_i64p, _i64p, _u16p, _u16p, _u16p, _f32p, _u16p, _u16p, _u16p,
                                         _u16p, _u16p, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64p]
        for name in ("orc_add_argmax", "orc_topc_argmax", "orc_latent", "orc_row_logits",
                     "orc_readout_bias", "orc_jacobi_pass", "orc_latent_ex", "orc_jacobi_pass_ex"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray, dtype, ptype):
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("arrays must be C-contiguous")
    return a.ctypes.data_as(ptype)


def _check(status: int) -> None:
    if status != 0:
        raise OracleError(_ERRORS.get(status, f"status {status}"))


def num_threads() -> int:
    return int(lib().orc_num_threads())


# --- bf16 helpers ---------------------------------------------------------

def bf16_from_float_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even on the bit pattern."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_float_array(_p(x, np.float32, _f32p), _p(out, np.uint16, _u16p), x.size)
    return out


def bf16_from_double(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bits, round to nearest even by arithmetic on the value."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_double_array(_p(x, np.float64, _f64p), _p(out, np.uint16, _u16p), x.size)
    return out


def bf16_to_float(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_add(a: int, b: int) -> int:
    return int(lib().orc_bf16_add(a, b))


# --- the method -----------------------------------------------------------

def add_argmax(base: np.ndarray, bias: np.ndarray, blk: np.ndarray) -> None:
    """blk[n, 1+b] = argmax_v bf16(base[r, v] + bias[r, v]), r = n*(B-1)+b (in place)."""
    rows, V = base.shape
    N, B = blk.shape
    _check(lib().orc_add_argmax(_p(base, np.uint16, _u16p), base.strides[0] // 2,
                                _p(bias, np.uint16, _u16p), bias.strides[0] // 2, rows, V,
                                _p(blk, np.int64, _i64p), N, B))


def topc_argmax(base_c: np.ndarray, bias_c: np.ndarray, cand: np.ndarray, blk: np.ndarray) -> None:
    """Top-C variant: blk[n, 1+b] = cand[r, argmax_c bf16(base_c + bias_c)]."""
    rows, C = base_c.shape
    N, B = blk.shape
    _check(lib().orc_topc_argmax(_p(base_c, np.uint16, _u16p), _p(bias_c, np.uint16, _u16p),
                                 _p(cand, np.int64, _i64p), rows, C, _p(blk, np.int64, _i64p), N, B))


def latent(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, blocks=None, want_u=False, do_mlp=True):
    """Latent stage.  Returns lat_out [N, B-1, R] bf16 bits (and the mixer
    output u [N, B, R] float64 when ``want_u``).  ``blocks=(lo, hi)`` limits the
    work to blocks lo..hi-1; the other rows of the outputs are left zero.
    ``do_mlp`` False selects the GEMM schedule of ``xpress_latent_pass``
    (bf16 u handed back, then u @ wgu_t, silu_and_mul, addmm_ in bf16)."""
    N, B = blk.shape
    V, D = E.shape
    R = W_lat.shape[1]
    H = Wg.shape[1]
    assert hcache.shape == (N, B, R) and W_lat.shape == (D, R) and L.shape == (B, B, R)
    assert Wg.shape == (R, H) and Wu.shape == (R, H) and Wd.shape == (H, R) and am1.shape == (N,)
    lo, hi = blocks if blocks is not None else (0, N)
    lat = np.zeros((N, B - 1, R), np.uint16)
    u = np.zeros((N, B, R), np.float64) if want_u else None
    _check(lib().orc_latent_ex(_p(blk, np.int64, _i64p), _p(am1, np.int64, _i64p),
                               _p(hcache, np.uint16, _u16p), _p(E, np.uint16, _u16p),
                               _p(W_lat, np.uint16, _u16p), _p(L, np.float32, _f32p),
                               _p(Wg, np.uint16, _u16p), _p(Wu, np.uint16, _u16p), _p(Wd, np.uint16, _u16p),
                               _p(lat, np.uint16, _u16p), N, B, V, D, R, H, 1 if do_mlp else 0,
                               _p(u, np.float64, _f64p) if want_u else None, lo, hi))
    return (lat, u) if want_u else lat


def readout_bias(lat: np.ndarray, W2: np.ndarray) -> np.ndarray:
    """bias = bf16(lat @ W2), lat [rows, R], W2 [R, V]; bf16 bits."""
    rows, R = lat.shape
    V = W2.shape[1]
    out = np.empty((rows, V), np.uint16)
    _check(lib().orc_readout_bias(_p(lat, np.uint16, _u16p), _p(W2, np.uint16, _u16p), rows, R, V,
                                  _p(out, np.uint16, _u16p)))
    return out


def row_logits(lat_row: np.ndarray, W2: np.ndarray, base_row: np.ndarray) -> np.ndarray:
    """s[v] = bf16(base[v] + bf16(lat_row . W2[:, v])) for one row, float64."""
    R, V = W2.shape
    out = np.empty(V, np.float64)
    _check(lib().orc_row_logits(_p(np.ascontiguousarray(lat_row), np.uint16, _u16p),
                                _p(W2, np.uint16, _u16p),
                                _p(np.ascontiguousarray(base_row), np.uint16, _u16p), R, V,
                                _p(out, np.float64, _f64p)))
    return out


def jacobi_pass(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2, base, do_mlp=True) -> int:
    """One pass in place on ``blk``; returns the number of slots that changed.
    ``do_mlp`` as in ``latent``."""
    N, B = blk.shape
    V, D = E.shape
    R = W_lat.shape[1]
    H = Wg.shape[1]
    changed = np.zeros(1, np.int64)
    _check(lib().orc_jacobi_pass_ex(_p(blk, np.int64, _i64p), _p(am1, np.int64, _i64p),
                                    _p(hcache, np.uint16, _u16p), _p(E, np.uint16, _u16p),
                                    _p(W_lat, np.uint16, _u16p), _p(L, np.float32, _f32p),
                                    _p(Wg, np.uint16, _u16p), _p(Wu, np.uint16, _u16p),
                                    _p(Wd, np.uint16, _u16p), _p(W2, np.uint16, _u16p),
                                    _p(base, np.uint16, _u16p), base.strides[0] // 2,
                                    N, B, V, D, R, H, 1 if do_mlp else 0, _p(changed, np.int64, _i64p)))
    return int(changed[0])


def jacobi_to_fixpoint(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2, base, max_passes=8):
    """Repeat the pass in place until a pass changes nothing or ``max_passes``
    passes ran.  Returns (passes, per-pass changed counts); the count includes
    the final pass that changed nothing."""
    counts = []
    for _ in range(max_passes):
        c = jacobi_pass(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2, base)
        counts.append(c)
        if c == 0:
            break
    return len(counts), counts
