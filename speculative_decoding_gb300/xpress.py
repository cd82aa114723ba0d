"""Thin Python binding of libxpress.so (argument marshalling only).

Every function takes torch CUDA tensors, checks dtype/device/contiguity, and
passes raw device pointers plus the current CUDA stream to the C entry point of
the same name (``latent_pass`` and ``jacobi_pass`` call the ``_ex`` forms, which
also take the MLP schedule; see include/xpress.h for the contracts).  Nothing
here computes: if the library is missing, ``lib()`` raises -- there is no
fallback.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libxpress.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "xpress.h")

XP_OK, XP_ERR_NULL, XP_ERR_SHAPE, XP_ERR_ALIGN, XP_ERR_WORKSPACE, XP_ERR_LAUNCH, XP_ERR_UNSUPPORTED = range(7)
XP_DEVERR_TOKEN, XP_DEVERR_TIMEOUT = 1, 2
NOALLOC_MAX_ROWS = 8192  # XP_ADD_ARGMAX_NOALLOC_MAX_ROWS


class XpressError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t

_SIGS = {
    "xp_status_string": (ctypes.c_char_p, [ctypes.c_int32]),
    "xp_version": (ctypes.c_int32, []),
    "xp_add_argmax_workspace_size": (_sz, [_i64, _i64]),
    "xp_add_argmax": (ctypes.c_int32, [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _sz, _vp]),
    "xp_add_argmax_noalloc": (ctypes.c_int32, [_vp, _i64, _vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp]),
    "xp_topc_argmax": (ctypes.c_int32, [_vp, _vp, _vp, _i64, _i64, _vp, _i64, _i64, _vp]),
    "xp_latent_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i64]),
    "xp_latent_pass": (ctypes.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _i64, _i64, _i64, _i64, _i64, _i64, _vp, _sz, _vp]),
    "xp_latent_pass_ex": (ctypes.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                           _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, _vp, _sz, _vp]),
    "xp_readout_workspace_size": (_sz, [_i64, _i64]),
    "xp_readout_argmax": (ctypes.c_int32, [_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _i64, _i64, _vp,
                                           _vp, _sz, _vp]),
    "xp_jacobi_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i64, _i64]),
    "xp_jacobi_pass": (ctypes.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                        _i64, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "xp_jacobi_pass_ex": (ctypes.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                           _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, _vp, _vp, _sz,
                                           _vp]),
    "xp_jacobi_fixpoint": (ctypes.c_int32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64,
                                            _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int32, _vp, _vp, _vp,
                                            _sz, _vp]),
    "xp_read_error": (ctypes.c_int32, [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]),
    "xp_selftest_wait_timeout": (ctypes.c_int32, [_vp, _sz, ctypes.c_uint32, _vp]),
}


def declared_symbols() -> list[str]:
    """Names of the functions include/xpress.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^XP_API\s+[\w\s\*]+?\b(xp_\w+)\s*\(", text, flags=re.M)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m speculative_decoding_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(st: int) -> str:
    return lib().xp_status_string(st).decode()


def _check(st: int) -> None:
    if st != XP_OK:
        raise XpressError(st, status_string(st))


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t, dtype, name, contiguous=True):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _rowmajor(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit column stride")
    return t.stride(0)


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed uint8 device buffer of ``nbytes`` (rounded up to 256)."""
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device or "cuda")


# --- entry points -----------------------------------------------------------

def add_argmax_workspace_size(rows: int, V: int) -> int:
    return int(lib().xp_add_argmax_workspace_size(rows, V))


def add_argmax(base, bias, blk, ws, stream=None) -> None:
    """blk[n, 1+j] = lowest argmax_v bf16(base[r, v] + bias[r, v]), r = n*(B-1)+j."""
    rows, V = base.shape
    N, B = blk.shape
    _check(lib().xp_add_argmax(_ptr(base, torch.bfloat16, "base", False), _rowmajor(base, "base"),
                               _ptr(bias, torch.bfloat16, "bias", False), _rowmajor(bias, "bias"),
                               rows, V, _ptr(blk, torch.int64, "blk"), N, B,
                               _ptr(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)))


def add_argmax_noalloc(base, bias, blk, stream=None) -> None:
    """add_argmax on the library's fixed scratch: no workspace, at most
    NOALLOC_MAX_ROWS rows, and calls that overlap in time race."""
    rows, V = base.shape
    N, B = blk.shape
    _check(lib().xp_add_argmax_noalloc(_ptr(base, torch.bfloat16, "base", False), _rowmajor(base, "base"),
                                       _ptr(bias, torch.bfloat16, "bias", False), _rowmajor(bias, "bias"),
                                       rows, V, _ptr(blk, torch.int64, "blk"), N, B, _stream(stream)))


def topc_argmax(base_c, bias_c, cand, blk, stream=None) -> None:
    """blk[n, 1+j] = cand[r, p*], p* the lowest argmax_p bf16(base_c[r, p] + bias_c[r, p]);
    base_c, bias_c, cand are [N, B-1, C] (or [rows, C])."""
    C = base_c.shape[-1]
    rows = base_c.numel() // C if C else 0
    N, B = blk.shape
    _check(lib().xp_topc_argmax(_ptr(base_c, torch.bfloat16, "base_c"), _ptr(bias_c, torch.bfloat16, "bias_c"),
                                _ptr(cand, torch.int64, "cand"), rows, C, _ptr(blk, torch.int64, "blk"), N, B,
                                _stream(stream)))


def latent_workspace_size(N: int, B: int, D: int, R: int, H: int) -> int:
    return int(lib().xp_latent_workspace_size(N, B, D, R, H))


def latent_pass(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, lat_out, ws, stream=None, do_mlp=True) -> None:
    """The latent stage into lat_out [N, B-1, R].  ``do_mlp`` False selects the
    GEMM schedule (bf16 g, v and residual; see xp_latent_pass_ex)."""
    N, B = blk.shape
    V, D = E.shape
    R = W_lat.shape[1]
    H = Wg.shape[1]
    bf = torch.bfloat16
    _check(lib().xp_latent_pass_ex(_ptr(blk, torch.int64, "blk"), _ptr(am1, torch.int64, "am1"),
                                   _ptr(hcache, bf, "hcache"), _ptr(E, bf, "E"), _ptr(W_lat, bf, "W_lat"),
                                   _ptr(L, torch.float32, "L"), _ptr(Wg, bf, "Wg"), _ptr(Wu, bf, "Wu"),
                                   _ptr(Wd, bf, "Wd"), _ptr(lat_out, bf, "lat_out"), N, B, V, D, R, H,
                                   1 if do_mlp else 0, _ptr(ws, torch.uint8, "workspace"), ws.numel(),
                                   _stream(stream)))


def readout_workspace_size(rows: int, V: int) -> int:
    return int(lib().xp_readout_workspace_size(rows, V))


def readout_argmax(lat, W2t, base, blk, ws, changed=None, stream=None) -> None:
    """blk[n, 1+j] = lowest argmax_v bf16(base[r, v] + bf16(lat[r] . W2t[v])); W2t is [V, R]."""
    rows, R = lat.shape
    V = W2t.shape[0]
    N, B = blk.shape
    bf = torch.bfloat16
    _check(lib().xp_readout_argmax(_ptr(lat, bf, "lat"), _ptr(W2t, bf, "W2t"),
                                   _ptr(base, bf, "base", False), _rowmajor(base, "base"), rows, V, R,
                                   _ptr(blk, torch.int64, "blk"), N, B, _ptr(changed, torch.int32, "changed"),
                                   _ptr(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)))


def jacobi_workspace_size(N: int, B: int, V: int, D: int, R: int, H: int) -> int:
    return int(lib().xp_jacobi_workspace_size(N, B, V, D, R, H))


def jacobi_pass(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2t, base, ws, changed=None, stream=None,
                do_mlp=True) -> None:
    """One pass in place on blk; W2t is the readout weight stored [V, R].
    ``do_mlp`` as in latent_pass."""
    N, B = blk.shape
    V, D = E.shape
    R = W_lat.shape[1]
    H = Wg.shape[1]
    bf = torch.bfloat16
    _check(lib().xp_jacobi_pass_ex(_ptr(blk, torch.int64, "blk"), _ptr(am1, torch.int64, "am1"),
                                   _ptr(hcache, bf, "hcache"), _ptr(E, bf, "E"), _ptr(W_lat, bf, "W_lat"),
                                   _ptr(L, torch.float32, "L"), _ptr(Wg, bf, "Wg"), _ptr(Wu, bf, "Wu"),
                                   _ptr(Wd, bf, "Wd"), _ptr(W2t, bf, "W2t"), _ptr(base, bf, "base", False),
                                   _rowmajor(base, "base"), N, B, V, D, R, H, 1 if do_mlp else 0,
                                   _ptr(changed, torch.int32, "changed"),
                                   _ptr(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)))


def jacobi_fixpoint(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, W2t, base, ws, passes, max_passes=8,
                    changed=None, stream=None) -> None:
    """Passes in place on blk until one changes nothing (counted) or max_passes;
    the count lands in the device int32 tensor ``passes`` (no host sync)."""
    N, B = blk.shape
    V, D = E.shape
    R = W_lat.shape[1]
    H = Wg.shape[1]
    bf = torch.bfloat16
    _check(lib().xp_jacobi_fixpoint(_ptr(blk, torch.int64, "blk"), _ptr(am1, torch.int64, "am1"),
                                    _ptr(hcache, bf, "hcache"), _ptr(E, bf, "E"), _ptr(W_lat, bf, "W_lat"),
                                    _ptr(L, torch.float32, "L"), _ptr(Wg, bf, "Wg"), _ptr(Wu, bf, "Wu"),
                                    _ptr(Wd, bf, "Wd"), _ptr(W2t, bf, "W2t"), _ptr(base, bf, "base", False),
                                    _rowmajor(base, "base"), N, B, V, D, R, H, int(max_passes),
                                    _ptr(passes, torch.int32, "passes"), _ptr(changed, torch.int32, "changed"),
                                    _ptr(ws, torch.uint8, "workspace"), ws.numel(), _stream(stream)))


def read_error(ws, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().xp_read_error(_ptr(ws, torch.uint8, "workspace"), _stream(stream), ctypes.byref(bits)))
    return int(bits.value)


def selftest_wait_timeout(ws, limit_us: int = 1000, stream=None) -> None:
    """Enqueue the failure-detection self-test: a bounded device wait that runs
    out after limit_us and sets XP_DEVERR_TIMEOUT (read it with read_error)."""
    _check(lib().xp_selftest_wait_timeout(_ptr(ws, torch.uint8, "workspace"), ws.numel(), limit_us,
                                          _stream(stream)))
