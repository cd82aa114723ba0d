"""Pins of the oracle's bf16 rounding (CPU only).

The pass rounds to bf16 with round-to-nearest-even wherever the vLLM
``xpress.kernels`` pages cast to the input dtype (``.to(dtype)`` in
``_xpress_add_argmax_partial_kernel`` and ``_xpress_latent_kernel``)."""

import os
import struct
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

from exact import round_bf16

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.slow
def test_exhaustive_rounding_and_sum(orc, tmp_path):
    """Every fp32 pattern: bit-trick rounding == value-arithmetic rounding.
    Every pair of finite bf16 values: fp32 add + RNE == correctly rounded sum
    (so a kernel's fp32 add followed by a bf16 convert computes the pages'
    rounded bf16 sum exactly)."""
    exe = tmp_path / "exh"
    subprocess.run(["gcc", "-O2", "-fopenmp", os.path.join(HERE, "csrc", "exhaustive_bf16.c"),
                    "-o", str(exe), "-ldl"], check=True)
    r = subprocess.run([str(exe), orc.build()], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("OK 4294967296")


def test_rounding_matches_torch_sample(orc):
    """torch's fp32 -> bf16 cast is round-to-nearest-even: a library pin."""
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    ours = orc.bf16_from_float_bits(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


@pytest.mark.parametrize("x", [1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-8 + 2**-30, -(1.0 + 2**-8),
                               3.0e38, 3.4e38, 2**-133, 2**-134, 3 * 2**-135, 0.0, -0.0,
                               255.5, 256.5, 16.03125, 15.96875])
def test_rounding_special_values(orc, x):
    """Ties to even, overflow to inf, subnormals, signed zero, against a
    pure-Python Fraction rounding."""
    got = orc.bf16_from_double(np.array([x]))[0]
    want = round_bf16(Fraction(x))
    got_f = struct.unpack("<f", struct.pack("<I", int(got) << 16))[0]
    assert got_f == float(want)
    if x == 0.0:
        assert (int(got) >> 15) == (1 if str(x).startswith("-") else 0)


def test_tie_to_even_cases(orc):
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even mantissa is 1.0
    assert orc.bf16_from_double(np.array([1.0 + 2**-8]))[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even)
    assert orc.bf16_from_double(np.array([1.0 + 3 * 2**-8]))[0] == 0x3F82
    assert orc.bf16_from_float_bits(np.array([1.0 + 3 * 2**-8], np.float32))[0] == 0x3F82
