"""Pins for the oracle's own binary32 -> fp16 / bf16 rounding and the decoders.

- Format facts the pages print (fp16's largest finite value 65504 and smallest
  normal 2^-14; 11 against 8 significand bits): "Mixed-Precision Kernels"
  sections "The Precision Hierarchy and What Each Format Costs" and "When It
  Falls Down"; "Precision" section "Dtype policy".  Stored in golden/formats.json.
- Every one of the 2^32 binary32 inputs against the compiler's _Float16 and
  __bf16 conversions (round to nearest, ties to even), in a native harness.
- Every 16-bit pattern decoded against numpy's float16 and torch's bfloat16.
"""
import math
import os
import platform
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle_pins import golden

HERE = os.path.dirname(os.path.abspath(__file__))


def check_page_format_facts(L):
    g = golden("formats.json")
    fmax = g["f16_max_finite"]
    assert L.oracle_f32_to_f16(fmax) == 0x7BFF
    assert L.oracle_f16_to_f32(0x7BFF) == fmax
    # beyond the largest finite value: 65519 still rounds down, 65520 is the tie that overflows
    assert L.oracle_f32_to_f16(65519.0) == 0x7BFF
    assert L.oracle_f32_to_f16(65520.0) == 0x7C00
    assert L.oracle_f32_to_f16(-70000.0) == 0xFC00
    tiny = 2.0 ** g["f16_min_normal_log2"]
    assert L.oracle_f32_to_f16(tiny) == 0x0400
    assert L.oracle_f16_to_f32(0x0400) == tiny
    assert L.oracle_f32_to_f16(tiny / 2) == 0x0200  # subnormal below the smallest normal
    # significand widths: 1 + 2^-10 is an fp16 value but not a bf16 one; 1 + 2^-7 is both
    p16, pb = g["significand_bits"]["f16"], g["significand_bits"]["bf16"]
    one_16 = 1.0 + 2.0 ** -(p16 - 1)
    assert L.oracle_f16_to_f32(L.oracle_f32_to_f16(one_16)) == one_16
    assert L.oracle_bf16_to_f32(L.oracle_f32_to_bf16(one_16)) == 1.0
    one_b = 1.0 + 2.0 ** -(pb - 1)
    assert L.oracle_bf16_to_f32(L.oracle_f32_to_bf16(one_b)) == one_b
    # bf16 shares binary32's exponent range: no overflow below binary32's top binade
    assert g["bf16_exponent_width_equals_f32"]
    assert L.oracle_bf16_to_f32(L.oracle_f32_to_bf16(1e38)) == pytest.approx(1e38, rel=2 ** -8)


def check_converter_boundaries(L):
    f16 = L.oracle_f32_to_f16
    bf = L.oracle_f32_to_bf16
    # ties to even in the normal range
    assert f16(1.0 + 2.0 ** -11) == 0x3C00            # halfway 1 .. 1+2^-10 -> 1
    assert f16(1.0 + 3 * 2.0 ** -11) == 0x3C02        # halfway 1+2^-10 .. 1+2^-9 -> even
    assert bf(1.0 + 2.0 ** -8) == 0x3F80
    assert bf(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # subnormal ties and underflow
    assert f16(2.0 ** -25) == 0x0000                  # half the smallest subnormal -> 0 (even)
    assert f16(3 * 2.0 ** -25) == 0x0002              # 1.5 subnormal quanta -> 2 (even)
    assert f16(-(2.0 ** -26)) == 0x8000               # signed zero
    assert bf(2.0 ** -134) == 0x0000                  # half bf16's smallest subnormal
    assert bf(3 * 2.0 ** -134) == 0x0002
    # binade crossing by rounding
    assert f16(2047.5) == 0x6800                      # 2047.5 -> 2048 (tie, even)
    assert bf(float(np.float32(3.3961514e38))) == 0x7F7F  # largest finite bf16
    assert bf(float(np.finfo(np.float32).max)) == 0x7F80  # binary32 max rounds to inf in bf16
    # specials
    assert f16(math.inf) == 0x7C00 and f16(-math.inf) == 0xFC00
    assert (f16(math.nan) & 0x7C00) == 0x7C00 and (f16(math.nan) & 0x03FF)
    assert (bf(math.nan) & 0x7F80) == 0x7F80 and (bf(math.nan) & 0x007F)


def test_page_format_facts():
    check_page_format_facts(oracle.lib())


def test_converter_boundaries():
    check_converter_boundaries(oracle.lib())


def test_f16_matches_numpy_on_a_sample():
    L = oracle.lib()
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    for v, want in zip(vals, ref):
        got = L.oracle_f32_to_f16(float(v))
        if np.isnan(v):
            assert (got & 0x7C00) == 0x7C00 and (got & 0x3FF)
        else:
            assert got == want, f"{v!r}: {got:#06x} vs numpy {want:#06x}"


def test_decoders_exhaustive():
    L = oracle.lib()
    pats = np.arange(65536, dtype=np.uint16)
    f16_ref = pats.view(np.float16).astype(np.float32)
    bf_ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    for p in range(65536):
        a, b = L.oracle_f16_to_f32(p), L.oracle_bf16_to_f32(p)
        ra, rb = f16_ref[p], bf_ref[p]
        assert (a == ra) or (math.isnan(a) and math.isnan(ra)), hex(p)
        assert (b == rb) or (math.isnan(b) and math.isnan(rb)), hex(p)
        if a == 0:
            assert math.copysign(1, a) == math.copysign(1, ra)


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    exe = tmp_path_factory.mktemp("conv") / "check_converters"
    flags = ["-O2", "-std=gnu11", "-pthread"]
    # on x86 hosts with F16C the compiler's _Float16 conversion is one hardware
    # instruction (round to nearest even) instead of a libgcc call: same result, faster
    if platform.machine() == "x86_64" and " f16c" in open("/proc/cpuinfo").read():
        flags.append("-mf16c")
    subprocess.check_call(["gcc", *flags, os.path.join(HERE, "native", "check_converters.c"),
                           "-o", str(exe), "-ldl"])
    return str(exe)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
def test_rounding_exhaustive_against_compiler(harness, fmt):
    r = subprocess.run([harness, oracle.build(), fmt], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
