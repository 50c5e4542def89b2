"""Pins for the oracle's quantised output (per-token scale, int8 or FP8 E4M3).

- Format: all 256 E4M3 codes decoded against torch's float8_e4m3fn; rounding of
  binary32 values against torch's conversion (round to nearest even) wherever
  both are finite, and saturation to +-448 above; int8 rounding against numpy's
  round-half-even.
- The quantised rows against the unquantised oracle output (itself pinned by
  test_oracle_pins): scale by its defining property in exact arithmetic, q
  rebuilt from out with numpy/torch primitives bit for bit, the largest
  element at exactly +-127 / +-448, the dequantisation error bound.
- Page fact: the INT8 divisor 127 (golden/quantisation.json).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import far_gen
import oracle
from oracle_pins import frac, golden, is_rne_f32

QMAX = {"int8": 127.0, "fp8": 448.0}


@pytest.fixture(scope="module")
def L():
    return oracle.lib()


def check_e4m3_format(L):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = L.oracle_e4m3_to_f32(c)
        assert (got == ref[c]) or (np.isnan(got) and np.isnan(ref[c])), hex(c)
    # every midpoint between neighbouring values, the values themselves, and random values
    vals = np.sort(np.unique(ref[~np.isnan(ref)]))
    mids = (vals[:-1] + vals[1:]) / 2
    rng = np.random.default_rng(3)
    sample = np.concatenate([vals, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                             rng.uniform(-464, 464, 20000), rng.uniform(-1, 1, 20000) * 2.0 ** -6]).astype(np.float32)
    sample = sample[np.abs(sample) < 464]
    tref = torch.from_numpy(sample).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, want in zip(sample, tref):
        got = L.oracle_f32_to_e4m3(float(v))
        if want in (0x00, 0x80) and got in (0x00, 0x80):
            continue  # signed zeros
        assert got == want, f"{v!r}: {got:#04x} vs torch {want:#04x}"
    # saturation of finite values, NaN kept
    for v in (464.0, 479.0, 480.0, 1e4, 3e38, float("inf")):
        assert L.oracle_f32_to_e4m3(v) == 0x7E and L.oracle_f32_to_e4m3(-v) == 0xFE
    assert (L.oracle_f32_to_e4m3(float("nan")) & 0x7F) == 0x7F


def check_int8(L):
    rng = np.random.default_rng(4)
    v = np.concatenate([np.arange(-130, 131, 0.5), rng.uniform(-127.5, 127.5, 20000)]).astype(np.float32)
    ref = np.clip(np.rint(v), -127, 127).astype(np.int32)  # numpy rint: ties to even
    for a, b in zip(v, ref):
        assert L.oracle_f32_to_int8(float(a)) == b, a
    assert L.oracle_f32_to_int8(float("nan")) == 0
    assert L.oracle_f32_to_int8(float("inf")) == 127 and L.oracle_f32_to_int8(float("-inf")) == -127


def _quant_cases():
    return [far_gen.make_inputs("c1"),
            far_gen.custom_inputs("f16", "f16", 12, 1000, seed=5, scale_lo=1e-3, scale_hi=30),
            far_gen.custom_inputs("bf16", "f32", 10, 777, seed=6),
            far_gen.custom_inputs("f32", "bf16", 8, 96, seed=7)]


def check_quant_rows(L, cases=None):
    assert golden("quantisation.json")["int8_scale_divisor"] == QMAX["int8"]
    for d in cases or _quant_cases():
        for qtype in ("int8", "fp8"):
            for with_res in (True, False):
                if with_res:
                    q, scale, res = oracle.fused_add_rmsnorm_quant(d["x"], d["r"], d["w"], d["eps"], d["act"],
                                                                  d["wd"], qtype, threads=1, L=L)
                    out, ref_res = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"],
                                                            threads=1, L=L)
                    assert torch.equal(res.view(torch.int16 if res.element_size() == 2 else torch.int32),
                                       ref_res.view(torch.int16 if res.element_size() == 2 else torch.int32))
                else:
                    q, scale = oracle.rmsnorm_quant(d["x"], d["w"], d["eps"], d["act"], d["wd"], qtype,
                                                    threads=1, L=L)
                    out = oracle.rmsnorm(d["x"], d["w"], d["eps"], d["act"], d["wd"], threads=1, L=L)
                o = out.float().numpy()
                amax = np.abs(o).max(axis=1).astype(np.float32)
                qm = np.float32(QMAX[qtype])
                for t in range(o.shape[0]):
                    # scale = RN32(amax / QMAX) by its defining property
                    assert is_rne_f32(np.float32(scale[t]), frac(amax[t]) / Fraction(int(qm))), (qtype, t)
                inv = np.where(amax == 0, np.float32(0), (qm / amax).astype(np.float32)).astype(np.float32)
                v = (o * inv[:, None]).astype(np.float32)  # numpy binary32 multiply
                if qtype == "int8":
                    ref = np.clip(np.rint(v), -127, 127).astype(np.int8)
                    assert np.array_equal(q.numpy(), ref), f"int8 q of {d['workload']} res={with_res}"
                    # the largest element lands on +-127; dequantisation within half a step
                    for t in range(o.shape[0]):
                        i = int(np.argmax(np.abs(o[t])))
                        assert abs(int(q[t, i])) == 127
                    err = np.abs(q.numpy().astype(np.float64) * scale.numpy()[:, None].astype(np.float64) - o)
                    assert (err <= scale.numpy()[:, None] * (0.5 + 1e-5)).all()
                else:
                    vv = np.clip(v, -448, 448)
                    ref = torch.from_numpy(vv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    got = q.numpy()
                    zero = ((ref & 0x7F) == 0) & ((got & 0x7F) == 0)
                    assert np.array_equal(np.where(zero, 0, got), np.where(zero, 0, ref)), \
                        f"fp8 q of {d['workload']} res={with_res}"
                    for t in range(o.shape[0]):
                        i = int(np.argmax(np.abs(o[t])))
                        assert (got[t, i] & 0x7F) == 0x7E  # +-448


def test_e4m3_format(L):
    check_e4m3_format(L)


def test_int8_rounding(L):
    check_int8(L)


def test_quantised_rows(L):
    check_quant_rows(L)


def test_quant_special_rows(L):
    """A zero row quantises to zeros with scale 0; a NaN row gives a NaN scale."""
    x = torch.zeros((2, 64), dtype=torch.float16)
    r = torch.zeros((2, 64), dtype=torch.float16)
    x[1, 3] = float("nan")
    w = torch.ones(64, dtype=torch.float16)
    for qtype in ("int8", "fp8"):
        q, scale, _ = oracle.fused_add_rmsnorm_quant(x, r, w, 1e-6, "f16", "f16", qtype)
        assert scale[0] == 0 and (q[0].int() & 0x7F == 0).all()
        assert torch.isnan(scale[1])
