"""Pins for the oracle's GEMM with fp16 storage and fp32 compute (the Luminal page
"Luminal FP16 Backend Repair and H100 Evidence", section "What Was Fixed": operands
widened exactly, fp32 products and sums, the projection cast to fp16, then the fp16
bias add).

- Exact arithmetic: on small random shapes the output is the fp16 (or binary32) value
  nearest the exact rational sum of products, ties to even; the bias add is the fp16
  value nearest the exact sum of the cast result and the bias.
- An independent library route: torch's binary64 matmul of the widened operands,
  rounded once to fp16 by torch's cast, bit for bit on random data.
- Fixtures whose answers follow from the definition alone: the page's product /
  accumulation fixture (rounding the products to fp16 first gives 0 instead of
  K/2 * 2^-20), a sum just above an fp16 tie that a detour through binary32 would
  round the wrong way, ties to even, identity and zero operands, overflow, NaN and
  infinity.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import far_gen
import oracle
from oracle_pins import frac, is_rne_f32

F16_MAX_NEXT = Fraction(65536)           # 2^16, the first value past the fp16 range
F16_OVERFLOW = Fraction(65520)           # halfway between 65504 and 2^16


@pytest.fixture(scope="module")
def L():
    return oracle.lib()


def is_rne_f16(y, exact: Fraction) -> bool:
    """True when the fp16 value y is the one nearest `exact`, ties to even."""
    y = np.float16(y)
    if math.isinf(float(y)):
        return (exact >= F16_OVERFLOW) if y > 0 else (exact <= -F16_OVERFLOW)
    if abs(exact) >= F16_OVERFLOW:
        return False
    yf = frac(np.float32(y))
    up = np.nextafter(y, np.float16(np.inf))
    dn = np.nextafter(y, np.float16(-np.inf))
    upf = F16_MAX_NEXT if math.isinf(float(up)) else frac(np.float32(up))
    dnf = -F16_MAX_NEXT if math.isinf(float(dn)) else frac(np.float32(dn))
    d, du, dd = abs(yf - exact), abs(upf - exact), abs(dnf - exact)
    if d > du or d > dd:
        return False
    if d == du or d == dd:
        return (int(np.float16(y).view(np.uint16)) & 1) == 0
    return True


def exact_products(x, wt):
    xf = [[frac(np.float32(v)) for v in row] for row in x.float().numpy()]
    wf = [[frac(np.float32(v)) for v in row] for row in wt.float().numpy()]
    return [[sum((a * b for a, b in zip(xr, wr)), Fraction(0)) for wr in wf] for xr in xf]


def check_exact_small(L):
    for seed, (M, N, K) in enumerate([(3, 4, 1), (2, 5, 7), (4, 3, 16), (3, 3, 33), (2, 2, 64)]):
        d = far_gen.gemm_inputs(M, N, K, seed=seed + 100)
        if seed % 2:  # wide dynamic range within a row: products of very different sizes
            scale = torch.tensor([2.0 ** ((k * 7) % 24 - 12) for k in range(K)])
            d["x"] = (d["x"].float() * scale).to(torch.float16)
        ex = exact_products(d["x"], d["wt"])
        p = oracle.gemm_f16(d["x"], d["wt"], None, "f16", L=L)
        y = oracle.gemm_f16(d["x"], d["wt"], d["bias"], "f16", L=L)
        o32 = oracle.gemm_f16(d["x"], d["wt"], None, "f32", L=L)
        for m in range(M):
            for n in range(N):
                assert is_rne_f16(p[m, n].numpy(), ex[m][n]), (seed, m, n)
                assert is_rne_f32(o32[m, n].numpy(), ex[m][n]), (seed, m, n)
                s = frac(np.float32(p[m, n].float())) + frac(np.float32(d["bias"][n].float()))
                assert is_rne_f16(y[m, n].numpy(), s), (seed, m, n)


def check_torch_fp64(L):
    d = far_gen.gemm_inputs(48, 40, 768, seed=7)
    ref = d["x"].double() @ d["wt"].double().T          # binary64 sums of exact products
    p = oracle.gemm_f16(d["x"], d["wt"], None, "f16", L=L)
    assert torch.equal(p.view(torch.int16), ref.to(torch.float16).view(torch.int16))
    y = oracle.gemm_f16(d["x"], d["wt"], d["bias"], "f16", L=L)
    ry = (p.double() + d["bias"].double()).to(torch.float16)  # exact sum, one rounding
    assert torch.equal(y.view(torch.int16), ry.view(torch.int16))
    o32 = oracle.gemm_f16(d["x"], d["wt"], None, "f32", L=L)
    assert torch.equal(o32.view(torch.int32), ref.float().view(torch.int32))


def f16(vals):
    return torch.tensor(vals, dtype=torch.float64).to(torch.float16)


def check_fixtures(L):
    # the page's product/accumulation fixture: (1 + e)^2 - (1 + 2e) = e^2 per pair, e = 2^-10;
    # with the products rounded to fp16 every pair would give 0
    K = 768
    e = 2.0 ** -10
    x = f16([1 + e if k % 2 == 0 else -(1 + 2 * e) for k in range(K)]).reshape(1, K)
    w = f16([1 + e if k % 2 == 0 else 1.0 for k in range(K)]).reshape(1, K)
    p = oracle.gemm_f16(x, w, None, "f16", L=L)
    assert float(p[0, 0]) == (K // 2) * 2.0 ** -20
    # just above the fp16 tie between 1 and 1 + 2^-10: a detour through binary32 would
    # drop the 2^-40 and then round the tie to 1
    x = f16([1.0, 2.0 ** -11, 2.0 ** -20]).reshape(1, 3)
    w = f16([1.0, 1.0, 2.0 ** -20]).reshape(1, 3)
    assert float(oracle.gemm_f16(x, w, None, "f16", L=L)[0, 0]) == 1 + 2.0 ** -10
    # ties to even: 2049 (between 2048 and 2050) -> 2048, 2051 -> 2052
    for K, want in ((2049, 2048.0), (2051, 2052.0)):
        ones = torch.ones((1, K), dtype=torch.float16)
        assert float(oracle.gemm_f16(ones, ones, None, "f16", L=L)[0, 0]) == want
    # identity weight: out = x bit for bit; zero x: out = bias (RN: +0 + -0 = +0)
    d = far_gen.gemm_inputs(5, 8, 8, seed=3)
    eye = torch.eye(8, dtype=torch.float16)
    assert torch.equal(oracle.gemm_f16(d["x"], eye, None, "f16", L=L).view(torch.int16), d["x"].view(torch.int16))
    zero = torch.zeros((5, 8), dtype=torch.float16)
    b = f16([0.5, -0.0, 0.0, -3.0, 65504.0, 1e-7, -1e-7, 2.0])
    y = oracle.gemm_f16(zero, d["wt"], b, "f16", L=L)
    want = b.clone()
    want[1] = 0.0
    assert torch.equal(y.view(torch.int16), want.expand(5, 8).contiguous().view(torch.int16))
    # overflow to infinity at the projection cast and at the bias add
    big = f16([256.0, 255.0]).reshape(1, 2)
    w = f16([256.0, 0.0]).reshape(1, 2)
    assert math.isinf(float(oracle.gemm_f16(big, w, None, "f16", L=L)[0, 0]))
    w = f16([255.0, 0.0]).reshape(1, 2)
    assert float(oracle.gemm_f16(big, w, f16([1024.0]), "f16", L=L)[0, 0]) == math.inf  # 65280 + 1024
    assert float(oracle.gemm_f16(big, w, None, "f32", L=L)[0, 0]) == 65280.0
    # NaN and infinity
    x = f16([math.inf, 1.0]).reshape(1, 2)
    assert math.isnan(float(oracle.gemm_f16(x, f16([0.0, 1.0]).reshape(1, 2), None, "f16", L=L)[0, 0]))
    assert float(oracle.gemm_f16(x, f16([1.0, 1.0]).reshape(1, 2), None, "f16", L=L)[0, 0]) == math.inf
    x = f16([math.inf, math.inf]).reshape(1, 2)
    assert math.isnan(float(oracle.gemm_f16(x, f16([1.0, -1.0]).reshape(1, 2), None, "f16", L=L)[0, 0]))
    # K = 0: an empty sum is +0
    z = oracle.gemm_f16(torch.empty((2, 0), dtype=torch.float16), torch.empty((3, 0), dtype=torch.float16),
                        None, "f16", L=L)
    assert torch.equal(z.view(torch.int16), torch.zeros((2, 3), dtype=torch.int16))


GEMM_CHECKS = (check_exact_small, check_torch_fp64, check_fixtures)


def test_exact_small(L):
    check_exact_small(L)


def test_torch_fp64(L):
    check_torch_fp64(L)


def test_fixtures(L):
    check_fixtures(L)


def test_rejections(L):
    x = torch.zeros((2, 3), dtype=torch.float16)
    with pytest.raises(ValueError):
        oracle.gemm_f16(x, x, torch.zeros(2, dtype=torch.float16), "f32", L=L)
    with pytest.raises(ValueError):
        oracle.gemm_f16(x, torch.zeros((2, 4), dtype=torch.float16), None, "f16", L=L)
