"""Pins for the oracle's LayerNorm (two-pass, under the rounding contract).

- The exact signed sum: the defining property of round-to-nearest-even against the
  exact rational sum, with heavy cancellation and ties.
- Each step by its defining property in exact arithmetic (mean, var, rstd), d and
  out rebuilt bit for bit from the oracle's mean and rstd with numpy/torch IEEE
  primitives.
- Closed forms: a constant row gives exactly beta; a row of +-pairs has mean 0, and
  with beta = 0 LayerNorm equals the (separately pinned) RMSNorm oracle bit for bit;
  a column permutation permutes the output.
- An absolute bound against the fp64 evaluation.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import far_gen
import oracle
from oracle_pins import TD, bits_equal, frac, is_rne_f32, is_rne_sqrt_f32


@pytest.fixture(scope="module")
def L():
    return oracle.lib()


def ln_cases():
    cases = [far_gen.make_inputs("c1"), far_gen.custom_inputs("f16", "f16", 6, 4096, seed=2),
             far_gen.custom_inputs("bf16", "f32", 5, 777, seed=3), far_gen.custom_inputs("f32", "bf16", 4, 96, seed=4)]
    for act, wd in [("bf16", "bf16"), ("f16", "f32"), ("f32", "f32")]:
        for H in (1, 2, 3, 33):
            cases.append(far_gen.custom_inputs(act, wd, 5, H, seed=H + 10, scale_lo=1e-3, scale_hi=10))
    g = torch.Generator().manual_seed(0)
    for d in cases:  # a beta in the weight dtype, and rows with a large common offset
        d["b"] = (0.1 * torch.randn(d["hidden"], generator=g)).to(d["w"].dtype)
    off = far_gen.custom_inputs("f16", "f16", 4, 512, seed=5)
    off["x"] = (off["x"].float() + 300.0).half()
    off["b"] = torch.zeros(512, dtype=torch.float16)
    cases.append(off)
    return cases


def check_signed_sum(L):
    rng = np.random.default_rng(0)
    for trial in range(40):
        n = int(rng.integers(1, 300))
        v = (rng.standard_normal(n) * 10.0 ** rng.uniform(-8, 8, n)).astype(np.float32)
        if trial % 3 == 0:  # heavy cancellation: append the negations of most terms
            v = np.concatenate([v, -v[: n - 1], np.float32([1e-3])]).astype(np.float32)
        got = oracle.exact_signed_sum(v, L=L)
        exact = sum((frac(a) for a in v), Fraction(0))
        assert is_rne_f32(got, exact), (trial, got, float(exact))
    for vals, want in [([1.0, 2.0 ** -24, -(2.0 ** -80)], 1.0), ([-1.0, -(2.0 ** -24)], -1.0),
                       ([3.0, -3.0], 0.0), ([1e30, -1e30, 1.0], 1.0), ([], 0.0),
                       ([-(2.0 ** 24), -1.0], -(2.0 ** 24))]:
        assert float(oracle.exact_signed_sum(np.array(vals, np.float32), L=L)) == want, vals
    assert math.isnan(float(oracle.exact_signed_sum(np.array([np.inf, -np.inf], np.float32), L=L)))


def _s(d):
    return (d["x"].float() + d["r"].float()).numpy().astype(np.float32)


def check_steps(L, cases=None):
    for d in cases or ln_cases():
        H = d["hidden"]
        mean, rstd = oracle.ln_row_stats(d["x"], d["r"], d["eps"], d["act"], L=L)
        s = _s(d)
        dd = (s - mean[:, None]).astype(np.float32)  # numpy binary32 subtraction
        eps32 = np.float32(d["eps"])
        for t in range(s.shape[0]):
            S1 = sum((frac(v) for v in s[t]), Fraction(0))
            # mean = RN32(RN32(S1) / H): check the sum's rounding, then the quotient's
            S1r = oracle.exact_signed_sum(s[t], L=L)
            assert is_rne_f32(S1r, S1)
            assert is_rne_f32(mean[t], frac(S1r) / H), f"mean row {t} of {d['workload']}"
            sq = (dd[t] * dd[t]).astype(np.float32)
            S2 = np.float32(oracle.exact_sum(sq, L=L))
            assert is_rne_f32(S2, sum((frac(v) for v in sq), Fraction(0)))
            var = np.float32(S2 / np.float32(H))
            tv = np.float32(var + eps32)
            root = np.float32(np.sqrt(tv))
            assert is_rne_sqrt_f32(root, tv)
            assert is_rne_f32(rstd[t], 1 / frac(root)), f"rstd row {t} of {d['workload']}"
        out, res = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"],
                                              threads=1, L=L)
        assert bits_equal(res, torch.from_numpy(s).to(TD[d["act"]]))
        a = (dd * rstd[:, None]).astype(np.float32)
        n = torch.from_numpy(a).to(TD[d["wd"]]).float()
        t1 = n * d["w"].float()
        u = t1 + d["b"].float()
        od = "f32" if "f32" in (d["act"], d["wd"]) else d["act"]
        assert bits_equal(out, u.to(TD[od])), f"out of {d['workload']}"


def check_closed_forms(L):
    g = torch.Generator().manual_seed(3)
    for act, wd in [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32")]:
        od = "f32" if "f32" in (act, wd) else act
        for H in (1, 4, 64, 1000):
            x = torch.full((2, H), 0.75, dtype=TD[act])
            r = torch.full((2, H), -2.5, dtype=TD[act])
            gm = (1 + 0.1 * torch.randn(H, generator=g)).to(TD[wd])
            bt = (0.5 * torch.randn(H, generator=g)).to(TD[wd])
            out, _ = oracle.fused_add_layernorm(x, r, gm, bt, 1e-5, act, wd, threads=1, L=L)
            assert bits_equal(out, bt.float().to(TD[od]).expand(2, H)), f"constant row {act}/{wd} H={H}"
        # rows of +-pairs: mean 0; with beta = 0, LayerNorm equals RMSNorm
        d = far_gen.custom_inputs(act, wd, 6, 512, seed=8)
        half = d["x"][:, :256]
        x = torch.cat([half, -half], dim=1).contiguous()
        r = torch.zeros_like(x)
        zero = torch.zeros(512, dtype=TD[wd])
        ln, _ = oracle.fused_add_layernorm(x, r, d["w"], zero, d["eps"], act, wd, threads=1, L=L)
        rms, _ = oracle.fused_add_rmsnorm(x, r, d["w"], d["eps"], act, wd, threads=1, L=L)
        assert bits_equal(ln, rms), f"LayerNorm of a zero-mean row vs RMSNorm {act}/{wd}"
        # a column permutation permutes the output
        d = far_gen.custom_inputs(act, wd, 4, 300, seed=9)
        b = (0.1 * torch.randn(300, generator=g)).to(TD[wd])
        perm = torch.randperm(300, generator=g)
        o1, _ = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], b, d["eps"], act, wd, threads=1, L=L)
        o2, _ = oracle.fused_add_layernorm(d["x"][:, perm].contiguous(), d["r"][:, perm].contiguous(),
                                           d["w"][perm].contiguous(), b[perm].contiguous(), d["eps"], act, wd,
                                           threads=1, L=L)
        assert bits_equal(o2, o1[:, perm])
        # no residual == fused with a zero residual
        o3 = oracle.layernorm(d["x"], d["w"], b, d["eps"], act, wd, threads=1, L=L)
        o4, _ = oracle.fused_add_layernorm(d["x"], torch.zeros_like(d["x"]), d["w"], b, d["eps"], act, wd,
                                           threads=1, L=L)
        assert bits_equal(o3, o4)


def check_fp64(L, cases=None):
    """|out - LN_fp64| <= half an od ULP at out + half a weight-dtype ULP of a times |gamma|
    + the binary32 mean's ULP carried through rstd and gamma (+ binary32 slack)."""
    for d in cases or ln_cases():
        od = "f32" if "f32" in (d["act"], d["wd"]) else d["act"]
        out, _ = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"],
                                            threads=1, L=L)
        s = torch.from_numpy(_s(d)).double()
        mu = s.mean(dim=1, keepdim=True)
        var = ((s - mu) ** 2).mean(dim=1, keepdim=True)
        a = (s - mu) / torch.sqrt(var + float(np.float32(d["eps"])))
        exact = a * d["w"].double() + d["b"].double()

        def ulp(v, dt):
            fin = torch.finfo(TD[dt])
            return torch.pow(2.0, torch.floor(torch.log2(v.abs().clamp_min(fin.tiny)))) * fin.eps

        # the contract rounds the mean to binary32: every d_i carries up to one ULP of it
        rs = 1 / torch.sqrt(var + float(np.float32(d["eps"])))
        mean_err = ulp(mu, "f32") * rs * d["w"].double().abs()
        bound = 0.5 * ulp(exact, od) + 0.5 * ulp(a, d["wd"]) * d["w"].double().abs() + 4 * ulp(exact, "f32") \
            + 8 * 2.0 ** -23 * (a.abs() * d["w"].double().abs()) + mean_err
        err = (out.double() - exact).abs()
        assert bool((err <= bound * 1.0001 + 1e-30).all()), f"{d['workload']}: {float((err / bound).max()):.3f}"


def test_signed_sum(L):
    check_signed_sum(L)


def test_steps(L):
    check_steps(L)


def test_closed_forms(L):
    check_closed_forms(L)


def test_fp64_bound(L):
    check_fp64(L)


def test_rejects_f16_with_bf16(L):
    x = torch.zeros((1, 8), dtype=torch.float16)
    w = torch.ones(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.layernorm(x, w, w, 1e-5, "f16", "bf16")
