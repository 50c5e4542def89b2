"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (``oracle.bind(path)``)
and raises ``AssertionError`` when the oracle disagrees with what the pages
and the mathematics fix.  ``test_oracle_pins.py`` runs them on the oracle;
``test_oracle_mutants.py`` plants plausible mistakes in a copy of the oracle's
source and checks that at least one pin fails for each.

What pins what:
  pin_residual      residual_out = RNE_act(fl32(x + r)), rebuilt from torch's
                    binary32 add and its own RNE conversions (library routines).
  pin_sum           S is the correctly rounded binary32 value of the exact sum of
                    the binary32 squares: checked by the defining property of
                    round-to-nearest-even in exact rational arithmetic.
  pin_steps         var, rstd, and every element of out: each binary32 step is
                    checked by its defining property in exact arithmetic
                    (quotient, sum, square root, reciprocal), and out is rebuilt
                    from the oracle's rstd with numpy/torch primitives.
  pin_closed_forms  constant rows normalise to +-w exactly; hidden = 1; zero rows;
                    sign symmetry; scaling by 2^k with eps = 0; column
                    permutation; the no-residual variant equals the fused op with
                    a zero residual.
  pin_fp64          out within 2 ULP (4 for binary32) of the working dtype of the
                    unrounded fp64 evaluation, and within
                    the Luminal page's tolerance of the fp64 evaluation rounded at
                    the declared boundaries.
  pin_policy        fp16 with bf16 rejected; output dtype is the promotion.
  pin_exhaustive_h1 hidden = 1 over EVERY finite fp16 and every finite bf16 x, with
                    a few residuals (zero, a permutation of the same values, -x),
                    weights and eps: every binary32 step of every row against its
                    binary64 evaluation rounded once to binary32, which is the
                    correctly rounded binary32 result (the squares and products
                    of binary32 values are exact in binary64, and for + / sqrt
                    binary64 carries 53 >= 2 * 24 + 2 bits, so the double rounding
                    is innocuous: S. A. Figueroa, "When is double rounding
                    innocuous?", SIGNUM Newsletter 30(3), 1995); residual_out and
                    the two casts by torch's RNE conversions.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import far_gen
import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TD = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# exact-arithmetic helpers
# --------------------------------------------------------------------------

F32_MAX = Fraction(float(np.finfo(np.float32).max))
F32_OVERFLOW = Fraction(2) ** 128 - Fraction(2) ** 103  # RNE sends |v| >= this to infinity


def frac(v) -> Fraction:
    return Fraction(float(v))


def is_rne_f32(y: np.float32, exact: Fraction) -> bool:
    """True when y is the binary32 value nearest to `exact`, ties to even."""
    y = np.float32(y)
    if math.isinf(float(y)):
        return (exact >= F32_OVERFLOW) if y > 0 else (exact <= -F32_OVERFLOW)
    if abs(exact) >= F32_OVERFLOW:
        return False
    yf = frac(y)
    up = np.nextafter(y, np.float32(np.inf))
    dn = np.nextafter(y, np.float32(-np.inf))
    upf = Fraction(2) ** 128 if math.isinf(float(up)) else frac(up)
    dnf = -(Fraction(2) ** 128) if math.isinf(float(dn)) else frac(dn)
    d, du, dd = abs(yf - exact), abs(upf - exact), abs(dnf - exact)
    if d > du or d > dd:
        return False
    if d == du or d == dd:  # a tie: y must have the even significand
        return (int(np.float32(y).view(np.uint32)) & 1) == 0
    return True


def is_rne_sqrt_f32(y: np.float32, v: np.float32) -> bool:
    """True when y = RN32(sqrt(v)) for v > 0 (no ties are possible for binary32 v)."""
    y = np.float32(y)
    up = frac(np.nextafter(y, np.float32(np.inf)))
    dn = frac(np.nextafter(y, np.float32(0)))
    yf, vf = frac(y), frac(v)
    lo = (yf + dn) / 2
    hi = (yf + up) / 2
    return lo * lo <= vf <= hi * hi


def ordered(bits: np.ndarray, width: int) -> np.ndarray:
    """Map IEEE bit patterns to integers whose difference counts representable steps."""
    b = bits.astype(np.int64)
    sign = np.int64(1) << (width - 1)
    mag = b & (sign - 1)
    return np.where(b & sign, -mag, mag)


def ulp_distance(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    """Representable steps between equal-dtype tensors (NaN vs NaN counts 0, NaN vs number huge)."""
    assert a.dtype == b.dtype
    width = a.element_size() * 8
    view = {16: torch.int16, 32: torch.int32}[width]
    ai = a.contiguous().view(view).numpy().astype(np.int64) & ((1 << width) - 1)
    bi = b.contiguous().view(view).numpy().astype(np.int64) & ((1 << width) - 1)
    d = np.abs(ordered(ai, width) - ordered(bi, width))
    an, bn = torch.isnan(a.float()).numpy(), torch.isnan(b.float()).numpy()
    d = np.where(an & bn, 0, d)
    d = np.where(an ^ bn, 1 << 40, d)
    return d


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bit-for-bit equality, with +0 == -0 and any NaN equal to any NaN."""
    return bool((ulp_distance(a, b) == 0).all())


# --------------------------------------------------------------------------
# pin data (small: every pin runs in seconds)
# --------------------------------------------------------------------------

def _take(d: dict, rows: int) -> dict:
    d = dict(d)
    d["x"], d["r"] = d["x"][:rows].contiguous(), d["r"][:rows].contiguous()
    d["tokens"] = rows
    return d


def pin_cases() -> list[dict]:
    """Workload rows plus small shapes with tiny hidden sizes and var ~ eps rows."""
    cases = [far_gen.make_inputs("c1"),
             _take(far_gen.make_inputs("c2", rows=4), 4),
             _take(far_gen.make_inputs("c3", rows=6), 6),
             _take(far_gen.make_inputs("c4", rows=4), 4)]
    for act, wd in [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f16", "f32"),
                    ("f32", "f32"), ("f32", "bf16"), ("f32", "f16")]:
        for H in (1, 2, 3, 4, 7, 33):
            cases.append(far_gen.custom_inputs(act, wd, 6, H, seed=H, scale_lo=1e-3, scale_hi=10.0))
    # rows whose mean square is near eps, so that eps matters
    cases.append(far_gen.custom_inputs("f16", "f16", 8, 64, seed=7, scale_lo=1e-4, scale_hi=3e-3, eps=1e-6))
    cases.append(far_gen.custom_inputs("bf16", "f32", 8, 48, seed=8, scale_lo=1e-4, scale_hi=3e-3, eps=1e-5))
    return cases


# one call over all rows (threads=1), so that row strides inside the C code are exercised
def run_fused(L, d):
    return oracle_mod.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"],
                                        threads=1, L=L)


def run_norm(L, d):
    return oracle_mod.rmsnorm(d["x"], d["w"], d["eps"], d["act"], d["wd"], threads=1, L=L)


def _od(act, wd):
    return "f32" if "f32" in (act, wd) else act


# --------------------------------------------------------------------------
# pins
# --------------------------------------------------------------------------

def pin_residual(L, cases=None):
    for d in cases or pin_cases():
        _, res = run_fused(L, d)
        ref = (d["x"].float() + d["r"].float()).to(TD[d["act"]])  # binary32 add, one RNE rounding
        assert bits_equal(res, ref), f"residual_out differs on {d['workload']}"


def _squares_f32(d, with_residual=True) -> np.ndarray:
    s = d["x"].float() + d["r"].float() if with_residual else d["x"].float()
    s = s.numpy().astype(np.float32)
    return s, (s * s).astype(np.float32)  # numpy binary32 multiply


def pin_sum(L, cases=None):
    """S = RN32(exact sum of the binary32 squares), checked in exact arithmetic."""
    for d in cases or pin_cases():
        S, _, _ = oracle_mod.row_stats(d["x"], d["r"], d["eps"], d["act"], L=L)
        _, sq = _squares_f32(d)
        for t in range(min(d["tokens"], 4)):
            exact = sum((frac(v) for v in sq[t]), Fraction(0))
            assert is_rne_f32(S[t], exact), f"S row {t} of {d['workload']}: {S[t]!r} vs {float(exact)!r}"
    # adversarial sums: ties to even, near-overflow, subnormals
    tiny = float(np.float32(2.0 ** -149))
    cases = [
        ([1.0, 2.0 ** -24], 1.0),                      # exact midpoint, even is 1.0
        ([1.0 + 2.0 ** -23, 2.0 ** -24], 1.0 + 2.0 ** -22),  # midpoint, even is above
        ([1.0, 2.0 ** -24, 2.0 ** -60], 1.0 + 2.0 ** -23),   # just above the midpoint
        ([float(np.finfo(np.float32).max), 2.0 ** 103], math.inf),  # tie at the top: to infinity
        ([float(np.finfo(np.float32).max), 2.0 ** 102], float(np.finfo(np.float32).max)),
        ([tiny, tiny, tiny], 3 * tiny),
        ([2.0 ** 24] + [1.0] * 3, 2.0 ** 24 + 4.0),    # 2^24 + 3: a tie, even is + 4
        ([], 0.0),
    ]
    for vals, want in cases:
        got = oracle_mod.exact_sum(np.array(vals, dtype=np.float32), L=L)
        assert float(got) == want, f"exact_sum({vals}) = {got!r}, want {want!r}"
    assert math.isnan(float(oracle_mod.exact_sum(np.array([1.0, np.nan], np.float32), L=L)))
    assert math.isinf(float(oracle_mod.exact_sum(np.array([1.0, np.inf], np.float32), L=L)))


def pin_steps(L, cases=None):
    """Each binary32 step of a row by its defining property; out rebuilt by library primitives."""
    for d in cases or pin_cases():
        H = d["hidden"]
        eps32 = np.float32(d["eps"])
        S, var, rstd = oracle_mod.row_stats(d["x"], d["r"], d["eps"], d["act"], L=L)
        for t in range(d["tokens"]):
            assert is_rne_f32(var[t], frac(S[t]) / H), f"var row {t} of {d['workload']}"
            tv = np.float32(var[t] + eps32)  # numpy binary32 add
            assert is_rne_f32(tv, frac(var[t]) + frac(eps32))
            root = np.float32(np.sqrt(tv))  # numpy binary32 square root (IEEE)
            assert is_rne_sqrt_f32(root, tv)
            assert is_rne_f32(rstd[t], 1 / frac(root)), f"rstd row {t} of {d['workload']}"
        out, _ = run_fused(L, d)
        s, _ = _squares_f32(d)
        a = (s * rstd[:, None]).astype(np.float32)  # numpy binary32 multiply
        n = torch.from_numpy(a).to(TD[d["wd"]])      # torch RNE cast to the weight dtype
        prod = n.float() * d["w"].float()            # binary32 product
        ref = prod.to(TD[_od(d["act"], d["wd"])])
        assert bits_equal(out, ref), f"out differs from its rebuilt value on {d['workload']}"


def pin_closed_forms(L):
    gen = torch.Generator().manual_seed(1)
    # constant rows c = +-2^k: var = 4^k, rstd = 2^-k, a = +-1, so out = +-w exactly
    for act, wd in [("f16", "f16"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f32", "bf16")]:
        for H in (1, 2, 3, 4, 7, 64, 2048):
            for k, sign in ((3, 1.0), (5, -1.0), (4, 1.0)):
                c = sign * 2.0 ** k
                x = torch.full((1, H), c / 2, dtype=TD[act])
                r = torch.full((1, H), c / 2, dtype=TD[act])
                w = (1 + 0.1 * torch.randn(H, generator=gen)).to(TD[wd])
                out, res = oracle_mod.fused_add_rmsnorm(x, r, w, 1e-6, act, wd, threads=1, L=L)
                od = _od(act, wd)
                want = (sign * w.float()).to(TD[od]).reshape(1, H)
                assert bits_equal(out, want), f"constant row {c} H={H} {act}/{wd}"
                assert bits_equal(res, torch.full((1, H), c, dtype=TD[act]))
    # hidden = 1, eps = 0: out = sign(v) * w for v = +-2^k
    for v in (0.25, -8.0, 1024.0):
        x = torch.tensor([[v]], dtype=torch.float16)
        w = torch.tensor([1.375], dtype=torch.float16)
        out = oracle_mod.rmsnorm(x, w, 0.0, "f16", "f16", threads=1, L=L)
        assert float(out) == math.copysign(1.375, v)
    # zero row: out is a signed zero
    x = torch.zeros((1, 16), dtype=torch.bfloat16)
    w = torch.ones(16, dtype=torch.bfloat16)
    out, res = oracle_mod.fused_add_rmsnorm(x, x, w, 1e-6, "bf16", "bf16", threads=1, L=L)
    assert (out.float() == 0).all() and (res.float() == 0).all()
    for d in pin_cases()[:8]:
        act, wd = d["act"], d["wd"]
        out, res = run_fused(L, d)
        # negating x and r negates both outputs (round-to-nearest-even is symmetric)
        nd = dict(d, x=-d["x"], r=-d["r"])
        nout, nres = run_fused(L, nd)
        assert bits_equal(nout, -out) and bits_equal(nres, -res), f"sign symmetry {d['workload']}"
        # a column permutation of x, r and w permutes the outputs
        perm = torch.randperm(d["hidden"], generator=gen)
        pd = dict(d, x=d["x"][:, perm].contiguous(), r=d["r"][:, perm].contiguous(), w=d["w"][perm].contiguous())
        pout, pres = run_fused(L, pd)
        assert bits_equal(pout, out[:, perm]) and bits_equal(pres, res[:, perm]), f"permutation {d['workload']}"
        # no residual == fused with a zero residual (s = x + 0 = x for x != -0)
        zd = dict(d, r=torch.zeros_like(d["r"]))
        zout, _ = run_fused(L, zd)
        assert bits_equal(run_norm(L, d), zout), f"no-residual variant {d['workload']}"
        # scaling x and r by 2^k with eps = 0 leaves out unchanged (no overflow/underflow here)
        if act != "f32":
            e0 = dict(d, eps=0.0)
            base, _ = run_fused(L, e0)
            for k in (-3, 2):
                sx, sr = d["x"] * 2.0 ** k, d["r"] * 2.0 ** k
                if not (torch.equal(sx * 2.0 ** -k, d["x"]) and torch.equal(sr * 2.0 ** -k, d["r"])):
                    continue  # the scaled values left the normal range: the invariant does not apply
                sd = dict(e0, x=sx, r=sr)
                sout, _ = run_fused(L, sd)
                assert bits_equal(sout, base), f"2^{k} scaling {d['workload']}"
                snorm = run_norm(L, sd)
                assert bits_equal(snorm, run_norm(L, e0)), f"2^{k} scaling, no residual {d['workload']}"


def _fp64_reference(d, with_residual=True, rounded=False):
    s = d["x"].float() + d["r"].float() if with_residual else d["x"].float()
    s = s.double()
    var = (s * s).mean(dim=1, keepdim=True)
    a = s / torch.sqrt(var + float(np.float32(d["eps"])))
    if rounded:  # the declared rounding boundaries: weight-dtype cast, output cast
        a = a.to(TD[d["wd"]]).double()
        return (a * d["w"].double()).to(TD[_od(d["act"], d["wd"])]).double()
    return a * d["w"].double()


def pin_fp64(L, cases=None):
    tol = golden("tolerance.json")
    for d in cases or pin_cases():
        od = _od(d["act"], d["wd"])
        for with_res in (True, False):
            out = run_fused(L, d)[0] if with_res else run_norm(L, d)
            exact = _fp64_reference(d, with_res)
            # ULP of the working dtype at the fp64 value: the narrowest format the value
            # passes through (the weight-dtype cast, then od), with a subnormal floor
            work = min((d["wd"], od), key=lambda t: torch.finfo(TD[t]).eps * -1)
            fin = torch.finfo(TD[work])
            mag = exact.abs().clamp_min(fin.tiny)
            spacing = torch.pow(2.0, torch.floor(torch.log2(mag))) * fin.eps
            err = (out.double() - exact).abs() / spacing
            # 16-bit working dtype: half an ULP for each of the two casts plus binary32 noise;
            # binary32: the S, var, sqrt, reciprocal, a and product roundings add up to ~2.2 ULP
            bound_ulp = 4.0 if work == "f32" else 2.0
            assert float(err.max()) <= bound_ulp, f"{d['workload']} res={with_res}: {float(err.max()):.3f} ULP from fp64"
            # the Luminal page's tolerance was set for fp16 results; one bf16 ULP (2^-8
            # relative) already exceeds its relative term, so it is applied where the
            # working dtype is fp16 or binary32
            if work != "bf16":
                ref = _fp64_reference(d, with_res, rounded=True)
                bound = tol["abs"] + tol["rel"] * ref.abs()
                assert bool(((out.double() - ref).abs() <= bound).all()), \
                    f"{d['workload']}: outside the page tolerance"


def pin_policy(L):
    code = oracle_mod.DTYPE_CODE
    assert L.oracle_output_dtype(code["f16"], code["bf16"]) < 0
    assert L.oracle_output_dtype(code["bf16"], code["f16"]) < 0
    assert L.oracle_output_dtype(code["bf16"], code["bf16"]) == code["bf16"]
    assert L.oracle_output_dtype(code["f16"], code["f16"]) == code["f16"]
    for a in ("f16", "bf16", "f32"):
        assert L.oracle_output_dtype(code[a], code["f32"]) == code["f32"]
        assert L.oracle_output_dtype(code["f32"], code[a]) == code["f32"]
    assert L.oracle_output_dtype(7, 0) < 0


ALL_PINS = [pin_policy, pin_residual, pin_sum, pin_steps, pin_closed_forms, pin_fp64]


# --------------------------------------------------------------------------
# hidden = 1, exhaustively over the 16-bit inputs
# --------------------------------------------------------------------------

def finite_values(dt: str) -> torch.Tensor:
    """Every finite value of a 16-bit dtype (all 2^16 bit patterns but the infinities and
    NaNs), as a [N, 1] tensor."""
    bits = torch.from_numpy(np.arange(65536, dtype=np.uint16).view(np.int16).copy())
    v = bits.view(TD[dt])
    return v[torch.isfinite(v.float())].reshape(-1, 1).contiguous()


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _check_h1_rows(L, x, r, w, eps, act, wd, where):
    """One hidden = 1 call of the fused op (r given) or of the variant (r None), every row
    checked step by step against the binary64 evaluation rounded once to binary32."""
    od = _od(act, wd)
    eps32 = np.float32(eps)
    with np.errstate(all="ignore"):
        if r is not None:
            # fl32(x + r): the binary64 sum of two binary32 values rounded to binary32
            s32 = np.float32(_f64(x.float().numpy()[:, 0]) + _f64(r.float().numpy()[:, 0]))
        else:
            s32 = x.float().numpy()[:, 0].astype(np.float32)  # exact widening
        s64 = _f64(s32)
        S_ref = np.float32(s64 * s64)                       # one square: exact in binary64
        var_ref = np.float32(_f64(S_ref) / 1.0)             # S / hidden, hidden = 1
        tv_ref = np.float32(_f64(var_ref) + _f64(eps32))
        root_ref = np.float32(np.sqrt(_f64(tv_ref)))
        rstd_ref = np.float32(1.0 / _f64(root_ref))
        a_ref = np.float32(s64 * _f64(rstd_ref))            # exact product, one rounding
        n = torch.from_numpy(a_ref).to(TD[wd])              # RNE to the weight dtype
        prod = np.float32(_f64(n.float().numpy()) * float(w.float()[0]))  # exact product
        out_ref = torch.from_numpy(prod).to(TD[od]).reshape(-1, 1)
    S, var, rstd = oracle_mod.row_stats(x, r, eps, act, L=L)
    for name, got, want in (("S", S, S_ref), ("var", var, var_ref), ("rstd", rstd, rstd_ref)):
        assert bits_equal(torch.from_numpy(got), torch.from_numpy(want)), \
            f"{name} differs from its binary64 evaluation ({where})"
    if r is not None:
        out, res = oracle_mod.fused_add_rmsnorm(x, r, w, eps, act, wd, L=L)
        res_ref = torch.from_numpy(s32).to(TD[act]).reshape(-1, 1)  # RNE_act of the binary32 sum
        assert bits_equal(res, res_ref), f"residual_out ({where})"
    else:
        out = oracle_mod.rmsnorm(x, w, eps, act, wd, L=L)
    assert bits_equal(out, out_ref), f"out ({where})"


def pin_exhaustive_h1(L):
    """hidden = 1 over every finite fp16 and every finite bf16 x (see the module doc)."""
    for act in ("f16", "bf16"):
        x = finite_values(act)
        n = x.shape[0]
        perm = torch.from_numpy(np.random.default_rng(5).permutation(n))
        residuals = {"zero": torch.zeros_like(x), "permuted": x[perm].contiguous(), "negated": (-x).contiguous()}
        weights = [(act, 1.0), (act, -1.375), (act, 0.1), (act, 2.0 ** -20), ("f32", 0.7)]
        for wd, wv in weights:
            w = torch.tensor([wv], dtype=TD[wd])
            for rname, r in residuals.items():
                _check_h1_rows(L, x, r, w, 1e-6, act, wd, f"{act} x, r {rname}, w {wv} {wd}, eps 1e-6")
            _check_h1_rows(L, x, None, w, 1e-6, act, wd, f"{act} x, no residual, w {wv} {wd}, eps 1e-6")
        # eps 0 (a zero row then has rstd = inf and a NaN output) and a large eps
        w = torch.tensor([1.0], dtype=TD[act])
        for eps in (0.0, 0.5):
            _check_h1_rows(L, x, residuals["permuted"], w, eps, act, act, f"{act} x, r permuted, eps {eps}")
            _check_h1_rows(L, x, None, w, eps, act, act, f"{act} x, no residual, eps {eps}")
