"""A model of the staged kernel's sum of squares, in binary32 numpy arithmetic, on the CPU.

Each thread adds the squares of its values into four double-word chains (two packed pairs in
the kernel) that start at B, the largest of its squares with the mantissa cleared, and
only grow; each addition is Dekker's Fast2Sum without ordering its operands (s = hi + q,
t = q - (s - hi), lo += t), exact because a chain's exponent is never below a term's. At the
end B is taken off each chain (exact), the chains are folded with TwoSum, and the double
words are reduced across the 32 lanes and the row's warps with the ordered Fast2Sum
(max / min first), then rounded once. This file restates those steps (numpy float32 rounds
to nearest even and keeps subnormals, as the kernel's explicitly rounded operations do) and
checks them against the oracle's correctly rounded sum of the binary32 squares: every step
of the offset chains exact (checked in rational arithmetic), the row's result equal to the
oracle's on random and adversarial rows. A chain started at zero instead, with the same
unordered Fast2Sum, must lose exactness on rows whose squares grow along the chain, so the
offset is not vacuous.
"""
from fractions import Fraction

import numpy as np
import pytest

import far_gen

f32 = np.float32


def _pow2_floor(q):
    """The largest square's exponent field alone (0 for a subnormal, inf for inf or NaN)."""
    return (q.astype(f32).view(np.uint32) & np.uint32(0x7F800000)).view(f32)


def _fast2sum(a, b):
    s = (a + b).astype(f32)
    return s, (b - (s - a).astype(f32)).astype(f32)


def _two_sum(a, b):
    s = (a + b).astype(f32)
    bv = (s - a).astype(f32)
    av = (s - bv).astype(f32)
    return s, ((a - av).astype(f32) + (b - bv).astype(f32)).astype(f32)


def _combine_ordered(a, b):
    with np.errstate(invalid="ignore"):
        big = np.where(np.isnan(a[0]) | np.isnan(b[0]), np.float32(np.nan), np.maximum(a[0], b[0])).astype(f32)
        small = np.where(np.isnan(a[0]) | np.isnan(b[0]), np.float32(np.nan), np.minimum(a[0], b[0])).astype(f32)
        s, e = _fast2sum(big, small)
        return s, ((a[1] + b[1]).astype(f32) + e).astype(f32)


def _combine_signed(a, b):
    with np.errstate(invalid="ignore"):
        s, e = _two_sum(a[0], b[0])
        return s, ((a[1] + b[1]).astype(f32) + e).astype(f32)


def model_sum_of_squares(rows, G, offset=True, steps=None):
    """rows [R, H] binary32 values of s; G warps a row, 32 lanes, each lane taking 8-value
    chunks j * G * 32 + warp * 32 + lane. Returns RN32 of the double word, as the kernel."""
    R, H = rows.shape
    V = 8
    C = (H + V - 1) // V
    nch = (C + 32 * G - 1) // (32 * G)
    pad = np.zeros((R, nch * G * 32 * V), f32)
    pad[:, :H] = rows
    x = pad.reshape(R, nch, G, 32, V)  # chunk j of warp g, lane l: x[:, j, g, l, :]
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        sq = (x * x).astype(f32)  # fl32(s * s)
        B = _pow2_floor(np.nanmax(np.where(np.isnan(sq), np.float32(np.inf), sq), axis=(1, 4))) if offset \
            else np.zeros((R, G, 32), f32)
        B = np.where(np.isnan(sq).any(axis=(1, 4)), np.float32(np.inf), B).astype(f32)
        hi = [B.copy() for _ in range(4)]
        lo = [np.zeros((R, G, 32), f32) for _ in range(4)]
        for j in range(nch):
            for e in range(V // 2):
                for half in range(2):
                    k = 2 * (e & 1) + half
                    q = sq[:, j, :, :, 2 * e + half]
                    s, t = _fast2sum(hi[k], q)
                    if steps is not None:
                        steps.append((hi[k].copy(), q.copy(), s, t))
                    hi[k], lo[k] = s, (lo[k] + t).astype(f32)
        fin = np.isfinite(B)
        acc = [(np.where(fin, (hi[k] - B).astype(f32), hi[k]).astype(f32), lo[k]) for k in range(4)]
        # the packed pairs' halves folded with TwoSum, then the ordered combine
        d = _combine_ordered(_combine_signed(acc[0], acc[1]), _combine_signed(acc[2], acc[3]))
        for off in (16, 8, 4, 2, 1):
            perm = np.arange(32) ^ off
            d = _combine_ordered(d, (d[0][:, :, perm], d[1][:, :, perm]))
        part = (d[0][:, :, 0], d[1][:, :, 0])
        G8 = 1
        while G8 < G:
            G8 <<= 1
        t = (np.zeros((R, G8), f32), np.zeros((R, G8), f32))
        t[0][:, :G], t[1][:, :G] = part
        off = G8 >> 1
        while off:
            perm = np.arange(G8) ^ off
            t = _combine_ordered(t, (t[0][:, perm], t[1][:, perm]))
            off >>= 1
        h, l = t[0][:, 0], t[1][:, 0]
        return np.where(np.isfinite(h), (h + l).astype(f32), h).astype(f32)


def _oracle_sums(rows):
    import oracle

    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        return np.array([oracle.exact_sum((r * r).astype(f32)) for r in rows], f32)


def _same(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32)) or bool(
        np.all((a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))))


def _rows(kind, R, H, seed):
    rng = np.random.default_rng(seed)
    if kind == "workload":  # the generator's rows: N(0, 1) times a per-row log-uniform scale
        return far_gen.custom_inputs("f32", "f32", R, H, seed=seed)["x"].numpy()
    if kind == "fp16":
        return far_gen.custom_inputs("f16", "f16", R, H, seed=seed)["x"].float().numpy()
    if kind == "wide":  # magnitudes log-uniform over 2^-75 .. 2^60: squares from subnormal to 2^120
        return (rng.choice([-1.0, 1.0], (R, H)) * np.exp2(rng.uniform(-75, 60, (R, H)))).astype(f32)
    if kind == "dominant":  # one element far above the rest, in a random lane
        x = rng.standard_normal((R, H)).astype(f32)
        x[np.arange(R), rng.integers(0, H, R)] *= f32(2.0 ** 20)
        return x
    if kind == "growing":  # squares growing along each thread's chunks: every term above the chain
        return np.tile(np.exp2(np.repeat(np.arange(H // 256 + 1), 256)[:H] * 3.0).astype(f32), (R, 1)) \
            * (1 + rng.integers(0, 255, (R, H)) / 256).astype(f32)
    if kind == "subnormal":  # squares that are binary32 subnormals (rounded)
        return (rng.choice([-1.0, 1.0], (R, H)) * rng.uniform(1, 2, (R, H)) * 2.0 ** -70).astype(f32)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["workload", "fp16", "wide", "dominant", "growing", "subnormal"])
@pytest.mark.parametrize("H,G", [(8192, 4), (5120, 2), (1000, 1), (4096, 2)])
def test_offset_chains_give_the_correctly_rounded_sum(kind, H, G):
    rows = _rows(kind, 300, H, seed=H + G)
    got = model_sum_of_squares(rows, G)
    want = _oracle_sums(rows)
    assert _same(got, want), np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0][:10]


def test_every_offset_step_is_exact():
    """Each Fast2Sum step of the offset chains: s + t equals hi + q exactly (rationals)."""
    rng = np.random.default_rng(3)
    for kind in ("wide", "growing", "dominant", "subnormal"):
        rows = _rows(kind, 4, 1024, seed=int(rng.integers(1 << 30)))
        steps = []
        model_sum_of_squares(rows, 1, steps=steps)
        checked = 0
        for hi, q, s, t in steps:
            for a, b, ss, tt in zip(hi.ravel()[::2], q.ravel()[::2], s.ravel()[::2], t.ravel()[::2]):
                assert Fraction(float(ss)) + Fraction(float(tt)) == Fraction(float(a)) + Fraction(float(b))
                checked += 1
        assert checked > 500


def test_special_rows():
    """A zero row, a constant row, an infinite square, a NaN, squares that overflow."""
    H = 512
    rows = np.ones((6, H), f32)
    rows[0] = 0
    rows[1] = f32(3.0)
    rows[2, 17] = np.inf
    rows[3, 300] = np.nan
    rows[4, :] = f32(2.0 ** 70)  # every square overflows binary32
    rows[5, :] = f32(2.0 ** 60)  # the squares are finite; their sum overflows
    got = model_sum_of_squares(rows, 2)
    want = _oracle_sums(rows)
    assert _same(got, want)
    assert got[0] == 0 and got[1] == f32(9.0 * H) and np.isinf(got[2]) and np.isnan(got[3])
    assert np.isinf(got[4]) and np.isinf(got[5])


def test_chains_from_zero_lose_exactness():
    """The same unordered Fast2Sum on chains started at zero: rows whose squares grow along
    a thread's chunks break its exactness condition, and some step is inexact."""
    rows = _rows("growing", 4, 2048, seed=9)
    steps = []
    model_sum_of_squares(rows, 1, offset=False, steps=steps)
    inexact = 0
    for hi, q, s, t in steps:
        for a, b, ss, tt in zip(hi.ravel()[::7], q.ravel()[::7], s.ravel()[::7], t.ravel()[::7]):
            if Fraction(float(ss)) + Fraction(float(tt)) != Fraction(float(a)) + Fraction(float(b)):
                inexact += 1
    assert inexact > 0


# ---------------------------------------------------------------------------
# LayerNorm's mean: a signed sum. Each thread's values go into two packed pairs of chains:
# the pair of even pairs by the ordered Fast2Sum (the operand of larger magnitude first),
# the pair of odd pairs by TwoSum; both are exact for any signs. The halves are folded with
# TwoSum and the double words reduced across lanes and warps with TwoSum.
# ---------------------------------------------------------------------------

def _ordered_fast2sum(h, v):
    with np.errstate(invalid="ignore"):
        first = np.abs(h) >= np.abs(v)
        big, small = np.where(first, h, v).astype(f32), np.where(first, v, h).astype(f32)
        return _fast2sum(big, small)


def model_signed_sum(rows, G, steps=None):
    R, H = rows.shape
    V = 8
    C = (H + V - 1) // V
    nch = (C + 32 * G - 1) // (32 * G)
    pad = np.zeros((R, nch * G * 32 * V), f32)
    pad[:, :H] = rows
    x = pad.reshape(R, nch, G, 32, V)
    with np.errstate(over="ignore", invalid="ignore"):
        hi = [np.zeros((R, G, 32), f32) for _ in range(4)]  # chains: 2 * (pair parity) + half
        lo = [np.zeros((R, G, 32), f32) for _ in range(4)]
        for j in range(nch):
            for e in range(V // 2):
                for half in range(2):
                    k = 2 * (e & 1) + half
                    v = x[:, j, :, :, 2 * e + half]
                    s, t = _two_sum(hi[k], v) if e & 1 else _ordered_fast2sum(hi[k], v)
                    if steps is not None:
                        steps.append((hi[k].copy(), v.copy(), s, t))
                    hi[k], lo[k] = s, (lo[k] + t).astype(f32)
        d = _combine_signed(_combine_signed((hi[0], lo[0]), (hi[1], lo[1])),
                            _combine_signed((hi[2], lo[2]), (hi[3], lo[3])))
        for off in (16, 8, 4, 2, 1):
            perm = np.arange(32) ^ off
            d = _combine_signed(d, (d[0][:, :, perm], d[1][:, :, perm]))
        part = (d[0][:, :, 0], d[1][:, :, 0])
        G8 = 1
        while G8 < G:
            G8 <<= 1
        t = (np.zeros((R, G8), f32), np.zeros((R, G8), f32))
        t[0][:, :G], t[1][:, :G] = part
        off = G8 >> 1
        while off:
            perm = np.arange(G8) ^ off
            t = _combine_signed(t, (t[0][:, perm], t[1][:, perm]))
            off >>= 1
        h, l = t[0][:, 0], t[1][:, 0]
        return np.where(np.isfinite(h), (h + l).astype(f32), h).astype(f32)


def _rn32(q):
    """The binary32 value nearest the rational q, ties to even (q within the finite range)."""
    c = np.float32(float(q))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        dist = abs(Fraction(float(cand)) - q)
        key = (dist, int(cand.view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return best[1]


def _signed_rows(kind, R, H, seed):
    rng = np.random.default_rng(seed)
    if kind == "workload":
        return far_gen.custom_inputs("f32", "f32", R, H, seed=seed)["x"].numpy()
    if kind == "offset":  # a large mean over a small spread
        return (1000.0 + rng.standard_normal((R, H))).astype(f32)
    if kind == "cancelling":  # pairs of huge opposite values over small ones, in random lanes
        x = rng.standard_normal((R, H)).astype(f32)
        for r in range(R):
            i, k = rng.choice(H, 2, replace=False)
            big = f32(rng.uniform(1, 2) * 2.0 ** 40)
            x[r, i], x[r, k] = big, -big
        return x
    if kind == "wide":
        return (rng.choice([-1.0, 1.0], (R, H)) * np.exp2(rng.uniform(-100, 60, (R, H)))).astype(f32)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["workload", "offset", "wide"])
@pytest.mark.parametrize("H,G", [(8192, 4), (5120, 2), (1000, 1)])
def test_mean_chains_give_the_correctly_rounded_sum(kind, H, G):
    rows = _signed_rows(kind, 40, H, seed=H * 7 + G)
    got = model_signed_sum(rows, G)
    want = np.array([_rn32(sum((Fraction(float(v)) for v in r), Fraction(0))) for r in rows], f32)
    assert _same(got, want), np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0][:10]


@pytest.mark.parametrize("H,G", [(8192, 4), (5120, 2), (1000, 1)])
def test_mean_under_cancellation_stays_within_its_bound(H, G):
    """Where the row's partial sums dwarf its sum (two values of +-1.5 * 2^40 that cancel
    among N(0, 1) ones), the chains are still exact at every step, but the low parts that
    carry the small values are plain binary32 sums: their rounding errors, at most 2^-24 of
    each partial low sum, add up to a few tens of ulps of the mean's sum. Checked: the
    double word is within (chain length + 16) * 2^-24 * sum |t| of the exact sum, t the
    steps' error terms, and some rows do round differently (the limitation is real)."""
    rows = _signed_rows("cancelling", 40, H, seed=H * 7 + G)
    steps = []
    got = model_signed_sum(rows, G, steps=steps)
    chain_len = len(steps) // 4
    abs_t = sum(np.abs(t.astype(np.float64)).sum(axis=(1, 2)) for _, _, _, t in steps)  # per row
    off = 0
    for r in range(len(rows)):
        exact = sum((Fraction(float(v)) for v in rows[r]), Fraction(0))
        bound = Fraction((chain_len + 16) * abs_t[r]) * Fraction(1, 1 << 24) + abs(exact) * Fraction(1, 1 << 24)
        assert abs(Fraction(float(got[r])) - exact) <= bound, r
        off += got[r] != _rn32(exact)
    assert off > 0


def test_every_mean_step_is_exact():
    """Each step of both kinds of chain: s + t equals hi + v exactly (rationals)."""
    for kind in ("wide", "cancelling", "offset"):
        rows = _signed_rows(kind, 3, 1024, seed=11)
        steps = []
        model_signed_sum(rows, 1, steps=steps)
        for hi, v, s, t in steps:
            for a, b, ss, tt in zip(hi.ravel()[::3], v.ravel()[::3], s.ravel()[::3], t.ravel()[::3]):
                assert Fraction(float(ss)) + Fraction(float(tt)) == Fraction(float(a)) + Fraction(float(b))
