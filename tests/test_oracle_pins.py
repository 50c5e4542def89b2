"""The oracle against its pins (see oracle_pins for what pins what)."""
import itertools

import pytest
import torch

import far_gen
import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def L():
    return oracle.lib()


@pytest.fixture(scope="module")
def cases():
    return P.pin_cases()


def test_policy(L):
    P.pin_policy(L)


def test_residual(L, cases):
    P.pin_residual(L, cases)


def test_sum(L, cases):
    P.pin_sum(L, cases)


def test_steps(L, cases):
    P.pin_steps(L, cases)


def test_closed_forms(L):
    P.pin_closed_forms(L)


def test_fp64(L, cases):
    P.pin_fp64(L, cases)


def test_exhaustive_hidden_1(L):
    """Every finite fp16 and bf16 x at hidden = 1, every step against binary64."""
    assert P.finite_values("f16").shape[0] == 65536 - 2 * 1024   # 2 x (1023 NaN + 1 inf)
    assert P.finite_values("bf16").shape[0] == 65536 - 2 * 128   # 2 x (127 NaN + 1 inf)
    P.pin_exhaustive_h1(L)


def _matrix_cases():
    g = P.golden("contract.json")["test_matrix"]
    return list(itertools.product(g["dtypes"], g["tokens"], g["hidden"]))


@pytest.mark.parametrize("act,tokens,hidden", _matrix_cases())
def test_case_study_matrix(L, act, tokens, hidden):
    """The eight focused regressions of the case study: every pin on that shape.

    Exact-sum and step checks run on the first rows (they are exact-rational and
    slow); residual, fp64 and tolerance checks cover every row.
    """
    d = far_gen.custom_inputs(act, act, tokens, hidden, seed=tokens + hidden)
    P.pin_residual(L, [d])
    P.pin_fp64(L, [d])
    few = dict(d, x=d["x"][:2].contiguous(), r=d["r"][:2].contiguous(), tokens=2)
    P.pin_sum(L, [few])
    P.pin_steps(L, [few])


def test_threaded_driver_matches_single_call(L):
    d = far_gen.make_inputs("c3", rows=37)
    a = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], "bf16", "f32", threads=1)
    b = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], "bf16", "f32", threads=5)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = oracle.rmsnorm(d["x"], d["w"], d["eps"], "bf16", "f32", threads=1)
    e = oracle.rmsnorm(d["x"], d["w"], d["eps"], "bf16", "f32", threads=7)
    assert torch.equal(c, e)


def test_rejects_f16_with_bf16(L):
    x = torch.zeros((1, 8), dtype=torch.float16)
    w = torch.ones(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.fused_add_rmsnorm(x, x, w, 1e-6, "f16", "bf16")
    with pytest.raises(ValueError):
        oracle.rmsnorm(x, w, 1e-6, "f16", "bf16")


def test_empty_token_count(L):
    x = torch.zeros((0, 16), dtype=torch.bfloat16)
    w = torch.ones(16, dtype=torch.bfloat16)
    out, res = oracle.fused_add_rmsnorm(x, x, w, 1e-6, "bf16", "bf16")
    assert out.shape == (0, 16) and res.shape == (0, 16)


def test_special_values_propagate(L):
    """inf and NaN in a row: NaN spreads through the row's var; rows are independent."""
    x = torch.ones((3, 8), dtype=torch.float16)
    r = torch.zeros((3, 8), dtype=torch.float16)
    x[0, 3] = float("nan")
    x[1, 2] = float("inf")
    w = torch.ones(8, dtype=torch.float16)
    out, res = oracle.fused_add_rmsnorm(x, r, w, 1e-6, "f16", "f16")
    assert torch.isnan(out[0]).all()
    assert torch.isnan(res[0, 3]) and not torch.isnan(res[0, :3]).any()
    # an infinite element: S = inf, rstd = 0, finite elements give 0, the infinite one NaN
    assert torch.isinf(res[1, 2])
    assert torch.isnan(out[1, 2]) and (out[1, [0, 1, 3, 4, 5, 6, 7]] == 0).all()
    assert torch.equal(out[2], torch.ones(8, dtype=torch.float16))
