"""The large workloads at full size, in the launch configuration the bench times.

The fp16 65536 x 8192 workload (RMSNorm and LayerNorm) is compared with the oracle on sampled rows
(first, last and spread rows) and its residual_out on every element (a
property that holds at any size: RNE_act(fl32(x + r)), rebuilt with torch's
binary32 add and RNE cast); the bf16 16384 x 5120 workload is compared with
the oracle on every row, for both variants.
"""
import numpy as np
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import gate
from oracle_pins import bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    far.set_launch_override()
    return far


def _run(far, d):
    x, r, w = d["x"].cuda(), d["r"].cuda(), d["w"].cuda()
    out, res = far.fused_add_rmsnorm(x, r, w, d["eps"])
    nout = far.rmsnorm(x, w, d["eps"])
    assert far.device_status() == 0
    return out.cpu(), res.cpu(), nout.cpu()


def test_bf16_16384x5120_every_row(far):
    d = far_gen.make_inputs("c4")
    out, res, nout = _run(far, d)
    ref_out, ref_res = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], "bf16", "bf16")
    gate(out, ref_out, res, ref_res, "c4 fused")
    gate(nout, oracle.rmsnorm(d["x"], d["w"], d["eps"], "bf16", "bf16"), where="c4 rmsnorm")


def test_f16_65536x8192_sampled_rows(far):
    d = far_gen.make_inputs("c5")
    out, res, nout = _run(far, d)
    # residual_out everywhere, by its defining property (binary32 add, one RNE cast)
    for t0 in range(0, d["tokens"], 8192):
        sl = slice(t0, t0 + 8192)
        ref = (d["x"][sl].float() + d["r"][sl].float()).half()
        assert bits_equal(res[sl], ref), f"residual_out rows {t0}.."
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(d["tokens"] - 64, d["tokens"]),
                                     rng.choice(d["tokens"], 1920, replace=False)]))
    idx = torch.from_numpy(rows)
    x, r = d["x"][idx].contiguous(), d["r"][idx].contiguous()
    ref_out, ref_res = oracle.fused_add_rmsnorm(x, r, d["w"], d["eps"], "f16", "f16")
    gate(out[idx], ref_out, res[idx], ref_res, "c5 fused (sampled rows)")
    gate(nout[idx], oracle.rmsnorm(x, d["w"], d["eps"], "f16", "f16"), where="c5 rmsnorm (sampled rows)")


def test_layernorm_f16_65536x8192_sampled_rows(far):
    """LayerNorm on the same workload in the bench's launch plans, sampled rows."""
    d = far_gen.make_inputs("c5")
    b = far_gen.ln_beta(d)
    x, r, w, bb = d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), b.cuda()
    out, res = far.fused_add_layernorm(x, r, w, bb, d["eps"])
    nout = far.layernorm(x, w, bb, d["eps"])
    assert far.device_status() == 0
    out, res, nout = out.cpu(), res.cpu(), nout.cpu()
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(0, 32), np.arange(d["tokens"] - 32, d["tokens"]),
                                     rng.choice(d["tokens"], 960, replace=False)]))
    idx = torch.from_numpy(rows)
    xs, rs = d["x"][idx].contiguous(), d["r"][idx].contiguous()
    ref_out, ref_res = oracle.fused_add_layernorm(xs, rs, d["w"], b, d["eps"], "f16", "f16")
    gate(out[idx], ref_out, res[idx], ref_res, "c5 layernorm fused (sampled rows)")
    gate(nout[idx], oracle.layernorm(xs, d["w"], b, d["eps"], "f16", "f16"), where="c5 layernorm (sampled rows)")


def test_gemm_8192_cubed_sampled_rows(far):
    """The GEMM at the bench's shape and plan (256 x 256 tiles over CTA pairs): on dyadic
    operands (every binary32 sum exact) 32 sampled rows bit for bit; on random operands the
    same rows against the oracle under the page's tolerance and the bound that any order of
    binary32 additions meets (2 fp16 ULP + K * 2^-22 * sum |x * w|, two more fp16 ULP of the
    unbiased value for the bias add)."""
    M = N = K = 8192
    far.set_gemm_override()
    assert far.plan_gemm_for_sms(M, N, K, True, torch.float16, 152)["kind"] == 2
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, M - 1], rng.choice(M, 26, replace=False)]))
    idx = torch.from_numpy(rows)
    g = far_gen.gemm_dyadic_inputs(M, N, K, seed=3)
    y = far.gemm_f16_f32acc(g["x"].cuda(), g["wt"].cuda(), g["bias"].cuda())
    assert far.device_status() == 0
    ref = oracle.gemm_f16(g["x"][idx].contiguous(), g["wt"], g["bias"], "f16")
    assert torch.equal(y.cpu()[idx].view(torch.int16), ref.view(torch.int16)), "dyadic rows differ"
    g = far_gen.gemm_inputs(M, N, K, seed=4)
    y = far.gemm_f16_f32acc(g["x"].cuda(), g["wt"].cuda(), g["bias"].cuda())
    assert far.device_status() == 0
    assert len(rows) == 32
    xs = g["x"][idx].contiguous()
    ref = oracle.gemm_f16(xs, g["wt"], g["bias"], "f16")
    p_ref = oracle.gemm_f16(xs, g["wt"], None, "f16")
    got = y.cpu()[idx]
    assert np.isfinite(got.double().numpy()).all()
    from test_gpu_gemm import gate_f16

    gate_f16(got, ref, dict(g, x=xs, M=len(rows)), "8192^3 random, sampled rows", p_ref=p_ref)
    p = far.gemm_f16_f32acc(g["x"].cuda(), g["wt"].cuda(), None)
    assert far.device_status() == 0
    gate_f16(p.cpu()[idx], p_ref, dict(g, x=xs, M=len(rows)), "8192^3 random, no bias, sampled rows")
