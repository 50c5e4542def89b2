"""Fused residual-add + LayerNorm and its no-residual variant against the oracle,
through the C ABI, with the parity gate of the RMSNorm path: residual_out bit for
bit, out within 1 ULP of its dtype with fewer than 1% of elements differing.
Outputs sit between canary bands that must survive every call."""
import numpy as np
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import Guarded, gate, square_sensitive_rows, to_device
from oracle_pins import bits_equal

pytestmark = pytest.mark.gpu
PAIRS = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f16", "f32"), ("f32", "f32"), ("f32", "bf16"),
         ("f32", "f16")]


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    far.set_launch_override()
    return far


def with_beta(d, seed=0):
    d = dict(d)
    d["b"] = far_gen.ln_beta(d, seed)
    return d


def run_ln(far, d, residual=True, offset=0, inplace=False, beta_offset=0):
    """One call through the C ABI on guarded device buffers; CPU results."""
    x, w, b = to_device(d["x"], offset), to_device(d["w"]), to_device(d["b"], beta_offset)
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    tokens, hidden = d["x"].shape
    code = far.dtypes(d["x"].dtype, d["w"].dtype)
    stream = torch.cuda.current_stream().cuda_stream
    if residual:
        r = to_device(d["r"], offset)
        out = x if inplace and od == d["x"].dtype else Guarded(tuple(d["x"].shape), od, offset)
        res = r if inplace else Guarded(tuple(d["x"].shape), d["x"].dtype, offset)
        st = far.lib.fused_add_layernorm(x.t.data_ptr(), r.t.data_ptr(), w.t.data_ptr(), b.t.data_ptr(), d["eps"],
                                         out.t.data_ptr(), res.t.data_ptr(), tokens, hidden, code, stream)
    else:
        out = x if inplace and od == d["x"].dtype else Guarded(tuple(d["x"].shape), od, offset)
        res = None
        st = far.lib.layernorm(x.t.data_ptr(), w.t.data_ptr(), b.t.data_ptr(), d["eps"], out.t.data_ptr(), tokens,
                               hidden, code, stream)
    assert st == 0, far.lib.far_status_string(st)
    assert far.device_status() == 0
    for g in (out, res):
        if g is not None:
            assert g.guards_intact(), "a store landed outside its output"
    return out.t.cpu(), None if res is None else res.t.cpu()


def check_ln(far, d, where, offset=0, inplace=False):
    out, res = run_ln(far, d, True, offset, inplace)
    ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
    gate(out, ro, res, rr, where=f"{where} fused")
    out, _ = run_ln(far, d, False, offset, inplace)
    ro = oracle.layernorm(d["x"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
    gate(out, ro, where=f"{where} layernorm")


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_workloads(far, name):
    check_ln(far, with_beta(far_gen.make_inputs(name)), name)


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_workload_rows(far, name):
    check_ln(far, with_beta(far_gen.make_inputs(name, rows=600)), name)


@pytest.mark.parametrize("act,wd", PAIRS)
@pytest.mark.parametrize("hidden", [1, 8, 100, 2048, 4096, 5120, 8192])
def test_dtype_pairs(far, act, wd, hidden):
    d = with_beta(far_gen.custom_inputs(act, wd, 33, hidden, seed=hidden + 1, scale_lo=1e-3, scale_hi=30))
    check_ln(far, d, f"{act}/{wd} H={hidden}")


@pytest.mark.parametrize("act,wd", [("bf16", "bf16"), ("f16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("hidden", [256, 768, 1024, 2560, 3000, 3072, 5120, 6144, 10240])
@pytest.mark.parametrize("tokens", [600, 2500])
def test_default_plans_across_widths(far, act, wd, hidden, tokens):
    """The default plans (short one-warp rows in 7 groups, 8 chunks a thread above, the
    variant's exact 5 or 6 chunks on 16-bit rows of 2560, 3072 and 5120) at 4 and 17 rows
    an SM."""
    d = with_beta(far_gen.custom_inputs(act, wd, tokens, hidden, seed=hidden + tokens))
    check_ln(far, d, f"{act}/{wd} {tokens}x{hidden}")


@pytest.mark.parametrize("tokens", [1, 2, 151, 152, 153, 1000, 4096])
def test_token_counts(far, tokens):
    d = with_beta(far_gen.custom_inputs("bf16", "bf16", tokens, 4096, seed=tokens))
    check_ln(far, d, f"tokens={tokens}")


@pytest.mark.parametrize("hidden", [12288, 16384, 32768, 65536, 1 << 17])
def test_large_hidden(far, hidden):
    d = with_beta(far_gen.custom_inputs("f16", "f16", 24, hidden, seed=hidden))
    check_ln(far, d, f"H={hidden}")


def test_every_plan_gives_the_same_bits(far):
    """Generic kernel and staged plans of every shape: one set of bits."""
    d = with_beta(far_gen.custom_inputs("f16", "f16", 200, 8192, seed=9))
    ref = None
    try:
        for plan in [(1, 0, 0, 0), (0, 4, 1, 2), (0, 8, 1, 0), (0, 2, 0, 0), (0, 4, 3, 3), (0, 8, 2, 4),
                     (0, 1, 0, 0)]:
            far.set_launch_override(*plan)
            got = run_ln(far, d, True)
            if ref is None:
                ref = got
                ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
                gate(got[0], ro, got[1], rr, where=f"plan {plan}")
            else:
                assert bits_equal(got[0], ref[0]) and bits_equal(got[1], ref[1]), plan
    finally:
        far.set_launch_override()


@pytest.mark.parametrize("act", ["f16", "f32"])
def test_fp16_weight_extremes_every_plan(far, act):
    """fp16 gamma and beta at the fp16 extremes (largest finite, smallest subnormal, signed
    zeros, infinity): the generic kernel and staged plans of 1 to 8 chunks a thread give one
    set of bits, fused and not, with fp16 and binary32 x, and pass the oracle's gate."""
    d = with_beta(far_gen.custom_inputs(act, "f16", 96, 8192, seed=44, scale_lo=1e-2, scale_hi=60))
    w, b = d["w"].clone(), d["b"].clone()
    ext = torch.tensor([65504.0, -65504.0, 2.0 ** -24, -(2.0 ** -24), 2.0 ** -14, 0.0, -0.0, 1.0, 1024.5,
                        float("inf")], dtype=torch.float16)
    w[: 4 * len(ext)] = ext.repeat(4)
    b[: 4 * len(ext)] = ext.flip(0).repeat(4)
    b[100:140] = torch.tensor([65504.0, -(2.0 ** -24), -0.0, 3.0e-5], dtype=torch.float16).repeat(10)
    d = dict(d, w=w, b=b)
    for residual in (True, False):
        ref = None
        try:
            for plan in [(1, 0, 0, 0), (0, 1, 0, 0), (0, 2, 0, 0), (0, 4, 1, 2), (0, 4, 3, 3), (0, 8, 1, 0),
                         (0, 8, 2, 4)]:
                far.set_launch_override(*plan)
                got = run_ln(far, d, residual)
                if ref is None:
                    ref = got
                    if residual:
                        ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"],
                                                            d["wd"])
                        gate(got[0], ro, got[1], rr, where=f"{act}/f16 extremes fused")
                    else:
                        gate(got[0], oracle.layernorm(d["x"], d["w"], d["b"], d["eps"], d["act"], d["wd"]),
                             where=f"{act}/f16 extremes")
                else:
                    assert bits_equal(got[0], ref[0]), (residual, plan)
                    if residual:
                        assert bits_equal(got[1], ref[1]), (residual, plan)
        finally:
            far.set_launch_override()


@pytest.mark.parametrize("offset", [1, 3])
def test_misaligned_buffers(far, offset):
    d = with_beta(far_gen.custom_inputs("bf16", "bf16", 40, 1000, seed=offset))
    check_ln(far, d, f"offset={offset}", offset=offset)


def test_misaligned_beta(far):
    """Everything aligned but beta: the staged kernel's vector copy of beta would be
    misaligned, so the call must take the generic kernel and still match."""
    d = with_beta(far_gen.custom_inputs("bf16", "bf16", 40, 4096, seed=21))
    for residual in (True, False):
        out, res = run_ln(far, d, residual, beta_offset=1)
        if residual:
            ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
            gate(out, ro, res, rr, where="misaligned beta fused")
        else:
            gate(out, oracle.layernorm(d["x"], d["w"], d["b"], d["eps"], d["act"], d["wd"]),
                 where="misaligned beta")


def test_in_place(far):
    d = with_beta(far_gen.custom_inputs("bf16", "bf16", 64, 4096, seed=17))
    check_ln(far, d, "in place", inplace=True)


def test_special_rows(far):
    """A constant row (d = 0: out is beta exactly), a row with a large common offset
    (heavy cancellation in the mean), an all-zero row, NaN and infinity."""
    d = with_beta(far_gen.custom_inputs("bf16", "bf16", 8, 1024, seed=2))
    x, r = d["x"].clone(), d["r"].clone()
    x[0] = 1.5
    r[0] = 0.25
    x[1] = (x[1].float() + 1000.0).to(x.dtype)
    x[2] = 0.0
    r[2] = 0.0
    x[3, 5] = float("nan")
    x[4, 9] = float("inf")
    d = dict(d, x=x, r=r)
    check_ln(far, d, "special rows")
    out, _ = run_ln(far, d, True)
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    assert bits_equal(out[0], d["b"].to(od)), "a constant row must give beta"


def test_eps_values(far):
    for eps in (0.0, 1e-12, 1e-5, 1.0):
        d = with_beta(dict(far_gen.custom_inputs("f16", "f32", 16, 2048, seed=7), eps=eps))
        check_ln(far, d, f"eps={eps}")


def test_rejections(far):
    x = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    g = torch.ones(64, dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream().cuda_stream
    code = far.dtypes(x.dtype, g.dtype)
    assert far.lib.layernorm(x.data_ptr(), g.data_ptr(), None, 1e-5, out.data_ptr(), 4, 64, code, stream) == 3
    b = torch.zeros(4 * 64, dtype=torch.float16, device="cuda")
    # out overlapping beta
    assert far.lib.layernorm(x.data_ptr(), g.data_ptr(), b.data_ptr(), 1e-5, b.data_ptr(), 4, 64, code, stream) == 5
    # the fp16 / bf16 mix is refused as for RMSNorm
    gb = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    assert far.lib.layernorm(x.data_ptr(), gb.data_ptr(), gb.data_ptr(), 1e-5, out.data_ptr(), 4, 64,
                             1 | (2 << 4), stream) == 1  # act f16, weight bf16


def test_binding(far):
    d = with_beta(far_gen.custom_inputs("bf16", "f32", 32, 2048, seed=5))
    out, res = far.fused_add_layernorm(d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), d["b"].cuda(), d["eps"])
    ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
    gate(out.cpu(), ro, res.cpu(), rr, where="binding fused")
    out = far.layernorm(d["x"].cuda(), d["w"].cuda(), d["b"].cuda(), d["eps"])
    gate(out.cpu(), oracle.layernorm(d["x"], d["w"], d["b"], d["eps"], d["act"], d["wd"]), where="binding")


def test_rounded_squares_are_summed(far):
    """The variance sums fl32(d * d), each square rounded, not the exact squares (as a
    fused multiply-add would): rows where the two sums round to different binary32
    values and so change rstd must still pass the gate."""
    d = far_gen.custom_inputs("f32", "f32", 6000, 64, seed=31, scale_lo=0.5, scale_hi=2.0, eps=0.0)
    x = d["x"].numpy()
    mean, rstd = oracle.ln_row_stats(d["x"], None, 0.0, "f32")
    dev = (x - mean[:, None]).astype(np.float32)  # fl32(s - mean)
    var_sums = oracle_sums_of_squares(dev)
    rows = np.nonzero(square_sensitive_rows(dev, var_sums, 0.0))[0]
    assert len(rows) >= 20, len(rows)
    sel = dict(d, x=d["x"][rows].contiguous(), r=d["r"][rows].contiguous(), tokens=len(rows))
    sel = with_beta(sel)
    try:
        for plan in [(-1, 0, 0, 0), (1, 0, 0, 0)]:
            far.set_launch_override(*plan)
            out, _ = run_ln(far, sel, False)
            gate(out, oracle.layernorm(sel["x"], sel["w"], sel["b"], 0.0, "f32", "f32"),
                 where=f"rounded squares {plan}")
    finally:
        far.set_launch_override()


def oracle_sums_of_squares(dev):
    return np.array([oracle.exact_sum((row * row).astype(np.float32)) for row in dev], np.float32)


@pytest.mark.parametrize("act,wd,hidden", [("bf16", "bf16", 4096), ("f16", "f32", 1000), ("f32", "f32", 2048)])
def test_strided_rows(far, act, wd, hidden):
    """Column slices of wider buffers (x, residual, out, residual_out interleaved): bit for
    bit the contiguous result, and the oracle's gate."""
    d = with_beta(far_gen.custom_inputs(act, wd, 48, hidden, seed=hidden + 9))
    T, H = 48, hidden
    x_c, r_c, w, b = d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), d["b"].cuda()
    od = far.output_dtype(x_c.dtype, w.dtype)
    wide = torch.zeros((T, 4 * H), dtype=x_c.dtype, device="cuda")
    x, r = wide[:, 0:H], wide[:, 2 * H:3 * H]
    x.copy_(x_c)
    r.copy_(r_c)
    res = wide[:, 3 * H:4 * H]
    outw = torch.zeros((T, 2 * H), dtype=od, device="cuda")
    out = outw[:, H:2 * H]
    far.fused_add_layernorm(x, r, w, b, d["eps"], out=out, residual_out=res)
    ref_out, ref_res = far.fused_add_layernorm(x_c, r_c, w, b, d["eps"])
    assert far.device_status() == 0
    assert bits_equal(out.cpu(), ref_out.cpu()) and bits_equal(res.cpu(), ref_res.cpu())
    ro, rr = oracle.fused_add_layernorm(d["x"], d["r"], d["w"], d["b"], d["eps"], d["act"], d["wd"])
    gate(out.cpu(), ro, res.cpu(), rr, where=f"strided fused {act}/{wd}")
    nout = far.layernorm(x, w, b, d["eps"], out=outw[:, 0:H])
    assert far.device_status() == 0
    assert bits_equal(nout.cpu(), far.layernorm(x_c, w, b, d["eps"]).cpu())


def test_host_buffers(far):
    """The host-buffer pipeline (several chunks through a small workspace) gives the device
    path's bits."""
    d = with_beta(far_gen.custom_inputs("bf16", "f32", 300, 2048, seed=41))
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    ws = torch.empty(far.host_workspace_bytes_op(64, 2048, d["x"].dtype, d["w"].dtype, True, "layernorm"),
                     dtype=torch.uint8, device="cuda")
    xh, rh, wh, bh = (t.pin_memory() for t in (d["x"], d["r"], d["w"], d["b"]))
    out = torch.empty((300, 2048), dtype=od).pin_memory()
    res = torch.empty_like(d["x"]).pin_memory()
    far.fused_add_layernorm_host(xh, rh, wh, bh, d["eps"], out, res, ws)
    nout = torch.empty((300, 2048), dtype=od).pin_memory()
    far.layernorm_host(xh, wh, bh, d["eps"], nout, ws)
    torch.cuda.synchronize()
    assert far.device_status() == 0
    ref_out, ref_res = far.fused_add_layernorm(d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), d["b"].cuda(), d["eps"])
    assert bits_equal(out, ref_out.cpu()) and bits_equal(res, ref_res.cpu())
    assert bits_equal(nout, far.layernorm(d["x"].cuda(), d["w"].cuda(), d["b"].cuda(), d["eps"]).cpu())
