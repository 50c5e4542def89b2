"""The quantised-output variants (per-token scale, int8 or FP8 E4M3) against the
oracle, through the C ABI.  The gate: residual_out bit for bit; scale bit for bit
(it is a function of the row maximum, exact whenever out matches); q equal
wherever out matches the oracle, and within one quantisation step where out
differs by its allowed one ULP (fewer than 1% of elements)."""
import numpy as np
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import gate
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


def _q_gate(q, scale, ref_q, ref_scale, where):
    assert bits_equal(scale, ref_scale), f"{where}: scale differs"
    a = q.numpy().astype(np.int64)
    b = ref_q.numpy().astype(np.int64)
    if q.dtype == torch.uint8:  # E4M3 codes: compare decoded values, NaN equal to NaN
        av = q.view(torch.float8_e4m3fn).float().numpy()
        bv = ref_q.view(torch.float8_e4m3fn).float().numpy()
        same = (av == bv) | (np.isnan(av) & np.isnan(bv))
        # one E4M3 step apart where out itself differs by one ULP
        step_ok = np.abs(np.abs(a & 0x7F) - np.abs(b & 0x7F)) <= 1
        assert (same | step_ok).all(), f"{where}: q differs by more than one E4M3 step"
    else:
        same = a == b
        assert (np.abs(a - b) <= 1).all(), f"{where}: q differs by more than one int8 step"
    frac = float((~same).mean())
    assert frac < 0.01, f"{where}: {frac:.4%} of q differ"


def run_quant(far, d, qtype, residual=True):
    x, r, w = d["x"].cuda(), d["r"].cuda(), d["w"].cuda()
    if residual:
        q, scale, res = far.fused_add_rmsnorm_quant(x, r, w, d["eps"], qtype)
    else:
        q, scale = far.rmsnorm_quant(x, w, d["eps"], qtype)
        res = None
    assert far.device_status() == 0
    return q.cpu(), scale.cpu(), None if res is None else res.cpu()


def check_quant(far, d, where):
    for qtype in ("int8", "fp8"):
        q, scale, res = run_quant(far, d, qtype, True)
        rq, rs, rres = oracle.fused_add_rmsnorm_quant(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"], qtype)
        assert bits_equal(res, rres), f"{where} {qtype}: residual_out differs"
        _q_gate(q.view(torch.uint8) if qtype == "fp8" else q, scale, rq, rs, f"{where} {qtype} fused")
        q, scale, _ = run_quant(far, d, qtype, False)
        rq, rs = oracle.rmsnorm_quant(d["x"], d["w"], d["eps"], d["act"], d["wd"], qtype)
        _q_gate(q.view(torch.uint8) if qtype == "fp8" else q, scale, rq, rs, f"{where} {qtype} rmsnorm")


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_workloads(far, name):
    check_quant(far, far_gen.make_inputs(name), name)


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_workload_rows(far, name):
    check_quant(far, far_gen.make_inputs(name, rows=600), name)


@pytest.mark.parametrize("act,wd", PAIRS)
@pytest.mark.parametrize("hidden", [1, 8, 100, 2048, 4096, 5120, 8192])
def test_dtype_pairs(far, act, wd, hidden):
    d = far_gen.custom_inputs(act, wd, 33, hidden, seed=hidden + 1, scale_lo=1e-3, scale_hi=30)
    check_quant(far, d, f"{act}/{wd} H={hidden}")


@pytest.mark.parametrize("act,wd", [("bf16", "bf16"), ("f16", "f16"), ("f32", "f32")])
@pytest.mark.parametrize("hidden", [256, 1024, 2048, 3072, 4096, 6144, 7168, 12288])
@pytest.mark.parametrize("tokens", [600, 2500])
def test_default_plans_across_widths(far, act, wd, hidden, tokens):
    """The default plans (8 chunks a thread on rows they cover exactly, else 4; up to 12
    one-warp groups; 8 warps for fused rows of 2+ warps) at 4 and 17 rows an SM."""
    d = far_gen.custom_inputs(act, wd, tokens, hidden, seed=hidden + tokens, scale_lo=1e-2, scale_hi=50.0)
    check_quant(far, d, f"{act}/{wd} {tokens}x{hidden}")


def test_generic_path_and_plans(far):
    d = far_gen.custom_inputs("f16", "f16", 200, 8192, seed=9)
    try:
        for plan in [(1, 0, 0, 0), (0, 4, 1, 2), (0, 8, 1, 0), (0, 2, 0, 0)]:
            far.set_launch_override(*plan)
            check_quant(far, d, f"plan {plan}")
    finally:
        far.set_launch_override()


def test_special_rows(far):
    """All-zero rows (scale 0, q 0), rows with NaN (NaN scale) and infinity."""
    d = far_gen.custom_inputs("bf16", "bf16", 8, 1024, seed=2)
    x, r = d["x"].clone(), d["r"].clone()
    x[0] = 0.0
    r[0] = 0.0
    x[1, 5] = float("nan")
    x[2, 9] = float("inf")
    check_quant(far, dict(d, x=x, r=r), "special rows")


def test_quant_rejections(far):
    x = torch.zeros((4, 64), dtype=torch.float16, device="cuda")
    w = torch.ones(64, dtype=torch.float16, device="cuda")
    scale = torch.empty(4, dtype=torch.float32, device="cuda")
    q = torch.empty((4, 64), dtype=torch.int8, device="cuda")
    st = far.lib.fused_add_rmsnorm_quant(x.data_ptr(), x.data_ptr(), w.data_ptr(), 1e-6, q.data_ptr(),
                                         scale.data_ptr(), x.data_ptr(), 4, 64, far.dtypes(x.dtype, w.dtype), 3,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 2  # unknown quantisation type
    st = far.lib.rmsnorm_quant(x.data_ptr(), w.data_ptr(), 1e-6, x.data_ptr(), scale.data_ptr(), 4, 64,
                               far.dtypes(x.dtype, w.dtype), 1, torch.cuda.current_stream().cuda_stream)
    assert st == 5  # q over x


def _quantise_given_out(out, qtype, L):
    """The quantisation step alone, applied to given out values the way the oracle takes
    it: amax per row, scale = fl32(amax / QMAX), inv = fl32(QMAX / amax) (0 for a zero
    row), codes = Q(fl32(out * inv)) by the oracle's pinned converters; binary32 steps
    by numpy's IEEE float32 arithmetic."""
    o = out.float().numpy()
    qmax = np.float32(127.0 if qtype == "int8" else 448.0)
    amax = np.max(np.abs(o), axis=1).astype(np.float32)
    scale = (amax / qmax).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(amax == 0, np.float32(0), qmax / amax).astype(np.float32)
    v = (o * inv[:, None]).astype(np.float32)
    conv = L.oracle_f32_to_int8 if qtype == "int8" else L.oracle_f32_to_e4m3
    codes = np.array([conv(float(t)) for t in v.ravel()], dtype=np.int64).reshape(v.shape)
    return codes, scale


@pytest.mark.parametrize("act,wd,hidden", [("bf16", "bf16", 4096), ("f16", "f16", 8192), ("f32", "f32", 2048),
                                           ("bf16", "f32", 5120), ("f16", "f16", 1000)])
def test_quantisation_bit_exact_given_out(far, act, wd, hidden):
    """Where floating point decides the integer codes, both sides decide from the same
    values: the GPU's own out (from the plain kernel, same arithmetic) quantised by the
    oracle's steps must equal the quantised kernel's codes and scales bit for bit."""
    L = oracle.lib()
    d = far_gen.custom_inputs(act, wd, 48, hidden, seed=hidden + 3, scale_lo=1e-2, scale_hi=50)
    x, r, w = d["x"].cuda(), d["r"].cuda(), d["w"].cuda()
    for residual in (True, False):
        out = far.fused_add_rmsnorm(x, r, w, d["eps"])[0] if residual else far.rmsnorm(x, w, d["eps"])
        assert far.device_status() == 0
        for qtype in ("int8", "fp8"):
            q, scale, _ = run_quant(far, d, qtype, residual)
            codes, want_scale = _quantise_given_out(out.cpu(), qtype, L)
            got = q.numpy().astype(np.int64) if qtype == "int8" else q.view(torch.uint8).numpy().astype(np.int64)
            assert np.array_equal(scale.numpy().view(np.uint32), want_scale.view(np.uint32)), (qtype, residual)
            assert np.array_equal(got, codes), f"{act}/{wd} H={hidden} {qtype} residual={residual}: codes differ"


@pytest.mark.parametrize("act,wd,hidden", [("bf16", "bf16", 4096), ("f16", "f16", 1000), ("f32", "f32", 2048)])
def test_strided_inputs(far, act, wd, hidden):
    """x, the residual and residual_out as column slices: against the oracle (residual_out
    and scale bit for bit, q within the quantised gate), and bit for bit the contiguous
    call's (q and scale stay contiguous)."""
    d = far_gen.custom_inputs(act, wd, 40, hidden, seed=hidden + 2)
    T, H = 40, hidden
    x_c, r_c, w = d["x"].cuda(), d["r"].cuda(), d["w"].cuda()
    wide = torch.zeros((T, 3 * H), dtype=x_c.dtype, device="cuda")
    x, r, res = wide[:, 0:H], wide[:, H:2 * H], wide[:, 2 * H:3 * H]
    x.copy_(x_c)
    r.copy_(r_c)
    for qtype in ("int8", "fp8"):
        rq, rs, rres = oracle.fused_add_rmsnorm_quant(d["x"], d["r"], d["w"], d["eps"], act, wd, qtype)
        q, s, res_o = far.fused_add_rmsnorm_quant(x, r, w, d["eps"], qtype, residual_out=res)
        q_c, s_c, res_c = far.fused_add_rmsnorm_quant(x_c, r_c, w, d["eps"], qtype)
        assert far.device_status() == 0
        assert bits_equal(res.cpu(), rres), f"strided {qtype}: residual_out differs from the oracle"
        _q_gate(q.cpu().view(torch.uint8) if qtype == "fp8" else q.cpu(), s.cpu(), rq, rs, f"strided {qtype} fused")
        assert torch.equal(q.cpu(), q_c.cpu()) and bits_equal(s.cpu(), s_c.cpu()) and bits_equal(res.cpu(), res_c.cpu())
        rq, rs = oracle.rmsnorm_quant(d["x"], d["w"], d["eps"], act, wd, qtype)
        q, s = far.rmsnorm_quant(x, w, d["eps"], qtype)
        q_c, s_c = far.rmsnorm_quant(x_c, w, d["eps"], qtype)
        assert far.device_status() == 0
        _q_gate(q.cpu().view(torch.uint8) if qtype == "fp8" else q.cpu(), s.cpu(), rq, rs, f"strided {qtype}")
        assert torch.equal(q.cpu(), q_c.cpu()) and bits_equal(s.cpu(), s_c.cpu())


def test_host_buffers(far):
    """The host-buffer pipeline for the quantised outputs against the oracle (the quantised
    gate), and bit for bit the device path's."""
    d = far_gen.custom_inputs("f16", "f16", 300, 4096, seed=43)
    xh, rh, wh = (t.pin_memory() for t in (d["x"], d["r"], d["w"]))
    for qtype in ("int8", "fp8"):
        ws = torch.empty(far.host_workspace_bytes_op(64, 4096, d["x"].dtype, d["w"].dtype, True, "quant"),
                         dtype=torch.uint8, device="cuda")
        qdt = torch.int8 if qtype == "int8" else torch.uint8
        q = torch.empty((300, 4096), dtype=qdt).pin_memory()
        sc = torch.empty(300, dtype=torch.float32).pin_memory()
        res = torch.empty_like(d["x"]).pin_memory()
        far.fused_add_rmsnorm_quant_host(xh, rh, wh, d["eps"], qtype, q, sc, res, ws)
        q2 = torch.empty((300, 4096), dtype=qdt).pin_memory()
        sc2 = torch.empty(300, dtype=torch.float32).pin_memory()
        far.rmsnorm_quant_host(xh, wh, d["eps"], qtype, q2, sc2, ws)
        torch.cuda.synchronize()
        assert far.device_status() == 0
        oq, os_, ores = oracle.fused_add_rmsnorm_quant(d["x"], d["r"], d["w"], d["eps"], "f16", "f16", qtype)
        assert bits_equal(res, ores), f"host {qtype}: residual_out differs from the oracle"
        _q_gate(q.view(torch.uint8) if qtype == "fp8" else q, sc, oq, os_, f"host {qtype} fused")
        oq, os_ = oracle.rmsnorm_quant(d["x"], d["w"], d["eps"], "f16", "f16", qtype)
        _q_gate(q2.view(torch.uint8) if qtype == "fp8" else q2, sc2, oq, os_, f"host {qtype}")
        rq, rs, rr = far.fused_add_rmsnorm_quant(d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), d["eps"], qtype)
        assert torch.equal(q, rq.cpu()) and bits_equal(sc, rs.cpu()) and bits_equal(res, rr.cpu())
        rq2, rs2 = far.rmsnorm_quant(d["x"].cuda(), d["w"].cuda(), d["eps"], qtype)
        assert torch.equal(q2, rq2.cpu()) and bits_equal(sc2, rs2.cpu())
