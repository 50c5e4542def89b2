"""CUDA path against the CPU oracle, element by element, through the C ABI.

Sizes here are ones the oracle finishes in seconds but that still span many
rows per CTA, several CTAs per SM sweep and ragged tails; the full workload
sizes are in test_gpu_full.py.
"""
import itertools

import pytest
import torch

import far_gen
from gpu_helpers import (check_both, far_fused, far_norm, gate, oracle_fused, oracle_norm,
                         square_sensitive_rows)
from oracle_pins import bits_equal, golden

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

    far.set_launch_override()  # automatic plans
    return far


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_workloads(far, name):
    d = far_gen.make_inputs(name)
    check_both(far, d, name)


@pytest.mark.parametrize("name", ["c4", "c5"])
def test_workload_rows(far, name):
    """The large workloads' first rows (the full sizes run in test_gpu_full)."""
    d = far_gen.make_inputs(name, rows=700)
    check_both(far, d, name)


def _matrix():
    g = golden("contract.json")["test_matrix"]
    return list(itertools.product(g["dtypes"], g["tokens"], g["hidden"]))


@pytest.mark.parametrize("act,tokens,hidden", _matrix())
def test_case_study_matrix(far, act, tokens, hidden):
    d = far_gen.custom_inputs(act, act, tokens, hidden, seed=tokens + hidden)
    check_both(far, d, f"{act} {tokens}x{hidden}")


@pytest.mark.parametrize("act,wd", PAIRS)
@pytest.mark.parametrize("hidden", [1, 7, 8, 33, 1000, 2048, 4095, 4096, 4097, 5120, 8192, 12288])
def test_dtype_pairs_and_hidden_sizes(far, act, wd, hidden):
    tokens = 40 if hidden <= 8192 else 12
    d = far_gen.custom_inputs(act, wd, tokens, hidden, seed=hidden, scale_lo=1e-3, scale_hi=30.0)
    check_both(far, d, f"{act}/{wd} H={hidden}")


@pytest.mark.parametrize("act,wd", [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("hidden", [768, 1536, 2560, 3000, 3072, 6144, 7168, 10240, 12288])
@pytest.mark.parametrize("tokens", [600, 2500])
def test_default_plans_across_widths(far, act, wd, hidden, tokens):
    """The launch table's rules at 4 and 17 rows an SM (more groups, exact 5, 6 or 10
    chunks, 4 chunks on rows with idle lanes at 8, up to 19 warps for the variant):
    the default plans of both ops against the oracle."""
    d = far_gen.custom_inputs(act, wd, tokens, hidden, seed=hidden + tokens, scale_lo=1e-2, scale_hi=50.0)
    check_both(far, d, f"{act}/{wd} {tokens}x{hidden}")


@pytest.mark.parametrize("hidden", [16384, 24576, 32768, 65536, 100003])
def test_large_hidden(far, hidden):
    d = far_gen.custom_inputs("bf16", "bf16", 5, hidden, seed=3)
    check_both(far, d, f"H={hidden}")
    d = far_gen.custom_inputs("f16", "f32", 3, hidden, seed=4)
    check_both(far, d, f"f16/f32 H={hidden}")


@pytest.mark.parametrize("tokens", [1, 2, 151, 152, 153, 305, 1217])
def test_token_counts(far, tokens):
    d = far_gen.custom_inputs("f16", "f16", tokens, 5120, seed=tokens)
    check_both(far, d, f"T={tokens}")


def test_zero_tokens(far):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    out, res = far.fused_add_rmsnorm(x, x.clone(), w, 1e-6)
    assert out.shape == (0, 256)
    assert far.rmsnorm(x, w, 1e-6).shape == (0, 256)


@pytest.mark.parametrize("offset", [1, 3])
def test_misaligned_pointers(far, offset):
    """Buffers off a 16-byte boundary take the generic path: same results."""
    for act, wd in [("bf16", "bf16"), ("f16", "f32"), ("f32", "f32")]:
        d = far_gen.custom_inputs(act, wd, 50, 2048, seed=offset)
        check_both(far, d, f"misaligned {act}/{wd}", offset=offset)


def test_in_place(far):
    for act, wd in [("bf16", "bf16"), ("f16", "f16"), ("f32", "f32")]:
        d = far_gen.custom_inputs(act, wd, 300, 4096, seed=11)
        check_both(far, d, f"in-place {act}", inplace=True)


def test_every_plan_gives_the_same_bits(far):
    """Chunks per thread, rows in flight, ring depth and the generic kernel all change
    the reduction order; the double-word accumulator makes the results identical."""
    d = far_gen.custom_inputs("f16", "f16", 400, 8192, seed=5)
    ref_out, ref_res = oracle_fused(d)
    ref_norm = oracle_norm(d)
    plans = [(-1, 0, 0, 0), (1, 0, 0, 0), (0, 4, 1, 2), (0, 4, 2, 3), (0, 8, 1, 0), (0, 8, 4, 0), (0, 2, 0, 0)]
    results = []
    try:
        for kind, nch, groups, stages in plans:
            far.set_launch_override(kind, nch, groups, stages)
            out, res = far_fused(far, d)
            nout = far_norm(far, d)
            gate(out, ref_out, res, ref_res, f"plan {kind, nch, groups, stages}")
            gate(nout, ref_norm, where=f"plan {kind, nch, groups, stages} rmsnorm")
            results.append((out, nout))
    finally:
        far.set_launch_override()
    for out, nout in results[1:]:
        assert bits_equal(out, results[0][0]) and bits_equal(nout, results[0][1])


def test_exact_five_and_six_chunk_plans(far):
    """Rows that 5 or 6 chunks a thread cover exactly (hidden 2560 and 3072 in 16-bit, 1280
    and 1536 in binary32) get those plans by default; they must pass the gate and give the
    same bits as the 8-chunk plan with idle lanes and as the generic kernel."""
    cases = [("bf16", "bf16", 2560, 5), ("f16", "f16", 3072, 6), ("f32", "f32", 1280, 5),
             ("f32", "bf16", 1536, 6), ("bf16", "f32", 2560, 5)]
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for act, wd, hidden, nch in cases:
        for tokens in (1, 37, 1234):
            plan = far.plan_for_sms(tokens, hidden, dt[act], dt[wd], True, sms)
            if tokens >= sms:
                assert plan["nch"] == nch, (act, hidden, tokens, plan)
            d = far_gen.custom_inputs(act, wd, tokens, hidden, seed=tokens + hidden)
            ref_out, ref_res = oracle_fused(d)
            ref_norm = oracle_norm(d)
            results = []
            try:
                for ov in [(-1, 0, 0, 0), (0, 8, 2, 0), (1, 0, 0, 0), (0, nch, 3, 3)]:
                    far.set_launch_override(*ov)
                    out, res = far_fused(far, d)
                    nout = far_norm(far, d)
                    gate(out, ref_out, res, ref_res, f"{act}/{wd} {hidden}x{tokens} plan {ov}")
                    gate(nout, ref_norm, where=f"{act}/{wd} {hidden}x{tokens} plan {ov} rmsnorm")
                    results.append((out, nout))
            finally:
                far.set_launch_override()
            for out, nout in results[1:]:
                assert bits_equal(out, results[0][0]) and bits_equal(nout, results[0][1])


def test_ten_chunk_variant(far):
    """The no-residual variant on 16-bit rows that 2 warps cover exactly at 10 chunks a thread
    (hidden 5120): every plan, including 10 chunks with 1 to 9 groups, gives the same bits
    and passes the gate; the fused op asked for 10 chunks runs the generic kernel."""
    for act, wd in [("bf16", "bf16"), ("f16", "f16"), ("bf16", "f32"), ("f16", "f32")]:
        d = far_gen.custom_inputs(act, wd, 999, 5120, seed=77)
        ref_norm = oracle_norm(d)
        ref_out, ref_res = oracle_fused(d)
        results = []
        try:
            for ov in [(-1, 0, 0, 0), (0, 10, 1, 2), (0, 10, 6, 12), (0, 10, 9, 18), (0, 8, 6, 12), (1, 0, 0, 0)]:
                far.set_launch_override(*ov)
                nout = far_norm(far, d)
                gate(nout, ref_norm, where=f"{act}/{wd} 5120 plan {ov} rmsnorm")
                out, res = far_fused(far, d)
                gate(out, ref_out, res, ref_res, f"{act}/{wd} 5120 plan {ov}")
                results.append(nout)
        finally:
            far.set_launch_override()
        assert all(bits_equal(r, results[0]) for r in results[1:])


def test_special_values(far):
    """inf / NaN / huge / subnormal inputs: NaN spreads through its row only."""
    for act in ("f16", "bf16", "f32"):
        d = far_gen.custom_inputs(act, act, 16, 1024, seed=9)
        x, r = d["x"].clone(), d["r"].clone()
        x[0, 5] = float("nan")
        x[1, 7] = float("inf")
        r[2, 9] = float("-inf")
        x[3] = 0.0
        r[3] = 0.0
        big = {"f16": 60000.0, "bf16": 3.0e38, "f32": 3.0e38}[act]
        x[4, :4] = big
        r[4, :4] = big
        tiny = {"f16": 6e-8, "bf16": 1e-39, "f32": 1e-44}[act]
        x[5] = tiny
        r[5] = -tiny / 2
        x[6, 100] = -0.0
        r[6, 100] = -0.0
        d = dict(d, x=x, r=r)
        check_both(far, d, f"special {act}")


def test_eps_variants(far):
    for eps in (0.0, 1e-12, 1e-5, 0.5):
        d = dict(far_gen.custom_inputs("bf16", "f32", 64, 3072, seed=2, scale_lo=1e-4, scale_hi=1e-1), eps=eps)
        check_both(far, d, f"eps={eps}")


def test_host_buffer_entry_points(far):
    """The end-to-end entry points (host buffers, chunked through a small workspace)
    give the same bits as the device entry points."""
    for act, wd in [("f16", "f16"), ("bf16", "f32")]:
        d = far_gen.custom_inputs(act, wd, 1000, 4096, seed=21)
        od = far.output_dtype(d["x"].dtype, d["w"].dtype)
        ws = torch.empty(far.host_workspace_bytes(96, 4096, d["x"].dtype, d["w"].dtype), dtype=torch.uint8,
                         device="cuda")
        ref_out, ref_res = oracle_fused(d)
        for pinned in (True, False):
            x, r, w = (t.pin_memory() if pinned else t.clone() for t in (d["x"], d["r"], d["w"]))
            out = torch.empty(d["x"].shape, dtype=od, pin_memory=pinned)
            res = torch.empty(d["x"].shape, dtype=d["x"].dtype, pin_memory=pinned)
            far.fused_add_rmsnorm_host(x, r, w, d["eps"], out, res, ws)
            torch.cuda.current_stream().synchronize()
            gate(out, ref_out, res, ref_res, f"host {act}/{wd} pinned={pinned}")
            nout = torch.empty(d["x"].shape, dtype=od, pin_memory=pinned)
            far.rmsnorm_host(x, w, d["eps"], nout, ws)
            torch.cuda.current_stream().synchronize()
            gate(nout, oracle_norm(d), where=f"host rmsnorm {act}/{wd}")
    with pytest.raises(far.FarError):
        tiny = torch.empty(64, dtype=torch.uint8, device="cuda")
        far.fused_add_rmsnorm_host(x, r, w, d["eps"], out, res, tiny)


def test_errors_through_the_abi_on_device(far):
    x = torch.zeros((8, 256), dtype=torch.float16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(far.FarError) as e:
        far.fused_add_rmsnorm(x, x.clone(), w, 1e-6)
    assert e.value.status == 1
    w16 = torch.ones(256, dtype=torch.float16, device="cuda")
    buf = torch.zeros(8 * 256 + 8, dtype=torch.float16, device="cuda")
    with pytest.raises(far.FarError) as e:  # out overlapping x at an offset
        far.fused_add_rmsnorm(buf[:2048].view(8, 256), x, w16, 1e-6, out=buf[8:].view(8, 256))
    assert e.value.status == 5


@pytest.mark.parametrize("act", ["f16", "bf16"])
def test_subnormal_products(far, act):
    """Weights so small that n * w lands among the 16-bit subnormals (and rounds to
    zero at the bottom): the packed 16-bit multiply must keep subnormals and round
    them to nearest even exactly like the oracle."""
    d = far_gen.custom_inputs(act, act, 64, 4096, seed=17)
    tiny = {"f16": 2.0 ** -20, "bf16": 2.0 ** -130}[act]
    g = torch.Generator().manual_seed(5)
    w = (torch.rand(4096, generator=g, dtype=torch.float64) * 8 - 4) * tiny
    w[::7] = torch.linspace(-1, 1, len(w[::7]), dtype=torch.float64) * tiny * 2 ** -8
    d = dict(d, w=w.to(d["w"].dtype))
    check_both(far, d, f"subnormal products {act}")


def _canary_like(shape, dtype):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    t.view(torch.int16 if t.element_size() == 2 else torch.int32).fill_(0x3A5A)
    return t


@pytest.mark.parametrize("act,wd,extra", [("bf16", "bf16", 64), ("f16", "f32", 8), ("f32", "f32", 3),
                                          ("bf16", "bf16", 1)])
def test_strided_rows(far, act, wd, extra):
    """x, residual, out and residual_out as column slices of wider matrices (row stride
    hidden + extra elements); the columns outside the slices must stay untouched.  A
    stride that breaks 16-byte row alignment (extra = 1 or 3) takes the generic kernel."""
    T, H = 300, 2048
    d = far_gen.custom_inputs(act, wd, T, H, seed=extra)
    S = H + extra
    xbig = _canary_like((T, S), d["x"].dtype)
    rbig = _canary_like((T, S), d["x"].dtype)
    xbig[:, :H] = d["x"].cuda()
    rbig[:, :H] = d["r"].cuda()
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    obig = _canary_like((T, S), od)
    robig = _canary_like((T, S), d["x"].dtype)
    keep = [t[:, H:].clone() for t in (obig, robig)]
    out, res = far.fused_add_rmsnorm(xbig[:, :H], rbig[:, :H], d["w"].cuda(), d["eps"],
                                     out=obig[:, :H], residual_out=robig[:, :H])
    assert far.device_status() == 0
    ref_out, ref_res = oracle_fused(d)
    gate(out.cpu(), ref_out, res.cpu(), ref_res, f"strided {act}/{wd} +{extra}")
    assert torch.equal(obig[:, H:], keep[0]) and torch.equal(robig[:, H:], keep[1]), "wrote outside the slices"
    # the no-residual variant on the same slices
    o2big = _canary_like((T, S), od)
    nout = far.rmsnorm(xbig[:, :H], d["w"].cuda(), d["eps"], out=o2big[:, :H])
    assert far.device_status() == 0
    gate(nout.cpu(), oracle_norm(d), where=f"strided rmsnorm {act}/{wd} +{extra}")
    assert (o2big[:, H:].view(torch.int16 if o2big.element_size() == 2 else torch.int32) == 0x3A5A).all()


def test_interleaved_slices_of_one_buffer(far):
    """x, out, residual_out and residual as four interleaved column slices of one buffer."""
    T, H = 200, 1024
    d = far_gen.custom_inputs("f16", "f16", T, H, seed=31)
    buf = torch.empty((T, 4 * H), dtype=torch.float16, device="cuda")
    buf[:, 0:H] = d["x"].cuda()
    buf[:, 3 * H:4 * H] = d["r"].cuda()
    out, res = far.fused_add_rmsnorm(buf[:, 0:H], buf[:, 3 * H:], d["w"].cuda(), d["eps"],
                                     out=buf[:, H:2 * H], residual_out=buf[:, 2 * H:3 * H])
    assert far.device_status() == 0
    ref_out, ref_res = oracle_fused(d)
    gate(out.cpu(), ref_out, res.cpu(), ref_res, "interleaved slices")
    assert torch.equal(buf[:, 0:H].cpu(), d["x"]) and torch.equal(buf[:, 3 * H:].cpu(), d["r"])


def test_strided_in_place(far):
    T, H = 150, 4096
    d = far_gen.custom_inputs("bf16", "bf16", T, H, seed=32)
    xbig = torch.zeros((T, H + 512), dtype=torch.bfloat16, device="cuda")
    rbig = torch.zeros((T, H + 512), dtype=torch.bfloat16, device="cuda")
    xbig[:, :H] = d["x"].cuda()
    rbig[:, :H] = d["r"].cuda()
    out, res = far.fused_add_rmsnorm(xbig[:, :H], rbig[:, :H], d["w"].cuda(), d["eps"],
                                     out=xbig[:, :H], residual_out=rbig[:, :H])
    assert far.device_status() == 0
    ref_out, ref_res = oracle_fused(d)
    gate(xbig[:, :H].cpu(), ref_out, rbig[:, :H].cpu(), ref_res, "strided in place")


def _tiny_square_rows(T, H, seed):
    """bf16 rows whose squares fall in binary32's subnormal range and are rounded there:
    x = +-m/128 * 2^-68 with m odd in 129..255 (m and the signs drawn from the seeded
    generator), so x^2 = m^2 * 2^-150 lies halfway between two subnormals and, m^2/2 being
    4j + 1/2, rounds down to the even one: every square loses 2^-150, and a row of
    thousands loses enough to move var = S / hidden by about half its last place.  Every
    third row carries one element 2^8 larger (a normal square that dominates its thread's
    chain)."""
    import numpy as np

    d = far_gen.custom_inputs("bf16", "f32", T, H, seed=seed, eps=0.0)
    u = d["x"].double().numpy()
    m = 129.0 + 2.0 * (np.floor(np.abs(u) * 1000.0) % 64)
    x = np.sign(u) * m / 128.0 * 2.0 ** -68
    x[::3, 7] *= 2.0 ** 8
    return d, torch.from_numpy(x.astype(np.float32))


@pytest.mark.parametrize("wd", ["f32", "bf16"])
@pytest.mark.parametrize("hidden", [5120, 4096, 1000])
def test_subnormal_squares_of_16_bit_rows(far, hidden, wd):
    """The no-residual kernel keeps 16-bit x packed and sums its squares in chains that
    start at the largest square's power of two; the fused kernel (residual 0) sums
    fl32(s * s) in ordered chains.  On rows whose rounded squares (binary32 subnormals)
    give another rstd than their exact squares would, both must still match the oracle
    (with a binary32 out every element shows a change of rstd), on several plans."""
    import math

    import numpy as np

    import oracle

    d, x = _tiny_square_rows(1200, hidden, seed=hidden + 3)
    xb = x.to(torch.bfloat16)
    assert torch.equal(xb.float(), x)  # every value is a bf16
    H = np.float32(hidden)

    def rstd(S):
        return np.float32(1.0) / np.sqrt(np.float32(S / H))

    xf = x.numpy()
    keep = []
    for i, row in enumerate(xf):
        S_rounded = np.float32(oracle.exact_sum((row * row).astype(np.float32)))
        S_exact = np.float32(math.fsum(float(v) * float(v) for v in row.astype(np.float64)))
        keep.append(rstd(S_rounded) != rstd(S_exact))
    rows = np.nonzero(keep)[0]
    assert len(rows) >= 100 and (rows % 3 == 0).sum() >= 20, len(rows)
    w = d["w"] if wd == "f32" else d["w"].to(torch.bfloat16)
    sel = dict(d, x=xb[rows].contiguous(), r=torch.zeros_like(xb[rows]), w=w, wd=wd, tokens=len(rows))
    try:
        for plan in [(-1, 0, 0, 0), (0, 2, 0, 0), (0, 8, 0, 0), (1, 0, 0, 0)]:
            far.set_launch_override(*plan)
            gate(far_norm(far, sel), oracle_norm(sel), where=f"subnormal squares rmsnorm {plan}")
            out, res = far_fused(far, sel)
            ref_out, ref_res = oracle_fused(sel)
            gate(out, ref_out, res, ref_res, where=f"subnormal squares fused {plan}")
    finally:
        far.set_launch_override()


def test_rounded_squares_are_summed(far):
    """The sum of squares adds fl32(s * s), each square rounded, not the exact squares
    (as a fused multiply-add would): rows where the two sums round to different binary32
    values and so change rstd must still pass the gate, for both kernels."""
    import numpy as np

    import oracle

    d = far_gen.custom_inputs("f32", "f32", 6000, 64, seed=31, scale_lo=0.5, scale_hi=2.0, eps=0.0)
    x = d["x"].numpy()
    S = np.array([oracle.exact_sum((row * row).astype(np.float32)) for row in x], np.float32)
    rows = np.nonzero(square_sensitive_rows(x, S, 0.0))[0]
    assert len(rows) >= 20, len(rows)
    sel = dict(d, x=d["x"][rows].contiguous(), r=torch.zeros_like(d["x"][rows]), tokens=len(rows))
    try:
        for plan in [(-1, 0, 0, 0), (1, 0, 0, 0)]:
            far.set_launch_override(*plan)
            gate(far_norm(far, sel), oracle_norm(sel), where=f"rounded squares rmsnorm {plan}")
            out, res = far_fused(far, sel)  # residual 0: s = x + 0 = x
            ref_out, ref_res = oracle_fused(sel)
            gate(out, ref_out, res, ref_res, where=f"rounded squares fused {plan}")
    finally:
        far.set_launch_override()
