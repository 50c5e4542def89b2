"""How the staged kernel's CTAs share rows: fixed-stride rows against rows claimed from a
per-launch counter. Both give the same bits for every op (each row is computed the same
way by whichever CTA takes it). Claimed rows must also survive:
- launches back to back (each launch's last CTA must leave its counter zero, or the next
  launch given it would skip rows);
- launches side by side on two streams (they must never share a counter);
- more launches in flight on one stream than counters (they share the stream's counter),
  and more streams than counters (the rest take the fixed stride);
- graph capture (the fixed stride: a captured event cannot be polled).
Outputs start as NaN (0xFF bytes for quantised codes), so a row nobody wrote shows."""
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import gate
from oracle_pins import bits_equal

pytestmark = pytest.mark.gpu

SHAPES = [("bf16", "bf16", 16384, 5120), ("f16", "f16", 3001, 8192), ("f32", "f32", 2000, 4096),
          ("bf16", "bf16", 7777, 1024), ("f16", "f32", 5000, 2048)]


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    far.set_launch_override()
    far.set_row_schedule(1)
    yield far
    far.set_row_schedule(1)


def _nan(shape, dtype):
    if dtype in (torch.int8, torch.uint8):
        return torch.full(shape, -1 if dtype == torch.int8 else 255, dtype=dtype, device="cuda")
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def _run(far, op, t, stream=None):
    """One call of `op` on device tensors t, into NaN-filled outputs; returns the outputs."""
    x, r, w, b, eps = t["x"], t["r"], t["w"], t["b"], t["eps"]
    od = far.output_dtype(x.dtype, w.dtype)
    shape = tuple(x.shape)
    if op == "rms_fused":
        out, res = _nan(shape, od), _nan(shape, x.dtype)
        far.fused_add_rmsnorm(x, r, w, eps, out=out, residual_out=res, stream=stream)
        return [out, res]
    if op == "rms":
        out = _nan(shape, od)
        far.rmsnorm(x, w, eps, out=out, stream=stream)
        return [out]
    if op == "ln_fused":
        out, res = _nan(shape, od), _nan(shape, x.dtype)
        far.fused_add_layernorm(x, r, w, b, eps, out=out, residual_out=res)
        return [out, res]
    if op == "ln":
        return [far.layernorm(x, w, b, eps, out=_nan(shape, od))]
    if op == "q_fused":
        q, scale, res = _nan(shape, torch.int8), _nan((shape[0],), torch.float32), _nan(shape, x.dtype)
        far.fused_add_rmsnorm_quant(x, r, w, eps, "int8", q=q, scale=scale, residual_out=res)
        return [q, scale, res]
    q, scale = _nan(shape, torch.uint8), _nan((shape[0],), torch.float32)
    far.rmsnorm_quant(x, w, eps, "fp8", q=q, scale=scale)
    return [q, scale]


def _same(a, b):
    return all(bits_equal(u.cpu(), v.cpu()) if u.is_floating_point() else torch.equal(u.cpu(), v.cpu())
               for u, v in zip(a, b))


def _inputs(act, wd, tokens, hidden, seed):
    d = far_gen.custom_inputs(act, wd, tokens, hidden, seed=seed)
    d["b"] = far_gen.ln_beta(d, seed)
    t = {k: d[k].cuda() for k in ("x", "r", "w", "b")}
    t["eps"] = d["eps"]
    return d, t


@pytest.mark.parametrize("op", ["rms_fused", "rms", "ln_fused", "ln", "q_fused", "q"])
@pytest.mark.parametrize("act,wd,tokens,hidden", SHAPES)
def test_claimed_rows_give_the_fixed_stride_bits(far, op, act, wd, tokens, hidden):
    d, t = _inputs(act, wd, tokens, hidden, seed=tokens + hidden)
    try:
        far.set_row_schedule(1)
        ref = _run(far, op, t)
        assert not far.last_launch_claimed_rows()
        assert far.device_status() == 0
        far.set_row_schedule(2)
        for i in range(3):  # back to back: each launch must find its counter zero
            got = _run(far, op, t)
            assert far.last_launch_claimed_rows(), f"{op}: launch {i} did not claim rows"
            assert far.device_status() == 0
            assert _same(got, ref), f"{op} {act}/{wd} {tokens}x{hidden}: launch {i} differs"
    finally:
        far.set_row_schedule(1)
    assert not any(torch.isnan(o).any() for o in ref if o.is_floating_point()), "a row was left unwritten"


@pytest.mark.parametrize("op,act,tokens,hidden", [("rms", "bf16", 16384, 5120), ("rms", "bf16", 32768, 4608),
                                                  ("rms", "f16", 24576, 5120), ("q", "bf16", 16384, 5120),
                                                  ("q", "f16", 24576, 5120)])
def test_claims_over_the_last_quarter_give_the_fixed_stride_bits(far, op, act, tokens, hidden):
    """The automatic rule's three-row claims (packed no-residual kernels): each CTA takes the
    first three quarters of its rows at the fixed stride, then claims; back to back, each
    launch finds its counter zero, every row is written, and the bits are the fixed stride's."""
    d, t = _inputs(act, act, tokens, hidden, seed=tokens + hidden + 1)
    try:
        far.set_row_schedule(1)
        ref = _run(far, op, t)
        assert not far.last_launch_claimed_rows()
        far.set_row_schedule(0)
        assert far.row_schedule_for_sms(tokens, hidden, t["x"].dtype, t["w"].dtype, False,
                                        "rmsnorm" if op == "rms" else "quant",
                                        torch.cuda.get_device_properties(0).multi_processor_count) == 3
        for i in range(3):
            got = _run(far, op, t)
            assert far.last_launch_claimed_rows(), f"{op}: launch {i} did not claim rows"
            assert far.device_status() == 0
            assert _same(got, ref), f"{op} {act} {tokens}x{hidden}: launch {i} differs"
    finally:
        far.set_row_schedule(1)
    assert not any(torch.isnan(o).any() for o in ref if o.is_floating_point()), "a row was left unwritten"


def test_claimed_rows_against_the_oracle(far):
    """The fused op and the variant at many rows a CTA, claimed rows, against the oracle."""
    d, t = _inputs("bf16", "bf16", 6000, 2048, seed=77)
    try:
        far.set_row_schedule(2)
        out, res = _run(far, "rms_fused", t)
        assert far.last_launch_claimed_rows()
        ro, rr = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"])
        gate(out.cpu(), ro, res.cpu(), rr, where="claimed rows fused")
        (out,) = _run(far, "rms", t)
        assert far.last_launch_claimed_rows()
        gate(out.cpu(), oracle.rmsnorm(d["x"], d["w"], d["eps"], d["act"], d["wd"]), where="claimed rows")
    finally:
        far.set_row_schedule(1)


def test_default_schedule(far):
    """The default keeps the fixed stride (no state between calls). The automatic rule
    (mode 0) claims rows for the fused op at 16384 x 5120 bf16 (40 KB moved a row, two rows
    a claim, over 2 ring-fulls a CTA) and for its packed no-residual variant (20 KB a row,
    three a claim, 640 chunks), keeps the fixed stride for LayerNorm's variant on the same
    rows, for the variant at 16384 x 4096 (512 chunks) and for the fused op at 512 rows."""
    assert far.get_row_schedule() == 1
    _, t = _inputs("bf16", "bf16", 16384, 5120, seed=3)
    for op in ("rms_fused", "rms", "ln_fused", "q_fused"):
        _run(far, op, t)
        assert not far.last_launch_claimed_rows(), op
    try:
        far.set_row_schedule(0)
        _run(far, "rms_fused", t)
        assert far.last_launch_claimed_rows()
        _run(far, "rms", t)
        assert far.last_launch_claimed_rows()
        _run(far, "ln", t)
        assert not far.last_launch_claimed_rows()
        _, t4 = _inputs("bf16", "bf16", 16384, 4096, seed=5)
        _run(far, "rms", t4)
        assert not far.last_launch_claimed_rows()
        _, t = _inputs("bf16", "bf16", 512, 5120, seed=4)
        _run(far, "rms_fused", t)
        assert not far.last_launch_claimed_rows()
    finally:
        far.set_row_schedule(1)
    assert far.device_status() == 0


def test_two_streams_side_by_side(far):
    """Two inputs launched alternately on two streams, many times, with claimed rows: every
    result equals its fixed-stride reference (no two launches in flight share a counter)."""
    ins = [_inputs("bf16", "bf16", 8192, 4096, seed=s)[1] for s in (11, 12)]
    try:
        far.set_row_schedule(1)
        refs = [_run(far, "rms_fused", t) for t in ins]
        far.set_row_schedule(2)
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        torch.cuda.synchronize()
        outs = []
        for _ in range(12):
            for t, s in zip(ins, streams):
                with torch.cuda.stream(s):
                    outs.append((len(outs) % 2, _run(far, "rms_fused", t, stream=s)))
        torch.cuda.synchronize()
        assert far.device_status() == 0
        for which, got in outs:
            assert _same(got, refs[which]), "a launch on one stream lost rows to the other"
    finally:
        far.set_row_schedule(1)


def test_more_launches_in_flight_than_counters(far):
    """100 launches queued on one stream without a wait (more than the 64 counters): they
    share their stream's counter, which the stream's order keeps apart, so every one claims
    rows; all results equal the reference."""
    _, t = _inputs("bf16", "bf16", 4096, 4096, seed=21)
    try:
        far.set_row_schedule(1)
        ref = _run(far, "rms", t)
        far.set_row_schedule(2)
        outs, claimed = [], 0
        for _ in range(100):
            outs.append(_run(far, "rms", t))
            claimed += far.last_launch_claimed_rows()
        torch.cuda.synchronize()
        assert far.device_status() == 0
        assert claimed == 100
        for got in outs:
            assert _same(got, ref)
    finally:
        far.set_row_schedule(1)


def test_more_streams_than_counters(far):
    """One launch on each of 70 streams, queued without a wait: a stream finds no counter of
    its own, so it takes one that no launch is pending on and whose last launch has
    finished, or keeps the fixed stride; every result equals the reference."""
    _, t = _inputs("bf16", "bf16", 2048, 4096, seed=41)
    try:
        far.set_row_schedule(1)
        ref = _run(far, "rms_fused", t)
        far.set_row_schedule(2)
        streams = [torch.cuda.Stream() for _ in range(70)]
        torch.cuda.synchronize()
        outs = []
        for s in streams:
            with torch.cuda.stream(s):
                outs.append(_run(far, "rms_fused", t, stream=s))
        torch.cuda.synchronize()
        assert far.device_status() == 0
        for got in outs:
            assert _same(got, ref), "a launch lost rows to another stream's launch"
    finally:
        far.set_row_schedule(1)


def test_graph_capture_keeps_the_fixed_stride(far):
    _, t = _inputs("bf16", "bf16", 16384, 2048, seed=31)
    try:
        far.set_row_schedule(1)
        ref = _run(far, "rms_fused", t)
        far.set_row_schedule(2)
        out = torch.empty_like(ref[0])
        res = torch.empty_like(ref[1])
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            far.fused_add_rmsnorm(t["x"], t["r"], t["w"], t["eps"], out=out, residual_out=res, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            far.fused_add_rmsnorm(t["x"], t["r"], t["w"], t["eps"], out=out, residual_out=res,
                                  stream=torch.cuda.current_stream())
            claimed_in_capture = far.last_launch_claimed_rows()
        assert not claimed_in_capture
        for _ in range(3):
            out.fill_(float("nan"))
            res.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert _same([out, res], ref)
        assert far.device_status() == 0
    finally:
        far.set_row_schedule(1)
