"""The allocation-free entry point, fused_add_rmsnorm_host_noalloc.

It serves callers that cannot allocate device memory (a host program that owns
all device memory through its own pool, or a no-allocation-after-start-up
rule): host buffers in and out, staged through a fixed array inside the
library.  Here it is called through the C ABI on two calls in a row with
different shapes and dtypes, and each result is checked against the CPU oracle
and against the existing host-buffer entry point (which stages through a
caller workspace), under the same gate as every other parity test:
residual_out bit for bit, out within 1 ULP with fewer than 1% of elements
differing.  A further test checks the promise itself: across a call, the
device's free memory and torch's allocator counters do not move.  The file is
named to be collected last.
"""
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import gate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    return far


def _pinned(t):
    return t.contiguous().pin_memory()


def _with_workspace(far, d):
    """The existing host-buffer entry point, staging through a torch-allocated workspace."""
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    x, r, w = _pinned(d["x"]), _pinned(d["r"]), _pinned(d["w"])
    out = torch.empty(d["x"].shape, dtype=od, pin_memory=True)
    res = torch.empty(d["x"].shape, dtype=d["x"].dtype, pin_memory=True)
    ws = torch.empty(far.host_workspace_bytes(256, d["hidden"], d["x"].dtype, d["w"].dtype), dtype=torch.uint8,
                     device="cuda")
    far.fused_add_rmsnorm_host(x, r, w, d["eps"], out, res, ws)
    torch.cuda.current_stream().synchronize()
    return out, res


def _no_alloc(far, d):
    """The allocation-free entry point, called through the C ABI."""
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    x, r, w = _pinned(d["x"]), _pinned(d["r"]), _pinned(d["w"])
    out = torch.empty(d["x"].shape, dtype=od, pin_memory=True)
    res = torch.empty(d["x"].shape, dtype=d["x"].dtype, pin_memory=True)
    tokens, hidden = d["x"].shape
    st = far.lib.fused_add_rmsnorm_host_noalloc(x.data_ptr(), r.data_ptr(), w.data_ptr(), d["eps"], out.data_ptr(),
                                                res.data_ptr(), tokens, hidden,
                                                far.dtypes(d["x"].dtype, d["w"].dtype),
                                                torch.cuda.current_stream().cuda_stream)
    assert st == 0, far.lib.far_status_string(st)
    torch.cuda.current_stream().synchronize()
    assert far.device_status() == 0
    return out, res


def _oracle(d):
    return oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"])


def test_two_calls_in_a_row_match_the_oracle_and_the_workspace_entry_point(far):
    # first call: more rows than one pass through the 16 MiB array holds
    d1 = far_gen.make_inputs("c5", rows=1500)
    out1, res1 = _no_alloc(far, d1)
    ref_out1, ref_res1 = _oracle(d1)
    gate(out1, ref_out1, res1, ref_res1, "no-alloc call 1 (fp16 1500x8192) against the oracle")
    ws_out1, ws_res1 = _with_workspace(far, d1)
    gate(out1, ws_out1, res1, ws_res1, "no-alloc call 1 against the workspace entry point")
    # second call right after: another shape and dtype pair through the same array
    d2 = far_gen.make_inputs("c3", rows=700)
    out2, res2 = _no_alloc(far, d2)
    ref_out2, ref_res2 = _oracle(d2)
    gate(out2, ref_out2, res2, ref_res2, "no-alloc call 2 (bf16/fp32 700x4096) against the oracle")
    ws_out2, ws_res2 = _with_workspace(far, d2)
    gate(out2, ws_out2, res2, ws_res2, "no-alloc call 2 against the workspace entry point")


def test_a_call_allocates_no_device_memory(far):
    """After a first call (which loads the library's device code and looks up the array's
    address), further calls leave the device's free memory and torch's allocator counters
    exactly as they were."""
    d = far_gen.make_inputs("c2", rows=300)
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    x, r, w = _pinned(d["x"]), _pinned(d["r"]), _pinned(d["w"])
    out = torch.empty(d["x"].shape, dtype=od, pin_memory=True)
    res = torch.empty(d["x"].shape, dtype=d["x"].dtype, pin_memory=True)
    stream = torch.cuda.current_stream()
    args = (x.data_ptr(), r.data_ptr(), w.data_ptr(), d["eps"], out.data_ptr(), res.data_ptr(), 300, d["hidden"],
            far.dtypes(d["x"].dtype, d["w"].dtype), stream.cuda_stream)
    assert far.lib.fused_add_rmsnorm_host_noalloc(*args) == 0
    stream.synchronize()

    def counters():
        s = torch.cuda.memory_stats()
        return (torch.cuda.mem_get_info()[0], s.get("allocation.all.allocated", 0),
                s.get("segment.all.allocated", 0), torch.cuda.memory_reserved())

    before = counters()
    for _ in range(3):
        assert far.lib.fused_add_rmsnorm_host_noalloc(*args) == 0
    stream.synchronize()
    after = counters()
    assert after == before, f"device memory moved across the calls: {before} -> {after}"
    assert far.device_status() == 0
    ref_out, ref_res = _oracle(d)
    gate(out, ref_out, res, ref_res, "no-alloc, repeated calls")


def test_rejects_a_row_too_large_for_the_array(far):
    hidden = 1 << 21  # 2M fp16 elements: one row of the four tensors plus the weight exceeds 16 MiB
    x = torch.zeros((1, hidden), dtype=torch.float16)
    w = torch.ones(hidden, dtype=torch.float16)
    out = torch.empty_like(x)
    res = torch.empty_like(x)
    st = far.lib.fused_add_rmsnorm_host_noalloc(x.data_ptr(), x.data_ptr() + 0, w.data_ptr(), 1e-6, out.data_ptr(),
                                                res.data_ptr(), 1, hidden, far.dtypes(x.dtype, w.dtype),
                                                torch.cuda.current_stream().cuda_stream)
    assert st == 10, far.lib.far_status_string(st)  # FAR_ERR_SCRATCH
    assert b"scratch" in far.lib.far_status_string(st)
