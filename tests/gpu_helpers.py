"""Helpers for the GPU parity tests: guarded device buffers, calls through the
C ABI, and the parity gate.

The gate (after the case study "Aligning fused RMSNorm rounding across vLLM
backends", section "Testing the contract"):
residual_out bit for bit equal to the oracle's; out within 1 ULP of its dtype
everywhere, with fewer than 1% of elements differing at all.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle_pins import ulp_distance

GUARD = 64  # elements of canary before and after every output (keeps 16-byte alignment)
CANARY = {torch.float16: 0x7E5A, torch.bfloat16: 0x7FA5, torch.float32: 0x7FC0A5A5}


class Guarded:
    """A device tensor with canary bands on both sides, to catch out-of-bounds stores."""

    def __init__(self, shape, dtype, offset_elems=0, fill=None):
        n = int(np.prod(shape))
        self.dtype = dtype
        self.n = n
        self.lead = GUARD + offset_elems
        self.buf = torch.empty(self.lead + n + GUARD, dtype=dtype, device="cuda")
        ibits = {2: torch.int16, 4: torch.int32}[self.buf.element_size()]
        self.canary = CANARY[dtype]
        v = self.canary if self.canary < (1 << (8 * self.buf.element_size() - 1)) else self.canary - (1 << 32)
        self.buf.view(ibits).fill_(v)
        self.t = self.buf[self.lead:self.lead + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self) -> bool:
        ibits = {2: torch.int16, 4: torch.int32}[self.buf.element_size()]
        b = self.buf.view(ibits).cpu().numpy().astype(np.int64) & ((1 << (8 * self.buf.element_size())) - 1)
        return bool((b[:self.lead] == self.canary).all() and (b[self.lead + self.n:] == self.canary).all())


def to_device(t: torch.Tensor, offset_elems: int = 0) -> Guarded:
    return Guarded(tuple(t.shape), t.dtype, offset_elems, fill=t)


def gate(out_gpu: torch.Tensor, out_ref: torch.Tensor, res_gpu=None, res_ref=None, where=""):
    """Assert the parity gate; return (max ULP, differing fraction)."""
    if res_gpu is not None:
        rd = ulp_distance(res_gpu, res_ref)
        assert int(rd.max(initial=0)) == 0, f"{where}: residual_out differs in {int((rd > 0).sum())} elements"
    d = ulp_distance(out_gpu, out_ref)
    mx = int(d.max(initial=0))
    frac = float((d > 0).mean()) if d.size else 0.0
    assert mx <= 1, f"{where}: out differs by up to {mx} ULP ({int((d > 1).sum())} elements > 1 ULP)"
    assert frac < 0.01, f"{where}: {frac:.4%} of out elements differ"
    return mx, frac


def far_fused(far, d, offset=0, inplace=False):
    """Run the fused op on the GPU through the C ABI with guarded buffers; CPU results."""
    x, r, w = to_device(d["x"], offset), to_device(d["r"], offset), to_device(d["w"], 0)
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    if inplace:
        out_t = x.t if od == x.t.dtype else None
        out = x if out_t is not None else Guarded(tuple(d["x"].shape), od, offset)
        res = r
    else:
        out = Guarded(tuple(d["x"].shape), od, offset)
        res = Guarded(tuple(d["x"].shape), d["x"].dtype, offset)
    tokens, hidden = d["x"].shape
    st = far.lib.fused_add_rmsnorm(x.t.data_ptr(), r.t.data_ptr(), w.t.data_ptr(), d["eps"], out.t.data_ptr(),
                                   res.t.data_ptr(), tokens, hidden, far.dtypes(d["x"].dtype, d["w"].dtype),
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0, far.lib.far_status_string(st)
    assert far.device_status() == 0
    for g in (out, res):
        assert g.guards_intact(), "a store landed outside its output"
    return out.t.cpu(), res.t.cpu()


def far_norm(far, d, offset=0, inplace=False):
    x, w = to_device(d["x"], offset), to_device(d["w"], 0)
    od = far.output_dtype(d["x"].dtype, d["w"].dtype)
    out = x if (inplace and od == d["x"].dtype) else Guarded(tuple(d["x"].shape), od, offset)
    tokens, hidden = d["x"].shape
    st = far.lib.rmsnorm(x.t.data_ptr(), w.t.data_ptr(), d["eps"], out.t.data_ptr(), tokens, hidden,
                         far.dtypes(d["x"].dtype, d["w"].dtype), torch.cuda.current_stream().cuda_stream)
    assert st == 0, far.lib.far_status_string(st)
    assert far.device_status() == 0
    assert out.guards_intact(), "a store landed outside its output"
    return out.t.cpu()


def oracle_fused(d):
    return oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], d["act"], d["wd"])


def oracle_norm(d):
    return oracle.rmsnorm(d["x"], d["w"], d["eps"], d["act"], d["wd"])


def check_both(far, d, where, offset=0, inplace=False):
    """The fused op and the no-residual variant against the oracle."""
    out, res = far_fused(far, d, offset, inplace)
    ref_out, ref_res = oracle_fused(d)
    a = gate(out, ref_out, res, ref_res, where + " fused")
    nout = far_norm(far, d, offset, inplace)
    b = gate(nout, oracle_norm(d), where=where + " rmsnorm")
    return a, b


def square_sensitive_rows(dev: np.ndarray, S: np.ndarray, eps: float) -> np.ndarray:
    """Rows whose rstd depends on rounding each square before the sum.

    dev: [rows, hidden] binary32 values whose squares are summed (s for RMSNorm, the
    deviations d for LayerNorm); S: the oracle's binary32 sums RN32(sum fl32(v^2)).
    A row is kept when RN32 of the exact sum of the EXACT squares is another binary32
    value and that changes fl32(1 / fl32(sqrt(fl32(fl32(S / H) + eps)))).  math.fsum
    rounds correctly, so the sign of (exact sum - rounding boundary) it returns is exact.
    """
    import math

    rows, H = dev.shape
    keep = np.zeros(rows, bool)
    for i in range(rows):
        sq = [float(v) * float(v) for v in dev[i].astype(np.float64)]  # exact in binary64
        r = np.float32(S[i])
        up, down = np.nextafter(r, np.float32(np.inf)), np.nextafter(r, np.float32(-np.inf))
        hi = (float(r) + float(up)) / 2
        lo = (float(r) + float(down)) / 2
        if math.fsum(sq + [-hi]) > 0:
            alt = up
        elif math.fsum(sq + [-lo]) < 0:
            alt = down
        else:
            continue

        def rstd(s):
            var = np.float32(s / np.float32(H))
            return np.float32(np.float32(1.0) / np.sqrt(np.float32(var + np.float32(eps))))

        keep[i] = rstd(r) != rstd(alt)
    return keep
