"""The C-ABI library: it loads, exports every symbol include/*.h declares, and
its host-side validation returns the documented statuses.  No compute runs
here: every call below is rejected (or is a no-op) before any CUDA call."""
import ctypes
import itertools
import glob
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def far():
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    return far


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)  # drop comments
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("defined",):
                names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("fused_add_rmsnorm", "rmsnorm", "far_output_dtype", "far_status_string",
                     "far_device_status", "fused_add_rmsnorm_host", "rmsnorm_host"):
        assert required in names


def test_every_declared_symbol_is_exported(far):
    lib = ctypes.CDLL(far.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


D = {"f32": 0, "f16": 1, "bf16": 2}


def code(a, w):
    return D[a] | (D[w] << 4)


def test_output_dtype_policy(far):
    L = far.lib
    assert L.far_output_dtype(code("f16", "bf16")) == -1  # -FAR_ERR_DTYPE_MIX
    assert L.far_output_dtype(code("bf16", "f16")) == -1
    assert L.far_output_dtype(code("bf16", "bf16")) == D["bf16"]
    assert L.far_output_dtype(code("f16", "f16")) == D["f16"]
    for a in ("f16", "bf16", "f32"):
        assert L.far_output_dtype(code(a, "f32")) == D["f32"]
        assert L.far_output_dtype(code("f32", a)) == D["f32"]
    assert L.far_output_dtype(3) == -2 and L.far_output_dtype(0x100) == -2 and L.far_output_dtype(-1) == -2


FAKE = 1 << 40  # never dereferenced: every call below fails validation first


def call(far, x=FAKE, r=FAKE + (1 << 30), w=FAKE + (2 << 30), eps=1e-6, out=FAKE + (3 << 30),
         ro=FAKE + (4 << 30), tokens=4, hidden=64, dtype=None):
    dtype = code("bf16", "bf16") if dtype is None else dtype
    return far.lib.fused_add_rmsnorm(x, r, w, eps, out, ro, tokens, hidden, dtype, None)


def test_validation_statuses(far):
    assert call(far, dtype=code("f16", "bf16")) == 1   # FAR_ERR_DTYPE_MIX
    assert call(far, dtype=code("bf16", "f16")) == 1
    assert call(far, dtype=7) == 2                      # FAR_ERR_DTYPE
    assert call(far, x=None) == 3                       # FAR_ERR_NULL
    assert call(far, w=None) == 3
    assert call(far, ro=None) == 3
    assert call(far, hidden=0) == 4                     # FAR_ERR_SHAPE
    assert call(far, hidden=(1 << 24) + 1) == 4
    assert call(far, tokens=-1) == 4
    assert call(far, tokens=1 << 62, hidden=1 << 20) == 4
    assert call(far, eps=-1e-6) == 6                    # FAR_ERR_EPS
    assert call(far, eps=float("nan")) == 6
    assert call(far, eps=float("inf")) == 6
    # aliasing: exact in-place is allowed, partial overlap is not
    assert call(far, out=FAKE + 2) == 5                 # out overlaps x partially
    assert call(far, ro=FAKE + (1 << 30) + 64) == 5     # residual_out overlaps residual partially
    assert call(far, out=FAKE + (4 << 30)) == 5         # out == residual_out
    assert call(far, out=FAKE + (2 << 30)) == 5         # out overlaps the weight
    assert call(far, dtype=code("bf16", "f32"), out=FAKE) == 5  # fp32 out cannot alias a bf16 x
    # no-residual variant
    assert far.lib.rmsnorm(FAKE, FAKE + (2 << 30), 1e-6, FAKE + 2, 4, 64, code("f16", "f16"), None) == 5
    assert far.lib.rmsnorm(FAKE, None, 1e-6, FAKE + (3 << 30), 4, 64, code("f16", "f16"), None) == 3
    assert far.lib.rmsnorm(FAKE, FAKE + (2 << 30), 1e-6, FAKE + (3 << 30), 4, 64, code("f16", "bf16"), None) == 1


def test_zero_tokens_is_a_noop(far):
    assert call(far, tokens=0, x=None, r=None, w=None, out=None, ro=None) == 0
    assert far.lib.rmsnorm(None, None, 1e-6, None, 0, 128, code("f32", "f32"), None) == 0


def test_row_schedule_hook(far):
    """The default row schedule is the fixed stride (mode 1: no state kept between calls);
    far_set_row_schedule takes 0, 1 or 2 and refuses anything else (FAR_ERR_SHAPE), leaving
    the mode as it was; nothing launched on this thread means no rows claimed (a zero-token
    call launches nothing)."""
    assert far.lib.far_get_row_schedule() == 1
    try:
        for mode in (0, 1, 2):
            assert far.lib.far_set_row_schedule(mode) == 0
            assert far.get_row_schedule() == mode
        for mode in (-1, 3, 1 << 20):
            assert far.lib.far_set_row_schedule(mode) == 4
            assert far.get_row_schedule() == 2
    finally:
        assert far.lib.far_set_row_schedule(1) == 0
    assert far.lib.fused_add_rmsnorm(FAKE, FAKE, FAKE, 1e-6, FAKE, FAKE, 0, 64, code("bf16", "bf16"), None) == 0
    assert far.lib.far_last_launch_claimed_rows() == 0
    assert far.last_launch_claimed_rows() is False


def test_row_schedule_rule(far):
    """The default keeps the fixed stride everywhere. The automatic claimed-row rule (mode 0,
    host logic): one row a claim where a row moves 45 KB or more, two down to 23 KB, the
    fixed stride on shorter rows and on launches with fewer than four ring-fulls of rows a
    CTA; three rows a claim (15-22 KB) only for the packed no-residual kernels on 16-bit
    rows (16-bit or quantised out) with eight ring-fulls or more and a row that is not a
    whole number of 256 chunks; mode 2 claims wherever rows are left."""
    f16, bf16, f32 = torch.float16, torch.bfloat16, torch.float32

    def rows(tokens, hidden, act, wd, residual, op, sms=152):
        return far.row_schedule_for_sms(tokens, hidden, act, wd, residual, op, sms)

    assert far.get_row_schedule() == 1
    for op in ("rmsnorm", "layernorm", "quant"):
        assert rows(65536, 8192, f16, f16, True, op) == 0
        assert rows(65536, 8192, f16, f16, False, op) == 0
    far.set_row_schedule(0)
    for op in ("rmsnorm", "layernorm", "quant"):
        assert rows(65536, 8192, f16, f16, True, op) == 1      # 64 KB (56 KB quantised) a row
        assert rows(65536, 8192, f16, f16, False, op) == 2     # 32 KB (24 KB)
    assert rows(16384, 5120, bf16, bf16, True, "rmsnorm") == 2   # 40 KB
    assert rows(16384, 5120, bf16, bf16, False, "rmsnorm") == 3  # 20 KB, packed: 3 a claim
    assert rows(16384, 5120, bf16, bf16, False, "quant") == 3    # 15.4 KB
    assert rows(32768, 4608, bf16, bf16, False, "rmsnorm") == 3  # 18 KB, 576 chunks
    assert rows(16384, 4096, f16, f16, False, "rmsnorm") == 0    # 16 KB, 512 chunks: stride
    assert rows(8192, 5120, f16, f16, False, "rmsnorm") == 0     # 5.4 ring-fulls a CTA
    assert rows(16384, 5120, bf16, bf16, False, "layernorm") == 0  # LayerNorm keeps the stride
    assert rows(32768, 2048, f16, f16, True, "rmsnorm") == 0     # 16 KB fused: stride
    assert rows(16384, 3072, bf16, f32, False, "rmsnorm") == 0   # binary32 out: stride
    assert rows(4096, 4096, bf16, f32, True, "rmsnorm") == 2     # 40 KB
    assert rows(65536, 1024, bf16, bf16, True, "rmsnorm") == 0   # 8 KB
    for tokens, hidden, dt in ((512, 8192, f16), (512, 5120, bf16), (8, 2048, bf16)):
        assert rows(tokens, hidden, dt, dt, True, "rmsnorm") == 0  # under four ring-fulls a CTA
    # bf16 / fp32-weight 4096 x 4096 variant: 24 KB a row (two a claim) but 10 ring slots, so
    # 4096 rows are 2.7 ring-fulls of 152 CTAs: the fixed stride
    assert rows(4096, 4096, bf16, f32, False, "rmsnorm") == 0
    assert rows(65536, 1888, bf16, bf16, False, "quant") == 0
    try:
        far.set_row_schedule(1)
        assert rows(65536, 8192, f16, f16, True, "rmsnorm") == 0
        far.set_row_schedule(2)
        assert rows(65536, 1024, bf16, bf16, True, "rmsnorm") == 6  # ceil(45333 / 8192)
        assert rows(16384, 5120, bf16, bf16, False, "rmsnorm") == 3
        # a quantised row also moves its 4-byte scale: 1888 x (2 + 1) + 4 = 5668 B, so
        # ceil(45333 / 5668) = 8 rows a claim (9 if the scale were left out)
        assert rows(65536, 1888, bf16, bf16, False, "quant") == 8
        assert rows(65536, 2048, bf16, bf16, False, "rmsnorm") == 6  # ceil(45333 / 8192)
    finally:
        far.set_row_schedule(1)
    out = ctypes.c_int(0)
    for args in ((0, 8192, 1, 1, 0, 152), (64, 8192, 1, 1, 3, 152), (64, 8192, 1, 1, 0, 0)):
        assert far.lib.far_row_schedule_for_sms(*args, ctypes.addressof(out)) == 4  # FAR_ERR_SHAPE


def test_host_workspace_size(far):
    n1 = far.lib.far_host_workspace_bytes(1, 4096, code("bf16", "f32"), 1)
    n8 = far.lib.far_host_workspace_bytes(8, 4096, code("bf16", "f32"), 1)
    # weight + two slots of (x, residual, residual_out in bf16, out in fp32)
    assert n8 == 4096 * 4 + 2 * 8 * 4096 * (2 + 2 + 2 + 4)
    assert n1 < n8
    assert far.lib.far_host_workspace_bytes(8, 4096, code("f16", "bf16"), 1) == -1
    assert far.lib.far_host_workspace_bytes(0, 4096, code("f16", "f16"), 1) == -4


def test_status_strings(far):
    for s in range(10):
        assert far.lib.far_status_string(s)
    assert b"bf16" in far.lib.far_status_string(1)


def test_binding_rejects_mixed_halves_before_the_call(far):
    with pytest.raises(far.FarError):
        far.output_dtype(torch.float16, torch.bfloat16)


def test_launch_plans_are_consistent(far):
    """The host planner, over shapes, dtype pairs, SM counts and every override the
    tests and the bench use: each ring slot belongs to one group (stages a multiple of
    groups), the CTA fits the register and shared-memory budgets, the grid covers
    the rows, and a row is covered by its group's warps."""
    T16, B16, F32 = torch.float16, torch.bfloat16, torch.float32
    overrides = [(-1, 0, 0, 0), (0, 4, 1, 2), (0, 4, 2, 3), (0, 8, 1, 0), (0, 8, 4, 0), (0, 2, 0, 0),
                 (0, 4, 2, 0), (0, 8, 3, 0), (0, 4, 2, 4), (0, 8, 2, 4), (0, 1, 0, 0), (0, 4, 16, 5), (0, 5, 0, 0),
                 (0, 6, 3, 6), (0, 10, 0, 0), (0, 10, 9, 18), (0, 8, 6, 12)]
    try:
        for kind, nch, groups, stages in overrides:
            far.set_launch_override(kind, nch, groups, stages)
            for (act, wd), hidden, tokens, res, sms in itertools.product(
                    [(T16, T16), (B16, B16), (B16, F32), (F32, F32), (F32, B16)],
                    [1, 8, 64, 1000, 1536, 2048, 2560, 3072, 4096, 5120, 6144, 8192, 12288, 16384, 24576, 32768],
                    [1, 8, 151, 152, 4096, 65536], (True, False), (152, 148, 1)):
                p = far.plan_for_sms(tokens, hidden, act, wd, res, sms)
                if p["kind"] == 1:  # generic kernel
                    assert p["threads"] == 256 and p["smem"] == 0 and 1 <= p["grid"] <= min(tokens, 8 * sms)
                    continue
                sa = 4 if act == F32 else 2
                chunks = hidden * sa // 16
                G, g, st = p["warps_per_row"], p["groups"], p["stages"]
                assert p["nch"] in (1, 2, 4, 5, 6, 8, 10)
                if p["nch"] in (5, 6, 10):  # only as exact plans
                    assert hidden * (4 if act == F32 else 2) // 16 == p["nch"] * p["warps_per_row"] * 32, p
                assert st >= 2 and st % g == 0, p
                packed = not res and act != F32  # the no-residual variant keeps 16-bit x packed
                if p["nch"] == 10:
                    assert packed, p
                # 19 consumer warps for packed rows (96 registers a thread), else 12 or 16
                assert g * G <= (19 if packed else 12 if p["nch"] == 8 else 16), p
                if kind == -1 and not (packed and wd != F32):
                    assert g * G <= 16, p  # the default plans keep to 16 but for the 16-bit variant
                assert p["threads"] == (1 + g * G) * 32
                assert p["smem"] <= 227 * 1024
                # the group's warps cover the row, and one warp fewer would not
                assert (G - 1) * 32 * p["nch"] < chunks <= G * 32 * p["nch"], p
                assert 1 <= p["grid"] <= min(sms, -(-tokens // g))
    finally:
        far.set_launch_override()


def strided(far, x=FAKE, xs=256, r=FAKE + (1 << 30), rs=256, w=FAKE + (2 << 30), out=FAKE + (3 << 30), os_=256,
            ro=FAKE + (4 << 30), ros=256, tokens=4, hidden=64, dtype=None, res=1):
    """The strided entry point's argument checks alone (host logic, no CUDA call)."""
    dtype = code("bf16", "bf16") if dtype is None else dtype
    return far.lib.far_validate_strided(x, xs, r, rs, w, 1e-6, out, os_, ro, ros, tokens, hidden, dtype, res)


def test_strided_validation(far):
    """Strided aliasing: equal-stride column slices of one buffer may interleave; any
    shared byte is rejected; an output may be exactly its input (in place)."""
    B = FAKE + (8 << 30)  # a [4, 256] bf16 buffer holding four [4, 64] column slices
    ok = dict(x=B, xs=256, out=B + 128, os_=256, ro=B + 256, ros=256, r=B + 384, rs=256)
    assert strided(far, **ok) == 0                      # interleaved slices share no byte
    assert strided(far, **dict(ok, out=B + 64)) == 5     # out shares half its columns with x
    assert strided(far, **dict(ok, out=B + 512)) == 5    # out rows shifted by one row: overlap
    assert strided(far, **dict(ok, out=B + 2)) == 5      # a partial overlap
    assert strided(far, **dict(ok, out=B)) == 0          # out exactly x: in place
    assert strided(far, **dict(ok, ro=B + 384)) == 0     # residual_out exactly the residual: in place
    assert strided(far, **dict(ok, ro=B + 128)) == 5     # residual_out == out
    assert strided(far, **dict(ok, os_=320)) == 5        # different strides whose spans overlap
    assert strided(far, **dict(ok, xs=32)) == 4          # a stride below hidden
    assert strided(far, **dict(ok, ros=63)) == 4
    assert strided(far, **dict(ok, x=None)) == 3
    # rows far apart in memory (stride much larger than the row) never touch
    assert strided(far, x=B, xs=4096, out=B + 1024, os_=4096, ro=B + 2048, ros=4096, r=B + 3072, rs=4096) == 0
    # the no-residual variant ignores the residual arguments
    assert strided(far, res=0, r=B, ro=B, **{k: v for k, v in ok.items() if k not in ("r", "ro")}) == 0
    assert strided(far, res=0, r=None, ro=None, x=B, xs=256, out=B + 100, os_=256) == 5


def test_quantised_launch_plans_are_consistent(far):
    """The planner's quantised plans: slots belong to one group, the CTA fits the 12-warp
    (8 chunks) or 16-warp budget of the fused quantised kernels or the 19-warp budget of the
    no-residual variant on 16-bit rows, shared memory fits, rows covered."""
    T16, B16, F32 = torch.float16, torch.bfloat16, torch.float32
    try:
        for override in [(-1, 0, 0, 0), (0, 8, 3, 0), (0, 4, 2, 3), (0, 2, 0, 0), (0, 8, 8, 8)]:
            far.set_launch_override(*override)
            for (act, wd), hidden, tokens, res, qtype in itertools.product(
                    [(T16, T16), (B16, B16), (B16, F32), (F32, F32)], [8, 1000, 4096, 5120, 8192, 16384],
                    [1, 151, 4096, 65536], (True, False), ("int8", "fp8")):
                p = far.plan_quant_for_sms(tokens, hidden, act, wd, res, qtype, 152)
                if p["kind"] == 1:
                    continue
                G, g, st = p["warps_per_row"], p["groups"], p["stages"]
                assert st >= 2 and st % g == 0, p
                packed = not res and act != F32  # x kept packed: 96 registers a thread
                assert g * G <= (19 if packed else 12 if p["nch"] == 8 else 16), p
                assert p["threads"] == (1 + g * G) * 32 and p["smem"] <= 227 * 1024
                chunks = hidden * (4 if act == F32 else 2) // 16
                assert (G - 1) * 32 * p["nch"] < chunks <= G * 32 * p["nch"], p
    finally:
        far.set_launch_override()


def test_layernorm_validation(far):
    """LayerNorm's checks (every call below is rejected before any CUDA call): beta
    must be given, and no output may overlap it; the rest is RMSNorm's validation."""
    x, r, g, b = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (5 << 30)
    out, ro = FAKE + (3 << 30), FAKE + (4 << 30)
    bf = code("bf16", "bf16")
    L = far.lib
    assert L.fused_add_layernorm(x, r, g, None, 1e-5, out, ro, 4, 64, bf, None) == 3
    assert L.layernorm(x, g, None, 1e-5, out, 4, 64, bf, None) == 3
    assert L.fused_add_layernorm(x, r, g, b, 1e-5, b + 64, ro, 4, 64, bf, None) == 5   # out over beta
    assert L.fused_add_layernorm(x, r, g, b, 1e-5, out, b - 64, 4, 64, bf, None) == 5  # residual_out over beta
    assert L.layernorm(x, g, b, 1e-5, b, 4, 64, bf, None) == 5
    assert L.layernorm(x, g, b, 1e-5, out, 4, 64, code("f16", "bf16"), None) == 1
    assert L.layernorm(x, g, b, -1.0, out, 4, 64, bf, None) == 6
    assert L.layernorm(x, g, b, 1e-5, x + 2, 4, 64, bf, None) == 5
    assert L.layernorm(None, None, None, 1e-5, None, 0, 64, bf, None) == 0  # zero tokens: a no-op


def test_layernorm_launch_plans_are_consistent(far):
    """LayerNorm plans: gamma and beta both in shared memory, four reduction buffers,
    slots owned by one group, the CTA within its warp and shared-memory budgets."""
    T16, B16, F32 = torch.float16, torch.bfloat16, torch.float32
    try:
        for override in [(-1, 0, 0, 0), (0, 8, 3, 0), (0, 4, 2, 3), (0, 2, 0, 0), (0, 8, 8, 8), (0, 1, 0, 0)]:
            far.set_launch_override(*override)
            for (act, wd), hidden, tokens, res, sms in itertools.product(
                    [(T16, T16), (B16, B16), (B16, F32), (F32, F32), (F32, T16)],
                    [1, 8, 1000, 4096, 5120, 8192, 16384, 32768], [1, 151, 4096, 65536], (True, False),
                    (152, 1)):
                p = far.plan_ln_for_sms(tokens, hidden, act, wd, res, sms)
                if p["kind"] == 1:
                    assert p["threads"] == 256 and p["smem"] == 0
                    continue
                G, g, st = p["warps_per_row"], p["groups"], p["stages"]
                assert st >= 2 and st % g == 0, p
                assert g * G <= (12 if p["nch"] == 8 else 16), p
                assert p["threads"] == (1 + g * G) * 32 and p["smem"] <= 227 * 1024
                sa, sw = (4 if act == F32 else 2), (4 if wd == F32 else 2)
                chunks = hidden * sa // 16
                assert (G - 1) * 32 * p["nch"] < chunks <= G * 32 * p["nch"], p
                # shared memory holds gamma and beta besides the ring
                w16 = -(-hidden * sw // 16) * 16
                assert p["smem"] >= 2 * w16 + st * hidden * sa * (2 if res else 1), p
    finally:
        far.set_launch_override()


def test_layernorm_plan_needs_aligned_beta(far):
    """The staged kernel copies gamma and beta with 16-byte loads: a beta off a 16-byte
    boundary must route the call to the generic kernel (host logic only)."""
    B16 = torch.bfloat16
    assert far.plan_ln_for_sms(4096, 4096, B16, B16, True, 152)["kind"] == 0
    for off in (2, 8):
        assert far.plan_ln_for_sms(4096, 4096, B16, B16, True, 152, beta_offset=off)["kind"] == 1
        assert far.plan_ln_for_sms(4096, 4096, B16, B16, False, 152, beta_offset=off)["kind"] == 1


def test_gemm_validation(far):
    """The GEMM's checks, every call rejected before any CUDA call (or a no-op)."""
    L = far.lib
    x, wt, b, out = FAKE, FAKE + (1 << 30), FAKE + (2 << 30), FAKE + (3 << 30)
    assert L.gemm_f16_f32acc(x, wt, None, out, 4, 8, 16, 7, None) == 2         # unknown out dtype
    assert L.gemm_f16_f32acc(x, wt, b, out, 4, 8, 16, 0, None) == 2            # a bias with fp32 out
    assert L.gemm_f16_f32acc(x, wt, None, out, -1, 8, 16, 1, None) == 4
    assert L.gemm_f16_f32acc(x, wt, None, out, 4, 8, 1 << 31, 1, None) == 4
    assert L.gemm_f16_f32acc(None, wt, None, out, 4, 8, 16, 1, None) == 3
    assert L.gemm_f16_f32acc(x, wt, None, None, 4, 8, 16, 1, None) == 3
    assert L.gemm_f16_f32acc(x, wt, None, x + 8, 4, 8, 16, 1, None) == 5       # out over x
    assert L.gemm_f16_f32acc(x, wt, b, b - 16, 4, 8, 16, 1, None) == 5         # out over the bias
    assert L.gemm_f16_f32acc(None, None, None, None, 0, 8, 16, 1, None) == 0   # empty output: no-op


def test_gemm_plans(far):
    """Tensor cores for aligned shapes with k and n multiples of 8, else the plain kernel;
    the tile width keeps a tile per SM where it can; the shared memory fits."""
    T16, F32 = torch.float16, torch.float32
    p = far.plan_gemm_for_sms(1024, 1024, 768, True, T16, 152)
    assert p["kind"] == 0 and p["bn"] == 64 and p["grid"] == 8 * 16
    p = far.plan_gemm_for_sms(8192, 8192, 8192, False, F32, 152)
    assert p["kind"] == 2 and p["bn"] == 256 and p["grid"] == 152  # CTA pairs, one CTA per SM
    assert far.plan_gemm_for_sms(4096, 2048, 4096, True, T16, 152)["bn"] == 256
    # 64 pair tiles (half the pairs or more): pairs, whole tiles in one round
    assert far.plan_gemm_for_sms(1024, 4096, 4096, True, T16, 152)["kind"] == 2
    assert far.plan_gemm_for_sms(2048, 2048, 8192, True, T16, 152)["kind"] == 2
    assert far.plan_gemm_for_sms(1024, 1024, 4096, True, T16, 152)["kind"] == 0  # 16 pair tiles: one CTA a tile
    # one CTA a tile: the width of least estimated time (waves x width x the width's cost a
    # column): 144 tiles of 128 in one wave rather than 288 of 64 in two
    p = far.plan_gemm_for_sms(1536, 1536, 4096, True, T16, 152)
    assert p["kind"] == 0 and p["bn"] == 128 and p["grid"] == 144
    assert far.plan_gemm_for_sms(1024, 2048, 2048, True, T16, 152)["bn"] == 128
    try:
        far.set_gemm_override(0, 0)
        assert far.plan_gemm_for_sms(4096, 2048, 4096, True, T16, 152)["bn"] == 256
    finally:
        far.set_gemm_override()
    for m, n, k in [(100, 8, 8), (1, 8, 4096), (5000, 1000, 64)]:
        p = far.plan_gemm_for_sms(m, n, k, True, T16, 152)
        assert p["kind"] in (0, 2) and p["smem"] <= 227 * 1024 and p["threads"] == 192
        assert p["grid"] % 2 == 0 or p["kind"] == 0  # pairs launch whole clusters
    for m, n, k in [(64, 12, 64), (64, 64, 12), (64, 64, 0), (3, 5, 7)]:
        assert far.plan_gemm_for_sms(m, n, k, True, T16, 152)["kind"] == 1


def test_strided_layernorm_and_quant_validation(far):
    """The strided LayerNorm and quantised entry points reject before any CUDA call: a
    stride below hidden, a missing beta or scale, an output over beta or over x."""
    L = far.lib
    B = FAKE + (8 << 30)
    g, b = FAKE + (2 << 30), FAKE + (5 << 30)
    bf = code("bf16", "bf16")
    assert L.fused_add_layernorm_strided(B, 32, B + 128, 256, g, b, 1e-5, B + 256, 256, B + 384, 256, 4, 64, bf,
                                         None) == 4   # x stride below hidden
    assert L.fused_add_layernorm_strided(B, 256, B + 128, 256, g, None, 1e-5, B + 256, 256, B + 384, 256, 4, 64, bf,
                                         None) == 3   # no beta
    assert L.layernorm_strided(B, 256, g, b, 1e-5, B + 64, 256, 4, 64, bf, None) == 5      # out shares x's columns
    assert L.layernorm_strided(B, 256, g, b, 1e-5, b, 256, 4, 64, bf, None) == 5           # out over beta
    q, sc = FAKE + (3 << 30), FAKE + (6 << 30)
    assert L.rmsnorm_quant_strided(B, 63, g, 1e-6, q, sc, 4, 64, bf, 1, None) == 4
    assert L.rmsnorm_quant_strided(B, 256, g, 1e-6, q, None, 4, 64, bf, 1, None) == 3
    assert L.rmsnorm_quant_strided(B, 256, g, 1e-6, B + 16, sc, 4, 64, bf, 1, None) == 5   # q inside x's rows
    assert L.fused_add_rmsnorm_quant_strided(B, 256, B + 128, 256, g, 1e-6, q, sc, B + 130, 256, 4, 64, bf, 2,
                                             None) == 5  # residual_out overlaps the residual partially
    assert L.fused_add_rmsnorm_quant_strided(B, 256, B + 128, 256, g, 1e-6, q, sc, B + 256, 256, 4, 64, bf, 3,
                                             None) == 2  # unknown quantised type


def test_host_workspace_size_per_op(far):
    """RMSNorm's layout is unchanged; LayerNorm keeps beta beside gamma; a quantised output
    holds q (one byte an element) and the per-row scales in place of out."""
    T, H, bf = 8, 4096, code("bf16", "f32")
    a256 = lambda n: -(-n // 256) * 256
    assert far.lib.far_host_workspace_bytes_op(T, H, bf, 1, 0) == far.lib.far_host_workspace_bytes(T, H, bf, 1)
    assert far.lib.far_host_workspace_bytes_op(T, H, bf, 1, 1) == 2 * a256(H * 4) + 2 * (3 * a256(T * H * 2) + a256(T * H * 4))
    assert far.lib.far_host_workspace_bytes_op(T, H, bf, 0, 2) == a256(H * 4) + 2 * (a256(T * H * 2) + a256(T * H) + a256(T * 4))
    assert far.lib.far_host_workspace_bytes_op(T, H, bf, 1, 3) == -4


def test_counter_pool_bookkeeping(far):
    """The claimed-row counter pool as host logic (far_sched_pool_model): a stream keeps
    reusing its own pair, even with launches still pending on it and no event completed; a
    pair with a launch pending, or whose last launch's event has not completed, is never
    handed to another stream; a completed event frees it; a pair whose launch got no event
    is retired for good; with every pair busy a launch gets none (fixed stride)."""
    ACQ, REL = 1, 2
    LAUNCHED, RECORDED = 1, 2
    done_none, done_all = 0, (1 << 64) - 1
    m = far.sched_pool_model
    # one stream: the same pair over and over, with launches pending and no event done
    assert m([(ACQ, 7, done_none), (REL, 0, LAUNCHED | RECORDED), (ACQ, 7, done_none), (ACQ, 7, done_none)]) == \
        [0, 0, 0, 0]
    # another stream while pair 0 is pending on stream 7: a fresh pair
    assert m([(ACQ, 7, done_none), (ACQ, 8, done_none)]) == [0, 1]
    # pair 0 released, its event not yet done: stream 8 takes a fresh pair; done: next free in turn
    ops = [(ACQ, 7, done_none), (REL, 0, LAUNCHED | RECORDED), (ACQ, 8, done_none)]
    assert m(ops) == [0, 0, 1]
    # after every other pair is taken by other streams, pair 0 goes to stream 9 once its event is done
    ops = [(ACQ, 7, done_none), (REL, 0, LAUNCHED | RECORDED)]
    ops += [(ACQ, 100 + s, done_none) for s in range(1, 64)]
    assert m(ops + [(ACQ, 9, done_none)])[-1] == -1       # every pair busy or unfinished
    assert m(ops + [(ACQ, 9, 1 << 0)])[-1] == 0            # pair 0's event completed
    assert m(ops + [(ACQ, 7, done_none)])[-1] == 0         # its own stream still may
    # a launched pair without an event is retired: neither its stream nor any other gets it back
    ops = [(ACQ, 7, done_none), (REL, 0, LAUNCHED)]
    assert m(ops + [(ACQ, 7, done_all)])[-1] == 1
    assert m(ops + [(ACQ, 8, done_all)])[-1] == 1
    # a launch that failed to enqueue gives its pair back unused: any stream may take it
    ops = [(ACQ, 7, done_none), (REL, 0, 0)] + [(ACQ, 100 + s, done_none) for s in range(1, 64)]
    assert m(ops + [(ACQ, 8, done_none)])[-1] == 0
    # 64 streams with a launch pending each exhaust the pool; the 65th gets none
    res = m([(ACQ, 1000 + s, done_all) for s in range(65)])
    assert sorted(res[:64]) == list(range(64)) and res[64] == -1
    # errors: an unknown op, giving back a pair that is not handed out
    flat = (ctypes.c_int64 * 3)(3, 0, 0)
    out = (ctypes.c_int * 1)()
    assert far.lib.far_sched_pool_model(ctypes.addressof(flat), 1, ctypes.addressof(out)) == 4
    flat = (ctypes.c_int64 * 3)(2, 5, 1)
    assert far.lib.far_sched_pool_model(ctypes.addressof(flat), 1, ctypes.addressof(out)) == 4


def test_plan_queries_take_the_largest_shapes(far):
    """The host-only plan queries answer for every shape the entry points accept, however
    large: their stand-in addresses are never checked for overlap, so they cannot wrap into
    a false FAR_ERR_ALIAS."""
    out = (ctypes.c_int * 8)()
    one = ctypes.c_int(0)
    code_ = code("f32", "f32")
    tokens = (2 ** 63 - 1) // 8 // (1 << 24)  # the largest accepted at hidden 2^24
    assert far.lib.far_plan_for_sms(tokens, 1 << 24, code_, 1, 152, ctypes.addressof(out)) == 0
    assert far.lib.far_row_schedule_for_sms(tokens, 1 << 24, code_, 1, 0, 152, ctypes.addressof(one)) == 0
    assert far.lib.far_plan_quant_for_sms(tokens, 1 << 24, code_, 1, 1, 152, ctypes.addressof(out)) == 0
    assert far.lib.far_plan_ln_for_sms(tokens, 1 << 24, code_, 1, 0, 152, ctypes.addressof(out)) == 0
    # one more row is a shape error, as for the entry points
    assert far.lib.far_plan_for_sms(tokens + 1, 1 << 24, code_, 1, 152, ctypes.addressof(out)) == 4


def test_plans_of_the_bench_workloads(far):
    """The planner's choices on a 152-SM GB300 for the five workloads, fused op and variant,
    and LayerNorm and int8 on the fp16 65536 x 8192 one: {kind, chunks a thread, warps a
    row, groups, ring slots, grid}. Each was chosen from timed sweeps of every plan (a change
    here should come with new measurements)."""
    f16, bf16, f32 = torch.float16, torch.bfloat16, torch.float32
    keys = ("kind", "nch", "warps_per_row", "groups", "stages", "grid")
    want = {
        ("c1", True): [0, 1, 8, 1, 4, 8], ("c1", False): [0, 1, 8, 1, 4, 8],
        ("c2", True): [0, 8, 4, 2, 2, 152], ("c2", False): [0, 8, 4, 4, 4, 128],
        ("c3", True): [0, 8, 2, 3, 3, 152], ("c3", False): [0, 8, 2, 5, 10, 152],
        ("c4", True): [0, 5, 4, 3, 3, 152], ("c4", False): [0, 10, 2, 5, 10, 152],
        ("c5", True): [0, 8, 4, 2, 2, 152], ("c5", False): [0, 8, 4, 4, 4, 152],
    }
    shapes = {"c1": (bf16, bf16, 8, 2048), "c2": (f16, f16, 512, 8192), "c3": (bf16, f32, 4096, 4096),
              "c4": (bf16, bf16, 16384, 5120), "c5": (f16, f16, 65536, 8192)}
    for (name, residual), plan in want.items():
        a, w, T, H = shapes[name]
        p = far.plan_for_sms(T, H, a, w, residual, 152)
        assert [p[k] for k in keys] == plan, (name, residual, p)
    for residual, ln, q8 in ((True, [0, 8, 4, 2, 2, 152], [0, 8, 4, 2, 2, 152]),
                             (False, [0, 8, 4, 3, 6, 152], [0, 8, 4, 4, 8, 152])):
        p = far.plan_ln_for_sms(65536, 8192, f16, f16, residual, 152)
        assert [p[k] for k in keys] == ln, ("layernorm", residual, p)
        p = far.plan_quant_for_sms(65536, 8192, f16, f16, residual, "int8", 152)
        assert [p[k] for k in keys] == q8, ("int8", residual, p)
