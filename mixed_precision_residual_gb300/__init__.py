"""GB300 fused residual-add + RMSNorm under the mixed-precision rounding contract.

A thin ctypes binding of the C ABI in ``include/far.h`` (library
``_build/libfar.so``, built for sm_103a by ``build.py``).  The functions keep
the C names and only marshal arguments: every step of the computation runs in
the library's CUDA kernels.  PyTorch provides device memory and streams.

    out, residual_out = fused_add_rmsnorm(x, residual, weight, eps)
    out = rmsnorm(x, weight, eps)

There is no fallback: importing this package fails loudly when the library
has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libfar.so")

F32, F16, BF16 = 0, 1, 2
STATUS = {0: "FAR_OK", 1: "FAR_ERR_DTYPE_MIX", 2: "FAR_ERR_DTYPE", 3: "FAR_ERR_NULL", 4: "FAR_ERR_SHAPE",
          5: "FAR_ERR_ALIAS", 6: "FAR_ERR_EPS", 7: "FAR_ERR_CUDA", 8: "FAR_ERR_TIMEOUT",
          9: "FAR_ERR_WORKSPACE", 10: "FAR_ERR_SCRATCH"}
FAR_OK, FAR_ERR_TIMEOUT = 0, 8
TORCH_TO_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
CODE_TO_TORCH = {v: k for k, v in TORCH_TO_CODE.items()}

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(python -c 'import __graft_entry__ as g; g.build()')")

lib = ctypes.CDLL(LIB_PATH)
_vp, _f32, _i64, _int, _u32 = ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
lib.fused_add_rmsnorm.argtypes = [_vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _vp]
lib.fused_add_rmsnorm.restype = _int
lib.rmsnorm.argtypes = [_vp, _vp, _f32, _vp, _i64, _i64, _int, _vp]
lib.rmsnorm.restype = _int
lib.fused_add_rmsnorm_strided.argtypes = [_vp, _i64, _vp, _i64, _vp, _f32, _vp, _i64, _vp, _i64, _i64, _i64, _int, _vp]
lib.fused_add_rmsnorm_strided.restype = _int
lib.rmsnorm_strided.argtypes = [_vp, _i64, _vp, _f32, _vp, _i64, _i64, _i64, _int, _vp]
lib.rmsnorm_strided.restype = _int
lib.far_validate_strided.argtypes = [_vp, _i64, _vp, _i64, _vp, _f32, _vp, _i64, _vp, _i64, _i64, _i64, _int, _int]
lib.far_validate_strided.restype = _int
lib.fused_add_rmsnorm_quant.argtypes = [_vp, _vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp]
lib.fused_add_rmsnorm_quant.restype = _int
lib.rmsnorm_quant.argtypes = [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _int, _vp]
lib.rmsnorm_quant.restype = _int
lib.far_plan_quant_for_sms.argtypes = [_i64, _i64, _int, _int, _int, _int, _vp]
lib.far_plan_quant_for_sms.restype = _int
lib.fused_add_layernorm.argtypes = [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _vp]
lib.fused_add_layernorm.restype = _int
lib.layernorm.argtypes = [_vp, _vp, _vp, _f32, _vp, _i64, _i64, _int, _vp]
lib.layernorm.restype = _int
lib.far_plan_ln_for_sms.argtypes = [_i64, _i64, _int, _int, _int, _int, _vp]
lib.far_plan_ln_for_sms.restype = _int
lib.far_host_workspace_bytes_op.argtypes = [_i64, _i64, _int, _int, _int]
lib.far_host_workspace_bytes_op.restype = _i64
lib.fused_add_layernorm_host.argtypes = [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _vp, _i64, _vp]
lib.fused_add_layernorm_host.restype = _int
lib.layernorm_host.argtypes = [_vp, _vp, _vp, _f32, _vp, _i64, _i64, _int, _vp, _i64, _vp]
lib.layernorm_host.restype = _int
lib.fused_add_rmsnorm_quant_host.argtypes = [_vp, _vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp, _i64,
                                             _vp]
lib.fused_add_rmsnorm_quant_host.restype = _int
lib.rmsnorm_quant_host.argtypes = [_vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _int, _vp, _i64, _vp]
lib.rmsnorm_quant_host.restype = _int
lib.fused_add_layernorm_strided.argtypes = [_vp, _i64, _vp, _i64, _vp, _vp, _f32, _vp, _i64, _vp, _i64, _i64, _i64,
                                            _int, _vp]
lib.fused_add_layernorm_strided.restype = _int
lib.layernorm_strided.argtypes = [_vp, _i64, _vp, _vp, _f32, _vp, _i64, _i64, _i64, _int, _vp]
lib.layernorm_strided.restype = _int
lib.fused_add_rmsnorm_quant_strided.argtypes = [_vp, _i64, _vp, _i64, _vp, _f32, _vp, _vp, _vp, _i64, _i64, _i64,
                                                _int, _int, _vp]
lib.fused_add_rmsnorm_quant_strided.restype = _int
lib.rmsnorm_quant_strided.argtypes = [_vp, _i64, _vp, _f32, _vp, _vp, _i64, _i64, _int, _int, _vp]
lib.rmsnorm_quant_strided.restype = _int
lib.gemm_f16_f32acc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
lib.gemm_f16_f32acc.restype = _int
lib.far_plan_gemm_for_sms.argtypes = [_i64, _i64, _i64, _int, _int, _int, _vp]
lib.far_plan_gemm_for_sms.restype = _int
lib.far_set_gemm_override.argtypes = [_int, _int]
lib.far_set_gemm_override.restype = _int
lib.far_output_dtype.argtypes = [_int]
lib.far_output_dtype.restype = _int
lib.far_status_string.argtypes = [_int]
lib.far_status_string.restype = ctypes.c_char_p
lib.far_device_status.argtypes = [_vp]
lib.far_device_status.restype = _int
lib.far_host_workspace_bytes.argtypes = [_i64, _i64, _int, _int]
lib.far_host_workspace_bytes.restype = _i64
lib.fused_add_rmsnorm_host.argtypes = [_vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _vp, _i64, _vp]
lib.fused_add_rmsnorm_host.restype = _int
lib.rmsnorm_host.argtypes = [_vp, _vp, _f32, _vp, _i64, _i64, _int, _vp, _i64, _vp]
lib.rmsnorm_host.restype = _int
lib.fused_add_rmsnorm_host_noalloc.argtypes = [_vp, _vp, _vp, _f32, _vp, _vp, _i64, _i64, _int, _vp]
lib.fused_add_rmsnorm_host_noalloc.restype = _int
lib.far_selftest_wait_timeout.argtypes = [_u32, _vp]
lib.far_selftest_wait_timeout.restype = _int
lib.far_set_launch_override.argtypes = [_int, _int, _int, _int]
lib.far_set_launch_override.restype = _int
lib.far_set_row_schedule.argtypes = [_int]
lib.far_set_row_schedule.restype = _int
lib.far_last_launch_claimed_rows.argtypes = []
lib.far_last_launch_claimed_rows.restype = _int
lib.far_get_row_schedule.argtypes = []
lib.far_get_row_schedule.restype = _int
lib.far_set_programmatic_launch.argtypes = [_int]
lib.far_set_programmatic_launch.restype = _int
lib.far_get_programmatic_launch.argtypes = []
lib.far_get_programmatic_launch.restype = _int
lib.far_sched_pool_model.argtypes = [_vp, _int, _vp]
lib.far_sched_pool_model.restype = _int
lib.far_row_schedule_for_sms.argtypes = [_i64, _i64, _int, _int, _int, _int, _vp]
lib.far_row_schedule_for_sms.restype = _int
lib.far_describe_launch.argtypes = [_i64, _i64, _int, _int, _vp]
lib.far_describe_launch.restype = _int
lib.far_plan_for_sms.argtypes = [_i64, _i64, _int, _int, _int, _vp]
lib.far_plan_for_sms.restype = _int


class FarError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {lib.far_status_string(status).decode()}")


def _check(status: int) -> None:
    if status != FAR_OK:
        raise FarError(status)


def dtypes(act: torch.dtype, wd: torch.dtype) -> int:
    """The packed dtype argument FAR_DTYPES(act, wd)."""
    return TORCH_TO_CODE[act] | (TORCH_TO_CODE[wd] << 4)


def output_dtype(act: torch.dtype, wd: torch.dtype) -> torch.dtype:
    code = lib.far_output_dtype(dtypes(act, wd))
    if code < 0:
        raise FarError(-code)
    return CODE_TO_TORCH[code]


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _rows(x: torch.Tensor) -> tuple[int, int]:
    hidden = x.shape[-1]
    return (x.numel() // hidden if hidden else 0), hidden


def _row_stride(t: torch.Tensor) -> int | None:
    """Row stride in elements of a 2-D tensor with contiguous rows, else None."""
    if t.dim() == 2 and (t.stride(1) == 1 or t.shape[1] == 1):
        return t.stride(0) if t.shape[0] > 1 else t.shape[1]
    return None


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor, eps: float,
                      out: torch.Tensor | None = None, residual_out: torch.Tensor | None = None,
                      stream=None):
    """out, residual_out = RMSNorm(x + residual) * weight under the rounding contract.

    x, residual: [..., hidden] CUDA tensors of one dtype, contiguous, or 2-D with
    contiguous rows and any row stride (column slices); weight: [hidden].  Outputs
    are allocated when not given (out in the promoted dtype); pass out=x /
    residual_out=residual for in-place use.
    """
    if not weight.is_contiguous():
        raise ValueError("weight must be contiguous")
    code = dtypes(x.dtype, weight.dtype)
    if residual.dtype != x.dtype:
        raise ValueError("x and residual must share a dtype")
    if out is None:
        out = torch.empty(x.shape, dtype=output_dtype(x.dtype, weight.dtype), device=x.device)
    if residual_out is None:
        residual_out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    tokens, hidden = _rows(x)
    if weight.numel() != hidden or residual.shape != x.shape or out.shape != x.shape or residual_out.shape != x.shape:
        raise ValueError("shape mismatch")
    ts = (x, residual, out, residual_out)
    if all(t.is_contiguous() for t in ts):
        _check(lib.fused_add_rmsnorm(_ptr(x), _ptr(residual), _ptr(weight), eps, _ptr(out), _ptr(residual_out),
                                     tokens, hidden, code, _stream_handle(stream)))
    else:
        st = [_row_stride(t) for t in ts]
        if None in st:
            raise ValueError("non-contiguous tensors must be 2-D with contiguous rows")
        _check(lib.fused_add_rmsnorm_strided(_ptr(x), st[0], _ptr(residual), st[1], _ptr(weight), eps, _ptr(out),
                                             st[2], _ptr(residual_out), st[3], tokens, hidden, code,
                                             _stream_handle(stream)))
    return out, residual_out


def rmsnorm(x: torch.Tensor, weight: torch.Tensor, eps: float, out: torch.Tensor | None = None, stream=None):
    """out = RMSNorm(x) * weight under the rounding contract (no residual)."""
    if not weight.is_contiguous():
        raise ValueError("weight must be contiguous")
    code = dtypes(x.dtype, weight.dtype)
    if out is None:
        out = torch.empty(x.shape, dtype=output_dtype(x.dtype, weight.dtype), device=x.device)
    tokens, hidden = _rows(x)
    if weight.numel() != hidden or out.shape != x.shape:
        raise ValueError("shape mismatch")
    if x.is_contiguous() and out.is_contiguous():
        _check(lib.rmsnorm(_ptr(x), _ptr(weight), eps, _ptr(out), tokens, hidden, code, _stream_handle(stream)))
    else:
        sx, so = _row_stride(x), _row_stride(out)
        if sx is None or so is None:
            raise ValueError("non-contiguous tensors must be 2-D with contiguous rows")
        _check(lib.rmsnorm_strided(_ptr(x), sx, _ptr(weight), eps, _ptr(out), so, tokens, hidden, code,
                                   _stream_handle(stream)))
    return out


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word's status."""
    return lib.far_device_status(_stream_handle(stream))


def host_workspace_bytes(chunk_tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype,
                         residual: bool = True) -> int:
    n = lib.far_host_workspace_bytes(chunk_tokens, hidden, dtypes(act, wd), int(residual))
    if n < 0:
        raise FarError(-n)
    return n


def fused_add_rmsnorm_host(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor, eps: float,
                           out: torch.Tensor, residual_out: torch.Tensor, workspace: torch.Tensor,
                           stream=None) -> None:
    """End-to-end call on host (CPU, ideally pinned) tensors through a device workspace."""
    tokens, hidden = _rows(x)
    _check(lib.fused_add_rmsnorm_host(_ptr(x), _ptr(residual), _ptr(weight), eps, _ptr(out), _ptr(residual_out),
                                      tokens, hidden, dtypes(x.dtype, weight.dtype), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def rmsnorm_host(x: torch.Tensor, weight: torch.Tensor, eps: float, out: torch.Tensor, workspace: torch.Tensor,
                 stream=None) -> None:
    tokens, hidden = _rows(x)
    _check(lib.rmsnorm_host(_ptr(x), _ptr(weight), eps, _ptr(out), tokens, hidden,
                            dtypes(x.dtype, weight.dtype), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def selftest_wait_timeout(timeout_us: int = 20000, stream=None) -> None:
    _check(lib.far_selftest_wait_timeout(timeout_us, _stream_handle(stream)))


def set_launch_override(kind: int = -1, nch: int = 0, groups: int = 0, stages: int = 0) -> None:
    _check(lib.far_set_launch_override(kind, nch, groups, stages))


def set_row_schedule(mode: int = 1) -> None:
    """How the staged kernel's CTAs share rows: 1 the fixed stride (the default, no state kept
    between calls), 0 claimed rows by the automatic rule, 2 claimed rows whenever possible
    (the same bits in every mode)."""
    _check(lib.far_set_row_schedule(mode))


def set_programmatic_launch(enable: bool = True) -> None:
    """Launch the normalisation kernels as programmatic dependent launches (the default) or
    plainly (the same bits either way)."""
    _check(lib.far_set_programmatic_launch(int(bool(enable))))


def get_programmatic_launch() -> bool:
    return bool(lib.far_get_programmatic_launch())


def get_row_schedule() -> int:
    """The current row-schedule mode (see set_row_schedule)."""
    return int(lib.far_get_row_schedule())


def sched_pool_model(ops) -> list:
    """Run the counter pool's bookkeeping alone (host logic, no CUDA call) on a fresh pool:
    ops is a list of (1, stream_id, done_mask) acquisitions and (2, pair, flags) releases;
    returns each operation's result (the pair handed out or -1; 0 for a release)."""
    n = len(ops)
    flat = (ctypes.c_int64 * (3 * max(n, 1)))(*[int(v) for op in ops for v in op])
    res = (ctypes.c_int * max(n, 1))()
    _check(lib.far_sched_pool_model(ctypes.addressof(flat), n, ctypes.addressof(res)))
    return list(res)[:n]


def row_schedule_for_sms(tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool, op: str,
                         sms: int) -> int:
    """Rows a claim for such a call under the current mode, 0 for the fixed stride (host
    logic only); op "rmsnorm", "layernorm" or "quant"."""
    out = ctypes.c_int(0)
    _check(lib.far_row_schedule_for_sms(tokens, hidden, dtypes(act, wd), int(residual),
                                        {"rmsnorm": 0, "layernorm": 1, "quant": 2}[op], sms, ctypes.addressof(out)))
    return out.value


def last_launch_claimed_rows() -> bool:
    """Whether this thread's last launch by the library claimed rows from a counter."""
    return bool(lib.far_last_launch_claimed_rows())


def describe_launch(tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool = True) -> dict:
    buf = (ctypes.c_int * 6)()
    _check(lib.far_describe_launch(tokens, hidden, dtypes(act, wd), int(residual), ctypes.addressof(buf)))
    return dict(zip(("kind", "nch", "warps_per_row", "groups", "stages", "grid"), list(buf)))


def plan_for_sms(tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool, sms: int) -> dict:
    """The launch plan for a device with `sms` SMs (host logic only, no GPU needed)."""
    buf = (ctypes.c_int * 8)()
    _check(lib.far_plan_for_sms(tokens, hidden, dtypes(act, wd), int(residual), sms, ctypes.addressof(buf)))
    return dict(zip(("kind", "nch", "warps_per_row", "groups", "stages", "grid", "threads", "smem"), list(buf)))


QUANT = {"int8": 1, "fp8": 2}


def fused_add_rmsnorm_quant(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor, eps: float,
                            qtype: str = "int8", q: torch.Tensor | None = None, scale: torch.Tensor | None = None,
                            residual_out: torch.Tensor | None = None, stream=None):
    """(q, scale, residual_out): the fused op with a per-token quantised output.

    q is int8 for "int8" and uint8 E4M3 codes for "fp8" (view as torch.float8_e4m3fn);
    dequantise as q * scale[:, None].
    """
    if not weight.is_contiguous():
        raise ValueError("weight must be contiguous")
    tokens, hidden = _rows(x)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8 if qtype == "int8" else torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(tokens, dtype=torch.float32, device=x.device)
    if residual_out is None:
        residual_out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    if not (q.is_contiguous() and scale.is_contiguous()):
        raise ValueError("q and scale must be contiguous")
    code = dtypes(x.dtype, weight.dtype)
    ts = (x, residual, residual_out)
    if all(t.is_contiguous() for t in ts):
        _check(lib.fused_add_rmsnorm_quant(_ptr(x), _ptr(residual), _ptr(weight), eps, _ptr(q), _ptr(scale),
                                           _ptr(residual_out), tokens, hidden, code, QUANT[qtype],
                                           _stream_handle(stream)))
    else:
        st = [_row_stride(t) for t in ts]
        if None in st:
            raise ValueError("non-contiguous tensors must be 2-D with contiguous rows")
        _check(lib.fused_add_rmsnorm_quant_strided(_ptr(x), st[0], _ptr(residual), st[1], _ptr(weight), eps, _ptr(q),
                                                   _ptr(scale), _ptr(residual_out), st[2], tokens, hidden, code,
                                                   QUANT[qtype], _stream_handle(stream)))
    return q, scale, residual_out


def rmsnorm_quant(x: torch.Tensor, weight: torch.Tensor, eps: float, qtype: str = "int8",
                  q: torch.Tensor | None = None, scale: torch.Tensor | None = None, stream=None):
    """(q, scale): the no-residual variant with a per-token quantised output."""
    if not weight.is_contiguous():
        raise ValueError("weight must be contiguous")
    tokens, hidden = _rows(x)
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8 if qtype == "int8" else torch.uint8, device=x.device)
    if scale is None:
        scale = torch.empty(tokens, dtype=torch.float32, device=x.device)
    code = dtypes(x.dtype, weight.dtype)
    if x.is_contiguous():
        _check(lib.rmsnorm_quant(_ptr(x), _ptr(weight), eps, _ptr(q), _ptr(scale), tokens, hidden, code,
                                 QUANT[qtype], _stream_handle(stream)))
    else:
        sx = _row_stride(x)
        if sx is None:
            raise ValueError("a non-contiguous x must be 2-D with contiguous rows")
        _check(lib.rmsnorm_quant_strided(_ptr(x), sx, _ptr(weight), eps, _ptr(q), _ptr(scale), tokens, hidden, code,
                                         QUANT[qtype], _stream_handle(stream)))
    return q, scale


def plan_quant_for_sms(tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool, qtype: str,
                       sms: int) -> dict:
    buf = (ctypes.c_int * 8)()
    _check(lib.far_plan_quant_for_sms(tokens, hidden, dtypes(act, wd), int(residual), QUANT[qtype], sms,
                                      ctypes.addressof(buf)))
    return dict(zip(("kind", "nch", "warps_per_row", "groups", "stages", "grid", "threads", "smem"), list(buf)))


def fused_add_layernorm(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor,
                        eps: float, out: torch.Tensor | None = None, residual_out: torch.Tensor | None = None,
                        stream=None):
    """out, residual_out = LayerNorm(x + residual) * gamma + beta under the rounding contract.

    x, residual: [..., hidden] CUDA tensors of one dtype, contiguous or 2-D with contiguous
    rows and any row stride; gamma, beta: contiguous [hidden] in the weight dtype.
    Outputs are allocated when not given.
    """
    if not (gamma.is_contiguous() and beta.is_contiguous()):
        raise ValueError("gamma and beta must be contiguous")
    if residual.dtype != x.dtype or beta.dtype != gamma.dtype:
        raise ValueError("x and residual, gamma and beta must share a dtype")
    code = dtypes(x.dtype, gamma.dtype)
    if out is None:
        out = torch.empty(x.shape, dtype=output_dtype(x.dtype, gamma.dtype), device=x.device)
    if residual_out is None:
        residual_out = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    tokens, hidden = _rows(x)
    if (gamma.numel() != hidden or beta.numel() != hidden or residual.shape != x.shape or out.shape != x.shape
            or residual_out.shape != x.shape):
        raise ValueError("shape mismatch")
    ts = (x, residual, out, residual_out)
    if all(t.is_contiguous() for t in ts):
        _check(lib.fused_add_layernorm(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(beta), eps, _ptr(out),
                                       _ptr(residual_out), tokens, hidden, code, _stream_handle(stream)))
    else:
        st = [_row_stride(t) for t in ts]
        if None in st:
            raise ValueError("non-contiguous tensors must be 2-D with contiguous rows")
        _check(lib.fused_add_layernorm_strided(_ptr(x), st[0], _ptr(residual), st[1], _ptr(gamma), _ptr(beta), eps,
                                               _ptr(out), st[2], _ptr(residual_out), st[3], tokens, hidden, code,
                                               _stream_handle(stream)))
    return out, residual_out


def layernorm(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float,
              out: torch.Tensor | None = None, stream=None):
    """out = LayerNorm(x) * gamma + beta under the rounding contract (no residual)."""
    if not (gamma.is_contiguous() and beta.is_contiguous()):
        raise ValueError("gamma and beta must be contiguous")
    if beta.dtype != gamma.dtype:
        raise ValueError("gamma and beta must share a dtype")
    code = dtypes(x.dtype, gamma.dtype)
    if out is None:
        out = torch.empty(x.shape, dtype=output_dtype(x.dtype, gamma.dtype), device=x.device)
    tokens, hidden = _rows(x)
    if gamma.numel() != hidden or beta.numel() != hidden or out.shape != x.shape:
        raise ValueError("shape mismatch")
    if x.is_contiguous() and out.is_contiguous():
        _check(lib.layernorm(_ptr(x), _ptr(gamma), _ptr(beta), eps, _ptr(out), tokens, hidden, code,
                             _stream_handle(stream)))
    else:
        sx, so = _row_stride(x), _row_stride(out)
        if sx is None or so is None:
            raise ValueError("non-contiguous tensors must be 2-D with contiguous rows")
        _check(lib.layernorm_strided(_ptr(x), sx, _ptr(gamma), _ptr(beta), eps, _ptr(out), so, tokens, hidden, code,
                                     _stream_handle(stream)))
    return out


def plan_ln_for_sms(tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool, sms: int,
                    beta_offset: int = 0) -> dict:
    buf = (ctypes.c_int * 8)()
    _check(lib.far_plan_ln_for_sms(tokens, hidden, dtypes(act, wd), int(residual), beta_offset, sms,
                                   ctypes.addressof(buf)))
    return dict(zip(("kind", "nch", "warps_per_row", "groups", "stages", "grid", "threads", "smem"), list(buf)))


_OUT_CODE = {torch.float16: 1, torch.float32: 0}


def gemm_f16_f32acc(x: torch.Tensor, wt: torch.Tensor, bias: torch.Tensor | None = None,
                    out: torch.Tensor | None = None, out_dtype: torch.dtype = torch.float16, stream=None):
    """y = RNE_f16(RNE_f16(x @ wt^T) + bias) with fp32 products and sums (fp16 storage).

    x [M, K] and wt [N, K] (the transposed weight) fp16, contiguous; bias [N] fp16 or
    None; out_dtype torch.float32 returns the fp32 sums (no bias)."""
    if x.dtype != torch.float16 or wt.dtype != torch.float16 or (bias is not None and bias.dtype != torch.float16):
        raise ValueError("fp16 operands expected")
    if not (x.is_contiguous() and wt.is_contiguous() and (bias is None or bias.is_contiguous())):
        raise ValueError("contiguous operands expected")
    M, K = x.shape
    N, K2 = wt.shape
    if K2 != K or (bias is not None and bias.numel() != N):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    if out.shape != (M, N) or not out.is_contiguous() or out.dtype not in _OUT_CODE:
        raise ValueError("out must be a contiguous [M, N] fp16 or fp32 tensor")
    _check(lib.gemm_f16_f32acc(_ptr(x), _ptr(wt), _ptr(bias), _ptr(out), M, N, K, _OUT_CODE[out.dtype],
                               _stream_handle(stream)))
    return out


def plan_gemm_for_sms(m: int, n: int, k: int, bias: bool, out_dtype: torch.dtype, sms: int) -> dict:
    buf = (ctypes.c_int * 6)()
    _check(lib.far_plan_gemm_for_sms(m, n, k, int(bias), _OUT_CODE[out_dtype], sms, ctypes.addressof(buf)))
    return dict(zip(("kind", "bn", "grid", "threads", "smem", "stages"), list(buf)))


def set_gemm_override(kind: int = -1, bn: int = 0) -> None:
    _check(lib.far_set_gemm_override(kind, bn))


HOST_OP = {"rmsnorm": 0, "layernorm": 1, "quant": 2}


def host_workspace_bytes_op(chunk_tokens: int, hidden: int, act: torch.dtype, wd: torch.dtype, residual: bool,
                            op: str) -> int:
    """Workspace bytes of the host-buffer pipeline for `op` ("rmsnorm", "layernorm", "quant")."""
    n = lib.far_host_workspace_bytes_op(chunk_tokens, hidden, dtypes(act, wd), int(residual), HOST_OP[op])
    if n < 0:
        raise FarError(-n)
    return n


def _wsb(workspace: torch.Tensor) -> int:
    return workspace.numel() * workspace.element_size()


def fused_add_layernorm_host(x, residual, gamma, beta, eps, out, residual_out, workspace, stream=None) -> None:
    """End-to-end LayerNorm on host (ideally pinned) tensors through a device workspace."""
    tokens, hidden = _rows(x)
    _check(lib.fused_add_layernorm_host(_ptr(x), _ptr(residual), _ptr(gamma), _ptr(beta), eps, _ptr(out),
                                        _ptr(residual_out), tokens, hidden, dtypes(x.dtype, gamma.dtype),
                                        _ptr(workspace), _wsb(workspace), _stream_handle(stream)))


def layernorm_host(x, gamma, beta, eps, out, workspace, stream=None) -> None:
    tokens, hidden = _rows(x)
    _check(lib.layernorm_host(_ptr(x), _ptr(gamma), _ptr(beta), eps, _ptr(out), tokens, hidden,
                              dtypes(x.dtype, gamma.dtype), _ptr(workspace), _wsb(workspace), _stream_handle(stream)))


def fused_add_rmsnorm_quant_host(x, residual, weight, eps, qtype, q, scale, residual_out, workspace,
                                 stream=None) -> None:
    tokens, hidden = _rows(x)
    _check(lib.fused_add_rmsnorm_quant_host(_ptr(x), _ptr(residual), _ptr(weight), eps, _ptr(q), _ptr(scale),
                                            _ptr(residual_out), tokens, hidden, dtypes(x.dtype, weight.dtype),
                                            QUANT[qtype], _ptr(workspace), _wsb(workspace), _stream_handle(stream)))


def rmsnorm_quant_host(x, weight, eps, qtype, q, scale, workspace, stream=None) -> None:
    tokens, hidden = _rows(x)
    _check(lib.rmsnorm_quant_host(_ptr(x), _ptr(weight), eps, _ptr(q), _ptr(scale), tokens, hidden,
                                  dtypes(x.dtype, weight.dtype), QUANT[qtype], _ptr(workspace), _wsb(workspace),
                                  _stream_handle(stream)))
