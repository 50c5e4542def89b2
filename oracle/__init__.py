"""CPU oracle for fused residual-add + RMSNorm (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under
``mixed_precision_residual_gb300`` never does: the oracle is the independent
reference that the CUDA path is checked against, and the two share no code.

The arithmetic lives in ``far_oracle.c`` (plain C, binary32 steps as the
contract states them, an exact accumulator for the sum of squares).  This
module compiles it with gcc, loads it with ctypes and splits rows across host
threads; it adds no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "far_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fno-unsafe-math-optimizations"]

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
CODE_DTYPE = {v: k for k, v in DTYPE_CODE.items()}
TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}

_lib = None
_lock = threading.Lock()


def compile_oracle(source: str, target: str) -> str:
    """Compile an oracle source file into a shared library at `target`."""
    os.makedirs(os.path.dirname(target), exist_ok=True)
    tmp = target + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, source, "-o", tmp, "-lm"])
    os.replace(tmp, target)
    return target


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def bind(path: str) -> ctypes.CDLL:
    """Load an oracle shared library and declare its entry points."""
    l = ctypes.CDLL(path)
    vp, f32, i64, i32, u16 = (ctypes.c_void_p, ctypes.c_float, ctypes.c_int64, ctypes.c_int,
                              ctypes.c_uint16)
    l.oracle_fused_add_rmsnorm.argtypes = [vp, vp, vp, f32, vp, vp, i64, i64, i32, i32]
    l.oracle_fused_add_rmsnorm.restype = i32
    l.oracle_rmsnorm.argtypes = [vp, vp, f32, vp, i64, i64, i32, i32]
    l.oracle_rmsnorm.restype = i32
    l.oracle_row_stats.argtypes = [vp, vp, f32, i64, i64, i32, vp, vp, vp]
    l.oracle_row_stats.restype = i32
    l.oracle_exact_sum.argtypes = [vp, i64]
    l.oracle_exact_sum.restype = f32
    l.oracle_output_dtype.argtypes = [i32, i32]
    l.oracle_output_dtype.restype = i32
    l.oracle_f32_to_f16.argtypes = [f32]
    l.oracle_f32_to_f16.restype = u16
    l.oracle_f32_to_bf16.argtypes = [f32]
    l.oracle_f32_to_bf16.restype = u16
    l.oracle_f16_to_f32.argtypes = [u16]
    l.oracle_f16_to_f32.restype = f32
    l.oracle_bf16_to_f32.argtypes = [u16]
    l.oracle_bf16_to_f32.restype = f32
    l.oracle_fused_add_rmsnorm_quant.argtypes = [vp, vp, vp, f32, vp, vp, vp, i64, i64, i32, i32, i32]
    l.oracle_fused_add_rmsnorm_quant.restype = i32
    l.oracle_rmsnorm_quant.argtypes = [vp, vp, f32, vp, vp, i64, i64, i32, i32, i32]
    l.oracle_rmsnorm_quant.restype = i32
    l.oracle_f32_to_e4m3.argtypes = [f32]
    l.oracle_f32_to_e4m3.restype = ctypes.c_uint8
    l.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    l.oracle_e4m3_to_f32.restype = f32
    l.oracle_f32_to_int8.argtypes = [f32]
    l.oracle_f32_to_int8.restype = i32
    l.oracle_fused_add_layernorm.argtypes = [vp, vp, vp, vp, f32, vp, vp, i64, i64, i32, i32]
    l.oracle_fused_add_layernorm.restype = i32
    l.oracle_layernorm.argtypes = [vp, vp, vp, f32, vp, i64, i64, i32, i32]
    l.oracle_layernorm.restype = i32
    l.oracle_ln_row_stats.argtypes = [vp, vp, f32, i64, i64, i32, vp, vp]
    l.oracle_ln_row_stats.restype = i32
    l.oracle_exact_signed_sum.argtypes = [vp, i64]
    l.oracle_exact_signed_sum.restype = f32
    l.oracle_gemm_f16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32]
    l.oracle_gemm_f16.restype = i32
    return l


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def output_dtype(act: str, wd: str, L: ctypes.CDLL | None = None) -> str | None:
    code = (L or lib()).oracle_output_dtype(DTYPE_CODE[act], DTYPE_CODE[wd])
    return None if code < 0 else CODE_DTYPE[code]


def _rows_parallel(fn, tokens: int, threads: int):
    """Run fn(t0, t1) over row blocks on host threads (ctypes releases the GIL)."""
    if tokens == 0:
        return
    threads = max(1, min(threads, tokens))
    if threads == 1:
        fn(0, tokens)
        return
    step = -(-tokens // (threads * 4))
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda t0: fn(t0, min(tokens, t0 + step)), range(0, tokens, step)))


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor, weight: torch.Tensor, eps: float,
                      act: str, wd: str, threads: int | None = None, L: ctypes.CDLL | None = None):
    """Oracle of the fused op on CPU tensors; returns (out, residual_out)."""
    L = L or lib()
    od = output_dtype(act, wd, L)
    if od is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, residual, weight = x.contiguous(), residual.contiguous(), weight.contiguous()
    out = torch.empty((T, H), dtype=TORCH_DTYPE[od])
    res_out = torch.empty((T, H), dtype=TORCH_DTYPE[act])
    sa, so = x.element_size(), out.element_size()

    def work(t0, t1):
        rc = L.oracle_fused_add_rmsnorm(
            x.data_ptr() + t0 * H * sa, residual.data_ptr() + t0 * H * sa, weight.data_ptr(),
            eps, out.data_ptr() + t0 * H * so, res_out.data_ptr() + t0 * H * sa,
            t1 - t0, H, DTYPE_CODE[act], DTYPE_CODE[wd])
        if rc != 0:
            raise RuntimeError(f"oracle_fused_add_rmsnorm returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return out, res_out


def rmsnorm(x: torch.Tensor, weight: torch.Tensor, eps: float, act: str, wd: str,
            threads: int | None = None, L: ctypes.CDLL | None = None):
    """Oracle of the no-residual variant on CPU tensors; returns out."""
    L = L or lib()
    od = output_dtype(act, wd, L)
    if od is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, weight = x.contiguous(), weight.contiguous()
    out = torch.empty((T, H), dtype=TORCH_DTYPE[od])
    sa, so = x.element_size(), out.element_size()

    def work(t0, t1):
        rc = L.oracle_rmsnorm(x.data_ptr() + t0 * H * sa, weight.data_ptr(), eps,
                              out.data_ptr() + t0 * H * so, t1 - t0, H,
                              DTYPE_CODE[act], DTYPE_CODE[wd])
        if rc != 0:
            raise RuntimeError(f"oracle_rmsnorm returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return out


def row_stats(x: torch.Tensor, residual: torch.Tensor | None, eps: float, act: str,
              L: ctypes.CDLL | None = None):
    """Per-row (S, var, rstd) as binary32 numpy arrays."""
    L = L or lib()
    T, H = x.shape
    S = np.empty(T, np.float32)
    var = np.empty(T, np.float32)
    rstd = np.empty(T, np.float32)
    rc = L.oracle_row_stats(x.contiguous().data_ptr(),
                            None if residual is None else residual.contiguous().data_ptr(),
                            eps, T, H, DTYPE_CODE[act], S.ctypes.data, var.ctypes.data,
                            rstd.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_row_stats returned {rc}")
    return S, var, rstd


def exact_sum(values: np.ndarray, L: ctypes.CDLL | None = None) -> np.float32:
    v = np.ascontiguousarray(values, dtype=np.float32)
    return np.float32((L or lib()).oracle_exact_sum(v.ctypes.data, v.size))


QTYPE_CODE = {"int8": 1, "fp8": 2}
Q_TORCH = {"int8": torch.int8, "fp8": torch.uint8}  # fp8 E4M3 codes held as bytes


def fused_add_rmsnorm_quant(x, residual, weight, eps, act, wd, qtype, threads=None, L=None):
    """Oracle of the fused op with a per-token quantised output: (q, scale, residual_out)."""
    L = L or lib()
    if output_dtype(act, wd, L) is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, residual, weight = x.contiguous(), residual.contiguous(), weight.contiguous()
    q = torch.empty((T, H), dtype=Q_TORCH[qtype])
    scale = torch.empty(T, dtype=torch.float32)
    res_out = torch.empty((T, H), dtype=TORCH_DTYPE[act])
    sa = x.element_size()

    def work(t0, t1):
        rc = L.oracle_fused_add_rmsnorm_quant(
            x.data_ptr() + t0 * H * sa, residual.data_ptr() + t0 * H * sa, weight.data_ptr(), eps,
            q.data_ptr() + t0 * H, scale.data_ptr() + t0 * 4, res_out.data_ptr() + t0 * H * sa,
            t1 - t0, H, DTYPE_CODE[act], DTYPE_CODE[wd], QTYPE_CODE[qtype])
        if rc != 0:
            raise RuntimeError(f"oracle_fused_add_rmsnorm_quant returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return q, scale, res_out


def rmsnorm_quant(x, weight, eps, act, wd, qtype, threads=None, L=None):
    """Oracle of the no-residual variant with a per-token quantised output: (q, scale)."""
    L = L or lib()
    if output_dtype(act, wd, L) is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, weight = x.contiguous(), weight.contiguous()
    q = torch.empty((T, H), dtype=Q_TORCH[qtype])
    scale = torch.empty(T, dtype=torch.float32)
    sa = x.element_size()

    def work(t0, t1):
        rc = L.oracle_rmsnorm_quant(x.data_ptr() + t0 * H * sa, weight.data_ptr(), eps, q.data_ptr() + t0 * H,
                                    scale.data_ptr() + t0 * 4, t1 - t0, H, DTYPE_CODE[act], DTYPE_CODE[wd],
                                    QTYPE_CODE[qtype])
        if rc != 0:
            raise RuntimeError(f"oracle_rmsnorm_quant returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return q, scale


def fused_add_layernorm(x, residual, gamma, beta, eps, act, wd, threads=None, L=None):
    """Oracle of fused residual-add + LayerNorm on CPU tensors: (out, residual_out)."""
    L = L or lib()
    od = output_dtype(act, wd, L)
    if od is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, residual, gamma, beta = x.contiguous(), residual.contiguous(), gamma.contiguous(), beta.contiguous()
    out = torch.empty((T, H), dtype=TORCH_DTYPE[od])
    res_out = torch.empty((T, H), dtype=TORCH_DTYPE[act])
    sa, so = x.element_size(), out.element_size()

    def work(t0, t1):
        rc = L.oracle_fused_add_layernorm(x.data_ptr() + t0 * H * sa, residual.data_ptr() + t0 * H * sa,
                                          gamma.data_ptr(), beta.data_ptr(), eps, out.data_ptr() + t0 * H * so,
                                          res_out.data_ptr() + t0 * H * sa, t1 - t0, H, DTYPE_CODE[act],
                                          DTYPE_CODE[wd])
        if rc != 0:
            raise RuntimeError(f"oracle_fused_add_layernorm returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return out, res_out


def layernorm(x, gamma, beta, eps, act, wd, threads=None, L=None):
    """Oracle of LayerNorm without a residual on CPU tensors: out."""
    L = L or lib()
    od = output_dtype(act, wd, L)
    if od is None:
        raise ValueError(f"dtype pair ({act}, {wd}) is rejected by the dtype policy")
    T, H = x.shape
    x, gamma, beta = x.contiguous(), gamma.contiguous(), beta.contiguous()
    out = torch.empty((T, H), dtype=TORCH_DTYPE[od])
    sa, so = x.element_size(), out.element_size()

    def work(t0, t1):
        rc = L.oracle_layernorm(x.data_ptr() + t0 * H * sa, gamma.data_ptr(), beta.data_ptr(), eps,
                                out.data_ptr() + t0 * H * so, t1 - t0, H, DTYPE_CODE[act], DTYPE_CODE[wd])
        if rc != 0:
            raise RuntimeError(f"oracle_layernorm returned {rc}")

    _rows_parallel(work, T, threads or default_threads())
    return out


def ln_row_stats(x, residual, eps, act, L=None):
    """Per-row (mean, rstd) of the fused LayerNorm as binary32 numpy arrays."""
    L = L or lib()
    T, H = x.shape
    mean = np.empty(T, np.float32)
    rstd = np.empty(T, np.float32)
    rc = L.oracle_ln_row_stats(x.contiguous().data_ptr(),
                               None if residual is None else residual.contiguous().data_ptr(), eps, T, H,
                               DTYPE_CODE[act], mean.ctypes.data, rstd.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"oracle_ln_row_stats returned {rc}")
    return mean, rstd


def exact_signed_sum(values, L=None):
    v = np.ascontiguousarray(values, dtype=np.float32)
    return np.float32((L or lib()).oracle_exact_signed_sum(v.ctypes.data, v.size))


def gemm_f16(x, wt, bias=None, out_dtype="f16", threads=None, L=None):
    """Oracle of the fp16-storage / fp32-compute GEMM on CPU tensors.

    x [M, K] and wt [N, K] fp16 (the transposed weight, row-major), bias [N] fp16 or
    None.  out_dtype "f16": RNE_f16(RNE_f16(exact x @ wt^T) + bias); "f32": the exact
    sum rounded once to binary32 (no bias)."""
    L = L or lib()
    if x.dtype != torch.float16 or wt.dtype != torch.float16 or (bias is not None and bias.dtype != torch.float16):
        raise ValueError("the GEMM oracle takes fp16 operands")
    if out_dtype == "f32" and bias is not None:
        raise ValueError("the fp32 output takes no bias")
    M, K = x.shape
    N, K2 = wt.shape
    if K != K2 or (bias is not None and bias.numel() != N):
        raise ValueError("shape mismatch")
    x, wt = x.contiguous(), wt.contiguous()
    bias = None if bias is None else bias.contiguous()
    out = torch.empty((M, N), dtype=TORCH_DTYPE[out_dtype])
    so = out.element_size()

    def work(t0, t1):
        rc = L.oracle_gemm_f16(x.data_ptr() + t0 * K * 2, wt.data_ptr(), None if bias is None else bias.data_ptr(),
                               out.data_ptr() + t0 * N * so, t1 - t0, N, K, DTYPE_CODE[out_dtype])
        if rc != 0:
            raise RuntimeError(f"oracle_gemm_f16 returned {rc}")

    _rows_parallel(work, M, threads or default_threads())
    return out
