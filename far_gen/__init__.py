"""Seeded synthetic inputs for fused residual-add + RMSNorm.

Random-number generation only: the normalisation itself is computed elsewhere
(the CUDA library and, independently, the CPU oracle); this module feeds both
the same bytes.  Values come from a counter-based generator (Philox4x32-10,
Box-Muller normals, see ``gen.c``) so any row range of any workload can be
produced alone and the result does not depend on the thread count.

The workloads follow the shapes the case study "Aligning fused RMSNorm rounding
across vLLM backends" (section "Testing the contract") tests: bf16 and fp16,
token counts 8 and 512, hidden sizes 2048 and 8192, with non-uniform rows so
that normalisation cannot cancel a rounding error, plus three larger ones.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_build", "libfargen.so")

# stream ids: one independent random sequence per role
STREAM_X, STREAM_R, STREAM_W, STREAM_SCALE, STREAM_OUTLIER, STREAM_SIGN, STREAM_BETA = 1, 2, 3, 4, 5, 6, 7
STREAM_GEMM_X, STREAM_GEMM_W, STREAM_GEMM_BIAS = 8, 9, 10

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: dtypes, shape, eps and the value recipe."""

    name: str
    act: str  # dtype of x, residual and residual_out: "f16" | "bf16" | "f32"
    wd: str  # dtype of the weight
    tokens: int
    hidden: int
    eps: float
    recipe: str  # "rowscale" | "outliers"
    scale_lo: float = 0.1
    scale_hi: float = 10.0
    r_sd: float = 1.0
    outlier_p: float = 0.0
    outlier_value: float = 0.0
    note: str = ""
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "c1": Workload("c1", "bf16", "bf16", 8, 2048, 1e-6, "rowscale", 0.1, 10.0,
                   note="bf16 8x2048: per-row log-uniform scale in [0.1, 10]"),
    "c2": Workload("c2", "f16", "f16", 512, 8192, 1e-6, "rowscale", 0.1, 10.0,
                   note="fp16 512x8192: per-row log-uniform scale in [0.1, 10]"),
    "c3": Workload("c3", "bf16", "f32", 4096, 4096, 1e-5, "outliers", r_sd=2.0,
                   outlier_p=1e-3, outlier_value=200.0,
                   note="bf16 activations, fp32 weight (fp32 out) 4096x4096: "
                        "x~N(0,1), r~N(0,4) with 0.1% outliers at +-200"),
    "c4": Workload("c4", "bf16", "bf16", 16384, 5120, 1e-6, "rowscale", 0.01, 100.0,
                   note="bf16 16384x5120: per-row log-uniform scale in [0.01, 100]"),
    "c5": Workload("c5", "f16", "f16", 65536, 8192, 1e-6, "rowscale", 0.1, 10.0,
                   note="fp16 65536x8192: per-row log-uniform scale in [0.1, 10], |x+r| < 60000"),
}

# Largest |Z| Box-Muller can return here: u1 >= 0.5 / 2^32, so |Z| <= sqrt(-2 ln u1).
MAX_ABS_NORMAL = math.sqrt(-2.0 * math.log(0.5 / 4294967296.0))

_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile gen.c into an in-tree shared library (gcc, no GPU needed)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lib_lock:
        if _lib is None:
            build()
            l = ctypes.CDLL(_LIB)
            i64, u64, u32, dbl, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                      ctypes.c_double, ctypes.c_void_p)
            l.fargen_normal_f32.argtypes = [u64, u32, i64, i64, dbl, dbl, vp]
            l.fargen_rows_f32.argtypes = [u64, u32, i64, i64, i64, vp, dbl, vp]
            l.fargen_uniform_f64.argtypes = [u64, u32, i64, i64, vp]
            l.fargen_uniform_at_f64.argtypes = [u64, u32, vp, i64, vp]
            l.fargen_philox_block.argtypes = [u64, u32, u64, vp]
            l.fargen_philox_raw.argtypes = [vp, vp, vp]
            for f in (l.fargen_normal_f32, l.fargen_rows_f32, l.fargen_uniform_f64,
                      l.fargen_uniform_at_f64,
                      l.fargen_philox_block, l.fargen_philox_raw):
                f.restype = None
            _lib = l
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def normal(seed: int, stream: int, start: int, n: int, mean: float = 0.0, sd: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().fargen_normal_f32(seed, stream, start, n, mean, sd, _ptr(out))
    return out


def uniform(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    lib().fargen_uniform_f64(seed, stream, start, n, _ptr(out))
    return out


def row_scales(w: Workload, seed: int, row0: int, rows: int) -> np.ndarray:
    """Per-row scale shared by x and r: exp(U(ln lo, ln hi)), in binary64."""
    if w.recipe != "rowscale":
        return np.ones(rows, dtype=np.float64)
    u = uniform(seed, STREAM_SCALE, row0, rows)
    lo, hi = math.log(w.scale_lo), math.log(w.scale_hi)
    return np.exp(lo + (hi - lo) * u)


def _fill_rows(seed, stream, row0, rows, hidden, scales, sd, out_f32):
    lib().fargen_rows_f32(seed, stream, row0, rows, hidden, _ptr(scales), sd, _ptr(out_f32))


def _default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _matrix(w: Workload, seed: int, stream: int, row0: int, rows: int, sd: float,
            scales: np.ndarray, dtype: torch.dtype, threads: int) -> torch.Tensor:
    """rows x hidden tensor of sd * scale[t] * Z, rounded once from binary32 to `dtype`."""
    H = w.hidden
    out = torch.empty((rows, H), dtype=dtype)
    if rows == 0:
        return out
    # at most ~16 MB of binary32 per chunk, and several chunks per thread
    chunk = max(1, min((1 << 22) // max(1, H), -(-rows // (4 * threads))))

    def work(c0):
        c1 = min(rows, c0 + chunk)
        tmp = np.empty((c1 - c0, H), dtype=np.float32)
        _fill_rows(seed, stream, row0 + c0, c1 - c0, H, np.ascontiguousarray(scales[c0:c1]), sd, tmp)
        out[c0:c1].copy_(torch.from_numpy(tmp))  # one RNE rounding binary32 -> dtype

    starts = list(range(0, rows, chunk))
    if threads <= 1 or len(starts) == 1:
        for c0 in starts:
            work(c0)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, starts))
    return out


def uniform_at(seed: int, stream: int, idx: np.ndarray) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(idx.size, dtype=np.float64)
    lib().fargen_uniform_at_f64(seed, stream, _ptr(idx), idx.size, _ptr(out))
    return out


def _apply_outliers(w: Workload, seed: int, row0: int, r: torch.Tensor, threads: int) -> None:
    """Replace each element of r, independently with probability p, by +-value (fair sign)."""
    rows, H = r.shape
    start = row0 * H
    n = rows * H
    step = 1 << 22

    def hits(c0):
        u = uniform(seed, STREAM_OUTLIER, start + c0, min(step, n - c0))
        return np.nonzero(u < w.outlier_p)[0] + c0

    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        parts = list(ex.map(hits, range(0, n, step)))
    hit = np.concatenate(parts) if parts else np.zeros(0, np.int64)
    if hit.size == 0:
        return
    sign_u = uniform_at(seed, STREAM_SIGN, hit + start)
    vals = np.where(sign_u < 0.5, -w.outlier_value, w.outlier_value).astype(np.float32)
    flat = r.view(-1)
    flat[torch.from_numpy(hit)] = torch.from_numpy(vals).to(r.dtype)


def make_inputs(w: Workload | str, seed: int = 0, row0: int = 0, rows: int | None = None,
                threads: int | None = None) -> dict:
    """Inputs of workload `w` for rows [row0, row0 + rows): x, residual (r) and weight (w).

    Returns CPU tensors in the workload's storage dtypes plus the scalar
    parameters.  Any row range reproduces the same rows of the full matrices.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if rows is None:
        rows = w.tokens - row0
    threads = threads or _default_threads()
    act = TORCH_DTYPE[w.act]
    scales = row_scales(w, seed, row0, rows)
    x = _matrix(w, seed, STREAM_X, row0, rows, 1.0, scales, act, threads)
    r = _matrix(w, seed, STREAM_R, row0, rows, w.r_sd, scales, act, threads)
    if w.recipe == "outliers":
        _apply_outliers(w, seed, row0, r, threads)
    # The clip |x + r| < 60000 of the fp16 roofline workload never binds: |Z| is
    # bounded by MAX_ABS_NORMAL, so |x + r| <= 2 * scale_hi * MAX_ABS_NORMAL (+ rounding).
    weight = torch.from_numpy(normal(seed, STREAM_W, 0, w.hidden, 1.0, 0.1)).to(TORCH_DTYPE[w.wd])
    return {"x": x, "r": r, "w": weight, "eps": w.eps, "act": w.act, "wd": w.wd,
            "tokens": rows, "hidden": w.hidden, "row0": row0, "workload": w.name}


def custom_inputs(act: str, wd: str, tokens: int, hidden: int, seed: int = 0,
                  scale_lo: float = 0.1, scale_hi: float = 10.0, eps: float = 1e-6) -> dict:
    """Inputs for an arbitrary shape/dtype pair with the row-scale recipe (used by parity sweeps)."""
    w = Workload(f"custom_{act}_{wd}_{tokens}x{hidden}", act, wd, tokens, hidden, eps,
                 "rowscale", scale_lo, scale_hi)
    return make_inputs(w, seed)


def ln_beta(d: dict, seed: int = 0, sd: float = 0.1) -> torch.Tensor:
    """A LayerNorm shift for inputs `d`: [hidden] in the weight dtype, N(0, sd^2)."""
    return torch.from_numpy(normal(seed, STREAM_BETA, 0, d["hidden"], 0.0, sd)).to(d["w"].dtype)


def gemm_inputs(M: int, N: int, K: int, seed: int = 0, bias: bool = True) -> dict:
    """Operands of the fp16 GEMM: x [M, K] ~ N(0, 1), the transposed weight wt [N, K]
    ~ N(0, 1/K) (so each output is about N(0, 1)), bias [N] ~ N(0, 0.1^2); fp16 CPU
    tensors (each value drawn in binary64, rounded to binary32, then to fp16)."""
    x = torch.from_numpy(normal(seed, STREAM_GEMM_X, 0, M * K, 0.0, 1.0)).reshape(M, K).to(torch.float16)
    wt = torch.from_numpy(normal(seed, STREAM_GEMM_W, 0, N * K, 0.0, 1.0 / math.sqrt(max(K, 1))))
    wt = wt.reshape(N, K).to(torch.float16)
    b = torch.from_numpy(normal(seed, STREAM_GEMM_BIAS, 0, N, 0.0, 0.1)).to(torch.float16) if bias else None
    return {"x": x, "wt": wt, "bias": b, "M": M, "N": N, "K": K}


def gemm_dyadic_inputs(M: int, N: int, K: int, seed: int = 0) -> dict:
    """GEMM operands on a dyadic grid: x, wt in {k/8 : -8 <= k <= 8}, bias in {k/16 : -16
    <= k <= 16}.  Every product is a multiple of 2^-6 of magnitude <= 1, so every partial
    sum of up to 2^18 products (at most 2^18 in magnitude, on a 2^-6 grid: 24 bits) is
    exact in binary32 whatever the order of the additions."""
    def grid(stream, n, half, scale):
        u = uniform(seed, stream, 0, n)
        return torch.from_numpy((np.floor(u * (2 * half + 1)) - half) / scale).to(torch.float16)

    x = grid(STREAM_GEMM_X, M * K, 8, 8.0).reshape(M, K)
    wt = grid(STREAM_GEMM_W, N * K, 8, 8.0).reshape(N, K)
    b = grid(STREAM_GEMM_BIAS, N, 16, 16.0)
    return {"x": x, "wt": wt, "bias": b, "M": M, "N": N, "K": K}
