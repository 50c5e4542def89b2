"""The fp16-storage / fp32-compute GEMM against the oracle, through the C ABI.

Gates (the Luminal page "Luminal FP16 Backend Repair and H100 Evidence", section
"Validation and Experimental Design", and the fp32 accumulation the page specifies).
With E = K * 2^-22 * sum_k |x w|, a bound on the error of binary32 sums of K exact
products in any order (rounded or truncated additions):
- random operands, fp16 output: the page's |y - ref| <= 2e-4 + 2e-3 |ref| everywhere;
  |y - ref| <= 2 ulp16(ref) + E everywhere (ref = RNE_f16 of the exact sum, y the cast of
  a binary32 sum within E of it); the same non-finite pattern.  With the bias, 2 ulp16 of
  the cast value more.  fp32 output: |out - ref| <= E + ulp32.
- dyadic operands (every partial sum exact in binary32 in any order): bit for bit equal
  to the oracle, fp16 with and without bias and fp32.
(Neither one fp16 ULP everywhere nor a fixed share of differing elements is implied by
fp32 compute: near zero the fp16 spacing is finer than the accumulation error, and the
share of sums that cross an fp16 rounding boundary grows with K.)
Outputs sit between canary bands that must survive every call.
"""
import numpy as np
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import Guarded, to_device
from oracle_pins import ulp_distance

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    far.set_gemm_override()
    return far


def run_gemm(far, d, bias=True, out_dtype=torch.float16, offsets=(0, 0, 0, 0)):
    """One call through the C ABI on guarded device buffers; the CPU result."""
    x = to_device(d["x"], offsets[0])
    wt = to_device(d["wt"], offsets[1])
    b = to_device(d["bias"], offsets[2]) if bias and d["bias"] is not None else None
    M, N, K = d["M"], d["N"], d["K"]
    out = Guarded((M, N), out_dtype, offsets[3])
    st = far.lib.gemm_f16_f32acc(x.t.data_ptr(), wt.t.data_ptr(), None if b is None else b.t.data_ptr(),
                                 out.t.data_ptr(), M, N, K, 1 if out_dtype == torch.float16 else 0,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 0, far.lib.far_status_string(st)
    assert far.device_status() == 0
    assert out.guards_intact(), "a store landed outside the output"
    return out.t.cpu()


def f16_ulp(v: torch.Tensor) -> np.ndarray:
    """The fp16 spacing at |v| (the subnormal spacing 2^-24 at the bottom)."""
    a = np.abs(v.float().numpy()).astype(np.float64)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def accumulation_bound(d) -> np.ndarray:
    absprod = d["x"].double().abs() @ d["wt"].double().abs().T
    return max(d["K"], 1) * 2.0 ** -22 * absprod.numpy()


def gate_f16(got, ref, d, where, p_ref=None):
    """The fp16 gates above; p_ref (the oracle's cast value) when a bias was added."""
    g, r = got.double().numpy(), ref.double().numpy()
    nan_g, nan_r = np.isnan(g), np.isnan(r)
    assert (nan_g == nan_r).all(), f"{where}: NaN pattern differs"
    inf_r = np.isinf(r)
    assert (g[inf_r] == r[inf_r]).all() and not np.isinf(g[~inf_r & ~nan_r]).any(), f"{where}: infinities differ"
    fin = np.isfinite(r)
    err = np.abs(g[fin] - r[fin])
    # The page's tolerance. With a bias, the unbiased value p is cast to fp16 first, and any
    # order of the binary32 additions may leave p one fp16 step from the oracle's p_ref; the
    # bias add keeps that step in absolute terms while it can cancel |y| towards zero, where
    # a relative tolerance cannot absorb it. So the biased output gets that one step of p_ref
    # on top (the unbiased output is held to the page's tolerance alone).
    page = 2e-4 + 2e-3 * np.abs(r[fin])
    if p_ref is not None:
        page = page + f16_ulp(p_ref)[fin]
    assert (err <= page).all(), f"{where}: the page's tolerance fails"
    bound = 2 * f16_ulp(ref) + accumulation_bound(d)
    if p_ref is not None:
        bound = bound + 2 * f16_ulp(p_ref)
    assert (err <= bound[fin]).all(), f"{where}: beyond the accumulation bound"
    u = ulp_distance(got, ref)
    return int(u.max(initial=0)), float((u > 0).mean())


def gate_f32(got, ref, d, where):
    bound = accumulation_bound(d) + np.abs(ref.double().numpy()) * 2.0 ** -23
    err = np.abs(got.double().numpy() - ref.double().numpy())
    fin = np.isfinite(ref.numpy())
    assert (err[fin] <= bound[fin] + 1e-45).all(), f"{where}: fp32 sums beyond the accumulation bound"


def check_all(far, d, where, offsets=(0, 0, 0, 0)):
    p = run_gemm(far, d, bias=False, offsets=offsets)
    p_ref = oracle.gemm_f16(d["x"], d["wt"], None, "f16")
    gate_f16(p, p_ref, d, f"{where} fp16")
    if d["bias"] is not None:
        y = run_gemm(far, d, bias=True, offsets=offsets)
        y_ref = oracle.gemm_f16(d["x"], d["wt"], d["bias"], "f16")
        gate_f16(y, y_ref, d, f"{where} fp16 + bias", p_ref=p_ref)
    o = run_gemm(far, d, bias=False, out_dtype=torch.float32, offsets=offsets)
    gate_f32(o, oracle.gemm_f16(d["x"], d["wt"], None, "f32"), d, f"{where} fp32")


def test_page_shape(far):
    """The page's H100 shape, M = N = 1024, K = 768."""
    check_all(far, far_gen.gemm_inputs(1024, 1024, 768, seed=1), "1024x1024x768")


def force(far, bn):
    """The plan under test: a single-CTA tile width, "pair" (256 x 256 over CTA pairs) or "plain"."""
    if bn == "pair":
        far.set_gemm_override(2, 0)
    elif bn == "plain":
        far.set_gemm_override(1, 0)
    else:
        far.set_gemm_override(0, bn)


@pytest.mark.parametrize("bn", [64, 128, 256, "pair"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 200, 136), (257, 520, 1000), (1, 8, 8), (128, 64, 4096),
                                   (768, 768, 512)])
def test_tiles_and_tails(far, bn, M, N, K):
    """Every tile width on full tiles and ragged tails in M, N and K, a single row and
    a long K (the slice ring wraps many times); several tiles per CTA."""
    d = far_gen.gemm_inputs(M, N, K, seed=M + N + K)
    try:
        force(far, bn)
        check_all(far, d, f"bn={bn} {M}x{N}x{K}")
    finally:
        far.set_gemm_override()


@pytest.mark.parametrize("M,N,K", [(64, 12, 64), (33, 40, 7), (5, 3, 1), (16, 16, 0)])
def test_plain_kernel_shapes(far, M, N, K):
    """Shapes the tensor-core path does not take (n or k not a multiple of 8, k = 0)."""
    d = far_gen.gemm_inputs(M, N, K, seed=7)
    assert far.plan_gemm_for_sms(M, N, K, True, torch.float16, 152)["kind"] == 1
    check_all(far, d, f"plain {M}x{N}x{K}")


def test_plain_kernel_forced(far):
    d = far_gen.gemm_inputs(200, 136, 320, seed=11)
    try:
        far.set_gemm_override(1, 0)
        check_all(far, d, "plain forced")
    finally:
        far.set_gemm_override()


def test_misaligned_operands(far):
    """An fp16 offset on any operand rules out TMA: the plain kernel must run and match."""
    d = far_gen.gemm_inputs(96, 64, 128, seed=5)
    for offs in [(1, 0, 0, 0), (0, 1, 0, 0), (0, 0, 1, 0), (0, 0, 0, 1)]:
        check_all(far, d, f"offsets {offs}", offsets=offs)


def test_product_accumulation_fixture(far):
    """The page's fixture that rejects fp16-rounded products: pairs (1 + e)^2 and
    -(1 + 2e) * 1, e = 2^-10, leave e^2 each; K = 768 gives 384 * 2^-20 exactly."""
    K, e = 768, 2.0 ** -10
    x = torch.tensor([1 + e if k % 2 == 0 else -(1 + 2 * e) for k in range(K)], dtype=torch.float64)
    w = torch.tensor([1 + e if k % 2 == 0 else 1.0 for k in range(K)], dtype=torch.float64)
    d = {"x": x.to(torch.float16).repeat(128, 1), "wt": w.to(torch.float16).repeat(64, 1), "bias": None,
         "M": 128, "N": 64, "K": K}
    p = run_gemm(far, d, bias=False)
    want = (K // 2) * 2.0 ** -20
    assert np.all(np.abs(p.double().numpy() - want) <= 2e-4 + 2e-3 * want), "products were not kept in fp32"
    gate_f16(p, oracle.gemm_f16(d["x"], d["wt"], None, "f16"), d, "product fixture")


def test_special_values(far):
    """Overflow to infinity at the cast, infinity and NaN propagation."""
    d = far_gen.gemm_inputs(128, 64, 64, seed=3)
    x = d["x"].clone()
    x[0, :] = 60000.0                 # sums far above the fp16 range -> +-inf
    x[1, 3] = float("inf")
    x[2, 5] = float("nan")
    d = dict(d, x=x)
    p = run_gemm(far, d, bias=False)
    gate_f16(p, oracle.gemm_f16(d["x"], d["wt"], None, "f16"), d, "special values")


def test_binding_and_rejections(far):
    d = far_gen.gemm_inputs(256, 128, 192, seed=2)
    y = far.gemm_f16_f32acc(d["x"].cuda(), d["wt"].cuda(), d["bias"].cuda())
    gate_f16(y.cpu(), oracle.gemm_f16(d["x"], d["wt"], d["bias"], "f16"), d, "binding",
             p_ref=oracle.gemm_f16(d["x"], d["wt"], None, "f16"))
    x = d["x"].cuda()
    out = torch.empty((256, 128), dtype=torch.float16, device="cuda")
    st = far.lib.gemm_f16_f32acc(x.data_ptr(), x.data_ptr(), None, x.data_ptr(), 256, 128, 192, 1,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == 5  # out over x
    assert far.device_status() == 0
    del out


def check_exact(far, d, where):
    for bias, dt in ((False, torch.float16), (True, torch.float16), (False, torch.float32)):
        got = run_gemm(far, d, bias=bias, out_dtype=dt)
        ref = oracle.gemm_f16(d["x"], d["wt"], d["bias"] if bias else None, "f16" if dt == torch.float16 else "f32")
        ib = torch.int16 if dt == torch.float16 else torch.int32
        assert torch.equal(got.view(ib), ref.view(ib)), f"{where} bias={bias} {dt}: not bit for bit"


@pytest.mark.parametrize("bn", [64, 128, 256, "pair", "plain"])
@pytest.mark.parametrize("M,N,K", [(1024, 1024, 768), (300, 200, 136), (257, 520, 1000), (129, 72, 8),
                                   (2048, 1536, 256)])
def test_dyadic_bit_exact(far, bn, M, N, K):
    """Exact sums: the cast, the bias after the cast, the indexing and every tail bit for bit."""
    d = far_gen.gemm_dyadic_inputs(M, N, K, seed=M * 7 + K)
    try:
        force(far, bn)
        check_exact(far, d, f"dyadic bn={bn} {M}x{N}x{K}")
    finally:
        far.set_gemm_override()


def test_bias_after_cast_fixture(far):
    """x . w = 1 + 2^-11 exactly (an fp16 tie: the cast gives 1), bias 2^-11: the contract
    gives RNE_f16(1 + 2^-11) = 1, adding the bias before the cast would give 1 + 2^-10."""
    K = 64
    x = torch.zeros((128, K), dtype=torch.float16)
    x[:, 0], x[:, 1] = 1.0, 2.0 ** -11
    wt = torch.zeros((64, K), dtype=torch.float16)
    wt[:, 0], wt[:, 1] = 1.0, 1.0
    d = {"x": x, "wt": wt, "bias": torch.full((64,), 2.0 ** -11, dtype=torch.float16), "M": 128, "N": 64, "K": K}
    y = run_gemm(far, d, bias=True)
    assert bool((y == 1.0).all()), "the bias must be added after the fp16 cast"


def test_default_plan_uses_pairs_when_tiles_abound(far):
    """A large GEMM takes the CTA-pair path by default (the device holds pairs) and matches."""
    assert far.plan_gemm_for_sms(4096, 4096, 512, True, torch.float16, 152)["kind"] == 2
    d = far_gen.gemm_dyadic_inputs(4096, 4096, 512, seed=9)
    check_exact(far, d, "default plan 4096x4096x512")


def test_last_wave_in_whole_tiles(far):
    """A last wave of tiles for more than half the pairs runs as whole 256 x 256 tiles (two
    rounds of half tiles would take longer): 2048 x 2048 (64 tiles, one round) bit for bit
    on dyadic operands and within the gates on random ones; 3072 x 3072 (a full wave, then
    68 tiles) on sampled rows of every tile band."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert far.plan_gemm_for_sms(2048, 2048, 256, True, torch.float16, sms)["kind"] == 2
    check_exact(far, far_gen.gemm_dyadic_inputs(2048, 2048, 256, seed=12), "dyadic 2048x2048x256 last wave whole")
    check_all(far, far_gen.gemm_inputs(2048, 2048, 256, seed=13), "2048x2048x256 last wave whole")
    M = N = 3072
    K = 512
    assert far.plan_gemm_for_sms(M, N, K, True, torch.float16, sms)["kind"] == 2
    rows = sorted({r for band in range(0, M, 256) for r in (band, band + 129)} | {M - 1})
    d = far_gen.gemm_dyadic_inputs(M, N, K, seed=14)
    got = run_gemm(far, d, bias=True)
    ref = oracle.gemm_f16(d["x"][rows], d["wt"], d["bias"], "f16")
    assert torch.equal(got[rows].view(torch.int16), ref.view(torch.int16))
