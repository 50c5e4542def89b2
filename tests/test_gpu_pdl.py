"""Programmatic dependent launch: each normalisation kernel may be dispatched while the
kernel ahead of it on the stream finishes, and waits for that kernel's completion before
it touches global memory.  A chain of launches in which every launch reads the previous
launch's output must therefore give the same bits as the same chain launched plainly
(a launch that read its input before the previous kernel finished writing it would see
stale or partly written rows).  Staged and generic kernels, every op family, and a
launch that follows a kernel of another library (torch's fill) are covered."""
import pytest
import torch

import far_gen
import oracle
from gpu_helpers import gate
from oracle_pins import bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    far.set_launch_override()
    assert far.get_programmatic_launch(), "programmatic launches are the default"
    yield far
    far.set_programmatic_launch(True)


def _chain(far, x0, r, w, b, eps, links, offset=0):
    """links launches, each on the previous one's output: fused RMSNorm, RMSNorm, fused
    LayerNorm, LayerNorm, in turn; every output buffer starts as NaN, written right before
    (torch's fill on the same stream is the kernel ahead of the first link)."""
    outs = []
    x = x0
    for i in range(links):
        n = x.numel() + offset
        buf = torch.full((n,), float("nan"), dtype=x.dtype, device="cuda")
        out = buf[offset:].view(x.shape)
        res = torch.full(x.shape, float("nan"), dtype=x.dtype, device="cuda")
        k = i % 4
        if k == 0:
            far.fused_add_rmsnorm(x, r, w, eps, out=out, residual_out=res)
        elif k == 1:
            far.rmsnorm(x, w, eps, out=out)
        elif k == 2:
            far.fused_add_layernorm(x, r, w, b, eps, out=out, residual_out=res)
        else:
            far.layernorm(x, w, b, eps, out=out)
        outs.append(out)
        x = out
    torch.cuda.synchronize()
    assert far.device_status() == 0
    return [o.cpu() for o in outs]


@pytest.mark.parametrize("act,tokens,hidden,offset", [("bf16", 4096, 4096, 0), ("f16", 16384, 2048, 0),
                                                      ("bf16", 300, 5120, 0), ("f16", 1000, 1000, 1)])
def test_chain_of_dependent_launches(far, act, tokens, hidden, offset):
    """Every launch reads what the one before it wrote (offset 1: misaligned outputs, so the
    generic kernel runs from the second link on)."""
    d = far_gen.custom_inputs(act, act, tokens, hidden, seed=tokens + hidden)
    b = far_gen.ln_beta(d)
    x, r, w, bb = d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), b.cuda()
    try:
        far.set_programmatic_launch(False)
        ref = _chain(far, x, r, w, bb, d["eps"], 12, offset)
        far.set_programmatic_launch(True)
        for _ in range(3):
            got = _chain(far, x, r, w, bb, d["eps"], 12, offset)
            for i, (a, e) in enumerate(zip(got, ref)):
                assert bits_equal(a, e), f"link {i} differs under programmatic launch"
    finally:
        far.set_programmatic_launch(True)
    assert not any(torch.isnan(o.float()).all() for o in ref)


def test_first_links_against_the_oracle(far):
    """The first two links of a chain (fused RMSNorm, then RMSNorm of its output) against
    the oracle."""
    d = far_gen.custom_inputs("bf16", "bf16", 2048, 4096, seed=5)
    b = far_gen.ln_beta(d)
    outs = _chain(far, d["x"].cuda(), d["r"].cuda(), d["w"].cuda(), b.cuda(), d["eps"], 2)
    ro, _ = oracle.fused_add_rmsnorm(d["x"], d["r"], d["w"], d["eps"], "bf16", "bf16")
    gate(outs[0], ro, where="link 0")
    gate(outs[1], oracle.rmsnorm(outs[0], d["w"], d["eps"], "bf16", "bf16"), where="link 1")


def test_hook(far):
    assert far.lib.far_set_programmatic_launch(2) == 4
    assert far.lib.far_set_programmatic_launch(-1) == 4
    assert far.get_programmatic_launch()
