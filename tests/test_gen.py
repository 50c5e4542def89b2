"""The seeded input generator: published test vectors, reproducibility, recipes."""
import math

import numpy as np
import pytest
import torch

import far_gen


def test_philox_known_answers():
    """Philox4x32-10 test vectors published with the algorithm (Salmon et al., SC'11)."""
    L = far_gen.lib()
    out = np.zeros(4, np.uint32)
    vectors = [
        ([0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
        ([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
        ([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
         [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
    ]
    for ctr, key, want in vectors:
        c, k = np.array(ctr, np.uint32), np.array(key, np.uint32)
        L.fargen_philox_raw(c.ctypes.data, k.ctypes.data, out.ctypes.data)
        assert out.tolist() == want


def test_row_ranges_reproduce_full_matrices():
    full = far_gen.make_inputs("c3", rows=64)
    part = far_gen.make_inputs("c3", row0=20, rows=7, threads=3)
    assert torch.equal(part["x"], full["x"][20:27])
    assert torch.equal(part["r"], full["r"][20:27])
    assert torch.equal(part["w"], full["w"])


def test_thread_count_does_not_change_values():
    a = far_gen.make_inputs("c4", rows=40, threads=1)
    b = far_gen.make_inputs("c4", rows=40, threads=6)
    assert torch.equal(a["x"], b["x"]) and torch.equal(a["r"], b["r"])


def test_normal_moments():
    z = far_gen.normal(0, 9, 0, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs(np.mean(z ** 4) - 3.0) < 0.05  # Gaussian kurtosis
    assert np.abs(z).max() <= far_gen.MAX_ABS_NORMAL


def test_recipes():
    for name, w in far_gen.WORKLOADS.items():
        d = far_gen.make_inputs(name, rows=min(w.tokens, 64))
        assert d["x"].dtype == far_gen.TORCH_DTYPE[w.act] and d["w"].dtype == far_gen.TORCH_DTYPE[w.wd]
        assert d["x"].shape == (min(w.tokens, 64), w.hidden)
        wv = d["w"].double()
        assert abs(wv.mean().item() - 1.0) < 0.02 and abs(wv.std().item() - 0.1) < 0.01
        if w.recipe == "rowscale":
            s = far_gen.row_scales(w, 0, 0, 4096)
            assert s.min() >= w.scale_lo and s.max() <= w.scale_hi
            # log-uniform: log-scale mean at the centre of [ln lo, ln hi]
            assert abs(np.log(s).mean() - 0.5 * (math.log(w.scale_lo) + math.log(w.scale_hi))) < 0.1
            # x and r share the row scale: their row RMS ratio is ~1
            ratio = d["x"].double().pow(2).mean(1).sqrt() / d["r"].double().pow(2).mean(1).sqrt()
            assert (ratio - 1).abs().max() < 0.1


def test_outlier_recipe():
    d = far_gen.make_inputs("c3", rows=512)
    r = d["r"].float()
    hits = (r.abs() == 200).float().mean().item()
    assert 0.0007 < hits < 0.0013
    clean = r[r.abs() != 200]
    assert abs(clean.std().item() - 2.0) < 0.02  # r ~ N(0, 4): sd 2
    assert abs(d["x"].float().std().item() - 1.0) < 0.01


def test_fp16_clip_never_binds():
    w = far_gen.WORKLOADS["c5"]
    # the largest |x + r| this generator can produce, with rounding slack
    assert 2 * w.scale_hi * far_gen.MAX_ABS_NORMAL * (1 + 2 ** -10) < 60000
