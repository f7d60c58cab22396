"""The seeded input generator: determinism, distribution and rounding."""
import numpy as np
import pytest

import gdn_inputs as gi


def test_streams_are_deterministic_and_independent():
    a = gi.normal(0, "q", 1000)
    assert np.array_equal(a, gi.normal(0, "q", 1000))
    assert np.array_equal(a[:333], gi.normal(0, "q", 333))     # prefix-stable
    assert not np.array_equal(a, gi.normal(0, "k", 1000))
    assert not np.array_equal(a, gi.normal(1, "q", 1000))
    assert np.array_equal(gi.raw_u64(0, "x", 50)[10:], gi.raw_u64(0, "x", 40, offset=10))


def test_normal_moments():
    z = gi.normal(0, "moments", 400_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    assert abs(np.mean(z ** 4) - 3) < 0.1


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = (gi.normal(0, "bf", 100_000) * np.exp(gi.normal(1, "sc", 100_000) * 4)).astype(np.float32)
    ties = np.array([1.00390625, 1.01171875, -1.00390625, 3.0e-39], np.float32)  # exact halfway cases, subnormal
    x = np.concatenate([x, ties])
    bits = gi.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
    back = gi.bf16_bits_to_f32(bits)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_workload_recipes():
    wl = gi.varlen_8seq_hk16_hv32()
    assert len(wl.lengths) == 8 and all(256 <= L <= 8192 for L in wl.lengths)
    small = gi.Workload("s", [3, 5], 2, 4, dk=16, dv=8, dtype="bf16")
    x = gi.make_inputs(small)
    assert x["q"].shape == (8, 2, 16) and x["v"].shape == (8, 4, 8)
    assert x["state0"].shape == (2, 4, 16, 8)
    n = np.linalg.norm(x["q"].astype(np.float64), axis=-1)
    assert np.all(np.abs(n - 1) < 1e-2)                  # unit rows up to bf16 rounding
    assert np.all(x["g"] < 0) and np.all((x["beta"] > 0) & (x["beta"] < 1))
    assert np.array_equal(gi.bf16_bits_to_f32(x["v_st"]), x["v"])
    assert list(x["cu_seqlens"]) == [0, 3, 8]
    d1 = gi.make_inputs(small, step=1)
    assert not np.array_equal(d1["q"], x["q"]) and np.array_equal(d1["state0"], x["state0"])
