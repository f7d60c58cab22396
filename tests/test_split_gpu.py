"""GPU parity of the sequence-split prompt pass (gdn_prefill_split) against the float64
oracle: sequences cut into segments that run side by side, their maps combined in order,
then rerun from their incoming states.  Bounds as for the chunked pass: max |x - ref| /
rms(ref) over the tensor, 2e-2 for bf16 q/k/v and 1e-4 for fp32."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import device_inputs, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def _split(x, wl, seg, state_in=True, inplace=False, algo=0, chunk=None):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    d = device_inputs(x, wl.dtype)
    s_in = d["state0"] if state_in else None
    if inplace:
        s_in = s_in.clone()
        s_out = s_in
    else:
        s_out = torch.full_like(d["state0"], float("nan"))
    o = torch.full(d["v"].shape, float("nan"), device="cuda", dtype=torch.float32)
    gdn.gdn_prefill_split(d["q"], d["k"], d["v"], d["g"], d["beta"], s_in, s_out,
                          d["cu_seqlens"], o, segment_len=seg, chunk=chunk or wl.chunk, algo=algo)
    torch.cuda.synchronize()
    return to_np(o), to_np(s_out)


def _ref(x, state_in=True):
    s0 = x["state0"] if state_in else np.zeros_like(x["state0"])
    return oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], s0, x["cu_seqlens"])


def _check(o, s, o_ref, s_ref, dtype, what):
    assert np.isfinite(o).all() and np.isfinite(s).all(), what
    assert rel_err(o, o_ref) <= TOL[dtype], "%s o err %.3g" % (what, rel_err(o, o_ref))
    assert rel_err(s, s_ref) <= TOL[dtype], "%s state err %.3g" % (what, rel_err(s, s_ref))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_long_sequence(dtype):
    """T = 1000 in segments of 256 (the last one 232 tokens), 2 v-heads on one k-head."""
    wl = gi.Workload("split1", [1000], 1, 2, chunk=64, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=31)
    o, s = _split(x, wl, 256)
    _check(o, s, *_ref(x), dtype, "one sequence")


@pytest.mark.parametrize("chunk,seg", [(64, 128), (16, 48), (32, 32)])
def test_varlen_batch_with_empty_and_short_sequences(chunk, seg):
    wl = gi.Workload("split2", [300, 0, 65, 1000, 17, 128], 2, 4, chunk=chunk, dtype="bf16",
                     s0_scale=0.1)
    x = gi.make_inputs(wl, seed=32)
    o, s = _split(x, wl, seg)
    _check(o, s, *_ref(x), "bf16", "varlen")
    # an empty sequence passes its state through unchanged
    assert np.array_equal(s[1], x["state0"][1].astype(np.float64))


@pytest.mark.parametrize("algo", [1, 2, 3, 5])
def test_each_inner_schedule(algo):
    """The three passes run on the chunked schedule the shape asks for (with
    GDN_ALGO_TWO_PASS_TENSOR the shared pass 1 and the chain-only and output runs of the
    mma.sync second pass, in that schedule's larger workspace)."""
    wl = gi.Workload("split3", [700, 300], 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=33)
    o, s = _split(x, wl, 192, algo=algo)
    _check(o, s, *_ref(x), "bf16", "algo %d" % algo)


def test_in_place_and_zero_state():
    wl = gi.Workload("split4", [513, 64, 1], 2, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=34)
    o, s = _split(x, wl, 128, inplace=True)
    _check(o, s, *_ref(x), "bf16", "in place")
    o, s = _split(x, wl, 128, state_in=False)
    _check(o, s, *_ref(x, state_in=False), "bf16", "zero state")


def test_default_segment_length():
    """segment_len None: the binding's one-wave rule for the device (3000 tokens on 2 heads:
    9 segments of 384 tokens on 152 SMs)."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("split7", [3000], 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=37)
    d = device_inputs(x, "bf16")
    s_out = torch.full_like(d["state0"], float("nan"))
    o = torch.full(d["v"].shape, float("nan"), device="cuda", dtype=torch.float32)
    gdn.gdn_prefill_split(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                          d["cu_seqlens"], o)
    torch.cuda.synchronize()
    _check(to_np(o), to_np(s_out), *_ref(x), "bf16", "default segments")


def test_segment_longer_than_the_sequences():
    """One segment per sequence: the map of step 2 is applied to the incoming state, and
    the outputs come from the plain chunked pass of step 4."""
    wl = gi.Workload("split5", [200, 90], 1, 1, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=35)
    o, s = _split(x, wl, 4096)
    _check(o, s, *_ref(x), "bf16", "one segment")


@pytest.mark.slow
def test_long_single_head_sequence():
    """The regime the split is for: one head, T = 16,384, segments of 1024."""
    wl = gi.Workload("split6", [16384], 1, 1, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=36)
    o, s = _split(x, wl, 1024)
    _check(o, s, *_ref(x), "bf16", "T=16384")


@pytest.mark.slow
def test_bench_configuration():
    """The configuration the bench times: one sequence of 65,536 tokens on 2 heads in
    9 segments of 7,296 tokens (two-pass inner schedule, one chain-only launch)."""
    wl = gi.long_t65536_h2()
    x = gi.make_inputs(wl)
    o, s = _split(x, wl, 7296)
    _check(o, s, *_ref(x), "bf16", "T=65536, H=2")
