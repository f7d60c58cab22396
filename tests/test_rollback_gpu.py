"""GPU parity of the draft-verify accept step: the verify block that captures per-token
deltas, the state rollback to an accepted prefix, and the conv FIFO rollback, against
the float64 oracle (the per-token rule run over the accepted tokens only).

Bounds as for the layer: max |x - ref| / rms(ref) over the tensor, 2e-2 for bf16 q/k/v
and 1e-4 for fp32; the conv FIFO is a copy of raw inputs and must match bit for bit."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import device_inputs, rel_err, to_dev, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def _capture(x, wl, chunk=16, algo=0):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    d = device_inputs(x, wl.dtype)
    s_out = torch.full_like(d["state0"], float("nan"))
    o = torch.full(d["v"].shape, float("nan"), device="cuda",
                   dtype=torch.float32 if wl.dtype == "f32" else torch.float32)
    o, s, delta = gdn.gdn_verify_block_capture(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                               d["state0"], s_out, d["cu_seqlens"], o, chunk=chunk,
                                               algo=algo)
    torch.cuda.synchronize()
    return d, o, s, delta


CASES = [([16] * 6, 2, 4, "bf16", 16), ([16, 3, 1, 16, 9], 1, 2, "f32", 16),
         ([40, 17, 64], 2, 2, "bf16", 16), ([70, 5], 1, 1, "bf16", 64), ([33, 16], 1, 2, "f32", 32)]


@pytest.mark.parametrize("algo", [0, 4])  # AUTO (the single-pass schedule), the token loop
@pytest.mark.parametrize("lengths,hk,hv,dtype,chunk", CASES)
def test_capture_outputs_and_deltas(lengths, hk, hv, dtype, chunk, algo):
    wl = gi.Workload("cap", lengths, hk, hv, chunk=chunk, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=len(lengths))
    d, o, s, delta = _capture(x, wl, chunk, algo)
    o_ref, s_ref, d_ref = oracle.recurrent_deltas(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                  x["state0"], x["cu_seqlens"])
    for name, a, r in (("o", to_np(o), o_ref), ("state", to_np(s), s_ref),
                       ("delta", to_np(delta), d_ref)):
        assert np.isfinite(a).all(), name
        assert rel_err(a, r) <= TOL[dtype], "%s err %.3g" % (name, rel_err(a, r))
    # the snapshot is untouched
    assert np.array_equal(to_np(d["state0"]), x["state0"].astype(np.float64))


def test_capture_matches_the_plain_single_pass_verify():
    """Capturing adds stores only: o and the state equal the same schedule's plain call."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("cap", [16] * 9, 2, 4, chunk=16, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=2)
    d, o, s, _ = _capture(x, wl)
    s2 = torch.empty_like(s)
    o2 = torch.empty_like(o)
    gdn.gdn_verify_block(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s2,
                         d["cu_seqlens"], o2, chunk=16, algo=gdn.GDN_ALGO_SINGLE_PASS)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(s, s2)


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("lengths,hk,hv,dtype,chunk", CASES)
def test_rollback_to_accepted_prefix(lengths, hk, hv, dtype, chunk, inplace):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("rb", lengths, hk, hv, chunk=chunk, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=7 + len(lengths))
    d, _, _, delta = _capture(x, wl, chunk)
    # accepted lengths: none, one, some, all, and past the end (clamped)
    pick = [0, 1, 5, 10 ** 6, 2, 37, 15]
    acc = np.array([pick[i % len(pick)] for i in range(wl.num_seqs)], np.int32)
    acc_d = to_dev(acc, "i32")
    s_in = d["state0"].clone() if inplace else d["state0"]
    s_out = s_in if inplace else torch.full_like(s_in, float("nan"))
    gdn.gdn_state_rollback(d["k"], d["g"], delta, s_in, acc_d, s_out, d["cu_seqlens"])
    torch.cuda.synchronize()
    ref = oracle.state_after_prefix(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"], acc)
    got = to_np(s_out)
    assert np.isfinite(got).all()
    assert rel_err(got, ref) <= TOL[dtype], rel_err(got, ref)
    # a = 0 keeps the snapshot exactly
    for n in range(wl.num_seqs):
        if acc[n] == 0:
            assert np.array_equal(got[n], x["state0"][n].astype(np.float64))


@pytest.mark.slow
def test_capture_and_rollback_full_verify_workload():
    """128 sequences x 32 heads, 16-token drafts, accepted lengths spread over 0..16."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.verify_b128_h32()
    x = gi.make_inputs(wl)
    d, o, s, delta = _capture(x, wl)
    acc = (gi.raw_u64(0, "accept", wl.num_seqs) % np.uint64(17)).astype(np.int32)
    s_rb = torch.empty_like(s)
    gdn.gdn_state_rollback(d["k"], d["g"], delta, d["state0"], to_dev(acc, "i32"), s_rb,
                           d["cu_seqlens"])
    torch.cuda.synchronize()
    o_ref, s_ref, d_ref = oracle.recurrent_deltas(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                  x["state0"], x["cu_seqlens"])
    assert rel_err(to_np(delta), d_ref) <= TOL["bf16"]
    ref = oracle.state_after_prefix(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"], acc)
    assert rel_err(to_np(s_rb), ref) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("inplace", [False, True])
def test_conv_state_rollback(dtype, inplace):
    """The FIFO after the accepted prefix equals the oracle prologue's FIFO after those
    tokens (bit for bit)."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("crb", [16, 16, 5, 2, 16, 0, 9], 2, 4, dtype=dtype)
    x = gi.make_block_inputs(wl, seed=4)
    acc = np.array([0, 1, 2, 3, 16, 4, 100], np.int32)
    raw = {n: to_dev(x[n + "_st"], dtype) for n in ("q_raw", "k_raw", "v_raw")}
    cs_in = to_dev(x["conv_state0_st"], dtype)
    cs_out = cs_in if inplace else torch.full_like(cs_in, float("nan"))
    gdn.gdn_conv_state_rollback(raw["q_raw"], raw["k_raw"], raw["v_raw"], cs_in,
                                to_dev(acc, "i32"), cs_out, to_dev(x["cu_seqlens"], "i32"))
    torch.cuda.synchronize()
    # the oracle's FIFO after the accepted tokens only
    cu = x["cu_seqlens"]
    keep, lens = [], []
    for n in range(wl.num_seqs):
        a = min(int(acc[n]), int(cu[n + 1] - cu[n]))
        keep.extend(range(int(cu[n]), int(cu[n]) + a))
        lens.append(a)
    sub = {n: x[n][keep] for n in ("q_raw", "k_raw", "v_raw", "a", "b")}
    csi = np.ascontiguousarray(np.transpose(x["conv_state0"], (0, 2, 1)))
    *_, cso = oracle.prologue(sub["q_raw"], sub["k_raw"], sub["v_raw"], sub["a"], sub["b"],
                              x["conv_w"], x["A_log"], x["dt_bias"], csi,
                              np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
    assert np.array_equal(to_np(cs_out), np.transpose(cso, (0, 2, 1)))
