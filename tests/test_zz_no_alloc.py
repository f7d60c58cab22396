"""gdn_prefill_chunked_noalloc, the entry point for callers that cannot allocate.

Some callers may not call cudaMalloc (or any allocator) where they run the layer,
for example a host runtime that only hands out pre-registered buffers or a real-time
path where an allocation could block.  This entry point takes the same inputs and
outputs as gdn_prefill_chunked but uses scratch compiled into the library instead
of a caller workspace.  The test calls it through the C-ABI twice in a row (on
different inputs, so the second call starts from the first call's leftover scratch)
and checks that each result is bit-identical to gdn_prefill_chunked's on the same
inputs (both run the same two-pass schedule, so any leftover scratch that leaked into a
result would show), and the first against the float64 oracle within the bf16 bound of
the parity tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import device_inputs, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module")
def gdn():
    from gated_deltanet_linear_05_gb300 import build
    build.build()
    import gated_deltanet_linear_05_gb300 as mod
    mod.lib()
    return mod


def _noalloc(gdn, d, s_in, s_out, o, chunk):
    import torch
    T, hk, _ = d["q"].shape
    hv = d["v"].shape[1]
    shape = gdn.make_shape(s_out.shape[0], T, hk, hv, chunk=chunk, dtype=gdn.GDN_BF16,
                           o_fp32=int(o.dtype == torch.float32))
    p = lambda t: None if t is None else t.data_ptr()
    return gdn.lib().gdn_prefill_chunked_noalloc(
        ctypes.byref(shape), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]), p(d["beta"]), p(s_in),
        p(s_out), p(d["cu_seqlens"]), p(o), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("o_fp32", [False, True])
def test_noalloc_matches_workspace_entry_on_two_calls(gdn, o_fp32):
    import torch
    odt = torch.float32 if o_fp32 else torch.bfloat16
    cases = [(gi.Workload("a", [300, 77, 129], 2, 4, chunk=64, dtype="bf16", s0_scale=0.1), 1),
             (gi.Workload("b", [1000, 16, 5], 16, 16, chunk=16, dtype="bf16", s0_scale=0.1), 2)]
    runs = []
    for wl, seed in cases:
        x = gi.make_inputs(wl, seed=seed)
        if not runs:
            first = (x, oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                         x["cu_seqlens"]))
        d = device_inputs(x, "bf16")
        shape = gdn.make_shape(wl.num_seqs, wl.total_tokens, wl.num_k_heads, wl.num_v_heads,
                               chunk=wl.chunk)
        assert gdn.gdn_workspace_size(shape, gdn.GDN_OP_PREFILL) <= (64 << 20)
        # the existing entry point, with a caller workspace
        o_ref = torch.empty(d["v"].shape, dtype=odt, device="cuda")
        s_ref = torch.empty_like(d["state0"])
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_ref,
                                d["cu_seqlens"], o_ref, chunk=wl.chunk)
        o = torch.full(d["v"].shape, float("nan"), dtype=odt, device="cuda")
        s = torch.full_like(d["state0"], float("nan"))
        runs.append((wl, d, o, s, o_ref, s_ref))
    torch.cuda.synchronize()
    # two calls of the no-allocation entry point in a row
    for wl, d, o, s, _, _ in runs:
        st = _noalloc(gdn, d, d["state0"], s, o, wl.chunk)
        assert st == gdn.GDN_OK, gdn.gdn_status_string(st)
    torch.cuda.synchronize()
    for wl, d, o, s, o_ref, s_ref in runs:
        assert torch.equal(o, o_ref), wl.name + ": o differs from gdn_prefill_chunked's"
        assert torch.equal(s, s_ref), wl.name + ": state differs from gdn_prefill_chunked's"
    # the first call against the oracle (the bf16 o within half a bf16 spacing more)
    _, (oo, so) = first
    wl, _, o, s, _, _ = runs[0]
    slack = 0.0 if o_fp32 else np.max(np.abs(to_np(o))) * 2.0 ** -9 / np.sqrt(np.mean(oo ** 2))
    assert rel_err(to_np(o), oo) <= TOL + slack, wl.name
    assert rel_err(to_np(s), so) <= TOL, wl.name


def test_noalloc_rejects_requests_beyond_its_scratch(gdn):
    import torch
    # one sequence of 8192 tokens over 16 heads needs ~119 MB of scratch, more than the
    # 64 MiB built in
    T, H = 8192, 16
    shape = gdn.make_shape(1, T, H, H, chunk=64)
    assert gdn.gdn_workspace_size(shape, gdn.GDN_OP_PREFILL) > (64 << 20)
    d = {"q": torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")}
    d["k"] = torch.zeros_like(d["q"])
    d["v"] = torch.zeros_like(d["q"])
    d["g"] = torch.zeros((T, H), device="cuda")
    d["beta"] = torch.zeros((T, H), device="cuda")
    d["cu_seqlens"] = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    s = torch.zeros((1, H, 128, 128), device="cuda")
    o = torch.zeros_like(d["v"])
    assert _noalloc(gdn, d, s, torch.zeros_like(s), o, 64) == gdn.GDN_ERR_WORKSPACE
