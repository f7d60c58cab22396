"""GPU parity of the block steps around the layer -- the input prologue (causal conv +
SiLU, q/k L2 norm, gates) and the gated-RMSNorm epilogue -- against the float64 oracle
on the same seeded inputs, through the C ABI.

Bounds, per element: a bf16 output may differ from the exact value by its own
rounding (half a bf16 spacing) plus the fp32 arithmetic before it; fp32 outputs by
the fp32 arithmetic alone (a few units in the last place of each step, taken as
1e-5 relative plus 1e-6 of the tensor's rms).  The advanced conv FIFO is a copy of
raw inputs and must match bit for bit.
"""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import half_ulp_bf16, to_dev, to_np

pytestmark = pytest.mark.gpu

W = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def _close(x, ref, dtype, what):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(x).all(), what
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 1.0
    bound = 1e-5 * np.abs(ref) + 1e-6 * rms
    if dtype == "bf16":
        bound = bound + half_ulp_bf16(x)
    excess = np.abs(x - ref) - bound
    assert excess.max(initial=-1.0) <= 0, "%s: worst excess %.3g at %s" % (
        what, excess.max(), np.unravel_index(np.argmax(excess), excess.shape))


def _oracle_prologue(x, cs_in, cu):
    """The oracle takes the FIFO as [N, C, W-1]; the library's layout is [N, W-1, C]."""
    csi = None if cs_in is None else np.ascontiguousarray(np.transpose(cs_in, (0, 2, 1)))
    q, k, v, g, beta, cso = oracle.prologue(x["q_raw"], x["k_raw"], x["v_raw"], x["a"], x["b"],
                                            x["conv_w"], x["A_log"], x["dt_bias"], csi, cu)
    return q, k, v, g, beta, np.transpose(cso, (0, 2, 1))


def _gpu_prologue(x, wl, per_token=False, state_in=True, state_out=True, inplace=False):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    dt = wl.dtype
    d = {n: to_dev(x[n + "_st"], dt) for n in ("q_raw", "k_raw", "v_raw")}
    for n in ("a", "b", "conv_w", "A_log", "dt_bias"):
        d[n] = to_dev(x[n], "f32")
    cs_in = to_dev(x["conv_state0_st"], dt) if state_in else None
    if inplace:
        cs_out = cs_in
    elif state_out:
        cs_out = torch.full(tuple(x["conv_state0"].shape), float("nan"), device="cuda",
                            dtype=d["q_raw"].dtype)
    else:
        cs_out = None
    cu = None if per_token else to_dev(x["cu_seqlens"], "i32")
    nan = lambda t: torch.full_like(t, float("nan"))
    q, k, v = nan(d["q_raw"]), nan(d["k_raw"]), nan(d["v_raw"])
    g = torch.full(tuple(x["a"].shape), float("nan"), device="cuda")
    beta = torch.full_like(g, float("nan"))
    gdn.gdn_input_prologue(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"], d["conv_w"],
                           d["A_log"], d["dt_bias"], cs_in, cs_out, cu, 1e-6, q, k, v, g, beta)
    torch.cuda.synchronize()
    outs = [to_np(t) for t in (q, k, v, g, beta)]
    return outs, (None if cs_out is None else to_np(cs_out))


def _check_prologue(x, wl, per_token=False, state_in=True, state_out=True, inplace=False):
    got, cs = _gpu_prologue(x, wl, per_token, state_in, state_out, inplace)
    ref = _oracle_prologue(x, x["conv_state0"] if state_in else None,
                           None if per_token else x["cu_seqlens"])
    for name, a, r in zip(("q", "k", "v"), got[:3], ref[:3]):
        _close(a, r, wl.dtype, name)
    _close(got[3], ref[3], "f32", "g")
    _close(got[4], ref[4], "f32", "beta")
    if cs is not None:
        assert np.array_equal(cs, ref[5]), "conv state out"
    return got, ref


PROLOGUE_CASES = [
    ([1], 1, 1), ([2], 1, 2), ([3], 1, 1), ([17], 2, 2),
    ([1, 2, 3, 5, 40, 0, 130], 2, 4),          # short sequences, an empty one, runs crossing
    ([0, 16, 16, 15, 1, 0], 1, 2),             # boundaries on and off the 16-token runs
    ([300, 257], 4, 8),
    ([40, 3, 19], 3, 3),                       # odd head count: a q/k pair, a lone last head
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("lengths,hk,hv", PROLOGUE_CASES)
def test_prologue_packed_sequences(dtype, lengths, hk, hv):
    wl = gi.Workload("pro", lengths, hk, hv, dtype=dtype)
    x = gi.make_block_inputs(wl, seed=len(lengths) + hk)
    _check_prologue(x, wl)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prologue_packing_does_not_change_a_bit(dtype):
    """A token's outputs (and its sequence's advanced FIFO) are the same bits whether the
    sequence runs packed behind others or alone: the kernel's 16-token units and their
    boundary path fall on different tokens in the two runs."""
    lengths = [37, 5, 90, 16, 3, 21]
    wl = gi.Workload("pack", lengths, 2, 4, dtype=dtype)
    x = gi.make_block_inputs(wl, seed=12)
    packed, cs_packed = _gpu_prologue(x, wl)
    cu = x["cu_seqlens"]
    for n, L in enumerate(lengths):
        a, b = int(cu[n]), int(cu[n + 1])
        xn = dict(x)
        for name in ("q_raw", "k_raw", "v_raw"):
            xn[name], xn[name + "_st"] = x[name][a:b], x[name + "_st"][a:b]
        xn["a"], xn["b"] = x["a"][a:b], x["b"][a:b]
        xn["conv_state0"], xn["conv_state0_st"] = x["conv_state0"][n:n + 1], x["conv_state0_st"][n:n + 1]
        xn["cu_seqlens"] = np.array([0, L], np.int32)
        alone, cs_alone = _gpu_prologue(xn, gi.Workload("one", [L], 2, 4, dtype=dtype))
        for i, name in enumerate(("q", "k", "v", "g", "beta")):
            assert np.array_equal(packed[i][a:b], alone[i]), (n, name)
        assert np.array_equal(cs_packed[n:n + 1], cs_alone), n


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prologue_in_place_state(dtype):
    wl = gi.Workload("pro", [5, 1, 70, 2, 33], 2, 4, dtype=dtype)
    x = gi.make_block_inputs(wl, seed=11)
    _check_prologue(x, wl, inplace=True)


def test_prologue_without_states():
    wl = gi.Workload("pro", [4, 19, 2], 1, 2)
    x = gi.make_block_inputs(wl, seed=12)
    _check_prologue(x, wl, state_in=False)
    got, _ = _gpu_prologue(x, wl, state_out=False)
    ref = _oracle_prologue(x, x["conv_state0"], x["cu_seqlens"])
    _close(got[2], ref[2], "bf16", "v without a state_out")


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("n,hk,hv", [(1, 1, 1), (37, 2, 4), (9, 3, 3), (512, 16, 32)])
def test_prologue_decode_step(n, hk, hv, inplace):
    """One token per sequence (no cu_seqlens), the FIFO updated in place or not."""
    wl = gi.Workload("pro_dec", [1] * n, hk, hv)
    x = gi.make_block_inputs(wl, seed=n, step=3)
    _check_prologue(x, wl, per_token=True, inplace=inplace)


def test_prologue_decode_steps_chain():
    """Eight decode steps through one in-place FIFO equal one packed 8-token call."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    n, hk, hv, steps = 6, 1, 2, 8
    wl = gi.Workload("pro_chain", [steps] * n, hk, hv)
    x = gi.make_block_inputs(wl, seed=5)
    ref = _oracle_prologue(x, x["conv_state0"], x["cu_seqlens"])
    cs = to_dev(x["conv_state0_st"], "bf16")
    d = {nm: to_dev(x[nm], "f32") for nm in ("conv_w", "A_log", "dt_bias")}
    for t in range(steps):
        rows = [s * steps + t for s in range(n)]   # token t of every sequence
        sub = lambda a: np.ascontiguousarray(a[rows])
        qr, kr, vr = (to_dev(sub(x[nm + "_st"]), "bf16") for nm in ("q_raw", "k_raw", "v_raw"))
        q, k, v, g, beta = gdn.gdn_input_prologue(qr, kr, vr, to_dev(sub(x["a"]), "f32"),
                                                  to_dev(sub(x["b"]), "f32"), d["conv_w"],
                                                  d["A_log"], d["dt_bias"], cs, cs)
        torch.cuda.synchronize()
        for nm, a, r in zip(("q", "k", "v"), (q, k, v), ref[:3]):
            _close(to_np(a), r[rows], "bf16", "%s step %d" % (nm, t))
        _close(to_np(g), ref[3][rows], "f32", "g step %d" % t)
    assert np.array_equal(to_np(cs), ref[5])


@pytest.mark.slow
def test_prologue_varlen_full_size():
    """The packed workload of 8 sequences (Hk 16, Hv 32), all tokens against the oracle."""
    wl = gi.varlen_8seq_hk16_hv32()
    x = gi.make_block_inputs(wl)
    _check_prologue(x, wl)


# ------------------------------------------------------------------ gated RMSNorm

def _gpu_norm(x, wl, o, o_fp32=False, inplace=None):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    od = to_dev(o.astype(np.float32), "f32") if (o_fp32 or wl.dtype == "f32") else \
        to_dev(gi.f32_to_bf16_bits(o.astype(np.float32)), "bf16")
    z = to_dev(x["z_st"], wl.dtype)
    w = to_dev(x["norm_w"], "f32")
    y = {"o": od, "z": z}.get(inplace)
    y = gdn.gdn_gated_rmsnorm(od, z, w, 1e-6, y)
    torch.cuda.synchronize()
    return to_np(y), to_np(od)


@pytest.mark.parametrize("o_fp32", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("lengths,hv", [([1], 1), ([7], 3), ([129, 64, 1], 4), ([4096], 16)])
def test_gated_rmsnorm(dtype, o_fp32, lengths, hv):
    if dtype == "f32" and o_fp32:
        pytest.skip("o is fp32 already")
    wl = gi.Workload("norm", lengths, 1, hv, dtype=dtype)
    x = gi.make_block_inputs(wl, seed=hv)
    o = gi.normal(7, "o", wl.total_tokens * hv * 128).reshape(-1, hv, 128) * 0.3
    y, od = _gpu_norm(x, wl, o, o_fp32)
    ref = oracle.gated_rmsnorm(od.astype(np.float32), x["z"], x["norm_w"])
    _close(y, ref, dtype, "y")


@pytest.mark.parametrize("where", ["o", "z"])
def test_gated_rmsnorm_in_place(where):
    wl = gi.Workload("norm", [300], 1, 4)
    x = gi.make_block_inputs(wl, seed=2)
    o = gi.normal(8, "o", 300 * 4 * 128).reshape(300, 4, 128)
    ref = oracle.gated_rmsnorm(gi.bf16_bits_to_f32(gi.f32_to_bf16_bits(o.astype(np.float32))),
                               x["z"], x["norm_w"])
    y, _ = _gpu_norm(x, wl, o, inplace=where)
    _close(y, ref, "bf16", "in place over " + where)


def test_block_prologue_layer_epilogue():
    """The three steps chained on the GPU (prologue -> chunked layer -> gated norm) against
    the same chain in the oracle; the layer's own bound (2e-2 of the rms) applies."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("block", [100, 64, 1, 37], 2, 4)
    x = gi.make_block_inputs(wl, seed=21)
    d = {n: to_dev(x[n + "_st"], "bf16") for n in ("q_raw", "k_raw", "v_raw", "z")}
    for n in ("a", "b", "conv_w", "A_log", "dt_bias", "norm_w"):
        d[n] = to_dev(x[n], "f32")
    cs = to_dev(x["conv_state0_st"], "bf16")
    cu = to_dev(x["cu_seqlens"], "i32")
    s0 = 0.1 * gi.normal(4, "s0", wl.num_seqs * 4 * 128 * 128).reshape(wl.num_seqs, 4, 128, 128)
    s0 = s0.astype(np.float32)
    q, k, v, g, beta = gdn.gdn_input_prologue(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                              d["conv_w"], d["A_log"], d["dt_bias"], cs, cs, cu)
    s = to_dev(s0, "f32")
    o = torch.empty(v.shape, dtype=torch.float32, device="cuda")
    gdn.gdn_prefill_chunked(q, k, v, g, beta, s, s, cu, o, chunk=64)
    y = gdn.gdn_gated_rmsnorm(o, d["z"], d["norm_w"])
    torch.cuda.synchronize()
    rq, rk, rv, rg, rb, _ = _oracle_prologue(x, x["conv_state0"], x["cu_seqlens"])
    # q, k, v cross between the steps in their storage dtype (bf16) on both sides: with
    # slow decays the state is a near-interpolating fit of the keys, sensitive to the
    # keys' own rounding far beyond the layer's bound
    rq, rk, rv = (gi.round_to(a, "bf16")[0] for a in (rq, rk, rv))
    o_ref, s_ref = oracle.recurrent(rq, rk, rv, rg, rb, s0, x["cu_seqlens"])
    y_ref = oracle.gated_rmsnorm(o_ref.astype(np.float32), x["z"], x["norm_w"])
    s_np, y_np = to_np(s), to_np(y)
    assert np.max(np.abs(s_np - s_ref)) / np.sqrt(np.mean(s_ref ** 2)) <= 2e-2
    # y is stored in bf16: the bound applies beyond its own rounding
    excess = np.maximum(np.abs(y_np - y_ref) - half_ulp_bf16(y_np), 0.0)
    assert excess.max() / np.sqrt(np.mean(y_ref ** 2)) <= 2e-2


def test_prefix_reuse_two_turns_equal_one_pass():
    """Prefix reuse: turn 2 run from the conv FIFO and state kept after turn 1 gives the
    outputs and final state of one pass over both turns (against the oracle's one pass)."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    turn1, turn2 = [70, 5, 33], [40, 17, 1]
    both = [a + b for a, b in zip(turn1, turn2)]
    wl = gi.Workload("reuse", both, 1, 2)
    x = gi.make_block_inputs(wl, seed=31)
    cu = x["cu_seqlens"]
    idx1 = np.concatenate([np.arange(cu[n], cu[n] + turn1[n]) for n in range(3)])
    idx2 = np.concatenate([np.arange(cu[n] + turn1[n], cu[n + 1]) for n in range(3)])
    s0 = (0.1 * gi.normal(5, "s0", 3 * 2 * 128 * 128)).astype(np.float32).reshape(3, 2, 128, 128)
    w = {n: to_dev(x[n], "f32") for n in ("conv_w", "A_log", "dt_bias")}
    cs = to_dev(x["conv_state0_st"], "bf16")
    s = to_dev(s0, "f32")
    outs = []
    for idx, lens in ((idx1, turn1), (idx2, turn2)):
        raw = {n: to_dev(np.ascontiguousarray(x[n + "_st"][idx]), "bf16")
               for n in ("q_raw", "k_raw", "v_raw")}
        ab = {n: to_dev(np.ascontiguousarray(x[n][idx]), "f32") for n in ("a", "b")}
        cu_t = to_dev(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), "i32")
        q, k, v, g, beta = gdn.gdn_input_prologue(raw["q_raw"], raw["k_raw"], raw["v_raw"],
                                                  ab["a"], ab["b"], w["conv_w"], w["A_log"],
                                                  w["dt_bias"], cs, cs, cu_t)
        o = torch.empty(v.shape, dtype=torch.float32, device="cuda")
        gdn.gdn_prefill_chunked(q, k, v, g, beta, s, s, cu_t, o, chunk=64)
        torch.cuda.synchronize()
        outs.append(to_np(o))
    rq, rk, rv, rg, rb, rcs = _oracle_prologue(x, x["conv_state0"], cu)
    rq, rk, rv = (gi.round_to(a, "bf16")[0] for a in (rq, rk, rv))
    o_ref, s_ref = oracle.recurrent(rq, rk, rv, rg, rb, s0, cu)
    assert np.array_equal(to_np(cs), rcs)
    for got, idx in zip(outs, (idx1, idx2)):
        ref = o_ref[idx]
        assert np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2)) <= 2e-2
    assert np.max(np.abs(to_np(s) - s_ref)) / np.sqrt(np.mean(s_ref ** 2)) <= 2e-2
