"""gdn_decode_block_step: the block's one-token decode step in one launch (input prologue,
state step, gated RMSNorm) against the same chain in the float64 oracle, and against the
three separate launches on the GPU.

q, k and v cross between the oracle's steps rounded to the storage dtype, as the fused
kernel (and the separate prologue) round them; the layer's bound (2e-2 of the rms) applies
to the state and to y beyond y's own bf16 rounding; the FIFO is data movement (exact)."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import half_ulp_bf16, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def _state0(n, hv, seed):
    s0 = 0.1 * gi.normal(seed, "s0", n * hv * 128 * 128)
    return s0.astype(np.float32).reshape(n, hv, 128, 128)


def _oracle_step(x, cs_in, s_in, dt):
    """One token per sequence through the oracle chain; returns y, state, FIFO, o."""
    csi = np.ascontiguousarray(np.transpose(cs_in, (0, 2, 1)))
    q, k, v, g, beta, cso = oracle.prologue(x["q_raw"], x["k_raw"], x["v_raw"], x["a"], x["b"],
                                            x["conv_w"], x["A_log"], x["dt_bias"], csi, None)
    if dt == "bf16":
        q, k, v = (gi.round_to(a, "bf16")[0] for a in (q, k, v))
    o, s = oracle.recurrent(q, k, v, g, beta, s_in, np.arange(len(q) + 1, dtype=np.int32))
    y = oracle.gated_rmsnorm(o.astype(np.float32), x["z"], x["norm_w"])
    return y, s, np.transpose(cso, (0, 2, 1)), o


def _dev_block(x, dt):
    d = {n: to_dev(x[n + "_st"], dt) for n in ("q_raw", "k_raw", "v_raw", "z")}
    for n in ("a", "b", "conv_w", "A_log", "dt_bias", "norm_w"):
        d[n] = to_dev(x[n], "f32")
    return d


def _check_y(y, y_ref, dt):
    rms = np.sqrt(np.mean(y_ref ** 2))
    if dt == "bf16":
        excess = np.maximum(np.abs(y - y_ref) - half_ulp_bf16(y), 0.0)
        assert excess.max() / rms <= 2e-2
    else:
        assert np.max(np.abs(y - y_ref)) / rms <= 1e-4


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("hk,hv", [(4, 4), (2, 4), (1, 4), (2, 16)])
def test_fused_decode_steps_in_place_against_the_oracle_chain(dt, hk, hv):
    """Four consecutive steps, FIFO and state updated in place, fresh token inputs per
    step, one workspace zeroed once and reused (its counters must come back to zero);
    every step's y, the FIFO and the state against the oracle's chain.  Grouped heads up
    to 8 v-heads per k-head: 32 CTAs count in on one k-head's FIFO."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    n = 6
    wl = gi.Workload("dec", [1] * n, hk, hv, dtype=dt)
    tol = 2e-2 if dt == "bf16" else 1e-4
    s_ref = _state0(n, hv, 3)
    s = to_dev(s_ref, "f32")
    cs_ref = None
    cs = None
    shape = gdn.make_shape(n, n, hk, hv)
    ws = torch.zeros(gdn.gdn_workspace_size(shape, gdn.GDN_OP_DECODE_BLOCK) + 256,
                     dtype=torch.uint8, device="cuda")
    for step in range(4):
        x = gi.make_block_inputs(wl, seed=17, step=step)
        if cs is None:
            cs_ref = x["conv_state0"]
            cs = to_dev(x["conv_state0_st"], dt)
        d = _dev_block(x, dt)
        o = torch.empty((n, hv, 128), dtype=torch.float32, device="cuda")
        y, _ = gdn.gdn_decode_block_step(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                         d["conv_w"], d["A_log"], d["dt_bias"], cs, cs, s, s,
                                         d["z"], d["norm_w"], o=o, workspace=ws)
        torch.cuda.synchronize()
        y_ref, s_ref, cs_ref, o_ref = _oracle_step(x, cs_ref, s_ref, dt)
        assert np.array_equal(to_np(cs), cs_ref), "FIFO step %d" % step
        s_np = to_np(s)
        assert np.max(np.abs(s_np - s_ref)) / np.sqrt(np.mean(s_ref ** 2)) <= tol, step
        o_np = to_np(o)
        assert np.max(np.abs(o_np - o_ref)) / np.sqrt(np.mean(o_ref ** 2)) <= tol, step
        _check_y(to_np(y), y_ref, dt)
        s_ref = s_ref.astype(np.float64)


def test_fused_decode_matches_the_three_launches():
    """Decode batch 32 x 16 heads: the fused step against gdn_input_prologue ->
    gdn_decode_step -> gdn_gated_rmsnorm on the same inputs (FIFO bit for bit; state and
    y within the sums' reordering), and against the oracle."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    n, hk, hv = 32, 16, 16
    wl = gi.Workload("dec", [1] * n, hk, hv, dtype="bf16")
    x = gi.make_block_inputs(wl, seed=23)
    d = _dev_block(x, "bf16")
    s0 = _state0(n, hv, 4)
    cs_in = to_dev(x["conv_state0_st"], "bf16")
    # the three launches
    cs3 = torch.empty_like(cs_in)
    q, k, v, g, beta = gdn.gdn_input_prologue(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                              d["conv_w"], d["A_log"], d["dt_bias"], cs_in, cs3, None)
    s3 = to_dev(s0, "f32")
    o3 = torch.empty((n, hv, 128), dtype=torch.float32, device="cuda")
    gdn.gdn_decode_step(q, k, v, g, beta, s3, s3, None, o3)
    y3 = gdn.gdn_gated_rmsnorm(o3, d["z"], d["norm_w"])
    # fused
    cs1 = torch.empty_like(cs_in)
    s1 = to_dev(s0, "f32")
    y1, _ = gdn.gdn_decode_block_step(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                      d["conv_w"], d["A_log"], d["dt_bias"], cs_in, cs1, s1, s1,
                                      d["z"], d["norm_w"])
    torch.cuda.synchronize()
    assert torch.equal(cs1, cs3)
    s1n, s3n = to_np(s1), to_np(s3)
    assert np.max(np.abs(s1n - s3n)) / np.sqrt(np.mean(s3n ** 2)) <= 1e-2
    y1n, y3n = to_np(y1), to_np(y3)
    assert np.max(np.abs(y1n - y3n)) / np.sqrt(np.mean(y3n ** 2)) <= 2e-2
    y_ref, s_ref, cs_ref, _ = _oracle_step(x, x["conv_state0"], s0.astype(np.float64), "bf16")
    assert np.array_equal(to_np(cs1), cs_ref)
    assert np.max(np.abs(s1n - s_ref)) / np.sqrt(np.mean(s_ref ** 2)) <= 2e-2
    _check_y(y1n, y_ref, "bf16")


def test_fused_decode_zero_initial_states_and_no_fifo_output():
    """state_in NULL (zero state), conv_state_in NULL (zero FIFO), conv_state_out NULL."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    n, hk, hv = 3, 1, 2
    wl = gi.Workload("dec0", [1] * n, hk, hv, dtype="bf16")
    x = gi.make_block_inputs(wl, seed=29)
    d = _dev_block(x, "bf16")
    s = torch.full((n, hv, 128, 128), float("nan"), device="cuda")
    y, _ = gdn.gdn_decode_block_step(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                     d["conv_w"], d["A_log"], d["dt_bias"], None, None, None, s,
                                     d["z"], d["norm_w"])
    torch.cuda.synchronize()
    zeros = np.zeros_like(x["conv_state0"])
    y_ref, s_ref, _, _ = _oracle_step(x, zeros, np.zeros((n, hv, 128, 128)), "bf16")
    s_np = to_np(s)
    assert np.isfinite(s_np).all()
    assert np.max(np.abs(s_np - s_ref)) / np.sqrt(np.mean(s_ref ** 2)) <= 2e-2
    _check_y(to_np(y), y_ref, "bf16")
