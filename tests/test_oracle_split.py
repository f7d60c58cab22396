"""CPU pin of the sequence split's algebra, on the float64 oracle alone: a segment maps its
incoming state affinely, S -> M S + L (the chunkwise form's per-block state update,
"Qwen3.5-9B-npu" model card, "How it works", composed over the segment's tokens), with
L the segment's final state from a zero start and M its final state from the identity
with v = 0.  Combining (M, L) in segment order and re-running each segment from its
incoming state must reproduce the unsplit outputs and final state up to rounding -- the
identity gdn_prefill_split is built on, checked here independently of any GPU code."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle


def _segments(length, seg):
    return [(a, min(a + seg, length)) for a in range(0, length, seg)]


def _one(x, a, b, state, v_zero=False):
    """The oracle over tokens [a, b) of sequence 0 (head layout kept) from `state`; with
    v_zero the values are zero and have dk columns, so that the state is dk x dk."""
    k = x["k"][a:b]
    v = np.zeros(k.shape[:1] + x["v"].shape[1:2] + k.shape[2:], np.float32) if v_zero else x["v"][a:b]
    return oracle.recurrent(x["q"][a:b], x["k"][a:b], v, x["g"][a:b], x["beta"][a:b], state,
                            np.array([0, b - a], np.int32))


@pytest.mark.parametrize("length,seg", [(97, 32), (64, 16), (50, 64), (130, 7)])
def test_segment_maps_compose_to_the_unsplit_pass(length, seg):
    """Every segment run from exact inputs only (a zero state, or the identity with v = 0);
    the composition in float64: S_out = M S_in + L, and o_t = o_t(0) + r_t^T S_in with
    r_t the output of the identity run (the outputs are linear in the incoming state)."""
    wl = gi.Workload("split_pin", [length], 1, 2, dk=16, dv=8, dtype="f32", s0_scale=0.3)
    x = gi.make_inputs(wl, seed=41)
    hv, dk = 2, 16
    o_full, s_full = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                      x["cu_seqlens"])
    eye = np.broadcast_to(np.eye(dk), (1, hv, dk, dk)).copy()
    s_in = x["state0"].astype(np.float64)[0]            # [Hv, dk, dv]
    o_split = np.zeros_like(o_full)
    for a, b in _segments(length, seg):
        o_loc, L = _one(x, a, b, None)                  # from zero: L, o(0)
        r, M = _one(x, a, b, eye, v_zero=True)          # from the identity, v = 0: M, r_t
        o_split[a:b] = o_loc + np.einsum("thk,hkj->thj", r, s_in)
        s_in = np.einsum("hik,hkj->hij", M[0], s_in) + L[0]
    np.testing.assert_allclose(o_split, o_full, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(s_in, s_full[0], rtol=1e-10, atol=1e-12)


def test_map_is_independent_of_the_values_and_of_the_state():
    """M_s depends on k, g, beta only: the same map from two different v and states."""
    wl = gi.Workload("split_pin2", [40], 1, 1, dk=8, dv=8, dtype="f32", s0_scale=0.3)
    x = gi.make_inputs(wl, seed=42)
    eye = np.eye(8)[None, None].copy()
    _, M1 = _one(x, 0, 40, eye, v_zero=True)
    y = dict(x, v=x["v"] * -3.0 + 1.0)
    # the affine map: S(S0) - S(0) = M S0 for any S0, whatever v is
    s0 = x["state0"].astype(np.float64)
    _, s_a = _one(y, 0, 40, s0)
    _, s_b = _one(y, 0, 40, None)
    np.testing.assert_allclose(s_a - s_b, np.einsum("nhik,nhkj->nhij", M1, s0), rtol=1e-11,
                               atol=1e-12)
