"""Pins of the oracle's per-token deltas and prefix states (the draft-verify accept
step: the state after the accepted prefix of a verified block).

The chunkwise form of "Qwen3.5-9B-npu" ("How it works") writes the end-of-block state
as e^{G_T} S0 + K^T diag(e^{G_T - G}) D with D the per-token deltas; cut after a
tokens it gives the state after the prefix.  The pins check the oracle's deltas
against a hand-worked example, against that cut form rebuilt from the per-token loop's
own prefix states, and against special cases."""
import json
import os

import numpy as np
import pytest

import gdn_inputs as gi
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _small(lengths, hk=1, hv=2, dk=8, dv=6, seed=0, s0=0.5):
    wl = gi.Workload("r", lengths, hk, hv, dk=dk, dv=dv, dtype="f32", s0_scale=s0)
    return wl, gi.make_inputs(wl, seed=seed)


def test_hand_example_deltas_and_first_token_state():
    fx = json.load(open(os.path.join(GOLDEN, "hand_example_dk2_dv2_T2.json")))
    inp = fx["inputs"]
    args = [np.array(inp[n], np.float32) for n in ("q", "k", "v")]
    g = np.log(np.array(inp["g_exp"], np.float64)).astype(np.float32)
    beta = np.array(inp["beta"], np.float32)
    s0 = np.array(inp["state0"], np.float32)
    cu = np.array(inp["cu_seqlens"], np.int32)
    o, s, d = oracle.recurrent_deltas(*args, g, beta, s0, cu)
    np.testing.assert_allclose(d, fx["expected"]["delta"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(s, fx["expected"]["state_out"], rtol=1e-6, atol=1e-6)
    s1 = oracle.state_after_prefix(*args, g, beta, s0, cu, [1])
    np.testing.assert_allclose(s1, fx["expected"]["state_after_first_token"], rtol=1e-6, atol=1e-6)
    s2 = oracle.state_after_prefix(*args, g, beta, s0, cu, [5])   # clamped to the length
    np.testing.assert_array_equal(s2, s)
    s0_ = oracle.state_after_prefix(*args, g, beta, s0, cu, [0])
    np.testing.assert_array_equal(s0_, s0.astype(np.float64))


def test_deltas_rebuild_every_prefix_state():
    """e^{G_a} S0 + sum_{t<a} e^{G_a - G_t} k_t delta_t^T equals the loop's state after a
    tokens, for every a of every sequence (GQA, ragged lengths)."""
    wl, x = _small([9, 1, 4], hk=1, hv=2)
    _, _, d = oracle.recurrent_deltas(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                      x["cu_seqlens"])
    cu = x["cu_seqlens"]
    for a in range(0, 10):
        pref = [min(a, L) for L in wl.lengths]
        s_loop = oracle.state_after_prefix(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                           x["state0"], cu, pref)
        for n in range(wl.num_seqs):
            for h in range(wl.num_v_heads):
                kh = h // (wl.num_v_heads // wl.num_k_heads)
                toks = range(cu[n], cu[n] + pref[n])
                G = np.cumsum([float(x["g"][t, h]) for t in toks])
                Ga = G[-1] if len(G) else 0.0
                S = np.exp(Ga) * x["state0"][n, h].astype(np.float64)
                for i, t in enumerate(toks):
                    S += np.exp(Ga - G[i]) * np.outer(x["k"][t, kh], d[t, h])
                np.testing.assert_allclose(S, s_loop[n, h], rtol=1e-12, atol=1e-12)


def test_zero_write_strength_gives_zero_deltas():
    wl, x = _small([6, 3])
    x["beta"][:] = 0.0
    _, s, d = oracle.recurrent_deltas(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                      x["cu_seqlens"])
    assert not d.any()


def test_orthonormal_keys_from_zero_state_store_v():
    """g = 0, beta = 1, S0 = 0, keys e_0, e_1, ...: each delta is the token's v."""
    T, d = 5, 8
    q = np.zeros((T, 1, d), np.float32)
    k = np.eye(d, dtype=np.float32)[:T].reshape(T, 1, d)
    v = gi.normal(3, "v", T * 6).reshape(T, 1, 6).astype(np.float32)
    g = np.zeros((T, 1), np.float32)
    beta = np.ones((T, 1), np.float32)
    _, _, dl = oracle.recurrent_deltas(q, k, v, g, beta, None, np.array([0, T], np.int32))
    np.testing.assert_array_equal(dl, v.astype(np.float64))
