"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Every check here compares the oracle with something it does not compute:
a hand-worked example, a closed form that follows from the page's
equations for a special input, an identity of linear algebra, or the
chunkwise form of the same page (a different formula that reaches the
same result exactly).  Source for all of them: "Qwen3.5-9B-npu" model card,
section "How it works" (per-token recurrence, 1-token matrix form,
chunkwise form, block-doubling inverse, token_valid padding) and the
packed-varlen / grouped-head workload recipe.
"""
import json
import os

import numpy as np
import pytest

import gdn_inputs as gi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.sqrt(np.mean(np.square(b))), 1e-300))


def _small(lengths, hk=1, hv=1, dk=8, dv=6, s0=0.3, seed=0, gate_scale=1.0):
    wl = gi.Workload("small", list(lengths), hk, hv, dk=dk, dv=dv, chunk=4, dtype="f32",
                     s0_scale=s0)
    x = gi.make_inputs(wl, seed=seed, gate_scale=gate_scale)
    return wl, x


def _run(x, **kw):
    return oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                            x["cu_seqlens"], **kw)


# ---------------------------------------------------------------- hand example

def test_hand_worked_example():
    """Two tokens worked by hand in exact arithmetic (tests/golden fixture)."""
    fx = json.load(open(os.path.join(GOLDEN, "hand_example_dk2_dv2_T2.json")))
    inp = fx["inputs"]
    q = np.array(inp["q"], np.float32)
    k = np.array(inp["k"], np.float32)
    v = np.array(inp["v"], np.float32)
    g = np.log(np.array(inp["g_exp"], np.float64)).astype(np.float32)
    beta = np.array(inp["beta"], np.float32)
    s0 = np.array(inp["state0"], np.float32)
    cu = np.array(inp["cu_seqlens"], np.int32)
    o_ref = np.array(fx["expected"]["o"])
    s_ref = np.array(fx["expected"]["state_out"])
    o, s = oracle.recurrent(q, k, v, g, beta, s0, cu)
    np.testing.assert_allclose(o, o_ref, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(s, s_ref, rtol=1e-6, atol=1e-6)
    for C in (1, 2, 4):
        for solve in ("forward", "doubling"):
            o2, s2 = oracle.chunked(q, k, v, g, beta, s0, cu, C, solve)
            np.testing.assert_allclose(o2, o_ref, rtol=1e-6, atol=1e-6)
            np.testing.assert_allclose(s2, s_ref, rtol=1e-6, atol=1e-6)


# ---------------------------------------------------------------- chunk form

@pytest.mark.parametrize("C", [1, 4, 16, 64])
@pytest.mark.parametrize("solve", ["forward", "doubling"])
def test_chunked_form_equals_token_loop(C, solve):
    """The chunkwise form equals the per-token loop (exact in real arithmetic)."""
    wl, x = _small([70, 1, 17, 16, 33], hk=2, hv=4, dk=8, dv=6)
    o1, s1 = _run(x)
    o2, s2 = oracle.chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                            x["cu_seqlens"], C, solve)
    assert _rel(o2, o1) < 1e-12
    assert _rel(s2, s1) < 1e-12


def test_chunked_form_slow_decay_dk128():
    """Full head size, slow decay (state carries across many blocks)."""
    wl = gi.Workload("s", [150], 1, 2, dk=128, dv=128, dtype="f32", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=3, gate_scale=0.01)
    o1, s1 = _run(x)
    for C in (16, 64):
        o2, s2 = oracle.chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                x["cu_seqlens"], C, "doubling")
        assert _rel(o2, o1) < 1e-11 and _rel(s2, s1) < 1e-11


def test_chunked_form_strong_decay():
    """g ~ -28 per token: e^G of a 64-token block underflows to zero in float64 long before
    its end.  The chunk form takes every decay as the exp of a difference of cumsums, so it
    stays finite and equal to the token loop (a product e^G_t e^-G_j would be 0 * inf)."""
    wl = gi.Workload("s", [150, 7, 64], 1, 2, dk=16, dv=8, dtype="f32", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=5, gate_scale=40.0)
    G = np.cumsum(x["g"][:64, 0].astype(np.float64))
    assert np.exp(G[-1]) == 0.0  # the regime the pin is about
    o1, s1 = _run(x)
    for C in (16, 64):
        o2, s2 = oracle.chunked(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                x["cu_seqlens"], C, "doubling")
        assert np.isfinite(o2).all() and np.isfinite(s2).all()
        assert _rel(o2, o1) < 1e-12 and _rel(s2, s1) < 1e-12


# ---------------------------------------------------------------- closed forms

def test_beta_zero_is_pure_decay():
    """beta = 0: no writes, S_T = exp(G_T) S0 and o_t = exp(G_t) S0^T q_t."""
    wl, x = _small([23], dk=5, dv=7)
    x["beta"][:] = 0.0
    o, s = _run(x)
    G = np.cumsum(x["g"][:, 0].astype(np.float64))
    S0 = x["state0"][0, 0].astype(np.float64)
    np.testing.assert_allclose(s[0, 0], np.exp(G[-1]) * S0, rtol=1e-13, atol=1e-300)
    o_ref = np.exp(G)[:, None] * (x["q"][:, 0].astype(np.float64) @ S0)
    assert _rel(o[:, 0], o_ref) < 1e-13


def test_orthonormal_keys_store_values():
    """g = 0, beta = 1, orthonormal keys: the state maps each k_i to v_i, for any S0."""
    dk, dv, T = 16, 9, 12
    wl, x = _small([T], dk=dk, dv=dv, s0=1.0)
    basis, _ = np.linalg.qr(gi.normal(5, "basis", dk * dk).reshape(dk, dk))
    K = basis[:, :T].T                       # T orthonormal rows
    x["k"] = K.astype(np.float32).reshape(T, 1, dk)
    x["g"][:] = 0.0
    x["beta"][:] = 1.0
    o, s = _run(x)
    recalled = x["k"][:, 0].astype(np.float64) @ s[0, 0]          # rows: S_T^T k_i
    np.testing.assert_allclose(recalled, x["v"][:, 0], atol=5e-6)   # float32 keys: ~1e-7 off-orthogonal


def test_single_token_matches_matrix_form():
    """T = 1 equals the 1-token matrix form: o = d q^T S + (q.k) delta, S' = d S + k delta^T."""
    dk, dv = 8, 5
    wl, x = _small([1, 1, 1], hk=1, hv=2, dk=dk, dv=dv, s0=0.7)
    o, s = _run(x)
    for n in range(3):
        for h in range(2):
            q = x["q"][n, 0].astype(np.float64)
            k = x["k"][n, 0].astype(np.float64)
            v = x["v"][n, h].astype(np.float64)
            d = np.exp(np.float64(x["g"][n, h]))
            b = np.float64(x["beta"][n, h])
            S = x["state0"][n, h].astype(np.float64)
            delta = b * (v - d * (k @ S))
            assert _rel(o[n, h], d * (q @ S) + (q @ k) * delta) < 1e-13
            assert _rel(s[n, h], d * S + np.outer(k, delta)) < 1e-13


def test_single_token_zero_state():
    """T = 1, S0 = 0: o = beta (q.k) v."""
    wl, x = _small([1], dk=8, dv=8, s0=None)
    o, s = _run(x)
    q, k, v = (x[n][0, 0].astype(np.float64) for n in ("q", "k", "v"))
    np.testing.assert_allclose(o[0, 0], x["beta"][0, 0] * (q @ k) * v, rtol=1e-13)


def test_delta_rule_write_property():
    """One step with |k| = 1: S'^T k = (1 - beta) d S^T k + beta v."""
    wl, x = _small([1], dk=12, dv=7, s0=0.5)
    o, s = _run(x)
    k = x["k"][0, 0].astype(np.float64)
    k_norm2 = k @ k                           # 1 up to float32 rounding of k
    d = np.exp(np.float64(x["g"][0, 0]))
    b = np.float64(x["beta"][0, 0])
    S = x["state0"][0, 0].astype(np.float64)
    lhs = k @ s[0, 0]
    rhs = d * (k @ S) * (1 - b * k_norm2) + b * k_norm2 * x["v"][0, 0]
    assert _rel(lhs, rhs) < 1e-12


# ---------------------------------------------------------------- structure

def test_padding_leaves_state_bit_identical():
    """Tokens with g = 0, beta = 0 appended to a sequence change nothing, bit for bit."""
    wl, x = _small([13], dk=8, dv=8)
    o, s = _run(x)
    pad = 7
    y = {}
    for name in ("q", "k", "v"):
        extra = gi.normal(9, name + "pad", pad * x[name][0].size).astype(np.float32)
        y[name] = np.concatenate([x[name], extra.reshape((pad,) + x[name].shape[1:])])
    y["g"] = np.concatenate([x["g"], np.zeros((pad, 1), np.float32)])
    y["beta"] = np.concatenate([x["beta"], np.zeros((pad, 1), np.float32)])
    o2, s2 = oracle.recurrent(y["q"], y["k"], y["v"], y["g"], y["beta"], x["state0"],
                              np.array([0, 13 + pad], np.int32))
    assert np.array_equal(s2, s)
    assert np.array_equal(o2[:13], o)


def test_varlen_packed_equals_separate():
    """A packed batch equals each sequence run alone from its own initial state."""
    lengths = [5, 0, 19, 1, 40]
    wl, x = _small(lengths, hk=2, hv=2)
    o, s = _run(x)
    cu = x["cu_seqlens"]
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        o1, s1 = oracle.recurrent(x["q"][a:b], x["k"][a:b], x["v"][a:b], x["g"][a:b],
                                  x["beta"][a:b], x["state0"][n:n + 1],
                                  np.array([0, L], np.int32))
        assert np.array_equal(o1, o[a:b])
        assert np.array_equal(s1[0], s[n])


def test_grouped_heads_equal_duplicated_heads():
    """Hv = 2 Hk: q/k head i serves v heads 2i and 2i+1 (same as duplicating q/k heads)."""
    wl, x = _small([9, 14], hk=2, hv=4)
    o, s = _run(x)
    qd = np.repeat(x["q"], 2, axis=1)
    kd = np.repeat(x["k"], 2, axis=1)
    o2, s2 = oracle.recurrent(qd, kd, x["v"], x["g"], x["beta"], x["state0"], x["cu_seqlens"])
    assert np.array_equal(o, o2) and np.array_equal(s, s2)


def test_value_columns_are_independent():
    """Permuting the value columns of v and S0 permutes those of o and S_T."""
    wl, x = _small([21], dk=8, dv=6)
    o, s = _run(x)
    perm = np.array([3, 0, 5, 1, 4, 2])
    o2, s2 = oracle.recurrent(x["q"], x["k"], x["v"][..., perm], x["g"], x["beta"],
                              x["state0"][..., perm], x["cu_seqlens"])
    assert np.array_equal(o2, o[..., perm]) and np.array_equal(s2, s[..., perm])


def test_linear_in_values_and_state():
    """For fixed q, k, g, beta the layer is linear in (V, S0) jointly."""
    wl, x = _small([17], dk=6, dv=5)
    _, y = _small([17], dk=6, dv=5, seed=4)
    o1, s1 = _run(x)
    x2 = dict(x, v=y["v"], state0=y["state0"])
    o2, s2 = _run(x2)
    x3 = dict(x, v=(2.0 * x["v"].astype(np.float64) - 3.0 * y["v"]).astype(np.float32),
              state0=(2.0 * x["state0"].astype(np.float64) - 3.0 * y["state0"]).astype(np.float32))
    o3, s3 = _run(x3)
    assert _rel(o3, 2 * o1 - 3 * o2) < 1e-6   # float32 rounding of the combined inputs
    assert _rel(s3, 2 * s1 - 3 * s2) < 1e-6


def test_chain_subset_matches_full_run():
    """Computing a subset of (sequence, head) chains gives the same rows."""
    wl, x = _small([11, 30, 7], hk=1, hv=3)
    o, s = _run(x)
    pairs = [(1, 2), (0, 0), (2, 1)]
    o2, s2 = _run(x, pairs=pairs)
    cu = x["cu_seqlens"]
    for n, h in pairs:
        assert np.array_equal(o2[cu[n]:cu[n + 1], h], o[cu[n]:cu[n + 1], h])
        assert np.array_equal(s2[n, h], s[n, h])


# ---------------------------------------------------------------- inverse

@pytest.mark.parametrize("n", [1, 2, 3, 7, 16, 33, 64])
def test_triangular_inverse(n):
    """(I + N) X = I, and block doubling equals forward substitution."""
    N = np.tril(gi.normal(n, "tri", n * n).reshape(n, n), -1) * 0.5
    Xf = oracle.tril_inverse(N, "forward")
    Xd = oracle.tril_inverse(N, "doubling")
    M = np.eye(n) + N
    scale = max(1.0, np.max(np.abs(Xf)))
    assert np.max(np.abs(M @ Xf - np.eye(n))) < 1e-12 * scale
    assert np.max(np.abs(M @ Xd - np.eye(n))) < 1e-12 * scale
    assert np.max(np.abs(Xf - Xd)) < 1e-12 * scale
    assert np.allclose(np.triu(Xd, 1), 0) and np.allclose(np.diag(Xd), 1)


def test_neumann_product_cancels_on_correlated_keys():
    """The page's warning: with highly correlated keys the product series
    (I - N)(I + N^2)(I + N^4)... is exact in exact arithmetic but loses
    everything in fp16, while the doubling inverse stays accurate."""
    C, dk = 64, 128
    base = gi.normal(1, "base", dk)
    keys = base[None, :] + 0.05 * gi.normal(2, "jit", C * dk).reshape(C, dk)
    keys /= np.linalg.norm(keys, axis=1, keepdims=True)
    beta = np.full(C, 0.9)
    N = np.tril(beta[:, None] * (keys @ keys.T), -1)
    X = oracle.tril_inverse(N, "doubling")
    ref = np.linalg.inv(np.eye(C) + N)
    assert np.max(np.abs(X - ref)) / np.max(np.abs(ref)) < 1e-9
    # fp16 evaluation of the product series
    h = np.float16
    with np.errstate(all="ignore"):
        P = (np.eye(C) - N).astype(h)
        Nk = N.astype(h)
        for _ in range(6):
            Nk = (Nk.astype(np.float32) @ Nk.astype(np.float32)).astype(h)
            P = (P.astype(np.float32) @ (np.eye(C) + Nk.astype(np.float32))).astype(h)
        diff = np.abs(P.astype(np.float64) - ref)
    err = np.max(np.where(np.isfinite(diff), diff, np.inf)) / np.max(np.abs(ref))
    assert err > 0.1
