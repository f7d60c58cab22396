"""Pins of the oracle's input prologue and gated-RMSNorm epilogue (the steps around the
recurrence in the GDN block), each against a special case or an invariant that does not
restate the oracle: tap orientation through the conv FIFO, chained calls equal one call,
one-token calls equal one block, unit norms, closed-form gate values, zero gate, scale
invariance and constant rows of the norm."""
import numpy as np
import pytest

import oracle

W = oracle.CONV_WIDTH


def _rand_block(T, hk=1, hv=2, d=128, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    C = 2 * hk * d + hv * d
    return dict(
        q_raw=rng.standard_normal((T, hk, d)).astype(np.float32) * scale,
        k_raw=rng.standard_normal((T, hk, d)).astype(np.float32) * scale,
        v_raw=rng.standard_normal((T, hv, d)).astype(np.float32) * scale,
        a=rng.standard_normal((T, hv)).astype(np.float32),
        b=rng.standard_normal((T, hv)).astype(np.float32),
        conv_w=(rng.standard_normal((C, W)) * 0.5).astype(np.float32),
        A_log=(rng.standard_normal(hv) * 0.5).astype(np.float32),
        dt_bias=(rng.standard_normal(hv) * 0.5).astype(np.float32),
    ), C


def _silu(u):
    return u / (1.0 + np.exp(-u))


def _run(blk, state, cu):
    return oracle.prologue(blk["q_raw"], blk["k_raw"], blk["v_raw"], blk["a"], blk["b"],
                           blk["conv_w"], blk["A_log"], blk["dt_bias"], state, cu)


def _sub(blk, lo, hi):
    out = dict(blk)
    for name in ("q_raw", "k_raw", "v_raw", "a", "b"):
        out[name] = blk[name][lo:hi]
    return out


def test_single_tap_shifts_through_the_fifo():
    """conv weights with one 1 at tap i: y_t = SiLU(x_{t - (W-1) + i}), the first inputs
    coming from the state in order (oldest first)."""
    T = 7
    blk, C = _rand_block(T, seed=1)
    rng = np.random.default_rng(2)
    state = rng.standard_normal((1, C, W - 1)).astype(np.float32)
    cv0 = 2 * 128  # first v channel
    for tap in range(W):
        w = np.zeros((C, W), np.float32)
        w[:, tap] = 1.0
        blk["conv_w"] = w
        _, _, v, _, _, _ = _run(blk, state, [0, T])
        x = np.concatenate([state[0, cv0:].T.reshape(W - 1, 2, 128).astype(np.float64),
                            blk["v_raw"].astype(np.float64)])  # positions -(W-1) .. T-1
        shift = W - 1 - tap
        # libm and numpy exponentials may differ in the last bit
        assert np.allclose(v, _silu(x[W - 1 - shift:W - 1 - shift + T]), rtol=1e-14, atol=0)


def test_two_chained_calls_equal_one_call():
    T = 11
    blk, C = _rand_block(T, seed=3)
    rng = np.random.default_rng(4)
    state = rng.standard_normal((1, C, W - 1)).astype(np.float32)
    full = _run(blk, state, [0, T])
    for cut in (1, 2, 3, 5, 10):
        a = _run(_sub(blk, 0, cut), state, [0, cut])
        b = _run(_sub(blk, cut, T), a[5].astype(np.float32), [0, T - cut])
        for i in range(5):
            assert np.array_equal(np.concatenate([a[i], b[i]]), full[i]), (cut, i)
        assert np.array_equal(b[5], full[5])


def test_one_token_calls_equal_one_block():
    T = 6
    blk, C = _rand_block(T, seed=5)
    full = _run(blk, None, [0, T])
    state = None
    for t in range(T):
        step = _run(_sub(blk, t, t + 1), state, None)  # one token per sequence
        for i in range(5):
            assert np.array_equal(step[i][0], full[i][t]), (t, i)
        state = step[5].astype(np.float32)
    assert np.array_equal(state, full[5].astype(np.float32))


def test_state_out_holds_the_last_raw_inputs():
    blk, C = _rand_block(5, seed=6)
    rng = np.random.default_rng(7)
    state = rng.standard_normal((2, C, W - 1)).astype(np.float32)
    *_, cso = _run(blk, state, [0, 1, 5])  # sequences of 1 and 4 tokens
    x = np.concatenate([blk["q_raw"].reshape(5, -1), blk["k_raw"].reshape(5, -1),
                        blk["v_raw"].reshape(5, -1)], axis=1)  # [T, C]
    assert np.array_equal(cso[1], x[2:5].T)                    # last three of sequence 1
    assert np.array_equal(cso[0], np.concatenate([state[0, :, 1:], x[0:1].T], axis=1))


def test_q_k_rows_have_unit_norm_and_zero_stays_zero():
    blk, C = _rand_block(4, seed=8)
    q, k, *_ = _run(blk, None, [0, 4])
    nq, nk = np.linalg.norm(q, axis=-1), np.linalg.norm(k, axis=-1)
    assert np.all(np.abs(nq - 1) < 1e-6) and np.all(np.abs(nk - 1) < 1e-6)
    zero = {n: np.zeros_like(x) for n, x in blk.items()}
    zero["conv_w"] = blk["conv_w"]
    q0, k0, v0, *_ = _run(zero, None, [0, 4])
    assert not q0.any() and not k0.any() and not v0.any()


def test_gates_closed_forms():
    blk, _ = _rand_block(3, seed=9)
    A_log, dt = blk["A_log"].astype(np.float64), blk["dt_bias"].astype(np.float64)
    blk["a"] = np.stack([-blk["dt_bias"], np.full(2, 40, np.float32) - blk["dt_bias"],
                         np.full(2, -40, np.float32) - blk["dt_bias"]])
    blk["b"] = np.array([[0, 0], [40, 40], [-40, -40]], np.float32)
    _, _, _, g, beta, _ = _run(blk, None, [0, 3])
    a = blk["a"].astype(np.float64)
    assert np.allclose(g[0], -np.exp(A_log) * np.log(2.0), rtol=1e-15, atol=0)
    assert np.allclose(g[1], -np.exp(A_log) * (a[1] + dt), rtol=1e-12)   # softplus(u) ~ u
    assert np.all(g[2] < 0) and np.all(g[2] > -np.exp(A_log) * 1e-16)     # ~ e^-40
    assert np.array_equal(beta[0], [0.5, 0.5])
    assert np.all(beta[1] == 1.0) and np.all(beta[2] < 1e-17)


def test_gated_rmsnorm_pins():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((5, 128)).astype(np.float32)
    w = rng.standard_normal(128).astype(np.float32)
    z = rng.standard_normal((5, 128)).astype(np.float32)
    # the gate SiLU(0) = 0 silences the row
    assert not oracle.gated_rmsnorm(o, np.zeros_like(z), w).any()
    # scale invariance (eps = 0) and odd symmetry in o
    y = oracle.gated_rmsnorm(o, z, w, eps=0.0)
    assert np.allclose(oracle.gated_rmsnorm(o * 8, z, w, eps=0.0), y, rtol=1e-14, atol=0)
    assert np.allclose(oracle.gated_rmsnorm(-o, z, w, eps=0.0), -y, rtol=1e-14, atol=0)
    # a constant row c has rms |c|: y = sign(c) * w * SiLU(z) (a sum in place of the mean
    # would give sign(c) / sqrt(128) instead)
    c = np.full((2, 128), -2.5, np.float32)
    yc = oracle.gated_rmsnorm(c, z[:2], w, eps=0.0)
    assert np.allclose(yc, -w.astype(np.float64) * _silu(z[:2].astype(np.float64)), rtol=1e-14)
    # eps enters inside the root: o / sqrt(mean o^2 + eps)
    ye = oracle.gated_rmsnorm(c, z[:2], w, eps=6.25 * 3)
    assert np.allclose(ye, yc / 2.0, rtol=1e-14)
