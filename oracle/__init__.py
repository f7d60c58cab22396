"""Float64 CPU oracle of the gated delta-rule layer (ctypes binding).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg import this module; the product path never
does.  It shares no code with the CUDA library.

The arithmetic lives in ``gdn_oracle.c`` (plain C, double precision); see
its header for what each function follows ("Qwen3.5-9B-npu" model card,
section "How it works": the per-token recurrence, the chunkwise form,
token_valid padding and the block-doubling triangular inverse; and the steps
around the recurrence in the GDN block: the input prologue -- causal conv FIFO,
SiLU, q/k L2 norm, gates -- and the gated RMSNorm output epilogue).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgdn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.gdn_oracle_recurrent.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, I]
        lib.gdn_oracle_recurrent.restype = I
        lib.gdn_oracle_recurrent_deltas.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I]
        lib.gdn_oracle_recurrent_deltas.restype = I
        lib.gdn_oracle_chunked.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, I, I, I, I]
        lib.gdn_oracle_chunked.restype = I
        lib.gdn_oracle_tril_inverse.argtypes = [I, P, P, I]
        lib.gdn_oracle_tril_inverse.restype = I
        D = ctypes.c_double
        lib.gdn_oracle_prologue.argtypes = [I, I, I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, D,
                                            P, P, P, P, P, P]
        lib.gdn_oracle_prologue.restype = I
        lib.gdn_oracle_gated_rmsnorm.argtypes = [I, I, P, P, P, D, P]
        lib.gdn_oracle_gated_rmsnorm.restype = I
        _lib = lib
    return _lib


def _f32(x):
    return None if x is None else np.ascontiguousarray(x, np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _prep(q, k, v, g, beta, state_in, cu_seqlens, pairs):
    q, k, v, g, beta, state_in = map(_f32, (q, k, v, g, beta, state_in))
    T, hk, dk = q.shape
    _, hv, dv = v.shape
    assert k.shape == (T, hk, dk) and v.shape[0] == T
    assert g.shape == (T, hv) and beta.shape == (T, hv)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    n = len(cu) - 1
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    if state_in is not None:
        assert state_in.shape == (n, hv, dk, dv)
    pr = None if pairs is None else np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    o = np.zeros((T, hv, dv), np.float64)
    s_out = np.zeros((n, hv, dk, dv), np.float64)
    return q, k, v, g, beta, state_in, cu, pr, o, s_out, (n, hk, hv, dk, dv)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def recurrent(q, k, v, g, beta, state_in, cu_seqlens,
              pairs: Optional[Sequence[Tuple[int, int]]] = None,
              threads: Optional[int] = None):
    """Per-token gated delta rule in float64.

    Returns (o [T, Hv, dv], state_out [N, Hv, dk, dv]) as float64.  With
    `pairs`, only those (sequence, v-head) chains are computed; the other
    entries of both outputs stay zero.
    """
    q, k, v, g, beta, s_in, cu, pr, o, s_out, (n, hk, hv, dk, dv) = \
        _prep(q, k, v, g, beta, state_in, cu_seqlens, pairs)
    rc = _load().gdn_oracle_recurrent(
        n, hk, hv, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s_in),
        _ptr(o), _ptr(s_out), _ptr(pr), 0 if pr is None else len(pr),
        threads or default_threads())
    if rc:
        raise RuntimeError("gdn_oracle_recurrent failed (%d)" % rc)
    return o, s_out


def recurrent_deltas(q, k, v, g, beta, state_in, cu_seqlens, threads: Optional[int] = None):
    """The per-token rule in float64, also returning each token's delta
    delta_t = beta_t (v_t - S'^T k_t) (S' the decayed state before the write).

    Returns (o [T, Hv, dv], state_out [N, Hv, dk, dv], delta [T, Hv, dv]), float64."""
    q, k, v, g, beta, s_in, cu, _, o, s_out, (n, hk, hv, dk, dv) = \
        _prep(q, k, v, g, beta, state_in, cu_seqlens, None)
    delta = np.zeros_like(o)
    rc = _load().gdn_oracle_recurrent_deltas(
        n, hk, hv, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s_in),
        _ptr(o), _ptr(s_out), _ptr(delta), threads or default_threads())
    if rc:
        raise RuntimeError("gdn_oracle_recurrent_deltas failed (%d)" % rc)
    return o, s_out, delta


def state_after_prefix(q, k, v, g, beta, state_in, cu_seqlens, prefix_len,
                       threads: Optional[int] = None):
    """The state of every (sequence, v-head) after the first prefix_len[n] tokens of
    sequence n (clamped to its length), by running the per-token rule over those
    tokens only.  Returns [N, Hv, dk, dv] float64."""
    cu = np.asarray(cu_seqlens, np.int64)
    n = len(cu) - 1
    keep = []
    lens = []
    for s in range(n):
        a = int(min(max(int(prefix_len[s]), 0), cu[s + 1] - cu[s]))
        keep.extend(range(int(cu[s]), int(cu[s]) + a))
        lens.append(a)
    keep = np.asarray(keep, np.int64)
    cu_p = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    sub = [np.asarray(x)[keep] for x in (q, k, v, g, beta)]
    _, s_out = recurrent(*sub, state_in, cu_p, threads=threads)
    return s_out


def chunked(q, k, v, g, beta, state_in, cu_seqlens, chunk: int, solve: str = "forward",
            pairs: Optional[Sequence[Tuple[int, int]]] = None,
            threads: Optional[int] = None):
    """Chunkwise-parallel closed form in float64 (solve: "forward" or "doubling")."""
    q, k, v, g, beta, s_in, cu, pr, o, s_out, (n, hk, hv, dk, dv) = \
        _prep(q, k, v, g, beta, state_in, cu_seqlens, pairs)
    rc = _load().gdn_oracle_chunked(
        n, hk, hv, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s_in),
        _ptr(o), _ptr(s_out), _ptr(pr), 0 if pr is None else len(pr), int(chunk),
        {"forward": 0, "doubling": 1}[solve], threads or default_threads())
    if rc:
        raise RuntimeError("gdn_oracle_chunked failed (%d)" % rc)
    return o, s_out


def tril_inverse(Nm: np.ndarray, method: str = "forward") -> np.ndarray:
    """(I + tril(Nm, -1))^-1 in float64 by forward substitution or block doubling."""
    Nm = np.ascontiguousarray(Nm, np.float64)
    n = Nm.shape[0]
    X = np.zeros((n, n), np.float64)
    rc = _load().gdn_oracle_tril_inverse(n, _ptr(Nm), _ptr(X), {"forward": 0, "doubling": 1}[method])
    if rc:
        raise RuntimeError("gdn_oracle_tril_inverse failed")
    return X


CONV_WIDTH = 4  # the short causal convolution of the input prologue


def prologue(q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in, cu_seqlens,
             eps: float = 1e-6, conv_width: int = CONV_WIDTH):
    """Input prologue in float64: causal conv (width W) over the raw q | k | v channels with
    the per-sequence FIFO state, SiLU, q/k L2 norm, gates.

    Shapes: q_raw, k_raw [T, Hk, dk]; v_raw [T, Hv, dv]; a, b [T, Hv]; conv_w [C, W] with
    C = 2 Hk dk + Hv dv; A_log, dt_bias [Hv]; conv_state_in [N, C, W - 1] or None;
    cu_seqlens [N + 1] or None (one token per sequence).
    Returns q, k, v, g, beta, conv_state_out (float64)."""
    q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, csi = map(
        _f32, (q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in))
    T, hk, dk = q_raw.shape
    _, hv, dv = v_raw.shape
    C = 2 * hk * dk + hv * dv
    assert conv_w.shape == (C, conv_width) and a.shape == (T, hv) and b.shape == (T, hv)
    if cu_seqlens is None:
        n, cu = T, None
    else:
        cu = np.ascontiguousarray(cu_seqlens, np.int32)
        n = len(cu) - 1
        assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    if csi is not None:
        assert csi.shape == (n, C, conv_width - 1)
    q = np.zeros((T, hk, dk)); k = np.zeros((T, hk, dk)); v = np.zeros((T, hv, dv))
    g = np.zeros((T, hv)); beta = np.zeros((T, hv))
    cso = np.zeros((n, C, conv_width - 1))
    rc = _load().gdn_oracle_prologue(n, T, hk, hv, dk, dv, conv_width, _ptr(cu), _ptr(q_raw),
                                     _ptr(k_raw), _ptr(v_raw), _ptr(a), _ptr(b), _ptr(conv_w),
                                     _ptr(A_log), _ptr(dt_bias), _ptr(csi), float(eps), _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cso))
    if rc:
        raise RuntimeError("gdn_oracle_prologue failed (%d)" % rc)
    return q, k, v, g, beta, cso


def gated_rmsnorm(o, z, weight, eps: float = 1e-6):
    """Gated RMSNorm of each row of the last axis in float64:
    o / sqrt(mean(o^2) + eps) * weight * SiLU(z)."""
    o, z, weight = map(_f32, (o, z, weight))
    d = o.shape[-1]
    assert z.shape == o.shape and weight.shape == (d,)
    y = np.zeros(o.shape, np.float64)
    rc = _load().gdn_oracle_gated_rmsnorm(int(o.size // d), d, _ptr(o), _ptr(z), _ptr(weight),
                                          float(eps), _ptr(y))
    if rc:
        raise RuntimeError("gdn_oracle_gated_rmsnorm failed")
    return y
