"""Seeded synthetic inputs for the gated delta-rule layer.

This module is shared by the float64 oracle tests and by the CUDA path's
tests and benchmark, so that both sides see the same bytes.  It holds none
of the layer's own arithmetic: only

* a counter-based random stream (splitmix64's output mix applied to
  ``key + (i + 1) * 0x9E3779B97F4A7C15``, i the element counter),
* the Box-Muller transform to N(0, 1),
* the input recipe of the workloads (q, k L2-normalised per token and
  head, g = -softplus(x), beta = sigmoid(x), S0 = scale * N(0, 1), varlen
  lengths drawn uniformly), and
* rounding to the storage dtype (float64 -> float32 round-to-nearest-even,
  then float32 -> bfloat16 round-to-nearest-even on the bit pattern).

Every tensor is keyed by (seed, tag, element index), so a tensor's values
do not depend on which other tensors were drawn or in what order.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_BLOCK = 1 << 22


def _mix(z: np.ndarray, t: Optional[np.ndarray] = None) -> np.ndarray:
    """splitmix64 output function on an array of uint64 (wrapping arithmetic, in place).

    `t` is an optional scratch array of at least z's size."""
    t = np.empty_like(z) if t is None else t[:z.size]
    np.right_shift(z, np.uint64(30), out=t)
    z ^= t
    z *= _M1
    np.right_shift(z, np.uint64(27), out=t)
    z ^= t
    z *= _M2
    np.right_shift(z, np.uint64(31), out=t)
    z ^= t
    return z


def _tag_hash(tag: str) -> int:
    """64-bit FNV-1a of the tag string."""
    h = 0xCBF29CE484222325
    for b in tag.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def _key(seed: int, tag: str) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF], np.uint64)
        s ^= np.uint64(_tag_hash(tag))
        return _mix(s)[0]


def raw_u64(seed: int, tag: str, n: int, offset: int = 0) -> np.ndarray:
    """Counters offset .. offset+n-1 of the stream (seed, tag) as uint64."""
    key = _key(seed, tag)
    out = np.empty(n, np.uint64)
    B = max(1, min(_BLOCK, n))
    base = np.arange(1, B + 1, dtype=np.int64).view(np.uint64)
    tmp = np.empty(B, np.uint64)
    with np.errstate(over="ignore"):
        for s in range(0, n, B):
            c = out[s:min(n, s + B)]
            np.add(base[:len(c)], np.uint64(offset + s), out=c)
            c *= _GAMMA
            c += key
            _mix(c, tmp)
    return out


def uniform(seed: int, tag: str, n: int) -> np.ndarray:
    """n uniforms in [0, 1) with 53 random bits each."""
    z = raw_u64(seed, tag, n) >> np.uint64(11)
    return z.view(np.int64).astype(np.float64) * 2.0 ** -53


def normal(seed: int, tag: str, n: int) -> np.ndarray:
    """n standard normals by Box-Muller: elements 2j, 2j+1 come from counters 2j, 2j+1.

    u1 = (bits + 1) * 2**-53 in (0, 1] from counter 2j, u2 = bits * 2**-53
    in [0, 1) from counter 2j+1 (bits: the top 53 bits of the mixed word);
    element 2j = sqrt(-2 ln u1) cos(2 pi u2), element 2j+1 the sine.
    """
    pairs = (n + 1) // 2
    out = np.empty(2 * pairs, np.float64)
    key = _key(seed, tag)
    B = max(1, min(_BLOCK, pairs))
    base = np.arange(1, 2 * B + 1, dtype=np.int64).view(np.uint64)
    cbuf = np.empty(2 * B, np.uint64)
    tbuf = np.empty(2 * B, np.uint64)
    fbuf = np.empty(2 * B, np.float64)
    r = np.empty(B, np.float64)
    th = np.empty(B, np.float64)
    tmp = np.empty(B, np.float64)
    with np.errstate(over="ignore"):
        for s in range(0, pairs, B):
            m = min(B, pairs - s)
            c = cbuf[:2 * m]
            np.add(base[:2 * m], np.uint64(2 * s), out=c)
            c *= _GAMMA
            c += key
            _mix(c, tbuf)
            c >>= np.uint64(11)
            f = fbuf[:2 * m]
            np.copyto(f, c.view(np.int64), casting="unsafe")
            f *= 2.0 ** -53
            rr, tt, xx = r[:m], th[:m], tmp[:m]
            np.add(f[0::2], 2.0 ** -53, out=rr)
            np.log(rr, out=rr)
            rr *= -2.0
            np.sqrt(rr, out=rr)
            np.multiply(f[1::2], 2.0 * np.pi, out=tt)
            np.cos(tt, out=xx)
            np.multiply(rr, xx, out=out[2 * s:2 * (s + m):2])
            np.sin(tt, out=xx)
            np.multiply(rr, xx, out=out[2 * s + 1:2 * (s + m):2])
    return out[:n]


# ---------------------------------------------------------------- rounding

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    # finite inputs only: the sum stays below 2**32 for every finite pattern
    r = (b >> np.uint32(16)) & np.uint32(1)
    r += np.uint32(0x7FFF)
    r += b
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str):
    """Round float64 values to the storage dtype.

    Returns (values as float32, storage array): for "f32" both are the same
    float32 array; for "bf16" the storage array holds the uint16 bit patterns.
    """
    x32 = x.astype(np.float32)
    if dtype == "f32":
        return x32, x32
    if dtype == "bf16":
        bits = f32_to_bf16_bits(x32)
        return bf16_bits_to_f32(bits), bits
    raise ValueError(dtype)


# ---------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    """Shape and recipe of one synthetic workload."""
    name: str
    lengths: List[int]          # tokens per sequence
    num_k_heads: int            # heads of q and k
    num_v_heads: int            # heads of v, g, beta, state, o
    dk: int = 128
    dv: int = 128
    chunk: int = 64
    dtype: str = "bf16"         # storage dtype of q, k, v and o
    s0_scale: Optional[float] = 0.1   # None: zero initial state
    steps: int = 1              # decode: consecutive one-token steps

    @property
    def num_seqs(self) -> int:
        return len(self.lengths)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)


def varlen_lengths(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """n lengths uniform in [lo, hi]: lo + (u64 mod (hi - lo + 1))."""
    u = raw_u64(seed, "lens", n)
    return [int(lo + int(x) % (hi - lo + 1)) for x in u]


def chunk_vs_sequential_fp32() -> Workload:
    """fp32, one sequence, one head, T=64, chunk 16, zero initial state."""
    return Workload("chunk_vs_sequential_fp32_T64_C16", [64], 1, 1, chunk=16,
                    dtype="f32", s0_scale=None)


def decode_b32_h16(steps: int = 100) -> Workload:
    """Decode: 32 sequences x 16 heads, one token each per step, 100 steps."""
    return Workload("decode_B32_H16", [1] * 32, 16, 16, chunk=64, dtype="bf16",
                    s0_scale=0.1, steps=steps)


def prefill_t4096_h16() -> Workload:
    """Single-sequence prefill: H=16, T=4096, chunk 64, bf16 q/k/v."""
    return Workload("prefill_B1_H16_T4096_C64", [4096], 16, 16, chunk=64, dtype="bf16",
                    s0_scale=0.1)


def long_t65536_h2() -> Workload:
    """Few heads and one long sequence: H=2, T=65,536, chunk 64, bf16 q/k/v."""
    return Workload("prefill_B1_H2_T65536_C64", [65536], 2, 2, chunk=64, dtype="bf16",
                    s0_scale=0.1)


def varlen_8seq_hk16_hv32(seed: int = 0) -> Workload:
    """Packed varlen prefill: 8 sequences, lengths U[256, 8192], Hk=16, Hv=32."""
    return Workload("varlen_N8_Hk16_Hv32_C64", varlen_lengths(seed, 8, 256, 8192), 16, 32,
                    chunk=64, dtype="bf16", s0_scale=0.1)


def verify_b128_h32() -> Workload:
    """Draft-verify blocks: 128 sequences x 32 heads, T=16, chunk 16."""
    return Workload("verify_B128_H32_T16_C16", [16] * 128, 32, 32, chunk=16, dtype="bf16",
                    s0_scale=0.1)


def all_workloads() -> List[Workload]:
    return [chunk_vs_sequential_fp32(), decode_b32_h16(), prefill_t4096_h16(),
            varlen_8seq_hk16_hv32(), verify_b128_h32()]


# ---------------------------------------------------------------- tensors

def _unit_rows(x: np.ndarray) -> np.ndarray:
    """L2-normalise the last axis in float64 (input recipe for q and k)."""
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True))


def make_inputs(wl: Workload, seed: int = 0, step: Optional[int] = None,
                gate_scale: float = 1.0) -> dict:
    """Draw one batch of inputs for `wl`.

    Returns a dict of numpy arrays:
      q, k       float32 [T, Hk, dk]   (values exactly representable in wl.dtype)
      v          float32 [T, Hv, dv]
      q_st, k_st, v_st  storage arrays (uint16 bf16 bits, or the float32 arrays)
      g, beta    float32 [T, Hv]
      state0     float32 [N, Hv, dk, dv] or None
      cu_seqlens int32 [N+1]
    `step` selects a fresh draw of the per-token tensors (decode steps);
    the initial state does not depend on it.  `gate_scale` multiplies g
    (slow-decay stress inputs use 0.01).
    """
    T, Hk, Hv, dk, dv = wl.total_tokens, wl.num_k_heads, wl.num_v_heads, wl.dk, wl.dv
    sfx = "" if step is None else "/step%d" % step
    q = _unit_rows(normal(seed, "q" + sfx, T * Hk * dk).reshape(T, Hk, dk))
    k = _unit_rows(normal(seed, "k" + sfx, T * Hk * dk).reshape(T, Hk, dk))
    v = normal(seed, "v" + sfx, T * Hv * dv).reshape(T, Hv, dv)
    xg = normal(seed, "g" + sfx, T * Hv).reshape(T, Hv)
    xb = normal(seed, "beta" + sfx, T * Hv).reshape(T, Hv)
    g = (-gate_scale * np.logaddexp(0.0, xg)).astype(np.float32)      # -softplus
    beta = (1.0 / (1.0 + np.exp(-xb))).astype(np.float32)             # sigmoid
    out = {}
    out["q"], out["q_st"] = round_to(q, wl.dtype)
    out["k"], out["k_st"] = round_to(k, wl.dtype)
    out["v"], out["v_st"] = round_to(v, wl.dtype)
    out["g"], out["beta"] = g, beta
    if wl.s0_scale is None:
        out["state0"] = None
    else:
        s0 = wl.s0_scale * normal(seed, "state0", wl.num_seqs * Hv * dk * dv)
        out["state0"] = s0.astype(np.float32).reshape(wl.num_seqs, Hv, dk, dv)
    out["cu_seqlens"] = wl.cu_seqlens()
    return out


def make_block_inputs(wl: Workload, seed: int = 0, step: Optional[int] = None,
                      conv_width: int = 4) -> dict:
    """Draw the inputs of the block steps around the layer for `wl`: the raw projections
    before the input prologue and the gate projection after the layer.

    Returns a dict of numpy arrays (storage arrays *_st as in make_inputs):
      q_raw, k_raw  float32 [T, Hk, dk]  N(0, 1), exactly representable in wl.dtype
      v_raw         float32 [T, Hv, dv]  N(0, 1)
      a, b          float32 [T, Hv]      N(0, 1)
      conv_w        float32 [C, W]       0.5 N(0, 1), C = 2 Hk dk + Hv dv
      A_log         float32 [Hv]         log A, A uniform in [1, 16]
      dt_bias       float32 [Hv]         log(e^dt - 1), dt log-uniform in [1e-3, 1e-1]
      conv_state0   float32 [N, W-1, C]  N(0, 1) (oldest input first), in wl.dtype
      z             float32 [T, Hv, dv]  N(0, 1), in wl.dtype
      norm_w        float32 [dv]         1 + 0.1 N(0, 1)
      cu_seqlens    int32 [N+1]
    `step` selects a fresh draw of the per-token tensors; the weights and the initial
    conv state do not depend on it."""
    T, Hk, Hv, dk, dv = wl.total_tokens, wl.num_k_heads, wl.num_v_heads, wl.dk, wl.dv
    C = 2 * Hk * dk + Hv * dv
    sfx = "" if step is None else "/step%d" % step
    out = {}
    out["q_raw"], out["q_raw_st"] = round_to(normal(seed, "q_raw" + sfx, T * Hk * dk).reshape(T, Hk, dk), wl.dtype)
    out["k_raw"], out["k_raw_st"] = round_to(normal(seed, "k_raw" + sfx, T * Hk * dk).reshape(T, Hk, dk), wl.dtype)
    out["v_raw"], out["v_raw_st"] = round_to(normal(seed, "v_raw" + sfx, T * Hv * dv).reshape(T, Hv, dv), wl.dtype)
    out["a"] = normal(seed, "a" + sfx, T * Hv).reshape(T, Hv).astype(np.float32)
    out["b"] = normal(seed, "b" + sfx, T * Hv).reshape(T, Hv).astype(np.float32)
    out["conv_w"] = (0.5 * normal(seed, "conv_w", C * conv_width)).reshape(C, conv_width).astype(np.float32)
    out["A_log"] = np.log(1.0 + 15.0 * uniform(seed, "A", Hv)).astype(np.float32)
    dt = np.exp(np.log(1e-3) + (np.log(1e-1) - np.log(1e-3)) * uniform(seed, "dt", Hv))
    out["dt_bias"] = np.log(np.expm1(dt)).astype(np.float32)
    cs = normal(seed, "conv_state0", wl.num_seqs * (conv_width - 1) * C)
    out["conv_state0"], out["conv_state0_st"] = round_to(cs.reshape(wl.num_seqs, conv_width - 1, C), wl.dtype)
    out["z"], out["z_st"] = round_to(normal(seed, "z" + sfx, T * Hv * dv).reshape(T, Hv, dv), wl.dtype)
    out["norm_w"] = (1.0 + 0.1 * normal(seed, "norm_w", dv)).astype(np.float32)
    out["cu_seqlens"] = wl.cu_seqlens()
    return out
