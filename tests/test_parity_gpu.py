"""GPU parity: libgdn's CUDA path against the float64 oracle on the same seeded inputs.

Tolerances (max |x - ref| / rms(ref) over the whole tensor, o and the final state
separately): 1e-4 for fp32 q/k/v, 2e-2 for bf16 q/k/v with fp32 g/beta/state.

bf16 outputs: o has heavy tails (max/rms ~16 on the T=4096 workload), so rounding
even the exact result to bf16 already moves its largest entries by ~3e-2 of the rms.
The bound is therefore applied to the kernel's fp32 result (o_fp32 = 1), and the
stored bf16 o of the same computation must be exactly its round-to-nearest-even
rounding (bit for bit), with the state bit-identical between the two runs.
"""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import device_inputs, gpu_prefill, half_ulp_bf16, rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
# the schedules of the bf16 chunked pass (f32 q/k/v: the fp32 kernel, or the token loop)
ALGOS = {"two_pass": 1, "single_pass": 2, "tensor_memory": 3, "recurrent": 4, "two_pass_tensor": 5}
# schedules built for every block length (tensor_memory: 64-token blocks only)
ALGOS_ANY_C = ["two_pass", "single_pass", "recurrent"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def _oracle(x, pairs=None):
    return oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                            x["cu_seqlens"], pairs=pairs)


def _check(o, s, o_ref, s_ref, dtype, what=""):
    eo, es = rel_err(o, o_ref), rel_err(s, s_ref)
    assert np.isfinite(o).all() and np.isfinite(s).all(), what
    assert eo <= TOL[dtype], "%s o err %.3g" % (what, eo)
    assert es <= TOL[dtype], "%s state err %.3g" % (what, es)
    return eo, es


def _run_and_check(x, wl, o_ref, s_ref, what="", **kw):
    """Chunked GPU pass checked against the oracle; for bf16 also the stored-output rounding."""
    import torch
    if wl.dtype == "f32":
        o, s, _ = gpu_prefill(x, wl, **kw)
        return _check(o, s, o_ref, s_ref, "f32", what)
    o32, s32, d32 = gpu_prefill(x, wl, o_fp32=True, **kw)
    err = _check(o32, s32, o_ref, s_ref, "bf16", what)
    o16, s16, d16 = gpu_prefill(x, wl, **kw)
    assert np.array_equal(s16, s32), what + ": state differs between output dtypes"
    assert torch.equal(d16["o_raw"], d32["o_raw"].to(torch.bfloat16)), what + ": bf16 o != RNE(fp32 o)"
    # the literal bound on the stored bf16 output, beyond its own rounding
    excess = np.maximum(np.abs(o16 - o_ref) - half_ulp_bf16(o16), 0.0)
    assert excess.max() / np.sqrt(np.mean(o_ref ** 2)) <= TOL["bf16"], what
    return err


# ------------------------------------------------------------------ chunked prefill

def test_chunk_vs_sequential_fp32_T64_C16():
    wl = gi.chunk_vs_sequential_fp32()
    x = gi.make_inputs(wl)
    o, s, _ = gpu_prefill(x, wl, state_in=False)
    o_ref, s_ref = _oracle(x)
    _check(o, s, o_ref, s_ref, "f32")


SMALL_CASES = [([1], 1, 1), ([2], 1, 1), ([15], 1, 2), ([16], 2, 2), ([17], 1, 1),
               ([63, 64, 65], 1, 2), ([200, 3, 129], 2, 4), ([0, 70, 0, 1], 1, 1)]


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("lengths,hk,hv", SMALL_CASES)
def test_prefill_small_shapes_f32(chunk, lengths, hk, hv):
    wl = gi.Workload("small", lengths, hk, hv, chunk=chunk, dtype="f32", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=len(lengths) + chunk)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "T=%s C=%d" % (lengths, chunk))


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("lengths,hk,hv", SMALL_CASES)
def test_prefill_small_shapes_bf16(algo, chunk, lengths, hk, hv):
    if algo not in ALGOS_ANY_C and chunk != 64:
        pytest.skip("64-token blocks only")
    wl = gi.Workload("small", lengths, hk, hv, chunk=chunk, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=len(lengths) + chunk)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "T=%s C=%d %s" % (lengths, chunk, algo),
                   algo=ALGOS[algo])


@pytest.mark.parametrize("dtype,algo", [("f32", None), ("bf16", "two_pass"),
                                        ("bf16", "single_pass"), ("bf16", "tensor_memory"),
                                        ("bf16", "recurrent"), ("f32", "recurrent"),
                                        ("bf16", "two_pass_tensor")])
def test_prefill_zero_initial_state_and_in_place(dtype, algo):
    kw = {"algo": ALGOS[algo]} if algo else {}
    chunk = 32 if algo in (None, *ALGOS_ANY_C) else 64
    wl = gi.Workload("small", [37, 90], 2, 2, chunk=chunk, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=7)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "in place", inplace=True, **kw)
    x0 = dict(x, state0=None)
    o_ref0, s_ref0 = _oracle(x0)
    _run_and_check(x0, wl, o_ref0, s_ref0, "zero state", state_in=False, **kw)


@pytest.mark.parametrize("verify", [False, True])
@pytest.mark.parametrize("inplace", [False, True])
def test_single_pass_16_token_blocks_many_units(verify, inplace):
    """16-token blocks on the single-pass schedule: each CTA walks several (sequence, head)
    units (400 here, more than one per SM) and prefetches the next unit's first block and
    state while it computes; empty sequences among them pass their state through."""
    if verify and inplace:
        pytest.skip("the verify block keeps its snapshot: no in-place state")
    lengths = [(0, 1, 16, 17, 40, 5, 0, 33)[i % 8] for i in range(200)]
    wl = gi.Workload("many16", lengths, 1, 2, chunk=16, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=21)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "many units", inplace=inplace, verify=verify,
                   algo=ALGOS["single_pass"])


@pytest.mark.parametrize("algo", list(ALGOS))
def test_prefill_slow_decay_bf16(algo):
    """g = -0.01 softplus(.): the state carries across many blocks."""
    wl = gi.Workload("slow", [1000], 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=11, gate_scale=0.01)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "slow decay", algo=ALGOS[algo])


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("chunk", [16, 64])
def test_prefill_strong_decay_bf16(algo, chunk):
    """g ~ -28 per token: the in-block decays underflow to zero within a few tokens, which
    only the exp of a difference of cumsums survives (a product of e^G_t and e^-G_j would
    give 0 * inf); every schedule must stay finite and match the oracle."""
    if algo not in ALGOS_ANY_C and chunk != 64:
        pytest.skip("64-token blocks only")
    wl = gi.Workload("strong", [200, 37, 64], 1, 2, chunk=chunk, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=13, gate_scale=40.0)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "strong decay C=%d" % chunk, algo=ALGOS[algo])


@pytest.mark.parametrize("algo", [None, "recurrent"])
@pytest.mark.parametrize("chunk", [16, 64])
def test_prefill_strong_decay_f32(algo, chunk):
    """As above for fp32 q/k/v (the fp32 chunk kernel, and the token loop)."""
    kw = {"algo": ALGOS[algo]} if algo else {}
    wl = gi.Workload("strong", [200, 37, 64], 1, 2, chunk=chunk, dtype="f32", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=14, gate_scale=40.0)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "strong decay f32 C=%d" % chunk, **kw)


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("hk,hv", [(1, 8), (2, 16)])
def test_prefill_wide_head_groups_bf16(algo, hk, hv):
    """8 v-heads per k-head: every v-head of a group reads the same q, k rows (h / 8)."""
    wl = gi.Workload("gqa8", [90, 1, 130], hk, hv, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=17 + hv)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "Hk=%d Hv=%d" % (hk, hv), algo=ALGOS[algo])


@pytest.mark.parametrize("algo", list(ALGOS))
def test_prefill_T4096_H16_full(algo):
    wl = gi.prefill_t4096_h16()
    x = gi.make_inputs(wl)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "T=4096", algo=ALGOS[algo])


def test_many_heads_take_the_single_pass_schedule_by_default():
    """AUTO: at least GDN_SINGLE_PASS_MIN_HEADS (sequence, head) pairs -> single pass,
    which is bit-identical to asking for it."""
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("many", [5, 40, 17, 64] * 8, 2, 4, chunk=32, dtype="bf16", s0_scale=0.1)
    assert wl.num_seqs * wl.num_v_heads >= gdn.GDN_SINGLE_PASS_MIN_HEADS
    x = gi.make_inputs(wl, seed=21)
    o_ref, s_ref = _oracle(x)
    _run_and_check(x, wl, o_ref, s_ref, "many heads")
    o_a, s_a, _ = gpu_prefill(x, wl, o_fp32=True)
    o_1, s_1, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS["single_pass"])
    assert np.array_equal(o_a, o_1) and np.array_equal(s_a, s_1)
    # 64-token blocks: the tensor-memory schedule
    wl64 = gi.Workload("many", [5, 40, 17, 64, 130] * 8, 2, 4, chunk=64, dtype="bf16", s0_scale=0.1)
    x64 = gi.make_inputs(wl64, seed=22)
    o_a, s_a, _ = gpu_prefill(x64, wl64, o_fp32=True)
    o_t, s_t, _ = gpu_prefill(x64, wl64, o_fp32=True, algo=ALGOS["tensor_memory"])
    assert np.array_equal(o_a, o_t) and np.array_equal(s_a, s_t)


_VARLEN = {}


def _varlen():
    """The packed varlen workload and its float64 oracle (all 256 chains, computed once)."""
    if not _VARLEN:
        wl = gi.varlen_8seq_hk16_hv32()
        x = gi.make_inputs(wl)
        _VARLEN["v"] = (wl, x) + tuple(_oracle(x))
    return _VARLEN["v"]


@pytest.mark.slow
@pytest.mark.parametrize("algo", list(ALGOS))
def test_varlen_N8_Hk16_Hv32_full(algo):
    """Every (sequence, head) chain of the packed batch, element by element, and the stored
    bf16 o as the exact rounding of the fp32 result."""
    wl, x, o_ref, s_ref = _varlen()
    _run_and_check(x, wl, o_ref, s_ref, "varlen", algo=ALGOS[algo])


# ------------------------------------------------------------------ verify

@pytest.mark.parametrize("algo", ALGOS_ANY_C)
def test_verify_B128_H32_T16_full(algo):
    import torch
    wl = gi.verify_b128_h32()
    x = gi.make_inputs(wl)
    d = device_inputs(x, "bf16")
    snap = d["state0"].clone()
    s_out = torch.empty_like(snap)
    o = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    import gated_deltanet_linear_05_gb300 as gdn
    o, s = gdn.gdn_verify_block(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                                d["cu_seqlens"], o, chunk=16, algo=ALGOS[algo])
    torch.cuda.synchronize()
    assert torch.equal(d["state0"], snap)  # the snapshot is untouched, bit for bit
    o_ref, s_ref = _oracle(x)
    _check(to_np(o), to_np(s), o_ref, s_ref, "bf16", "verify")
    _run_and_check(x, wl, o_ref, s_ref, "verify", verify=True, algo=ALGOS[algo])


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hk,hv", [(1, 3), (2, 16)])
def test_decode_one_token_per_sequence(dtype, hk, hv):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("dec", [1] * 5, hk, hv, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=2 + hv)
    d = device_inputs(x, dtype)
    s_out = torch.empty_like(d["state0"])
    o32 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    o, s = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                               None, o32)
    torch.cuda.synchronize()
    o_ref, s_ref = _oracle(x)
    _check(to_np(o), to_np(s), o_ref, s_ref, dtype, "decode")
    o16, s16 = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"],
                                   torch.empty_like(s_out))
    torch.cuda.synchronize()
    assert torch.equal(s16, s) and torch.equal(o16, o32.to(o16.dtype))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_one_token_zero_state_and_token_loop(dtype):
    """One token per sequence from no state (state_in None: zero state), against the
    oracle; and the one-token kernel (cu_seqlens None) against the token-loop kernel
    (cu_seqlens = 0, 1, ..., N) on the same batch, both against the oracle."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("dec0", [1] * 7, 2, 4, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=8)
    d = device_inputs(x, dtype)
    s_out = torch.full_like(d["state0"], float("nan"))
    o32 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], None, s_out, None, o32)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                    np.zeros_like(x["state0"]), x["cu_seqlens"])
    _check(to_np(o32), to_np(s_out), o_ref, s_ref, dtype, "decode from zero state")
    o_ref, s_ref = _oracle(x)
    for cu in (None, d["cu_seqlens"]):
        s2 = torch.full_like(d["state0"], float("nan"))
        o2 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s2, cu, o2)
        torch.cuda.synchronize()
        _check(to_np(o2), to_np(s2), o_ref, s_ref, dtype, "cu_seqlens %s" % (cu is not None))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_token_loop_varlen(dtype):
    """With cu_seqlens the decode kernel walks every sequence token by token."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("loop", [40, 0, 3, 17], 2, 4, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=5)
    d = device_inputs(x, dtype)
    s_out = torch.empty_like(d["state0"])
    o32 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    o, s = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                               d["cu_seqlens"], o32)
    torch.cuda.synchronize()
    o_ref, s_ref = _oracle(x)
    _check(to_np(o), to_np(s), o_ref, s_ref, dtype, "decode loop")


def test_decode_B32_H16_100_steps_in_place():
    """100 consecutive in-place steps; the oracle runs the same 100 tokens per sequence
    as one chain in float64."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.decode_b32_h16()
    steps = [gi.make_inputs(wl, step=s) for s in range(wl.steps)]
    state = device_inputs(steps[0], "bf16")["state0"]
    outs = []
    for xs in steps:
        d = device_inputs(xs, "bf16")
        o = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
        gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, state, None, o)
        outs.append(o)
    torch.cuda.synchronize()
    o_gpu = np.stack([to_np(o) for o in outs], axis=1)          # [N, steps, H, dv]
    # oracle: sequence n = its 100 tokens in step order
    cat = {}
    for name in ("q", "k", "v", "g", "beta"):
        cat[name] = np.stack([xs[name] for xs in steps], axis=1).reshape(
            (wl.num_seqs * wl.steps,) + steps[0][name].shape[1:])
    cu = np.arange(0, wl.num_seqs * wl.steps + 1, wl.steps, dtype=np.int32)
    o_ref, s_ref = oracle.recurrent(cat["q"], cat["k"], cat["v"], cat["g"], cat["beta"],
                                    steps[0]["state0"], cu)
    o_ref = o_ref.reshape(wl.num_seqs, wl.steps, wl.num_v_heads, wl.dv)
    _check(o_gpu, to_np(state), o_ref, s_ref, "bf16", "100 steps")


# ------------------------------------------------------------------ self-consistency

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunked_matches_gpu_decode_loop(dtype):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("cons", [64, 130, 16], 1, 2, chunk=16, dtype=dtype, s0_scale=0.1)
    x = gi.make_inputs(wl, seed=9)
    o_c, s_c, d = gpu_prefill(x, wl, o_fp32=True)
    s_out = torch.empty_like(d["state0"])
    o32 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    o_d, s_d = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"],
                                   s_out, d["cu_seqlens"], o32)
    torch.cuda.synchronize()
    _check(o_c, s_c, to_np(o_d), to_np(s_d), dtype, "chunked vs decode loop")


@pytest.mark.parametrize("algo", list(ALGOS))
def test_chunk16_matches_chunk64_bf16(algo):
    """The block length changes only the rounding: C = 64 under `algo` against C = 16
    (two-pass for the schedules built for 64-token blocks only)."""
    wl = gi.Workload("c", [300, 77], 2, 2, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=4)
    a16 = algo if algo in ALGOS_ANY_C else "two_pass"
    o16, s16, _ = gpu_prefill(x, wl, chunk=16, o_fp32=True, algo=ALGOS[a16])
    o64, s64, _ = gpu_prefill(x, wl, chunk=64, o_fp32=True, algo=ALGOS[algo])
    _check(o16, s16, o64, s64, "bf16", "C16 vs C64")


@pytest.mark.parametrize("algo", ["single_pass", "tensor_memory", "recurrent"])
def test_schedules_agree_bf16(algo):
    wl = gi.Workload("c", [300, 77, 1], 2, 4, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=5)
    o1, s1, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS["two_pass"])
    o2, s2, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS[algo])
    _check(o2, s2, o1, s1, "bf16", "%s vs two pass" % algo)


@pytest.mark.parametrize("algo", list(ALGOS))
def test_varlen_packed_matches_separate_runs_bf16(algo):
    lengths = [100, 5, 64]
    wl = gi.Workload("v", lengths, 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=3)
    o, s, _ = gpu_prefill(x, wl, algo=ALGOS[algo])
    cu = x["cu_seqlens"]
    for n, L in enumerate(lengths):
        a, b = cu[n], cu[n + 1]
        xs = {k: x[k][a:b] for k in ("q", "k", "v", "g", "beta", "q_st", "k_st", "v_st")}
        xs["state0"] = x["state0"][n:n + 1]
        xs["cu_seqlens"] = np.array([0, L], np.int32)
        wl1 = gi.Workload("v1", [L], 1, 2, chunk=64, dtype="bf16")
        o1, s1, _ = gpu_prefill(xs, wl1, algo=ALGOS[algo])
        np.testing.assert_array_equal(o1, o[a:b])
        np.testing.assert_array_equal(s1[0], s[n])


@pytest.mark.parametrize("algo", list(ALGOS))
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_repeated_runs_are_bit_identical(chunk, algo):
    """Races between warps or CTAs show up as run-to-run differences."""
    if algo not in ALGOS_ANY_C and chunk != 64:
        pytest.skip("64-token blocks only")
    wl = gi.Workload("det", [40, 15, 130], 1, 2, chunk=chunk, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=12)
    o0, s0, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS[algo])
    for _ in range(8):
        o1, s1, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS[algo])
        assert np.array_equal(o0, o1) and np.array_equal(s0, s1)
