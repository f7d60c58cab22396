"""The C-ABI library: it loads, exports every entry point the header declares, and
rejects bad arguments on the host before launching anything.  No GPU needed: every
call here fails validation (or is a pure query), so no kernel is ever launched.  The
calls pass made-up device addresses, so the module runs only where no GPU is visible:
a mistake in one of these tests must never reach a kernel launch on a real device."""
import ctypes
import os
import re

import pytest

import gated_deltanet_linear_05_gb300 as gdn
from gated_deltanet_linear_05_gb300 import build as gdn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


pytestmark = pytest.mark.skipif(_gpu_visible(), reason="fake device addresses: CPU-only checks")


@pytest.fixture(scope="module")
def L():
    gdn_build.build()
    return gdn.lib()


def _declared():
    txt = open(os.path.join(ROOT, "include", "gdn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:gdn_status|size_t|const char \*)\s*(gdn_\w+)\(", txt, re.M)))


def test_header_declares_the_entry_points():
    assert set(_declared()) == set(gdn.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_status_strings(L):
    for s in range(6):
        assert gdn.gdn_status_string(s).startswith(
            ["GDN_OK", "GDN_ERR_INVALID_ARG", "GDN_ERR_UNSUPPORTED", "GDN_ERR_ALIAS",
             "GDN_ERR_WORKSPACE", "GDN_ERR_CUDA"][s])


def test_workspace_size(L):
    sh = gdn.make_shape(8, 4096, 16, 32, chunk=64, algo=gdn.GDN_ALGO_TWO_PASS)
    n = gdn.gdn_workspace_size(sh, gdn.GDN_OP_PREFILL)
    # a 256-byte header, then one slot per (v-head, block) for T / C + N blocks per head:
    # -W and U (64 x 128 fp16 each), A in 64 rows of 2 x 64 + 16 bytes, 3 x 64 fp32 decays
    mma_slot = -(-(2 * 64 * 128 * 2 + 64 * (2 * 64 + 16) + 3 * 64 * 4) // 128) * 128
    assert n == 256 + 32 * (4096 // 64 + 8) * mma_slot
    # with the tensor-memory second pass the slot holds its operand layouts instead: W^T,
    # diag(e^G) Q and K (64 x 128 fp16), A (64 x 64 fp16), U^T in 128 rows of 144 bytes
    tc_slot = 3 * 64 * 128 * 2 + 64 * 64 * 2 + 128 * 144 + 3 * 64 * 4
    sh5 = gdn.make_shape(8, 4096, 16, 32, chunk=64, algo=gdn.GDN_ALGO_TWO_PASS_TENSOR)
    assert gdn.gdn_workspace_size(sh5, gdn.GDN_OP_PREFILL) == 256 + 32 * (4096 // 64 + 8) * tc_slot
    assert n == gdn.gdn_workspace_size(sh, gdn.GDN_OP_VERIFY)
    assert gdn.gdn_workspace_size(sh, gdn.GDN_OP_DECODE) == 0
    assert gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, chunk=16, dtype=gdn.GDN_F32),
                                  gdn.GDN_OP_PREFILL) == 0
    with pytest.raises(gdn.GdnError):
        gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, dk=64), gdn.GDN_OP_PREFILL)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_workspace_size(sh, 7)


def test_workspace_size_follows_the_schedule(L):
    """The single-pass schedule needs no workspace; AUTO picks it from the head count."""
    for n, hv in [(8, 32), (1, 16), (127, 1), (128, 1), (2, 64)]:
        two = gdn.gdn_workspace_size(gdn.make_shape(n, 64 * n, 1, hv, chunk=64,
                                                    algo=gdn.GDN_ALGO_TWO_PASS), gdn.GDN_OP_PREFILL)
        one = gdn.gdn_workspace_size(gdn.make_shape(n, 64 * n, 1, hv, chunk=64,
                                                    algo=gdn.GDN_ALGO_SINGLE_PASS),
                                     gdn.GDN_OP_PREFILL)
        auto = gdn.gdn_workspace_size(gdn.make_shape(n, 64 * n, 1, hv, chunk=64),
                                      gdn.GDN_OP_VERIFY)
        assert two > 0 and one == 0
        assert auto == (0 if n * hv >= gdn.GDN_SINGLE_PASS_MIN_HEADS else two)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, algo=6), gdn.GDN_OP_PREFILL)
    # the two-pass schedule with the tensor-memory second pass: larger slots, 64-token
    # blocks only
    sh2 = gdn.make_shape(3, 700, 2, 4, chunk=64, algo=gdn.GDN_ALGO_TWO_PASS)
    sh5 = gdn.make_shape(3, 700, 2, 4, chunk=64, algo=gdn.GDN_ALGO_TWO_PASS_TENSOR)
    assert gdn.gdn_workspace_size(sh5, gdn.GDN_OP_PREFILL) > gdn.gdn_workspace_size(sh2, gdn.GDN_OP_PREFILL)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, chunk=16,
                                              algo=gdn.GDN_ALGO_TWO_PASS_TENSOR), gdn.GDN_OP_PREFILL)
    # the token loop (recurrent schedule) needs none, for any block length
    for chunk in (16, 32, 64):
        for op in (gdn.GDN_OP_PREFILL, gdn.GDN_OP_VERIFY):
            assert gdn.gdn_workspace_size(gdn.make_shape(8, 4096, 16, 32, chunk=chunk,
                                                         algo=gdn.GDN_ALGO_RECURRENT), op) == 0
    # the tensor-memory schedule: 64-token blocks of bf16 q/k/v only, no workspace
    assert gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, chunk=64,
                                                 algo=gdn.GDN_ALGO_TENSOR_MEMORY),
                                  gdn.GDN_OP_PREFILL) == 0
    with pytest.raises(gdn.GdnError):
        gdn.gdn_workspace_size(gdn.make_shape(1, 64, 1, 1, chunk=16,
                                              algo=gdn.GDN_ALGO_TENSOR_MEMORY), gdn.GDN_OP_PREFILL)


# fake, well-aligned device addresses: every call below must fail validation first
A = 0x10000000


def _call(L, name, shape, q=A, k=A, v=A, g=A, beta=A, s_in=A + (1 << 24), s_out=A + (1 << 26),
          cu=A, o=A, ws=None, ws_bytes=0):
    fn = getattr(L, name)
    return fn(ctypes.byref(shape) if shape is not None else None, q, k, v, g, beta, s_in, s_out,
              cu, o, ws, ws_bytes, None)


@pytest.mark.parametrize("name", ["gdn_prefill_chunked", "gdn_verify_block", "gdn_decode_step"])
def test_validation(L, name):
    ok_shape = gdn.make_shape(2, 10, 1, 2, chunk=16)
    assert _call(L, name, None) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, gdn.make_shape(2, 10, 1, 2, dk=64)) == gdn.GDN_ERR_UNSUPPORTED
    assert _call(L, name, gdn.make_shape(2, 10, 2, 3)) == gdn.GDN_ERR_INVALID_ARG   # Hv % Hk
    assert _call(L, name, gdn.make_shape(-1, 10, 1, 1)) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, gdn.make_shape(2, 10, 1, 2, dtype=5)) == gdn.GDN_ERR_UNSUPPORTED
    assert _call(L, name, gdn.make_shape(2, 10, 1, 2, algo=-1)) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, ok_shape, q=None) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, ok_shape, o=None) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, ok_shape, s_out=None) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, ok_shape, v=A + 8) == gdn.GDN_ERR_INVALID_ARG            # misaligned
    assert _call(L, name, ok_shape, s_in=A + 4) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, name, ok_shape, cu=A + 2) == gdn.GDN_ERR_INVALID_ARG
    # partial overlap of the two state buffers
    assert _call(L, name, ok_shape, s_in=A, s_out=A + 4096) == gdn.GDN_ERR_ALIAS


@pytest.mark.parametrize("name", ["gdn_prefill_chunked", "gdn_verify_block"])
def test_chunked_validation(L, name):
    assert _call(L, name, gdn.make_shape(2, 10, 1, 2, chunk=24)) == gdn.GDN_ERR_UNSUPPORTED
    assert _call(L, name, gdn.make_shape(2, 10, 1, 2, chunk=16), cu=None) == gdn.GDN_ERR_INVALID_ARG
    sh = gdn.make_shape(2, 10, 1, 2, chunk=16)
    need = gdn.gdn_workspace_size(sh, gdn.GDN_OP_PREFILL)
    assert _call(L, name, sh, ws=None) == gdn.GDN_ERR_WORKSPACE
    assert _call(L, name, sh, ws=A, ws_bytes=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert _call(L, name, sh, ws=A + 16, ws_bytes=need) == gdn.GDN_ERR_WORKSPACE  # not 256-aligned


def test_verify_needs_a_separate_snapshot(L):
    sh = gdn.make_shape(2, 10, 1, 2, chunk=16)
    assert _call(L, "gdn_verify_block", sh, s_in=None) == gdn.GDN_ERR_INVALID_ARG
    assert _call(L, "gdn_verify_block", sh, s_in=A, s_out=A) == gdn.GDN_ERR_ALIAS


def test_decode_without_cu_seqlens_needs_one_token_per_sequence(L):
    sh = gdn.make_shape(3, 4, 1, 1)
    assert _call(L, "gdn_decode_step", sh, cu=None) == gdn.GDN_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(L):
    sh = gdn.make_shape(0, 0, 1, 1, chunk=16)
    for name in ("gdn_prefill_chunked", "gdn_verify_block", "gdn_decode_step"):
        assert _call(L, name, sh, q=None, k=None, v=None, g=None, beta=None, s_in=None,
                     s_out=None, cu=None, o=None) == gdn.GDN_OK


def _pro_args(**kw):
    """gdn_input_prologue arguments at disjoint fake addresses (1 MiB apart)."""
    names = ["q_raw", "k_raw", "v_raw", "a", "b", "conv_w", "A_log", "dt_bias", "cs_in", "cs_out",
             "cu", "q", "k", "v", "g", "beta"]
    args = {n: A + (i << 20) for i, n in enumerate(names)}
    args.update(kw)
    return args


def _prologue(L, shape, eps=1e-6, **kw):
    a = _pro_args(**kw)
    return L.gdn_input_prologue(
        ctypes.byref(shape) if shape is not None else None, a["q_raw"], a["k_raw"], a["v_raw"],
        a["a"], a["b"], a["conv_w"], a["A_log"], a["dt_bias"], a["cs_in"], a["cs_out"], a["cu"],
        eps, a["q"], a["k"], a["v"], a["g"], a["beta"], None)


def test_prologue_validation(L):
    ok = gdn.make_shape(2, 10, 1, 2)
    assert _prologue(L, None) == gdn.GDN_ERR_INVALID_ARG
    assert _prologue(L, gdn.make_shape(2, 10, 1, 2, dk=64)) == gdn.GDN_ERR_UNSUPPORTED
    assert _prologue(L, gdn.make_shape(2, 10, 2, 3)) == gdn.GDN_ERR_INVALID_ARG
    for name in ("q_raw", "v_raw", "a", "b", "conv_w", "A_log", "dt_bias", "q", "k", "g", "beta"):
        assert _prologue(L, ok, **{name: None}) == gdn.GDN_ERR_INVALID_ARG, name
    for name in ("q_raw", "k", "beta", "conv_w", "cs_in", "cs_out"):
        assert _prologue(L, ok, **{name: A + (1 << 30) + 8}) == gdn.GDN_ERR_INVALID_ARG, name
    assert _prologue(L, ok, A_log=A + (1 << 30) + 2) == gdn.GDN_ERR_INVALID_ARG
    assert _prologue(L, ok, cu=A + (1 << 30) + 2) == gdn.GDN_ERR_INVALID_ARG
    assert _prologue(L, ok, eps=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert _prologue(L, ok, eps=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    # one token per sequence without cu_seqlens
    assert _prologue(L, ok, cu=None) == gdn.GDN_ERR_INVALID_ARG
    # outputs overlapping the raw inputs; conv states overlapping partly
    assert _prologue(L, ok, q=A) == gdn.GDN_ERR_ALIAS
    assert _prologue(L, ok, v=A + (1 << 20) + 256) == gdn.GDN_ERR_ALIAS   # inside k_raw
    assert _prologue(L, ok, cs_out=A + (8 << 20) + 16) == gdn.GDN_ERR_ALIAS
    # an empty batch launches nothing
    assert _prologue(L, gdn.make_shape(0, 0, 1, 2), q_raw=None, q=None) == gdn.GDN_OK


def _norm(L, shape, o=A, z=A + (1 << 24), w=A + (2 << 24), y=A + (3 << 24), eps=1e-6):
    return L.gdn_gated_rmsnorm(ctypes.byref(shape) if shape is not None else None, o, z, w, eps,
                               y, None)


def test_gated_rmsnorm_validation(L):
    ok = gdn.make_shape(0, 10, 1, 2)
    assert _norm(L, None) == gdn.GDN_ERR_INVALID_ARG
    assert _norm(L, gdn.make_shape(0, 10, 1, 2, dv=64)) == gdn.GDN_ERR_UNSUPPORTED
    assert _norm(L, ok, o=None) == gdn.GDN_ERR_INVALID_ARG
    assert _norm(L, ok, w=A + 4) == gdn.GDN_ERR_INVALID_ARG
    assert _norm(L, ok, eps=-1e-3) == gdn.GDN_ERR_INVALID_ARG
    assert _norm(L, ok, y=A + 512) == gdn.GDN_ERR_ALIAS                 # partly over o
    assert _norm(L, ok, y=A + (1 << 24) + 16) == gdn.GDN_ERR_ALIAS      # partly over z
    # in place over an fp32 o with a bf16 y is not the same element size
    assert _norm(L, gdn.make_shape(0, 10, 1, 2, o_fp32=1), y=A) == gdn.GDN_ERR_ALIAS
    assert _norm(L, gdn.make_shape(0, 0, 1, 2), o=None, z=None, w=None, y=None) == gdn.GDN_OK


def test_capture_and_rollback_validation(L):
    sh = gdn.make_shape(2, 10, 1, 2, chunk=16)
    cap = L.gdn_verify_block_capture
    # q, k, v, g, beta, state_in, state_out, cu_seqlens, o (then delta, stream)
    base = [A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20), A + (5 << 24),
            A + (6 << 24), A + (7 << 20), A + (8 << 20)]
    assert len(base) + 3 == len(cap.argtypes)

    def c(shape, delta=A + (10 << 20), **kw):
        args = list(base)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return cap(ctypes.byref(shape), *args, delta, None)
    assert c(sh, delta=None) == gdn.GDN_ERR_INVALID_ARG
    assert c(sh, delta=A + (10 << 20) + 4) == gdn.GDN_ERR_INVALID_ARG
    assert c(gdn.make_shape(2, 10, 1, 2, chunk=16, algo=gdn.GDN_ALGO_TWO_PASS)) == gdn.GDN_ERR_UNSUPPORTED
    assert c(gdn.make_shape(2, 10, 1, 2, chunk=64, algo=gdn.GDN_ALGO_TENSOR_MEMORY)) == gdn.GDN_ERR_UNSUPPORTED
    assert c(sh, a5=None) == gdn.GDN_ERR_INVALID_ARG                       # no snapshot
    assert c(sh, a6=A + (5 << 24) + 4096) == gdn.GDN_ERR_ALIAS             # overlaps the snapshot
    rb = L.gdn_state_rollback
    # k, g, delta, state_in, prefix_len, state_out, cu_seqlens (then stream)
    ok = [A, A + (1 << 20), A + (2 << 20), A + (3 << 24), A + (4 << 20), A + (5 << 24), A + (6 << 20)]
    assert len(ok) + 2 == len(rb.argtypes)

    def r(shape, **kw):
        args = list(ok)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return rb(ctypes.byref(shape) if shape is not None else None, *args, None)
    assert r(None) == gdn.GDN_ERR_INVALID_ARG
    assert r(gdn.make_shape(2, 10, 1, 2, dk=64)) == gdn.GDN_ERR_UNSUPPORTED
    assert r(sh, a4=None) == gdn.GDN_ERR_INVALID_ARG                       # prefix_len
    assert r(sh, a6=None) == gdn.GDN_ERR_INVALID_ARG                       # cu_seqlens
    assert r(sh, a2=A + (2 << 20) + 8) == gdn.GDN_ERR_INVALID_ARG          # delta misaligned
    assert r(sh, a5=A + (3 << 24) + 1024) == gdn.GDN_ERR_ALIAS             # partial state overlap
    assert r(gdn.make_shape(0, 0, 1, 2), a0=None, a1=None, a2=None) == gdn.GDN_OK
    cs = L.gdn_conv_state_rollback
    assert len(cs.argtypes) == 9

    def cr(shape, **kw):
        args = [A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20), A + (5 << 20),
                A + (6 << 20)]
        for i, v in kw.items():
            args[int(i[1:])] = v
        return cs(ctypes.byref(shape), *args, None)
    assert cr(sh, a4=None) == gdn.GDN_ERR_INVALID_ARG
    assert cr(sh, a0=A + 8) == gdn.GDN_ERR_INVALID_ARG
    assert cr(sh, a5=A + (3 << 20) + 16) == gdn.GDN_ERR_ALIAS


def test_split_validation(L):
    """The sequence-split pass: segment length a positive multiple of the block length,
    no token loop, a workspace of the size its query returns; every failure before any
    launch."""
    sp = L.gdn_prefill_split
    base = [A, A + (1 << 20), A + (2 << 20), A + (3 << 20), A + (4 << 20), A + (5 << 24),
            A + (6 << 24), A + (7 << 20), A + (8 << 20)]
    assert len(base) + 5 == len(sp.argtypes)
    sh = gdn.make_shape(2, 4096, 1, 2, chunk=64)

    def c(shape, seg=1024, ws=A + (9 << 24), ws_bytes=1 << 40, **kw):
        args = list(base)
        for i, v in kw.items():
            args[int(i[1:])] = v
        return sp(ctypes.byref(shape), *args, seg, ws, ws_bytes, None)
    need = gdn.gdn_prefill_split_workspace_size(sh, 1024)
    # two segments of (4096 / 1024 + 2) sets of states at least
    assert need > 3 * (4096 // 1024 + 2) * 2 * 128 * 128 * 4
    for bad_seg in (0, -64, 100):
        assert c(sh, seg=bad_seg) == gdn.GDN_ERR_INVALID_ARG
        with pytest.raises(gdn.GdnError):
            gdn.gdn_prefill_split_workspace_size(sh, bad_seg)
    rec = gdn.make_shape(2, 4096, 1, 2, chunk=64, algo=gdn.GDN_ALGO_RECURRENT)
    assert c(rec) == gdn.GDN_ERR_UNSUPPORTED
    assert c(sh, a7=None) == gdn.GDN_ERR_INVALID_ARG                     # cu_seqlens required
    assert c(sh, a6=A + (5 << 24) + 4096) == gdn.GDN_ERR_ALIAS           # partly over state_in
    assert c(sh, ws=None) == gdn.GDN_ERR_WORKSPACE
    assert c(sh, ws_bytes=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert c(sh, ws=A + (9 << 24) + 128) == gdn.GDN_ERR_WORKSPACE        # not 256-byte aligned
    assert c(gdn.make_shape(0, 0, 1, 2, chunk=64)) == gdn.GDN_OK          # nothing to do


def test_split_segment_rule():
    """The binding's segment-length rule (one wave of two-pass chains)."""
    f = gdn.split_segment_len
    assert f(1, 2, 65536) == 7296          # 9 segments of 114 blocks on 152 SMs
    assert f(1, 1, 16384) == 896           # 19 segments
    assert f(1, 16, 4096) == 4096          # 16 heads fill the GPU already: one segment
    assert f(2, 2, 1000, chunk=16) == 256  # 4 segments, rounded up to the block length
    assert f(1, 2, 65536) % 64 == 0
    for n, hv, t in [(1, 2, 65536), (1, 1, 16384), (3, 1, 5000)]:
        seg = f(n, hv, t)
        segs = -(-t // seg)
        assert segs * n * hv * 8 <= 152 or segs == 1
    with pytest.raises(ValueError):
        f(0, 2, 100)


def test_status_entry_points_validate_before_any_cuda_call(L):
    """A null status pointer and a poll count outside 1 .. 2^22 are rejected on the host."""
    assert L.gdn_device_status(None, None) == gdn.GDN_ERR_INVALID_ARG
    for polls in (0, -1, (1 << 22) + 1):
        assert L.gdn_selftest_wait_timeout(polls, None) == gdn.GDN_ERR_INVALID_ARG


def test_decode_block_step_validation(L):
    """The fused decode step: one token per sequence, non-negative eps, a workspace of
    gdn_workspace_size(GDN_OP_DECODE_BLOCK) bytes on a 256-byte boundary; all rejected
    before any launch."""
    P = ctypes.c_void_p
    fake = [P(0x1000 * (i + 1)) for i in range(10)]
    fake[9] = fake[8]  # the FIFO updated in place

    def call(shape, eps_qk=1e-6, eps_norm=1e-6, ws=0x100000, ws_bytes=1 << 20):
        return L.gdn_decode_block_step(ctypes.byref(shape), *fake, ctypes.c_float(eps_qk),
                                       P(0x20000), P(0x20000), P(0x30000), P(0x40000),
                                       ctypes.c_float(eps_norm), P(0x50000), None, P(ws),
                                       ctypes.c_size_t(ws_bytes), None)

    sh = gdn.make_shape(2, 2, 1, 4)                                            # Hv / Hk = 4
    need = L.gdn_workspace_size(ctypes.byref(sh), gdn.GDN_OP_DECODE_BLOCK)
    # counters (2 x 4 + 2 x 1 words), quarter sums (2 x 4 x 4), o (2 x 4 x 128), 256-aligned
    assert need == 256 + 256 + 2 * 4 * 128 * 4
    assert call(sh, ws_bytes=need - 1) == gdn.GDN_ERR_WORKSPACE
    assert call(sh, ws=0x100080, ws_bytes=need) == gdn.GDN_ERR_WORKSPACE      # not 256-aligned
    assert call(sh, ws=0) == gdn.GDN_ERR_WORKSPACE
    assert call(gdn.make_shape(2, 3, 2, 4)) == gdn.GDN_ERR_INVALID_ARG        # T != N
    assert call(gdn.make_shape(2, 2, 2, 4), eps_qk=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.make_shape(2, 2, 2, 4), eps_norm=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    assert call(gdn.make_shape(0, 0, 2, 4)) == gdn.GDN_OK                     # empty batch
