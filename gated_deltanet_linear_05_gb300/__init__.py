"""Python binding of libgdn, the gated delta-rule layer for GB300 (sm_103a).

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libgdn.so`` (built in-tree by ``build.py``).  The functions carry the C-ABI's
names (include/gdn.h) and take torch CUDA tensors, which supply device memory
and the current stream; there is no CPU path.  If the library has not been
built, importing works but every call raises ``GdnUnavailable``.

Layer ("Qwen3.5-9B-npu" model card, section "How it works"): per head a state
S [dk, dv] evolves per token by S <- S exp(g_t); kv = S^T k_t;
S <- S + k_t (x) ((v_t - kv) beta_t); o_t = S^T q_t.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgdn.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_ALIAS, GDN_ERR_WORKSPACE, \
    GDN_ERR_CUDA = range(6)
GDN_F32, GDN_BF16 = 0, 1
GDN_OP_PREFILL, GDN_OP_DECODE, GDN_OP_VERIFY, GDN_OP_DECODE_BLOCK = 0, 1, 2, 3
GDN_ALGO_AUTO, GDN_ALGO_TWO_PASS, GDN_ALGO_SINGLE_PASS, GDN_ALGO_TENSOR_MEMORY = 0, 1, 2, 3
GDN_ALGO_RECURRENT = 4
GDN_ALGO_TWO_PASS_TENSOR = 5
GDN_SINGLE_PASS_MIN_HEADS = 128

GDN_CONV_WIDTH = 4

EXPORTS = ("gdn_prefill_chunked", "gdn_decode_step", "gdn_verify_block",
           "gdn_workspace_size", "gdn_status_string", "gdn_prefill_chunked_noalloc",
           "gdn_input_prologue", "gdn_gated_rmsnorm", "gdn_verify_block_capture",
           "gdn_state_rollback", "gdn_conv_state_rollback", "gdn_prefill_split",
           "gdn_prefill_split_workspace_size", "gdn_device_status", "gdn_selftest_wait_timeout",
           "gdn_decode_block_step")
GDN_STATUS_WAIT_TIMEOUT = 1


class GdnUnavailable(RuntimeError):
    """libgdn.so is missing or cannot be loaded."""


class GdnError(RuntimeError):
    """A libgdn entry point returned a status other than GDN_OK."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, gdn_status_string(status)))


class GdnShape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_k_heads", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32),
                ("o_fp32", ctypes.c_int32), ("algo", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libgdn.so (raises GdnUnavailable if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise GdnUnavailable("libgdn.so not built (run gated_deltanet_linear_05_gb300/build.py)")
        try:
            L = ctypes.CDLL(LIB_PATH)
        except OSError as e:
            raise GdnUnavailable("cannot load libgdn.so: %s" % e)
        P, S = ctypes.c_void_p, ctypes.c_size_t
        for name in ("gdn_prefill_chunked", "gdn_decode_step", "gdn_verify_block"):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(GdnShape), P, P, P, P, P, P, P, P, P, P, S, P]
            f.restype = ctypes.c_int
        L.gdn_workspace_size.argtypes = [ctypes.POINTER(GdnShape), ctypes.c_int]
        L.gdn_workspace_size.restype = ctypes.c_size_t
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        # for callers that cannot allocate: scratch built into the library, no workspace
        L.gdn_prefill_chunked_noalloc.argtypes = [ctypes.POINTER(GdnShape), P, P, P, P, P, P, P,
                                                  P, P, P]
        L.gdn_prefill_chunked_noalloc.restype = ctypes.c_int
        F = ctypes.c_float
        L.gdn_input_prologue.argtypes = [ctypes.POINTER(GdnShape)] + [P] * 11 + [F] + [P] * 6
        L.gdn_input_prologue.restype = ctypes.c_int
        L.gdn_gated_rmsnorm.argtypes = [ctypes.POINTER(GdnShape), P, P, P, F, P, P]
        L.gdn_gated_rmsnorm.restype = ctypes.c_int
        L.gdn_verify_block_capture.argtypes = [ctypes.POINTER(GdnShape)] + [P] * 11
        L.gdn_verify_block_capture.restype = ctypes.c_int
        L.gdn_state_rollback.argtypes = [ctypes.POINTER(GdnShape)] + [P] * 8
        L.gdn_state_rollback.restype = ctypes.c_int
        L.gdn_conv_state_rollback.argtypes = [ctypes.POINTER(GdnShape)] + [P] * 8
        L.gdn_conv_state_rollback.restype = ctypes.c_int
        I32 = ctypes.c_int32
        L.gdn_prefill_split.argtypes = [ctypes.POINTER(GdnShape)] + [P] * 9 + [I32, P, S, P]
        L.gdn_prefill_split.restype = ctypes.c_int
        L.gdn_prefill_split_workspace_size.argtypes = [ctypes.POINTER(GdnShape), I32]
        L.gdn_prefill_split_workspace_size.restype = ctypes.c_size_t
        L.gdn_decode_block_step.argtypes = ([ctypes.POINTER(GdnShape)] + [P] * 10 + [F] +
                                            [P] * 4 + [F, P, P, P, S, P])
        L.gdn_decode_block_step.restype = ctypes.c_int
        L.gdn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
        L.gdn_device_status.restype = ctypes.c_int
        L.gdn_selftest_wait_timeout.argtypes = [I32, P]
        L.gdn_selftest_wait_timeout.restype = ctypes.c_int
        _lib = L
    return _lib


def gdn_status_string(status: int) -> str:
    return lib().gdn_status_string(int(status)).decode()


def make_shape(num_seqs: int, total_tokens: int, num_k_heads: int, num_v_heads: int,
               dk: int = 128, dv: int = 128, chunk: int = 64, dtype: int = GDN_BF16,
               o_fp32: int = 0, algo: int = GDN_ALGO_AUTO) -> GdnShape:
    return GdnShape(num_seqs, total_tokens, num_k_heads, num_v_heads, dk, dv, chunk, dtype, o_fp32,
                    algo)


def gdn_device_status(stream=None) -> int:
    """Read and clear the library's status word on the current device (GDN_STATUS_* bits);
    synchronizes the stream first."""
    v = ctypes.c_uint32(0)
    st = lib().gdn_device_status(ctypes.byref(v), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_device_status")
    return v.value


def gdn_selftest_wait_timeout(polls: int = 1024, stream=None) -> None:
    """Launch the status path's self-test: one bounded wait that nothing completes."""
    st = lib().gdn_selftest_wait_timeout(int(polls), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_selftest_wait_timeout")


def gdn_workspace_size(shape: GdnShape, op: int) -> int:
    n = lib().gdn_workspace_size(ctypes.byref(shape), int(op))
    if n == ctypes.c_size_t(-1).value:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_workspace_size")
    return n


def gdn_prefill_split_workspace_size(shape: GdnShape, segment_len: int) -> int:
    n = lib().gdn_prefill_split_workspace_size(ctypes.byref(shape), int(segment_len))
    if n == ctypes.c_size_t(-1).value:
        raise GdnError(GDN_ERR_INVALID_ARG, "gdn_prefill_split_workspace_size")
    return n


# ------------------------------------------------------------------ torch marshalling

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _shape_of(q, v, o, state_out, cu_seqlens, chunk: int, algo: int = 0) -> GdnShape:
    """Shape from the tensors; o may be float32 while q/k/v are bf16 (o_fp32 = 1)."""
    T, hk, dk = q.shape
    hv, dv = v.shape[1], v.shape[2]
    n = state_out.shape[0] if state_out is not None else (len(cu_seqlens) - 1)
    code = _dtype_code(q)
    o_fp32 = int(code == GDN_BF16 and _dtype_code(o) == GDN_F32)
    if code == GDN_F32 and _dtype_code(o) != GDN_F32:
        raise TypeError("o must be float32 when q/k/v are float32")
    return make_shape(n, T, hk, hv, dk, dv, chunk, code, o_fp32, algo)


def _check_tensors(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libgdn takes contiguous CUDA tensors")


def _stream(stream) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _workspace(shape: GdnShape, op: int, device, workspace):
    need = gdn_workspace_size(shape, op)
    if need == 0:
        return None, 0
    if workspace is None:
        torch = _torch()
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=device)
    base = workspace.data_ptr()
    aligned = (base + 255) & ~255
    return aligned, workspace.numel() - (aligned - base)


def _call(name, op, q, k, v, g, beta, state_in, state_out, cu_seqlens, o, chunk,
          workspace, stream, algo=GDN_ALGO_AUTO):
    _check_tensors(q, k, v, g, beta, state_in, state_out, cu_seqlens, o, workspace)
    shape = _shape_of(q, v, o, state_out, cu_seqlens, chunk, algo)
    ws_ptr, ws_bytes = _workspace(shape, op, q.device, workspace)
    st = getattr(lib(), name)(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                              _ptr(beta), _ptr(state_in), _ptr(state_out), _ptr(cu_seqlens),
                              _ptr(o), ws_ptr, ws_bytes, _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, name)
    return o, state_out


def gdn_prefill_chunked(q, k, v, g, beta, state_in, state_out, cu_seqlens, o=None,
                        chunk: int = 64, workspace=None, stream=None, algo: int = GDN_ALGO_AUTO):
    """Chunkwise-parallel prompt pass.  Tensors as in include/gdn.h:
    q, k [T, Hk, 128]; v [T, Hv, 128]; g, beta [T, Hv] fp32; state_in (or None),
    state_out [N, Hv, 128, 128] fp32; cu_seqlens [N+1] int32.  algo: a GDN_ALGO_* schedule.
    Returns (o, state_out)."""
    if o is None:
        o = _torch().empty_like(v)
    return _call("gdn_prefill_chunked", GDN_OP_PREFILL, q, k, v, g, beta, state_in, state_out,
                 cu_seqlens, o, chunk, workspace, stream, algo)


def split_segment_len(num_seqs: int, num_v_heads: int, tokens_per_seq: int, chunk: int = 64,
                      sms: int = 152) -> int:
    """Segment length that fills the GPU in one wave on the two-pass schedule: each
    (segment, v-head) chain takes 8 CTAs of one SM, so P = sms // (8 * num_seqs *
    num_v_heads) segments per sequence (at least 1) and segment_len = ceil(T / P)
    rounded up to a multiple of chunk."""
    if num_seqs <= 0 or num_v_heads <= 0 or chunk <= 0:
        raise ValueError("num_seqs, num_v_heads and chunk must be positive")
    p = max(1, sms // (8 * num_seqs * num_v_heads))
    seg = -(-max(1, tokens_per_seq) // p)
    return -(-seg // chunk) * chunk


def gdn_prefill_split(q, k, v, g, beta, state_in, state_out, cu_seqlens, o=None,
                      segment_len=None, chunk: int = 64, workspace=None, stream=None,
                      algo: int = GDN_ALGO_AUTO):
    """Sequence-split prompt pass: the results of gdn_prefill_chunked, each sequence cut
    into segments of segment_len tokens (a multiple of chunk) that run side by side.
    segment_len None: split_segment_len for the device's SM count and the mean sequence
    length (total tokens / sequences, rounded up), so with ragged sequences the longest
    ones get more than one wave's worth of segments; with no sequences, one block.
    Returns (o, state_out)."""
    torch = _torch()
    if o is None:
        o = torch.empty_like(v)
    if segment_len is None:
        n = cu_seqlens.numel() - 1
        if n <= 0:
            segment_len = chunk  # nothing to split: the call only validates and returns
        else:
            sms = torch.cuda.get_device_properties(q.device).multi_processor_count
            segment_len = split_segment_len(n, v.shape[1], -(-q.shape[0] // n), chunk, sms)
    _check_tensors(q, k, v, g, beta, state_in, state_out, cu_seqlens, o, workspace)
    shape = _shape_of(q, v, o, state_out, cu_seqlens, chunk, algo)
    need = gdn_prefill_split_workspace_size(shape, segment_len)
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=q.device)
    base = workspace.data_ptr()
    aligned = (base + 255) & ~255
    st = lib().gdn_prefill_split(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(state_in), _ptr(state_out), _ptr(cu_seqlens),
                                 _ptr(o), int(segment_len), aligned,
                                 workspace.numel() - (aligned - base), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_prefill_split")
    return o, state_out


def gdn_verify_block(q, k, v, g, beta, state_in, state_out, cu_seqlens, o=None,
                     chunk: int = 16, workspace=None, stream=None, algo: int = GDN_ALGO_AUTO):
    """Draft-verify block from the snapshot state_in (left unchanged)."""
    if o is None:
        o = _torch().empty_like(v)
    return _call("gdn_verify_block", GDN_OP_VERIFY, q, k, v, g, beta, state_in, state_out,
                 cu_seqlens, o, chunk, workspace, stream, algo)


def gdn_decode_step(q, k, v, g, beta, state_in, state_out, cu_seqlens=None, o=None,
                    stream=None):
    """Token-by-token recurrence (cu_seqlens None: one token per sequence)."""
    if o is None:
        o = _torch().empty_like(v)
    return _call("gdn_decode_step", GDN_OP_DECODE, q, k, v, g, beta, state_in, state_out,
                 cu_seqlens, o, 64, None, stream)


def gdn_input_prologue(q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in,
                       conv_state_out, cu_seqlens=None, eps: float = 1e-6, q=None, k=None, v=None,
                       g=None, beta=None, stream=None):
    """The block's input prologue: causal conv (width GDN_CONV_WIDTH) + SiLU over the raw
    [q | k | v] channels, q/k L2 norm, gates.  q_raw, k_raw [T, Hk, 128]; v_raw
    [T, Hv, 128] (bf16 or fp32); a, b [T, Hv] fp32; conv_w [C, 4] fp32; A_log, dt_bias
    [Hv] fp32; conv_state_in / conv_state_out [N, 3, C] in q_raw's dtype (either may be
    None; they may be the same tensor); cu_seqlens [N+1] int32 or None (one token per
    sequence).  Returns (q, k, v, g, beta)."""
    torch = _torch()
    _check_tensors(q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in,
                   conv_state_out, cu_seqlens, q, k, v, g, beta)
    T, hk, dk = q_raw.shape
    hv, dv = v_raw.shape[1], v_raw.shape[2]
    n = T if cu_seqlens is None else cu_seqlens.numel() - 1
    for cs in (conv_state_in, conv_state_out):
        if cs is not None and (cs.dtype != q_raw.dtype or
                               tuple(cs.shape) != (n, GDN_CONV_WIDTH - 1, 2 * hk * dk + hv * dv)):
            raise ValueError("conv state must be [N, %d, C] in q_raw's dtype" % (GDN_CONV_WIDTH - 1))
    shape = make_shape(n, T, hk, hv, dk, dv, 64, _dtype_code(q_raw))
    q = torch.empty_like(q_raw) if q is None else q
    k = torch.empty_like(k_raw) if k is None else k
    v = torch.empty_like(v_raw) if v is None else v
    g = torch.empty(T, hv, dtype=torch.float32, device=q_raw.device) if g is None else g
    beta = torch.empty(T, hv, dtype=torch.float32, device=q_raw.device) if beta is None else beta
    st = lib().gdn_input_prologue(ctypes.byref(shape), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                                  _ptr(a), _ptr(b), _ptr(conv_w), _ptr(A_log), _ptr(dt_bias),
                                  _ptr(conv_state_in), _ptr(conv_state_out), _ptr(cu_seqlens),
                                  float(eps), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_input_prologue")
    return q, k, v, g, beta


def gdn_gated_rmsnorm(o, z, weight, eps: float = 1e-6, y=None, stream=None):
    """Gated RMSNorm of each (token, v-head) row: o / sqrt(mean(o^2) + eps) * weight * SiLU(z).
    o [T, Hv, 128] (z's dtype, or fp32 with bf16 z); z [T, Hv, 128]; weight [128] fp32.
    y (z's dtype) may be o or z itself.  Returns y."""
    _check_tensors(o, z, weight, y)
    T, hv, dv = z.shape
    code = _dtype_code(z)
    o_fp32 = int(code == GDN_BF16 and _dtype_code(o) == GDN_F32)
    if code == GDN_F32 and _dtype_code(o) != GDN_F32:
        raise TypeError("o must be float32 when z is float32")
    shape = make_shape(0, T, 1, hv, 128, dv, 64, code, o_fp32)
    y = _torch().empty_like(z) if y is None else y
    st = lib().gdn_gated_rmsnorm(ctypes.byref(shape), _ptr(o), _ptr(z), _ptr(weight), float(eps),
                                 _ptr(y), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_gated_rmsnorm")
    return y


def gdn_decode_block_step(q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in,
                          conv_state_out, state_in, state_out, z, norm_w, eps_qk: float = 1e-6,
                          eps_norm: float = 1e-6, y=None, o=None, workspace=None, stream=None):
    """The block's one-token decode step in one launch: input prologue, state step and
    gated RMSNorm.  q_raw, k_raw [N, Hk, 128], v_raw and z [N, Hv, 128] (bf16 or fp32),
    a, b [N, Hv], conv_w [C, 4], A_log, dt_bias [Hv], norm_w [128] fp32, conv states
    [N, 3, C] in q_raw's dtype (in may be None, out may be None or the same tensor),
    states [N, Hv, 128, 128] fp32 (in may be None or equal out).  Returns (y, state_out);
    o (fp32 [N, Hv, 128], optional) receives the layer output before the norm.
    workspace: a uint8 CUDA tensor of gdn_workspace_size(shape, GDN_OP_DECODE_BLOCK) + 256
    bytes, zeroed once and reused across steps (None: a fresh zeroed one per call)."""
    _check_tensors(q_raw, k_raw, v_raw, a, b, conv_w, A_log, dt_bias, conv_state_in,
                   conv_state_out, state_in, state_out, z, norm_w, y, o)
    N, hk, dk = q_raw.shape
    hv, dv = v_raw.shape[1], v_raw.shape[2]
    shape = make_shape(N, N, hk, hv, dk, dv, 64, _dtype_code(q_raw), 0)
    y = _torch().empty_like(z) if y is None else y
    if workspace is None:
        workspace = _torch().zeros(gdn_workspace_size(shape, GDN_OP_DECODE_BLOCK) + 256,
                                   dtype=_torch().uint8, device=z.device)
    _check_tensors(workspace)
    base = workspace.data_ptr()
    ws_ptr = (base + 255) & ~255
    ws_bytes = workspace.numel() - (ws_ptr - base)
    st = lib().gdn_decode_block_step(
        ctypes.byref(shape), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(a), _ptr(b),
        _ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(conv_state_in), _ptr(conv_state_out),
        float(eps_qk), _ptr(state_in), _ptr(state_out), _ptr(z), _ptr(norm_w), float(eps_norm),
        _ptr(y), _ptr(o), ws_ptr, ws_bytes, _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_decode_block_step")
    return y, state_out


def gdn_verify_block_capture(q, k, v, g, beta, state_in, state_out, cu_seqlens, o=None,
                             delta=None, chunk: int = 16, stream=None, algo: int = GDN_ALGO_AUTO):
    """Draft-verify block (state_in left unchanged) that also writes each token's delta
    [T, Hv, 128] fp32.  algo: GDN_ALGO_AUTO, GDN_ALGO_SINGLE_PASS or GDN_ALGO_RECURRENT.
    Returns (o, state_out, delta)."""
    torch = _torch()
    if o is None:
        o = torch.empty_like(v)
    if delta is None:
        delta = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    _check_tensors(q, k, v, g, beta, state_in, state_out, cu_seqlens, o, delta)
    shape = _shape_of(q, v, o, state_out, cu_seqlens, chunk, algo)
    st = lib().gdn_verify_block_capture(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(state_in), _ptr(state_out),
                                        _ptr(cu_seqlens), _ptr(o), _ptr(delta), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_verify_block_capture")
    return o, state_out, delta


def gdn_state_rollback(k, g, delta, state_in, prefix_len, state_out, cu_seqlens, stream=None):
    """State after the first prefix_len[n] tokens of each sequence's verified block,
    from the snapshot state_in and the captured deltas.  state_out may be state_in."""
    _check_tensors(k, g, delta, state_in, prefix_len, state_out, cu_seqlens)
    T, hk, dk = k.shape
    hv = g.shape[1]
    shape = make_shape(cu_seqlens.numel() - 1, T, hk, hv, dk, 128, 64, _dtype_code(k))
    st = lib().gdn_state_rollback(ctypes.byref(shape), _ptr(k), _ptr(g), _ptr(delta),
                                  _ptr(state_in), _ptr(prefix_len), _ptr(state_out),
                                  _ptr(cu_seqlens), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_state_rollback")
    return state_out


def gdn_conv_state_rollback(q_raw, k_raw, v_raw, conv_state_in, prefix_len, conv_state_out,
                            cu_seqlens, stream=None):
    """Conv FIFO after the first prefix_len[n] draft tokens of each sequence."""
    _check_tensors(q_raw, k_raw, v_raw, conv_state_in, prefix_len, conv_state_out, cu_seqlens)
    T, hk, dk = q_raw.shape
    hv, dv = v_raw.shape[1], v_raw.shape[2]
    shape = make_shape(cu_seqlens.numel() - 1, T, hk, hv, dk, dv, 64, _dtype_code(q_raw))
    st = lib().gdn_conv_state_rollback(ctypes.byref(shape), _ptr(q_raw), _ptr(k_raw), _ptr(v_raw),
                                       _ptr(conv_state_in), _ptr(prefix_len),
                                       _ptr(conv_state_out), _ptr(cu_seqlens), _stream(stream))
    if st != GDN_OK:
        raise GdnError(st, "gdn_conv_state_rollback")
    return conv_state_out
