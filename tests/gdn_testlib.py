"""Helpers shared by the GPU tests: move seeded inputs to the device and compare."""
import numpy as np

import gdn_inputs as gi


def rel_err(x, ref):
    """max |x - ref| / rms(ref) over the whole tensor (the tolerance metric)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(x - ref)) / max(rms, 1e-300)) if ref.size else 0.0


def to_dev(arr, dtype: str, device="cuda"):
    """Storage array (float32, or uint16 bf16 bits) -> torch CUDA tensor."""
    import torch
    if arr is None:
        return None
    if dtype == "bf16" and arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    if arr.dtype == np.int32:
        return torch.from_numpy(np.ascontiguousarray(arr)).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(device)


def device_inputs(x: dict, dtype: str, device="cuda"):
    d = {n: to_dev(x[n + "_st"], dtype, device) for n in ("q", "k", "v")}
    d["g"] = to_dev(x["g"], "f32", device)
    d["beta"] = to_dev(x["beta"], "f32", device)
    d["state0"] = to_dev(x["state0"], "f32", device)
    d["cu_seqlens"] = to_dev(x["cu_seqlens"], "i32", device)
    return d


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(x, wl, chunk=None, state_in=True, inplace=False, verify=False, o_fp32=False,
                algo=0):
    """Run the chunked path (or verify) on the seeded inputs; returns (o, state_out, dev).

    o_fp32: ask for the unrounded fp32 output even when q/k/v are bf16.
    algo: the bf16 schedule (0 auto, 1 two-pass, 2 single-pass)."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    d = device_inputs(x, wl.dtype)
    s_in = d["state0"] if state_in else None
    N, Hv = wl.num_seqs, wl.num_v_heads
    if inplace:
        s_out = s_in.clone() if s_in is not None else None
        s_in = s_out
    else:
        s_out = torch.full((N, Hv, wl.dk, wl.dv), float("nan"), device="cuda")
    o = torch.full(d["v"].shape, float("nan"), device="cuda",
                   dtype=torch.float32 if o_fp32 else d["v"].dtype)
    fn = gdn.gdn_verify_block if verify else gdn.gdn_prefill_chunked
    o, s = fn(d["q"], d["k"], d["v"], d["g"], d["beta"], s_in, s_out, d["cu_seqlens"], o,
              chunk=chunk or wl.chunk, algo=algo)
    torch.cuda.synchronize()
    d["o_raw"] = o
    return to_np(o), to_np(s), d


def half_ulp_bf16(x):
    """Half the bf16 spacing at |x| (the largest rounding error of a stored bf16 value)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, 2.0 ** (e - 8), 0.0)
