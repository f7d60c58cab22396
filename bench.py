#!/usr/bin/env python
"""Benchmark of libgdn (gated delta-rule layer) on GB300; prints ONE JSON line.

Headline: chunked prefill tokens/s on the single-sequence workload (B=1, H=16,
T=4096, chunk 64, bf16 q/k/v, fp32 g/beta/state).  One step = one
gdn_prefill_chunked call over that batch (the prompt path: block bookkeeping,
cumsum, Grams, triangular solve, block output and state carry).  The same line
carries the other rows of the path measured the same way: the decode step
(32 x 16 heads, state GB/s), the draft-verify block (128 x 32 heads, T=16) and
packed varlen prefill (8 sequences, Hk=16 / Hv=32).

Timing: CUDA events on the launching stream, L2 flushed (a 512 MiB write)
before every timed step and outside the events; decode rotates over 8 state
sets (268 MB > 2x L2) so each step streams its state from HBM.

--impl reference times the float64 CPU oracle (the reference arm)
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GDN prefill tokens/s (%TC roofline); decode state GB/s (%HBM peak)"
D = 128
EXTRA_ROWS = ("decode", "decode_block", "verify", "varlen", "prologue", "gated_rmsnorm", "accept",
              "split", "schedules")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--only", choices=EXTRA_ROWS, action="append",
                    help="run only these extra rows after the headline (repeatable)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(p))
        return {"hbm": float(j["hbm_gbs"]), "bf16": float(j["bf16_tflops"]),
                "bf16_sustained": float(j["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ algorithmic work

def prefill_work(lengths, hk, hv, chunk, s_qk=2, s_v=2):
    """(flops, bytes) the method itself must do / move for a prefill batch."""
    T = sum(lengths)
    flops = T * (hk * 2 * chunk * D + hv * (6 * D * D + 2 * chunk * D))
    byts = T * (hk * 2 * D * s_qk + hv * (2 * D * s_v + 8)) + len(lengths) * hv * 2 * D * D * 4
    return flops, byts


def decode_bytes(n, hv, hk, s=2):
    """State read + write, q/k (per k-head), v, o, g, beta for one decode step."""
    return n * hv * (2 * D * D * 4 + 2 * D * s + 8) + n * hk * 2 * D * s


# ------------------------------------------------------------------ clocks

class Clocks:
    """nvidia-smi samples (every 100 ms) while the timed regions run."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        mhz = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------ helpers

def dev_inputs(x, torch, device):
    import numpy as np

    def t(a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return {"q": t(x["q_st"]), "k": t(x["k_st"]), "v": t(x["v_st"]), "g": t(x["g"]),
            "beta": t(x["beta"]), "state0": t(x["state0"]), "cu": t(x["cu_seqlens"])}


def timed_steps(torch, fn, steps, warmup, flush=None):
    """Per-step CUDA-event times (ms) on the current stream, L2 flushed between steps."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    for i in range(steps):
        if flush is not None:
            flush(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def roofline(bound, achieved, peak, unit, traffic=None):
    return {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "traffic": traffic}


# ------------------------------------------------------------------ GPU arm

def run_gdn(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import gdn_inputs as gi
    import gated_deltanet_linear_05_gb300 as gdn
    from gated_deltanet_linear_05_gb300 import build as gdn_build
    from gated_deltanet_linear_05_gb300 import shard as gdn_shard

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    gdn_build.build()
    gdn.lib()
    pk = peaks()
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=device)

    def flush(i):
        flush_buf.fill_(i & 0xFF)

    def barrier_max(ms):  # the slowest rank's time (barrier first); ms itself at N = 1
        return gdn_shard.max_over_ranks(ms, device=device)

    clocks = Clocks(local)
    out = {}

    # ---- headline: prefill B=1, H=16, T=4096, C=64
    wl = gi.prefill_t4096_h16()
    x = gi.make_inputs(wl)
    d = dev_inputs(x, torch, device)
    N, Hk, Hv, C = wl.num_seqs, wl.num_k_heads, wl.num_v_heads, wl.chunk
    s_out = torch.empty_like(d["state0"])
    o = torch.empty_like(d["v"])
    shape = gdn.make_shape(N, wl.total_tokens, Hk, Hv, chunk=C)
    ws = torch.empty(gdn.gdn_workspace_size(shape, gdn.GDN_OP_PREFILL) + 256, dtype=torch.uint8,
                     device=device)

    def step():
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                                d["cu"], o, chunk=C, workspace=ws)

    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    times = timed_steps(torch, step, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    ms = barrier_max(statistics.mean(times))
    # the same step back to back, L2 not flushed (whatever the previous step left in L2)
    warm_ms = barrier_max(statistics.mean(timed_steps(torch, step, max(3, min(args.steps, 50)), 2)))
    flops, byts = prefill_work(wl.lengths, Hk, Hv, C)
    tok_s = world * wl.total_tokens / (ms * 1e-3)
    gbs = byts / (ms * 1e-3) / 1e9
    tfs = flops / (ms * 1e-3) / 1e12

    # e2e through the C-ABI from pinned host buffers
    host = {k: v.cpu().pin_memory() for k, v in d.items() if v is not None}
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    s_h = torch.empty(s_out.shape, dtype=s_out.dtype).pin_memory()
    bufs = {k: torch.empty_like(v) for k, v in d.items() if v is not None}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_h.numel() * o_h.element_size() + s_h.numel() * s_h.element_size()

    def e2e_step():
        for k, v in host.items():
            bufs[k].copy_(v, non_blocking=True)
        gdn.gdn_prefill_chunked(bufs["q"], bufs["k"], bufs["v"], bufs["g"], bufs["beta"],
                                bufs["state0"], s_out, bufs["cu"], o, chunk=C, workspace=ws)
        o_h.copy_(o, non_blocking=True)
        s_h.copy_(s_out, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 50))
    e2e_times = timed_steps(torch, e2e_step, e2e_steps, 2, flush)
    e2e_serial_ms = barrier_max(statistics.mean(e2e_times))
    e2e_ms = barrier_max(e2e_pipelined(torch, gdn, d, host, o, s_out, ws, C, e2e_steps))

    if not args.no_extra:
        rows = {"decode": lambda: bench_decode(torch, gdn, gi, device, pk, args),
                "decode_block": lambda: bench_decode_block(torch, gdn, gi, device, pk, args),
                "verify": lambda: bench_verify(torch, gdn, gi, device, pk, args, flush),
                "varlen": lambda: bench_varlen(torch, gdn, gi, device, pk, args, flush),
                "schedules": lambda: bench_schedules(torch, gdn, gi, device, pk, args, flush),
                "prologue": lambda: bench_prologue(torch, gdn, gi, device, pk, args, flush),
                "gated_rmsnorm": lambda: bench_gated_rmsnorm(torch, gdn, gi, device, pk, args, flush),
                "accept": lambda: bench_accept(torch, gdn, gi, device, pk, args, flush),
                "split": lambda: bench_split(torch, gdn, gi, device, pk, args, flush)}
        for name in EXTRA_ROWS:
            if not args.only or name in args.only:
                out[name] = rows[name]()
    clk = clocks.stop()

    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "num_seqs": N, "seq_len": wl.total_tokens,
                   "num_k_heads": Hk, "num_v_heads": Hv, "dk": D, "dv": D, "chunk": C,
                   "qkv": "bf16", "g_beta_state": "fp32",
                   "l2": "flushed (512 MiB write) before every timed step",
                   "parallelism": "dp%d (independent batches per GPU)" % world},
        # traffic: DRAM bytes of the step's two kernels from the committed ncu capture
        # (pass 1 53.9 MB + pass 2 80.1 MB; ncu flushes caches between kernels, so the
        # workspace round trip counts as DRAM traffic there)
        "roofline": roofline("hbm", gbs, pk["hbm"], "GB/s", traffic=134.0e6),
        "roofline_scope": "one gdn_prefill_chunked call (pass 1 + pass 2); the dominant "
                          "kernel, pass 2, takes ~57 of its ~87 us",
        "tensor": {"achieved": round(tfs, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                   "frac": round(tfs / pk["bf16"], 4), "algorithmic_flops": flops},
        "algorithmic_bytes": byts,
        "ms_per_step_warm_l2": round(warm_ms, 5),
        "peaks_source": pk["source"],
        "e2e": {"value": round(world * wl.total_tokens / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "method": "steps pipelined over 2 device buffer sets: step i+1's inputs copied in "
                          "(one packed copy) and step i-1's o and state copied out (one packed "
                          "copy) on their own streams while step i computes; every copy inside "
                          "the timed region",
                "ms_per_step_serial": round(e2e_serial_ms, 4)},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    line.update(out)
    line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def bench_decode(torch, gdn, gi, device, pk, args):
    """Decode step, 32 sequences x 16 heads; 8 state sets rotated (268 MB > 2x L2).

    The 100 steps are captured once in a CUDA graph and replayed, so the GPU sees the
    steps back to back (as a serving loop would issue them); the eager Python-driven
    loop is reported beside it."""
    wl = gi.decode_b32_h16()
    R, steps = 8, 100
    sets = []
    for r in range(R):
        x = gi.make_inputs(wl, seed=r, step=0)
        sets.append(dev_inputs(x, torch, device))
    o = torch.empty_like(sets[0]["v"])

    def one(i):
        s = sets[i % R]
        gdn.gdn_decode_step(s["q"], s["k"], s["v"], s["g"], s["beta"], s["state0"], s["state0"],
                            None, o)

    def run(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    for i in range(2 * R):
        one(i)
    torch.cuda.synchronize()
    ms_eager = run(lambda: [one(i) for i in range(steps)]) / steps
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graphs = {}
    for name, pick in (("rotated", lambda i: i), ("resident", lambda i: 0)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            one(0)  # warm the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(steps):
                    one(pick(i))
        graphs[name] = g
    for g in graphs.values():
        g.replay()
    torch.cuda.synchronize()
    times = {name: min(run(g.replay) for _ in range(3)) / steps for name, g in graphs.items()}
    ms = times["rotated"]
    byts = decode_bytes(wl.num_seqs, wl.num_v_heads, wl.num_k_heads)
    state_b = wl.num_seqs * wl.num_v_heads * 2 * D * D * 4
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": wl.name + "_x100steps", "us_per_step": round(ms * 1e3, 3),
            "state_GBps": round(state_b / (ms * 1e-3) / 1e9, 1),
            "roofline": roofline("hbm", gbs, pk["hbm"], "GB/s"),
            "bytes_per_step": byts, "l2": "8 state sets rotated (268 MB)",
            "launch": "100 steps replayed from one CUDA graph",
            "us_per_step_eager_launches": round(ms_eager * 1e3, 3),
            "us_per_step_l2_resident": round(times["resident"] * 1e3, 3), "gpu_launches": steps}


def decode_block_bytes(n, hk, hv, s=2, conv_width=4):
    """The block's decode step: the state read and written, the raw q/k/v projections, a and
    b, z read and y written, the conv FIFO read and written, the conv and norm weights (the
    fused kernel's 0.5 MB of scratch, o and its partial sums, stays in L2 and is not counted)."""
    C = (2 * hk + hv) * D
    return (n * hv * 2 * D * D * 4 + n * C * s + n * hv * 8 + 2 * n * hv * D * s +
            2 * n * (conv_width - 1) * C * s + C * conv_width * 4 + D * 4)


def bench_decode_block(torch, gdn, gi, device, pk, args):
    """The block's whole decode step (input prologue, state step, gated RMSNorm), 32
    sequences x 16 heads, one token each: one fused launch (gdn_decode_block_step) against
    the three separate launches; 8 state sets rotated (268 MB > 2x L2), conv FIFO in place,
    100 steps captured in one CUDA graph per form."""
    wl = gi.decode_b32_h16()
    R, steps = 8, 100
    d = block_dev_inputs(gi.make_block_inputs(wl), torch, device)
    S = [dev_inputs(gi.make_inputs(wl, seed=r, step=0), torch, device)["state0"] for r in range(R)]
    cs = d["conv_state0"]
    N, Hk, Hv = wl.num_seqs, wl.num_k_heads, wl.num_v_heads
    q = torch.empty((N, Hk, D), dtype=torch.bfloat16, device=device)
    k = torch.empty_like(q)
    v = torch.empty((N, Hv, D), dtype=torch.bfloat16, device=device)
    g = torch.empty((N, Hv), device=device)
    beta = torch.empty_like(g)
    o = torch.empty((N, Hv, D), device=device)
    y = torch.empty_like(d["z"])
    ws = torch.zeros(gdn.gdn_workspace_size(gdn.make_shape(N, N, Hk, Hv), gdn.GDN_OP_DECODE_BLOCK)
                     + 256, dtype=torch.uint8, device=device)

    def fused(i):
        st = S[i % R]
        gdn.gdn_decode_block_step(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"], d["conv_w"],
                                  d["A_log"], d["dt_bias"], cs, cs, st, st, d["z"], d["norm_w"],
                                  1e-6, 1e-6, y, workspace=ws)

    def three(i):
        st = S[i % R]
        gdn.gdn_input_prologue(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"], d["conv_w"],
                               d["A_log"], d["dt_bias"], cs, cs, None, 1e-6, q, k, v, g, beta)
        gdn.gdn_decode_step(q, k, v, g, beta, st, st, None, o)
        gdn.gdn_gated_rmsnorm(o, d["z"], d["norm_w"], 1e-6, y)

    def run(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    times = {}
    for name, fn in (("fused", fused), ("three_launches", three)):
        for i in range(2 * R):
            fn(i)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn(0)
            torch.cuda.synchronize()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(steps):
                    fn(i)
        gr.replay()
        torch.cuda.synchronize()
        times[name] = min(run(gr.replay) for _ in range(3)) / steps
    byts = decode_block_bytes(N, Hk, Hv)
    ms = times["fused"]
    return {"workload": wl.name + "_block_x100steps", "us_per_step": round(ms * 1e3, 3),
            "us_per_step_three_launches": round(times["three_launches"] * 1e3, 3),
            "speedup_over_three_launches": round(times["three_launches"] / ms, 3),
            "roofline": roofline("hbm", byts / (ms * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "bytes_per_step": byts, "l2": "8 state sets rotated (268 MB)",
            "launch": "100 steps replayed from one CUDA graph per form", "gpu_launches": steps}


SCHEDULES = (("two_pass", 1), ("single_pass", 2), ("tensor_memory", 3),  # C = 64 only
             ("recurrent", 4), ("two_pass_tensor", 5))                  # C = 64 only


def bench_chunked_schedules(torch, gdn, d, wl, chunk, fn, op, n, flush):
    """Mean ms per call of each bf16 schedule, and the one AUTO picks for this shape."""
    s_out = torch.empty_like(d["state0"])
    o = torch.empty_like(d["v"])
    res = {}
    for name, algo in SCHEDULES:
        if algo in (3, 5) and chunk != 64:
            continue
        shape = gdn.make_shape(wl.num_seqs, wl.total_tokens, wl.num_k_heads, wl.num_v_heads,
                               chunk=chunk, algo=algo)
        ws = torch.empty(gdn.gdn_workspace_size(shape, op) + 256, dtype=torch.uint8,
                         device=d["q"].device)

        def step():
            fn(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out, d["cu"], o,
               chunk=chunk, workspace=ws, algo=algo)

        res[name] = statistics.mean(timed_steps(torch, step, n, 3, flush))
        del ws  # the two-pass workspace of the packed workload is ~2 GB: give it back
        torch.cuda.empty_cache()
    many = wl.num_seqs * wl.num_v_heads >= gdn.GDN_SINGLE_PASS_MIN_HEADS
    auto = ("tensor_memory" if chunk == 64 else "single_pass") if many else "two_pass"
    return res, auto


def e2e_pipelined(torch, gdn, d, host, o, s_out, ws, C, steps):
    """ms per step of the prefill from pinned host inputs to pinned host outputs, the steps
    pipelined the way a caller streams batches: each direction's tensors packed into one
    buffer (one copy per step each way), two device buffer sets, the input copy of step
    i + 1 and the output copy of step i - 1 on their own streams while step i computes.
    The timed region starts before the first copy and ends after the last one."""
    def packed(tensors, device):
        offs, n = {}, 0
        for k, v in tensors.items():
            offs[k] = n
            n += (v.numel() * v.element_size() + 255) // 256 * 256
        buf = torch.empty(n, dtype=torch.uint8, device=device, pin_memory=(device == "cpu"))
        views = {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                 for k, v in tensors.items()}
        return buf, views

    dev = o.device
    h_in, h_in_v = packed(host, "cpu")
    for k, v in host.items():
        h_in_v[k].copy_(v)
    outs = {"o": o, "s": s_out}
    sets = []
    for _ in range(2):
        d_in, d_in_v = packed(host, dev)
        d_out, d_out_v = packed(outs, dev)
        h_out, _ = packed(outs, "cpu")
        sets.append((d_in, d_in_v, d_out, d_out_v, h_out))
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        up.wait_event(a)
        down.wait_event(a)
        for i in range(n):
            j = i & 1
            d_in, d_in_v, d_out, d_out_v, h_out = sets[j]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(drained[j])  # step i - 2 is computed and copied out
                d_in.copy_(h_in, non_blocking=True)
                copied[j].record(up)
            comp.wait_event(copied[j])
            gdn.gdn_prefill_chunked(d_in_v["q"], d_in_v["k"], d_in_v["v"], d_in_v["g"], d_in_v["beta"],
                                    d_in_v["state0"], d_out_v["s"], d_in_v["cu"], d_out_v["o"],
                                    chunk=C, workspace=ws)
            computed[j].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[j])
                h_out.copy_(d_out, non_blocking=True)
                drained[j].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
        b.record(comp)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    run(3)
    return run(steps)


def bench_schedules(torch, gdn, gi, device, pk, args, flush):
    """The headline prefill (B=1, H=16, T=4096, C=64) under every bf16 schedule, L2 flushed
    before each step; AUTO takes the two-pass one for these 16 (sequence, head) pairs."""
    wl = gi.prefill_t4096_h16()
    d = dev_inputs(gi.make_inputs(wl), torch, device)
    n = max(5, min(args.steps, 30))
    res, auto = bench_chunked_schedules(torch, gdn, d, wl, 64, gdn.gdn_prefill_chunked,
                                        gdn.GDN_OP_PREFILL, n, flush)
    return {"workload": wl.name, "schedule": auto,
            "us_per_step_by_schedule": {k: round(v * 1e3, 2) for k, v in res.items()},
            "gpu_launches": n * (len(res) + 2)}


def bench_verify(torch, gdn, gi, device, pk, args, flush):
    wl = gi.verify_b128_h32()
    d = dev_inputs(gi.make_inputs(wl), torch, device)
    n = max(5, min(args.steps, 50))
    res, auto = bench_chunked_schedules(torch, gdn, d, wl, 16, gdn.gdn_verify_block,
                                        gdn.GDN_OP_VERIFY, n, flush)
    ms = res[auto]
    flops, byts = prefill_work(wl.lengths, wl.num_k_heads, wl.num_v_heads, 16)
    return {"workload": wl.name, "schedule": auto, "us_per_step": round(ms * 1e3, 2),
            "us_per_step_by_schedule": {k: round(v * 1e3, 2) for k, v in res.items()},
            "tokens_per_s": round(wl.total_tokens / (ms * 1e-3), 1),
            "roofline": roofline("hbm", byts / (ms * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "algorithmic_bytes": byts,
            "gpu_launches": n * (1 if auto == "single_pass" else 2)}


def bench_varlen(torch, gdn, gi, device, pk, args, flush):
    wl = gi.varlen_8seq_hk16_hv32()
    d = dev_inputs(gi.make_inputs(wl), torch, device)
    n = max(5, min(args.steps, 30))
    res, auto = bench_chunked_schedules(torch, gdn, d, wl, 64, gdn.gdn_prefill_chunked,
                                        gdn.GDN_OP_PREFILL, n, flush)
    ms = res[auto]
    flops, byts = prefill_work(wl.lengths, wl.num_k_heads, wl.num_v_heads, 64)
    return {"workload": wl.name, "lengths": wl.lengths, "schedule": auto,
            "us_per_step": round(ms * 1e3, 2),
            "us_per_step_by_schedule": {k: round(v * 1e3, 2) for k, v in res.items()},
            "tokens_per_s": round(wl.total_tokens / (ms * 1e-3), 1),
            "roofline": roofline("hbm", byts / (ms * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "tensor_frac": round(flops / (ms * 1e-3) / 1e12 / pk["bf16"], 4),
            "gpu_launches": n * (1 if auto == "single_pass" else 2)}


def block_dev_inputs(x, torch, device):
    import numpy as np

    def t(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    d = {n: t(x[n + "_st"]) for n in ("q_raw", "k_raw", "v_raw", "z", "conv_state0")}
    for n in ("a", "b", "conv_w", "A_log", "dt_bias", "norm_w", "cu_seqlens"):
        d[n] = t(x[n])
    return d


def prologue_bytes(T, n, hk, hv, s=2, conv_width=4):
    """Raw q/k/v read + q/k/v written, a/b read + g/beta written, the conv FIFO read and
    written, the conv weights read once."""
    C = (2 * hk + hv) * D
    return 2 * T * C * s + 4 * T * hv * 4 + 2 * n * (conv_width - 1) * C * s + C * conv_width * 4


def bench_prologue(torch, gdn, gi, device, pk, args, flush):
    """Input prologue on the packed workload (8 sequences, Hk 16, Hv 32) and on the decode
    batch (32 sequences x 16 heads, one token each, FIFO updated in place)."""
    res = {}
    for key, wl, per_token in (("varlen", gi.varlen_8seq_hk16_hv32(), False),
                               ("decode", gi.decode_b32_h16(), True)):
        d = block_dev_inputs(gi.make_block_inputs(wl), torch, device)
        cu = None if per_token else d["cu_seqlens"]
        outs = [torch.empty_like(d[n]) for n in ("q_raw", "k_raw", "v_raw")]
        g = torch.empty_like(d["a"])
        beta = torch.empty_like(d["a"])
        cs = d["conv_state0"]

        def step():
            gdn.gdn_input_prologue(d["q_raw"], d["k_raw"], d["v_raw"], d["a"], d["b"],
                                   d["conv_w"], d["A_log"], d["dt_bias"], cs, cs, cu, 1e-6,
                                   *outs, g, beta)

        n = max(5, min(args.steps, 50))
        ms = statistics.mean(timed_steps(torch, step, n, 3, flush))
        byts = prologue_bytes(wl.total_tokens, wl.num_seqs, wl.num_k_heads, wl.num_v_heads)
        res[key] = {"workload": wl.name, "us_per_step": round(ms * 1e3, 2),
                    "tokens_per_s": round(wl.total_tokens / (ms * 1e-3), 1),
                    "roofline": roofline("hbm", byts / (ms * 1e-3) / 1e9, pk["hbm"], "GB/s"),
                    "algorithmic_bytes": byts,
                    "gpu_launches": n * (1 if per_token else 2)}
    return res


def bench_gated_rmsnorm(torch, gdn, gi, device, pk, args, flush):
    """Gated RMSNorm of the packed workload's output (bf16 o, z and y)."""
    wl = gi.varlen_8seq_hk16_hv32()
    d = block_dev_inputs(gi.make_block_inputs(wl), torch, device)
    o = torch.randn(d["z"].shape, device=device).to(torch.bfloat16)
    y = torch.empty_like(d["z"])

    def step():
        gdn.gdn_gated_rmsnorm(o, d["z"], d["norm_w"], 1e-6, y)

    n = max(5, min(args.steps, 50))
    ms = statistics.mean(timed_steps(torch, step, n, 3, flush))
    byts = 3 * o.numel() * 2 + D * 4
    return {"workload": wl.name + "_gated_rmsnorm", "us_per_step": round(ms * 1e3, 2),
            "rows_per_s": round(o.numel() // D / (ms * 1e-3), 1),
            "roofline": roofline("hbm", byts / (ms * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "algorithmic_bytes": byts, "gpu_launches": n}


def bench_split(torch, gdn, gi, device, pk, args, flush):
    """Few heads and one long sequence (N=1, H=2, T=65,536): the chunked pass (AUTO: two
    passes) against the sequence-split pass at a few segment lengths."""
    wl = gi.long_t65536_h2()
    d = dev_inputs(gi.make_inputs(wl), torch, device)
    s_out = torch.empty_like(d["state0"])
    o = torch.empty_like(d["v"])
    n = max(3, min(args.steps, 20))
    shape = gdn.make_shape(wl.num_seqs, wl.total_tokens, wl.num_k_heads, wl.num_v_heads, chunk=64)
    ws = torch.empty(gdn.gdn_workspace_size(shape, gdn.GDN_OP_PREFILL) + 256, dtype=torch.uint8,
                     device=device)

    def plain():
        gdn.gdn_prefill_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                                d["cu"], o, chunk=64, workspace=ws)

    res = {"chunked": statistics.mean(timed_steps(torch, plain, n, 2, flush))}
    del ws
    for seg in (2048, 4096, 7296):  # 33, 17 and 9 segments
        sws = torch.empty(gdn.gdn_prefill_split_workspace_size(shape, seg) + 256,
                          dtype=torch.uint8, device=device)

        def split():
            gdn.gdn_prefill_split(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], s_out,
                                  d["cu"], o, segment_len=seg, chunk=64, workspace=sws)

        res["split_%d" % seg] = statistics.mean(timed_steps(torch, split, n, 2, flush))
        del sws
    torch.cuda.empty_cache()
    best = min((v, k) for k, v in res.items() if k.startswith("split"))
    flops, byts = prefill_work(wl.lengths, wl.num_k_heads, wl.num_v_heads, 64)
    return {"workload": wl.name, "us_per_step_by_schedule": {k: round(v * 1e3, 2) for k, v in res.items()},
            "best_split": best[1], "tokens_per_s": round(wl.total_tokens / (best[0] * 1e-3), 1),
            "speedup_over_chunked": round(res["chunked"] / best[0], 3),
            "roofline": roofline("hbm", byts / (best[0] * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "gpu_launches": n * (2 + 3 * 9)}


def bench_accept(torch, gdn, gi, device, pk, args, flush):
    """Draft-verify accept step on the verify workload (128 x 32 heads, 16-token drafts):
    the verify block that captures the per-token deltas, and the rollback of every state
    to its accepted prefix (accepted lengths spread over 0..16)."""
    import numpy as np
    wl = gi.verify_b128_h32()
    d = dev_inputs(gi.make_inputs(wl), torch, device)
    s_out = torch.empty_like(d["state0"])
    o = torch.empty_like(d["v"])
    delta = torch.empty(d["v"].shape, dtype=torch.float32, device=device)
    acc = (gi.raw_u64(0, "accept", wl.num_seqs) % np.uint64(17)).astype(np.int32)
    acc_d = torch.from_numpy(acc).to(device)
    s_rb = torch.empty_like(d["state0"])
    n = max(5, min(args.steps, 50))

    def capture():
        gdn.gdn_verify_block_capture(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"],
                                     s_out, d["cu"], o, delta, chunk=16)

    def rollback():
        gdn.gdn_state_rollback(d["k"], d["g"], delta, d["state0"], acc_d, s_rb, d["cu"])

    ms_cap = statistics.mean(timed_steps(torch, capture, n, 3, flush))
    ms_rb = statistics.mean(timed_steps(torch, rollback, n, 3, flush))
    pairs = wl.num_seqs * wl.num_v_heads
    rb_bytes = pairs * 2 * D * D * 4 + int(acc.sum()) * wl.num_v_heads * (2 * D + 4 * D + 4)
    _, v_bytes = prefill_work(wl.lengths, wl.num_k_heads, wl.num_v_heads, 16)
    cap_bytes = v_bytes + wl.total_tokens * wl.num_v_heads * D * 4
    return {"workload": wl.name + "_accept",
            "capture_us": round(ms_cap * 1e3, 2),
            "capture_roofline": roofline("hbm", cap_bytes / (ms_cap * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "rollback_us": round(ms_rb * 1e3, 2),
            "rollback_roofline": roofline("hbm", rb_bytes / (ms_rb * 1e-3) / 1e9, pk["hbm"], "GB/s"),
            "accepted_tokens": int(acc.sum()), "gpu_launches": 2 * n}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(threads):
    """The prefill workload's inputs and a sample of (sequence, head) chains, one per thread."""
    import gdn_inputs as gi
    wl = gi.prefill_t4096_h16()
    x = gi.make_inputs(wl)
    chains = min(wl.num_v_heads, threads)
    pairs = [(0, h) for h in range(chains)]
    return wl, x, pairs


def cpu_baseline(seconds):
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    wl, x, pairs = oracle_sample(threads)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"], x["cu_seqlens"],
                         pairs=pairs, threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= 100:
            break
    tokens = reps * wl.total_tokens * len(pairs) / wl.num_v_heads
    # one thread: one head of the same workload, repeated for about a tenth of the time
    t1, reps1 = time.perf_counter(), 0
    while True:
        oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"], x["cu_seqlens"],
                         pairs=pairs[:1], threads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= max(0.1, seconds / 10) or reps1 >= 100:
            break
    tokens1 = reps1 * wl.total_tokens / wl.num_v_heads
    return {"value": round(tokens / el, 1), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": "%d of the %d heads of %s (full T), %d repetitions, %.1f s, float64 per-token "
                      "recurrence" % (len(pairs), wl.num_v_heads, wl.name, reps, el),
            "value_1thread": round(tokens1 / el1, 1),
            "sample_1thread": "1 head of %s (full T) on 1 thread, %d repetitions, %.2f s"
                              % (wl.name, reps1, el1)}


def run_reference(args):
    import numpy as np
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    oracle.build()
    threads = oracle.default_threads()
    wl, x, pairs = oracle_sample(threads)

    def make_step(xs):
        def step():
            oracle.recurrent(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], xs["state0"],
                             xs["cu_seqlens"], pairs=pairs, threads=threads)
        return step

    step = make_step(x)
    for _ in range(args.warmup):
        step()
    # exactly --steps timed steps, each a prefix of the sequence sized so that the whole
    # run stays within about two minutes (the recurrence's cost per token does not depend
    # on the prefix length)
    t0 = time.perf_counter()
    step()
    one = time.perf_counter() - t0
    steps = max(1, args.steps)
    T = wl.total_tokens
    if steps * one > 120.0:
        T = max(64, int(T * 120.0 / (steps * one)) // 64 * 64)
        xs = dict(x)
        for name in ("q", "k", "v", "g", "beta"):
            xs[name] = x[name][:T]
        xs["cu_seqlens"] = np.array([0, T], np.int32)
        step = make_step(xs)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t0
    ms = el / steps * 1e3
    tok_step = T * len(pairs) / wl.num_v_heads
    val = round(tok_step / (ms * 1e-3), 1)
    sample = ("%d of the %d heads of %s, the first %d tokens, per step; float64 per-token "
              "recurrence, %d steps" % (len(pairs), wl.num_v_heads, wl.name, T, steps))
    return {"metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "num_seqs": 1, "seq_len": wl.total_tokens,
                       "num_k_heads": wl.num_k_heads, "num_v_heads": wl.num_v_heads, "dk": D,
                       "dv": D, "chunk": wl.chunk, "sample": sample},
            "impl": "reference",
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    line = run_reference(args) if args.impl == "reference" else run_gdn(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
