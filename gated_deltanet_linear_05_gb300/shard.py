"""Data-parallel sharding of the layer across ranks (one process per GPU).

Every (sequence, v-head) chain of the gated delta rule is independent ("Qwen3.5-9B-npu"
model card, section "How it works": the state of one head of one sequence is carried
only through that sequence's own tokens), so a batch of sequences splits across ranks
by whole sequences with no exchange step: each rank runs the layer on its sequences'
tokens and states; nothing crosses ranks on the data path.  This module holds the host
side of that split -- the plan (which rank takes which sequences, balanced by tokens),
the slicing of the packed inputs and of the states, the merge of the per-rank results --
and the one reduction the benchmark needs (the slowest rank's time).

Works on numpy arrays or torch tensors (CPU or CUDA) alike; no GPU code lives here.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np


def plan(lengths: Sequence[int], world: int) -> List[List[int]]:
    """Sequence indices per rank: longest sequences first onto the least-loaded rank
    (greedy balancing of the token counts); each rank's list is in ascending order."""
    if world < 1:
        raise ValueError("world must be >= 1")
    load = [0] * world
    owned: List[List[int]] = [[] for _ in range(world)]
    for n in sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i)):
        r = min(range(world), key=lambda j: (load[j], j))
        owned[r].append(n)
        load[r] += int(lengths[n])
    return [sorted(o) for o in owned]


def _cat(parts, like):
    if hasattr(like, "new_empty"):  # torch
        import torch
        return torch.cat(parts) if parts else like[:0]
    return np.concatenate(parts) if parts else like[:0]


def slice_inputs(x: Dict[str, object], seqs: Sequence[int]) -> Dict[str, object]:
    """The inputs of the sequences `seqs` as a packed batch of their own.

    x holds q, k, v (token-major: [T, heads, d]), g, beta ([T, Hv]), state0
    ([N, Hv, dk, dv] or None) and cu_seqlens ([N + 1]); the result has the same keys."""
    cu = np.asarray(x["cu_seqlens"].cpu() if hasattr(x["cu_seqlens"], "cpu") else x["cu_seqlens"])
    out: Dict[str, object] = {}
    for name in ("q", "k", "v", "g", "beta"):
        a = x[name]
        out[name] = _cat([a[int(cu[n]):int(cu[n + 1])] for n in seqs], a)
    s0 = x.get("state0")
    out["state0"] = None if s0 is None else _cat([s0[n:n + 1] for n in seqs], s0)
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    new_cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    new_cu[1:] = np.cumsum(lens, dtype=np.int64)
    if hasattr(x["cu_seqlens"], "new_tensor"):
        out["cu_seqlens"] = x["cu_seqlens"].new_tensor(new_cu)
    else:
        out["cu_seqlens"] = new_cu
    return out


def merge(cu_seqlens, owned: List[List[int]], outputs: List[object], states: List[object]):
    """Reassemble per-rank outputs o ([T_r, Hv, dv]) and final states ([N_r, Hv, dk, dv])
    into the full batch's order.  Returns (o, state) as numpy arrays."""
    cu = np.asarray(cu_seqlens)
    n_seq = len(cu) - 1
    o_full = None
    s_full = None
    for seqs, o_r, s_r in zip(owned, outputs, states):
        o_r = np.asarray(o_r)
        s_r = np.asarray(s_r)
        if o_full is None:
            o_full = np.zeros((int(cu[-1]),) + o_r.shape[1:], dtype=o_r.dtype)
            s_full = np.zeros((n_seq,) + s_r.shape[1:], dtype=s_r.dtype)
        pos = 0
        for i, n in enumerate(seqs):
            ln = int(cu[n + 1] - cu[n])
            o_full[int(cu[n]):int(cu[n + 1])] = o_r[pos:pos + ln]
            s_full[n] = s_r[i]
            pos += ln
    return o_full, s_full


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (barrier first);
    `value` itself when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.barrier()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
