"""Edge cases of the layer on the GPU against the float64 oracle: batches whose sequences
are all empty, zero write strength (beta = 0: pure decay, a closed form), one long
sequence (65,536 tokens, index arithmetic far past the bench sizes) and a large decode
batch (256 sequences x 32 v-heads, sampled (sequence, head) chains)."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import device_inputs, gpu_prefill, rel_err, to_dev, to_np

pytestmark = pytest.mark.gpu

ALGOS = {"two_pass": 1, "single_pass": 2, "tensor_memory": 3, "recurrent": 4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


@pytest.mark.parametrize("algo", list(ALGOS))
def test_all_sequences_empty_pass_the_state_through(algo):
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    n, hv = 3, 4
    s0 = (0.1 * gi.normal(1, "s0", n * hv * 128 * 128)).astype(np.float32).reshape(n, hv, 128, 128)
    e = lambda shape, dt=torch.bfloat16: torch.empty(shape, dtype=dt, device="cuda")
    q, k, v = e((0, 2, 128)), e((0, 2, 128)), e((0, hv, 128))
    g, beta = e((0, hv), torch.float32), e((0, hv), torch.float32)
    cu = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    s_in = to_dev(s0, "f32")
    for fn in (gdn.gdn_prefill_chunked, gdn.gdn_verify_block):
        s_out = torch.full_like(s_in, float("nan"))
        fn(q, k, v, g, beta, s_in, s_out, cu, torch.empty_like(v), chunk=64, algo=ALGOS[algo])
        torch.cuda.synchronize()
        assert np.array_equal(to_np(s_out), s0.astype(np.float64)), fn.__name__
    s_out = torch.full_like(s_in, float("nan"))
    gdn.gdn_decode_step(q, k, v, g, beta, s_in, s_out, cu, torch.empty_like(v))
    torch.cuda.synchronize()
    assert np.array_equal(to_np(s_out), s0.astype(np.float64))


@pytest.mark.parametrize("algo", list(ALGOS))
def test_zero_write_strength_is_pure_decay(algo):
    """beta = 0: S_T = exp(G_T) S0 and o_t = exp(G_t) q_t^T S0 (the page's token_valid
    padding rule applied to every token)."""
    wl = gi.Workload("b0", [100, 64, 3], 2, 4, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=13)
    x["beta"][:] = 0.0
    o, s, _ = gpu_prefill(x, wl, o_fp32=True, algo=ALGOS[algo])
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"])
    cu = x["cu_seqlens"]
    for n in range(wl.num_seqs):
        G = np.cumsum(x["g"][cu[n]:cu[n + 1]].astype(np.float64), axis=0)   # [L, Hv]
        for h in range(wl.num_v_heads):
            gt = G[-1, h] if len(G) else 0.0
            closed = np.exp(gt) * x["state0"][n, h].astype(np.float64)
            np.testing.assert_allclose(s_ref[n, h], closed, rtol=1e-12, atol=1e-15)
    assert rel_err(s, s_ref) <= 2e-2 and rel_err(o, o_ref) <= 2e-2


def test_one_long_sequence():
    """T = 65,536 tokens (1,024 blocks), 2 v-heads sharing a k-head, two-pass schedule."""
    wl = gi.Workload("long", [65536], 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=17)
    o, s, _ = gpu_prefill(x, wl, o_fp32=True)
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"])
    assert rel_err(o, o_ref) <= 2e-2, rel_err(o, o_ref)
    assert rel_err(s, s_ref) <= 2e-2, rel_err(s, s_ref)


def test_large_decode_batch_sampled():
    """256 sequences x 32 v-heads (16 k-heads), one token each, in place; 64 sampled chains
    against the oracle and every state finite."""
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    wl = gi.Workload("dec_big", [1] * 256, 16, 32, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=19)
    d = device_inputs(x, "bf16")
    o32 = torch.empty(d["v"].shape, dtype=torch.float32, device="cuda")
    gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state0"], d["state0"],
                        None, o32)
    torch.cuda.synchronize()
    u = gi.raw_u64(0, "pairs", 64)
    pairs = sorted({(int(a % np.uint64(256)), int((a >> np.uint64(20)) % np.uint64(32))) for a in u})
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"], pairs=pairs)
    s = d["state0"]
    for n, h in pairs:
        sn = to_np(s[n, h])
        assert rel_err(sn, s_ref[n, h]) <= 2e-2, (n, h)
        assert rel_err(to_np(o32[n, h]), o_ref[n, h]) <= 2e-2, (n, h)
    assert torch.isfinite(s).all()
