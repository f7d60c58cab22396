"""The device status word: a bounded wait that runs out is reported to the caller, the
kernel returns normally and the context stays usable.  The wait that runs out is the
self-test's, on a shared-memory barrier that nothing completes and no copy targets."""
import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gdn_testlib import gpu_prefill, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gated_deltanet_linear_05_gb300 import build
    build.build()


def test_wait_timeout_reaches_the_caller_and_the_context_stays_usable():
    import torch
    import gated_deltanet_linear_05_gb300 as gdn
    torch.cuda.set_device(0)
    gdn.gdn_device_status()                      # start from a clear word
    assert gdn.gdn_device_status() == 0
    gdn.gdn_selftest_wait_timeout(polls=1000)    # the wait gives up after 1000 polls
    assert gdn.gdn_device_status() == gdn.GDN_STATUS_WAIT_TIMEOUT
    assert gdn.gdn_device_status() == 0          # reading clears it
    # the context still runs the layer correctly, and a normal call reports nothing
    wl = gi.Workload("after", [300, 65], 1, 2, chunk=64, dtype="bf16", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=5)
    o, s, _ = gpu_prefill(x, wl, o_fp32=True, algo=gdn.GDN_ALGO_TWO_PASS)
    o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"], x["state0"],
                                    x["cu_seqlens"])
    assert rel_err(o, o_ref) <= 2e-2 and rel_err(s, s_ref) <= 2e-2
    assert gdn.gdn_device_status() == 0
