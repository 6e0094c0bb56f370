"""Failure detection on the GPU without a fault: a bounded wait is made to run out (one warp
waits, with the tensor-core kernels' bounded mbarrier wait, on a barrier that nothing
completes), the timeout is read back through both status paths, and the context stays usable
for a prefill checked against the oracle."""
import time

import numpy as np
import pytest
import torch

import gdr_inputs as gi
import oracle
from tests.parity import TOL, dev_inputs, host, rel_rows, rel_states

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_wait_timeout_reported_and_context_usable():
    import gated_delta_rule_prefill_gb300 as g
    from gated_delta_rule_prefill_gb300 import _abi
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    g.gdr_query_device_status()  # start from a clear per-device word
    assert g.gdr_workspace_status(ws) == _abi.GDR_DEVCHECK_OK

    limit_ns = 50_000_000
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g.gdr_check_wait_timeout(ws, limit_ns)
    code = g.gdr_workspace_status(ws)  # synchronises
    waited = time.perf_counter() - t0
    assert code == _abi.GDR_DEVCHECK_TIMEOUT
    assert waited >= limit_ns * 1e-9, waited  # the wait ran to its limit, no longer than needed
    assert waited < 5.0, waited
    assert g.gdr_query_device_status() == _abi.GDR_ERR_DEVICE_CHECK
    assert g.gdr_query_device_status() == _abi.GDR_OK  # taken: cleared
    assert g.gdr_workspace_status(ws) == _abi.GDR_DEVCHECK_OK  # read and cleared above

    # the context is still usable: a clustered tensor-core prefill, checked against the oracle
    wl = gi.custom(seed=31, seqlens=[300, 65], H=2, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "bf16")
    out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    ro, rs = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                                cu_seqlens=a["cu_seqlens"])
    eo, es = rel_rows(host(out), ro), rel_states(host(Sf), rs)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)
    assert np.isfinite(host(out)).all()
    assert g.gdr_query_device_status() == _abi.GDR_OK
