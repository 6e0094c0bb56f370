"""GPU parity of the tensor-core prefill kernels with helper CTAs, which the library picks for
bf16, d = 128 workloads with few (sequence, head) chains: the clustered kernel (one chain CTA plus
1-7 helpers per cluster) and the work-queue kernel (one chain CTA per chain, every other SM a
helper taking chunks from a shared queue; needs the full workspace, chosen where clusters would
give a chain one helper).  Every case runs the default dispatch, the work-queue kernel
(GDR_FLAG_PREFER_QUEUE), the clustered kernel (minimum workspace) and the one-CTA-per-chain kernel
(GDR_FLAG_NO_CLUSTER), and checks each against the oracle.  The pair counts below reach different
helper counts."""
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


PATHS = ("default", "queue", "cluster", "one_cta")


def _run(a, path="default"):
    import gated_delta_rule_prefill_gb300 as g
    d = dev_inputs(a, "bf16")
    ws = None
    if path == "cluster":  # the minimum workspace: no operand rings, so no work-queue kernel
        n_seqs = d["cu_seqlens"].numel() - 1
        ws = torch.empty(256 + (n_seqs * 4 + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], workspace=ws,
                            no_cluster=(path == "one_cta"), prefer_queue=(path == "queue"))
    torch.cuda.synchronize()
    return host(out), host(Sf)


def _check(a, what):
    ref = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                             cu_seqlens=a["cu_seqlens"])
    for path in PATHS:
        o, s = _run(a, path)
        eo, es = rel_rows(o, ref[0]), rel_states(s, ref[1])
        print("%s %s: output err %.3g, state err %.3g" % (what, path, eo, es))
        assert eo <= TOL["bf16"] and es <= TOL["bf16"], (what, path, eo, es)
        assert np.isfinite(o).all() and np.isfinite(s).all()


# (sequence lengths, heads): 1, 8, 32, 48 and 72 chains
CASES = {
    "one_chain": ([2000], 1),
    "ragged_8": ([1, 63, 64, 65, 0, 130, 200, 700], 1),
    "chains_32": ([300, 517], 16),
    "chains_48": ([129, 64, 250], 16),
    "chains_72": ([190, 33, 260], 24),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_cluster_prefill(case, gate):
    lens, H = CASES[case]
    wl = gi.custom(seed=61 + len(lens) + H, seqlens=lens, H=H, d_k=128, d_v=128, dtype="bf16",
                   gate=gate, s0="normal")
    _check(gi.gen_full(wl), "%s %s" % (case, gate))


@pytest.mark.parametrize("case", ["alpha0", "tiny_alpha", "mixed_decay"])
def test_cluster_special_gates(case):
    """Resets and strong-decay chunks, which the helper CTAs form from direct pairwise
    exponentials instead of the factorised Gram product."""
    wl = gi.custom(seed=71, seqlens=[450, 77], H=2, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    if case == "alpha0":
        a["alpha"][::17] = 0.0
    elif case == "tiny_alpha":
        a["alpha"][:] = np.float32(1e-3)
    else:  # strong decay in some chunks only, so both forms meet in one chain
        a["alpha"][64:128] = np.float32(1e-3)
        a["alpha"][300:340] = np.float32(0.05)
    _check(a, case)


def test_cluster_two_calls_in_a_row():
    """Back-to-back launches on one stream reuse nothing: the second call's results do not
    depend on the first (different inputs, same shapes)."""
    wl = gi.custom(seed=91, seqlens=[640, 100], H=4, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    b = gi.gen_full(gi.custom(seed=92, seqlens=[640, 100], H=4, d_k=128, d_v=128, dtype="bf16",
                              s0="normal"))
    first = _run(a)
    second = _run(b)
    again = _run(a)
    np.testing.assert_array_equal(first[0], again[0])
    np.testing.assert_array_equal(first[1], again[1])
    ref = oracle.gated_delta(b["q"], b["k"], b["v"], b["alpha"], b["beta"], S0=b["S0"],
                             cu_seqlens=b["cu_seqlens"])
    assert rel_rows(second[0], ref[0]) <= TOL["bf16"]


def test_queue_repeated_calls():
    """The work-queue kernel (72 chains: one helper CTA per chain or so) called back to back:
    every call ends without a device-check failure and gives the same bits."""
    import gated_delta_rule_prefill_gb300 as g
    lens, H = CASES["chains_72"]
    wl = gi.custom(seed=93, seqlens=lens, H=H, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "bf16")
    n = g.gdr_prefill_workspace_size(len(lens), H, 128, 128, "bf16")
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    first = None
    for _ in range(6):
        out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                                cu_seqlens=d["cu_seqlens"], workspace=ws, prefer_queue=True)
        assert g.gdr_workspace_status(ws) == 0
        cur = (host(out), host(Sf))
        if first is None:
            first = cur
        else:
            np.testing.assert_array_equal(cur[0], first[0])
            np.testing.assert_array_equal(cur[1], first[1])


def test_cluster_back_to_back_launches():
    """Hundreds of launches with helper CTAs back to back on one stream (32 chains of 64
    chunks: the plain, output-gated and gated-linear clustered chains and the work-queue kernel
    with 3.75 helpers per chain, in turn): no bounded wait gives up -- a chain thread that slept
    through two phases of a barrier would -- and every repeat gives the same bits."""
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=94, seqlens=[4096], H=32, d_k=128, d_v=128, dtype="bf16", s0="normal")
    d = gi.device_full(wl, "cuda")
    gate_in = torch.randn_like(d["v"])
    ws = torch.empty(g.gdr_prefill_workspace_size(1, 32, 128, 128, "bf16"), dtype=torch.uint8,
                     device="cuda")
    g.gdr_query_device_status()
    outs = [torch.empty_like(d["v"]) for _ in range(4)]
    firsts = []
    for rep in range(100):
        o = [g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                           cu_seqlens=d["cu_seqlens"], out=outs[0], workspace=ws)[0],
             g.gdr_prefill_output_gate(d["q"], d["k"], d["v"], d["alpha"], d["beta"], gate_in,
                                       S0=d["S0"], cu_seqlens=d["cu_seqlens"], out=outs[1],
                                       workspace=ws)[0],
             g.gdr_gated_linear_attn(d["q"], d["k"], d["v"], d["alpha"], S0=d["S0"],
                                     cu_seqlens=d["cu_seqlens"], out=outs[2], workspace=ws)[0],
             g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                           cu_seqlens=d["cu_seqlens"], out=outs[3], workspace=ws,
                           prefer_queue=True)[0]]
        if rep == 0 or rep == 99:
            firsts.append([x.clone() for x in o])
    assert g.gdr_workspace_status(ws) == 0
    assert g.gdr_query_device_status() == g._abi.GDR_OK
    for x, y in zip(firsts[0], firsts[1]):
        assert torch.equal(x, y)
