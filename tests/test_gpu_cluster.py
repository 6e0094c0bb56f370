"""GPU parity of the clustered tensor-core prefill (one chain CTA plus helper CTAs per
(sequence, head) chain), which the library picks for bf16, d = 128 workloads with few chains.

The cluster size follows from the number of chains (the largest cluster of which one per chain
fits on the device), so the pair counts below reach different helper counts; each case runs the
default dispatch and the one-CTA kernel (GDR_FLAG_NO_CLUSTER) and checks both against the
oracle."""
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


def _run(a, no_cluster):
    import gated_delta_rule_prefill_gb300 as g
    d = dev_inputs(a, "bf16")
    out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], no_cluster=no_cluster)
    torch.cuda.synchronize()
    return host(out), host(Sf)


def _check(a, what):
    ref = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                             cu_seqlens=a["cu_seqlens"])
    for no_cluster in (False, True):
        o, s = _run(a, no_cluster)
        eo, es = rel_rows(o, ref[0]), rel_states(s, ref[1])
        print("%s no_cluster=%s: output err %.3g, state err %.3g" % (what, no_cluster, eo, es))
        assert eo <= TOL["bf16"] and es <= TOL["bf16"], (what, no_cluster, eo, es)
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
    first = _run(a, False)
    second = _run(b, False)
    again = _run(a, False)
    np.testing.assert_array_equal(first[0], again[0])
    np.testing.assert_array_equal(first[1], again[1])
    ref = oracle.gated_delta(b["q"], b["k"], b["v"], b["alpha"], b["beta"], S0=b["S0"],
                             cu_seqlens=b["cu_seqlens"])
    assert rel_rows(second[0], ref[0]) <= TOL["bf16"]
