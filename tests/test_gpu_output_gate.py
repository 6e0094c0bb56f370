"""GPU parity of gdr_prefill_output_gate (the prefill with out = o * sigmoid(g)) against the
oracle's gated delta rule followed by its output gate, on every prefill path: the clustered
and work-queue kernels with helper CTAs, the one-CTA tensor-core kernel, and the fp32 kernel
(fp32 inputs and forced).  Gate pre-activations ~ N(0, 2^2), so the gate spans nearly shut to
nearly open; final states must equal those of the ungated rule."""
import numpy as np
import pytest
import torch

import gdr_inputs as gi
import oracle
from tests.parity import TOL, dev_inputs, err_rows, err_states, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run(a, dtype, path="default", seed=401):
    import gated_delta_rule_prefill_gb300 as g
    T, H = a["q"].shape[:2]
    dv = a["v"].shape[2]
    gate = np.random.default_rng(seed).normal(0.0, 2.0, (T, H, dv))
    if dtype == "bf16":
        gate = gi.bf16_round(gate)
    d = dev_inputs(a, dtype)
    gd = to_dev(gate, dtype)
    out, sf = g.gdr_prefill_output_gate(d["q"], d["k"], d["v"], d["alpha"], d["beta"], gd,
                                        S0=d["S0"], cu_seqlens=d["cu_seqlens"],
                                        force_simt=(path == "simt"),
                                        no_cluster=(path == "one_cta"),
                                        prefer_queue=(path == "queue"))
    torch.cuda.synchronize()
    ref_o, ref_s = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                                      cu_seqlens=a["cu_seqlens"])
    ref = oracle.output_gate(ref_o, gate)
    eo, es = err_rows(host(out), ref, TOL[dtype]), err_states(host(sf), ref_s, TOL[dtype])
    print("%s %s: output err %.3g, state err %.3g" % (dtype, path, eo, es))
    assert eo <= TOL[dtype] and es <= TOL[dtype], (path, eo, es)


@pytest.mark.parametrize("path", ["default", "queue", "one_cta", "simt"])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_output_gate_bf16(path, gate):
    wl = gi.custom(seed=402, seqlens=[700, 1, 64, 65, 0, 300], H=4, d_k=128, d_v=128,
                   dtype="bf16", gate=gate, s0="normal")
    run(gi.gen_full(wl), "bf16", path)


def test_output_gate_fp32_d64():
    wl = gi.custom(seed=403, seqlens=[256, 37, 130], H=2, d_k=64, d_v=64, dtype="f32",
                   gate="channel", s0="normal")
    run(gi.gen_full(wl), "f32")

