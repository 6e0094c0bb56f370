"""GPU parity of gdr_gated_linear_attn (S <- Diag(alpha) S + k v^T, no erase, no beta) against
the oracle's gated-linear mode: the fp32 FFMA path (fp32 inputs, d = 64, or forced), the
clustered tensor-core kernel (helpers without the solve), the one-CTA tensor-core kernel with
both value-column splits (64 and 128 columns per CTA), both gate kinds, ragged and empty
sequences, entering states, resets and strong decay."""
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


def check(a, dtype, force_simt=False, what="", no_cluster=False):
    import gated_delta_rule_prefill_gb300 as g
    d = dev_inputs(a, dtype)
    out, sf = g.gdr_gated_linear_attn(d["q"], d["k"], d["v"], d["alpha"], S0=d["S0"],
                                      cu_seqlens=d["cu_seqlens"], force_simt=force_simt,
                                      no_cluster=no_cluster)
    torch.cuda.synchronize()
    ref = oracle.gated_linear(a["q"], a["k"], a["v"], a["alpha"], S0=a["S0"],
                              cu_seqlens=a["cu_seqlens"])
    eo, es = err_rows(host(out), ref[0], TOL[dtype]), err_states(host(sf), ref[1], TOL[dtype])
    print("%s: output err %.3g, state err %.3g" % (what, eo, es))
    assert eo <= TOL[dtype] and es <= TOL[dtype], (what, eo, es)
    assert np.isfinite(host(out)).all()


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_gla_fp32_d64(gate):
    wl = gi.custom(seed=301, seqlens=[256, 37, 0, 130], H=2, d_k=64, d_v=64, dtype="f32",
                   gate=gate, s0="normal")
    check(gi.gen_full(wl), "f32", what="fp32 d64 " + gate)


@pytest.mark.parametrize("gate", ["channel", "scalar"])
@pytest.mark.parametrize("case", ["cluster", "dv64", "dv128"])
def test_gla_tensor_core(gate, case):
    # few chains run in clusters with helper CTAs; without clusters, fewer than 120 (sequence,
    # head) pairs run 64 value columns per CTA and more run 128 (too many for clusters anyway)
    lens, H = ([700, 1, 64, 65, 0, 300], 4) if case != "dv128" else ([200, 131, 64, 90], 32)
    wl = gi.custom(seed=302, seqlens=lens, H=H, d_k=128, d_v=128, dtype="bf16", gate=gate,
                   s0="normal")
    check(gi.gen_full(wl), "bf16", what="bf16 %s %s" % (case, gate), no_cluster=(case == "dv64"))


def test_gla_forced_simt_bf16():
    wl = gi.custom(seed=303, seqlens=[300, 100], H=2, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    check(gi.gen_full(wl), "bf16", force_simt=True, what="bf16 forced fp32 path")


@pytest.mark.parametrize("case", ["alpha0", "tiny_alpha", "mixed_decay"])
def test_gla_special_gates(case):
    wl = gi.custom(seed=304, seqlens=[450, 77], H=2, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    if case == "alpha0":
        a["alpha"][::17] = 0.0
    elif case == "tiny_alpha":
        a["alpha"][:] = np.float32(1e-3)
    else:
        a["alpha"][64:128] = np.float32(1e-3)
        a["alpha"][300:340] = np.float32(0.05)
    check(a, "bf16", what=case)


@pytest.mark.parametrize("dtype,d,gate", [("bf16", 128, "channel"), ("bf16", 128, "scalar"),
                                          ("f32", 64, "channel")])
def test_gla_decode_step(dtype, d, gate):
    """gdr_gated_linear_decode_step from a given state, two steps (the second with alpha = 0 on
    some sequences: a reset, then the write), against the oracle's gated-linear mode on one-token
    sequences."""
    import gated_delta_rule_prefill_gb300 as g
    N, H = 40, 3
    wl = gi.Workload("dec", 702, H, d, d, dtype, gate, np.array([1] * N), "zeros")
    S = gi.random_state(703, N, H, d, d)
    Sd = torch.from_numpy(S).cuda()
    cu = np.arange(N + 1)
    for step in range(2):
        a = gi.gen_decode_step(wl, step)
        if step == 1:
            a["alpha"][:5] = 0.0
        d_ = {kk: to_dev(a[kk], dtype) for kk in ("q", "k", "v")}
        out = g.gdr_gated_linear_decode_step(d_["q"], d_["k"], d_["v"], to_dev(a["alpha"], "f32"),
                                             Sd)
        torch.cuda.synchronize()
        ro, rs = oracle.gated_linear(a["q"], a["k"], a["v"], a["alpha"], S0=S, cu_seqlens=cu)
        eo, es = err_rows(host(out), ro, TOL[dtype]), err_states(host(Sd), rs, TOL[dtype])
        print("gla decode %s %s step %d: out %.3g state %.3g" % (dtype, gate, step, eo, es))
        assert eo <= TOL[dtype] and es <= TOL[dtype], (eo, es)
        S = rs


def test_gla_decode_step_prologue():
    """The gated-linear decode step on raw projections (layer prologue on load)."""
    import gated_delta_rule_prefill_gb300 as g
    N, H, d = 32, 2, 128
    wl = gi.Workload("dec", 704, H, d, d, "bf16", "channel", np.array([1] * N), "zeros")
    S = gi.random_state(705, N, H, d, d)
    Sd = torch.from_numpy(S).cuda()
    a = gi.gen_decode_step(wl, 0, raw=True)
    d_ = {kk: to_dev(a[kk], "bf16") for kk in ("q", "k", "v")}
    out = g.gdr_gated_linear_decode_step(d_["q"], d_["k"], d_["v"], to_dev(a["alpha"], "f32"), Sd,
                                         prologue=True)
    torch.cuda.synchronize()
    q, k, al, _ = oracle.layer_prologue(a["q"], a["k"], a["alpha"], a["beta"])
    ro, rs = oracle.gated_linear(q, k, a["v"], al, S0=S, cu_seqlens=np.arange(N + 1))
    eo, es = err_rows(host(out), ro, TOL["bf16"]), err_states(host(Sd), rs, TOL["bf16"])
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)
