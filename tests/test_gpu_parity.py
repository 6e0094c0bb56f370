"""GPU parity of the three calls against the CPU oracle on seeded inputs (small and medium
sizes: several chunks, ragged tails, empty sequences, special gates).  Every call goes through
the C ABI (ctypes binding); every expected value comes from oracle/."""
import numpy as np
import pytest
import torch

import gdr_inputs as gi
import oracle
from tests.parity import TOL, dev_inputs, err_rows, err_states, host, rel_rows, rel_states, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_prefill_gb300 as g
    return g


def run_prefill(a, dtype, force_simt=False, linear=False, pass_cu=True):
    import gated_delta_rule_prefill_gb300 as g
    d = dev_inputs(a, dtype)
    cu = d["cu_seqlens"] if pass_cu else None
    if linear:
        out, Sf = g.gdr_linear_attn(d["q"], d["k"], d["v"], S0=d["S0"], cu_seqlens=cu,
                                    force_simt=force_simt)
    else:
        out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                                cu_seqlens=cu, force_simt=force_simt)
    torch.cuda.synchronize()
    return host(out), host(Sf)


def ref_prefill(a, linear=False):
    if linear:
        return oracle.linear_attn(a["q"], a["k"], a["v"], S0=a["S0"], cu_seqlens=a["cu_seqlens"])
    return oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                              cu_seqlens=a["cu_seqlens"])


def check(got, ref, tol, what):
    eo = err_rows(got[0], ref[0], tol)
    es = err_states(got[1], ref[1], tol)
    assert eo <= tol and es <= tol, "%s: output err %.3g, state err %.3g (tol %g)" % (
        what, eo, es, tol)
    return eo, es


def test_config0_kda_t256_d64_f32():
    wl = gi.workload("kda_t256_d64_f32")
    a = gi.gen_full(wl)
    check(run_prefill(a, "f32"), ref_prefill(a), TOL["f32"], wl.name)


RAGGED = [1, 63, 64, 65, 0, 130, 200]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("force_simt", [False, True])
def test_prefill_ragged(d, gate, dtype, force_simt):
    wl = gi.custom(seed=11 + d, seqlens=RAGGED, H=3, d_k=d, d_v=d, dtype=dtype, gate=gate,
                   s0="normal")
    a = gi.gen_full(wl)
    got = run_prefill(a, dtype, force_simt=force_simt)
    ref = ref_prefill(a)
    eo, es = check(got, ref, TOL[dtype], "prefill d=%d %s %s" % (d, gate, dtype))
    if dtype == "f32" or force_simt:
        # the fp32 FFMA path keeps the state to fp32 rounding even with bf16 inputs
        es = err_states(got[1], ref[1], TOL["f32"])
        assert es <= TOL["f32"], es


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_linear_attn_ragged(d, dtype):
    wl = gi.custom(seed=21 + d, seqlens=RAGGED, H=2, d_k=d, d_v=d, dtype=dtype, s0="normal")
    a = gi.gen_full(wl)
    check(run_prefill(a, dtype, linear=True), ref_prefill(a, linear=True), TOL[dtype],
          "linear d=%d %s" % (d, dtype))


# few (sequence, head) pairs and long sequences: the linear pass splits each sequence into runs of
# whole chunks, one CTA each, every run starting from the state its earlier chunks imply
@pytest.mark.parametrize("lens,H", [([9000], 1), ([5000, 4000, 64], 2), ([3000, 2500], 3)])
def test_linear_attn_segmented(lens, H):
    wl = gi.custom(seed=23 + H, seqlens=lens, H=H, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    check(run_prefill(a, "bf16", linear=True), ref_prefill(a, linear=True), TOL["bf16"],
          "linear segmented %s H=%d" % (lens, H))


@pytest.mark.parametrize("lens,H", [([9000], 1), ([5000, 4000, 64], 2)])
def test_linear_attn_segmented_min_workspace(lens, H):
    """The same runs with a workspace too small to hold the runs' sums (header and visiting
    order only): each run rebuilds its entering state from the chunks before it instead of
    reading the sums a first launch wrote.  Also the normalised phi-linear form, whose runs
    rebuild z the same way."""
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=33 + H, seqlens=lens, H=H, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "bf16")
    n = len(lens)
    ws = torch.empty(256 + (4 * n + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    out, sf = g.gdr_linear_attn(d["q"], d["k"], d["v"], S0=d["S0"], cu_seqlens=d["cu_seqlens"],
                                workspace=ws)
    torch.cuda.synchronize()
    check((host(out), host(sf)), ref_prefill(a, linear=True), TOL["bf16"],
          "linear min-workspace %s H=%d" % (lens, H))
    o2, s2, z2 = g.gdr_normalized_linear_attn(d["q"], d["k"], d["v"], eps=1e-6, S0=d["S0"],
                                              cu_seqlens=d["cu_seqlens"], workspace=ws)
    torch.cuda.synchronize()
    ro, rs, rz = oracle.normalized_linear(a["q"], a["k"], a["v"], S0=a["S0"],
                                          cu_seqlens=a["cu_seqlens"], eps=1e-6)
    check((host(o2), host(s2)), (ro, rs), TOL["bf16"], "normalised min-workspace")
    assert rel_rows(host(z2), rz) <= TOL["bf16"]


@pytest.mark.parametrize("linear", [False, True])
def test_in_place_state_hand_off(linear):
    """S_final = S0 (the documented in-place hand-off) on a workload whose linear pass would
    otherwise be split into runs, and whose gated pass runs with helper CTAs."""
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=27, seqlens=[5000, 4000], H=2, d_k=128, d_v=128, dtype="bf16",
                   s0="normal")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "bf16")
    S = d["S0"].clone()
    if linear:
        out, _ = g.gdr_linear_attn(d["q"], d["k"], d["v"], S0=S, S_final=S,
                                   cu_seqlens=d["cu_seqlens"])
    else:
        out, _ = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=S, S_final=S,
                               cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    check((host(out), host(S)), ref_prefill(a, linear=linear), TOL["bf16"],
          "in-place %s" % ("linear" if linear else "gated"))


@pytest.mark.parametrize("case", ["alpha0", "alpha1_beta0", "beta1", "tiny_alpha"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_special_gates(case, dtype):
    wl = gi.custom(seed=31, seqlens=[150, 77], H=2, d_k=128, d_v=128, dtype=dtype, s0="normal")
    a = gi.gen_full(wl)
    if case == "alpha0":
        a["alpha"][::17] = 0.0  # full resets, some inside chunks
    elif case == "alpha1_beta0":
        a["alpha"][40:90] = 1.0
        a["beta"][40:90] = 0.0
    elif case == "beta1":
        a["beta"][:] = 1.0
    elif case == "tiny_alpha":
        a["alpha"][:] = np.float32(1e-3)  # strong decay everywhere (G spans ~ -440 per chunk)
    check(run_prefill(a, dtype), ref_prefill(a), TOL[dtype], "%s %s" % (case, dtype))


def test_single_sequence_without_cu_seqlens():
    wl = gi.custom(seed=41, seqlens=[333], H=2, d_k=128, d_v=128, dtype="bf16", s0="normal")
    a = gi.gen_full(wl)
    check(run_prefill(a, "bf16", pass_cu=False), ref_prefill(a), TOL["bf16"], "no cu")


def test_empty_token_axis():
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=42, seqlens=[0, 0], H=2, d_k=64, d_v=64, dtype="f32", s0="normal")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "f32")
    out, Sf = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert out.numel() == 0
    np.testing.assert_array_equal(host(Sf), a["S0"])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps(d, gate, dtype):
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.Workload("dec", 51, 4, d, d, dtype, gate, np.array([1] * 37), "zeros")
    S = gi.random_state(52, 37, 4, d, d, std=0.3)
    S_dev = torch.from_numpy(S).cuda()
    S_ref = S.astype(np.float64)
    for step in range(3):
        x = gi.gen_decode_step(wl, step)
        if step == 1:
            x["alpha"][::5] = 0.0
            x["beta"][::7] = 1.0
        out = g.gdr_decode_step(to_dev(x["q"], dtype), to_dev(x["k"], dtype),
                                to_dev(x["v"], dtype), to_dev(x["alpha"], "f32"),
                                to_dev(x["beta"], "f32"), S_dev)
        ref_o, S_ref = oracle.decode_step(x["q"], x["k"], x["v"], x["alpha"], x["beta"], S_ref)
        torch.cuda.synchronize()
        eo = err_rows(host(out), ref_o, TOL[dtype])
        es = err_states(host(S_dev), S_ref, TOL["f32"])
        assert eo <= TOL[dtype] and es <= TOL["f32"], (step, eo, es)


def test_decode_continues_prefill():
    """A prefill of n tokens followed by m decode steps equals a prefill of n + m tokens."""
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=61, seqlens=[100, 70, 90], H=2, d_k=128, d_v=128, dtype="bf16",
                   s0="normal")
    a = gi.gen_full(wl)
    ref_o, ref_S = ref_prefill(a)
    d = dev_inputs(a, "bf16")
    m = 5
    cu = a["cu_seqlens"]
    lens = np.diff(cu)
    # prefill the first len - m tokens of every sequence
    keep = torch.from_numpy(np.concatenate([np.arange(cu[i], cu[i + 1] - m)
                                            for i in range(3)])).cuda()
    cu_p = np.concatenate([[0], np.cumsum(lens - m)]).astype(np.int32)
    _, S = g.gdr_prefill(d["q"][keep].contiguous(), d["k"][keep].contiguous(),
                         d["v"][keep].contiguous(), d["alpha"][keep].contiguous(),
                         d["beta"][keep].contiguous(), S0=d["S0"],
                         cu_seqlens=torch.from_numpy(cu_p).cuda())
    for j in range(m):
        idx = torch.from_numpy(cu[1:] - m + j).cuda()
        o = g.gdr_decode_step(d["q"][idx].contiguous(), d["k"][idx].contiguous(),
                              d["v"][idx].contiguous(), d["alpha"][idx].contiguous(),
                              d["beta"][idx].contiguous(), S)
        torch.cuda.synchronize()
        assert rel_rows(host(o), ref_o[cu[1:] - m + j]) <= TOL["bf16"]
    assert rel_states(host(S), ref_S) <= TOL["bf16"]


def test_device_check_bad_seqlens():
    import gated_delta_rule_prefill_gb300 as g
    from gated_delta_rule_prefill_gb300 import _abi
    wl = gi.custom(seed=71, seqlens=[10, 20], H=1, d_k=64, d_v=64, dtype="f32")
    a = gi.gen_full(wl)
    d = dev_inputs(a, "f32")
    ws = torch.empty(g.gdr_prefill_workspace_size(2), dtype=torch.uint8, device="cuda")
    g.gdr_query_device_status()  # start from a clear per-device word
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")  # not monotone
    g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], cu_seqlens=bad, workspace=ws)
    assert g.gdr_workspace_status(ws) == 1
    # the per-device word holds the failure until it is taken, then reads clear
    assert g.gdr_query_device_status() == _abi.GDR_ERR_DEVICE_CHECK
    assert g.gdr_query_device_status() == _abi.GDR_OK
    beyond = torch.tensor([0, 10, 31], dtype=torch.int32, device="cuda")  # past total_tokens
    g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], cu_seqlens=beyond, workspace=ws)
    assert g.gdr_workspace_status(ws) == 1
    # a later good call does not clear it: the word keeps the first failure since the last query
    g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], cu_seqlens=d["cu_seqlens"],
                  workspace=ws)
    assert g.gdr_workspace_status(ws) == 0
    assert g.gdr_query_device_status() == _abi.GDR_ERR_DEVICE_CHECK
    g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], cu_seqlens=d["cu_seqlens"],
                  workspace=ws)
    assert g.gdr_query_device_status() == _abi.GDR_OK
