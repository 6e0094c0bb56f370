"""GPU parity of the layer prologue on load (GDR_FLAG_LAYER_PROLOGUE): q, k, alpha, beta are the
layer's raw projections (xq, xk ~ N(0, 1); a = 4 - N(0, 1); b ~ N(0, 1)) and every kernel maps
them on load.  The expected values are the oracle's layer prologue followed by its rule, on
every prefill path (clustered, work-queue, one-CTA tensor-core, fp32), the output-gated and
gated-linear entries, the decode step and the host pipeline; plus the prologue's edge cases
(silu rows of zero, gates saturated shut and open)."""
import numpy as np
import pytest
import torch

import gdr_inputs as gi
import oracle
from tests.parity import TOL, dev_inputs, err_rows, err_states, host, rel_rows, rel_states, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def mapped(a):
    """The oracle's layer prologue on raw inputs: (q, k, alpha, beta) in fp64."""
    return oracle.layer_prologue(a["q"], a["k"], a["alpha"], a["beta"])


def check(name, out, sf, ref_o, ref_s, dtype):
    eo = err_rows(host(out), ref_o, TOL[dtype])
    es = err_states(host(sf), ref_s, TOL[dtype]) if sf is not None else 0.0
    print("%s: output err %.3g, state err %.3g" % (name, eo, es))
    assert eo <= TOL[dtype] and es <= TOL[dtype], (name, eo, es)


def run_prefill(a, dtype, path="default", g=None):
    import gated_delta_rule_prefill_gb300 as gd
    d = dev_inputs(a, dtype)
    kw = dict(S0=d["S0"], cu_seqlens=d["cu_seqlens"], force_simt=(path == "simt"),
              no_cluster=(path == "one_cta"), prefer_queue=(path == "queue"), prologue=True)
    if g is None:
        out, sf = gd.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], **kw)
    else:
        out, sf = gd.gdr_prefill_output_gate(d["q"], d["k"], d["v"], d["alpha"], d["beta"],
                                             to_dev(g, dtype), **kw)
    torch.cuda.synchronize()
    q, k, al, be = mapped(a)
    ref_o, ref_s = oracle.gated_delta(q, k, a["v"], al, be, S0=a["S0"],
                                      cu_seqlens=a["cu_seqlens"])
    if g is not None:
        ref_o = oracle.output_gate(ref_o, g)
    check("prefill %s %s" % (dtype, path), out, sf, ref_o, ref_s, dtype)


@pytest.mark.parametrize("path", ["default", "queue", "one_cta", "simt"])
@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_prologue_prefill_bf16(path, gate):
    wl = gi.custom(seed=501, seqlens=[700, 1, 64, 65, 0, 300], H=4, d_k=128, d_v=128,
                   dtype="bf16", gate=gate, s0="normal")
    run_prefill(gi.gen_full(wl, raw=True), "bf16", path)


def test_prologue_prefill_fp32_d64():
    wl = gi.custom(seed=502, seqlens=[256, 37, 130], H=2, d_k=64, d_v=64, dtype="f32",
                   gate="channel", s0="normal")
    run_prefill(gi.gen_full(wl, raw=True), "f32")


def test_prologue_prefill_bf16_d64():
    wl = gi.custom(seed=503, seqlens=[200, 129], H=3, d_k=64, d_v=64, dtype="bf16",
                   gate="scalar", s0="normal")
    run_prefill(gi.gen_full(wl, raw=True), "bf16")


def test_prologue_output_gate():
    wl = gi.custom(seed=504, seqlens=[513, 70], H=4, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    a = gi.gen_full(wl, raw=True)
    T = a["q"].shape[0]
    g = gi.bf16_round(np.random.default_rng(505).normal(0.0, 2.0, (T, 4, 128)))
    run_prefill(a, "bf16", "default", g=g)


def test_prologue_edge_rows_and_saturated_gates():
    """Rows of xq / xk that are all zero (silu 0, normalised to 0) or all very negative (silu
    underflows towards 0 relative to the row), and raw gates of -100 (alpha, beta = 0: the
    state resets, nothing is written) and +100 (alpha, beta = 1)."""
    wl = gi.custom(seed=506, seqlens=[300, 77], H=2, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    a = gi.gen_full(wl, raw=True)
    a["q"][5] = 0.0
    a["k"][9] = 0.0
    a["k"][11] = -30.0
    a["q"][12, :, :64] = -50.0
    a["alpha"][20:24] = -100.0
    a["alpha"][40:60] = 100.0
    a["beta"][30:33] = -100.0
    a["beta"][50:70] = 100.0
    for path in ("default", "simt"):
        run_prefill(a, "bf16", path)


@pytest.mark.parametrize("gate", ["channel", "scalar"])
def test_prologue_gated_linear(gate):
    import gated_delta_rule_prefill_gb300 as gd
    wl = gi.custom(seed=507, seqlens=[640, 3, 129], H=4, d_k=128, d_v=128, dtype="bf16",
                   gate=gate, s0="normal")
    a = gi.gen_full(wl, raw=True)
    d = dev_inputs(a, "bf16")
    q, k, al, _ = mapped(a)
    ref_o, ref_s = oracle.gated_linear(q, k, a["v"], al, S0=a["S0"], cu_seqlens=a["cu_seqlens"])
    for path in ("default", "one_cta", "simt"):
        out, sf = gd.gdr_gated_linear_attn(d["q"], d["k"], d["v"], d["alpha"], S0=d["S0"],
                                           cu_seqlens=d["cu_seqlens"],
                                           force_simt=(path == "simt"),
                                           no_cluster=(path == "one_cta"), prologue=True)
        torch.cuda.synchronize()
        check("gla %s %s" % (gate, path), out, sf, ref_o, ref_s, "bf16")


@pytest.mark.parametrize("dtype,d,gate", [("bf16", 128, "channel"), ("bf16", 128, "scalar"),
                                          ("f32", 64, "channel")])
def test_prologue_decode(dtype, d, gate):
    import gated_delta_rule_prefill_gb300 as gd
    wl = gi.Workload("dec", 508, 3, d, d, dtype, gate, np.array([1] * 40), "zeros")
    S = gi.random_state(509, 40, 3, d, d)
    step = gi.gen_decode_step(wl, 0, raw=True)
    st = torch.from_numpy(S).cuda()
    out = gd.gdr_decode_step(to_dev(step["q"], dtype), to_dev(step["k"], dtype),
                             to_dev(step["v"], dtype), to_dev(step["alpha"], "f32"),
                             to_dev(step["beta"], "f32"), st, prologue=True)
    torch.cuda.synchronize()
    q, k, al, be = oracle.layer_prologue(step["q"], step["k"], step["alpha"], step["beta"])
    ro, rs = oracle.decode_step(q, k, step["v"], al, be, S)
    check("decode %s d%d %s" % (dtype, d, gate), out, st, ro, rs, dtype)


def test_prologue_host_pipeline():
    import gated_delta_rule_prefill_gb300 as gd
    wl = gi.custom(seed=510, seqlens=[900, 5, 300], H=2, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    a = gi.gen_full(wl, raw=True)
    from tests.test_gpu_host import host_inputs
    h = host_inputs(a, "bf16")
    out, sf = gd.gdr_prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"], S0=h["S0"],
                                  cu_seqlens=h["cu_seqlens"], piece_tokens=512, prologue=True)
    torch.cuda.synchronize()
    q, k, al, be = mapped(a)
    ref_o, ref_s = oracle.gated_delta(q, k, a["v"], al, be, S0=a["S0"],
                                      cu_seqlens=a["cu_seqlens"])
    eo = rel_rows(out.float().numpy(), ref_o)
    es = rel_states(sf.numpy(), ref_s)
    print("host pipeline: output err %.3g, state err %.3g" % (eo, es))
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


def _close(got, ref, rtol, atol=1e-30):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= rtol * np.abs(ref) + atol), float(np.max(err / (np.abs(ref) + atol)))


@pytest.mark.parametrize("dtype,d,gate", [("bf16", 128, "channel"), ("f32", 64, "scalar"),
                                          ("bf16", 64, "channel"), ("f32", 128, "channel")])
def test_layer_prologue_pass(dtype, d, gate):
    """gdr_layer_prologue against the oracle's maps: q, k rows within one rounding to the dtype
    (row-relative 2^-8 for bf16, 1e-6 for fp32), alpha and beta elementwise within 1e-5; edge
    rows (all zero, all -30) and saturated gates included; a second call in place agrees."""
    import gated_delta_rule_prefill_gb300 as gd
    wl = gi.custom(seed=511, seqlens=[333, 3], H=3, d_k=d, d_v=d, dtype=dtype, gate=gate,
                   s0="zeros")
    a = gi.gen_full(wl, raw=True)
    a["q"][4] = 0.0
    a["k"][7] = -30.0
    a["alpha"][9] = -100.0
    a["beta"][10] = 100.0
    d_ = dev_inputs(a, dtype)
    q, k, al, be = gd.gdr_layer_prologue(d_["q"], d_["k"], d_["alpha"], d_["beta"])
    torch.cuda.synchronize()
    rq, rk, ral, rbe = mapped(a)
    tol = 2.0 ** -8 if dtype == "bf16" else 1e-6
    assert rel_rows(host(q), rq) <= tol and rel_rows(host(k), rk) <= tol
    _close(host(al), ral, 1e-5)
    _close(host(be), rbe, 1e-5)
    # in place: outputs are the inputs
    gd.gdr_layer_prologue(d_["q"], d_["k"], d_["alpha"], d_["beta"], q=d_["q"], k=d_["k"],
                          alpha=d_["alpha"], beta=d_["beta"])
    torch.cuda.synchronize()
    for x, y in ((d_["q"], q), (d_["k"], k), (d_["alpha"], al), (d_["beta"], be)):
        assert torch.equal(x, y)


def test_layer_prologue_then_prefill_matches_fused():
    """The unfused composition (gdr_layer_prologue, then gdr_prefill on its outputs) and the
    fused prefill both meet the oracle; they agree closely with each other."""
    import gated_delta_rule_prefill_gb300 as gd
    wl = gi.custom(seed=512, seqlens=[640, 65], H=4, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    a = gi.gen_full(wl, raw=True)
    d = dev_inputs(a, "bf16")
    q, k, al, be = gd.gdr_layer_prologue(d["q"], d["k"], d["alpha"], d["beta"])
    o1, s1 = gd.gdr_prefill(q, k, d["v"], al, be, S0=d["S0"], cu_seqlens=d["cu_seqlens"])
    o2, s2 = gd.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                            cu_seqlens=d["cu_seqlens"], prologue=True)
    torch.cuda.synchronize()
    rq, rk, ral, rbe = mapped(a)
    ref_o, ref_s = oracle.gated_delta(rq, rk, a["v"], ral, rbe, S0=a["S0"],
                                      cu_seqlens=a["cu_seqlens"])
    check("unfused", o1, s1, ref_o, ref_s, "bf16")
    check("fused", o2, s2, ref_o, ref_s, "bf16")
    assert rel_rows(host(o1), host(o2).astype(np.float64)) <= 2e-2
