"""GPU parity of gdr_normalized_linear_attn (normalised phi-linear attention, phi = elu + 1,
normaliser z) against the oracle's token-by-token statement: outputs, final states and final
normalisers, with and without entering (S0, z0), eps = 0 and eps > 0, ragged and empty
sequences, on the tensor-core path (bf16, d = 128) and the fp32 path (fp32 inputs, d = 64 and
128, and bf16 forced onto it)."""
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


def run(a, dtype, eps=0.0, with_state=True, force_simt=False, z0_scale=1.0):
    import gated_delta_rule_prefill_gb300 as g
    N, H, dk = a["S0"].shape[:3]
    z0 = z0_scale * np.abs(np.random.default_rng(601).normal(size=(N, H, dk))).astype(np.float32)
    d = dev_inputs(a, dtype)
    S0 = d["S0"] if with_state else None
    z0d = torch.from_numpy(z0).cuda() if with_state else None
    out, sf, zf = g.gdr_normalized_linear_attn(d["q"], d["k"], d["v"], eps=eps, S0=S0, z0=z0d,
                                               cu_seqlens=d["cu_seqlens"],
                                               force_simt=force_simt)
    torch.cuda.synchronize()
    ro, rs, rz = oracle.normalized_linear(a["q"], a["k"], a["v"],
                                          a["S0"] if with_state else None,
                                          z0 if with_state else None, a["cu_seqlens"], eps)
    eo, es = err_rows(host(out), ro, TOL[dtype]), err_states(host(sf), rs, TOL[dtype])
    ez = err_rows(host(zf), rz, TOL[dtype])
    print("%s eps %g simt %s: out %.3g state %.3g z %.3g" % (dtype, eps, force_simt, eo, es, ez))
    assert eo <= TOL[dtype] and es <= TOL[dtype] and ez <= TOL[dtype], (eo, es, ez)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("eps", [0.0, 1e-3])
def test_normlinear_fp32(d, eps):
    wl = gi.custom(seed=602, seqlens=[200, 1, 64, 65, 0, 130], H=2, d_k=d, d_v=d, dtype="f32",
                   s0="normal")
    run(gi.gen_full(wl, raw=True), "f32", eps)


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_normlinear_bf16(simt, with_state):
    wl = gi.custom(seed=603, seqlens=[700, 1, 64, 65, 0, 300], H=4, d_k=128, d_v=128,
                   dtype="bf16", s0="normal")
    run(gi.gen_full(wl, raw=True), "bf16", 0.0, with_state, simt)


def test_normlinear_long_bf16():
    """Long sequences (the normaliser grows to thousands), few heads (the tensor-core path splits
    each sequence into runs with recomputed entering states)."""
    wl = gi.custom(seed=604, seqlens=[6000, 2500], H=2, d_k=128, d_v=128, dtype="bf16",
                   s0="normal")
    run(gi.gen_full(wl, raw=True), "bf16", 1e-6)


def test_normlinear_edge_rows():
    """Queries of -20 everywhere (phi(q) ~ 2e-9: numerator and denominator tiny, their ratio
    still the weighted average), keys of -20 (their tokens add almost nothing), large positive
    entries (phi = x + 1)."""
    wl = gi.custom(seed=605, seqlens=[150, 90], H=2, d_k=128, d_v=128, dtype="bf16",
                   s0="normal")
    a = gi.gen_full(wl, raw=True)
    a["q"][3] = -20.0
    a["k"][7] = -20.0
    a["q"][11, :, :8] = 30.0
    a["k"][12, :, :8] = 30.0
    for simt in (False, True):
        run(a, "bf16", 0.0, True, simt)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_normlinear_decode_step(dtype, d):
    """gdr_normalized_linear_decode_step from a given (S, z), twice in a row, against the oracle
    stepping the same tokens (one-token sequences)."""
    import gated_delta_rule_prefill_gb300 as g
    N, H = 48, 3
    wl = gi.Workload("dec", 606, H, d, d, dtype, "channel", np.array([1] * N), "zeros")
    S = gi.random_state(607, N, H, d, d)
    z = np.abs(np.random.default_rng(608).normal(size=(N, H, d))).astype(np.float32) * 5
    Sd, zd = torch.from_numpy(S).cuda(), torch.from_numpy(z).cuda()
    cu = np.arange(N + 1)
    for step in range(2):
        a = gi.gen_decode_step(wl, step, raw=True)
        d_ = {kk: to_dev(a[kk], dtype) for kk in ("q", "k", "v")}
        out = g.gdr_normalized_linear_decode_step(d_["q"], d_["k"], d_["v"], Sd, zd, eps=1e-6)
        torch.cuda.synchronize()
        ro, rs, rz = oracle.normalized_linear(a["q"], a["k"], a["v"], S, z, cu, 1e-6)
        eo, es = err_rows(host(out), ro, TOL[dtype]), err_states(host(Sd), rs, TOL[dtype])
        ez = err_rows(host(zd), rz, TOL[dtype])
        print("norm decode %s step %d: out %.3g state %.3g z %.3g" % (dtype, step, eo, es, ez))
        assert eo <= TOL[dtype] and es <= TOL[dtype] and ez <= TOL[dtype], (eo, es, ez)
        S, z = rs, rz
