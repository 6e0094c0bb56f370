"""GPU parity of gdr_prefill_host: the prefill on host arrays, pipelined over pieces of the token
axis (copies in, kernels, copies out on three streams, states handed over in place between
pieces).  Each case is checked against the oracle and against gdr_prefill on device copies of
the same inputs; the piece sizes put cuts inside sequences, on sequence boundaries and next to
empty and one-token sequences."""
import numpy as np
import pytest
import torch

import gdr_inputs as gi
import oracle
from tests.parity import TOL, dev_inputs, err_rows, err_states, host, rel_rows, rel_states

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def host_inputs(a, dtype, pinned=True):
    def t(x, dt):
        if dt == "bf16":
            y = torch.from_numpy(gi.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
        else:
            y = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
        return y.pin_memory() if pinned else y.clone()
    d = dict(q=t(a["q"], dtype), k=t(a["k"], dtype), v=t(a["v"], dtype),
             alpha=t(a["alpha"], "f32"), beta=t(a["beta"], "f32"), S0=t(a["S0"], "f32"))
    d["cu_seqlens"] = torch.from_numpy(a["cu_seqlens"].astype(np.int32))
    return d


def run_case(a, dtype, piece, pinned=True, with_s0=True, with_final=True):
    import gated_delta_rule_prefill_gb300 as g
    h = host_inputs(a, dtype, pinned)
    out, sf = g.gdr_prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"],
                                 S0=h["S0"] if with_s0 else None, cu_seqlens=h["cu_seqlens"],
                                 piece_tokens=piece, want_final=with_final)
    torch.cuda.synchronize()
    s0 = a["S0"] if with_s0 else None
    ref = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=s0,
                             cu_seqlens=a["cu_seqlens"])
    eo = err_rows(out.float().numpy(), ref[0], TOL[dtype])
    assert eo <= TOL[dtype], eo
    if with_final:
        es = err_states(sf.numpy(), ref[1], TOL[dtype])
        assert es <= TOL[dtype], es
    # the same prefill on device copies (one call): identical chunking, so the results agree
    d = dev_inputs(a, dtype)
    o2, s2 = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"],
                           S0=d["S0"] if with_s0 else None, cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert rel_rows(out.float().numpy(), host(o2)) <= 1e-3
    if with_final:
        assert rel_states(sf.numpy(), host(s2)) <= 1e-3
    return eo


def test_host_kda_single_sequence_pieces():
    wl = gi.custom(seed=201, seqlens=[3000], H=4, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    run_case(gi.gen_full(wl), "bf16", piece=640)


def test_host_varlen_scalar_cuts_everywhere():
    wl = gi.custom(seed=202, seqlens=[100, 700, 0, 1500, 64, 1], H=2, d_k=128, d_v=128,
                   dtype="bf16", gate="scalar", s0="normal")
    run_case(gi.gen_full(wl), "bf16", piece=256)


def test_host_one_piece_and_no_states():
    wl = gi.custom(seed=203, seqlens=[500, 260], H=3, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    run_case(gi.gen_full(wl), "bf16", piece=0, with_s0=False, with_final=False)


def test_host_fp32_d64_pageable():
    wl = gi.custom(seed=204, seqlens=[300, 200], H=2, d_k=64, d_v=64, dtype="f32",
                   gate="channel", s0="normal")
    run_case(gi.gen_full(wl), "f32", piece=128, pinned=False)


def test_host_two_calls_share_the_streams():
    """Back-to-back calls on one stream (the internal copy streams and events are reused)."""
    import gated_delta_rule_prefill_gb300 as g
    wl = gi.custom(seed=205, seqlens=[900, 300], H=2, d_k=128, d_v=128, dtype="bf16",
                   gate="channel", s0="normal")
    a = gi.gen_full(wl)
    h = host_inputs(a, "bf16")
    first = g.gdr_prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"], S0=h["S0"],
                               cu_seqlens=h["cu_seqlens"], piece_tokens=256)
    second = g.gdr_prefill_host(h["q"], h["k"], h["v"], h["alpha"], h["beta"], S0=h["S0"],
                                cu_seqlens=h["cu_seqlens"], piece_tokens=256)
    torch.cuda.synchronize()
    assert torch.equal(first[0], second[0]) and torch.equal(first[1], second[1])
