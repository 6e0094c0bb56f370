"""gdr_prefill_noalloc: the prefill for callers that cannot provide a workspace.

Such callers have their device memory fully budgeted (a host framework's allocator or a static
memory plan), so they can neither pass a scratch buffer nor call cudaMalloc.  The entry point
keeps its scratch in a fixed device array inside the library.  These tests call it through the
C ABI and check it against gdr_prefill (the entry point with a caller workspace) on two calls in
a row, with different sequence counts so that the second call starts from the first call's
leftover scratch contents.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdr_inputs as gi
from tests.parity import TOL, dev_inputs, host, rel_rows, rel_states


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_rejects_too_many_sequences():
    """More sequences than the fixed scratch holds: a clear error before any GPU work."""
    from gated_delta_rule_prefill_gb300 import _abi, build, make_shape
    build.build_library()
    lib = _abi.load()
    sh = make_shape(_abi.GDR_NOALLOC_MAX_SEQS + 1, 1, 100, 128, 128, _abi.GDR_BF16)
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.gdr_prefill_noalloc(ctypes.byref(sh), fake, fake, fake, fake, fake, None, fake,
                                 ctypes.c_void_p(1 << 21), None, None)
    assert rc == _abi.GDR_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_prefill_matches_workspace_prefill():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_prefill_gb300 as g
    from gated_delta_rule_prefill_gb300 import _abi
    lib = _abi.load()
    cases = [gi.custom(seed=81, seqlens=[300, 0, 77, 129], H=4, d_k=128, d_v=128, dtype="bf16",
                       s0="normal"),
             gi.custom(seed=82, seqlens=[65, 190], H=3, d_k=128, d_v=128, dtype="bf16",
                       gate="scalar", s0="normal")]
    for call, wl in enumerate(cases):
        a = gi.gen_full(wl)
        d = dev_inputs(a, "bf16")
        ref_out, ref_S = g.gdr_prefill(d["q"], d["k"], d["v"], d["alpha"], d["beta"], S0=d["S0"],
                                       cu_seqlens=d["cu_seqlens"])
        out = torch.full_like(ref_out, float("nan"))
        S = torch.full_like(ref_S, float("nan"))
        T, H, dk = d["q"].shape
        gate = _abi.GDR_GATE_CHANNEL if d["alpha"].dim() == 3 else _abi.GDR_GATE_SCALAR
        sh = g.make_shape(wl.n_seqs, H, T, dk, dk, _abi.GDR_BF16, gate)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.gdr_prefill_noalloc(ctypes.byref(sh), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]),
                                     _ptr(d["alpha"]), _ptr(d["beta"]), _ptr(d["S0"]),
                                     _ptr(d["cu_seqlens"]), _ptr(out), _ptr(S), stream)
        assert rc == 0, _abi.status_string(rc)
        torch.cuda.synchronize()
        eo = rel_rows(host(out), host(ref_out))
        es = rel_states(host(S), host(ref_S))
        assert eo <= TOL["bf16"] and es <= TOL["bf16"], (call, eo, es)
        assert np.isfinite(host(out)).all()
