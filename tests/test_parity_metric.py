"""The element-wise parity metric's floor (tests/parity.py, ELEM_FLOOR) is a property of fp32
arithmetic, not of the kernels: the recurrence itself evaluated in fp32, token by token in the
stated order (fade, read the faded state, correct, read out), already misses a 1e-4 element-wise
bound at a floor of 1e-3 x RMS on the fp32 workload (256 tokens, d = 64), and meets it with a
10x margin at ELEM_FLOOR x RMS."""
import numpy as np

import gdr_inputs as gi
import oracle
from tests.parity import ELEM_FLOOR, TOL, rel_elem, rel_rows


def _fp32_token_loop(q, k, v, alpha, beta):
    q, k, v, alpha, beta = (np.asarray(x, np.float32) for x in (q, k, v, alpha, beta))
    T, H, dk = q.shape
    S = np.zeros((H, dk, v.shape[-1]), np.float32)
    o = np.zeros((T, H, v.shape[-1]), np.float32)
    for t in range(T):
        for h in range(H):
            Sa = S[h] * alpha[t, h][:, None]
            vh = Sa.T @ k[t, h]
            S[h] = Sa + beta[t, h] * np.outer(k[t, h], v[t, h] - vh)
            o[t, h] = S[h].T @ q[t, h]
    return o, S


def test_fp32_resolution_sets_the_floor():
    wl = gi.workload("kda_t256_d64_f32")
    a = gi.gen_full(wl)
    ro, rs = oracle.gated_delta(a["q"], a["k"], a["v"], a["alpha"], a["beta"], S0=a["S0"],
                                cu_seqlens=a["cu_seqlens"])
    o32, s32 = _fp32_token_loop(a["q"], a["k"], a["v"], a["alpha"], a["beta"])
    # row-normwise the fp32 loop is far inside the bound ...
    assert rel_rows(o32, ro) < 1e-5
    # ... element-wise it misses 1e-4 at the 1e-3 x RMS floor, and meets it at ELEM_FLOOR
    assert rel_elem(o32, ro, 1e-3) > TOL["f32"]
    assert rel_elem(o32, ro) <= 0.1 * TOL["f32"]
    assert rel_elem(s32[None], rs) <= 0.1 * TOL["f32"]
    assert ELEM_FLOOR == 0.1
