"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test ties the oracle to something other than itself: a value printed on a page (fixtures
under tests/golden/, each with its source), a closed form, a textbook routine it reduces to, an
invariant stated on a page, or brute force.  test_oracle_mutations.py then plants plausible
mistakes in a copy of the oracle and checks that these pins catch them.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def one_head(*arrs):
    """[L, d] per-head arrays -> token-major [L, 1, d] (or [L] -> [L, 1])."""
    return [np.asarray(a, dtype=np.float64)[:, None] for a in arrs]


def rand_inputs(rng, T, H, dk, dv, channel=True, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    alpha = rng.uniform(0.3, 1.0, (T, H, dk) if channel else (T, H))
    beta = rng.uniform(0.0, 1.0, (T, H))
    return q, k, v, alpha, beta


# ------------------------------------------------------------------------------------------
# values printed on the pages
# ------------------------------------------------------------------------------------------
def test_interference_read_em02e():
    g = golden("em_02e_interference_read.json")
    k = np.array(g["k"], float)
    v = np.array(g["v"], float)
    q = np.stack([g["q_read"], g["q_read"]]).astype(float)
    out, S = oracle.linear_attn(*one_head(q, k, v))
    np.testing.assert_allclose(out[1, 0], g["expected_read"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S[0, 0, 1], g["expected_row1"], rtol=0, atol=1e-12)
    # the error is exactly the interference law's crosstalk (k_cat . k_dog) v_rex
    np.testing.assert_allclose(out[1, 0] - v[0], (k[0] @ k[1]) * v[1], atol=1e-12)


def test_delta_overwrite_em03d():
    g = golden("em_03d_delta_overwrite.json")
    S0 = np.zeros((1, 1, 4, 4))
    S0[0, 0, 0] = g["row0_before"]
    S0[0, 0, 2] = [0.0, 0.0, 3.0, 1.0]  # another fact on a row the key does not touch
    S0[0, 0, 3] = [0.5, -1.0, 0.0, 2.0]
    k = np.array([g["k"]], float)
    v = np.array([g["v"]], float)
    a = np.ones((1, 4))
    b = np.array([g["beta"]])
    out, S = oracle.gated_delta(*one_head(k, k, v, a, b), S0=S0)
    np.testing.assert_allclose(S[0, 0, 0], g["expected_row0_after"], atol=1e-12)
    np.testing.assert_allclose(S[0, 0, 0] - S0[0, 0, 0], g["expected_u"], atol=1e-12)
    np.testing.assert_allclose(S[0, 0, 1:], S0[0, 0, 1:], atol=0)
    np.testing.assert_allclose(out[0, 0], g["v"], atol=1e-12)  # read-back is exact


def test_two_token_chunk_em04e():
    g = golden("em_04e_two_token_chunk.json")
    k = np.array(g["k"], float)
    v = np.array(g["v"], float)
    b = np.array(g["beta"], float)
    a = np.ones((2, 4))
    for qrow, key in ((k[1], "derived_read_k2"), (k[0], "derived_read_k1")):
        q = np.stack([k[0], qrow])
        out, S = oracle.gated_delta(*one_head(q, k, v, a, b))
        np.testing.assert_allclose(out[1, 0], g[key], atol=1e-12)
    # S2 = k1 u1^T + k2 u2^T with the printed corrections
    expect = np.outer(k[0], g["expected_u1"]) + np.outer(k[1], g["expected_u2"])
    np.testing.assert_allclose(S[0, 0], expect, atol=1e-12)
    # and the chunked (triangular solve) form reproduces the printed u2
    _, _, Us = chunked.gated_delta_seq(k, k, v, a, b, np.zeros((4, 4)), C=2)
    np.testing.assert_allclose(Us[0][0], g["expected_u1"], atol=1e-12)
    np.testing.assert_allclose(Us[0][1], g["expected_u2"], atol=1e-12)


@pytest.mark.parametrize("channel", [True, False])
def test_decay_survival_em05d(channel):
    g = golden("em_05d_decay_survival.json")
    d = 4
    L = g["write_step"] + len(g["gates_after_write"])
    rng = np.random.default_rng(0)
    k = np.zeros((L, d))
    q = np.zeros((L, d))
    v = rng.standard_normal((L, d))
    k[g["write_step"] - 1, 0] = 1.0
    q[-1, 0] = 1.0
    b = np.zeros(L)
    b[g["write_step"] - 1] = 1.0
    gates = np.ones(L)
    gates[g["write_step"]:] = g["gates_after_write"]
    if channel:
        a = np.ones((L, d))
        a[:, 0] = gates  # only channel 0 carries the fact
        a[:, 1:] = 0.3
    else:
        a = gates
    out, _ = oracle.gated_delta(*one_head(q, k, v, a, b))
    np.testing.assert_allclose(out[-1, 0], g["expected_strength"] * v[g["write_step"] - 1],
                               atol=1e-12)


def test_hand_2x2_steps():
    g = golden("hand_2x2_steps.json")
    for c in g["cases"]:
        S0 = np.array(c["S0"], float)[None, None]
        k = np.array([c["k"]], float)
        q = np.array([c["q"]], float)
        v = np.array([c["v"]], float)
        a = np.array([c["alpha"]], float) if np.ndim(c["alpha"]) else np.array([c["alpha"]])
        b = np.array([c["beta"]], float)
        out, S = oracle.gated_delta(*one_head(q, k, v, a, b), S0=S0)
        np.testing.assert_allclose(S[0, 0], c["expected_S1"], atol=1e-12)
        np.testing.assert_allclose(out[0, 0], c["expected_o"], atol=1e-12)
        # the read of the faded state that the correction was computed from
        np.testing.assert_allclose(S[0, 0].T @ k[0], (1 - c["beta"]) * np.array(c["v_hat"])
                                   + c["beta"] * np.array(c["v"]), atol=1e-12)


# ------------------------------------------------------------------------------------------
# closed forms and textbook reductions
# ------------------------------------------------------------------------------------------
def test_linear_attention_is_masked_qk_v():
    """alpha = 1 and no erase: O = tril(Q K^T) V (+ Q S0) per sequence, by brute force."""
    rng = np.random.default_rng(1)
    lens = [1, 17, 0, 40]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv = cu[-1], 3, 8, 5
    q, k, v, _, _ = rand_inputs(rng, T, H, dk, dv, unit_k=False)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    out, Sf = oracle.linear_attn(q, k, v, S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        for h in range(H):
            Q, K, V = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h]
            ref = np.tril(Q @ K.T) @ V + Q @ S0[n, h]
            np.testing.assert_allclose(out[t0:t1, h], ref, atol=1e-10)
            np.testing.assert_allclose(Sf[n, h], S0[n, h] + K.T @ V, atol=1e-10)


def test_gdn_matrix_form():
    """Scalar gate: S_t = alpha (I - beta k k^T) S_{t-1} + beta k v^T (Gated DeltaNet form)."""
    rng = np.random.default_rng(2)
    T, dk, dv = 9, 6, 4
    q, k, v, a, b = rand_inputs(rng, T, 1, dk, dv, channel=False)
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, Sf = oracle.gated_delta(q, k, v, a, b, S0=S0)
    S = S0[0, 0].copy()
    for t in range(T):
        kt = k[t, 0]
        S = a[t, 0] * (np.eye(dk) - b[t, 0] * np.outer(kt, kt)) @ S + b[t, 0] * np.outer(kt, v[t, 0])
        np.testing.assert_allclose(out[t, 0], S.T @ q[t, 0], atol=1e-12)
    np.testing.assert_allclose(Sf[0, 0], S, atol=1e-12)


def test_scalar_gate_equals_uniform_channel_gate():
    rng = np.random.default_rng(3)
    q, k, v, a, b = rand_inputs(rng, 20, 2, 8, 8, channel=False)
    S0 = rng.standard_normal((1, 2, 8, 8))
    o1, s1 = oracle.gated_delta(q, k, v, a, b, S0=S0)
    o2, s2 = oracle.gated_delta(q, k, v, np.repeat(a[:, :, None], 8, axis=2), b, S0=S0)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(s1, s2, atol=1e-13)


def test_alpha_zero_resets_memory():
    """alpha = 0: amnesia, the new state is exactly beta k v^T whatever came before."""
    rng = np.random.default_rng(4)
    q, k, v, a, b = rand_inputs(rng, 1, 1, 8, 6)
    S0 = rng.standard_normal((1, 1, 8, 6))
    _, Sf = oracle.gated_delta(q, k, v, np.zeros_like(a), b, S0=S0)
    np.testing.assert_allclose(Sf[0, 0], b[0, 0] * np.outer(k[0, 0], v[0, 0]), atol=1e-14)


def test_beta_zero_is_pure_decay():
    """beta = 0: no write at all; S_t = Diag(prod alpha) S0 and o_t reads that state."""
    rng = np.random.default_rng(5)
    T, dk, dv = 12, 8, 5
    q, k, v, a, _ = rand_inputs(rng, T, 1, dk, dv)
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, Sf = oracle.gated_delta(q, k, v, a, np.zeros((T, 1)), S0=S0)
    P = np.cumprod(a[:, 0], axis=0)
    for t in range(T):
        np.testing.assert_allclose(out[t, 0], (P[t][:, None] * S0[0, 0]).T @ q[t, 0], atol=1e-12)
    np.testing.assert_allclose(Sf[0, 0], P[-1][:, None] * S0[0, 0], atol=1e-12)


def test_idle_gates_coast():
    """alpha = 1, beta = 0: neither fade nor write, so the state carries over unchanged."""
    rng = np.random.default_rng(6)
    q, k, v, a, _ = rand_inputs(rng, 7, 2, 4, 4)
    S0 = rng.standard_normal((1, 2, 4, 4))
    out, Sf = oracle.gated_delta(q, k, v, np.ones_like(a), np.zeros((7, 2)), S0=S0)
    np.testing.assert_array_equal(Sf, S0)
    np.testing.assert_allclose(out, np.einsum("thc,hcd->thd", q, S0[0]), atol=1e-12)


def test_orthonormal_keys_store_last_value():
    """Keys cycling through e_0..e_{d-1} with beta = alpha = 1: row c = last value at key c."""
    rng = np.random.default_rng(7)
    d, T = 6, 20
    k = np.zeros((T, 1, d))
    for t in range(T):
        k[t, 0, t % d] = 1.0
    v = rng.standard_normal((T, 1, d))
    q = rng.standard_normal((T, 1, d))
    S0 = rng.standard_normal((1, 1, d, d))
    _, Sf = oracle.gated_delta(q, k, v, np.ones((T, 1, d)), np.ones((T, 1)), S0=S0)
    for c in range(d):
        last = max(t for t in range(T) if t % d == c)
        np.testing.assert_allclose(Sf[0, 0, c], v[last, 0], atol=1e-13)


def test_deltanet_householder_geometry():
    """alpha = 1, unit k: beta = 2 with v = 0 is a reflection (norm kept); beta = 1 with v = 0
    projects the k-direction out (k^T S = 0)."""
    rng = np.random.default_rng(8)
    T, d = 10, 7
    q, k, _, _, _ = rand_inputs(rng, T, 1, d, d)
    S0 = rng.standard_normal((1, 1, d, d))
    zero_v = np.zeros((T, 1, d))
    ones = np.ones((T, 1, d))
    _, Sf = oracle.gated_delta(q, k, zero_v, ones, 2 * np.ones((T, 1)), S0=S0)
    assert abs(np.linalg.norm(Sf) - np.linalg.norm(S0)) < 1e-12
    _, Sf = oracle.gated_delta(q[:1], k[:1], zero_v[:1], ones[:1], np.ones((1, 1)), S0=S0)
    np.testing.assert_allclose(k[0, 0] @ Sf[0, 0], 0, atol=1e-13)


# ------------------------------------------------------------------------------------------
# invariants stated on the pages
# ------------------------------------------------------------------------------------------
def _prefix_states(q, k, v, a, b, S0):
    """State before each token (the oracle's own S_final of each prefix)."""
    T = q.shape[0]
    states = [S0[0, 0]]
    for t in range(1, T):
        _, s = oracle.gated_delta(q[:t], k[:t], v[:t], a[:t], b[:t], S0=S0)
        states.append(s[0, 0])
    return states


def test_read_back_after_write():
    """Unit k: k_t^T S_t = (1 - beta) v_hat + beta v with v_hat the read of the faded state; the
    SGD view: ||S_t^T k - v|| = (1 - beta) ||v_hat - v||.  beta = 1 returns v exactly."""
    rng = np.random.default_rng(9)
    T, dk, dv = 8, 6, 5
    q, k, v, a, b = rand_inputs(rng, T, 1, dk, dv)
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, _ = oracle.gated_delta(k, k, v, a, b, S0=S0)  # read-out with q = k
    for t, S in enumerate(_prefix_states(k, k, v, a, b, S0)):
        vhat = (a[t, 0][:, None] * S).T @ k[t, 0]
        expect = (1 - b[t, 0]) * vhat + b[t, 0] * v[t, 0]
        np.testing.assert_allclose(out[t, 0], expect, atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(out[t, 0] - v[t, 0]),
                                   (1 - b[t, 0]) * np.linalg.norm(vhat - v[t, 0]), atol=1e-12)
    out1, _ = oracle.gated_delta(k, k, v, a, np.ones((T, 1)), S0=S0)
    np.testing.assert_allclose(out1[:, 0], v[:, 0], atol=1e-12)


def test_causality():
    """Changing tokens after t leaves every output up to t unchanged."""
    rng = np.random.default_rng(10)
    q, k, v, a, b = rand_inputs(rng, 30, 2, 8, 8)
    out, _ = oracle.gated_delta(q, k, v, a, b)
    q2, k2, v2, a2, b2 = (x.copy() for x in (q, k, v, a, b))
    t = 13
    for x in (q2, k2, v2, a2, b2):
        x[t + 1:] = rng.uniform(0.1, 0.9, x[t + 1:].shape)
    out2, _ = oracle.gated_delta(q2, k2, v2, a2, b2)
    np.testing.assert_array_equal(out[:t + 1], out2[:t + 1])
    assert not np.allclose(out[t + 1:], out2[t + 1:])


def test_continuation_and_varlen_and_decode():
    """prefill(T1) -> S; prefill(T2, S0=S) == prefill(T1+T2); packed == per-sequence;
    n decode steps == a prefill of n tokens; a (seq, head) subset == the full run."""
    rng = np.random.default_rng(11)
    H, dk, dv = 2, 8, 6
    lens = [23, 5, 0, 31]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, a, b = rand_inputs(rng, cu[-1], H, dk, dv)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    out, Sf = oracle.gated_delta(q, k, v, a, b, S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        o1, s1 = oracle.gated_delta(q[t0:t1], k[t0:t1], v[t0:t1], a[t0:t1], b[t0:t1],
                                    S0=S0[n:n + 1])
        np.testing.assert_array_equal(out[t0:t1], o1)
        np.testing.assert_array_equal(Sf[n], s1[0])
    # continuation of sequence 0 split at token 9
    t0, cut, t1 = cu[0], cu[0] + 9, cu[1]
    oa, sa = oracle.gated_delta(q[t0:cut], k[t0:cut], v[t0:cut], a[t0:cut], b[t0:cut], S0=S0[:1])
    ob, sb = oracle.gated_delta(q[cut:t1], k[cut:t1], v[cut:t1], a[cut:t1], b[cut:t1], S0=sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), out[t0:t1], atol=1e-13)
    np.testing.assert_allclose(sb[0], Sf[0], atol=1e-13)
    # decode steps (sequence 3, all heads, token by token)
    S = S0[3:4]
    for t in range(cu[3], cu[4]):
        o, S = oracle.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], a[t:t + 1], b[t:t + 1], S)
        np.testing.assert_allclose(o[0], out[t], atol=1e-13)
    np.testing.assert_allclose(S[0], Sf[3], atol=1e-13)
    # subset of pairs
    o_sub, s_sub = oracle.gated_delta(q, k, v, a, b, S0=S0, cu_seqlens=cu, pairs=[(3, 1), (0, 0)])
    np.testing.assert_array_equal(o_sub[cu[3]:cu[4], 1], out[cu[3]:cu[4], 1])
    np.testing.assert_array_equal(s_sub[0, 0], Sf[0, 0])
    assert np.all(o_sub[cu[3]:cu[4], 0] == 0)


# ------------------------------------------------------------------------------------------
# the chunk algebra (derivation check), against the token loop
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 2, 3, 16, 64, 200])
@pytest.mark.parametrize("channel", [True, False])
def test_chunked_equals_recurrence(C, channel):
    rng = np.random.default_rng(12 + C)
    lens = [70, 1, 0, 45]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, dk, dv = 2, 8, 6
    q, k, v, a, b = rand_inputs(rng, cu[-1], H, dk, dv, channel=channel)
    a[5] = 0.0  # a full reset inside a chunk
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    ref_o, ref_s = oracle.gated_delta(q, k, v, a, b, S0=S0, cu_seqlens=cu)
    o, s = chunked.run_packed(q, k, v, a, b, S0, cu, C)
    np.testing.assert_allclose(o, ref_o, atol=1e-10, rtol=1e-10)
    np.testing.assert_allclose(s, ref_s, atol=1e-10, rtol=1e-10)
    lo, ls = oracle.linear_attn(q, k, v, S0=S0, cu_seqlens=cu)
    o, s = chunked.run_packed(q, k, v, None, None, S0, cu, C, linear=True)
    np.testing.assert_allclose(o, lo, atol=1e-10, rtol=1e-10)
    np.testing.assert_allclose(s, ls, atol=1e-10, rtol=1e-10)


# ------------------------------------------------------------------------------------------
# gated linear attention (S <- Diag(alpha) S + k v^T): closed forms and brute force
# ------------------------------------------------------------------------------------------
def test_gated_linear_unit_gate_is_masked_qk_v():
    """alpha = 1: gated linear attention is plain linear attention, O = tril(Q K^T) V + Q S0."""
    rng = np.random.default_rng(21)
    lens = [13, 0, 30]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv = cu[-1], 2, 6, 5
    q, k, v, _, _ = rand_inputs(rng, T, H, dk, dv, unit_k=False)
    S0 = rng.standard_normal((len(lens), H, dk, dv))
    out, Sf = oracle.gated_linear(q, k, v, np.ones((T, H, dk)), S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        t0, t1 = cu[n], cu[n + 1]
        for h in range(H):
            Q, K, V = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h]
            np.testing.assert_allclose(out[t0:t1, h], np.tril(Q @ K.T) @ V + Q @ S0[n, h], atol=1e-10)
            np.testing.assert_allclose(Sf[n, h], S0[n, h] + K.T @ V, atol=1e-10)


@pytest.mark.parametrize("channel", [True, False])
def test_gated_linear_survival_sum(channel):
    """Unrolled recurrence: S_t = sum_{s<=t} Diag(prod_{s<i<=t} alpha_i) k_s v_s^T
    + Diag(prod_{i<=t} alpha_i) S0, so o_t = sum_s ((q_t * D_st) . k_s) v_s + (q_t * D_0t)^T S0
    (engineermaxxing §05d's survival products, a write at step s not decayed by alpha_s)."""
    rng = np.random.default_rng(22 + channel)
    T, dk, dv = 11, 5, 3
    q, k, v, alpha, _ = rand_inputs(rng, T, 1, dk, dv, channel=channel, unit_k=False)
    S0 = rng.standard_normal((1, 1, dk, dv))
    out, Sf = oracle.gated_linear(q, k, v, alpha, S0=S0)
    a = alpha[:, 0] if channel else np.repeat(alpha[:, 0:1], dk, axis=1)  # [T, dk]
    for t in range(T):
        D0 = np.prod(a[:t + 1], axis=0)
        ref = (q[t, 0] * D0) @ S0[0, 0]
        for s in range(t + 1):
            D = np.prod(a[s + 1:t + 1], axis=0)  # empty product = 1
            ref = ref + np.dot(q[t, 0] * D, k[s, 0]) * v[s, 0]
        np.testing.assert_allclose(out[t, 0], ref, atol=1e-12)
    D0 = np.prod(a, axis=0)
    Sref = D0[:, None] * S0[0, 0] + sum(np.prod(a[s + 1:], axis=0)[:, None] * np.outer(k[s, 0], v[s, 0])
                                       for s in range(T))
    np.testing.assert_allclose(Sf[0, 0], Sref, atol=1e-12)


def test_gated_linear_zero_gate_resets():
    """alpha_t = 0 forgets everything before t: S_t = k_t v_t^T, o_t = (q_t . k_t) v_t."""
    rng = np.random.default_rng(24)
    T, dk, dv = 6, 4, 3
    q, k, v, alpha, _ = rand_inputs(rng, T, 1, dk, dv, unit_k=False)
    alpha[3] = 0.0
    out, _ = oracle.gated_linear(q, k, v, alpha, S0=rng.standard_normal((1, 1, dk, dv)))
    np.testing.assert_allclose(out[3, 0], np.dot(q[3, 0], k[3, 0]) * v[3, 0], atol=1e-12)


# ------------------------------------------------------------------------------------------
# the output gate o * sigmoid(g): closed forms
# ------------------------------------------------------------------------------------------
def test_output_gate_closed_forms():
    """sigmoid(0) = 1/2; sigmoid(ln 3) = 3/4; sigmoid(x) + sigmoid(-x) = 1; the gate opens fully
    for large g and shuts for very negative g."""
    o = np.array([2.0, -4.0, 8.0, 1.0])
    np.testing.assert_allclose(oracle.output_gate(o, np.zeros(4)), o / 2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.output_gate(o, np.full(4, np.log(3.0))), 0.75 * o, atol=1e-14)
    x = np.linspace(-6, 6, 13)
    one = np.ones_like(x)
    np.testing.assert_allclose(oracle.output_gate(one, x) + oracle.output_gate(one, -x), one,
                               atol=1e-15)
    np.testing.assert_allclose(oracle.output_gate(o, np.full(4, 50.0)), o, rtol=1e-15)
    np.testing.assert_allclose(oracle.output_gate(o, np.full(4, -50.0)), 0 * o, atol=1e-20)


# ------------------------------------------------------------------------------------------
# the layer prologue (raw projections -> q, k, alpha, beta): closed forms
# ------------------------------------------------------------------------------------------
def test_layer_prologue_closed_forms():
    """Unit-length q and k along silu(x) = x / (1 + e^-x); alpha = sigmoid(a) =
    exp(-softplus(-a)); beta = sigmoid(b) with sigmoid(0) = 1/2; silu(0) = 0 rows stay zero."""
    rng = np.random.default_rng(31)
    xq = rng.normal(0, 1.5, (5, 3, 8))
    xk = rng.normal(0, 1.5, (5, 3, 8))
    a = rng.normal(4, 1, (5, 3, 8))
    b = rng.normal(0, 1, (5, 3))
    q, k, al, be = oracle.layer_prologue(xq, xk, a, b)
    for x, y in ((xq, q), (xk, k)):
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-14)
        silu = x / (1.0 + np.exp(-x))
        cos = np.sum(y * silu, axis=-1) / np.linalg.norm(silu, axis=-1)
        np.testing.assert_allclose(cos, 1.0, atol=1e-14)
    np.testing.assert_allclose(al, np.exp(-np.log1p(np.exp(-a))), atol=1e-15)
    np.testing.assert_allclose(oracle.layer_prologue(xq, xk, np.zeros(1), np.zeros(1))[3], 0.5)
    z = oracle.layer_prologue(np.zeros((1, 1, 4)), xk[:1, :1, :4], a[:1], b[:1])[0]
    assert np.all(z == 0.0)


# ------------------------------------------------------------------------------------------
# normalised phi-linear attention: the feature map, and the read as a weighted average
# ------------------------------------------------------------------------------------------
def test_phi_closed_forms():
    """phi = elu + 1: x + 1 above zero, e^x at and below zero; continuous with slope 1 at 0."""
    x = np.array([-50.0, -2.0, -1e-9, 0.0, 1e-9, 0.5, 3.0])
    np.testing.assert_allclose(oracle.phi(x), [np.exp(-50), np.exp(-2), np.exp(-1e-9), 1.0,
                                               1.0 + 1e-9, 1.5, 4.0], rtol=1e-15)
    h = 1e-7
    assert abs((oracle.phi(h) - oracle.phi(-h)) / (2 * h) - 1.0) < 1e-6
    assert np.all(oracle.phi(np.linspace(-700, 50, 1001)) > 0)


def test_normalized_linear_is_a_weighted_average():
    """From zero state with eps = 0 the read is sum_j w_j v_j with w_j = phi(q_t).phi(k_j) /
    sum_i<=t phi(q_t).phi(k_i): computed here pair by pair, not through the running state.  The
    first output is v_1 exactly; every output lies in the convex hull of the values so far."""
    rng = np.random.default_rng(41)
    T, H, dk, dv = 9, 2, 5, 3
    q, k, v = rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dv))
    out, S, z = oracle.normalized_linear(q, k, v)
    pq, pk = oracle.phi(q), oracle.phi(k)
    for h in range(H):
        for t in range(T):
            w = np.array([pq[t, h] @ pk[j, h] for j in range(t + 1)])
            ref = (w / w.sum()) @ v[: t + 1, h]
            np.testing.assert_allclose(out[t, h], ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(out[0, h], v[0, h], rtol=1e-14)
        np.testing.assert_allclose(z[0, h], pk[:, h].sum(0), rtol=1e-14)
        np.testing.assert_allclose(S[0, h], pk[:, h].T @ v[:, h], rtol=1e-13)


def test_normalized_linear_state_handoff_and_eps():
    """Two halves with (S, z) handed over equal one run; eps adds to the denominator only;
    packed sequences are independent."""
    rng = np.random.default_rng(42)
    T, H, dk, dv = 12, 1, 4, 4
    q, k, v = rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dk)), rng.normal(size=(T, H, dv))
    S0 = rng.normal(size=(1, H, dk, dv))
    z0 = np.abs(rng.normal(size=(1, H, dk)))
    full = oracle.normalized_linear(q, k, v, S0, z0)
    a = oracle.normalized_linear(q[:5], k[:5], v[:5], S0, z0)
    b = oracle.normalized_linear(q[5:], k[5:], v[5:], a[1], a[2])
    np.testing.assert_allclose(np.concatenate([a[0], b[0]]), full[0], rtol=1e-12)
    np.testing.assert_allclose(b[1], full[1], rtol=1e-12)
    np.testing.assert_allclose(b[2], full[2], rtol=1e-12)
    e = oracle.normalized_linear(q, k, v, S0, z0, eps=0.25)[0]
    pq = oracle.phi(q)
    num = full[0] * (np.einsum("thd,thd->th", pq, np.cumsum(oracle.phi(k), 0) + z0[0]))[..., None]
    den = np.einsum("thd,thd->th", pq, np.cumsum(oracle.phi(k), 0) + z0[0]) + 0.25
    np.testing.assert_allclose(e, num / den[..., None], rtol=1e-12)
    cu = np.array([0, 5, 12])
    pk = oracle.normalized_linear(q, k, v, cu_seqlens=cu)
    np.testing.assert_allclose(pk[0][5:], oracle.normalized_linear(q[5:], k[5:], v[5:])[0],
                               rtol=1e-12)


def test_prologue_and_phi_match_the_pages_expressions():
    """The pages print the maps as framework expressions (heqinghuang §09: normalize(silu(.)) and
    sigmoid(.); heqinghuang §07 / engineermaxxing §02g: elu(.) + 1).  Evaluated with those
    framework routines (torch, CPU, fp64) they agree with the oracle's own statement."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(77)
    x = rng.normal(0, 3, (6, 2, 16))
    a = rng.normal(3, 2, (6, 2, 16))
    b = rng.normal(0, 2, (6, 2))
    q, k, al, be = oracle.layer_prologue(x, -x, a, b)
    tx = torch.from_numpy(x)
    np.testing.assert_allclose(q, F.normalize(F.silu(tx), dim=-1).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(k, F.normalize(F.silu(-tx), dim=-1).numpy(), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(al, torch.sigmoid(torch.from_numpy(a)).numpy(), rtol=1e-12)
    np.testing.assert_allclose(be, torch.sigmoid(torch.from_numpy(b)).numpy(), rtol=1e-12)
    np.testing.assert_allclose(oracle.phi(x), (F.elu(tx) + 1).numpy(), rtol=1e-12)
