"""Chunk-parallel form of the gated delta rule in numpy fp64.  TEST INFRASTRUCTURE.

This is the derivation check for the chunk algebra the GPU kernels implement: the same
recurrence the oracle runs token by token, regrouped into chunks of C tokens.  Tests compare it
against the token loop (gated_delta / linear_attn in this package) for many C: chunking is a
cost dial, not a change of result (engineermaxxing "From GPT-2 to Kimi K3: one memory, seven
eviction policies" §04b and §04f, whose assertion pattern these tests follow).

Per chunk of n tokens (local index r = 0..n-1) entering with state S0 (d_k x d_v):
  D[r, j]  = prod_{j < m <= r} a_m          (per key channel; the survival of a write made at
                                              token j when read at token r, §05d of the same page)
  Gam[r]   = prod_{m <= r} a_m               (fade of the entering state up to token r)
  A[r, j]  = beta_r * sum_c k_r[c] k_j[c] D[r, j][c]   for j < r    (in-chunk coupling, §04e)
  M[r, j]  =          sum_c q_r[c] k_j[c] D[r, j][c]   for j <= r   (in-chunk read-out)
  T        = (I + A)^-1                      (unit lower triangular: forward substitution)
  W        = T diag(beta) (K * Gam)          U_tilde = T diag(beta) V
  U        = U_tilde - W S0                  (the chunk's corrections, all at once)
  O        = (Q * Gam) S0 + M U
  S        = Diag(Gam[n-1]) S0 + (K * D[n-1, :])^T U
With alpha = 1 this is the runnable per-chunk listing of §04f ((I + tril(diag(beta) K K^T, -1)) U
= diag(beta)(V - K S0); O = Q S0 + tril(Q K^T) U; S += K^T U) and heqinghuang "gpt2-to-kimi" §10;
the decay products are the running products of alpha folded through the same solve (§11 there).

Plain linear attention per chunk (same pages, §04b / §10): O = Q S0 + tril(Q K^T) V; S += K^T V.
The decay products here are formed by direct multiplication (no logarithms), so alpha = 0 is
exact.
"""
from __future__ import annotations

import numpy as np


def _pair_decay(a: np.ndarray) -> np.ndarray:
    """D[r, j, c] = prod_{j < m <= r} a[m, c] for j <= r (zero above the diagonal)."""
    n, dk = a.shape
    D = np.zeros((n, n, dk))
    for j in range(n):
        p = np.ones(dk)
        D[j, j] = p
        for r in range(j + 1, n):
            p = p * a[r]
            D[r, j] = p
    return D


def chunk_step(q, k, v, a, b, S):
    """One chunk: q, k [n,d_k]; v [n,d_v]; a [n,d_k] gates; b [n] write strengths;
    S [d_k,d_v] entering state.  Returns (O [n,d_v], S_new, U [n,d_v])."""
    n, dk = k.shape
    D = _pair_decay(a)
    Gam = np.cumprod(a, axis=0)
    A = np.einsum("rc,jc,rjc->rj", k, k, D)
    A = np.tril(A, -1) * b[:, None]
    M = np.tril(np.einsum("rc,jc,rjc->rj", q, k, D))
    T = np.linalg.inv(np.eye(n) + A)
    W = T @ (b[:, None] * (k * Gam))
    U_tilde = T @ (b[:, None] * v)
    U = U_tilde - W @ S
    O = (q * Gam) @ S + M @ U
    K_hat = k * D[n - 1]
    S_new = Gam[n - 1][:, None] * S + K_hat.T @ U
    return O, S_new, U


def gated_delta_seq(q, k, v, alpha, beta, S0, C):
    """One (sequence, head): q,k [L,d_k], v [L,d_v], alpha [L,d_k] or [L], beta [L],
    S0 [d_k,d_v].  Returns (O [L,d_v], S_final, list of per-chunk U)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    L, dk = k.shape
    a = np.asarray(alpha, dtype=np.float64)
    if a.ndim == 1:
        a = np.repeat(a[:, None], dk, axis=1)
    b = np.asarray(beta, dtype=np.float64)
    S = np.array(S0, dtype=np.float64)
    O = np.zeros((L, v.shape[1]))
    Us = []
    for s in range(0, L, C):
        e = min(s + C, L)
        O[s:e], S, U = chunk_step(q[s:e], k[s:e], v[s:e], a[s:e], b[s:e], S)
        Us.append(U)
    return O, S, Us


def linear_seq(q, k, v, S0, C):
    """Chunked plain linear attention for one (sequence, head)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    L = k.shape[0]
    S = np.array(S0, dtype=np.float64)
    O = np.zeros((L, v.shape[1]))
    for s in range(0, L, C):
        e = min(s + C, L)
        Q, K, V = q[s:e], k[s:e], v[s:e]
        O[s:e] = Q @ S + np.tril(Q @ K.T) @ V
        S = S + K.T @ V
    return O, S


def run_packed(q, k, v, alpha, beta, S0, cu_seqlens, C, linear=False):
    """Token-major packed inputs ([T,H,d]); returns (out [T,H,d_v], S_final [N,H,d_k,d_v])."""
    T, H, dk = q.shape
    dv = v.shape[2]
    N = len(cu_seqlens) - 1
    out = np.zeros((T, H, dv))
    Sf = np.zeros((N, H, dk, dv))
    for n in range(N):
        t0, t1 = int(cu_seqlens[n]), int(cu_seqlens[n + 1])
        for h in range(H):
            s0 = np.zeros((dk, dv)) if S0 is None else S0[n, h]
            if linear:
                o, s = linear_seq(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], s0, C)
            else:
                o, s, _ = gated_delta_seq(q[t0:t1, h], k[t0:t1, h], v[t0:t1, h],
                                          alpha[t0:t1, h], beta[t0:t1, h], s0, C)
            out[t0:t1, h] = o
            Sf[n, h] = s
    return out, Sf
