"""The oracle: a plain, slow, fp64 CPU statement of the gated delta rule.  TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import this package.
It shares no code with the GPU library and never imports it.

  gated_delta(...)  token-by-token recurrence (C, fp64, threads over (sequence, head) pairs):
                    S <- Diag(alpha_t) S;  v_hat = S^T k_t;  S <- S + beta_t k_t (v_t - v_hat)^T;
                    o_t = S^T q_t.
  linear_attn(...)  S <- S + k_t v_t^T;  o_t = S^T q_t   (alpha = 1, no erase term, no beta).
  gated_linear(...) S <- Diag(alpha_t) S + k_t v_t^T;  o_t = S^T q_t   (no erase term, no beta;
                    engineermaxxing §05b, heqinghuang §11; per key channel as dev.to §5).
  layer_prologue(xq, xk, a, b)  the layer's input maps (numpy fp64): q = normalize(silu(xq)),
                    k = normalize(silu(xk)) over d_k (x / max(||x||, 1e-12)) and beta = sigmoid(b)
                    as heqinghuang §09 writes them; alpha = sigmoid(a), scalar per head as
                    engineermaxxing §05c, per channel as its §06b.
  phi(x)            elu(x) + 1 (x + 1 for x > 0, e^x otherwise): the feature map of normalised
                    linear attention (heqinghuang §07, engineermaxxing §02g).
  normalized_linear(q, k, v, S0, z0, cu_seqlens, eps)  normalised phi-linear attention, token by
                    token in numpy fp64: S <- S + phi(k_t) v_t^T, z <- z + phi(k_t),
                    o_t = S^T phi(q_t) / (phi(q_t) . z + eps) (both after the write, as the pages'
                    listings order them).
  output_gate(o, g) o * sigmoid(g), element by element (numpy fp64): the KDA layer's output
                    gate (dev.to §5: full rank and input dependent in K3; a sigmoid multiplied
                    into the output feature by feature, as heqinghuang §15 describes the gate of
                    the attention layers).
  chunked           (module) the chunk-parallel rewrite of the same recurrence in numpy fp64; a
                    derivation check for the chunk algebra, itself compared against gated_delta.

Pages followed (sections as numbered on each page):
  dev.to "From GPT-2 to Kimi K3: How Language Models Learned to Manage Memory" §3-§5
  (fade, then read, then correct; one retention factor per key channel = row of S);
  engineermaxxing "From GPT-2 to Kimi K3: one memory, seven eviction policies" §03b, §05c, §06b;
  heqinghuang "gpt2-to-kimi" §09-§11 (the naive loop reads the output after the write);
  kylehh "Kimi K3: From KV Cache to Selective Memory" §5 (v_hat = S^T k).
Readings where the pages disagree (decay before erase; the read sees the faded state) are the
ones the C source states in its header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdr_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the C oracle into oracle/liboracle.so (gcc, -O2, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                               tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            lib = ctypes.CDLL(_LIB)
            f = lib.gdr_oracle_run
            P = ctypes.c_void_p
            f.argtypes = [ctypes.c_int] * 5 + [P, P, P, P, P, ctypes.c_int, P, P, P, P, P,
                                               ctypes.c_int, ctypes.c_int]
            f.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _run(mode, q, k, v, alpha, beta, S0, cu_seqlens, pairs, threads):
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, T], dtype=np.int64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    n_seqs = len(cu) - 1
    alpha = _f64(alpha)
    beta = _f64(beta)
    per_channel = 1
    if alpha is not None:
        per_channel = 1 if alpha.ndim == 3 else 0
    if S0 is not None:
        S0 = _f64(S0).reshape(n_seqs, H, dk, dv)
    out = np.zeros((T, H, dv), dtype=np.float64)
    S_final = np.zeros((n_seqs, H, dk, dv), dtype=np.float64)
    pl = None
    n_pairs = 0
    if pairs is not None:
        pl = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        n_pairs = int(pl.shape[0])
    threads = default_threads() if threads is None else int(threads)
    rc = _load().gdr_oracle_run(mode, n_seqs, H, dk, dv, _ptr(cu), _ptr(q), _ptr(k), _ptr(v),
                                _ptr(alpha), per_channel, _ptr(beta), _ptr(S0), _ptr(out),
                                _ptr(S_final), _ptr(pl), n_pairs, threads)
    if rc != 0:
        raise RuntimeError("oracle failed with code %d" % rc)
    return out, S_final


def gated_delta(q, k, v, alpha, beta, S0=None, cu_seqlens=None, pairs=None, threads=None):
    """Gated delta rule (per-channel alpha [T,H,d_k] or scalar alpha [T,H]); returns
    (out [T,H,d_v], S_final [N,H,d_k,d_v]) in fp64."""
    return _run(0, q, k, v, alpha, beta, S0, cu_seqlens, pairs, threads)


def linear_attn(q, k, v, S0=None, cu_seqlens=None, pairs=None, threads=None):
    """Unnormalised linear attention (alpha = 1, no erase term); returns (out, S_final)."""
    return _run(1, q, k, v, None, None, S0, cu_seqlens, pairs, threads)


def gated_linear(q, k, v, alpha, S0=None, cu_seqlens=None, pairs=None, threads=None):
    """Gated linear attention: S <- Diag(alpha_t) S + k_t v_t^T (per-channel alpha [T,H,d_k] or
    scalar alpha [T,H]), o_t = S^T q_t; returns (out, S_final) in fp64."""
    return _run(2, q, k, v, alpha, None, S0, cu_seqlens, pairs, threads)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def layer_prologue(xq, xk, a, b):
    """The layer's maps from raw projections to the rule's inputs, in fp64: returns
    (q, k, alpha, beta) with q = xq*sigmoid(xq) / max(||.||, 1e-12) over the last axis (likewise
    k), alpha = sigmoid(a) (per channel or scalar, as a's shape), beta = sigmoid(b)."""
    out = []
    for x in (xq, xk):
        x = np.asarray(x, dtype=np.float64)
        s = x * _sigmoid(x)
        n = np.sqrt(np.sum(s * s, axis=-1, keepdims=True))
        out.append(s / np.maximum(n, 1e-12))
    out.append(_sigmoid(np.asarray(a, dtype=np.float64)))
    out.append(_sigmoid(np.asarray(b, dtype=np.float64)))
    return tuple(out)


def phi(x):
    """elu(x) + 1 in fp64: x + 1 where x > 0, e^x elsewhere (always > 0)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def normalized_linear(q, k, v, S0=None, z0=None, cu_seqlens=None, eps=0.0):
    """Normalised phi-linear attention, per (sequence, head), one token at a time in fp64.
    q, k [T,H,d_k], v [T,H,d_v]; S0 [N,H,d_k,d_v] and z0 [N,H,d_k] or None (zeros).
    Returns (out [T,H,d_v], S_final [N,H,d_k,d_v], z_final [N,H,d_k])."""
    q, k, v = phi(q), phi(k), np.asarray(v, dtype=np.float64)
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    out = np.zeros((T, H, dv))
    S_fin = np.zeros((N, H, dk, dv))
    z_fin = np.zeros((N, H, dk))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if S0 is None else np.array(S0[n, h], dtype=np.float64)
            z = np.zeros(dk) if z0 is None else np.array(z0[n, h], dtype=np.float64)
            for t in range(cu[n], cu[n + 1]):
                S += np.outer(k[t, h], v[t, h])
                z += k[t, h]
                out[t, h] = (q[t, h] @ S) / (q[t, h] @ z + eps)
            S_fin[n, h] = S
            z_fin[n, h] = z
    return out, S_fin, z_fin


def output_gate(o, g):
    """o * sigmoid(g) in fp64 (o and g of one shape, e.g. [T, H, d_v])."""
    o = np.asarray(o, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    return o / (1.0 + np.exp(-g))


def decode_step(q, k, v, alpha, beta, S):
    """One token per sequence from the state S [N,H,d_k,d_v]; q,k [N,H,d_k], v [N,H,d_v],
    alpha [N,H,d_k] or [N,H], beta [N,H].  Returns (out [N,H,d_v], S_new)."""
    N = q.shape[0]
    cu = np.arange(N + 1, dtype=np.int64)
    return _run(0, q, k, v, alpha, beta, S, cu, None, None)
