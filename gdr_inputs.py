"""Seeded synthetic workloads for the gated delta rule (inputs only, no method arithmetic).

This module is shared by the oracle-side tests and the GPU-side tests / bench.  It draws the
inputs each workload is specified with and nothing else: it contains none of the recurrence,
none of the chunk algebra and no kernel logic.

Distributions (the same for every workload):
  * q, k  ~ N(0, 1) per element, then L2-normalised per (token, head) over d_k (done in fp64),
  * v     ~ N(0, 1),
  * beta  = sigmoid(N(0, 1))                     one scalar per (token, head),
  * alpha = exp(-softplus(N(-4, 1)))             per key channel, or one scalar per (token, head),
  * S0    ~ N(0, 0.01), i.e. standard deviation 0.1, per (sequence, head) (or zeros).
q, k, v are then rounded to the workload dtype (bf16 round-to-nearest-even, or kept fp32);
alpha, beta and S0 stay fp32.  Every array returned holds values that are exactly representable
in the dtype the GPU receives, as float32, so the oracle widens the very same numbers to fp64.

Each (tensor, sequence, head) block has its own PCG64 stream, keyed by
SeedSequence(seed, spawn_key=(tensor_id, seq, head)); any subset of blocks can therefore be
regenerated independently (the oracle side samples (sequence, head) pairs of large workloads).
Decode steps use one stream per (tensor, step) covering all [N, H, d] entries.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# tensor ids used in the stream keys
_Q, _K, _V, _ALPHA, _BETA, _S0, _LEN = 0, 1, 2, 3, 4, 5, 6
_STEP_BASE = 100  # decode step streams: tensor id + _STEP_BASE


# ----------------------------------------------------------------------------------------------
# bf16 helpers (numpy only)
# ----------------------------------------------------------------------------------------------
def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of float32 values that are already exactly bf16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------------------------
# workload descriptions
# ----------------------------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    H: int
    d_k: int
    d_v: int
    dtype: str  # "f32" or "bf16": dtype of q, k, v and out
    gate: str  # "channel" (alpha [T,H,d_k]) or "scalar" (alpha [T,H])
    seqlens: np.ndarray  # int64 [n_seqs]
    s0: str  # "zeros" or "normal"
    chunk_size: int = 0  # 0: the kernel's choice
    linear_pass: bool = False  # also run plain linear attention on the same q/k/v/S0
    decode_steps: int = 0  # >0: serving-decode workload (seqlens = prefill length per sequence)

    @property
    def n_seqs(self) -> int:
        return int(len(self.seqlens))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.seqlens)]).astype(np.int64)

    @property
    def total_tokens(self) -> int:
        return int(np.sum(self.seqlens))


def _loguniform_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(_LEN,))))
    u = rng.uniform(math.log(lo), math.log(hi), size=n)
    return np.floor(np.exp(u)).astype(np.int64)


def workload(name: str) -> Workload:
    """The five named workloads (sizes and distributions as specified for this method).

    kda_t256_d64_f32         single sequence, H=1, T=256, d=64, fp32, per-channel alpha, S0=0
    gdn_b4_h16_t4096         4 x 4096 tokens, H=16, d=128, bf16, scalar alpha, S0=0, chunk 64
    kda_b1_h32_t32768        1 x 32768 tokens, H=32, d=128, bf16, per-channel alpha, S0~N(0,.01)
    decode_n256_h32          256 sequences, H=32, d=128, states from a 2048-token prefill
                             (S0=0, bf16), then one-token decode steps
    varlen_n64_h16           64 sequences, lengths floor(exp(U(ln 128, ln 65536))), H=16, d=128,
                             bf16, per-channel alpha, per-sequence S0~N(0,.01), plus a plain
                             linear-attention pass over the same q/k/v/S0
    """
    if name == "kda_t256_d64_f32":
        return Workload(name, 1000, 1, 64, 64, "f32", "channel", np.array([256]), "zeros")
    if name == "gdn_b4_h16_t4096":
        return Workload(name, 1001, 16, 128, 128, "bf16", "scalar", np.array([4096] * 4), "zeros",
                        chunk_size=64)
    if name == "kda_b1_h32_t32768":
        return Workload(name, 1002, 32, 128, 128, "bf16", "channel", np.array([32768]), "normal")
    if name == "decode_n256_h32":
        return Workload(name, 1003, 32, 128, 128, "bf16", "channel", np.array([2048] * 256),
                        "zeros", decode_steps=1000)
    if name == "varlen_n64_h16":
        return Workload(name, 1004, 16, 128, 128, "bf16", "channel",
                        _loguniform_lengths(1004, 64, 128, 65536), "normal", linear_pass=True)
    raise KeyError(name)


WORKLOADS = ("kda_t256_d64_f32", "gdn_b4_h16_t4096", "kda_b1_h32_t32768", "decode_n256_h32",
             "varlen_n64_h16")


def custom(name="custom", seed=7, seqlens=(64,), H=1, d_k=64, d_v=64, dtype="f32", gate="channel",
           s0="zeros") -> Workload:
    """A small ad-hoc workload with the standard distributions (for tests)."""
    return Workload(name, seed, H, d_k, d_v, dtype, gate, np.asarray(seqlens, dtype=np.int64), s0)


# ----------------------------------------------------------------------------------------------
# drawing
# ----------------------------------------------------------------------------------------------
def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=key)))


def _unit_rows(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-30)).astype(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return np.where(x > 30, x, np.log1p(np.exp(np.minimum(x, 30))))


def _cast(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_round(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def draw_qkv_gates(rngs, L: int, d_k: int, d_v: int, dtype: str, gate: str):
    rq, rk, rv, ra, rb = rngs
    q = _cast(_unit_rows(rq.standard_normal((L, d_k), dtype=np.float32)), dtype)
    k = _cast(_unit_rows(rk.standard_normal((L, d_k), dtype=np.float32)), dtype)
    v = _cast(rv.standard_normal((L, d_v), dtype=np.float32), dtype)
    ashape = (L, d_k) if gate == "channel" else (L,)
    a = ra.standard_normal(ashape, dtype=np.float32).astype(np.float64) - 4.0
    alpha = np.exp(-_softplus(a)).astype(np.float32)
    b = rb.standard_normal((L,), dtype=np.float32).astype(np.float64)
    beta = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
    return q, k, v, alpha, beta


def draw_raw(rngs, L: int, d_k: int, d_v: int, dtype: str, gate: str):
    """Raw layer projections of the same workload: xq, xk ~ N(0, 1) (in the input dtype),
    v as draw_qkv_gates, a = 4 - N(0, 1) (sigmoid(a) has draw_qkv_gates' alpha distribution),
    b ~ N(0, 1) (fp32)."""
    rq, rk, rv, ra, rb = rngs
    xq = _cast(rq.standard_normal((L, d_k), dtype=np.float32), dtype)
    xk = _cast(rk.standard_normal((L, d_k), dtype=np.float32), dtype)
    v = _cast(rv.standard_normal((L, d_v), dtype=np.float32), dtype)
    ashape = (L, d_k) if gate == "channel" else (L,)
    a = (4.0 - ra.standard_normal(ashape, dtype=np.float32)).astype(np.float32)
    b = rb.standard_normal((L,), dtype=np.float32).astype(np.float32)
    return xq, xk, v, a, b


def gen_block(wl: Workload, seq: int, head: int, raw: bool = False) -> dict:
    """Inputs of one (sequence, head): q [L,d_k], k [L,d_k], v [L,d_v], alpha [L,d_k] or [L],
    beta [L], S0 [d_k,d_v] (all float32 holding exactly-representable values).  raw=True: q, k,
    alpha, beta hold the raw projections of draw_raw instead."""
    L = int(wl.seqlens[seq])
    rngs = [_rng(wl.seed, t, seq, head) for t in (_Q, _K, _V, _ALPHA, _BETA)]
    draw = draw_raw if raw else draw_qkv_gates
    q, k, v, alpha, beta = draw(rngs, L, wl.d_k, wl.d_v, wl.dtype, wl.gate)
    if wl.s0 == "normal":
        S0 = (0.1 * _rng(wl.seed, _S0, seq, head).standard_normal((wl.d_k, wl.d_v),
                                                                     dtype=np.float32))
        S0 = S0.astype(np.float32)
    else:
        S0 = np.zeros((wl.d_k, wl.d_v), dtype=np.float32)
    return dict(q=q, k=k, v=v, alpha=alpha, beta=beta, S0=S0)


def alloc_full(wl: Workload, heads=None, seqs=None):
    """Empty token-major arrays for the chosen sequences / heads."""
    seqs = list(range(wl.n_seqs)) if seqs is None else list(seqs)
    heads = list(range(wl.H)) if heads is None else list(heads)
    lens = wl.seqlens[seqs]
    T = int(np.sum(lens))
    Hs = len(heads)
    a = dict(
        q=np.empty((T, Hs, wl.d_k), np.float32),
        k=np.empty((T, Hs, wl.d_k), np.float32),
        v=np.empty((T, Hs, wl.d_v), np.float32),
        alpha=np.empty((T, Hs, wl.d_k) if wl.gate == "channel" else (T, Hs), np.float32),
        beta=np.empty((T, Hs), np.float32),
        S0=np.empty((len(seqs), Hs, wl.d_k, wl.d_v), np.float32),
        cu_seqlens=np.concatenate([[0], np.cumsum(lens)]).astype(np.int64),
    )
    return a, seqs, heads


def gen_full(wl: Workload, heads=None, seqs=None, threads: int = 8, raw: bool = False) -> dict:
    """Token-major inputs for the chosen sequences and heads:
    q, k [T,H',d_k]; v [T,H',d_v]; alpha [T,H',d_k] or [T,H']; beta [T,H']; S0 [N',H',d_k,d_v];
    cu_seqlens [N'+1] (int64).  Blocks are drawn in parallel threads (numpy releases the GIL).
    raw=True: q, k, alpha, beta hold raw projections (draw_raw)."""
    a, seqs, heads = alloc_full(wl, heads, seqs)
    cu = a["cu_seqlens"]

    def fill(job):
        si, hi = job
        blk = gen_block(wl, seqs[si], heads[hi], raw)
        t0, t1 = cu[si], cu[si + 1]
        for name in ("q", "k", "v", "alpha", "beta"):
            a[name][t0:t1, hi] = blk[name]
        a["S0"][si, hi] = blk["S0"]

    jobs = [(si, hi) for si in range(len(seqs)) for hi in range(len(heads))]
    if threads > 1 and len(jobs) > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, jobs))
    else:
        for j in jobs:
            fill(j)
    return a


def gen_decode_step(wl: Workload, step: int, raw: bool = False) -> dict:
    """Inputs of one decode step for all N sequences: q,k [N,H,d_k], v [N,H,d_v],
    alpha [N,H,d_k] (or [N,H]), beta [N,H] (raw=True: raw projections, draw_raw)."""
    N, H = wl.n_seqs, wl.H
    rngs = [_rng(wl.seed, _STEP_BASE + t, step) for t in (_Q, _K, _V, _ALPHA, _BETA)]
    draw = draw_raw if raw else draw_qkv_gates
    q, k, v, alpha, beta = draw(rngs, N * H, wl.d_k, wl.d_v, wl.dtype, wl.gate)
    shp = (N, H)
    return dict(q=q.reshape(shp + (wl.d_k,)), k=k.reshape(shp + (wl.d_k,)),
                v=v.reshape(shp + (wl.d_v,)),
                alpha=alpha.reshape(shp + ((wl.d_k,) if wl.gate == "channel" else ())),
                beta=beta.reshape(shp))


def random_state(seed: int, N: int, H: int, d_k: int, d_v: int, std: float = 0.1) -> np.ndarray:
    """A synthetic fp32 state [N,H,d_k,d_v] ~ N(0, std^2) (decode parity from a given state)."""
    return (std * _rng(seed, _S0, 99991).standard_normal((N, H, d_k, d_v), dtype=np.float32)
            ).astype(np.float32)


# ----------------------------------------------------------------------------------------------
# device-side drawing (timing only)
# ----------------------------------------------------------------------------------------------
def device_full(wl: Workload, device, seed_offset: int = 0, raw: bool = False):
    """The same distributions drawn on the device with torch's seeded generator (different
    numbers from the host streams above).  Used where only the shape and distribution of the
    inputs matter (throughput runs); parity always uses the host streams.  raw=True: q, k,
    alpha, beta are raw projections with draw_raw's distributions."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1000003 + seed_offset)
    T, H, dk, dv = wl.total_tokens, wl.H, wl.d_k, wl.d_v
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32

    def unit(shape):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        return (x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(tdt)

    def normal(shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32)

    ashape = (T, H, dk) if wl.gate == "channel" else (T, H)
    if raw:
        q = normal((T, H, dk)).to(tdt)
        k = normal((T, H, dk)).to(tdt)
        v = normal((T, H, dv)).to(tdt)
        alpha = 4.0 - normal(ashape)
        beta = normal((T, H))
    else:
        q = unit((T, H, dk))
        k = unit((T, H, dk))
        v = normal((T, H, dv)).to(tdt)
        alpha = torch.exp(-torch.nn.functional.softplus(normal(ashape) - 4.0))
        beta = torch.sigmoid(normal((T, H)))
    if wl.s0 == "normal":
        S0 = 0.1 * torch.randn((wl.n_seqs, H, dk, dv), generator=g, device=device)
    else:
        S0 = torch.zeros((wl.n_seqs, H, dk, dv), device=device)
    cu = torch.from_numpy(wl.cu_seqlens.astype(np.int32)).to(device)
    return dict(q=q, k=k, v=v, alpha=alpha.contiguous(), beta=beta.contiguous(), S0=S0,
                cu_seqlens=cu)


def device_decode_steps(wl: Workload, n_sets: int, device):
    """n_sets distinct decode-step input sets drawn on the device (throughput runs)."""
    one = dataclasses.replace(wl, seqlens=np.ones(wl.n_seqs, dtype=np.int64), s0="zeros")
    sets = []
    for i in range(n_sets):
        d = device_full(one, device, seed_offset=1 + i)
        sets.append({k: d[k] for k in ("q", "k", "v", "alpha", "beta")})
    return sets
