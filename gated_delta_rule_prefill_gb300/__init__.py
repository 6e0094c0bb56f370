"""gated_delta_rule_prefill_gb300 -- Python binding of libgdr (the gated delta rule on GB300).

Same names as the C ABI (include/gdr.h); this layer only marshals torch CUDA tensors into
pointers and sizes and raises on a non-zero status.  Every step of the computation runs in the
library's CUDA kernels; there is no Python or CPU fallback.

    gdr_prefill(q, k, v, alpha, beta, S0=None, cu_seqlens=None, out=None, S_final=None, ...)
    gdr_decode_step(q, k, v, alpha, beta, S_inout, out=None)
    gdr_linear_attn(q, k, v, S0=None, cu_seqlens=None, out=None, S_final=None, ...)
    gdr_gated_linear_attn(q, k, v, alpha, S0=None, cu_seqlens=None, out=None, S_final=None, ...)
    gdr_prefill_workspace_size(n_seqs, H, d_k, d_v, dtype)  /  gdr_workspace_status(workspace)
    gdr_query_device_status()  -- takes the library's error word on the current device
    gdr_check_wait_timeout(workspace, limit_ns)  -- a bounded wait made to run out (error path)
    gdr_prefill_host(q, k, v, alpha, beta, ...)  -- host (CPU) tensors in and out, copies inside
    gdr_prefill_host_buffer_size(n_seqs, H, total_tokens, d_k, d_v, dtype, gate, piece_tokens)
    gdr_layer_prologue(xq, xk, a=None, b=None, q=None, k=None, alpha=None, beta=None)
    gdr_normalized_linear_attn(q, k, v, eps=0.0, S0=None, z0=None, cu_seqlens=None, ...)
    gdr_gated_linear_decode_step(q, k, v, alpha, S_inout)  /  gdr_normalized_linear_decode_step(
        q, k, v, S_inout, z_inout, eps=0.0)

prologue=True (GDR_FLAG_LAYER_PROLOGUE) makes q, k, alpha, beta the layer's raw projections: the
kernels form q, k = normalize(silu(.)) and alpha, beta = sigmoid(.) as they load them.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (GDR_BF16, GDR_ERR_DEVICE_CHECK, GDR_F32, GDR_FLAG_FORCE_SIMT,
                   GDR_FLAG_LAYER_PROLOGUE, GDR_FLAG_NO_CLUSTER, GDR_FLAG_PREFER_QUEUE,
                   GDR_GATE_CHANNEL, GDR_GATE_SCALAR, GDR_OK, GdrError, GdrShape)

__all__ = ["gdr_prefill", "gdr_prefill_output_gate", "gdr_decode_step", "gdr_linear_attn",
           "gdr_gated_linear_attn", "gdr_layer_prologue", "gdr_normalized_linear_attn",
           "gdr_gated_linear_decode_step", "gdr_normalized_linear_decode_step",
           "gdr_prefill_workspace_size",
           "gdr_workspace_status", "gdr_query_device_status", "gdr_check_wait_timeout",
           "gdr_prefill_host",
           "gdr_prefill_host_buffer_size",
           "make_shape", "GdrError"]

_DT = {torch.float32: GDR_F32, torch.bfloat16: GDR_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def make_shape(n_seqs, H, total_tokens, d_k, d_v, dtype, gate=GDR_GATE_CHANNEL, chunk_size=0,
               flags=0) -> GdrShape:
    return GdrShape(n_seqs, H, total_tokens, d_k, d_v, dtype, gate, chunk_size, flags)


def gdr_prefill_workspace_size(n_seqs: int, H: int = 1, d_k: int = 128, d_v: int = 128,
                               dtype: str = "bf16") -> int:
    """Bytes of the workspace gdr_prefill / gdr_linear_attn use for this shape."""
    sh = make_shape(n_seqs, H, 0, d_k, d_v, GDR_BF16 if dtype == "bf16" else GDR_F32)
    return int(_abi.load().gdr_prefill_workspace_size(ctypes.byref(sh)))


def _workspace(n_seqs, H, d_k, d_v, dtype, device, workspace):
    if workspace is None:
        need = gdr_prefill_workspace_size(n_seqs, H, d_k, d_v, dtype)
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return workspace


def _prefill_like(kind, q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, workspace,
                  chunk_size, force_simt, stream, want_final, no_cluster=False,
                  prefer_queue=False, g=None, prologue=False):
    """kind: "delta" (gdr_prefill), "linear" (gdr_linear_attn) or "gla"
    (gdr_gated_linear_attn)."""
    linear = kind == "linear"
    T, H, dk = q.shape
    dv = v.shape[2]
    dtype = _DT.get(q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype)
    n_seqs = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    gate = GDR_GATE_CHANNEL
    if not linear:
        _check(alpha, "alpha", torch.float32)
        if kind == "delta":
            _check(beta, "beta", torch.float32)
        gate = GDR_GATE_CHANNEL if alpha.dim() == 3 else GDR_GATE_SCALAR
    _check(S0, "S0", torch.float32)
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.dtype)
    if S_final is None and want_final:
        S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
    _check(S_final, "S_final", torch.float32)
    ws = _workspace(n_seqs, H, dk, dv, "bf16" if dtype == GDR_BF16 else "f32", q.device,
                    workspace)
    flags = ((GDR_FLAG_FORCE_SIMT if force_simt else 0) | (GDR_FLAG_NO_CLUSTER if no_cluster else 0)
             | (GDR_FLAG_PREFER_QUEUE if prefer_queue else 0)
             | (GDR_FLAG_LAYER_PROLOGUE if prologue else 0))
    sh = make_shape(n_seqs, H, T, dk, dv, dtype, gate, chunk_size, flags)
    lib = _abi.load()
    if linear:
        rc = lib.gdr_linear_attn(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(S0),
                                 _ptr(cu_seqlens), _ptr(out), _ptr(S_final), _ptr(ws),
                                 ws.numel(), _stream(stream))
    elif g is not None:
        _check(g, "g", q.dtype)
        rc = lib.gdr_prefill_output_gate(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                         _ptr(beta), _ptr(g), _ptr(S0), _ptr(cu_seqlens),
                                         _ptr(out), _ptr(S_final), _ptr(ws), ws.numel(),
                                         _stream(stream))
    elif kind == "gla":
        rc = lib.gdr_gated_linear_attn(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                       _ptr(S0), _ptr(cu_seqlens), _ptr(out), _ptr(S_final),
                                       _ptr(ws), ws.numel(), _stream(stream))
    else:
        rc = lib.gdr_prefill(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                             _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(out), _ptr(S_final),
                             _ptr(ws), ws.numel(), _stream(stream))
    if rc != 0:
        raise GdrError(rc, {"linear": "gdr_linear_attn", "gla": "gdr_gated_linear_attn"}.get(
            kind, "gdr_prefill"))
    return out, S_final


def gdr_prefill(q, k, v, alpha, beta, S0=None, cu_seqlens=None, out=None, S_final=None,
                workspace=None, chunk_size=0, force_simt=False, stream=None, want_final=True,
                no_cluster=False, prefer_queue=False, prologue=False):
    """Chunked packed-varlen prefill.  q,k [T,H,d_k], v [T,H,d_v] (fp32 or bf16); alpha
    [T,H,d_k] or [T,H] fp32; beta [T,H] fp32; S0 [N,H,d_k,d_v] fp32 or None; cu_seqlens int32
    [N+1] or None.  Returns (out [T,H,d_v], S_final [N,H,d_k,d_v] or None)."""
    return _prefill_like("delta", q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, workspace,
                         chunk_size, force_simt, stream, want_final, no_cluster, prefer_queue,
                         prologue=prologue)


def gdr_prefill_output_gate(q, k, v, alpha, beta, g, S0=None, cu_seqlens=None, out=None,
                            S_final=None, workspace=None, chunk_size=0, force_simt=False,
                            stream=None, want_final=True, no_cluster=False, prefer_queue=False,
                            prologue=False):
    """gdr_prefill with the output gate: out = o * sigmoid(g), g [T,H,d_v] in q's dtype."""
    return _prefill_like("delta", q, k, v, alpha, beta, S0, cu_seqlens, out, S_final, workspace,
                         chunk_size, force_simt, stream, want_final, no_cluster, prefer_queue,
                         g=g, prologue=prologue)


def _check_host(t, name, dtype=None):
    if t is None:
        return
    if t.is_cuda:
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def gdr_prefill_host_buffer_size(n_seqs, H, total_tokens, d_k=128, d_v=128, dtype="bf16",
                                 gate=GDR_GATE_CHANNEL, piece_tokens=0) -> int:
    """Bytes of the device buffer gdr_prefill_host needs."""
    sh = make_shape(n_seqs, H, total_tokens, d_k, d_v, GDR_BF16 if dtype == "bf16" else GDR_F32,
                    gate)
    return int(_abi.load().gdr_prefill_host_buffer_size(ctypes.byref(sh), int(piece_tokens)))


def gdr_prefill_host(q, k, v, alpha, beta, S0=None, cu_seqlens=None, out=None, S_final=None,
                     piece_tokens=0, buffer=None, device=None, stream=None, want_final=True,
                     prologue=False):
    """gdr_prefill on host (CPU) tensors -- pinned memory lets the copies overlap the kernels.
    q, k, v, alpha, beta, S0, out, S_final and cu_seqlens (int32) are CPU tensors; `buffer` is
    a CUDA uint8 tensor of gdr_prefill_host_buffer_size bytes (allocated on `device` if None).
    The call is asynchronous on `stream`: synchronise it before reading out / S_final."""
    T, H, dk = q.shape
    dv = v.shape[2]
    dtype = _DT.get(q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_host(t, n, q.dtype)
    _check_host(alpha, "alpha", torch.float32)
    _check_host(beta, "beta", torch.float32)
    _check_host(S0, "S0", torch.float32)
    _check_host(cu_seqlens, "cu_seqlens", torch.int32)
    gate = GDR_GATE_CHANNEL if alpha.dim() == 3 else GDR_GATE_SCALAR
    n_seqs = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype).pin_memory()
    _check_host(out, "out", q.dtype)
    if S_final is None and want_final:
        S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32).pin_memory()
    _check_host(S_final, "S_final", torch.float32)
    sh = make_shape(n_seqs, H, T, dk, dv, dtype, gate, 0,
                    GDR_FLAG_LAYER_PROLOGUE if prologue else 0)
    lib = _abi.load()
    if buffer is None:
        need = int(lib.gdr_prefill_host_buffer_size(ctypes.byref(sh), int(piece_tokens)))
        dev = torch.device("cuda") if device is None else torch.device(device)
        buffer = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(buffer, "buffer", torch.uint8)
    rc = lib.gdr_prefill_host(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                              _ptr(beta), _ptr(S0), _ptr(cu_seqlens), _ptr(out), _ptr(S_final),
                              int(piece_tokens), _ptr(buffer), buffer.numel(), _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_prefill_host")
    return out, S_final


def gdr_linear_attn(q, k, v, S0=None, cu_seqlens=None, out=None, S_final=None, workspace=None,
                    chunk_size=0, force_simt=False, stream=None, want_final=True):
    """Plain linear attention (alpha = 1, no erase).  Returns (out, S_final)."""
    return _prefill_like("linear", q, k, v, None, None, S0, cu_seqlens, out, S_final, workspace,
                         chunk_size, force_simt, stream, want_final)


def gdr_gated_linear_attn(q, k, v, alpha, S0=None, cu_seqlens=None, out=None, S_final=None,
                          workspace=None, chunk_size=0, force_simt=False, stream=None,
                          want_final=True, no_cluster=False, prologue=False):
    """Gated linear attention: S <- Diag(alpha) S + k v^T (no erase, no beta); alpha [T,H,d_k]
    or [T,H] fp32.  Returns (out, S_final)."""
    return _prefill_like("gla", q, k, v, alpha, None, S0, cu_seqlens, out, S_final, workspace,
                         chunk_size, force_simt, stream, want_final, no_cluster,
                         prologue=prologue)


def gdr_normalized_linear_attn(q, k, v, eps=0.0, S0=None, z0=None, cu_seqlens=None, out=None,
                               S_final=None, z_final=None, workspace=None, chunk_size=0,
                               force_simt=False, stream=None, want_final=True):
    """Normalised phi-linear attention (phi = elu + 1): S <- S + phi(k) v^T, z <- z + phi(k),
    o = S^T phi(q) / (phi(q) . z + eps).  q, k [T,H,d_k], v [T,H,d_v]; S0 [N,H,d_k,d_v] and z0
    [N,H,d_k] fp32 or None.  Returns (out, S_final, z_final)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    dtype = _DT.get(q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype)
    n_seqs = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    _check(S0, "S0", torch.float32)
    _check(z0, "z0", torch.float32)
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    if out is None:
        out = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.dtype)
    if want_final:
        if S_final is None:
            S_final = torch.empty((n_seqs, H, dk, dv), dtype=torch.float32, device=q.device)
        if z_final is None:
            z_final = torch.empty((n_seqs, H, dk), dtype=torch.float32, device=q.device)
    _check(S_final, "S_final", torch.float32)
    _check(z_final, "z_final", torch.float32)
    ws = _workspace(n_seqs, H, dk, dv, "bf16" if dtype == GDR_BF16 else "f32", q.device,
                    workspace)
    sh = make_shape(n_seqs, H, T, dk, dv, dtype, GDR_GATE_CHANNEL, chunk_size,
                    GDR_FLAG_FORCE_SIMT if force_simt else 0)
    rc = _abi.load().gdr_normalized_linear_attn(
        ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), float(eps), _ptr(S0), _ptr(z0),
        _ptr(cu_seqlens), _ptr(out), _ptr(S_final), _ptr(z_final), _ptr(ws), ws.numel(),
        _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_normalized_linear_attn")
    return out, S_final, z_final


def gdr_layer_prologue(xq, xk, a=None, b=None, q=None, k=None, alpha=None, beta=None,
                       stream=None):
    """The layer prologue as its own pass: q, k = normalize(silu(xq, xk)) over d_k, alpha =
    sigmoid(a) ([T,H,d_k] or [T,H]), beta = sigmoid(b) ([T,H]).  Outputs are allocated when None
    and may be the inputs themselves (in place).  Returns (q, k, alpha, beta)."""
    T, H, dk = xq.shape
    dtype = _DT.get(xq.dtype)
    if dtype is None:
        raise ValueError("xq/xk must be float32 or bfloat16")
    _check(xq, "xq", xq.dtype)
    _check(xk, "xk", xq.dtype)
    _check(a, "a", torch.float32)
    _check(b, "b", torch.float32)
    q = torch.empty_like(xq) if q is None else q
    k = torch.empty_like(xk) if k is None else k
    if a is not None and alpha is None:
        alpha = torch.empty_like(a)
    if b is not None and beta is None:
        beta = torch.empty_like(b)
    for t, n in ((q, "q"), (k, "k")):
        _check(t, n, xq.dtype)
    _check(alpha, "alpha", torch.float32)
    _check(beta, "beta", torch.float32)
    gate = GDR_GATE_CHANNEL if (a is None or a.dim() == 3) else GDR_GATE_SCALAR
    sh = make_shape(1, H, T, dk, dk, dtype, gate)
    rc = _abi.load().gdr_layer_prologue(ctypes.byref(sh), _ptr(xq), _ptr(xk), _ptr(a), _ptr(b),
                                        _ptr(q), _ptr(k), _ptr(alpha), _ptr(beta),
                                        _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_layer_prologue")
    return q, k, alpha, beta


def gdr_decode_step(q, k, v, alpha, beta, S_inout, out=None, stream=None, prologue=False):
    """One token per sequence; S_inout [N,H,d_k,d_v] fp32 is updated in place.  Returns out."""
    N, H, dk = q.shape
    dv = v.shape[2]
    dtype = _DT.get(q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype)
    _check(alpha, "alpha", torch.float32)
    _check(beta, "beta", torch.float32)
    _check(S_inout, "S_inout", torch.float32)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.dtype)
    gate = GDR_GATE_CHANNEL if alpha.dim() == 3 else GDR_GATE_SCALAR
    sh = make_shape(N, H, N, dk, dv, dtype, gate, 0, GDR_FLAG_LAYER_PROLOGUE if prologue else 0)
    rc = _abi.load().gdr_decode_step(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                     _ptr(beta), _ptr(S_inout), _ptr(out), _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_decode_step")
    return out


def _decode_inputs(q, k, v, S_inout, out):
    N, H, dk = q.shape
    dv = v.shape[2]
    dtype = _DT.get(q.dtype)
    if dtype is None:
        raise ValueError("q/k/v must be float32 or bfloat16")
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, q.dtype)
    _check(S_inout, "S_inout", torch.float32)
    if out is None:
        out = torch.empty((N, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.dtype)
    return N, H, dk, dv, dtype, out


def gdr_gated_linear_decode_step(q, k, v, alpha, S_inout, out=None, stream=None, prologue=False):
    """One token per sequence of gated linear attention: S <- Diag(alpha) S + k v^T, o = S^T q;
    S_inout [N,H,d_k,d_v] fp32 updated in place; alpha [N,H,d_k] or [N,H].  Returns out."""
    N, H, dk, dv, dtype, out = _decode_inputs(q, k, v, S_inout, out)
    _check(alpha, "alpha", torch.float32)
    gate = GDR_GATE_CHANNEL if alpha.dim() == 3 else GDR_GATE_SCALAR
    sh = make_shape(N, H, N, dk, dv, dtype, gate, 0, GDR_FLAG_LAYER_PROLOGUE if prologue else 0)
    rc = _abi.load().gdr_gated_linear_decode_step(ctypes.byref(sh), _ptr(q), _ptr(k), _ptr(v),
                                                  _ptr(alpha), _ptr(S_inout), _ptr(out),
                                                  _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_gated_linear_decode_step")
    return out


def gdr_normalized_linear_decode_step(q, k, v, S_inout, z_inout, eps=0.0, out=None, stream=None):
    """One token per sequence of normalised phi-linear attention: S <- S + phi(k) v^T,
    z <- z + phi(k), o = S^T phi(q) / (phi(q) . z + eps); S_inout [N,H,d_k,d_v] and z_inout
    [N,H,d_k] fp32 updated in place.  Returns out."""
    N, H, dk, dv, dtype, out = _decode_inputs(q, k, v, S_inout, out)
    _check(z_inout, "z_inout", torch.float32)
    sh = make_shape(N, H, N, dk, dv, dtype, GDR_GATE_CHANNEL)
    rc = _abi.load().gdr_normalized_linear_decode_step(ctypes.byref(sh), _ptr(q), _ptr(k),
                                                       _ptr(v), float(eps), _ptr(S_inout),
                                                       _ptr(z_inout), _ptr(out), _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_normalized_linear_decode_step")
    return out


def gdr_workspace_status(workspace, stream=None) -> int:
    """Synchronise and return (then clear) the device-check code of a workspace."""
    code = ctypes.c_int32(0)
    rc = _abi.load().gdr_workspace_status(_ptr(workspace), _stream(stream), ctypes.byref(code))
    if rc != 0:
        raise GdrError(rc, "gdr_workspace_status")
    return int(code.value)


def gdr_query_device_status(stream=None) -> int:
    """Synchronise, then take (read and clear) the library's error word on the current device.
    Returns the C status: GDR_OK (0) if no device-side check failed since the last query,
    GDR_ERR_DEVICE_CHECK (4) if one did; raises on a CUDA failure."""
    rc = _abi.load().gdr_query_device_status(_stream(stream))
    if rc not in (GDR_OK, GDR_ERR_DEVICE_CHECK):
        raise GdrError(rc, "gdr_query_device_status")
    return int(rc)


def gdr_check_wait_timeout(workspace, limit_ns: int, stream=None) -> None:
    """Launch the library's failure-detection check: one warp waits, with the kernels' bounded
    wait, on a barrier that nothing completes and records GDR_DEVCHECK_TIMEOUT after limit_ns
    in the workspace word and the per-device word (read them with gdr_workspace_status and
    gdr_query_device_status).  Asynchronous on the stream."""
    rc = _abi.load().gdr_check_wait_timeout(_ptr(workspace), ctypes.c_uint64(int(limit_ns)),
                                            _stream(stream))
    if rc != 0:
        raise GdrError(rc, "gdr_check_wait_timeout")


def compute_dtype(dtype: str, d: int, force_simt: bool = False) -> str:
    """Arithmetic type of the prefill kernel the library selects for these inputs: bf16
    tensor-core operands with fp32 accumulation and state for bf16 inputs at d = 128, fp32
    FFMA otherwise."""
    return "bf16" if (dtype == "bf16" and d == 128 and not force_simt) else "f32"
