"""The C ABI on the CPU (no GPU needed): the library builds, loads, exports every symbol that
include/gdr.h declares, and rejects bad arguments synchronously, before any CUDA work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_prefill_gb300 import _abi, build
    build.build_library()
    return _abi.load()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gdr_[a-z0-9_]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    from gated_delta_rule_prefill_gb300 import _abi
    names = declared_functions()
    assert names and names == set(_abi.EXPORTS), names
    for n in names:
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    from gated_delta_rule_prefill_gb300 import _abi
    assert _abi.status_string(0) == "GDR_OK"
    assert _abi.status_string(2) == "GDR_ERR_UNSUPPORTED"
    assert _abi.status_string(99) == "GDR_ERR_UNKNOWN"


def _shape(**kw):
    from gated_delta_rule_prefill_gb300 import make_shape
    base = dict(n_seqs=2, H=4, total_tokens=100, d_k=128, d_v=128, dtype=1, gate=1)
    base.update(kw)
    return make_shape(**base)


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: every case below fails validation first


def _prefill(lib, sh, ws_bytes=1 << 16, **over):
    p = dict(q=FAKE, k=FAKE + 4096, v=FAKE + 8192, alpha=FAKE, beta=FAKE, S0=None, cu=FAKE,
             out=FAKE + 65536, Sf=None, ws=FAKE * 2)
    p.update(over)
    P = ctypes.c_void_p
    return lib.gdr_prefill(ctypes.byref(sh), P(p["q"]), P(p["k"]), P(p["v"]), P(p["alpha"]),
                           P(p["beta"]), P(p["S0"]), P(p["cu"]), P(p["out"]), P(p["Sf"]),
                           P(p["ws"]), ws_bytes, None)


def test_argument_errors(lib):
    INV, UNS = 1, 2
    assert lib.gdr_prefill(None, *([None] * 10), 0, None) == INV
    assert _prefill(lib, _shape(d_k=96, d_v=96)) == UNS
    assert _prefill(lib, _shape(d_k=128, d_v=64)) == UNS
    assert _prefill(lib, _shape(dtype=7)) == INV
    assert _prefill(lib, _shape(gate=5)) == INV
    assert _prefill(lib, _shape(n_seqs=0)) == INV
    assert _prefill(lib, _shape(total_tokens=-1)) == INV
    assert _prefill(lib, _shape(), q=FAKE + 2) == INV           # misaligned
    assert _prefill(lib, _shape(), q=None) == INV               # null input
    assert _prefill(lib, _shape(), alpha=None) == INV           # gated rule needs alpha
    assert _prefill(lib, _shape(), ws=None) == INV              # no workspace
    assert _prefill(lib, _shape(), ws=FAKE * 2 + 16) == INV     # workspace not 256-aligned
    assert _prefill(lib, _shape(), ws_bytes=8) == INV           # workspace too small
    assert _prefill(lib, _shape(), cu=None) == INV              # n_seqs > 1 needs cu_seqlens
    assert _prefill(lib, _shape(), out=FAKE) == INV             # out aliases q
    assert _prefill(lib, _shape(chunk_size=48)) == UNS
    assert _prefill(lib, _shape(flags=16)) == INV
    # decode: total_tokens must equal n_seqs
    P = ctypes.c_void_p
    sh = _shape(total_tokens=3)
    assert lib.gdr_decode_step(ctypes.byref(sh), *[P(FAKE + 4096 * i) for i in range(7)],
                               None) == INV


def test_workspace_size(lib):
    from gated_delta_rule_prefill_gb300 import _abi
    sh = _shape(n_seqs=64)
    n = lib.gdr_prefill_workspace_size(ctypes.byref(sh))
    assert n >= 256 + 64 * 4 and n % 256 == 0
    assert lib.gdr_prefill_workspace_size(None) == 0


def _host_call(lib, sh, cu, buf=FAKE * 4, buf_bytes=1 << 40, piece=0):
    """gdr_prefill_host with fake host pointers: every case here fails validation first."""
    P = ctypes.c_void_p
    cu_arr = None if cu is None else (ctypes.c_int32 * len(cu))(*cu)
    return lib.gdr_prefill_host(ctypes.byref(sh), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                None, cu_arr, P(FAKE), None, piece, P(buf), buf_bytes, None)


def test_host_pipeline_argument_errors(lib):
    INV, UNS = 1, 2
    sh = _shape(n_seqs=2, total_tokens=100)
    assert _host_call(lib, sh, [0, 60, 50]) == INV     # offsets decrease
    assert _host_call(lib, sh, [0, 60, 90]) == INV     # do not end at total_tokens
    assert _host_call(lib, sh, [4, 60, 100]) == INV    # do not start at 0
    assert _host_call(lib, sh, None) == INV            # two sequences need offsets
    assert _host_call(lib, sh, [0, 60, 100], buf=FAKE * 4 + 16) == INV  # buffer misaligned
    assert _host_call(lib, sh, [0, 60, 100], buf_bytes=4096) == INV     # buffer too small
    assert _host_call(lib, _shape(d_k=96, d_v=96), [0, 60, 100]) == UNS
    assert _host_call(lib, _shape(gate=5), [0, 60, 100]) == INV


def test_host_pipeline_buffer_size(lib):
    # states + offsets + workspace + two staging sets of (piece + 64) tokens
    sh = _shape(n_seqs=1, H=32, total_tokens=32768)
    small = lib.gdr_prefill_host_buffer_size(ctypes.byref(sh), 1024)
    big = lib.gdr_prefill_host_buffer_size(ctypes.byref(sh), 8192)
    per_tok = 32 * (2 * 128 * 2 + 128 * 2 + 128 * 4 + 4) + 32 * 128 * 2  # inputs + output
    assert small % 256 == 0 and big % 256 == 0
    assert big - small >= 2 * (8192 - 1024) * per_tok
    assert small >= 32 * 128 * 128 * 4 + 2 * (1024 + 64) * per_tok
    assert lib.gdr_prefill_host_buffer_size(None, 0) == 0
    # scalar gates stage one gate per (token, head)
    assert (lib.gdr_prefill_host_buffer_size(ctypes.byref(_shape(n_seqs=1, H=32, total_tokens=32768, gate=0)), 1024)
            < small)


def test_gated_linear_argument_errors(lib):
    """gdr_gated_linear_attn needs alpha but no beta."""
    INV = 1
    P = ctypes.c_void_p
    sh = _shape()

    def call(alpha=FAKE, ws=FAKE * 2):
        return lib.gdr_gated_linear_attn(ctypes.byref(sh), P(FAKE), P(FAKE + 4096), P(FAKE + 8192),
                                         P(alpha), None, P(FAKE), P(FAKE + 65536), None, P(ws),
                                         8, None)
    assert call(alpha=None) == INV
    assert call() == INV  # workspace too small (8 bytes): alpha present, beta not needed


def test_output_gate_needs_g(lib):
    """gdr_prefill_output_gate without its gate tensor is an argument error (no launch)."""
    sh = _shape(n_seqs=1, total_tokens=64)
    assert lib.gdr_prefill_output_gate(ctypes.byref(sh), *([None] * 11), 0, None) == 1


def test_layer_prologue_flag(lib):
    """GDR_FLAG_LAYER_PROLOGUE passes the shape checks of the rule's entry points (their other
    argument errors still come first) and is unsupported for plain linear attention; unknown
    flag bits stay argument errors."""
    from gated_delta_rule_prefill_gb300._abi import GDR_FLAG_LAYER_PROLOGUE
    P = ctypes.c_void_p
    sh = _shape(n_seqs=1, total_tokens=64)
    sh.flags = GDR_FLAG_LAYER_PROLOGUE
    assert lib.gdr_linear_attn(ctypes.byref(sh), P(FAKE), P(FAKE + 4096), P(FAKE + 8192), None,
                               None, P(FAKE + 65536), None, P(FAKE * 2), 1 << 20, None) == 2
    # the prologue flag alone is no error: a missing beta still is
    assert lib.gdr_prefill(ctypes.byref(sh), P(FAKE), P(FAKE + 4096), P(FAKE + 8192),
                           P(FAKE + 16384), None, None, None, P(FAKE + 65536), None,
                           P(FAKE * 2), 1 << 20, None) == 1
    sh.flags = 16
    assert lib.gdr_decode_step(ctypes.byref(sh), *([None] * 7), None) == 1


def test_layer_prologue_argument_errors(lib):
    """gdr_layer_prologue: shape checks, required q/k tensors, gate inputs and outputs in pairs,
    alignment and output aliasing -- all rejected before any launch; T = 0 is a no-op."""
    P = ctypes.c_void_p
    sh = _shape(n_seqs=1, total_tokens=64)

    def call(xq=FAKE, xk=FAKE + 65536, a=None, b=None, q=FAKE + 131072, k=FAKE + 196608,
             alpha=None, beta=None, shape=sh):
        return lib.gdr_layer_prologue(ctypes.byref(shape), P(xq), P(xk), P(a), P(b), P(q), P(k),
                                      P(alpha), P(beta), None)
    assert call(xq=None) == 1
    assert call(k=None) == 1
    assert call(a=FAKE * 4) == 1              # a without alpha
    assert call(beta=FAKE * 4) == 1           # beta without b
    assert call(q=FAKE + 8) == 1              # misaligned
    assert call(q=FAKE + 65536) == 1          # q onto xk
    assert call(k=FAKE) == 1                  # k onto xq
    assert call(shape=_shape(n_seqs=1, total_tokens=64, d_k=96, d_v=96)) == 2
    assert call(xq=None, shape=_shape(n_seqs=1, total_tokens=0)) == 0


def test_normalized_linear_argument_errors(lib):
    """gdr_normalized_linear_attn: eps must be finite and >= 0, z_final must not be z0, the
    layer-prologue flag is unsupported -- rejected before any launch."""
    P = ctypes.c_void_p
    sh = _shape(n_seqs=1, total_tokens=64)

    def call(eps=0.0, z0=None, zf=None, shape=sh):
        return lib.gdr_normalized_linear_attn(ctypes.byref(shape), P(FAKE), P(FAKE + 4096),
                                              P(FAKE + 8192), eps, None, P(z0), None,
                                              P(FAKE + 65536), None, P(zf), P(FAKE * 2), 8, None)
    assert call(eps=-1.0) == 1
    assert call(eps=float("nan")) == 1
    assert call(eps=float("inf")) == 1
    assert call(z0=FAKE * 4, zf=FAKE * 4) == 1
    assert call() == 1  # workspace too small (8 bytes)
    from gated_delta_rule_prefill_gb300._abi import GDR_FLAG_LAYER_PROLOGUE
    sh2 = _shape(n_seqs=1, total_tokens=64)
    sh2.flags = GDR_FLAG_LAYER_PROLOGUE
    assert call(shape=sh2) == 2


def test_decode_variants_argument_errors(lib):
    """gdr_gated_linear_decode_step needs alpha; gdr_normalized_linear_decode_step needs z_inout
    (not aliasing S_inout), a finite eps >= 0 and no layer-prologue flag."""
    P = ctypes.c_void_p
    sh = _shape(n_seqs=4, H=2, total_tokens=4)
    a = [P(FAKE), P(FAKE + 4096), P(FAKE + 8192)]
    assert lib.gdr_gated_linear_decode_step(ctypes.byref(sh), *a, None, P(FAKE * 2),
                                            P(FAKE * 3), None) == 1
    sh_bad = _shape(n_seqs=4, H=2, total_tokens=5)
    assert lib.gdr_gated_linear_decode_step(ctypes.byref(sh_bad), *a, P(FAKE * 4), P(FAKE * 2),
                                            P(FAKE * 3), None) == 1

    def norm(eps=0.0, S=FAKE * 2, z=FAKE * 5, shape=sh):
        return lib.gdr_normalized_linear_decode_step(ctypes.byref(shape), *a, eps, P(S), P(z),
                                                     P(FAKE * 3), None)
    assert norm(z=None) == 1
    assert norm(z=FAKE * 2) == 1
    assert norm(eps=-1.0) == 1
    assert norm(eps=float("nan")) == 1
    from gated_delta_rule_prefill_gb300._abi import GDR_FLAG_LAYER_PROLOGUE
    sh2 = _shape(n_seqs=4, H=2, total_tokens=4)
    sh2.flags = GDR_FLAG_LAYER_PROLOGUE
    assert norm(shape=sh2) == 2


def test_query_device_status_without_a_device(lib):
    # the call synchronises the stream first; with no usable GPU that fails cleanly with
    # GDR_ERR_CUDA instead of touching device memory, and on a GPU it returns a status
    from gated_delta_rule_prefill_gb300 import _abi
    import torch
    rc = lib.gdr_query_device_status(None)
    if torch.cuda.is_available():
        assert rc in (_abi.GDR_OK, _abi.GDR_ERR_DEVICE_CHECK)
    else:
        assert rc == _abi.GDR_ERR_CUDA


def test_check_wait_timeout_argument_errors(lib):
    # rejected before any CUDA work: null or unaligned workspace, limit out of range
    P = ctypes.c_void_p
    INV = 1
    assert lib.gdr_check_wait_timeout(None, 1000, None) == INV
    assert lib.gdr_check_wait_timeout(P(FAKE * 2 + 16), 1000, None) == INV
    assert lib.gdr_check_wait_timeout(P(FAKE * 2), 0, None) == INV
    assert lib.gdr_check_wait_timeout(P(FAKE * 2), 10_000_000_001, None) == INV
