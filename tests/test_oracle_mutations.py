"""Plant plausible mistakes in a copy of the C oracle and check the pins catch every one (CPU).

Each mutant is compiled from a modified copy of oracle/gdr_oracle.c into a temporary library and
swapped in for the real one while the pin tests of test_oracle_pins.py run against it.  A mutant
that passes every pin would mean the pins cannot tell that mistake from the method.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdr_oracle.c")

PIN_TESTS = [
    pins.test_interference_read_em02e,
    pins.test_delta_overwrite_em03d,
    pins.test_two_token_chunk_em04e,
    lambda: pins.test_decay_survival_em05d(True),
    lambda: pins.test_decay_survival_em05d(False),
    pins.test_hand_2x2_steps,
    pins.test_linear_attention_is_masked_qk_v,
    pins.test_gdn_matrix_form,
    pins.test_alpha_zero_resets_memory,
    pins.test_beta_zero_is_pure_decay,
    pins.test_read_back_after_write,
    pins.test_orthonormal_keys_store_last_value,
    pins.test_gated_linear_unit_gate_is_masked_qk_v,
    lambda: pins.test_gated_linear_survival_sum(True),
    lambda: pins.test_gated_linear_survival_sum(False),
    pins.test_gated_linear_zero_gate_resets,
]


def _block(src, start, end):
    i, j = src.index(start), src.index(end)
    return src[i:j]


def _swap_fade_and_read(src):
    fade = _block(src, "/* 1. fade", "/* 2. read")
    read = _block(src, "/* 2. read", "/* 3. write")
    return src.replace(fade + read, read + fade)


def _fade_after_write(src):
    fade = _block(src, "/* 1. fade", "/* 2. read")
    write_end = src.index("    }\n    /* 4. read-out")
    src2 = src[:write_end] + fade + src[write_end:]
    return src2.replace(fade, "", 1)


MUTANTS = {
    "gated linear: fade after the write": lambda s: s.replace(
        "Si[j] = ai * Si[j] + kt[i] * vt[j]", "Si[j] = ai * (Si[j] + kt[i] * vt[j])"),
    "gated linear: gate on the wrong channel": lambda s: s.replace(
        "J->alpha[((size_t)t * H + h) * dk + i]", "J->alpha[((size_t)t * H + h) * dk + (dk - 1 - i)]"),
    "gated linear: scalar gate ignored": lambda s: s.replace(
        ": J->alpha[(size_t)t * H + h];\n        double* Si", ": 1.0;\n        double* Si"),
    "read the unfaded state": _swap_fade_and_read,
    "erase before fade": _fade_after_write,
    "dropped beta": lambda s: s.replace("vhat[j] = bt * (vt[j] - vhat[j])",
                                        "vhat[j] = (vt[j] - vhat[j])"),
    "wrong sign of the correction": lambda s: s.replace("bt * (vt[j] - vhat[j])",
                                                        "bt * (vt[j] + vhat[j])"),
    "gate on the wrong channel": lambda s: s.replace("Si[j] *= at[i]", "Si[j] *= at[dk - 1 - i]"),
    "scalar gate ignored": lambda s: s.replace("S[e] *= at;", "S[e] *= 1.0;"),
    "read-out with the key": lambda s: s.replace("ot[j] += Si[j] * qt[i]",
                                                 "ot[j] += Si[j] * kt[i]"),
    "transposed key read": lambda s: s.replace("vhat[j] += Si[j] * kt[i]",
                                               "vhat[j] += Si[j] * kt[j % dk]"),
    "transposed linear write": lambda s: s.replace("Si[j] += kt[i] * vt[j]",
                                                   "Si[j] += kt[j % dk] * vt[i % dv]"),
    "output before the write": lambda s: s.replace(
        "    /* 4. read-out", "    /* 4. read-out").replace(
        "if (J->mode == ORACLE_LINEAR) {\n      /* S <- S + k v^T */",
        "for (int j = 0; j < dv; ++j) ot[j] = 0.0;\n    for (int i = 0; i < dk; ++i)"
        " for (int j = 0; j < dv; ++j) ot[j] += S[(size_t)i * dv + j] * qt[i];\n"
        "    if (J->mode == ORACLE_LINEAR) {\n      /* S <- S + k v^T */").replace(
        "    /* 4. read-out of the updated state: o = S^T q */\n"
        "    for (int j = 0; j < dv; ++j) ot[j] = 0.0;",
        "    /* 4. (mutant: output already read) */\n    if (0)"),
}


@pytest.fixture(scope="module")
def original_source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, original_source, tmp_path):
    src = MUTANTS[name](original_source)
    assert src != original_source, "mutation did not apply"
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(src)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           str(so), str(c)])
    real = oracle._load()
    lib = ctypes.CDLL(str(so))
    lib.gdr_oracle_run.argtypes = real.gdr_oracle_run.argtypes
    lib.gdr_oracle_run.restype = ctypes.c_int
    caught = []
    oracle._lib = lib
    try:
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                caught.append(getattr(t, "__name__", "lambda"))
    finally:
        oracle._lib = real
    assert caught, "no pin caught the mutant '%s'" % name


# ---- the numpy statement of normalised phi-linear attention: mutants of its source text
import inspect  # noqa: E402

import numpy as np  # noqa: E402

NL_PINS = [pins.test_phi_closed_forms, pins.test_normalized_linear_is_a_weighted_average,
           pins.test_normalized_linear_state_handoff_and_eps]
NL_MUTANTS = {
    "phi_without_plus_one": ("phi", "x + 1.0, np.exp", "x, np.exp"),
    "phi_threshold_sign": ("phi", "np.where(x > 0", "np.where(x < 0"),
    "read_before_key_sum": ("normalized_linear",
                            "                z += k[t, h]\n                out[t, h] = (q[t, h] @ S) / (q[t, h] @ z + eps)",
                            "                out[t, h] = (q[t, h] @ S) / (q[t, h] @ z + eps)\n                z += k[t, h]"),
    "eps_in_numerator": ("normalized_linear", "(q[t, h] @ S) / (q[t, h] @ z + eps)",
                         "(q[t, h] @ S + eps) / (q[t, h] @ z + eps)"),
    "outer_product_transposed": ("normalized_linear", "np.outer(k[t, h], v[t, h])",
                                 "np.outer(k[t, h], v[t, h][::-1])"),
    "query_without_phi": ("normalized_linear", "q, k, v = phi(q), phi(k)", "q, k, v = q, phi(k)"),
}


@pytest.mark.parametrize("name", sorted(NL_MUTANTS))
def test_pins_catch_normalized_linear_mutant(name, monkeypatch):
    fn, old, new = NL_MUTANTS[name]
    src = inspect.getsource(getattr(oracle, fn))
    assert old in src, name
    ns = {"np": np, "phi": oracle.phi}
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(oracle, fn, ns[fn])
    caught = 0
    for pin in NL_PINS:
        try:
            with np.errstate(all="ignore"):  # a mutant may divide by a zero normaliser
                pin()
        except AssertionError:
            caught += 1
    assert caught > 0, "no pin catches mutant %s" % name
