"""Helpers of the GPU parity tests: move generator inputs to the device, run the library through
the binding, run the oracle on the same numbers, and measure the error.

Error metrics (the tolerances are the ones stated for this method: a maximum relative error of
1e-4 for fp32 inputs, 2e-2 relative to the output row norm for bf16 inputs with an fp32 state):
  row-normwise, every dtype:
    outputs: max over (token, head) of ||o_gpu - o_ref||_2 / max(||o_ref||_2, floor)
    states:  max over (seq, head)  of ||S_gpu - S_ref||_F / max(||S_ref||_F, floor)
  with floor = 1e-3 x the RMS of the reference row (or state) norms, so that rows whose
  reference is nearly zero are judged against the typical magnitude instead of blowing up;
  element-wise, asserted wherever the bound is the fp32 one:
    max over elements of |x_gpu - x_ref| / max(|x_ref|, ELEM_FLOOR x RMS of the reference)
  A relative error has no meaning for elements near zero, so the element-wise metric needs a
  floor; ELEM_FLOOR = 0.1 holds every element of at least a tenth of the typical magnitude to
  1e-4 relative and every smaller one to 1e-5 x RMS absolute.  A smaller floor asks for more
  than fp32 arithmetic gives: the recurrence itself evaluated in fp32, token by token in the
  stated order, misses 1e-4 at a floor of 1e-3 x RMS on the fp32 workload
  (tests/test_parity_metric.py pins this).  The value at the 1e-3 floor is still printed.
  err_rows / err_states give the row-normwise error, and for the fp32 bound the larger of the
  two.
"""
import numpy as np
import torch

import gdr_inputs as gi

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_dev(x: np.ndarray, dtype: str, device="cuda"):
    if dtype == "bf16":
        bits = gi.bf16_bits(x)
        return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def dev_inputs(a: dict, dtype: str, device="cuda"):
    d = dict(q=to_dev(a["q"], dtype, device), k=to_dev(a["k"], dtype, device),
             v=to_dev(a["v"], dtype, device), alpha=to_dev(a["alpha"], "f32", device),
             beta=to_dev(a["beta"], "f32", device), S0=to_dev(a["S0"], "f32", device))
    d["cu_seqlens"] = torch.from_numpy(a["cu_seqlens"].astype(np.int32)).to(device)
    return d


def rel_rows(got: np.ndarray, ref: np.ndarray) -> float:
    """Largest row-normwise relative error over the leading axes (last axis = the row)."""
    got = got.reshape(-1, got.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1]).astype(np.float64)
    if ref.size == 0:
        return 0.0
    rn = np.linalg.norm(ref, axis=1)
    floor = max(1e-3 * np.sqrt(np.mean(rn ** 2)), 1e-30)
    return float(np.max(np.linalg.norm(got - ref, axis=1) / np.maximum(rn, floor)))


def rel_states(got: np.ndarray, ref: np.ndarray) -> float:
    d = got.shape[-1] * got.shape[-2]
    return rel_rows(got.reshape(-1, d), ref.reshape(-1, d))


ELEM_FLOOR = 0.1


def rel_elem(got: np.ndarray, ref: np.ndarray, floor_frac: float = ELEM_FLOOR) -> float:
    """Largest element-wise relative error, the denominator floored at floor_frac x the RMS of
    the reference's elements."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if ref.size == 0:
        return 0.0
    floor = max(floor_frac * np.sqrt(np.mean(ref ** 2)), 1e-30)
    return float(np.max(np.abs(got - ref) / np.maximum(np.abs(ref), floor)))


def _elem_report(got, ref):
    print("element-wise relative error: %.3g (floor 1e-3 x RMS), %.3g (floor %g x RMS)"
          % (rel_elem(got, ref, 1e-3), rel_elem(got, ref), ELEM_FLOOR))


def err_rows(got: np.ndarray, ref: np.ndarray, tol: float) -> float:
    """The error checked against `tol`: row-normwise, and element-wise too for the fp32 bound."""
    e = rel_rows(got, ref)
    if tol <= TOL["f32"]:
        _elem_report(got, ref)
    return max(e, rel_elem(got, ref)) if tol <= TOL["f32"] else e


def err_states(got: np.ndarray, ref: np.ndarray, tol: float) -> float:
    e = rel_states(got, ref)
    if tol <= TOL["f32"]:
        _elem_report(got, ref)
    return max(e, rel_elem(got, ref)) if tol <= TOL["f32"] else e


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()
