"""Error metrics and tolerances shared by the GPU parity tests.

Tolerances (stated for the hot path):
  O    max-abs error <= 1e-2, measured on top of the bf16 rounding of the
       output: |O_gpu - O_oracle| - ulp_bf16(O_oracle)/2 <= 1e-2.  O is
       returned in bf16, whose half-ulp is 2^-6 = 0.0156 for |O| in [4, 8), so a
       plain 1e-2 bound could not be met by any bf16 output there; the reading
       keeps 1e-2 as the bound on the computation itself.
  LSE  max-abs error <= 1e-3 (fp32 output).
  dQ, dK, dV  relative Frobenius error ||g - g_oracle|| / ||g_oracle|| <= 2e-2.

Row diagnostic.  A whole-tensor Frobenius norm can hide one wrong row (at
N = 8192 a fully wrong row adds about 1% to it), so the gradient tests also log
the worst row: max_r ||g_r - g_oracle_r|| / rms_r ||g_oracle_r|| (rows of dQ are
queries, rows of dK, dV are keys; the denominator is the root-mean-square row
norm, so rows whose exact gradient is near zero, such as the first causal
query's dQ, do not blow it up).  A row that is wrong as a whole scores about 1;
the tests require <= ROW_TOL.
"""
from __future__ import annotations

import json
import os

import numpy as np

O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_RTOL = 2e-2
ROW_TOL = 0.25


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    a = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def o_error(o_gpu, o_ref) -> float:
    """Max over elements of |o_gpu - o_ref| minus the bf16 half-ulp of o_ref."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    if o_gpu.size == 0:
        return 0.0
    return float(np.max(np.abs(o_gpu - o_ref) - half_ulp_bf16(o_ref)))


def max_abs(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    return float(np.max(np.where(both_inf, 0.0, np.abs(a - b))))


def rel_fro(g, g_ref) -> float:
    g = np.asarray(g, np.float64)
    g_ref = np.asarray(g_ref, np.float64)
    den = np.linalg.norm(g_ref)
    return float(np.linalg.norm(g - g_ref) / (den if den > 0 else 1.0))


def row_err(g, g_ref) -> float:
    """Worst row error relative to the RMS row norm of g_ref (rows = all axes but the last)."""
    g = np.asarray(g, np.float64)
    g_ref = np.asarray(g_ref, np.float64)
    if g_ref.size == 0:
        return 0.0
    d = g_ref.shape[-1]
    diff = np.linalg.norm((g - g_ref).reshape(-1, d), axis=1)
    rms = float(np.sqrt(np.mean(np.sum(g_ref.reshape(-1, d) ** 2, axis=1))))
    return float(diff.max() / (rms if rms > 0 else 1.0))


def to64(t) -> np.ndarray:
    """torch tensor (any device, any float dtype) -> numpy float64."""
    return t.detach().to("cpu").double().numpy()


def record(test: str, **metrics) -> None:
    """Append the measured errors of one parity check to $FA_PARITY_LOG (JSON lines)."""
    path = os.environ.get("FA_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, **{k: (float(v) if isinstance(v, (float, np.floating)) else v)
                                             for k, v in metrics.items()}}) + "\n")
