"""Helpers of the GPU parity tests: device uploads, oracle inputs, comparisons.

Inputs come from ``workloads`` (seeded, shared); expected values come only
from ``oracle``.  Nothing here computes the method.
"""
from __future__ import annotations

import functools

import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from oracle import layout as OL
from workloads import WORKLOADS, ROW_BYTES, token_map

DEV = torch.device("cuda:0")

# Tolerances fixed by the benchmark spec for floating point: gate absolute,
# residual relative (to the largest term of the sum, see residual_close).
GATE_ATOL = 2e-3
RESID_RTOL = 1e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    eg.lib()  # raises loudly when the library is missing


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def i64(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int64)).to(DEV)


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(DEV)


def bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(DEV).view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def status() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@functools.lru_cache(maxsize=None)
def setup(name: str):
    """(workload, token map, oracle layout, library layout) of a workload."""
    w = WORKLOADS[name]
    tm = token_map(w.v_raw, w.v, w.seed)
    pad = int(tm[0])
    lay_o = OL.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=pad)
    lay = eg.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=pad)
    return w, tm, lay_o, lay


def device_table(total_rows: int, seed: int) -> torch.Tensor:
    """Synthetic table filled on the device (exact size, no tail padding)."""
    t = torch.empty(total_rows * ROW_BYTES, dtype=torch.uint8, device=DEV)
    eg.engram_fill_synthetic_table(t, total_rows, seed)
    return t


def dot_error_bound(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Bound on the error of fp32-accumulated dot products a @ b (float64 inputs).

    For a K-term sum accumulated in floating point with unit roundoff u,
    |fl(sum) - sum| <= K u sum |terms| (Higham, "Accuracy and Stability of
    Numerical Algorithms", 2nd ed., section 3.1).  u = 2^-23 covers fp32
    accumulation that truncates instead of rounding.
    """
    K = a.shape[-1]
    return K * 2.0 ** -23 * (np.abs(a) @ np.abs(b))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits, fp32 exponent range)."""
    _, E = np.frexp(np.abs(x))
    return np.exp2(np.maximum(E - 1, -126) - 7.0)


def bf16_flip(v_ref: np.ndarray, v_err: np.ndarray) -> np.ndarray:
    """One bf16 ulp where the exact v lies within v_err of a bf16 rounding
    midpoint (a correct fp32 v may round to the other side there), else 0."""
    from oracle.dequant import bf16_round
    ulp = bf16_ulp(v_ref)
    to_midpoint = ulp / 2 - np.abs(v_ref - bf16_round(v_ref))
    return np.where(to_midpoint <= v_err, ulp, 0.0)


def residual_close(got: np.ndarray, ref: np.ndarray, h_in: np.ndarray, g_ref: np.ndarray,
                   v_ref: np.ndarray, v_err: np.ndarray, rtol: float = RESID_RTOL):
    """|got - ref| <= rtol * max(|ref|, |h_in|, |g v|) + g * (v_err + flip), elementwise.

    The first term is the stated relative tolerance, measured against the
    largest term of the sum h + g v (the sum can cancel).  The second is the
    projection's fp32 accumulation bound on v (dot_error_bound), which the
    relative term cannot cover where v itself cancels.  v is rounded to bf16
    before the add (a step function), so where the exact v lies within v_err
    of a bf16 rounding midpoint the device's bf16(v) may land one bf16 ulp
    away from the oracle's: flip is that ulp there and 0 elsewhere.
    Returns (ok, worst ratio of error to tolerance, strict-relative fail count).
    """
    gv = np.abs(g_ref[:, :, None] * v_ref[:, None, :])
    scale = np.maximum(np.maximum(np.abs(ref), np.abs(h_in)), gv)
    flip = bf16_flip(v_ref, v_err)
    tol = rtol * scale + np.abs(g_ref)[:, :, None] * (v_err + flip)[:, None, :] + 1e-30
    ratio = np.abs(got - ref) / tol
    strict = np.abs(got - ref) > rtol * np.abs(ref)
    ok = bool((ratio <= 1.0).all())
    if not ok:
        t, m, i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        worst = dict(t=int(t), m=int(m), i=int(i), got=float(got[t, m, i]), ref=float(ref[t, m, i]),
                     h=float(h_in[t, m, i]), g=float(g_ref[t, m]), v=float(v_ref[t, i]),
                     v_err=float(v_err[t, i]), tol=float(tol[t, m, i]), ratio=float(ratio[t, m, i]))
        return ok, worst, int(strict.sum())
    return ok, float(ratio.max()), int(strict.sum())
