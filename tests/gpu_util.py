"""Helpers of the GPU parity tests: device uploads, oracle inputs, comparisons.

Inputs come from ``workloads`` (seeded, shared); expected values come only
from ``oracle``.  Nothing here computes the method.
"""
from __future__ import annotations

import dataclasses
import functools

import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from oracle import layout as OL
from workloads import WORKLOADS, ROW_BYTES, bf16_bits_to_f64, token_map

DEV = torch.device("cuda:0")

# Tolerances fixed by the benchmark spec for floating point: gate absolute,
# residual relative (to the largest term of the sum, see residual_close).
GATE_ATOL = 2e-3
RESID_RTOL = 1e-2
# Multiple of the typical fp32 accumulation error in dot_error_bound.
V_ERR_LAMBDA = 8.0


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


def dot_error_bound(a: np.ndarray, b: np.ndarray, lam: float = V_ERR_LAMBDA) -> np.ndarray:
    """High-probability bound on the error of fp32-accumulated dot products a @ b.

    lam * u * sqrt(K) * sqrt(sum_k (a_k b_k)^2), u = 2^-24, elementwise over
    the output (float64 inputs of exact bf16 values, K = a.shape[-1]).

    Model: every product of two bf16 values is exact in fp32, and each fp32
    addition adds an error delta_j |S_j| to the running sum S_j with
    independent, mean-zero delta_j, |delta_j| <= u (Higham and Mary, "A new
    approach to probabilistic rounding error analysis", SIAM J. Sci. Comput.
    41(5), 2019).  The total error sum_j delta_j S_j then spreads as
    u sqrt(sum_j S_j^2); with terms of independent sign E[S_j^2] <= sum_k
    (a_k b_k)^2, so the spread is at most u sqrt(K) ||a b||_2 whatever the
    order or blocking of the sum.  lam = 8 puts the bound far in the tail of
    that spread and still covers a truncating fp32 adder that errs by half an
    ulp on average at each of the K/16 steps of a 16-deep MMA.  The worst-case
    bound K u sum|a_k b_k| (Higham, "Accuracy and Stability of Numerical
    Algorithms", 2nd ed., section 3.1) is at least 2 sqrt(K) / lam (~20 at
    K = 6144) times larger, since sum|a_k b_k| >= ||a b||_2, and is not what a
    correct GEMM reaches.  The GPU tests check this
    bound against the device's own bf16(v): the two round apart only where
    the exact v lies within it of a bf16 midpoint (v_flips_explained).
    """
    K = a.shape[-1]
    return lam * 2.0 ** -24 * np.sqrt(K) * np.sqrt((a * a) @ (b * b))


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


@dataclasses.dataclass
class ResidualCheck:
    ok: bool
    worst: object        # ratio of error to allowed tolerance, or the worst element (a dict) when not ok
    stated_ratio: float  # max |got - ref| / (rtol * largest term) over all elements
    outside_ratio: float  # the same outside the flip and cancel sets (<= 1 whenever ok)
    strict: int          # elements beyond the bare stated tolerance (all inside flip or cancel)
    flip: int            # elements in the flip set (exact v within v_err of a bf16 midpoint)
    cancel: int          # elements in the cancellation set (g v_err above the stated tolerance)
    n: int


def residual_close(got: np.ndarray, ref: np.ndarray, h_in: np.ndarray, g_ref: np.ndarray,
                   v_ref: np.ndarray, v_err: np.ndarray, rtol: float = RESID_RTOL) -> ResidualCheck:
    """Residual h <- bf16(h + g bf16(v)) against the oracle at the stated tolerance.

    stated = rtol * max(|ref|, |h_in|, |g v|): 1e-2 relative to the largest
    term of the sum (h + g v can cancel).  Every element must meet it, except
    in two sets where a correct fp32 computation may not:

    * flip set: the exact v lies within v_err (dot_error_bound) of a bf16
      rounding midpoint, so a correctly accumulated fp32 v may round to the
      neighbouring bf16 value; the update then moves by g ulp(v), at most
      2^-7 of g|v|.  Allowed there: stated + g (v_err + ulp(v)).
    * cancel set: g v_err alone exceeds the stated tolerance (v nearly cancels
      and h is small), so the fp32 sum of v is not known to that precision.
      Allowed there: stated + g v_err.

    Outside both sets the check is the stated tolerance alone.  Returns a
    ResidualCheck with the counts of each set and of the elements beyond the
    bare stated tolerance (``strict``).
    """
    g = np.abs(g_ref)[:, :, None]
    gv = np.abs(g_ref[:, :, None] * v_ref[:, None, :])
    stated = rtol * np.maximum(np.maximum(np.abs(ref), np.abs(h_in)), gv) + 1e-30
    in_flip = np.broadcast_to(bf16_flip(v_ref, v_err)[:, None, :] > 0, stated.shape)
    in_cancel = g * v_err[:, None, :] > stated
    extra = g * (v_err + bf16_flip(v_ref, v_err))[:, None, :]
    tol = stated + np.where(in_flip | in_cancel, extra, 0.0)
    err = np.abs(got - ref)
    ratio = err / tol
    strict = err > stated
    ok = bool((ratio <= 1.0).all())
    worst: object = float(ratio.max()) if ratio.size else 0.0
    if not ok:
        t, m, i = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
        worst = dict(t=int(t), m=int(m), i=int(i), got=float(got[t, m, i]), ref=float(ref[t, m, i]),
                     h=float(h_in[t, m, i]), g=float(g_ref[t, m]), v=float(v_ref[t, i]),
                     v_err=float(v_err[t, i]), tol=float(tol[t, m, i]), ratio=float(ratio[t, m, i]),
                     flip=bool(in_flip[t, m, i]), cancel=bool(in_cancel[t, m, i]))
    outside = ~(in_flip | in_cancel)
    r_stated = err / stated
    return ResidualCheck(ok, worst, float(r_stated.max()) if err.size else 0.0,
                         float(r_stated[outside].max()) if outside.any() else 0.0, int(strict.sum()),
                         int(in_flip.sum()), int(in_cancel.sum()), int(err.size))


def v_flips_explained(v_dev_bits: np.ndarray, v_ref: np.ndarray, v_err: np.ndarray) -> int:
    """Check the device's bf16(v) against the oracle's exact v.

    Where the exact v is farther than v_err from every bf16 rounding midpoint
    the device must round to the same bf16 value as the oracle, bit for bit;
    inside that band it may land one bf16 step away (more where v_err exceeds
    an ulp of v, i.e. where v cancels).  This tests v_err
    (dot_error_bound) against the device's own accumulation.  Returns the
    number of elements that rounded the other way (all inside the band).
    """
    from oracle.dequant import bf16_bits, bf16_round
    vr = bf16_bits(bf16_round(v_ref))
    vd = np.asarray(v_dev_bits, dtype=np.uint16)
    differ = vd != vr
    band = bf16_flip(v_ref, v_err) > 0
    assert not (differ & ~band).any(), f"{int((differ & ~band).sum())} bf16(v) differ outside the flip band"
    # |bf16(v_dev) - bf16(v)| <= |v_dev - v| + half an ulp on each side: one
    # bf16 step where v_err is below an ulp, more where v cancels
    step = np.abs(bf16_bits_to_f64(vd) - bf16_bits_to_f64(vr))
    limit = v_err + bf16_ulp(np.abs(v_ref) + v_err)
    assert (step[differ] <= limit[differ] * 1.0000001).all(), "bf16(v) differs by more than v_err + one step"
    return int(differ.sum())
