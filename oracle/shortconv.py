"""Short causal convolution on the gated value (oracle; test infrastructure only).

The original Engram layer, before DeepSeek-V4.1 dropped it, refines the gated
value with a short depthwise causal convolution.

Sources:
  [P-DETAIL] §4.2 "Short convolution：补回一点局部连续性":
      Y = SiLU(Conv1D(RMSNorm(V~))) + V~, and the block's hidden state gets
      H <- H + Y.  The convolution is depthwise (one filter per channel) and
      causal, with kernel size 4 and dilation equal to the largest n-gram
      order (3), so position t combines positions t, t-3, t-6 and t-9.
      Zero-initialised filters leave Y = V~.
  [P-DETAIL] §五 (tensor pseudo code):
      refined = silu(depthwise_causal_conv(rmsnorm(gated)));
      hidden = hidden + gated + refined.
  [P-DETAIL] §9.5: incremental decode keeps the normalised values of the past
      (kernel-1)*dilation = 9 positions; chunked prefill carries the same state.
  [P-V41] §"V4.1 相对原版的两处改动": a depthwise causal convolution of
      kernel 4 over the gated value, per channel, along the sequence.
  [P-V41] §多模态细节: the gate is forced to 0 at image (DEAD) positions.

Readings:
  * With hc residual streams the gated value is per stream,
    V~^(m)_t = g^(m)_t * bf16(v_t), so RMSNorm (over the H channels of one
    stream and position, with a learned weight gamma^(m)) and the filters
    w[k][m][i] are per stream.  Weights shared by the streams are the special
    case of equal rows.
  * w[k] multiplies the normalised value k*dilation positions back (k = 0 is
    the current position).  The convolution has no bias (the pages list none;
    zero filters then give Y = V~ as [P-DETAIL] §4.2 states).
  * Before the start of a sequence the convolution reads zeros, or the carried
    state (the normalised values of the previous chunk's last positions).
  * RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gamma with the layer's eps; the
    normalised value of an all-zero row (a masked position) is 0.
  * A masked position has gate 0, so V~ = 0 there, and it still receives
    Y = SiLU(conv) from the earlier positions: the formula above applies to
    every position of the sequence.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from .dequant import bf16_round


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2 over the last axis) + eps) * gamma, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def silu(x: np.ndarray) -> np.ndarray:
    """x * sigmoid(x)."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def gated_value(g: np.ndarray, v: np.ndarray) -> np.ndarray:
    """V~^(m)_t = g^(m)_t * bf16(v_t): g [T][hc], v [T][H] -> [T][hc][H]."""
    return np.asarray(g, dtype=np.float64)[:, :, None] * bf16_round(v)[:, None, :]


def causal_conv(n: np.ndarray, w: np.ndarray, dilation: int, past: Optional[np.ndarray] = None) -> np.ndarray:
    """c_t = sum_k w[k] * n_{t - k*dilation} over one sequence.

    n [T][hc][H] normalised values; w [K][hc][H]; past [R][hc][H] holds the
    normalised values of the R = (K-1)*dilation positions before the sequence
    (oldest first), or None for zeros.
    """
    K = w.shape[0]
    R = (K - 1) * dilation
    T = n.shape[0]
    if past is None:
        past = np.zeros((R,) + n.shape[1:])
    full = np.concatenate([np.asarray(past, dtype=np.float64), n], axis=0)
    c = np.zeros(n.shape, dtype=np.float64)
    for t in range(T):
        for k in range(K):
            c[t] += w[k] * full[R + t - k * dilation]
    return c


def short_conv(gated: np.ndarray, cu_seqlens: Sequence[int], w: np.ndarray, gamma: np.ndarray, dilation: int,
               eps: float, state: Optional[List[Optional[np.ndarray]]] = None):
    """Y = SiLU(conv(RMSNorm(V~))) + V~ per sequence.

    gated [T][hc][H]; cu_seqlens [n_seqs+1]; state[s] = the previous R
    normalised values of sequence s (oldest first) or None.  Returns
    (Y [T][hc][H], new_state) where new_state[s] is the last R normalised
    values of the carried state followed by this chunk (oldest first).
    """
    gated = np.asarray(gated, dtype=np.float64)
    K = w.shape[0]
    R = (K - 1) * dilation
    n = rmsnorm(gated, gamma, eps)
    y = np.empty_like(gated)
    new_state = []
    for s in range(len(cu_seqlens) - 1):
        a, b = int(cu_seqlens[s]), int(cu_seqlens[s + 1])
        past = None if state is None else state[s]
        c = causal_conv(n[a:b], w, dilation, past)
        y[a:b] = silu(c) + gated[a:b]
        hist = np.zeros((R,) + gated.shape[1:]) if past is None else np.asarray(past, dtype=np.float64)
        new_state.append(np.concatenate([hist, n[a:b]], axis=0)[len(hist) + (b - a) - R:])
    return y, new_state


def conv_residual(h: np.ndarray, y: np.ndarray) -> np.ndarray:
    """H <- bf16(H + Y) at every position (fp64 sum, one rounding)."""
    return bf16_round(np.asarray(h, dtype=np.float64) + y)
