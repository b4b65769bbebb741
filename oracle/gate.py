"""wkv projection, context gate and gated residual add (oracle; test infrastructure only).

Sources:
  [P-V41] §"门控：用当前的上下文决定查到的向量用多少": one linear map turns
      the 6144-dim lookup vector e_t into four 5120-dim keys k^(1..4) and one
      value v; for each of the 4 mHC residual streams m,
      s = RMSNorm(h^(m)) . RMSNorm(k^(m)) / sqrt(d), the gate is a scalar in
      (0, 1), and h^(m) <- h^(m) + gate * v (the same v for all streams).
  [P-V41] §"sigmoid 之前多一步带符号的平方根": the released code computes the
      dot of h * weight * key, multiplies by the two RMS reciprocals and by
      dim^-0.5, and applies sigmoid(copysign(sqrt(max(|dot|, clamp)), dot)).
  [P-V41] §"每条流一个 key 的设计沿用自原版": the projections are one
      [6144, 25600] matrix wkv, one matmul.
  [P-DS4] §消费：学习投影 + 余弦门控: dot = sum_i h_i (q_w_i k_w_i) k_i with
      per-stream elementwise learned scales q_w, k_w (fp32 [5120, 4]);
      dot *= rsqrt(mean(h^2)+eps) rsqrt(mean(k^2)+eps) * (scale);
      h <- bf16(h + gate * bf16(v)); masked positions return without writing.
  [P-O1] §2.3: the gate kernel runs entirely in FP32 (this oracle uses fp64).

Readings:
  * The pages disagree on the final scale of the score: [P-V41] divides by
    sqrt(d) (its code line and its derivation s = sqrt(d) cos(theta), range
    +-71.6 at d = 5120), [P-DS4] writes a factor sqrt(width).  The oracle takes
    the score scale as a parameter and uses d^-0.5 (d = hidden width) by
    default, as [P-V41]'s derivation pins the scale.
  * eps = 1e-6 and clamp = 1e-6 (not printed on the pages).
  * wkv columns are [k^(1) | k^(2) | k^(3) | k^(4) | v], each H wide, and
    kv = e @ wkv with wkv stored [6144, 5H] (keys first, as listed on [P-V41]).
  * Only v is rounded to bf16 before the residual add; keys stay unrounded.
"""
from __future__ import annotations

import numpy as np

from .dequant import bf16_round


def project(e: np.ndarray, wkv: np.ndarray) -> np.ndarray:
    """kv = e @ wkv in float64 (a library GEMM of exact bf16 values)."""
    return np.asarray(e, dtype=np.float64) @ np.asarray(wkv, dtype=np.float64)


def split_kv(kv: np.ndarray, hidden: int, hc: int):
    """k [T][hc][H] and v [T][H] from kv [T][(hc+1)H]."""
    T = kv.shape[0]
    k = kv[:, : hc * hidden].reshape(T, hc, hidden)
    v = kv[:, hc * hidden: (hc + 1) * hidden]
    return k, v


def gate(h: np.ndarray, k: np.ndarray, q_w: np.ndarray, k_w: np.ndarray, mask: np.ndarray,
         eps: float = 1e-6, clamp: float = 1e-6, score_scale=None) -> np.ndarray:
    """Gate g[t][m] in (0, 1); 0 at masked positions.

    h, k: float64 [T][hc][H]; q_w, k_w: [H][hc].
    """
    h = np.asarray(h, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    H = h.shape[2]
    if score_scale is None:
        score_scale = H ** -0.5
    w = (np.asarray(q_w, dtype=np.float64) * np.asarray(k_w, dtype=np.float64)).T  # [hc][H]
    dot = np.einsum("tmi,mi,tmi->tm", h, w, k)
    rstd_h = 1.0 / np.sqrt(np.mean(h * h, axis=2) + eps)
    rstd_k = 1.0 / np.sqrt(np.mean(k * k, axis=2) + eps)
    s = dot * rstd_h * rstd_k * score_scale
    z = np.copysign(np.sqrt(np.maximum(np.abs(s), clamp)), s)
    g = 1.0 / (1.0 + np.exp(-z))
    return np.where(np.asarray(mask, dtype=bool)[:, None], 0.0, g)


def residual(h: np.ndarray, g: np.ndarray, v: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """h' = bf16(h + g * bf16(v)) per stream; masked positions keep h bit for bit.

    h: float64 [T][hc][H] of bf16 values; v: float64 [T][H] (unrounded).
    """
    vb = bf16_round(v)
    out = bf16_round(np.asarray(h, dtype=np.float64) + g[:, :, None] * vb[:, None, :])
    m = np.asarray(mask, dtype=bool)
    out[m] = h[m]
    return out
