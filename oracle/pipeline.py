"""The five stages composed (oracle; test infrastructure only).

Stage order follows [P-V41] ("DeepSeek-V4.1 模型结构（5）：记忆，Engram")
§"哈希函数" -> §"一层只有一张表" -> §"196B 参数怎么存、怎么取" -> §"门控", and the
summary of [P-LMNT] ("Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理")
§小结: compress tokens -> rolling XOR hash of 2/3/4-grams -> prime buckets in
an FP8 table -> gate decides how much is injected.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

from . import dequant, gate, hashing, shortconv
from .layout import Layout


@dataclasses.dataclass
class LayerResult:
    rows: np.ndarray       # int64 [T][n_cols]
    mask: np.ndarray       # bool [T]
    hist: np.ndarray       # int64 [S][max_ngram-1]
    e: np.ndarray          # float64 [T][n_cols*256] (bf16 values)
    gate: np.ndarray       # float64 [T][hc]
    v: np.ndarray          # float64 [T][H] (unrounded)
    h_out: np.ndarray      # float64 [T][hc][H] (bf16 values)


def layer_forward(layout: Layout, layer: int, raw_ids, cu_seqlens, token_map, table_rows,
                  wkv, h, q_w, k_w, hist: Optional[np.ndarray] = None, eps: float = 1e-6,
                  clamp: float = 1e-6, score_scale=None, gather=dequant.gather_dequant) -> LayerResult:
    """Prefill of one Engram layer on packed sequences.

    wkv: float64 [n_cols*row_dim][(hc+1)H]; h: float64 [T][hc][H].  ``gather``
    turns row ids into e: the E4M3 + E8M0 rows by default, or
    dequant.gather_rows for a table of plain bf16 rows.
    """
    rows, mask, new_hist = hashing.hash_prefill(raw_ids, cu_seqlens, token_map, layout, layer, hist)
    e = gather(rows, table_rows)
    hc, H = h.shape[1], h.shape[2]
    kv = gate.project(e, wkv)
    k, v = gate.split_kv(kv, H, hc)
    g = gate.gate(h, k, q_w, k_w, mask, eps, clamp, score_scale)
    h_out = gate.residual(h, g, v, mask)
    return LayerResult(rows, mask, new_hist, e, g, v, h_out)


def layer_decode_step(layout: Layout, layer: int, raw_ids, slots, hist: np.ndarray, token_map, table_rows,
                      wkv, h, q_w, k_w, eps: float = 1e-6, clamp: float = 1e-6, score_scale=None) -> LayerResult:
    """One decode step of one Engram layer: entry b hashes raw_ids[b] against
    the carried history hist[slots[b]] (slot -1 = padding, masked), then the
    same gather, projection, gate and residual as prefill.  h: float64 [B][hc][H]."""
    rows, mask, new_hist = hashing.hash_step(raw_ids, slots, hist, token_map, layout, layer)
    e = dequant.gather_dequant(rows, table_rows)
    hc, H = h.shape[1], h.shape[2]
    kv = gate.project(e, wkv)
    k, v = gate.split_kv(kv, H, hc)
    g = gate.gate(h, k, q_w, k_w, mask, eps, clamp, score_scale)
    h_out = gate.residual(h, g, v, mask)
    return LayerResult(rows, mask, new_hist, e, g, v, h_out)


@dataclasses.dataclass
class ConvParams:
    """The short convolution of the original Engram layer ([P-DETAIL] §4.2)."""
    w: np.ndarray          # float64 [K][hc][H], w[k] multiplies the value k*dilation positions back
    gamma: np.ndarray      # float64 [hc][H] RMSNorm weight
    dilation: int
    eps: float = 1e-6


def layer_forward_conv(layout: Layout, layer: int, raw_ids, cu_seqlens, token_map, table_rows, wkv, h, q_w, k_w,
                       conv: ConvParams, hist: Optional[np.ndarray] = None, conv_state=None, eps: float = 1e-6,
                       clamp: float = 1e-6, score_scale=None):
    """Prefill of the original Engram layer: the gated value is refined by the
    short convolution and H <- bf16(H + V~ + SiLU(conv(RMSNorm(V~)))) at every
    position ([P-DETAIL] §4.2 and the pseudo code of §五).

    Returns (LayerResult with h_out of this variant, new conv state per sequence).
    """
    rows, mask, new_hist = hashing.hash_prefill(raw_ids, cu_seqlens, token_map, layout, layer, hist)
    e = dequant.gather_dequant(rows, table_rows)
    hc, H = h.shape[1], h.shape[2]
    k, v = gate.split_kv(gate.project(e, wkv), H, hc)
    g = gate.gate(h, k, q_w, k_w, mask, eps, clamp, score_scale)
    y, state = shortconv.short_conv(shortconv.gated_value(g, v), cu_seqlens, conv.w, conv.gamma, conv.dilation,
                                    conv.eps, conv_state)
    return LayerResult(rows, mask, new_hist, e, g, v, shortconv.conv_residual(h, y)), state
