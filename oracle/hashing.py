"""Token map, suffix windows and multiplicative-XOR hash (oracle; test infrastructure only).

Sources:
  [P-V41] §"tokenizer 压缩": x'_t = P(x_t); n-grams are taken over
      compressed ids, g_{t,n} = (x'_{t-n+1}, ..., x'_t).
  [P-V41] §"哈希函数", eq. (H): mix_{t,n} = XOR_{i=0}^{n-1} (x'_{t-i} * m_i),
      z_{t,n,k} = mix_{t,n} mod p_{n,k}; the lookback at distance i uses m_i;
      the mix of order n+1 is the mix of order n XOR x'_{t-n} * m_n; the 8
      heads of one order share one mix; a short sequence start is padded
      with the pad id (the first token's 2-gram is (current token, pad)).
  [P-V41] §"一层只有一张表" and [P-DS4] §布局与哈希探测 step 3:
      row = mix mod p + offset of the column's segment.
  [P-DETAIL] §3.2: suffix windows are left-padded with the compressed pad id.
  [P-V41] §"V4.1 相对原版的两处改动" (image tokens) and [P-LMNT] §多模态细节:
      an image position is DEAD (-1); looking back, the first DEAD slot and
      every slot farther back are treated as pad; the gate is 0 at an image
      position itself.  [P-DS4] §布局与哈希探测 step 4: masked positions
      write nothing to the residual.
  [P-LMNT] §第二步 and [P-DS4] §布局与哈希探测 (last paragraph): prefill and
      decode share one history; the hash state is the last 3 ids, a copy of
      it is a snapshot.
  [P-O1] §4.4: decode hashing is fused with the history commit; padding
      rows must not pollute the history.

Readings:
  * The window at a DEAD position is all pad (the first DEAD slot is slot 0);
    its row ids are still produced, and the position is masked.
  * History holds compressed ids, most recent first, with DEAD kept as -1.
    A fresh sequence has the history (pad, pad, pad), which is the same as
    left padding.
  * A raw id outside [0, V_raw) other than -1 is an error.
  * A decode entry with slot -1 (a padding row) is hashed with an all-pad
    history, is masked, and commits nothing.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

from .layout import Layout

DEAD = -1


def compress(raw_ids: np.ndarray, token_map: np.ndarray) -> np.ndarray:
    """x' = P(x) as int64; DEAD (-1) stays DEAD.  Raises on other out-of-range ids."""
    x = np.asarray(raw_ids, dtype=np.int64)
    dead = x == DEAD
    bad = ~dead & ((x < 0) | (x >= len(token_map)))
    if bad.any():
        raise ValueError(f"raw token id out of range at {np.flatnonzero(bad)[:8]}")
    out = np.asarray(token_map, dtype=np.int64)[np.where(dead, 0, x)]
    out[dead] = DEAD
    return out


def seq_index(cu_seqlens: np.ndarray) -> np.ndarray:
    """Sequence number of every packed position."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return np.repeat(np.arange(len(cu) - 1), np.diff(cu))


def windows(xc: np.ndarray, cu_seqlens: np.ndarray, hist: Optional[np.ndarray], pad_id: int,
            max_ngram: int) -> Tuple[np.ndarray, np.ndarray]:
    """Window slots g[t][i] = x'_{t-i}, i < max_ngram, after pad and DEAD handling.

    Slots before the sequence start come from the carried history
    ``hist[s][i - 1 - (t - start)]`` (most recent first) or, without history,
    are the pad id.  From the first DEAD slot on, every slot is the pad id.
    Returns (g int64 [T][max_ngram], mask bool [T]) with mask = position is DEAD.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    T = len(xc)
    s = seq_index(cu)
    t = np.arange(T, dtype=np.int64)
    start = cu[:-1][s]
    g = np.empty((T, max_ngram), dtype=np.int64)
    for i in range(max_ngram):
        src = t - i
        inside = src >= start
        val = np.full(T, pad_id, dtype=np.int64)
        val[inside] = xc[src[inside]]
        if hist is not None and i > 0:
            hidx = i - 1 - (t - start)
            use = ~inside
            val[use] = np.asarray(hist, dtype=np.int64)[s[use], hidx[use]]
        g[:, i] = val
    # DEAD cascade: the first DEAD slot and all farther slots become pad
    seen_dead = np.zeros(T, dtype=bool)
    for i in range(max_ngram):
        seen_dead |= g[:, i] == DEAD
        g[seen_dead, i] = pad_id
    mask = np.asarray(xc) == DEAD
    return g, mask


def mixes(g: np.ndarray, mults) -> np.ndarray:
    """mix[t][n-2] = XOR_{i<n} g[t][i] * m_i for n = 2..max_ngram, uint64, eq. (H)."""
    T, max_ngram = g.shape
    gu = g.astype(np.uint64)
    out = np.zeros((T, max_ngram - 1), dtype=np.uint64)
    acc = gu[:, 0] * np.uint64(mults[0])
    for n in range(2, max_ngram + 1):
        acc = acc ^ (gu[:, n - 1] * np.uint64(mults[n - 1]))
        out[:, n - 2] = acc
    return out


def row_ids(mix: np.ndarray, layout: Layout, layer: int) -> np.ndarray:
    """row[t][j] = mix[t][n(j)-2] mod p_j + offset_j, int64 [T][n_cols]."""
    L = layout.layers[layer]
    T = mix.shape[0]
    out = np.empty((T, layout.n_cols), dtype=np.int64)
    for j in range(layout.n_cols):
        n = layout.column_order(j)
        out[:, j] = (mix[:, n - 2] % np.uint64(L.primes[j])).astype(np.int64) + L.offsets[j]
    return out


def commit_history(xc: np.ndarray, cu_seqlens: np.ndarray, hist: Optional[np.ndarray],
                   pad_id: int, depth: int) -> np.ndarray:
    """History after the chunk: the last ``depth`` compressed ids, most recent first."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    n = len(cu) - 1
    out = np.empty((n, depth), dtype=np.int64)
    for s in range(n):
        old = [pad_id] * depth if hist is None else [int(v) for v in hist[s]]
        # oldest first: h_{depth-1} .. h_0, then the chunk's ids
        ext = old[::-1] + [int(v) for v in xc[cu[s]:cu[s + 1]]]
        out[s] = ext[::-1][:depth]
    return out


def hash_prefill(raw_ids, cu_seqlens, token_map, layout: Layout, layer: int,
                 hist: Optional[np.ndarray] = None):
    """Stages 1-3 over packed sequences.

    Returns (rows int64 [T][n_cols], mask bool [T], new_hist int64 [S][max_ngram-1]).
    """
    xc = compress(raw_ids, token_map)
    g, mask = windows(xc, cu_seqlens, hist, layout.pad_id, layout.max_ngram)
    rows = row_ids(mixes(g, layout.layers[layer].multipliers), layout, layer)
    new_hist = commit_history(xc, cu_seqlens, hist, layout.pad_id, layout.max_ngram - 1)
    return rows, mask, new_hist


def hash_step(raw_ids, slots, hist: np.ndarray, token_map, layout: Layout, layer: int):
    """One decode step: one new raw id per batch entry, history in ``hist[slot]``.

    Returns (rows [B][n_cols], mask [B], new_hist) where new_hist is a copy of
    ``hist`` with every used slot rolled: (h0, h1, h2) <- (x', h0, h1).
    """
    raw_ids = np.asarray(raw_ids, dtype=np.int64)
    slots = np.asarray(slots, dtype=np.int64)
    used = slots[slots >= 0]
    if len(np.unique(used)) != len(used):
        raise ValueError("duplicate history slots in one decode step")
    xc = compress(raw_ids, token_map)
    depth = layout.max_ngram - 1
    B = len(raw_ids)
    hb = np.full((B, depth), layout.pad_id, dtype=np.int64)
    hb[slots >= 0] = np.asarray(hist, dtype=np.int64)[slots[slots >= 0]]
    # one-position "sequences" whose history is hb
    cu = np.arange(B + 1, dtype=np.int64)
    g, mask = windows(xc, cu, hb, layout.pad_id, layout.max_ngram)
    mask = mask | (slots < 0)
    rows = row_ids(mixes(g, layout.layers[layer].multipliers), layout, layer)
    new_hist = np.array(hist, dtype=np.int64, copy=True)
    for b in range(B):
        if slots[b] >= 0:
            new_hist[slots[b]] = [xc[b]] + list(hb[b][:depth - 1])
    return rows, mask, new_hist
