"""Row codec e4m3_e8m0_32_row264 and bf16 rounding (oracle; test infrastructure only).

Sources:
  [P-V41] §"196B 参数怎么存、怎么取": the table is FP8 (1 byte per
      parameter) with one quantisation scale per 32 dimensions, 8 per row,
      so each row dequantises on its own; 24 rows of 256 B + 8 B per token.
  [P-DS4] §布局与哈希探测 (DS4_ENGRAM_ROW_BYTES = 264) and §永不常驻的 I/O 设计:
      a row is 256 E4M3 weight bytes followed by 8 E8M0 block-scale bytes,
      one scale per 32 dimensions, the block-scaled family of MXFP4.
  [P-O1] §2.3: table payload fp8 e4m3 with e8m0 block scales; the lookup
      outputs bf16.
  [P-V41] §"门控" (e_t is the 6144-dim lookup result): the 24 rows are
      concatenated in column order.
  [P-O1] §2.3: the projection weights of the released model are block-FP8,
      and the table payload is E4M3 with E8M0 block scales.

Readings (weights):
  * Block-FP8 wkv is taken in the same E4M3 x E8M0-per-32 family as the
    rows, blocked along the contraction axis k (dequant_mx_weights); its
    values are exact in fp64, so the FP8 projection's oracle is the same fp64
    GEMM on these values.

Readings:
  * E4M3 is the OCP FP8 E4M3 format (bias 7, no infinities, 0x7F/0xFF are
    NaN, largest finite 448, subnormals M/8 * 2^-6), and E8M0 is the OCP
    scale format (value 2^(e-127), 0xFF is NaN) -- the variants used with
    32-element block scales.
  * value = E4M3(b) * 2^(e-127) is exact in fp64 and is rounded once to bf16,
    round-to-nearest-even, with gradual underflow and overflow to infinity;
    -0 is kept.
"""
from __future__ import annotations

import numpy as np

ROW_BYTES = 264
HEAD_DIM = 256
BLOCK = 32


def e4m3_value(code) -> np.ndarray:
    """Decode E4M3 codes to float64 by the closed form."""
    b = np.asarray(code, dtype=np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = sign * (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    subnormal = sign * (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, subnormal, normal)
    return np.where((e == 0xF) & ((b & 0x7) == 0x7), np.nan, v)


def e8m0_value(code) -> np.ndarray:
    """Decode E8M0 scale codes: 2^(e-127), NaN for 0xFF."""
    e = np.asarray(code, dtype=np.int64)
    return np.where(e == 0xFF, np.nan, np.exp2((e - 127).astype(np.float64)))


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even (as float64).

    A bf16 number has 8 significant bits and the fp32 exponent range, so the
    spacing of representable values near |x| is 2^(max(E, -126) - 7) where
    2^E <= |x| < 2^(E+1).  Dividing by that spacing is exact; numpy's
    ``round`` rounds halves to even.  Results beyond the largest finite bf16
    value become infinities; NaN stays NaN; zeros keep their sign.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x) & (x != 0)
    xf = x[fin]
    _, E = np.frexp(xf)                  # |x| = f * 2^E, f in [0.5, 1)
    lead = np.maximum(E - 1, -126)
    q = np.exp2((lead - 7).astype(np.float64))
    y = np.round(xf / q) * q
    y = np.where(np.abs(y) > BF16_MAX, np.copysign(np.inf, y), y)
    out[fin] = y
    return out


def bf16_bits(x) -> np.ndarray:
    """Bit patterns (uint16) of float64 values that are already bf16 values."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """uint8 [n][264] -> float64 [n][256] of bf16 values."""
    rows = np.asarray(rows, dtype=np.uint8)
    w = e4m3_value(rows[:, :HEAD_DIM])
    s = e8m0_value(rows[:, HEAD_DIM:HEAD_DIM + HEAD_DIM // BLOCK])
    return bf16_round(w * np.repeat(s, BLOCK, axis=1))


def dequant_mx_weights(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Block-FP8 weights to float64: w[k][n] = E4M3(codes[k][n]) * 2^(scales[k // 32][n] - 127),
    the same E4M3 x E8M0-per-32 family as the table rows, blocked along k (the
    contraction axis of kv = e @ wkv).  Exact; no rounding."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    return e4m3_value(codes) * e8m0_value(np.repeat(scales, BLOCK, axis=0))


def gather_dequant(row_ids: np.ndarray, table_rows) -> np.ndarray:
    """e[t] = concat_j dequant(row row_ids[t][j]), float64 [T][n_cols * 256].

    ``table_rows(ids)`` returns the bytes of the requested rows, uint8 [n][264].
    """
    rid = np.asarray(row_ids, dtype=np.int64)
    T, C = rid.shape
    vals = dequant_rows(table_rows(rid.reshape(-1)))
    return vals.reshape(T, C * HEAD_DIM)


def gather_rows(row_ids: np.ndarray, table_rows) -> np.ndarray:
    """e[t] = concat_j row(row_ids[t][j]) for a table of plain bf16 rows,
    float64 [T][n_cols * row_dim] ([P-DETAIL] §5: the per-head rows are
    concatenated in column order into the memory vector).

    ``table_rows(ids)`` returns the rows as float64 bf16 values [n][row_dim].
    """
    rid = np.asarray(row_ids, dtype=np.int64)
    T, C = rid.shape
    vals = np.asarray(table_rows(rid.reshape(-1)), dtype=np.float64)
    return vals.reshape(T, C * vals.shape[1])
