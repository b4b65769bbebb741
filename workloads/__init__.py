"""Seeded synthetic inputs for the Engram lookup layer.

This module is the only code shared by the CPU oracle (``oracle/``) and the
CUDA path (``hashed_gram_conditional_gb300``).  It draws random inputs and
holds the five workload definitions; it contains none of the method's
arithmetic (no token mapping, hashing, modulo, dequantisation, projection,
gate or residual).

Pages cited (by title):
  [P-V41]    "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
  [P-LMNT]   "Engram条件记忆：DeepSeek-V4.1-Flash中196B稀疏参数N-gram哈希查表的实现原理"
  [P-DS4]    "ds4.c 学习笔记" — glossary entry "Engram"
  [P-DETAIL] "DeepSeek Engram 详解：把静态知识从计算里拆出来"

Generators
----------
* token map: a seeded surjection from the raw vocabulary onto the compressed
  one.  The real map comes from text normalisation of a tokenizer vocabulary
  ([P-V41] §"tokenizer 压缩"), which is not available, so a random
  surjection with the same sizes (129280 -> 99092) stands in for it.
* Zipf(1.1) token streams over raw ids (truncated to the vocabulary).
* image (DEAD) spans: contiguous runs of raw id -1 ([P-LMNT] §多模态细节).
* table rows: 264-byte rows (256 E4M3 bytes + 8 E8M0 bytes, [P-DS4]
  §布局与哈希探测) drawn from a counter-based SplitMix64 stream, so any row
  can be produced on demand without holding a 101 GB table on the host.
  The CUDA library fills device tables with its own implementation of the
  same published generator (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014).
* dense tensors (wkv, residual h, q_w, k_w) as bf16 bit patterns / fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

DEAD = -1          # raw / compressed id of an image position ([P-LMNT] §多模态细节)
ROW_BYTES = 264    # 256 E4M3 weights + 8 E8M0 scales ([P-DS4] §布局与哈希探测)
HEAD_DIM = 256
WORDS_PER_ROW = ROW_BYTES // 8  # 33 little-endian 64-bit words per row

# ---------------------------------------------------------------------------
# Workload definitions
# ---------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    v_raw: int            # raw tokenizer vocabulary
    v: int                # compressed vocabulary
    base_rows: int        # prime search starts strictly above this value
    layer_id: int         # Engram layer id (seeds the multipliers)
    n_seqs: int
    seq_len: int          # tokens per sequence (prefill) / max prefix (decode)
    hidden: int           # H (0 = no projection stage in this workload)
    hc: int               # hyper-connection streams
    dead_frac: float      # fraction of positions inside image spans
    chunks: int = 1       # prefill chunks (history carried between them)
    decode_steps: int = 0
    seed: int = 0

    @property
    def tokens(self) -> int:
        return self.n_seqs * self.seq_len


WORKLOADS = {
    # raw 1300 -> 1000; 24 primes above 4099; T=128; hidden 256, hc 4
    "tiny": Workload("tiny", 1300, 1000, 4099, 1, 1, 128, 256, 4, 0.0),
    # hash+gather microbench: 1 x 65536 tokens, table from base 2,000,000
    "microbench": Workload("microbench", 129280, 99092, 2_000_000, 1, 1, 65536, 0, 4, 0.0),
    # full layer prefill: 4 x 4096 tokens, 5% DEAD spans, hidden 5120
    "prefill": Workload("prefill", 129280, 99092, 2_000_000, 1, 4, 4096, 5120, 4, 0.05),
    # decode: 256 sequences, prefix lengths U[0, 8192], 1000 one-token steps
    "decode": Workload("decode", 129280, 99092, 2_000_000, 1, 256, 8192, 5120, 4, 0.0,
                       decode_steps=1000),
    # profiling case: 4 x 1024 tokens over a 4.8M-row (1.27 GB) table, hidden 5120;
    # small enough for multi-pass counter captures, every input still larger than L2
    "profile": Workload("profile", 129280, 99092, 200_000, 1, 4, 1024, 5120, 4, 0.05),
    # full scale: primes above 16,000,000 (384,006,168 rows), 131072 tokens in 8 chunks
    "fullscale": Workload("fullscale", 129280, 99092, 16_000_000, 1, 1, 131072, 5120, 4, 0.0,
                          chunks=8),
}


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """Independent numpy Generator for (seed, stream...)."""
    return np.random.default_rng([seed, *stream])


# ---------------------------------------------------------------------------
# Token-level inputs
# ---------------------------------------------------------------------------


def token_map(v_raw: int, v: int, seed: int = 0) -> np.ndarray:
    """Seeded surjection raw id -> compressed id, int32 [v_raw].

    The first ``v`` slots are a permutation of [0, v) (so every compressed id
    is hit), the remaining ``v_raw - v`` slots are uniform compressed ids, and
    the raw axis is then shuffled.
    """
    if not (0 < v <= v_raw):
        raise ValueError("need 0 < v <= v_raw")
    g = rng_for(seed, 1)
    base = np.concatenate([g.permutation(v), g.integers(0, v, v_raw - v)])
    return base[g.permutation(v_raw)].astype(np.int32)


def zipf_tokens(v_raw: int, n: int, s: float = 1.1, seed: int = 0, stream: int = 2) -> np.ndarray:
    """n raw ids from a truncated Zipf(s) law over ranks 1..v_raw, int32.

    P(rank r) is proportional to r**-s; ranks map to raw ids through a seeded
    permutation so that frequent tokens are scattered over the vocabulary.
    """
    g = rng_for(seed, stream)
    ranks = np.arange(1, v_raw + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    rank_to_id = g.permutation(v_raw)
    idx = g.choice(v_raw, size=n, p=p)
    return rank_to_id[idx].astype(np.int32)


def add_dead_spans(ids: np.ndarray, frac: float, span=(32, 256), seed: int = 0,
                   stream: int = 3) -> np.ndarray:
    """Overwrite about ``frac`` of a sequence with non-overlapping runs of DEAD.

    Span lengths are uniform in [span[0], span[1]]; positions are uniform
    among non-overlapping placements.  Returns a new array.
    """
    out = ids.copy()
    n = len(out)
    if frac <= 0 or n == 0:
        return out
    g = rng_for(seed, stream)
    target = int(round(frac * n))
    lens = []
    while sum(lens) < target:
        lens.append(int(g.integers(span[0], span[1] + 1)))
    lens[-1] -= sum(lens) - target
    lens = [length for length in lens if length > 0]
    free = n - sum(lens)
    if free < 0:
        raise ValueError("sequence too short for the requested DEAD fraction")
    # choose k gap sizes summing to at most `free` (stars and bars)
    k = len(lens)
    cuts = np.sort(g.integers(0, free + 1, size=k))
    pos = 0
    prev = 0
    for length, c in zip(lens, cuts):
        pos += int(c - prev)
        prev = int(c)
        out[pos:pos + length] = DEAD
        pos += length
    return out


@dataclasses.dataclass
class PrefillBatch:
    raw_ids: np.ndarray      # int32 [T] packed sequences
    cu_seqlens: np.ndarray   # int64 [n_seqs + 1]


def prefill_batch(w: Workload, seed: Optional[int] = None) -> PrefillBatch:
    """Packed sequences of ``w.seq_len`` Zipf tokens with DEAD spans."""
    seed = w.seed if seed is None else seed
    seqs = []
    for s in range(w.n_seqs):
        ids = zipf_tokens(w.v_raw, w.seq_len, seed=seed, stream=100 + s)
        ids = add_dead_spans(ids, w.dead_frac, seed=seed, stream=10_000 + s)
        seqs.append(ids)
    raw = np.concatenate(seqs).astype(np.int32) if seqs else np.zeros(0, np.int32)
    cu = np.zeros(w.n_seqs + 1, np.int64)
    cu[1:] = np.cumsum([len(x) for x in seqs])
    return PrefillBatch(raw, cu)


@dataclasses.dataclass
class DecodeWorkload:
    prefix: PrefillBatch         # per-sequence prefixes (history source)
    steps: np.ndarray            # int32 [n_steps][n_seqs] one new raw id per sequence


def decode_workload(w: Workload, n_steps: Optional[int] = None, seed: Optional[int] = None) -> DecodeWorkload:
    """Prefix lengths U[0, seq_len] (sequences 0, 1, 2 forced to 0, 1, 2)."""
    seed = w.seed if seed is None else seed
    n_steps = w.decode_steps if n_steps is None else n_steps
    g = rng_for(seed, 4)
    lens = g.integers(0, w.seq_len + 1, size=w.n_seqs)
    lens[: min(3, w.n_seqs)] = np.arange(min(3, w.n_seqs))
    total = int(lens.sum())
    flat = zipf_tokens(w.v_raw, total, seed=seed, stream=5)
    cu = np.zeros(w.n_seqs + 1, np.int64)
    cu[1:] = np.cumsum(lens)
    steps = zipf_tokens(w.v_raw, n_steps * w.n_seqs, seed=seed, stream=6).reshape(n_steps, w.n_seqs)
    return DecodeWorkload(PrefillBatch(flat, cu), steps)


# ---------------------------------------------------------------------------
# Table rows: counter-based SplitMix64
# ---------------------------------------------------------------------------

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def splitmix64_at(seed: int, counter: np.ndarray) -> np.ndarray:
    """Output number ``counter + 1`` of a SplitMix64 stream whose state starts at ``seed``.

    SplitMix64 advances its state by the golden-gamma constant and returns the
    state passed through a two-multiply xor-shift finaliser, so the n-th output
    depends only on seed + n * gamma.  uint64 arithmetic wraps modulo 2**64.
    """
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (counter.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def table_rows(seed: int, rows: np.ndarray) -> np.ndarray:
    """Bytes of the requested table rows, uint8 [len(rows)][264].

    Row r is the little-endian bytes of words splitmix64_at(seed, 33*r + j),
    j = 0..32.  Weight bytes equal to an E4M3 NaN code (0x7F, 0xFF) are
    replaced by byte ^ 1; each scale byte b becomes 120 + (b mod 11), so scales
    are uniform over [120, 130].
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    ctr = rows[:, None] * WORDS_PER_ROW + np.arange(WORDS_PER_ROW, dtype=np.int64)[None, :]
    words = splitmix64_at(seed, ctr)                                  # [n][33] uint64
    b = words.astype("<u8").view(np.uint8).reshape(len(rows), ROW_BYTES).copy()
    w = b[:, :256]
    nan = (w & 0x7F) == 0x7F
    w[nan] ^= 1
    b[:, 256:] = 120 + (b[:, 256:] % 11)
    return b


def table_bytes(seed: int, n_rows: int) -> np.ndarray:
    """A whole table on the host (small tables only)."""
    return table_rows(seed, np.arange(n_rows, dtype=np.int64))


# ---------------------------------------------------------------------------
# Dense tensors
# ---------------------------------------------------------------------------


def normal_bf16_bits(shape, std: float, seed: int, stream: int) -> np.ndarray:
    """N(0, std^2) samples stored as bf16 bit patterns (uint16).

    The fp32 sample is truncated to its upper 16 bits; the result is a valid
    bf16 sample of (almost) the same law.
    """
    g = rng_for(seed, stream)
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def uniform_f32(shape, lo: float, hi: float, seed: int, stream: int) -> np.ndarray:
    g = rng_for(seed, stream)
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (no rounding)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


@dataclasses.dataclass
class LayerWeights:
    wkv_bits: np.ndarray   # uint16 [24*256][(hc+1)*H] bf16 bits, kv = e @ wkv
    q_w: np.ndarray        # float32 [H][hc]
    k_w: np.ndarray        # float32 [H][hc]


def table_rows_bf16(seed: int, rows: np.ndarray, row_dim: int) -> np.ndarray:
    """bf16 bit patterns of the requested rows of a synthetic bf16-row table,
    uint16 [len(rows)][row_dim].

    Element c of row r is 16-bit piece (c mod 4) (little-endian) of
    splitmix64_at(seed, r*(row_dim/4) + c/4), with its 8 exponent bits
    (bits 7..14) replaced by 120 + (those bits mod 11): finite values of
    magnitude in [2^-7, 2^4).
    """
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    per = row_dim // 4
    ctr = rows[:, None] * per + np.arange(per, dtype=np.int64)[None, :]
    b = splitmix64_at(seed, ctr).astype("<u8").view("<u2").reshape(len(rows), row_dim).astype(np.uint32)
    ex = np.uint32(120) + ((b >> np.uint32(7)) & np.uint32(0xFF)) % np.uint32(11)
    return ((b & np.uint32(0x807F)) | (ex << np.uint32(7))).astype(np.uint16)


def layer_weights(w: Workload, n_cols: int = 24, seed: Optional[int] = None,
                  row_dim: int = HEAD_DIM) -> LayerWeights:
    seed = w.seed if seed is None else seed
    k = n_cols * row_dim
    n = (w.hc + 1) * w.hidden
    wkv = normal_bf16_bits((k, n), 0.02, seed, 20)
    q_w = uniform_f32((w.hidden, w.hc), 0.5, 1.5, seed, 21)
    k_w = uniform_f32((w.hidden, w.hc), 0.5, 1.5, seed, 22)
    return LayerWeights(wkv, q_w, k_w)


def conv_weights(kernel: int, hc: int, hidden: int, seed: int):
    """Short-convolution inputs: filters N(0, 0.5^2) f32 [kernel][hc][hidden] and
    RMSNorm weights U[0.5, 1.5] f32 [hc][hidden]."""
    w = (rng_for(seed, 40).standard_normal((kernel, hc, hidden)) * 0.5).astype(np.float32)
    return w, uniform_f32((hc, hidden), 0.5, 1.5, seed, 41)


def gate_values(tokens: int, hc: int, seed: int, masked: Optional[np.ndarray] = None) -> np.ndarray:
    """Gate values U[0.02, 0.98] f32 [tokens][hc], 0 at masked positions."""
    g = uniform_f32((tokens, hc), 0.02, 0.98, seed, 42)
    if masked is not None:
        g[np.asarray(masked, dtype=bool)] = 0.0
    return g


def mxfp8_weights(k: int, n: int, seed: int):
    """A wkv matrix in the block-FP8 checkpoint form: E4M3 codes uint8 [k][n]
    (uniform bytes, the NaN codes 0x7F / 0xFF replaced by byte ^ 1) and one
    E8M0 scale per 32 consecutive rows of each column, uint8 [k/32][n],
    uniform over [114, 118] (factors 2^-13 .. 2^-9)."""
    g = rng_for(seed, 50)
    w = g.integers(0, 256, size=(k, n), dtype=np.int64).astype(np.uint8)
    nan = (w & 0x7F) == 0x7F
    w[nan] ^= 1
    sf = (114 + rng_for(seed, 51).integers(0, 5, size=(k // 32, n))).astype(np.uint8)
    return w, sf


def residual_bits(tokens: int, hc: int, hidden: int, seed: int, stream: int = 30) -> np.ndarray:
    """Residual streams h, bf16 bits [T][hc][H], N(0, 1)."""
    return normal_bf16_bits((tokens, hc, hidden), 1.0, seed, stream)
