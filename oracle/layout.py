"""Layout of one physical Engram table per layer (oracle; test infrastructure only).

Sources:
  [P-V41] §"一层只有一张表": one physical table per layer; each of the 24
      (order, head) pairs owns a contiguous segment; the table's row count is
      the sum of 24 primes found by searching upward from
      ``engram_vocab_size`` (16,000,000), one prime per head, never reused;
      the printed table gives min/max/sum for layers 1 and 14.
  [P-O1] §2.2: primes are drawn in (layer, order, head) order from one
      ascending sequence; §2.2 and §"一层只有一张表": segment offsets are the
      cumulative sum of the primes.
  [P-V41] §"哈希函数" items under eq. (H): the multipliers m_0..m_3 are large
      odd numbers bounded so that any compressed id times a multiplier fits in
      a signed 64-bit integer, i.e. below (2^63-1)/V.
  [P-O1] §4.3 and [P-LMNT] §第二步: the multipliers are drawn per layer from a
      generator seeded with 10007 * layer_id, bounded by int64max // V // 2.

Readings (the pages leave these open):
  * "search upward for the next prime" is read as: primes strictly greater
    than the base (the printed table for base 16,000,000 cannot tell > from
    >=, since 16,000,000 is not prime).
  * The pages name numpy's PCG64 generator for the multipliers.  This layout
    uses a SplitMix64 stream seeded with 10007 * layer_id instead; r_i is the
    i-th output modulo half = ((2^63-1) // V) // 2 and m_i = 2 r_i + 1.  Real
    checkpoint multipliers can be supplied through ``multipliers_override``.
    Parity of the generated values against a real checkpoint is therefore
    unpinned; the tests pin the bound, oddness and library == oracle.
  * Primality here is decided by trial division, independent of the CUDA
    library's Miller-Rabin test.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

INT64_MAX = (1 << 63) - 1
MASK64 = (1 << 64) - 1


def is_prime(n: int) -> bool:
    """Trial division up to floor(sqrt(n))."""
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    d = 3
    while d * d <= n:
        if n % d == 0:
            return False
        d += 2
    return True


def primes_above(base: int, count: int) -> List[int]:
    """The ``count`` consecutive primes strictly greater than ``base``."""
    out = []
    c = base
    while len(out) < count:
        c += 1
        if is_prime(c):
            out.append(c)
    return out


def splitmix64(seed: int, count: int) -> List[int]:
    """First ``count`` outputs of SplitMix64 with initial state ``seed``.

    Steele, Lea & Flood (OOPSLA 2014): state += 0x9E3779B97F4A7C15, then the
    state goes through z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
    z *= 0x94D049BB133111EB; z ^= z >> 31 (all modulo 2^64).
    """
    s = seed & MASK64
    out = []
    for _ in range(count):
        s = (s + 0x9E3779B97F4A7C15) & MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        out.append(z ^ (z >> 31))
    return out


def multipliers(layer_id: int, vocab: int, max_ngram: int) -> List[int]:
    """Odd multipliers m_0..m_{max_ngram-1} for one layer (reading above)."""
    half = (INT64_MAX // vocab) // 2
    return [2 * (r % half) + 1 for r in splitmix64(10007 * layer_id, max_ngram)]


@dataclasses.dataclass
class LayerLayout:
    layer_id: int
    primes: List[int]        # column j = (n - 2) * n_heads + k
    offsets: List[int]       # exclusive cumulative sum of primes
    total_rows: int          # sum of primes
    multipliers: List[int]   # m_0 .. m_{max_ngram-1}


@dataclasses.dataclass
class Layout:
    vocab: int
    base_rows: int
    max_ngram: int
    n_heads: int
    pad_id: int
    layers: List[LayerLayout]

    @property
    def n_cols(self) -> int:
        return (self.max_ngram - 1) * self.n_heads

    def column_order(self, j: int) -> int:
        """n-gram order n of column j."""
        return 2 + j // self.n_heads


def build_layout(vocab: int, base_rows: int, layer_ids: Sequence[int], max_ngram: int = 4,
                 n_heads: int = 8, pad_id: int = 0, expected_vocab: Optional[int] = None,
                 multipliers_override: Optional[Sequence[Sequence[int]]] = None) -> Layout:
    """Primes, offsets and multipliers for every Engram layer.

    ``expected_vocab``: the inference code refuses to start when the
    compressed vocabulary differs from the checkpoint's ([P-V41] under
    eq. (H); [P-O1] §2.1), because every multiplier depends on it.
    """
    if expected_vocab is not None and expected_vocab != vocab:
        raise ValueError(f"compressed vocabulary {vocab} != expected {expected_vocab}")
    if not (0 <= pad_id < vocab):
        raise ValueError("pad id must be a compressed id")
    n_cols = (max_ngram - 1) * n_heads
    all_primes = primes_above(base_rows, n_cols * len(layer_ids))
    layers = []
    for li, layer_id in enumerate(layer_ids):
        ps = all_primes[li * n_cols:(li + 1) * n_cols]
        offs = []
        acc = 0
        for p in ps:
            offs.append(acc)
            acc += p
        if multipliers_override is not None:
            ms = [int(m) for m in multipliers_override[li]]
            for m in ms:
                if m <= 0 or m % 2 == 0 or (vocab - 1) * m > INT64_MAX:
                    raise ValueError("override multipliers must be odd and keep (V-1)*m in int64")
        else:
            ms = multipliers(layer_id, vocab, max_ngram)
        layers.append(LayerLayout(layer_id, ps, offs, acc, ms))
    return Layout(vocab, base_rows, max_ngram, n_heads, pad_id, layers)
