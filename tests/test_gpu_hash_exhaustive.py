"""Exhaustive GPU hash over a small compressed vocabulary, bit-exact against the oracle.

Every compressed 4-gram over V = 12 ids (12^4 = 20,736 windows) is hashed:
ids 0 and V-1 and the pad id appear in every slot of the window.  Windows
are built three ways -- as the last position of a 4-token prefill sequence,
as a decode step on a carried 3-id history, and split over two prefill
chunks at every offset -- with DEAD at every slot offset, in the sequence and
in the carried history.  Multipliers are the library's own and a set at the
int64 bound (V-1) m <= 2^63 - 1, so that every mix reaches the top of the
range.  The rolling hash is eq. (H) of "DeepSeek-V4.1 模型结构（5）：记忆，Engram"
§哈希函数, and the DEAD rule is its §V4.1 相对原版的两处改动.
"""
import itertools

import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import i32, i64, require_gpu, status
from oracle import hashing as OH
from oracle import layout as OL
from workloads import DEAD, rng_for

pytestmark = pytest.mark.gpu

V = 12                 # compressed vocabulary
V_RAW = V + 5          # raw vocabulary: a permutation of [0, V) plus 5 duplicates
BASE = 16_000_000      # the full-scale prime base


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _token_map():
    g = rng_for(11, 1)
    tm = np.concatenate([g.permutation(V), g.integers(0, V, V_RAW - V)]).astype(np.int32)
    return tm


def _raw_of(tm):
    """One raw id for every compressed id (the first that maps to it)."""
    inv = np.full(V, -1, dtype=np.int64)
    for r in range(V_RAW - 1, -1, -1):
        inv[tm[r]] = r
    assert (inv >= 0).all()
    return inv


def _bound_multipliers():
    m = (2 ** 63 - 1) // (V - 1)
    m -= 1 - m % 2                     # largest odd multiplier with (V-1) m <= 2^63 - 1
    return [[m, m - 2, m - 4, m - 6]]


def _layouts(pad):
    out = []
    for mults in (None, _bound_multipliers()):
        lay_o = OL.build_layout(V, BASE, [1], pad_id=pad, multipliers_override=mults)
        lay = eg.build_layout(V, BASE, [1], pad_id=pad, multipliers=mults)
        assert list(lay_o.layers[0].multipliers) == [int(x) for x in lay.multipliers(0)]
        out.append((lay_o, lay))
    return out


def _all_4grams():
    return np.array(list(itertools.product(range(V), repeat=4)), dtype=np.int64)   # [V^4][4], oldest first


def _sequences(grams, raw_of, dead_at=None):
    """Each 4-gram (oldest first) as a 4-token sequence of raw ids; DEAD at position dead_at."""
    raw = raw_of[grams].astype(np.int32)
    if dead_at is not None:
        raw[:, dead_at] = DEAD
    n = len(grams)
    return raw.reshape(-1), np.arange(n + 1, dtype=np.int64) * 4


@pytest.mark.parametrize("pad", [0, 5, V - 1])
def test_every_4gram_prefill_bit_exact(pad):
    tm = _token_map()
    raw_of = _raw_of(tm)
    grams = _all_4grams()
    for lay_o, lay in _layouts(pad):
        for dead_at in (None, 0, 1, 2, 3):
            raw, cu = _sequences(grams, raw_of, dead_at)
            rows_o, mask_o, hist_o = OH.hash_prefill(raw, cu, tm, lay_o, 0)
            hist_d = i32(np.full((len(grams), 3), pad))
            st = status()
            rows, mask = eg.engram_hash(lay, 0, i32(raw), i64(cu), i32(tm), hist_d, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert (rows.cpu().numpy() == rows_o).all(), (pad, dead_at)
            assert (mask.cpu().numpy().astype(bool) == mask_o).all(), (pad, dead_at)
            assert (hist_d.cpu().numpy() == hist_o).all(), (pad, dead_at)


@pytest.mark.parametrize("pad", [0, 5])
def test_every_4gram_split_over_two_chunks(pad):
    """The first k tokens of every sequence in one call, the rest in the next
    with the history carried, for k = 1, 2, 3: the same ids as one call, with
    DEAD at every offset on either side of the chunk boundary."""
    tm = _token_map()
    raw_of = _raw_of(tm)
    grams = _all_4grams()
    n = len(grams)
    lay_o, lay = _layouts(pad)[1]
    for dead_at in (None, 0, 1, 2, 3):
        raw, cu = _sequences(grams, raw_of, dead_at)
        whole_o, _, _ = OH.hash_prefill(raw, cu, tm, lay_o, 0)
        seqs = raw.reshape(n, 4)
        for k in (1, 2, 3):
            hist_d = i32(np.full((n, 3), pad))
            a = seqs[:, :k].reshape(-1)
            b = seqs[:, k:].reshape(-1)
            ra, _ = eg.engram_hash(lay, 0, i32(a), i64(np.arange(n + 1) * k), i32(tm), hist_d)
            rb, _ = eg.engram_hash(lay, 0, i32(b), i64(np.arange(n + 1) * (4 - k)), i32(tm), hist_d)
            got = np.concatenate([ra.cpu().numpy().reshape(n, k, 24), rb.cpu().numpy().reshape(n, 4 - k, 24)],
                                 axis=1).reshape(-1, 24)
            assert (got == whole_o).all(), (dead_at, k)


@pytest.mark.parametrize("pad", [0, 5, V - 1])
def test_every_4gram_decode_step(pad):
    """One decode step per 4-gram: history (c, b, a) in its own slot, new id d;
    DEAD in every history slot and as the new id.  The rows equal the oracle's
    step and the last position of the prefill of (a, b, c, d)."""
    tm = _token_map()
    raw_of = _raw_of(tm)
    grams = _all_4grams()
    n = len(grams)
    slots = np.arange(n, dtype=np.int32)
    for lay_o, lay in _layouts(pad):
        for dead_slot in (None, 0, 1, 2, "new"):
            hist = grams[:, [2, 1, 0]].copy()          # compressed, most recent first
            raw_new = raw_of[grams[:, 3]].astype(np.int32)
            if dead_slot == "new":
                raw_new[:] = DEAD
            elif dead_slot is not None:
                hist[:, dead_slot] = DEAD
            rows_o, mask_o, hist_o = OH.hash_step(raw_new, slots, hist, tm, lay_o, 0)
            hist_d = i32(hist)
            st = status()
            rows, mask = eg.engram_hash_step(lay, 0, i32(raw_new), i32(slots), i32(tm), hist_d, status=st)
            torch.cuda.synchronize()
            assert int(st.item()) == 0
            assert (rows.cpu().numpy() == rows_o).all(), (pad, dead_slot)
            assert (mask.cpu().numpy().astype(bool) == mask_o).all(), (pad, dead_slot)
            assert (hist_d.cpu().numpy() == hist_o).all(), (pad, dead_slot)
            if dead_slot is None:
                raw, cu = _sequences(grams, raw_of)
                pre_o, _, _ = OH.hash_prefill(raw, cu, tm, lay_o, 0)
                assert (rows.cpu().numpy() == pre_o.reshape(n, 4, 24)[:, 3]).all(), pad
