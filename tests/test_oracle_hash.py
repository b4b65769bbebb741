"""Pins of the oracle's token map, windows and multiplicative-XOR hash."""
import itertools
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import hashing as Hs
from oracle import layout as L
from workloads import WORKLOADS, prefill_batch, token_map

DEAD = Hs.DEAD


def _worked_layout(g):
    sizes = g["prime_sizes"]
    primes = sizes["2"] + sizes["3"]
    lay = L.LayerLayout(0, primes, [0, 0, 0, 0], sum(primes), list(g["multipliers"]))
    return L.Layout(vocab=1000, base_rows=0, max_ngram=3, n_heads=2, pad_id=0, layers=[lay])


def test_worked_example_from_page():
    """Mixes 549 / 174 and indices [44, 34] / [67, 65] of the hand-computed example."""
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    lay = _worked_layout(g)
    toks = np.array(g["tokens"])
    ident = np.arange(1000, dtype=np.int32)
    rows, mask, _ = Hs.hash_prefill(toks, np.array([0, 4]), ident, lay, 0)
    xc = Hs.compress(toks, ident)
    win, _ = Hs.windows(xc, np.array([0, 4]), None, 0, 3)
    mix = Hs.mixes(win, g["multipliers"])
    assert int(mix[3, 0]) == g["expected"]["2"]["mix"]
    assert int(mix[3, 1]) == g["expected"]["3"]["mix"]
    assert list(rows[3, :2]) == g["expected"]["2"]["indices"]
    assert list(rows[3, 2:]) == g["expected"]["3"]["indices"]
    assert not mask.any()


def test_first_token_pairs_with_pad():
    """The first token's 2-gram is (current token, pad) and is looked up normally."""
    m = [11, 13, 17, 19]
    lay = L.Layout(1000, 0, 4, 1, pad_id=7,
                   layers=[L.LayerLayout(0, [1_000_003, 1_000_033, 1_000_037], [0, 0, 0], 0, m)])
    xc = np.array([5])
    win, _ = Hs.windows(xc, np.array([0, 1]), None, 7, 4)
    assert list(win[0]) == [5, 7, 7, 7]
    mix = Hs.mixes(win, m)
    assert int(mix[0, 0]) == (5 * 11) ^ (7 * 13)


def test_rolling_identity_and_order_sensitivity():
    """mix3 = mix2 ^ x'_{t-2} m_2, mix4 = mix3 ^ x'_{t-3} m_3; (A, B) != (B, A)."""
    lay = L.build_layout(99092, 2_000_000, [1])
    m = lay.layers[0].multipliers
    rng = np.random.default_rng(0)
    g = rng.integers(0, 99092, size=(1000, 4))
    mix = Hs.mixes(g, m)
    for t in range(0, 1000, 97):
        a = [int(x) for x in g[t]]
        m2 = (a[0] * m[0]) ^ (a[1] * m[1])
        assert int(mix[t, 0]) == m2
        assert int(mix[t, 1]) == m2 ^ (a[2] * m[2])
        assert int(mix[t, 2]) == m2 ^ (a[2] * m[2]) ^ (a[3] * m[3])
    ab = Hs.mixes(np.array([[3, 9, 0, 0]]), m)
    ba = Hs.mixes(np.array([[9, 3, 0, 0]]), m)
    assert int(ab[0, 0]) != int(ba[0, 0])


def test_mix_below_2_63():
    lay = L.build_layout(99092, 2_000_000, [1])
    g = np.full((1, 4), 99091)
    assert int(Hs.mixes(g, lay.layers[0].multipliers).max()) < 2 ** 63


def test_crt_bound_base_16m_bruteforce():
    """Distinct mixes collide in at most 2 of the 8 heads (every 3 primes multiply past 2^63).

    Brute force over all 2/3/4-grams of a 12-id vocabulary (20,736 4-grams):
    for every triple of heads the residue triples of distinct mixes are distinct.
    """
    V = 12
    lay = L.build_layout(V, 16_000_000, [1])
    ps = lay.layers[0].primes
    assert ps[0] * ps[1] * ps[2] > 2 ** 63  # the three smallest primes of the layer
    g = np.array(list(itertools.product(range(V), repeat=4)))
    mix = Hs.mixes(g, lay.layers[0].multipliers)
    for n in range(2, 5):
        col = np.unique(mix[:, n - 2])
        heads = ps[(n - 2) * 8:(n - 1) * 8]
        res = np.stack([col % np.uint64(p) for p in heads], axis=1)
        for a, b, c in itertools.combinations(range(8), 3):
            trip = res[:, [a, b, c]]
            assert len(np.unique(trip, axis=0)) == len(col)


def test_crt_bound_fails_without_premise():
    """Base 4099: three small primes multiply below 2^63, so a 3-head collision exists."""
    ps = L.build_layout(1000, 4099, [1]).layers[0].primes
    a = 123456789
    b = a + ps[0] * ps[1] * ps[2]
    assert b < 2 ** 63
    same = [a % p == b % p for p in ps[:8]]
    assert sum(same) >= 3


def _tiny():
    w = WORKLOADS["tiny"]
    tm = token_map(w.v_raw, w.v, 0)
    lay = L.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    return w, tm, lay


def test_dead_cascade_restarts_windows():
    """Past an image span the windows are those of a fresh sequence; DEAD is masked."""
    w, tm, lay = _tiny()
    a, b, c, d = 10, 20, 30, 40
    seq = np.array([a, b, DEAD, c, d])
    rows, mask, _ = Hs.hash_prefill(seq, np.array([0, 5]), tm, lay, 0)
    fresh, fmask, _ = Hs.hash_prefill(np.array([c, d]), np.array([0, 2]), tm, lay, 0)
    assert (rows[3] == fresh[0]).all() and (rows[4] == fresh[1]).all()
    assert list(mask) == [False, False, True, False, False]
    # at the DEAD position every slot is pad: same rows as a pad-only window
    win, _ = Hs.windows(np.array([DEAD]), np.array([0, 1]), None, lay.pad_id, 4)
    assert (win == lay.pad_id).all()


def test_prefill_equals_chunked_equals_replay():
    """Prefill and decode share one history ([P-LMNT] §第二步): whole == chunks == steps."""
    w, tm, lay = _tiny()
    rng = np.random.default_rng(1)
    lens = [0, 1, 2, 3, 9, 40]
    seqs = [rng.integers(0, w.v_raw, n) for n in lens]
    seqs[4][3] = DEAD
    seqs[5][[5, 6, 20]] = DEAD
    raw = np.concatenate(seqs)
    cu = np.concatenate([[0], np.cumsum(lens)])
    rows, mask, hist = Hs.hash_prefill(raw, cu, tm, lay, 0)
    # chunked: split every sequence at a cut point, carry the history
    cut = [min(c, n) for c, n in zip([0, 0, 1, 2, 4, 17], lens)]
    first = [s[:c] for s, c in zip(seqs, cut)]
    second = [s[c:] for s, c in zip(seqs, cut)]
    cu1 = np.concatenate([[0], np.cumsum([len(x) for x in first])])
    cu2 = np.concatenate([[0], np.cumsum([len(x) for x in second])])
    r1, m1, h1 = Hs.hash_prefill(np.concatenate(first), cu1, tm, lay, 0)
    r2, m2, h2 = Hs.hash_prefill(np.concatenate(second), cu2, tm, lay, 0, hist=h1)
    for s in range(len(lens)):
        whole = rows[cu[s]:cu[s + 1]]
        parts = np.concatenate([r1[cu1[s]:cu1[s + 1]], r2[cu2[s]:cu2[s + 1]]])
        assert (whole == parts).all()
    assert (h2 == hist).all()
    # replay: one decode step per token, starting from an all-pad history
    H = np.full((len(lens), 3), lay.pad_id)
    for s, seq in enumerate(seqs):
        for t, tok in enumerate(seq):
            r, m, H = Hs.hash_step(np.array([tok]), np.array([s]), H, tm, lay, 0)
            assert (r[0] == rows[cu[s] + t]).all() and m[0] == mask[cu[s] + t]
    assert (H == hist).all()


def test_step_padding_row_commits_nothing():
    w, tm, lay = _tiny()
    H = np.array([[1, 2, 3], [4, 5, 6]])
    r, m, H2 = Hs.hash_step(np.array([7, 8]), np.array([-1, 1]), H, tm, lay, 0)
    assert m[0] and not m[1]
    assert (H2[0] == H[0]).all()
    assert list(H2[1]) == [tm[8], 4, 5]


def test_bad_token_rejected():
    w, tm, lay = _tiny()
    with pytest.raises(ValueError):
        Hs.compress(np.array([5, w.v_raw]), tm)
    with pytest.raises(ValueError):
        Hs.compress(np.array([-2]), tm)


def test_rows_in_column_segments():
    w, tm, lay = _tiny()
    b = prefill_batch(w)
    rows, _, _ = Hs.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay, 0)
    x = lay.layers[0]
    for j in range(24):
        assert (rows[:, j] >= x.offsets[j]).all() and (rows[:, j] < x.offsets[j] + x.primes[j]).all()


def test_token_map_is_surjection():
    tm = token_map(1300, 1000, 0)
    assert tm.min() == 0 and tm.max() == 999 and len(np.unique(tm)) == 1000
