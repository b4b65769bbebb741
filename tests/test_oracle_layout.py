"""Pins of the oracle's table layout against what the pages and arithmetic fix."""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import layout as L


def _golden():
    with open(os.path.join(GOLDEN, "prime_table.json")) as f:
        return json.load(f)


@pytest.fixture(scope="module")
def v41_layout():
    g = _golden()
    return L.build_layout(99092, g["base_rows"], g["layer_ids"], g["max_ngram"], g["n_heads"])


def test_prime_table_matches_page(v41_layout):
    """min / max / sum of the 24 primes of layers 1 and 14 as printed on the page."""
    g = _golden()
    for lay in v41_layout.layers:
        exp = g["layers"][str(lay.layer_id)]
        assert min(lay.primes) == exp["min_prime"]
        assert max(lay.primes) == exp["max_prime"]
        assert lay.total_rows == exp["sum"] == sum(lay.primes)
    assert sum(x.total_rows for x in v41_layout.layers) == g["sum_both_layers"]


def test_primes_are_prime_increasing_unique(v41_layout):
    sympy = pytest.importorskip("sympy")
    allp = [p for lay in v41_layout.layers for p in lay.primes]
    assert all(sympy.isprime(p) for p in allp)
    assert allp == sorted(allp) and len(set(allp)) == len(allp)
    # consecutive: no prime is skipped between the base and the last prime used
    assert sympy.nextprime(16_000_000) == allp[0]
    for a, b in zip(allp, allp[1:]):
        assert sympy.nextprime(a) == b


def test_segments_disjoint_and_cover(v41_layout):
    for lay in v41_layout.layers:
        ends = [o + p for o, p in zip(lay.offsets, lay.primes)]
        assert lay.offsets[0] == 0
        assert all(e == o for e, o in zip(ends[:-1], lay.offsets[1:]))
        assert ends[-1] == lay.total_rows


@pytest.mark.parametrize("vocab", [1000, 99092, 129280, 2])
def test_multipliers_odd_and_bounded(vocab):
    lay = L.build_layout(vocab, 4099, [1, 14], 4, 8)
    for x in lay.layers:
        assert len(x.multipliers) == 4
        for m in x.multipliers:
            assert m % 2 == 1
            assert (vocab - 1) * m <= L.INT64_MAX          # x' * m never overflows int64
            assert m < L.INT64_MAX // vocab                # the page's bound (2^63-1)/V
    # layers draw independent multipliers
    assert lay.layers[0].multipliers != lay.layers[1].multipliers


def test_splitmix64_published_vector():
    """SplitMix64 with state 0: first outputs as published with the generator."""
    assert L.splitmix64(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_vocab_guard():
    with pytest.raises(ValueError):
        L.build_layout(99091, 16_000_000, [1], expected_vocab=99092)


def test_small_bases_are_consecutive_primes():
    lay = L.build_layout(1000, 4099, [1])
    ps = lay.layers[0].primes
    assert ps[0] == 4111  # 4099 itself is prime: primes strictly above the base
    sympy = pytest.importorskip("sympy")
    assert ps == list(sympy.primerange(4100, ps[-1] + 1))
    assert lay.layers[0].total_rows == 100966


def test_base_2m_total_rows():
    lay = L.build_layout(99092, 2_000_000, [1])
    assert lay.layers[0].total_rows == 48004402


def test_override_validated():
    with pytest.raises(ValueError):
        L.build_layout(1000, 4099, [1], multipliers_override=[[2, 3, 5, 7]])
    lay = L.build_layout(1000, 4099, [1], multipliers_override=[[3, 5, 7, 9]])
    assert lay.layers[0].multipliers == [3, 5, 7, 9]
