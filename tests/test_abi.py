"""The C-ABI library loads, exports every declared symbol, and its host-side
layout builder and argument checks agree with the oracle (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import hashed_gram_conditional_gb300 as eg
from conftest import ROOT
from oracle import layout as OL

HEADER = os.path.join(ROOT, "include", "engram.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(eg.library_path()):
        from hashed_gram_conditional_gb300 import build
        build.build()
    return eg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(engram_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for required in ["engram_build_layout", "engram_hash", "engram_hash_step", "engram_gather_dequant",
                     "engram_project", "engram_gate_add"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_sizes_match(lib):
    assert lib.engram_layout_size() == ctypes.sizeof(eg._Layout)
    assert lib.engram_layout_params_size() == ctypes.sizeof(eg._LayoutParams)
    assert lib.engram_abi_version() == 3


@pytest.mark.parametrize("vocab,base,layers", [(1000, 4099, [1]), (99092, 2_000_000, [1]),
                                               (99092, 16_000_000, [1, 14]), (12, 16_000_000, [0, 3, 7])])
def test_layout_equals_oracle(lib, vocab, base, layers):
    ref = OL.build_layout(vocab, base, layers, 4, 8, pad_id=min(7, vocab - 1))
    got = eg.build_layout(vocab, base, layers, 4, 8, pad_id=min(7, vocab - 1))
    assert got.n_cols == 24 and got.n_layers == len(layers)
    for li, x in enumerate(ref.layers):
        assert got.layer_id(li) == x.layer_id
        assert got.primes(li) == x.primes
        assert got.offsets(li) == x.offsets
        assert got.total_rows(li) == x.total_rows
        assert got.multipliers(li) == x.multipliers
        for j, p in enumerate(x.primes):
            assert got._raw.reciprocal[li][j] == (2 ** 64 - 1) // p


def test_layout_generic_orders_heads(lib):
    for max_ngram, heads in [(2, 8), (3, 8), (4, 4), (3, 16)]:
        ref = OL.build_layout(1000, 4099, [2, 15], max_ngram, heads)
        got = eg.build_layout(1000, 4099, [2, 15], max_ngram, heads)
        assert got.n_cols == (max_ngram - 1) * heads
        for li, x in enumerate(ref.layers):
            assert got.primes(li) == x.primes and got.multipliers(li) == x.multipliers


def test_layout_override(lib):
    got = eg.build_layout(1000, 4099, [1], multipliers=[[3, 5, 7, 9]])
    assert got.multipliers(0) == [3, 5, 7, 9]
    with pytest.raises(eg.EngramError, match="RANGE"):
        eg.build_layout(1000, 4099, [1], multipliers=[[4, 5, 7, 9]])
    with pytest.raises(eg.EngramError, match="RANGE"):
        eg.build_layout(1000, 4099, [1], multipliers=[[(2 ** 63 - 1) // 999 + 2, 5, 7, 9]])


def test_layout_errors(lib):
    with pytest.raises(eg.EngramError, match="VOCAB"):
        eg.build_layout(99091, 16_000_000, [1], expected_vocab=99092)
    with pytest.raises(eg.EngramError, match="SHAPE"):
        eg.build_layout(1000, 4099, [1], head_dim=128)
    with pytest.raises(eg.EngramError, match="SHAPE"):
        eg.build_layout(1000, 4099, [1], max_ngram=5)
    with pytest.raises(eg.EngramError, match="INVALID"):
        eg.build_layout(1000, 4099, [1], pad_id=1000)
    with pytest.raises(eg.EngramError, match="RANGE"):
        eg.build_layout(1000, 2 ** 31 - 1000, [1])  # row count would pass 2^31
    assert lib.engram_build_layout(None, None) == -1
    assert b"null" in lib.engram_last_error()


def test_host_side_argument_checks(lib):
    """Entry points reject bad sizes before touching a device."""
    P = ctypes.c_void_p
    assert lib.engram_gather_dequant(P(16), 10, 10 * 264, P(16), 4, 0, P(16), None, None) == -3
    assert lib.engram_gather_dequant(P(16), 10, 10 * 264 - 1, P(16), 4, 24, P(16), None, None) == -3
    assert lib.engram_project(P(16), 128, 6144, P(16), 100, 4, P(16), P(16), P(16), P(16), P(16), None, None) == -3
    assert lib.engram_project(P(16), 128, 6100, P(16), 256, 4, P(16), P(16), P(16), P(16), P(16), None, None) == -3
    assert lib.engram_gate_add(P(16), P(16), P(16), None, 4, 256, 9, 1e-6, 1e-6, 0.0625, None, None) == -3
    lay = eg.build_layout(1000, 4099, [1])
    assert lib.engram_hash(lay.ref, 3, P(16), 4, P(16), 1, P(16), 1300, None, P(16), P(16), None, None) == -1
    assert lib.engram_project_partials_bytes(16384, 5120, 4) == 16384 * 4 * 20 * 16


def test_host_side_argument_checks_of_the_wider_path(lib):
    """The FP8, fused hash + gather, short-convolution and host-gather entry
    points reject bad shapes and pointers before touching a device."""
    P = ctypes.c_void_p
    E_INVALID, E_SHAPE, E_ALIGN = -1, -3, -4
    lay = eg.build_layout(1000, 4099, [1])
    # FP8 packing: K and N multiples of 128; nothing to do for empty batches
    assert lib.engram_pack_wkv_fp8(P(16), P(16), 100, 256, P(16), P(16), None) == E_SHAPE
    assert lib.engram_pack_wkv_fp8(P(16), P(16), 256, 100, P(16), P(16), None) == E_SHAPE
    assert lib.engram_pack_wkv_fp8(None, P(16), 256, 256, P(16), P(16), None) == E_INVALID
    # FP8 projection: K % 128, hidden % 256, hc range
    args = (P(16), P(16), 128, 6100, P(16), P(16), 256, 4, P(16), P(16), P(16), P(16), P(16), None, None)
    assert lib.engram_project_fp8(*args) == E_SHAPE
    args = (P(16), P(16), 128, 6144, P(16), P(16), 200, 4, P(16), P(16), P(16), P(16), P(16), None, None)
    assert lib.engram_project_fp8(*args) == E_SHAPE
    args = (P(16), P(16), 128, 6144, P(16), P(16), 256, 9, P(16), P(16), P(16), P(16), P(16), None, None)
    assert lib.engram_project_fp8(*args) == E_SHAPE
    assert lib.engram_project_fp8(P(16), P(16), 0, 6144, P(16), P(16), 256, 4, P(16), P(16), P(16), P(16),
                                  P(16), None, None) == 0
    # FP8 gather: n_cols, table size, alignment
    assert lib.engram_gather_fp8(P(16), 10, 10 * 264, P(16), 4, 0, P(16), P(16), None, None) == E_SHAPE
    assert lib.engram_gather_fp8(P(16), 10, 10 * 264 - 1, P(16), 4, 24, P(16), P(16), None, None) == E_SHAPE
    assert lib.engram_gather_fp8(P(17), 10, 10 * 264, P(16), 4, 24, P(16), P(16), None, None) == E_ALIGN
    # fused hash + gather: layer range, sequence count, table size
    assert lib.engram_hash_gather(lay.ref, 3, P(16), 4, P(16), 1, P(16), 1300, None, P(16), 10 ** 9, P(16), P(16),
                                  None, None, None) == E_INVALID
    assert lib.engram_hash_gather(lay.ref, 0, P(16), 4, P(16), 0, P(16), 1300, None, P(16), 10 ** 9, P(16), P(16),
                                  None, None, None) == E_INVALID
    assert lib.engram_hash_gather(lay.ref, 0, P(16), 4, P(16), 1, P(16), 1300, None, P(16), 264, P(16), P(16),
                                  None, None, None) == E_SHAPE
    assert lib.engram_hash_gather_fp8(lay.ref, 0, P(16), 4, P(16), 1, P(16), 1300, None, P(16), 264, P(16), P(16),
                                      P(16), None, None, None) == E_SHAPE
    # short convolution: kernel size, dilation, ring length, shapes
    conv = lambda K, dil, hidden=256, hc=4, n_seqs=4, cu=None: lib.engram_short_conv_add(  # noqa: E731
        P(16), P(16), P(16), None, 4, hidden, hc, cu, n_seqs, None, P(16), P(16), K, dil, 1e-6, None, None, 0,
        P(256), 1 << 20, None, None)
    assert conv(5, 3) == E_SHAPE
    assert conv(0, 3) == E_SHAPE
    assert conv(4, 0) == E_SHAPE
    assert conv(4, 30) == E_SHAPE                 # (K-1)*dilation = 90 > 64
    assert conv(4, 3, hidden=200) == E_SHAPE
    assert conv(4, 3, hc=9) == E_SHAPE
    assert conv(4, 3, n_seqs=3) == E_SHAPE        # without cu_seqlens every position is a sequence
    assert lib.engram_short_conv_workspace_bytes(1000, 4) == 2 * 16128 + 3 * 4096
    # host gather: sizes and pointers
    assert lib.engram_host_gather(None, 10, None, 5, None, 0, None) == E_INVALID
    assert lib.engram_host_gather(None, -1, None, 0, None, 0, None) == E_INVALID


def test_kernel_options_round_trip_and_range_checks(lib):
    """engram_set/get_kernel_options: host-only, no device needed."""
    prev = eg.kernel_options()
    assert prev == dict(projection_cta=0, gather_copy=0, fp8_pair=0, fp8_fused=0, plain_launch=0)
    try:
        eg.set_kernel_options(projection_cta=2, plain_launch=1)
        assert eg.kernel_options() == dict(projection_cta=2, gather_copy=0, fp8_pair=0, fp8_fused=0, plain_launch=1)
        with pytest.raises(eg.EngramError):
            eg.set_kernel_options(projection_cta=3)
        with pytest.raises(eg.EngramError):
            eg.set_kernel_options(gather_copy=-1)
        # a rejected call changes nothing
        assert eg.kernel_options()["projection_cta"] == 2
        with pytest.raises(ValueError):
            eg.set_kernel_options(no_such_option=1)
        assert lib.engram_set_kernel_options(None) == -1
    finally:
        eg.set_kernel_options(**prev)
    assert eg.kernel_options() == prev


def test_fp8_scale_layout_helpers():
    """sf_cols rounds a token count up to whole 128-position blocks, and
    sf_word_index is the order the header states for block-FP8 scale words:
    within each 128 words, word 4r + c holds position (or column) r + 32c, a
    permutation of the block."""
    assert [eg.sf_cols(n) for n in (0, 1, 127, 128, 129, 16384)] == [0, 128, 128, 128, 256, 16384]
    for base in (0, 128, 4096):
        idx = [eg.sf_word_index(base + r + 32 * c) for r in range(32) for c in range(4)]
        assert idx == list(range(base, base + 128))
