"""GPU parity of the hash stages (token map, window, mix, modulo): bit-exact."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import DEV, device_table, i32, i64, require_gpu, setup, status
from oracle import hashing as OH
from oracle import layout as OL
from workloads import DEAD, WORKLOADS, decode_workload, prefill_batch, zipf_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _run_hash(lay, raw, cu, tm, hist=None):
    st = status()
    h = None if hist is None else i32(hist)
    rows, mask = eg.engram_hash(lay, 0, i32(raw), i64(cu), i32(tm), h, status=st)
    torch.cuda.synchronize()
    return rows.cpu().numpy(), mask.cpu().numpy().astype(bool), (None if h is None else h.cpu().numpy()), \
        int(st.item())


@pytest.mark.parametrize("name", ["tiny", "microbench", "prefill"])
def test_hash_config_bit_exact(name):
    w, tm, lay_o, lay = setup(name)
    b = prefill_batch(w)
    rows_o, mask_o, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    rows, mask, _, st = _run_hash(lay, b.raw_ids, b.cu_seqlens, tm)
    assert st == 0
    assert (rows == rows_o).all()
    assert (mask == mask_o).all()
    if w.dead_frac > 0:
        assert mask.any()


def test_hash_ragged_sequences_history_and_dead():
    w, tm, lay_o, lay = setup("tiny")
    rng = np.random.default_rng(7)
    lens = [0, 1, 2, 3, 5, 31, 32, 33, 200, 0, 7]
    seqs = [rng.integers(0, w.v_raw, n).astype(np.int32) for n in lens]
    seqs[4][1] = DEAD
    seqs[8][[0, 1, 50, 51, 52, 199]] = DEAD
    seqs[7][-1] = DEAD
    raw = np.concatenate(seqs)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    hist0 = rng.integers(0, w.v, size=(len(lens), 3)).astype(np.int64)
    hist0[2, 1] = DEAD
    hist0[5, 0] = DEAD
    rows_o, mask_o, hist_o = OH.hash_prefill(raw, cu, tm, lay_o, 0, hist=hist0)
    rows, mask, hist, st = _run_hash(lay, raw, cu, tm, hist=hist0)
    assert st == 0
    assert (rows == rows_o).all() and (mask == mask_o).all()
    assert (hist.reshape(hist_o.shape) == hist_o).all()


def test_hash_chunked_equals_whole():
    w, tm, lay_o, lay = setup("prefill")
    b = prefill_batch(w)
    whole, wmask, _, _ = _run_hash(lay, b.raw_ids, b.cu_seqlens, tm)
    hist = np.full((w.n_seqs, 3), lay.pad_id, dtype=np.int32)
    hist_d = i32(hist)
    parts = []
    L = w.seq_len
    for c0, c1 in [(0, 1000), (1000, 1001), (1001, 1003), (1003, L)]:
        raw = np.concatenate([b.raw_ids[s * L + c0: s * L + c1] for s in range(w.n_seqs)])
        cu = np.arange(w.n_seqs + 1, dtype=np.int64) * (c1 - c0)
        r, m = eg.engram_hash(lay, 0, i32(raw), i64(cu), i32(tm), hist_d)
        parts.append(r.cpu().numpy().reshape(w.n_seqs, c1 - c0, 24))
    chunked = np.concatenate(parts, axis=1).reshape(-1, 24)
    assert (chunked == whole).all()


def test_hash_bad_tokens_flagged():
    w, tm, lay_o, lay = setup("tiny")
    raw = np.array([5, w.v_raw, 7, -5, 9], dtype=np.int32)
    rows, mask, _, st = _run_hash(lay, raw, np.array([0, 5]), tm)
    assert st & eg.ST_BAD_TOKEN
    assert list(mask) == [False, True, False, True, False]   # a bad id is treated as DEAD


def test_hash_empty_and_single():
    w, tm, lay_o, lay = setup("tiny")
    rows, mask = eg.engram_hash(lay, 0, i32(np.zeros(0)), i64([0, 0]), i32(tm))
    assert rows.shape == (0, 24)
    raw = np.array([3], dtype=np.int32)
    rows_o, mask_o, _ = OH.hash_prefill(raw, np.array([0, 1]), tm, lay_o, 0)
    rows, mask, _, _ = _run_hash(lay, raw, np.array([0, 1]), tm)
    assert (rows == rows_o).all()


def test_hash_override_multipliers_and_generic_orders():
    """Large override multipliers (mixes near 2^63) and 2-/3-gram layouts with 16 heads."""
    w, tm, _, _ = setup("tiny")
    big = (2 ** 63 - 1) // (w.v - 1)
    big -= 1 - big % 2
    mults = [[big, big - 2, big - 4, big - 6]]
    b = prefill_batch(w)
    for max_ngram, heads, mm in [(4, 8, mults), (2, 8, None), (3, 16, None)]:
        lay_o = OL.build_layout(w.v, w.base_rows, [1], max_ngram, heads, pad_id=int(tm[0]),
                                multipliers_override=None if mm is None else [m[:max_ngram] for m in mm])
        lay = eg.build_layout(w.v, w.base_rows, [1], max_ngram, heads, pad_id=int(tm[0]),
                              multipliers=None if mm is None else [m[:max_ngram] for m in mm])
        rows_o, mask_o, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
        rows, mask = eg.engram_hash(lay, 0, i32(b.raw_ids), i64(b.cu_seqlens), i32(tm))
        assert (rows.cpu().numpy() == rows_o).all()


def test_selftest_mod_edge_values():
    """Device modulo against Python's % on edge and random 64-bit values."""
    w, tm, lay_o, lay = setup("microbench")
    ps = lay_o.layers[0].primes
    vals = [0, 1, 2 ** 63 - 1, 2 ** 63, 2 ** 64 - 1, 2 ** 32, 2 ** 32 - 1]
    for p in ps[:6]:
        for k in [1, 2, 3, 10 ** 6, (2 ** 63 - 1) // p, (2 ** 64 - 1) // p]:
            for d in (-1, 0, 1):
                x = k * p + d
                if 0 <= x < 2 ** 64:
                    vals.append(x)
    rng = np.random.default_rng(3)
    vals += [int(x) for x in rng.integers(0, 2 ** 63, size=20000, dtype=np.uint64)]
    vals += [int(x) | (1 << 63) for x in rng.integers(0, 2 ** 63, size=2000, dtype=np.uint64)]
    x = np.array(vals, dtype=np.uint64)
    out = eg.engram_selftest_mod(lay, 0, torch.from_numpy(x.view(np.int64)).to(DEV)).cpu().numpy()
    off = lay_o.layers[0].offsets
    for j, p in enumerate(ps):
        exp = (x % np.uint64(p)).astype(np.int64) + off[j]
        assert (out[:, j] == exp).all(), j


def test_hash_step_decode_replay():
    """Decode steps from prefix histories equal the oracle, and equal prefill of prefix+token."""
    w, tm, lay_o, lay = setup("decode")
    dw = decode_workload(w, n_steps=12)
    pre = dw.prefix
    S = w.n_seqs
    # histories from prefill of the prefixes (GPU and oracle independently)
    _, _, hist_o = OH.hash_prefill(pre.raw_ids, pre.cu_seqlens, tm, lay_o, 0)
    hist_d = i32(np.full((S, 3), lay.pad_id))
    eg.engram_hash(lay, 0, i32(pre.raw_ids), i64(pre.cu_seqlens), i32(tm), hist_d)
    assert (hist_d.cpu().numpy() == hist_o).all()
    slots = np.arange(S, dtype=np.int32)
    slots[5] = -1  # a padding entry commits nothing
    st = status()
    H = hist_o.copy()
    for step in range(dw.steps.shape[0]):
        raw = dw.steps[step]
        rows_o, mask_o, H = OH.hash_step(raw, slots, H, tm, lay_o, 0)
        rows, mask = eg.engram_hash_step(lay, 0, i32(raw), i32(slots), i32(tm), hist_d, status=st)
        assert (rows.cpu().numpy() == rows_o).all(), step
        assert (mask.cpu().numpy().astype(bool) == mask_o).all(), step
        assert (hist_d.cpu().numpy() == H).all(), step
    assert int(st.item()) == 0


def test_hash_step_bad_slot():
    w, tm, lay_o, lay = setup("tiny")
    hist = i32(np.full((4, 3), lay.pad_id))
    st = status()
    rows, mask = eg.engram_hash_step(lay, 0, i32([1, 2]), i32([0, 9]), i32(tm), hist, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & eg.ST_BAD_SLOT
    assert list(mask.cpu().numpy()) == [0, 1]


def test_hash_zero_tokens_keeps_history():
    """A call with no tokens still runs the history commit on its own (as a
    programmatic dependent of whatever the stream ran last): every sequence
    is empty, so each history row comes back unchanged, DEAD slots included."""
    w, tm, lay_o, lay = setup("tiny")
    rng = np.random.default_rng(11)
    hist0 = rng.integers(0, w.v, size=(5, 3)).astype(np.int32)
    hist0[1, 2] = DEAD
    hist_d = i32(hist0)
    cu = np.zeros(6, dtype=np.int64)
    st = status()
    # something on the stream first: a real hash call whose kernel allows early dependent launch
    b = prefill_batch(w)
    eg.engram_hash(lay, 0, i32(b.raw_ids), i64(b.cu_seqlens), i32(tm), status=st)
    rows, mask = eg.engram_hash(lay, 0, i32(np.zeros(0, dtype=np.int32)), i64(cu), i32(tm), hist_d, status=st)
    torch.cuda.synchronize()
    assert rows.shape[0] == 0
    assert int(st.item()) == 0
    assert (hist_d.cpu().numpy() == hist0).all()
    _, _, hist_o = OH.hash_prefill(np.zeros(0, dtype=np.int32), cu, tm, lay_o, 0, hist=hist0.astype(np.int64))
    assert (hist_o == hist0).all()


def test_history_commit_after_a_decode_step():
    """A decode step (which rolls the history inside its gather kernel) and,
    straight after it on the stream, prefill chunks of one token per sequence:
    the chunk's history commit must build on the step's history, not on the
    one before it."""
    w, tm, lay_o, lay = setup("tiny")
    table = device_table(lay_o.layers[0].total_rows, w.seed)
    S = 6
    rng = np.random.default_rng(5)
    hist0 = rng.integers(0, w.v, size=(S, 3)).astype(np.int32)
    step_raw = rng.integers(0, w.v_raw, size=S).astype(np.int32)
    chunk_raw = rng.integers(0, w.v_raw, size=S).astype(np.int32)
    slots = np.arange(S, dtype=np.int32)
    _, _, h1 = OH.hash_step(step_raw, slots, hist0.astype(np.int64), tm, lay_o, 0)
    cu = np.arange(S + 1, dtype=np.int64)
    _, _, h2 = OH.hash_prefill(chunk_raw, cu, tm, lay_o, 0, hist=h1)
    for _ in range(3):  # back to back, several times
        hist_d = i32(hist0)
        st = status()
        eg.engram_hash_gather_step(lay, 0, i32(step_raw), i32(slots), i32(tm), table, hist_d, status=st)
        eg.engram_hash(lay, 0, i32(chunk_raw), i64(cu), i32(tm), hist_d, status=st)
        eg.engram_hash(lay, 0, i32(np.zeros(0, dtype=np.int32)), i64(np.zeros(S + 1, dtype=np.int64)), i32(tm),
                       hist_d, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert (hist_d.cpu().numpy() == h2).all()
