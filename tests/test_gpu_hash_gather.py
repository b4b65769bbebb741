"""GPU parity of the fused hash + gather (engram_hash_gather): row ids, mask
and history equal the oracle's; the dequantised rows equal the oracle's and,
bit for bit, the separate hash and gather calls."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import bits, device_table, i32, i64, require_gpu, setup, status
from oracle import dequant as OD
from oracle import hashing as OH
from workloads import DEAD, prefill_batch, table_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _fused(lay, raw, cu, tm, table, hist0=None, rows=True):
    T = len(raw)
    hist = i32(hist0) if hist0 is not None else None
    rid = torch.empty((T, lay.n_cols), dtype=torch.int32, device="cuda") if rows else None
    st = status()
    e, mask = eg.engram_hash_gather(lay, 0, i32(raw), i64(cu), i32(tm), table, hist, row_ids=rid, status=st)
    torch.cuda.synchronize()
    return (e, mask.cpu().numpy().astype(bool), None if rid is None else rid.cpu().numpy(),
            None if hist is None else hist.cpu().numpy(), int(st.item()))


def test_tiny_ragged_history_dead_all_tokens():
    w, tm, lay_o, lay = setup("tiny")
    rng = np.random.default_rng(11)
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
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    e, mask, rows, hist, st = _fused(lay, raw, cu, tm, table, hist0)
    assert st == 0
    rows_o, mask_o, hist_o = OH.hash_prefill(raw, cu, tm, lay_o, 0, hist=hist0)
    assert (rows == rows_o).all() and (mask == mask_o).all()
    assert (hist.reshape(hist_o.shape) == hist_o).all()
    ref = OD.gather_dequant(rows_o, lambda r: table_rows(w.seed, r))
    assert (bits(e) == OD.bf16_bits(ref)).all()


def test_prefill_batch_equals_separate_calls_and_oracle():
    """4 x 4096 Zipf tokens with image spans over the 12.67 GB table, with and
    without the row ids written out."""
    w, tm, lay_o, lay = setup("prefill")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    b = prefill_batch(w)
    hist0 = np.full((w.n_seqs, 3), int(tm[0]), dtype=np.int64)
    hist0[1] = [5, DEAD, 7]
    e, mask, rows, hist, st = _fused(lay, b.raw_ids, b.cu_seqlens, tm, table, hist0)
    assert st == 0
    rows_o, mask_o, hist_o = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0, hist=hist0)
    assert (rows == rows_o).all() and (mask == mask_o).all() and mask_o.any()
    assert (hist.reshape(hist_o.shape) == hist_o).all()
    # the separate calls
    r2, m2 = eg.engram_hash(lay, 0, i32(b.raw_ids), i64(b.cu_seqlens), i32(tm), i32(hist0))
    e2 = eg.engram_gather_dequant(table, total, r2)
    e3, _, none_rows, _, _ = _fused(lay, b.raw_ids, b.cu_seqlens, tm, table, hist0, rows=False)
    torch.cuda.synchronize()
    assert none_rows is None
    assert (bits(e) == bits(e2)).all() and (bits(e3) == bits(e)).all()
    idx = np.unique(np.concatenate([np.arange(0, len(rows_o), 61), [len(rows_o) - 1]]))
    ref = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
    assert (bits(e)[idx] == OD.bf16_bits(ref)).all()


def test_bad_tokens_masked_and_flagged():
    w, tm, lay_o, lay = setup("tiny")
    table = device_table(lay_o.layers[0].total_rows, w.seed)
    raw = np.array([5, w.v_raw, 7, -5, 9], dtype=np.int32)
    _, mask, _, _, st = _fused(lay, raw, np.array([0, 5]), tm, table)
    assert st & eg.ST_BAD_TOKEN
    assert list(mask) == [False, True, False, True, False]


def test_empty_batch_commits_history_only():
    w, tm, lay_o, lay = setup("tiny")
    table = device_table(lay_o.layers[0].total_rows, w.seed)
    hist0 = np.array([[3, 4, 5], [6, DEAD, 8]], dtype=np.int64)
    e, mask, _, hist, st = _fused(lay, np.zeros(0, np.int32), np.array([0, 0, 0]), tm, table, hist0, rows=False)
    assert st == 0 and e.shape[0] == 0
    assert (hist == hist0).all()


def test_decode_step_fused_equals_oracle_and_separate_calls():
    """engram_hash_gather_step (bf16) and its FP8 variant over 6 decode steps:
    row ids, mask and rolled history equal the oracle's decode step; the rows
    equal the oracle's dequantised rows and, bit for bit, engram_hash_step +
    engram_gather_dequant / engram_gather_fp8.  Entry 3 is padding (slot -1),
    entry 5 names slot 40 of 12 (ST_BAD_SLOT, treated as padding), and the
    slots are a permutation, so entries do not hit their own rows."""
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    S, B = 12, 9
    rng = np.random.default_rng(11)
    hist0 = rng.integers(0, w.v, size=(S, 3)).astype(np.int64)
    hist0[2, 1] = DEAD                      # a DEAD entry carried in the history
    slots = rng.permutation(S)[:B].astype(np.int32)
    slots[3] = -1
    slots[5] = 40
    H = hist0.copy()
    h_fused, h_sep, h_fp8 = i32(hist0), i32(hist0), i32(hist0)
    st_f, st_s, st_8 = status(), status(), status()
    for step in range(6):
        raw = rng.integers(0, w.v_raw, size=B).astype(np.int32)
        if step == 2:
            raw[0] = DEAD                   # an image position
        slots_o = slots.copy()
        slots_o[5] = -1                     # what the kernel does with the bad slot
        rows_o, mask_o, H = OH.hash_step(raw, slots_o, H, tm, lay_o, 0)
        rid = torch.empty((B, lay.n_cols), dtype=torch.int32, device="cuda")
        e, mask = eg.engram_hash_gather_step(lay, 0, i32(raw), i32(slots), i32(tm), table, h_fused, row_ids=rid,
                                             status=st_f)
        rows_s, mask_s = eg.engram_hash_step(lay, 0, i32(raw), i32(slots), i32(tm), h_sep, status=st_s)
        e_s = eg.engram_gather_dequant(table, total, rows_s)
        rid8 = torch.empty((B, lay.n_cols), dtype=torch.int32, device="cuda")
        e8, sf, mask8 = eg.engram_hash_gather_step_fp8(lay, 0, i32(raw), i32(slots), i32(tm), table, h_fp8,
                                                       row_ids=rid8, status=st_8)
        e8_s, sf_s = eg.engram_gather_fp8(table, total, rows_s)
        torch.cuda.synchronize()
        assert (rid.cpu().numpy() == rows_o).all(), step
        assert (mask.cpu().numpy().astype(bool) == mask_o).all(), step
        assert (h_fused.cpu().numpy() == H).all(), step
        assert (bits(e) == bits(e_s)).all(), step
        ref = OD.gather_dequant(rows_o, lambda r: table_rows(w.seed, r))
        assert (OD.bf16_bits(ref) == bits(e)).all(), step
        assert (rid8.cpu().numpy() == rows_o).all() and (mask8.cpu().numpy() == mask.cpu().numpy()).all()
        assert (e8.cpu().numpy() == e8_s.cpu().numpy()).all() and (sf.cpu().numpy() == sf_s.cpu().numpy()).all()
        assert (h_fp8.cpu().numpy() == H).all() and (h_sep.cpu().numpy() == H).all()
    for st in (st_f, st_s, st_8):
        assert int(st.item()) == eg.ST_BAD_SLOT
