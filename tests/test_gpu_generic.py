"""Layouts beyond the DeepSeek-V4.1 shape: several layers hashed in one launch,
and 2/3-gram layouts with 16 columns feeding a hidden size of 2560 (the
Engram-27B shape family of the Engram paper, here with 256-dim rows)."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bits, device_table, dot_error_bound, f32, i32, i64, require_gpu,
                      residual_close, status)
from oracle import dequant as OD
from oracle import gate as OG
from oracle import hashing as OH
from oracle import layout as OL
from workloads import (WORKLOADS, Workload, bf16_bits_to_f64, layer_weights, prefill_batch, residual_bits,
                       table_rows, token_map)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def test_hash_all_layers_matches_per_layer_oracle():
    """Layers 1 and 14 from base 16,000,000 (the page's layout) in one launch."""
    w = WORKLOADS["prefill"]
    tm = token_map(w.v_raw, w.v, w.seed)
    pad = int(tm[0])
    lay_o = OL.build_layout(w.v, 16_000_000, [1, 14], pad_id=pad)
    lay = eg.build_layout(w.v, 16_000_000, [1, 14], pad_id=pad)
    b = prefill_batch(w)
    hist0 = np.full((w.n_seqs, 3), pad, dtype=np.int32)
    hist0[1, 0] = -1
    hist_d = i32(hist0)
    st = status()
    rows, mask = eg.engram_hash_all_layers(lay, i32(b.raw_ids), i64(b.cu_seqlens), i32(tm), hist_d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = rows.cpu().numpy()
    for li in range(2):
        r_o, m_o, h_o = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, li, hist=hist0.astype(np.int64))
        assert (rows[li] == r_o).all(), li
        assert (mask.cpu().numpy().astype(bool) == m_o).all()
        assert (hist_d.cpu().numpy() == h_o).all()
    # the two layers address unrelated rows
    assert not (rows[0] == rows[1]).all(axis=1).any()


@pytest.mark.parametrize("T", [300, 1700])
def test_layer_2_3_grams_16_columns_hidden_2560(T):
    """max_ngram 3, 8 heads (16 columns, K = 4096), hidden 2560, 4 streams; T = 300
    runs the two-kernel projection path, T = 1700 the fused cooperative kernel."""
    w = Workload("generic", 1300, 1000, 4099, 2, 3, T // 3, 2560, 4, 0.05)
    tm = token_map(w.v_raw, w.v, 3)
    pad = int(tm[0])
    lay_o = OL.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    lay = eg.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    assert lay.n_cols == 16
    lw = layer_weights(w, n_cols=16, seed=5)
    total = lay_o.layers[1].total_rows
    table = device_table(total, 9)
    layer = eg.EngramLayer(lay, 1, table, i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)), f32(lw.q_w), f32(lw.k_w))
    b = prefill_batch(w, seed=4)
    n = len(b.raw_ids)
    h_bits = residual_bits(n, w.hc, w.hidden, 6)
    h_d = bf16(h_bits)
    gate = torch.empty((n, w.hc), dtype=torch.float32, device=DEV)
    st = status()
    buf = layer.prefill(i32(b.raw_ids), i64(b.cu_seqlens), h_d, status=st, gate_out=gate)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_o, mask_o, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 1)
    assert (buf["rows"].cpu().numpy() == rows_o).all()
    idx = np.unique(np.concatenate([np.arange(0, n, 7), [n - 1]]))
    e = OD.gather_dequant(rows_o[idx], lambda r: table_rows(9, r))
    assert (bits(buf["e"])[idx] == OD.bf16_bits(e)).all()
    W = bf16_bits_to_f64(lw.wkv_bits)
    k, v = OG.split_kv(OG.project(e, W), w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits[idx])
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o[idx])
    out = OG.residual(hf, g, v, mask_o[idx])
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v,
                                       dot_error_bound(e, W[:, w.hc * w.hidden:]))
    assert r.ok, r


def _bf16_table(total, row_dim, seed):
    t = torch.empty((total, row_dim), dtype=torch.bfloat16, device=DEV)
    return eg.engram_fill_synthetic_rows_bf16(t, seed)


def test_bf16_row_table_fill_matches_host_generator():
    t = _bf16_table(1003, 80, 21)
    from workloads import table_rows_bf16
    assert (bits(t) == table_rows_bf16(21, np.arange(1003), 80)).all()


@pytest.mark.parametrize("row_dim", [80, 8, 256])
def test_gather_rows_bf16_copies_rows_and_flags_bad_ids(row_dim):
    from workloads import table_rows_bf16
    total, T, C = 5000, 333, 16
    table = _bf16_table(total, row_dim, 4)
    rng = np.random.default_rng(8)
    rows = rng.integers(0, total, size=(T, C)).astype(np.int32)
    rows[10, 3] = total
    rows[200, 15] = -1
    st = status()
    e = eg.engram_gather_rows_bf16(table, i32(rows), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == eg.ST_BAD_ROW
    bad = (rows < 0) | (rows >= total)
    ref = OD.gather_rows(np.clip(rows, 0, total - 1),
                         lambda r: bf16_bits_to_f64(table_rows_bf16(4, r, row_dim)))
    ref = ref.reshape(T, C, row_dim)
    ref[bad] = 0.0
    assert (bits(e).reshape(T, C, row_dim) == OD.bf16_bits(ref)).all()


@pytest.mark.parametrize("T", [300, 1700])
def test_engram_27b_shaped_layer_with_80_dim_bf16_rows(T):
    """The Engram-27B shape of the Engram paper: 2/3-grams x 8 heads = 16 rows
    of 80 bf16 elements (K = 1280) into hidden 2560, 4 streams, ragged packed
    sequences with DEAD spans, through EngramLayer with a bf16-row table
    (fused hash + copy, then the projection: two-kernel path at 300 tokens,
    fused cooperative kernel at 1700).  Rows, mask, history and e bit-exact;
    sampled gates and residuals against the oracle."""
    from workloads import table_rows_bf16
    R = 80
    w = Workload("generic27b", 1300, 1000, 4099, 2, 3, T // 3, 2560, 4, 0.05)
    tm = token_map(w.v_raw, w.v, 3)
    pad = int(tm[0])
    lay_o = OL.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    lay = eg.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    lw = layer_weights(w, n_cols=16, seed=5, row_dim=R)
    total = lay_o.layers[1].total_rows
    table = _bf16_table(total, R, 9)
    layer = eg.EngramLayer(lay, 1, table, i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)), f32(lw.q_w), f32(lw.k_w))
    b = prefill_batch(w, seed=4)
    n = len(b.raw_ids)
    h_bits = residual_bits(n, w.hc, w.hidden, 6)
    h_d = bf16(h_bits)
    hist0 = np.full((w.n_seqs, 2), pad, dtype=np.int32)
    hist0[0, 0] = 17
    hist_d = i32(hist0)
    gate = torch.empty((n, w.hc), dtype=torch.float32, device=DEV)
    st = status()
    buf = layer.prefill(i32(b.raw_ids), i64(b.cu_seqlens), h_d, hist_d, status=st, gate_out=gate)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_o, mask_o, hist_o = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 1, hist=hist0.astype(np.int64))
    assert (buf["rows"].cpu().numpy() == rows_o).all()
    assert (buf["mask"].cpu().numpy().astype(bool) == mask_o).all()
    assert (hist_d.cpu().numpy() == hist_o).all()
    e_all = OD.gather_rows(rows_o, lambda r: bf16_bits_to_f64(table_rows_bf16(9, r, R)))
    assert (bits(buf["e"]) == OD.bf16_bits(e_all)).all()
    idx = np.unique(np.concatenate([np.arange(0, n, 7), [n - 1]]))
    e = e_all[idx]
    W = bf16_bits_to_f64(lw.wkv_bits)
    k, v = OG.split_kv(OG.project(e, W), w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits[idx])
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o[idx])
    out = OG.residual(hf, g, v, mask_o[idx])
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v,
                                       dot_error_bound(e, W[:, w.hc * w.hidden:]))
    assert r.ok, r
