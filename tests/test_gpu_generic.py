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
    ok, worst, strict = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v,
                                       dot_error_bound(e, W[:, w.hc * w.hidden:]))
    assert ok, (worst, strict)
