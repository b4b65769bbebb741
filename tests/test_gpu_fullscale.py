"""Full-scale parity: a 384,006,168-row (101.4 GB) table from base 16,000,000,
131,072 Zipf tokens prefilled in 8 chunks of 16,384 with the 3-id history
carried between chunks, hidden 5120, 4 streams.

Row ids are compared bit-exactly on every token (the oracle hashes the whole
sequence in one pass, so chunk boundaries test the history carry); dequantised
rows, gates and residuals on a sample: every 16th token plus the first and
last three tokens of every chunk.
"""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bits, device_table, dot_error_bound, f32, i32, i64, require_gpu,
                      residual_close, setup, status)
from oracle import dequant as OD
from oracle import gate as OG
from oracle import hashing as OH
from workloads import bf16_bits_to_f64, layer_weights, prefill_batch, residual_bits, table_rows

pytestmark = pytest.mark.gpu


def test_fullscale_chunked_prefill():
    require_gpu()
    w, tm, lay_o, lay = setup("fullscale")
    total = lay_o.layers[0].total_rows
    assert total == 384_006_168
    free, _ = torch.cuda.mem_get_info()
    if free < total * 264 + (8 << 30):
        pytest.skip("needs ~110 GB of free device memory")
    table = device_table(total, w.seed)
    lw = layer_weights(w)
    layer = eg.EngramLayer(lay, 0, table, i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)), f32(lw.q_w),
                           f32(lw.k_w))
    b = prefill_batch(w)
    T = len(b.raw_ids)
    C = T // w.chunks
    h_bits = residual_bits(C, w.hc, w.hidden, w.seed)      # the same residual enters every chunk
    h0 = bf16(h_bits)
    hist = i32(np.full((1, 3), lay.pad_id))
    st = status()
    rows_all = np.empty((T, 24), dtype=np.int64)
    sample = {}
    for c in range(w.chunks):
        raw = b.raw_ids[c * C:(c + 1) * C]
        h = h0.clone()
        gate = torch.empty((C, w.hc), dtype=torch.float32, device=DEV)
        buf = layer.prefill(i32(raw), i64([0, C]), h, hist, status=st, gate_out=gate)
        torch.cuda.synchronize()
        rows_all[c * C:(c + 1) * C] = buf["rows"].cpu().numpy()
        local = np.unique(np.concatenate([np.arange(0, C, 16), [0, 1, 2, C - 3, C - 2, C - 1]]))
        sample[c] = (local, bits(buf["e"][torch.from_numpy(local).to(DEV)]), gate.cpu().numpy()[local],
                     bits(h)[local])
    assert int(st.item()) == 0
    del table
    torch.cuda.empty_cache()

    rows_o, mask_o, hist_o = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    assert (rows_all == rows_o).all()
    assert (hist.cpu().numpy() == hist_o).all()
    W = bf16_bits_to_f64(lw.wkv_bits)
    Wv = W[:, w.hc * w.hidden:]
    for c, (local, e_gpu, g_gpu, h_gpu) in sample.items():
        idx = c * C + local
        e = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
        assert (e_gpu == OD.bf16_bits(e)).all(), c
        kv = OG.project(e, W)
        k, v = OG.split_kv(kv, w.hidden, w.hc)
        hf = bf16_bits_to_f64(h_bits[local])
        g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o[idx])
        out = OG.residual(hf, g, v, mask_o[idx])
        gerr = np.abs(g_gpu - g)
        assert gerr.max() <= GATE_ATOL, c
        r = residual_close(bf16_bits_to_f64(h_gpu), out, hf, g, v, dot_error_bound(e, Wv))
        assert r.ok, f"chunk {c}: {r} gate_err_max={float(gerr.max())}"
