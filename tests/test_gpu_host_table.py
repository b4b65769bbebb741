"""Host-resident table on GB300: the gather kernel reading a pinned host table
over NVLink-C2C, and the prefetch pipeline (GPU hash -> row ids to host ->
host gather ordered on a stream -> one DMA -> dequantisation of contiguous
rows), both bit-exact against the device-table path and the oracle."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import bf16, bits, device_table, f32, i32, i64, require_gpu, setup, status
from oracle import dequant as OD
from oracle import hashing as OH
from workloads import ROW_BYTES, layer_weights, prefill_batch, residual_bits, table_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _host_table(total, seed):
    """Pinned host table filled by the device filler through the mapped pointer."""
    t = torch.empty(total * ROW_BYTES, dtype=torch.uint8, pin_memory=True)
    eg.engram_fill_synthetic_table(t, total, seed)   # device kernel writes host memory over C2C
    torch.cuda.synchronize()
    return t


def test_host_table_filled_over_c2c_matches_generator():
    total = 50_021
    t = _host_table(total, 7)
    assert (t.numpy().reshape(total, ROW_BYTES) == table_rows(7, np.arange(total))).all()


def test_zero_copy_gather_from_host_table():
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    host = _host_table(total, w.seed)
    b = prefill_batch(w)
    rows_o, _, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    st = status()
    e_host = eg.engram_gather_dequant(host, total, i32(rows_o), status=st)
    e_dev = eg.engram_gather_dequant(device_table(total, w.seed), total, i32(rows_o))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert (bits(e_host) == bits(e_dev)).all()
    ref = OD.gather_dequant(rows_o, lambda r: table_rows(w.seed, r))
    assert (bits(e_host) == OD.bf16_bits(ref)).all()


def test_prefetch_pipeline_matches_device_table():
    """Prefill batches of 4 x 4096 tokens over the 12.67 GB table kept in host
    memory, fetched ahead by EngramLayer.prefetch (two in flight), against the
    same layer over the device table: row ids equal the oracle's, e and the
    updated residual are bit-identical to the device-table path."""
    w, tm, lay_o, lay = setup("prefill")
    total = lay_o.layers[0].total_rows
    try:
        host = _host_table(total, w.seed)
    except RuntimeError as ex:  # not enough pinnable host memory on this machine
        pytest.skip(f"pinned host table unavailable: {ex}")
    lw = layer_weights(w)
    args = (i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)), f32(lw.q_w), f32(lw.k_w))
    dev_layer = eg.EngramLayer(lay, 0, device_table(total, w.seed), *args)
    host_layer = eg.EngramLayer(lay, 0, host, *args)
    batches = [prefill_batch(w, seed=s) for s in (w.seed, w.seed + 1, w.seed + 2)]
    T = len(batches[0].raw_ids)
    h_bits = residual_bits(T, w.hc, w.hidden, 3)
    copy = torch.cuda.Stream()
    st = status()
    pend = [host_layer.prefetch(i32(b.raw_ids), i64(b.cu_seqlens), status=st, copy_stream=copy)
            for b in batches[:2]]
    with pytest.raises(eg.EngramError):   # a third batch must wait for a prefill
        host_layer.prefetch(i32(batches[2].raw_ids), i64(batches[2].cu_seqlens), copy_stream=copy)
    outs = []
    for i, b in enumerate(batches):
        pf = pend.pop(0)
        h = bf16(h_bits)
        host_layer.prefill_prefetched(pf, h, st)     # the next batch's fetch is still in flight
        torch.cuda.synchronize()
        assert pf.bad_rows == 0
        h_ref = bf16(h_bits)
        buf = dev_layer.prefill(i32(b.raw_ids), i64(b.cu_seqlens), h_ref, status=st)
        torch.cuda.synchronize()
        assert (bits(pf.e) == bits(buf["e"])).all(), i
        assert (bits(h) == bits(h_ref)).all(), i
        outs.append((b, pf.row_ids.cpu().numpy(), bits(pf.e)))
        if i + 2 < len(batches):                       # reuses the slot just consumed
            pend.append(host_layer.prefetch(i32(batches[i + 2].raw_ids), i64(batches[i + 2].cu_seqlens),
                                            status=st, copy_stream=copy))
    assert int(st.item()) == 0
    b, rows, e_bits = outs[0]
    rows_o, _, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    assert (rows == rows_o).all()
    idx = np.arange(0, T, 97)
    ref = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
    assert (e_bits[idx] == OD.bf16_bits(ref)).all()


def test_fp8_prefetch_from_host_table_matches_device_table():
    """A layer with block-FP8 weights over a pinned host table (tiny layout):
    prefetch (host gather -> DMA -> rows regrouped as stored for the FP8
    projection) then prefill_prefetched gives, bit for bit, the FP8 layer's
    result over the device table."""
    from workloads import mxfp8_weights
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    host = _host_table(total, w.seed)
    K, N = 24 * 256, (w.hc + 1) * w.hidden
    w8, sfw = mxfp8_weights(K, N, 31)
    packed = eg.engram_pack_wkv_fp8(torch.from_numpy(w8).cuda(), torch.from_numpy(sfw).cuda())
    lw = layer_weights(w)
    args = (i32(tm), packed, f32(lw.q_w), f32(lw.k_w))
    dev_layer = eg.EngramLayer(lay, 0, device_table(total, w.seed), *args)
    host_layer = eg.EngramLayer(lay, 0, host, *args)
    rng = np.random.default_rng(17)
    raw = rng.integers(0, w.v_raw, size=300).astype(np.int32)
    cu = np.array([0, 120, 300], dtype=np.int64)
    h_bits = residual_bits(300, w.hc, w.hidden, 19)
    st = status()
    pf = host_layer.prefetch(i32(raw), i64(cu), status=st, copy_stream=torch.cuda.Stream())
    h = bf16(h_bits)
    host_layer.prefill_prefetched(pf, h, st)
    h_ref = bf16(h_bits)
    dev_layer.prefill(i32(raw), i64(cu), h_ref, status=st)
    torch.cuda.synchronize()
    assert pf.bad_rows == 0 and int(st.item()) == 0
    assert (bits(h) == bits(h_ref)).all()
