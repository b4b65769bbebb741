"""End-to-end GPU parity of one Engram layer (hash -> gather -> project -> gate/add)
on the tiny, layer-prefill and decode workloads."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bits, device_table, dot_error_bound, f32, i32, i64, require_gpu,
                      residual_close, setup, status, v_flips_explained)
from oracle import dequant as OD
from oracle import gate as OG
from oracle import hashing as OH
from workloads import (bf16_bits_to_f64, decode_workload, layer_weights, normal_bf16_bits, prefill_batch,
                       residual_bits, table_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _make_layer(name, fused=True):
    w, tm, lay_o, lay = setup(name)
    lw = layer_weights(w)
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    layer = eg.EngramLayer(lay, 0, table, i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)), f32(lw.q_w),
                           f32(lw.k_w), fused=fused)
    return w, tm, lay_o, lay, lw, layer


def _oracle_tokens(w, lay_o, lw, W, rows_o, mask_o, h_bits, idx):
    """Oracle e, gate, v and h_out for the positions idx (rows from the oracle hash).

    W is wkv widened to float64 once per test."""
    e = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
    kv = OG.project(e, W)
    k, v = OG.split_kv(kv, w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits[idx])
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o[idx])
    out = OG.residual(hf, g, v, mask_o[idx])
    v_err = dot_error_bound(e, W[:, w.hc * w.hidden:])
    return e, g, v, hf, out, v_err


def _check_layer(name, idx_fn, fused=True):
    w, tm, lay_o, lay, lw, layer = _make_layer(name, fused)
    b = prefill_batch(w)
    T = len(b.raw_ids)
    h_bits = residual_bits(T, w.hc, w.hidden, w.seed)
    rows_o, mask_o, hist_o = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    h_d = bf16(h_bits)
    hist_d = i32(np.full((w.n_seqs, 3), lay.pad_id))
    gate = torch.empty((T, w.hc), dtype=torch.float32, device=DEV)
    st = status()
    buf = layer.prefill(i32(b.raw_ids), i64(b.cu_seqlens), h_d, hist_d, status=st, gate_out=gate)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert (buf["rows"].cpu().numpy() == rows_o).all()
    assert (buf["mask"].cpu().numpy().astype(bool) == mask_o).all()
    assert (hist_d.cpu().numpy() == hist_o).all()
    idx = idx_fn(T, mask_o, b.cu_seqlens)
    e, g, v, hf, out, v_err = _oracle_tokens(w, lay_o, lw, bf16_bits_to_f64(lw.wkv_bits), rows_o, mask_o, h_bits,
                                             idx)
    assert (bits(buf["e"])[idx] == OD.bf16_bits(e)).all()
    gg = gate.cpu().numpy()[idx]
    assert np.abs(gg - g).max() <= GATE_ATOL
    hb = bits(h_d)[idx]
    assert (hb[mask_o[idx]] == h_bits[idx][mask_o[idx]]).all()
    if not fused:
        v_flips_explained(bits(buf["v"]).reshape(T, w.hidden)[idx], v, v_err)
    r = residual_close(bf16_bits_to_f64(hb), out, hf, g, v, v_err)
    assert r.ok, r


@pytest.mark.parametrize("fused", [True, False])
def test_layer_tiny_all_tokens(fused):
    _check_layer("tiny", lambda T, m, cu: np.arange(T), fused)


def test_layer_prefill_sampled():
    """4 x 4096 Zipf tokens with 5% DEAD spans, hidden 5120: sampled positions incl.
    sequence boundaries and positions on both sides of image spans."""
    def idx_fn(T, mask, cu):
        rng = np.random.default_rng(5)
        edges = np.flatnonzero(np.diff(mask.astype(np.int8)) != 0)
        pick = [rng.integers(0, T, 48), cu[:-1], cu[1:] - 1, edges[:8], edges[:8] + 1]
        return np.unique(np.concatenate(pick).astype(np.int64))
    _check_layer("prefill", idx_fn)


def test_layer_decode_steps():
    """256 sequences, histories from their prefixes; steps 0-9 and every 100th of 1000
    checked against the oracle, each with a fresh residual."""
    w, tm, lay_o, lay, lw, layer = _make_layer("decode")
    dw = decode_workload(w)
    pre = dw.prefix
    S = w.n_seqs
    _, _, H = OH.hash_prefill(pre.raw_ids, pre.cu_seqlens, tm, lay_o, 0)
    hist_d = i32(np.full((S, 3), lay.pad_id))
    eg.engram_hash(lay, 0, i32(pre.raw_ids), i64(pre.cu_seqlens), i32(tm), hist_d)
    slots = np.arange(S, dtype=np.int32)
    slots_d = i32(slots)
    check = set(range(10)) | set(range(0, dw.steps.shape[0], 100))
    W = bf16_bits_to_f64(lw.wkv_bits)
    gate = torch.empty((S, w.hc), dtype=torch.float32, device=DEV)
    st = status()
    for step in range(dw.steps.shape[0]):
        raw = dw.steps[step]
        h_bits = normal_bf16_bits((S, w.hc, w.hidden), 1.0, w.seed, 1000 + step) if step in check else None
        h_d = bf16(h_bits) if h_bits is not None else torch.zeros((S, w.hc, w.hidden), dtype=torch.bfloat16,
                                                                 device=DEV)
        buf = layer.decode(i32(raw), slots_d, hist_d, h_d, status=st, gate_out=gate)
        rows_o, mask_o, H = OH.hash_step(raw, slots, H, tm, lay_o, 0)
        if step in check:
            torch.cuda.synchronize()
            assert (buf["rows"].cpu().numpy() == rows_o).all()
            idx = np.arange(S)
            e, g, v, hf, out, v_err = _oracle_tokens(w, lay_o, lw, W, rows_o, mask_o, h_bits, idx)
            assert (bits(buf["e"]) == OD.bf16_bits(e)).all()
            assert np.abs(gate.cpu().numpy() - g).max() <= GATE_ATOL
            r = residual_close(bf16_bits_to_f64(bits(h_d)), out, hf, g, v, v_err)
            assert r.ok, (step, r)
    torch.cuda.synchronize()
    assert (hist_d.cpu().numpy() == H).all()
    assert int(st.item()) == 0


@pytest.mark.parametrize("conv", [False, True])
def test_decode_graph_replays_equal_eager_steps(conv):
    """A captured decode step replayed for 6 steps (new raw ids written in
    place each time, one padding entry) gives bit for bit the residual, gates,
    history (and short-convolution state) of eager EngramLayer.decode calls."""
    w, tm, lay_o, lay, lw, layer = _make_layer("tiny")
    if conv:
        from workloads import conv_weights
        cw, gamma = conv_weights(4, w.hc, w.hidden, w.seed)
        layer = eg.EngramLayer(lay, 0, layer.table, layer.token_map, layer.wkv_packed, layer.q_w, layer.k_w,
                               conv=eg.ShortConv(f32(cw), f32(gamma), 3))
    B, S = 37, 40
    rng = np.random.default_rng(3)
    hist0 = i32(rng.integers(0, w.v, size=(S, 3)))
    h0 = bf16(normal_bf16_bits((B, w.hc, w.hidden), 1.0, 5, 1))
    slots = rng.permutation(S)[:B].astype(np.int32)
    slots[7] = -1
    states = []
    for _ in range(2):
        cs = layer.new_conv_state(S, DEV) if conv else None
        states.append((hist0.clone(), h0.clone(), torch.empty((B, w.hc), dtype=torch.float32, device=DEV),
                       status(), cs))
    hist_e, h_e, g_e, st_e, cs_e = states[0]
    hist_g, h_g, g_g, st_g, cs_g = states[1]
    graph = layer.decode_graph(B, hist_g, h_g, st_g, g_g, cs_g)
    graph.slots.copy_(i32(slots))
    for step in range(6):
        raw = rng.integers(0, w.v_raw, size=B).astype(np.int32)
        layer.decode(i32(raw), i32(slots), hist_e, h_e, st_e, g_e, cs_e)
        graph.raw_ids.copy_(i32(raw))
        graph.replay()
        torch.cuda.synchronize()
        assert (bits(h_g) == bits(h_e)).all(), step
        assert (g_g.cpu().numpy() == g_e.cpu().numpy()).all(), step
        assert (hist_g.cpu().numpy() == hist_e.cpu().numpy()).all(), step
        if conv:
            assert (cs_g[0].cpu().numpy() == cs_e[0].cpu().numpy()).all(), step
            assert (cs_g[1].cpu().numpy() == cs_e[1].cpu().numpy()).all(), step
    assert int(st_e.item()) == 0 and int(st_g.item()) == 0
