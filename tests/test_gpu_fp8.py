"""GPU parity of the block-scaled FP8 path ([P-O1] §2.3: block-FP8 weights,
E4M3 + E8M0 table payload): the gather that copies the rows as stored, the
repacking of the FP8 weights, and the tcgen05 kind::mxf8f6f4 projection with
the gate and residual against the fp64 oracle on the exact dequantised
values (the tolerance is the bf16 path's: fp32 accumulation bound)."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bits, device_table, dot_error_bound, f32, i32, i64, require_gpu,
                      residual_close, setup, status, u8)
from oracle import dequant as OD
from oracle import gate as OG
from oracle import hashing as OH
from workloads import (ROW_BYTES, bf16_bits_to_f64, layer_weights, mxfp8_weights, prefill_batch, residual_bits,
                       table_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _sf_bytes(sf_words: torch.Tensor) -> np.ndarray:
    """int32 [2C][T128] words -> uint8 [2C][T128][4]."""
    return sf_words.cpu().numpy().view(np.uint8).reshape(sf_words.shape[0], sf_words.shape[1], 4)


def _sf_perm(i: np.ndarray) -> np.ndarray:
    """Documented word order of a block-FP8 scale row: within each 128 words,
    word 4 r + c holds position (or column) r + 32 c."""
    return (i // 128) * 128 + (i % 32) * 4 + (i % 128) // 32


def test_gather_fp8_copies_rows_and_groups_scales():
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    rng = np.random.default_rng(3)
    T = 77
    rows = rng.integers(0, total, size=(T, 24)).astype(np.int32)
    rows[5, 3] = total          # bad
    rows[60, 0] = -2            # bad
    st = status()
    e8, sf = eg.engram_gather_fp8(table, total, i32(rows), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & eg.ST_BAD_ROW
    ref = table_rows(w.seed, np.clip(rows, 0, total - 1).reshape(-1)).reshape(T, 24, ROW_BYTES)
    bad = (rows < 0) | (rows >= total)
    ref_w = ref[:, :, :256].copy()
    ref_s = ref[:, :, 256:].copy()
    ref_w[bad] = 0
    ref_s[bad] = 127
    assert (e8.cpu().numpy().reshape(T, 24, 256) == ref_w).all()
    T128 = (T + 127) // 128 * 128
    assert tuple(sf.shape) == (48, T128)
    sb = _sf_bytes(sf)                                         # [48][T128][4]
    got_s = sb[:, _sf_perm(np.arange(T))].reshape(24, 2, T, 4).transpose(2, 0, 1, 3).reshape(T, 24, 8)
    assert (got_s == ref_s).all()
    # positions T .. T128-1 of the last 128-block hold scale 127 (the value 1)
    assert (sb[:, _sf_perm(np.arange(T, T128))] == 127).all()
    # a permutation of each 128-block: every word is some position's
    assert sorted(_sf_perm(np.arange(T128)).tolist()) == list(range(T128))


def test_hash_gather_fp8_matches_hash_and_gather():
    w, tm, lay_o, lay = setup("prefill")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    b = prefill_batch(w)
    rid = torch.empty((len(b.raw_ids), 24), dtype=torch.int32, device=DEV)
    e8, sf, mask = eg.engram_hash_gather_fp8(lay, 0, i32(b.raw_ids), i64(b.cu_seqlens), i32(tm), table,
                                             row_ids=rid)
    rows_o, mask_o, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    assert (rid.cpu().numpy() == rows_o).all() and (mask.cpu().numpy().astype(bool) == mask_o).all()
    e8b, sfb = eg.engram_gather_fp8(table, total, rid)
    torch.cuda.synchronize()
    assert (e8.cpu().numpy() == e8b.cpu().numpy()).all() and (sf.cpu().numpy() == sfb.cpu().numpy()).all()


def test_pack_wkv_fp8_layout():
    K, N = 384, 640
    w8, sf = mxfp8_weights(K, N, 4)
    w8p, sfp = eg.engram_pack_wkv_fp8(u8(w8), u8(sf))
    torch.cuda.synchronize()
    got = w8p.cpu().numpy()
    k, n = np.meshgrid(np.arange(K), np.arange(N), indexing="ij")
    idx = (((n // 128) * (K // 128) + k // 128) * 128 + n % 128) * 128 + k % 128
    assert (got[idx] == w8).all()
    words = sfp.cpu().numpy().view(np.uint8).reshape(K // 128, N, 4)
    assert (words[:, _sf_perm(np.arange(N))] == sf.reshape(K // 128, 4, N).transpose(0, 2, 1)).all()


def _fp8_layer_case(name, T_cut=None, seed=0, sample=None):
    w, tm, lay_o, lay = setup(name)
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    b = prefill_batch(w)
    raw, cu = b.raw_ids, b.cu_seqlens
    if T_cut is not None:          # a shorter or longer batch from the same generator
        reps = -(-T_cut // len(raw))
        raw = np.tile(raw, reps)[:T_cut]
        cu = np.array([0, T_cut], dtype=np.int64)
    T = len(raw)
    K = 24 * 256
    N = (w.hc + 1) * w.hidden
    w8, sfw = mxfp8_weights(K, N, 7 + seed)
    w8p, sfb = eg.engram_pack_wkv_fp8(u8(w8), u8(sfw))
    lw = layer_weights(w)
    rid = torch.empty((T, 24), dtype=torch.int32, device=DEV)
    e8, sfa, mask = eg.engram_hash_gather_fp8(lay, 0, i32(raw), i64(cu), i32(tm), table, row_ids=rid)
    h_bits = residual_bits(T, w.hc, w.hidden, 11 + seed)
    h = bf16(h_bits)
    gate = torch.empty((T, w.hc), dtype=torch.float32, device=DEV)
    st = status()
    eg.engram_project_gate_fp8(e8, sfa, w8p, sfb, h, f32(lw.q_w), f32(lw.k_w), mask, gate_out=gate, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_o, mask_o, _ = OH.hash_prefill(raw, cu, tm, lay_o, 0)
    assert (rid.cpu().numpy() == rows_o).all()
    idx = np.arange(T) if sample is None else np.unique(np.concatenate([np.arange(0, T, sample), [T - 1]]))
    e = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
    W = OD.dequant_mx_weights(w8, sfw)
    k, v = OG.split_kv(OG.project(e, W), w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits[idx])
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o[idx])
    out = OG.residual(hf, g, v, mask_o[idx])
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h)[idx]), out, hf, g, v,
                                       dot_error_bound(e, W[:, w.hc * w.hidden:]))
    assert r.ok, r


@pytest.mark.parametrize("T", [128, 300, 1])
def test_fp8_layer_two_kernel_path(T):
    """tiny layout (hidden 256, N 1280): projection + separate gate kernel."""
    _fp8_layer_case("tiny", T_cut=T)


def test_fp8_layer_1700_tokens():
    """1700 tokens (ragged M tail): the FP8 projection and the gate kernel, or the
    fused cooperative FP8 kernel when engram_kernel_options.fp8_fused is set."""
    _fp8_layer_case("tiny", T_cut=1700, seed=1)


def test_fp8_layer_prefill_sampled():
    """The prefill batch (16,384 tokens, hidden 5120) through the FP8 path, every 61st token."""
    _fp8_layer_case("prefill", sample=61, seed=2)


@pytest.mark.parametrize("T", [256, 37])
def test_fp8_layer_decode_size(T):
    """Decode-size batches at hidden 5120 through the two-kernel FP8 path, every 16th token."""
    _fp8_layer_case("prefill", T_cut=T, sample=16, seed=3)


def test_engram_layer_with_fp8_weights_prefill_and_decode():
    """EngramLayer built with (w8p, sfb) from engram_pack_wkv_fp8: prefill of a
    ragged batch against the oracle, then decode steps bit for bit against the
    direct calls (fused FP8 decode step + FP8 projection and gate)."""
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    K, N = 24 * 256, (w.hc + 1) * w.hidden
    w8, sfw = mxfp8_weights(K, N, 21)
    w8p, sfb = eg.engram_pack_wkv_fp8(u8(w8), u8(sfw))
    lw = layer_weights(w)
    layer = eg.EngramLayer(lay, 0, table, i32(tm), (w8p, sfb), f32(lw.q_w), f32(lw.k_w))
    rng = np.random.default_rng(12)
    lens = [1, 150, 149]
    raw = rng.integers(0, w.v_raw, size=sum(lens)).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = len(raw)
    h_bits = residual_bits(T, w.hc, w.hidden, 13)
    h = bf16(h_bits)
    gate = torch.empty((T, w.hc), dtype=torch.float32, device=DEV)
    hist = i32(np.full((3, 3), lay.pad_id))
    st = status()
    layer.prefill(i32(raw), i64(cu), h, hist, status=st, gate_out=gate)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_o, mask_o, hist_o = OH.hash_prefill(raw, cu, tm, lay_o, 0)
    assert (hist.cpu().numpy() == hist_o).all()
    e = OD.gather_dequant(rows_o, lambda r: table_rows(w.seed, r))
    W = OD.dequant_mx_weights(w8, sfw)
    k, v = OG.split_kv(OG.project(e, W), w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits)
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o)
    out = OG.residual(hf, g, v, mask_o)
    assert np.abs(gate.cpu().numpy() - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h)), out, hf, g, v,
                                       dot_error_bound(e, W[:, w.hc * w.hidden:]))
    assert r.ok, r
    # decode: the layer against the direct calls, from the same history
    slots = i32(np.array([2, 0, 1], dtype=np.int32))
    hist_d = hist.clone()
    h_l = bf16(residual_bits(3, w.hc, w.hidden, 14))
    h_d = h_l.clone()
    work = eg.project_gate_workspace(3, w.hidden, w.hc, DEV)
    for step in range(3):
        new = i32(rng.integers(0, w.v_raw, size=3).astype(np.int32))
        layer.decode(new, slots, hist, h_l, status=st)
        e8, sf, m = eg.engram_hash_gather_step_fp8(lay, 0, new, slots, i32(tm), table, hist_d)
        eg.engram_project_gate_fp8(e8, sf, w8p, sfb, h_d, f32(lw.q_w), f32(lw.k_w), m, workspace=work)
        torch.cuda.synchronize()
        assert (bits(h_l) == bits(h_d)).all(), step
        assert (hist.cpu().numpy() == hist_d.cpu().numpy()).all(), step
    assert int(st.item()) == 0
