"""Pins of the oracle's projection, gate and residual add."""
import numpy as np
import pytest

from oracle import dequant as D
from oracle import gate as G
from oracle import hashing as Hs
from oracle import layout as L
from oracle import pipeline as P
from workloads import (WORKLOADS, bf16_bits_to_f64, layer_weights, prefill_batch, residual_bits,
                       table_rows, token_map)

SIG = lambda z: 1.0 / (1.0 + np.exp(-z))  # noqa: E731


def _unit(H, hc, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((1, hc, H))


@pytest.mark.parametrize("H", [256, 5120])
def test_aligned_opposite_orthogonal(H):
    """q_w = k_w = 1: s = sqrt(H) cos(theta) ([P-V41] §除以√d), so k = c h gives s = sqrt(H)."""
    hc = 4
    h = _unit(H, hc, 0)
    ones = np.ones((H, hc))
    no = np.zeros(1, dtype=bool)
    g_par = G.gate(h, 3.0 * h, ones, ones, no, eps=0.0)
    g_anti = G.gate(h, -0.5 * h, ones, ones, no, eps=0.0)
    np.testing.assert_allclose(g_par, SIG(H ** 0.25), rtol=1e-12)
    np.testing.assert_allclose(g_anti, SIG(-H ** 0.25), rtol=1e-12)
    # orthogonal key (disjoint supports, dot exactly +0): the clamp makes the
    # gate sigmoid(+sqrt(clamp)); copysign(., +0) is positive
    hs = h.copy()
    hs[..., H // 2:] = 0.0
    k = np.random.default_rng(1).standard_normal((1, hc, H))
    k[..., : H // 2] = 0.0
    g_orth = G.gate(hs, k, ones, ones, no, eps=0.0, clamp=1e-6)
    np.testing.assert_allclose(g_orth, SIG(1e-3), atol=1e-12)


def test_score_range_and_scale_71_6():
    """|s| <= sqrt(d) with unit weights; at d = 5120 the extreme is 71.6."""
    H = 5120
    assert round(H ** 0.5, 1) == 71.6
    rng = np.random.default_rng(2)
    h = rng.standard_normal((64, 4, H))
    k = rng.standard_normal((64, 4, H)) + 0.3 * h
    ones = np.ones((H, 4))
    g = G.gate(h, k, ones, ones, np.zeros(64, bool), eps=0.0)
    z = np.log(g / (1 - g))                       # signed sqrt of s
    assert (np.abs(z) <= H ** 0.25 + 1e-9).all()
    # unrelated vectors: s has standard deviation about 1
    g0 = G.gate(h, rng.standard_normal((64, 4, H)), ones, ones, np.zeros(64, bool), eps=0.0)
    z0 = np.log(g0 / (1 - g0))
    s0 = np.sign(z0) * z0 ** 2
    assert 0.6 < np.std(s0) < 1.5


def test_weights_scale_each_stream():
    """q_w * k_w enters the dot elementwise per stream ([P-DS4] §消费)."""
    H, hc = 256, 4
    rng = np.random.default_rng(3)
    h = rng.standard_normal((2, hc, H))
    k = rng.standard_normal((2, hc, H))
    qw = np.ones((H, hc))
    kw = np.ones((H, hc))
    qw[:, 2] = 2.0                               # doubles stream 2's dot only
    base = G.gate(h, k, np.ones((H, hc)), np.ones((H, hc)), np.zeros(2, bool), eps=0.0)
    twice = G.gate(h, k, qw, kw, np.zeros(2, bool), eps=0.0)
    zb = np.log(base / (1 - base))
    zt = np.log(twice / (1 - twice))
    np.testing.assert_allclose(zt[:, [0, 1, 3]], zb[:, [0, 1, 3]], rtol=1e-12)
    np.testing.assert_allclose(np.sign(zt[:, 2]) * zt[:, 2] ** 2, 2 * np.sign(zb[:, 2]) * zb[:, 2] ** 2,
                               rtol=1e-9)


def test_masked_gate_zero_and_h_untouched():
    H, hc = 256, 4
    rng = np.random.default_rng(4)
    hb = rng.integers(0, 2 ** 16, size=(3, hc, H), dtype=np.uint64).astype(np.uint16)
    hb[(hb & 0x7F80) == 0x7F80] = 0x8000          # avoid NaN/inf patterns; keep a -0
    h = bf16_bits_to_f64(hb)
    k = rng.standard_normal((3, hc, H))
    v = rng.standard_normal((3, H)) * 100
    mask = np.array([False, True, False])
    g = G.gate(h, k, np.ones((H, hc)), np.ones((H, hc)), mask)
    assert (g[1] == 0).all() and (g[[0, 2]] > 0).all()
    out = G.residual(h, g, v, mask)
    assert (D.bf16_bits(out[1]) == hb[1]).all()
    # unmasked rows: bf16(h + g bf16(v)) against a per-element re-derivation via fp32 ties
    assert not (D.bf16_bits(out[0]) == hb[0]).all()


def test_zero_gate_keeps_h():
    H, hc = 256, 4
    rng = np.random.default_rng(5)
    h = bf16_bits_to_f64(rng.integers(0, 0x3F00, size=(2, hc, H)).astype(np.uint16))
    out = G.residual(h, np.zeros((2, hc)), rng.standard_normal((2, H)), np.zeros(2, bool))
    assert (out == h).all()


def test_projection_block_order():
    """kv = e @ wkv; keys k^(1..4) first, then v: a one-hot e selects one wkv row."""
    H, hc, K = 8, 4, 16
    W = np.arange(K * (hc + 1) * H, dtype=np.float64).reshape(K, (hc + 1) * H)
    e = np.zeros((1, K))
    e[0, 5] = 1.0
    kv = G.project(e, W)
    k, v = G.split_kv(kv, H, hc)
    for m in range(hc):
        assert (k[0, m] == W[5, m * H:(m + 1) * H]).all()
    assert (v[0] == W[5, hc * H:]).all()


def test_tiny_pipeline_runs_and_is_consistent():
    w = WORKLOADS["tiny"]
    tm = token_map(w.v_raw, w.v, 0)
    lay = L.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    b = prefill_batch(w)
    lw = layer_weights(w)
    h = bf16_bits_to_f64(residual_bits(w.tokens, w.hc, w.hidden, 0))
    res = P.layer_forward(lay, 0, b.raw_ids, b.cu_seqlens, tm, lambda r: table_rows(0, r),
                          bf16_bits_to_f64(lw.wkv_bits), h, lw.q_w, lw.k_w)
    assert res.e.shape == (w.tokens, 6144)
    assert res.gate.shape == (w.tokens, w.hc)
    assert ((res.gate > 0) & (res.gate < 1)).all()
    assert np.isfinite(res.h_out).all()
    # the e of a token is the concatenation of its 24 dequantised rows
    t = 17
    direct = D.dequant_rows(table_rows(0, res.rows[t]))
    assert (res.e[t].reshape(24, 256) == direct).all()


def test_decode_step_equals_prefill_of_prefix_plus_token():
    """Three sequences (prefix lengths 0, 2, 9): a decode step from the
    prefill-carried history gives the rows, mask, gate and residual of the
    last position of prefill over prefix + token."""
    w = WORKLOADS["tiny"]
    tm = token_map(w.v_raw, w.v, 0)
    lay = L.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    lw = layer_weights(w)
    W = bf16_bits_to_f64(lw.wkv_bits)
    rng = np.random.default_rng(5)
    lens = [0, 2, 9]
    prefixes = [rng.integers(0, w.v_raw, size=n).astype(np.int64) for n in lens]
    new = rng.integers(0, w.v_raw, size=3).astype(np.int64)
    h = bf16_bits_to_f64(residual_bits(3, w.hc, w.hidden, 9))
    cu = np.concatenate([[0], np.cumsum(lens)])
    _, _, hist = Hs.hash_prefill(np.concatenate(prefixes), cu, tm, lay, 0)
    # history slot i holds sequence perm[i]; entry b names the slot of sequence b
    perm = np.array([1, 2, 0])
    slots = np.argsort(perm)
    step = P.layer_decode_step(lay, 0, new, slots, hist[perm], tm, lambda r: table_rows(0, r), W, h, lw.q_w, lw.k_w)
    for b in range(3):
        seq = np.concatenate([prefixes[b], [new[b]]])
        full = P.layer_forward(lay, 0, seq, np.array([0, len(seq)]), tm, lambda r: table_rows(0, r), W,
                               np.repeat(h[b:b + 1], len(seq), axis=0), lw.q_w, lw.k_w)
        assert (step.rows[b] == full.rows[-1]).all() and step.mask[b] == full.mask[-1]
        assert (step.e[b] == full.e[-1]).all()
        # the fp64 GEMM of one row and of a batch may round differently in the last bits
        assert np.abs(step.gate[b] - full.gate[-1]).max() <= 1e-12
        d = np.abs(step.h_out[b] - full.h_out[-1])
        assert (d <= 2.0 ** -7 * np.abs(full.h_out[-1])).all() and (d == 0).mean() > 0.999


def test_residual_rounds_v_before_the_product_worked_example():
    """A hand-worked case where rounding v to bf16 first decides the result
    (the residual uses bf16(v), and h + g bf16(v) is rounded once):
    h = 1, g = 1/2, v = 3 + 2^-6 + 2^-20.  bf16(v) = 3 + 2^-6, so the sum is
    2.5 + 2^-7, exactly half a bf16 step (2^-6) above 2.5: a tie, which goes
    to the even significand, 2.5.  With v unrounded the sum would sit above
    the tie and round up to 2.5 + 2^-6."""
    H, hc = 256, 1
    h = np.ones((1, hc, H))
    g = np.full((1, hc), 0.5)
    v = np.full((1, H), 3 + 2.0 ** -6 + 2.0 ** -20)
    out = G.residual(h, g, v, np.zeros(1, bool))
    assert (out == 2.5).all()
    assert (D.bf16_round(np.float64(3 + 2.0 ** -6 + 2.0 ** -20)) == 3 + 2.0 ** -6)
