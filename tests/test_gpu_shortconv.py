"""GPU parity of the short causal convolution (the original Engram layer's
branch, [P-DETAIL] §4.2) against the oracle: packed prefill with ragged
sequences and image spans, chunked prefill with the carried state, decode
steps with padding entries, several kernel sizes and dilations, and the
whole layer (hash -> gather -> projection -> gates -> convolution).

Tolerance: the device evaluates in fp32 and rounds once to bf16.  A result
passes when it is the bf16 rounding of some value within a stated bound of
the exact (fp64) sum; the bound is the fp32 evaluation error, plus, for the
whole layer, what the gate and v differences of the earlier stages carry in.
"""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bf16_flip, bits, device_table, dot_error_bound, f32, i32, i64,
                      require_gpu, status)
from oracle import dequant as OD
from oracle import gate as OG
from oracle import hashing as OH
from oracle import layout as OL
from oracle import shortconv as SC
from workloads import (DEAD, Workload, bf16_bits_to_f64, conv_weights, gate_values, layer_weights,
                       normal_bf16_bits, prefill_batch, residual_bits, table_rows, token_map)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _within(got, exact, err):
    """got is the bf16 rounding of a value within err of exact."""
    lo = OD.bf16_round(exact - err)
    hi = OD.bf16_round(exact + err)
    return (got >= lo) & (got <= hi)


def _fp32_bound(h, gated, y, n, w, dil, cu, past=None):
    """fp32 evaluation error of h + (V~ + SiLU(sum_k w_k n_{t-k dil})): a few
    roundings of each term, the relative error of the normalisation (a
    5120-term fp32 sum) carried by every filter tap, and the fast SiLU's
    (6 + 1.2|c|) ulp."""
    K = w.shape[0]
    R = (K - 1) * dil
    taps = np.zeros_like(y)
    c = np.zeros_like(y)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        pa = np.zeros((R,) + n.shape[1:]) if past is None or past[s] is None else past[s]
        full = np.concatenate([pa, n[a:b]])
        for t in range(b - a):
            for k in range(K):
                taps[a + t] += np.abs(w[k] * full[R + t - k * dil])
                c[a + t] += w[k] * full[R + t - k * dil]
    silu = y - gated
    return (2.0 ** -21 * (np.abs(h) + np.abs(gated) + np.abs(silu)) + 3e-5 * taps
            + 2.0 ** -24 * (6 + 1.2 * np.abs(c)) * np.abs(silu) + 1e-30)


def _inputs(T, hc, H, K, seed, dead=()):
    mask = np.zeros(T, dtype=bool)
    mask[list(dead)] = True
    g = gate_values(T, hc, seed, mask)
    v_bits = normal_bf16_bits((T, H), 1.0, seed, 43)
    h_bits = residual_bits(T, hc, H, seed)
    w, gamma = conv_weights(K, hc, H, seed)
    return mask, g, v_bits, h_bits, w, gamma


def _oracle(cu, mask, g, v_bits, h_bits, w, gamma, dil, eps, state=None):
    gated = SC.gated_value(g.astype(np.float64), bf16_bits_to_f64(v_bits))
    y, new_state = SC.short_conv(gated, cu, w.astype(np.float64), gamma.astype(np.float64), dil, eps, state)
    h = bf16_bits_to_f64(h_bits)
    n = SC.rmsnorm(gated, gamma.astype(np.float64), eps)
    return h + y, y, gated, n, new_state


@pytest.mark.parametrize("K,dil", [(4, 3), (4, 4), (3, 2), (1, 1)])
def test_packed_prefill_matches_oracle(K, dil):
    T, hc, H = 1 + 7 + 300 + 45, 4, 512
    cu = np.array([0, 1, 8, 308, T])
    mask, g, v_bits, h_bits, w, gamma = _inputs(T, hc, H, K, 3, dead=range(100, 140))
    h = bf16(h_bits)
    st = status()
    eg.engram_short_conv_add(f32(g), bf16(v_bits), h, torch.from_numpy(mask.astype(np.uint8)).to(DEV), f32(w),
                             f32(gamma), dil, 1e-6, cu_seqlens=i64(cu), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact, y, gated, n, _ = _oracle(cu, mask, g, v_bits, h_bits, w, gamma, dil, 1e-6)
    got = bf16_bits_to_f64(bits(h))
    err = _fp32_bound(bf16_bits_to_f64(h_bits), gated, y, n, w.astype(np.float64), dil, cu)
    ok = _within(got, exact, err)
    assert ok.all(), (np.argwhere(~ok)[:5], got[~ok][:5], exact[~ok][:5])
    assert (got == OD.bf16_round(exact)).mean() > 0.999
    # masked positions still receive SiLU(conv) of earlier positions (none with kernel 1)
    assert (got[100] != bf16_bits_to_f64(h_bits[100])).any() == (K > 1)


@pytest.mark.parametrize("hc,H,K,dil", [(1, 256, 4, 3), (3, 768, 2, 2), (6, 512, 4, 3), (8, 1280, 3, 1)])
def test_stream_groups_and_widths_match_oracle(hc, H, K, dil):
    """Stream counts that leave a block's group of four streams partly empty
    or need two groups, and hidden sizes that leave warps of the last
    512-channel block without channels: packed prefill against the oracle,
    and one sequence in two chunks with the ring carried bit-identical to one
    pass."""
    T = 97 + 64
    cu = np.array([0, 97, T])
    mask, g, v_bits, h_bits, w, gamma = _inputs(T, hc, H, K, 11 + hc, dead=range(20, 26))
    md = torch.from_numpy(mask.astype(np.uint8)).to(DEV)
    wd, gd = f32(w), f32(gamma)
    h = bf16(h_bits)
    st = status()
    eg.engram_short_conv_add(f32(g), bf16(v_bits), h, md, wd, gd, dil, 1e-6, cu_seqlens=i64(cu), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    exact, y, gated, n, _ = _oracle(cu, mask, g, v_bits, h_bits, w, gamma, dil, 1e-6)
    got = bf16_bits_to_f64(bits(h))
    err = _fp32_bound(bf16_bits_to_f64(h_bits), gated, y, n, w.astype(np.float64), dil, cu)
    ok = _within(got, exact, err)
    assert ok.all(), (np.argwhere(~ok)[:5], got[~ok][:5], exact[~ok][:5])
    # the first sequence again, as chunks of 40 and 57 with the ring carried
    R = (K - 1) * dil
    ring = torch.zeros((1, max(R, 1), hc, H), dtype=torch.float32, device=DEV)
    head = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for a, b in [(0, 40), (40, 97)]:
        hk = bf16(h_bits[a:b])
        eg.engram_short_conv_add(f32(g[a:b]), bf16(v_bits[a:b]), hk, md[a:b].contiguous(), wd, gd, dil, 1e-6,
                                 cu_seqlens=i64([0, b - a]), state=ring, state_head=head)
        outs.append(bits(hk))
    torch.cuda.synchronize()
    assert (np.concatenate(outs) == bits(h)[:97]).all()


def test_chunked_prefill_with_state_equals_one_pass():
    """A 300-position sequence in chunks of 5, 1, 144, 150 with the ring carried:
    every chunk matches the oracle's whole-sequence result, the device chunks
    are bit-identical to one device pass, and the ring holds the oracle's last
    9 normalised values."""
    T, hc, H, K, dil = 300, 4, 512, 4, 3
    mask, g, v_bits, h_bits, w, gamma = _inputs(T, hc, H, K, 5, dead=range(40, 52))
    exact, y, gated, n, st_o = _oracle(np.array([0, T]), mask, g, v_bits, h_bits, w, gamma, dil, 1e-6)
    err = _fp32_bound(bf16_bits_to_f64(h_bits), gated, y, n, w.astype(np.float64), dil, [0, T])
    ring = torch.zeros((1, (K - 1) * dil, hc, H), dtype=torch.float32, device=DEV)
    head = torch.zeros(1, dtype=torch.int32, device=DEV)
    wd, gd, md = f32(w), f32(gamma), torch.from_numpy(mask.astype(np.uint8)).to(DEV)
    h_one = bf16(h_bits)
    eg.engram_short_conv_add(f32(g), bf16(v_bits), h_one, md, wd, gd, dil, cu_seqlens=i64([0, T]))
    outs = []
    for a, b in [(0, 5), (5, 6), (6, 150), (150, 300)]:
        hc_ = bf16(h_bits[a:b])
        eg.engram_short_conv_add(f32(g[a:b]), bf16(v_bits[a:b]), hc_, md[a:b].contiguous(), wd, gd, dil,
                                 cu_seqlens=i64([0, b - a]), state=ring, state_head=head)
        outs.append(bits(hc_))
    torch.cuda.synchronize()
    chunked = np.concatenate(outs)
    assert (chunked == bits(h_one)).all()
    assert _within(bf16_bits_to_f64(chunked), exact, err).all()
    R = (K - 1) * dil
    hd = int(head.item())
    assert hd == T % R
    ring_t = ring.cpu().numpy()[0][[(hd + j) % R for j in range(R)]] * gamma   # the ring holds n / gamma
    assert np.allclose(ring_t, st_o[0], rtol=1e-4, atol=1e-4 * np.abs(st_o[0]).max())


def test_decode_steps_with_padding_match_oracle():
    """16 slots: prefixes of 0..40 positions prefilled with the state kept, then
    12 decode steps in which slots 3 and 9 are padding on odd steps."""
    hc, H, K, dil, B, steps = 4, 256, 4, 3, 16, 12
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 41, size=B)
    lens[:3] = [0, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    mask, g, v_bits, h_bits, w, gamma = _inputs(T, hc, H, K, 8)
    wd, gd = f32(w), f32(gamma)
    ring = torch.zeros((B, (K - 1) * dil, hc, H), dtype=torch.float32, device=DEV)
    head = torch.zeros(B, dtype=torch.int32, device=DEV)
    h0 = bf16(h_bits)
    eg.engram_short_conv_add(f32(g), bf16(v_bits), h0, None, wd, gd, dil, cu_seqlens=i64(cu), state=ring,
                             state_head=head)
    exact, y, gated, n, state_o = _oracle(cu, mask, g, v_bits, h_bits, w, gamma, dil, 1e-6)
    torch.cuda.synchronize()
    err = _fp32_bound(bf16_bits_to_f64(h_bits), gated, y, n, w.astype(np.float64), dil, cu)
    assert _within(bf16_bits_to_f64(bits(h0)), exact, err).all()
    st = status()
    for k in range(steps):
        _, gk, vk, hk, _, _ = _inputs(B, hc, H, K, 100 + k)
        slots = np.arange(B, dtype=np.int32)
        if k % 2:
            slots[[3, 9]] = -1
        h = bf16(hk)
        eg.engram_short_conv_add(f32(gk), bf16(vk), h, None, wd, gd, dil, slots=i32(slots), state=ring,
                                 state_head=head, status=st)
        torch.cuda.synchronize()
        live = slots >= 0
        cu1 = np.arange(int(live.sum()) + 1)
        past = [state_o[b] for b in np.flatnonzero(live)]
        ex, y, gated, n, new = _oracle(cu1, np.zeros(int(live.sum()), bool), gk[live], vk[live], hk[live], w, gamma,
                                       dil, 1e-6, past)
        for j, b in enumerate(np.flatnonzero(live)):
            state_o[b] = new[j]
        got = bf16_bits_to_f64(bits(h))
        err = _fp32_bound(bf16_bits_to_f64(hk[live]), gated, y, n, w.astype(np.float64), dil, cu1, past)
        assert _within(got[live], ex, err).all(), k
        assert (bits(h)[~live] == hk[~live]).all()                 # padding untouched
    assert int(st.item()) == 0
    R = (K - 1) * dil
    ring_np, head_np = ring.cpu().numpy(), head.cpu().numpy()
    for b in range(B):
        n_seen = lens[b] + steps - (steps // 2 if b in (3, 9) else 0)
        assert head_np[b] == n_seen % R
        ordered = ring_np[b][[(head_np[b] + j) % R for j in range(R)]] * gamma
        assert np.allclose(ordered, state_o[b], rtol=1e-4, atol=1e-4 * max(1.0, np.abs(state_o[b]).max())), b


def test_bad_slot_sets_status_and_is_skipped():
    hc, H, K, dil = 2, 256, 4, 3
    _, g, v_bits, h_bits, w, gamma = _inputs(3, hc, H, K, 9)
    ring = torch.zeros((2, 9, hc, H), dtype=torch.float32, device=DEV)
    head = torch.zeros(2, dtype=torch.int32, device=DEV)
    h = bf16(h_bits)
    st = status()
    eg.engram_short_conv_add(f32(g), bf16(v_bits), h, None, f32(w), f32(gamma), dil, slots=i32([0, 5, 1]),
                             state=ring, state_head=head, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 4
    assert (bits(h)[1] == h_bits[1]).all()
    assert (head.cpu().numpy() == [1, 1]).all()


def test_layer_with_short_conv_matches_oracle():
    """The original layer shape family: 2/3-grams, 16 columns, hidden 2560,
    4 streams, kernel 4, dilation 3; 2 sequences of 150 with an image span."""
    w = Workload("conv", 1300, 1000, 4099, 2, 2, 150, 2560, 4, 0.0)
    tm = token_map(w.v_raw, w.v, 3)
    pad = int(tm[0])
    lay_o = OL.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    lay = eg.build_layout(w.v, w.base_rows, [2, 15], max_ngram=3, n_heads=8, pad_id=pad)
    lw = layer_weights(w, n_cols=16, seed=5)
    cw, gamma = conv_weights(4, w.hc, w.hidden, 6)
    total = lay_o.layers[0].total_rows
    layer = eg.EngramLayer(lay, 0, device_table(total, 9), i32(tm), eg.engram_pack_wkv(bf16(lw.wkv_bits)),
                           f32(lw.q_w), f32(lw.k_w), conv=eg.ShortConv(f32(cw), f32(gamma), 3))
    b = prefill_batch(w, seed=4)
    b.raw_ids[60:70] = DEAD
    T = len(b.raw_ids)
    h_bits = residual_bits(T, w.hc, w.hidden, 6)
    h = bf16(h_bits)
    gate = torch.empty((T, w.hc), dtype=torch.float32, device=DEV)
    ring, head = layer.new_conv_state(w.n_seqs, DEV)
    st = status()
    layer.prefill(i32(b.raw_ids), i64(b.cu_seqlens), h, status=st, gate_out=gate, conv_state=(ring, head))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows_o, mask_o, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    e = OD.gather_dequant(rows_o, lambda r: table_rows(9, r))
    W = bf16_bits_to_f64(lw.wkv_bits)
    k, v = OG.split_kv(OG.project(e, W), w.hidden, w.hc)
    hf = bf16_bits_to_f64(h_bits)
    g = OG.gate(hf, k, lw.q_w, lw.k_w, mask_o)
    assert np.abs(gate.cpu().numpy() - g).max() <= GATE_ATOL
    gated = SC.gated_value(g, v)
    y, _ = SC.short_conv(gated, b.cu_seqlens, cw.astype(np.float64), gamma.astype(np.float64), 3, 1e-6)
    exact = hf + y
    # what the earlier stages carry in: |dg| <= GATE_ATOL; v carries the
    # projection's fp32 accumulation bound, and bf16(v) may flip by one ulp
    # where v is within that bound of a midpoint (the residual reading)
    vb = OD.bf16_round(v)
    v_err = dot_error_bound(e, W[:, w.hc * w.hidden:])
    d_v = v_err + bf16_flip(v, v_err)
    d_gated = GATE_ATOL * np.abs(vb)[:, None, :] + np.abs(g)[:, :, None] * d_v[:, None, :]
    r = np.sqrt(np.mean(gated ** 2, axis=-1, keepdims=True) + 1e-6)
    d_rms = np.sqrt(np.mean(d_gated ** 2, axis=-1, keepdims=True))
    d_n = np.abs(gamma) * (d_gated + np.abs(gated) * d_rms / r) / r
    d_c = np.zeros_like(d_n)
    cu = b.cu_seqlens
    for s in range(len(cu) - 1):
        a, bb = cu[s], cu[s + 1]
        for t in range(bb - a):
            for kk in range(4):
                if t - 3 * kk >= 0:
                    d_c[a + t] += np.abs(cw[kk]) * d_n[a + t - 3 * kk]
    n = SC.rmsnorm(gated, gamma.astype(np.float64), 1e-6)
    err = d_gated + 1.1 * d_c + _fp32_bound(hf, gated, y, n, cw.astype(np.float64), 3, cu)
    got = bf16_bits_to_f64(bits(h))
    ok = _within(got, exact, err)
    assert ok.all(), (np.argwhere(~ok)[:5], got[~ok][:5], exact[~ok][:5])
    assert (got == OD.bf16_round(exact)).mean() > 0.99
    assert (head.cpu().numpy() == [150 % 9, 150 % 9]).all()
