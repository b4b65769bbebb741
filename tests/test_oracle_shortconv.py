"""Pins of the short-convolution oracle against closed forms, library routines
and the invariants the pages state ([P-DETAIL] §4.2, §9.5)."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import shortconv as SC


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_zero_filters_leave_the_gated_value():
    """[P-DETAIL] §4.2: zero-initialised filters make the branch leave V~ unchanged."""
    g = _rand((12, 2, 16), 1)
    y, _ = SC.short_conv(g, [0, 5, 12], np.zeros((4, 2, 16)), _rand((2, 16), 2), 3, 1e-6)
    assert (y == g).all()


def test_conv_is_numpy_convolve_with_dilated_taps():
    """One channel: sum_k w[k] n[t-k*d] is a full convolution with the filter
    spread to taps 0, d, 2d, 3d, cut to the sequence length (zeros before)."""
    T, d = 40, 3
    n = _rand((T, 1, 1), 3)
    w = _rand((4, 1, 1), 4)
    c = SC.causal_conv(n, w, d)
    spread = np.zeros(3 * d + 1)
    spread[::d] = w[:, 0, 0]
    assert np.allclose(c[:, 0, 0], np.convolve(n[:, 0, 0], spread)[:T], rtol=0, atol=1e-12)


def test_conv_with_past_is_convolution_of_the_concatenation():
    T, d = 17, 3
    R = 3 * d
    past = _rand((R, 1, 2), 5)
    n = _rand((T, 1, 2), 6)
    w = _rand((4, 1, 2), 7)
    c = SC.causal_conv(n, w, d, past)
    for ch in range(2):
        spread = np.zeros(R + 1)
        spread[::d] = w[:, 0, ch]
        full = np.convolve(np.concatenate([past[:, 0, ch], n[:, 0, ch]]), spread)
        assert np.allclose(c[:, 0, ch], full[R:R + T], rtol=0, atol=1e-12)


def test_impulse_reaches_t_plus_0_3_6_9():
    """Kernel 4, dilation 3: position t reads t, t-3, t-6, t-9 ([P-DETAIL] §4.2)."""
    T, p = 30, 7
    n = np.zeros((T, 1, 1))
    n[p] = 1.0
    w = np.array([1.0, 2.0, 3.0, 4.0]).reshape(4, 1, 1)
    c = SC.causal_conv(n, w, 3)[:, 0, 0]
    expect = np.zeros(T)
    expect[[p, p + 3, p + 6, p + 9]] = [1.0, 2.0, 3.0, 4.0]
    assert (c == expect).all()


def test_rmsnorm_closed_form_and_scale_invariance():
    x = _rand((5, 3, 64), 8)
    ref = x * np.sqrt(64) / np.linalg.norm(x, axis=-1, keepdims=True)
    assert np.allclose(SC.rmsnorm(x, np.ones(64), 0.0), ref, rtol=1e-13, atol=0)
    gamma = _rand((3, 64), 9)
    assert np.allclose(SC.rmsnorm(7.5 * x, gamma, 0.0), SC.rmsnorm(x, gamma, 0.0), rtol=1e-12, atol=1e-12)
    assert (SC.rmsnorm(np.zeros((2, 64)), np.ones(64), 1e-6) == 0).all()


def test_silu_is_x_times_logistic():
    x = np.linspace(-30, 30, 1001)
    assert np.allclose(SC.silu(x), x * expit(x), rtol=1e-14, atol=1e-300)


def test_gated_value_rounds_v_once_and_masks():
    v = np.array([[1.0 + 2 ** -9, -3.0]])        # below half a bf16 ulp of 1: rounds to 1.0
    g = np.array([[0.5, 0.0]])
    out = SC.gated_value(g, v)
    assert out.shape == (1, 2, 2)
    assert (out[0, 0] == [0.5, -1.5]).all() and (out[0, 1] == 0).all()


@pytest.mark.parametrize("cuts", [[0, 5, 17, 41], [0, 1, 2, 3, 41], [0, 9, 10, 41]])
def test_chunks_with_carried_state_equal_one_pass(cuts):
    """[P-DETAIL] §9.5: chunked prefill carries the past normalised values."""
    T, hc, H = 41, 2, 8
    gated = _rand((T, hc, H), 10)
    w = _rand((4, hc, H), 11)
    gamma = _rand((hc, H), 12)
    y_all, st_all = SC.short_conv(gated, [0, T], w, gamma, 3, 1e-6)
    state = None
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        y, st = SC.short_conv(gated[a:b], [0, b - a], w, gamma, 3, 1e-6, state)
        parts.append(y)
        state = st
    assert np.allclose(np.concatenate(parts), y_all, rtol=0, atol=1e-12)
    assert np.allclose(state[0], st_all[0], rtol=0, atol=0)


def test_decode_steps_equal_prefill_and_sequences_are_isolated():
    T, hc, H = 23, 1, 4
    gated = _rand((2 * T, hc, H), 13)
    w = _rand((4, hc, H), 14)
    gamma = np.ones((hc, H))
    y_pack, _ = SC.short_conv(gated, [0, T, 2 * T], w, gamma, 3, 1e-6)
    y_alone, _ = SC.short_conv(gated[T:], [0, T], w, gamma, 3, 1e-6)
    assert (y_pack[T:] == y_alone).all()
    # two sequences decoded one token per step, batched
    state = [None, None]
    out = np.empty_like(gated)
    for t in range(T):
        y, state = SC.short_conv(np.stack([gated[t], gated[T + t]]), [0, 1, 2], w, gamma, 3, 1e-6, state)
        out[t], out[T + t] = y[0], y[1]
    assert np.allclose(out, y_pack, rtol=0, atol=1e-12)


def test_state_keeps_older_entries_when_chunk_is_short():
    R = 9
    past = np.arange(R, dtype=np.float64).reshape(R, 1, 1) + 1
    gated = np.full((2, 1, 1), 4.0)
    _, st = SC.short_conv(gated, [0, 2], np.zeros((4, 1, 1)), np.ones((1, 1)), 3, 0.0, [past])
    assert (st[0][:, 0, 0] == [3, 4, 5, 6, 7, 8, 9, 1, 1]).all()   # rmsnorm of a 1-wide 4.0 is 1.0


def test_conv_residual_rounds_once():
    """bf16 has a 2^-7 ulp at 1: 1 + 2^-8 is a tie (to even: 1), just above it rounds up."""
    h = np.array([1.0, 1.0])
    y = np.array([2 ** -8 + 2 ** -30, 2 ** -8])
    assert (SC.conv_residual(h, y) == [1.0 + 2 ** -7, 1.0]).all()


def test_layer_forward_conv_with_zero_filters_matches_plain_layer_off_mask():
    """Zero filters: the conv variant adds V~ = g*bf16(v) exactly like the
    V4.1 layer, and at masked positions (g = 0) adds 0."""
    from oracle import layout as OL, pipeline as OP
    from workloads import DEAD, WORKLOADS, bf16_bits_to_f64, layer_weights, prefill_batch, residual_bits, table_rows, \
        token_map
    w = WORKLOADS["tiny"]
    tm = token_map(w.v_raw, w.v, w.seed)
    lay = OL.build_layout(w.v, w.base_rows, [w.layer_id], pad_id=int(tm[0]))
    b = prefill_batch(w)
    b.raw_ids[40:52] = DEAD                     # an image span
    lw = layer_weights(w)
    T = len(b.raw_ids)
    h = bf16_bits_to_f64(residual_bits(T, w.hc, w.hidden, 1))
    args = (lay, 0, b.raw_ids, b.cu_seqlens, tm, lambda r: table_rows(w.seed, r), bf16_bits_to_f64(lw.wkv_bits),
            h, lw.q_w, lw.k_w)
    plain = OP.layer_forward(*args)
    conv = OP.ConvParams(np.zeros((4, w.hc, w.hidden)), np.ones((w.hc, w.hidden)), 3)
    res, state = OP.layer_forward_conv(*args, conv)
    assert plain.mask.any()
    assert (res.h_out == plain.h_out).all()
    assert len(state) == w.n_seqs and state[0].shape == (9, w.hc, w.hidden)
