"""GPU parity of the tensor-core projection, the fused gate partials and the residual add."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import (DEV, GATE_ATOL, bf16, bits, dot_error_bound, f32, i32, require_gpu, residual_close,
                      status, u8, v_flips_explained)
from oracle import dequant as OD
from oracle import gate as OG
from workloads import bf16_bits_to_f64, normal_bf16_bits, uniform_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _inputs(T, H, hc, K=6144, seed=0, e_std=1.0):
    e = normal_bf16_bits((T, K), e_std, seed, 1)
    w = normal_bf16_bits((K, (hc + 1) * H), 0.02, seed, 2)
    h = normal_bf16_bits((T, hc, H), 1.0, seed, 3)
    qw = uniform_f32((H, hc), 0.5, 1.5, seed, 4)
    kw = uniform_f32((H, hc), 0.5, 1.5, seed, 5)
    return e, w, h, qw, kw


def _oracle(e, w, h, qw, kw, mask, T, H, hc):
    ef, wf = bf16_bits_to_f64(e), bf16_bits_to_f64(w)
    kv = OG.project(ef, wf)
    k, v = OG.split_kv(kv, H, hc)
    hf = bf16_bits_to_f64(h)
    g = OG.gate(hf, k, qw, kw, mask)
    out = OG.residual(hf, g, v, mask)
    err = dot_error_bound(ef, wf)            # fp32 accumulation bound of every kv element
    k_err, v_err = OG.split_kv(err, H, hc)
    return k, v, hf, g, out, k_err, v_err


@pytest.mark.parametrize("T,H,hc", [(128, 256, 4), (300, 256, 4), (1, 256, 4), (129, 512, 2), (257, 256, 1)])
def test_project_partials_v_gate_residual(T, H, hc):
    e, w, h, qw, kw = _inputs(T, H, hc, seed=T)
    mask = np.zeros(T, dtype=bool)
    mask[::17] = True
    k, v, hf, g, out, k_err, v_err = _oracle(e, w, h, qw, kw, mask, T, H, hc)
    wp = eg.engram_pack_wkv(bf16(w))
    # the repack is a pure permutation of the bf16 bits into 128 x 64 tiles of w^T
    Kd, Nd = w.shape
    tiled = w.T.reshape(Nd // 128, 128, Kd // 64, 64).transpose(0, 2, 1, 3)
    assert (bits(wp).reshape(-1) == tiled.reshape(-1)).all()
    h_d = bf16(h)
    st = status()
    partials, v_d = eg.engram_project(bf16(e), wp, h_d, f32(qw), f32(kw), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # v: fp32 accumulation then one bf16 rounding; the oracle rounds the exact
    # value.  Bit-equal except where the exact v is within the accumulation
    # bound of a bf16 midpoint, and there one bf16 step away at most.
    vb = bf16_bits_to_f64(bits(v_d))
    assert (np.abs(vb - v) <= 2.0 ** -8 * np.abs(v) + v_err).all()   # one bf16 rounding + fp32 sum
    v_flips_explained(bits(v_d), v, v_err)
    # partials per 256-column tile
    P = partials.cpu().numpy().astype(np.float64)
    ntile = H // 256
    qk = (qw.astype(np.float64) * kw.astype(np.float64)).T.reshape(hc, ntile, 256)
    kt = k.reshape(T, hc, ntile, 256)
    ht = hf.reshape(T, hc, ntile, 256)
    ke = k_err.reshape(T, hc, ntile, 256)
    dot = np.einsum("tmqc,mqc,tmqc->tmq", ht, qk, kt)
    dot_abs = np.einsum("tmqc,mqc,tmqc->tmq", np.abs(ht), qk, np.abs(kt))
    dot_tol = np.einsum("tmqc,mqc,tmqc->tmq", np.abs(ht), qk, ke) + 1e-5 * dot_abs
    assert (np.abs(P[..., 0] - dot) <= dot_tol).all()
    kk = np.sum(kt * kt, axis=3)
    assert (np.abs(P[..., 1] - kk) <= np.sum(2 * np.abs(kt) * ke + ke ** 2, axis=3) + 1e-5 * kk).all()
    np.testing.assert_allclose(P[..., 2], np.sum(ht * ht, axis=3), rtol=1e-5)
    # gate + residual
    gate = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    eg.engram_gate_add(partials, v_d, h_d, u8(mask), gate_out=gate)
    gg = gate.cpu().numpy()
    assert np.abs(gg - g).max() <= GATE_ATOL
    assert (gg[mask] == 0).all()
    hb = bits(h_d)
    assert (hb[mask] == h[mask]).all()                     # masked rows bit-identical
    r = residual_close(bf16_bits_to_f64(hb), out, hf, g, v, v_err)
    assert r.ok, r


def test_project_identity_selects_rows():
    """e = one-hot rows: kv reproduces wkv rows exactly (checks operand order and tiling)."""
    T, H, hc, K = 256, 256, 4, 6144
    e = np.zeros((T, K), dtype=np.uint16)
    sel = (np.arange(T) * 37) % K
    e[np.arange(T), sel] = 0x3F80                          # 1.0
    w = normal_bf16_bits((K, (hc + 1) * H), 0.02, 9, 1)
    h = normal_bf16_bits((T, hc, H), 1.0, 9, 2)
    ones = np.ones((H, hc), dtype=np.float32)
    partials, v_d = eg.engram_project(bf16(e), eg.engram_pack_wkv(bf16(w)), bf16(h), f32(ones), f32(ones))
    vb = bits(v_d)
    assert (vb == w[sel, hc * H:]).all()
    P = partials.cpu().numpy().astype(np.float64)
    wf = bf16_bits_to_f64(w)
    for m in range(hc):
        km = wf[sel, m * H:(m + 1) * H]
        np.testing.assert_allclose(P[:, m, 0, 1], np.sum(km * km, axis=1), rtol=1e-5)


def test_project_large_m_tiles():
    """T = 1024 over the full 5120-wide key/value layout (100 N tiles), sampled rows."""
    T, H, hc = 1024, 5120, 4
    e, w, h, qw, kw = _inputs(T, H, hc, seed=42)
    h_d = bf16(h)
    partials, v_d = eg.engram_project(bf16(e), eg.engram_pack_wkv(bf16(w)), h_d, f32(qw), f32(kw))
    gate = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    mask = np.zeros(T, dtype=bool)
    eg.engram_gate_add(partials, v_d, h_d, u8(mask), gate_out=gate)
    idx = np.array([0, 1, 127, 128, 500, 1023])
    k, v, hf, g, out, k_err, v_err = _oracle(e[idx], w, h[idx], qw, kw, mask[idx], len(idx), H, hc)
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v, v_err)
    assert r.ok, r


def _assert_same_update(hu_bits, hb_bits, g_u, v_u, g_b=None, v_err=None):
    """Two computations of h <- bf16(h + g bf16(v)) whose fp32 sums ran in a
    different order (fused or not, K split or not).  bf16(v) may differ by one
    bf16 step (2^-7 of |v|), plus twice the fp32 accumulation bound of v when
    it is given (a sum that nearly cancels has a large relative error); g
    differs by fp32 rounding (|g_u - g_b| when the other gates are given, else
    1e-5).  So h may differ by one step of the result, plus g times the
    difference of bf16(v), plus the gate difference times v."""
    hu, hb = bf16_bits_to_f64(hu_bits), bf16_bits_to_f64(hb_bits)
    v = np.abs(bf16_bits_to_f64(bits(v_u)))[:, None, :]
    gu = g_u.cpu().numpy().astype(np.float64)
    dg = 1e-5 if g_b is None else np.abs(gu - g_b.cpu().numpy().astype(np.float64))[:, :, None] + 1e-7
    dv = 2.0 ** -7 * v + (0.0 if v_err is None else 2.0 * np.asarray(v_err)[:, None, :])
    bound = 2.0 ** -7 * np.abs(hu) + 2.0 * np.abs(gu)[:, :, None] * dv + 2.0 * dg * v + 1e-30
    assert (np.abs(hu - hb) <= bound).all()


@pytest.mark.parametrize("T,H,hc", [(128, 256, 4), (300, 256, 4), (1, 256, 4), (129, 512, 2), (257, 256, 1),
                                    (1537, 256, 4), (1600, 512, 2), (2100, 256, 4),
                                    (100, 256, 8), (300, 256, 6), (1600, 256, 8), (1800, 256, 5)])
def test_project_gate_fused(T, H, hc):
    """engram_project_gate against the oracle and against the unfused kernels.

    Up to 1536 tokens the entry point runs the two-kernel path in its
    workspace; from 1537 tokens on (ragged: 6 pair blocks + 1 row) the fused
    cooperative kernel.  5 to 8 residual streams take the fused value
    epilogue's path for streams beyond the fourth."""
    e, w, h, qw, kw = _inputs(T, H, hc, seed=1000 + T)
    mask = np.zeros(T, dtype=bool)
    mask[5::11] = True
    k, v, hf, g, out, k_err, v_err = _oracle(e, w, h, qw, kw, mask, T, H, hc)
    wp = eg.engram_pack_wkv(bf16(w))
    e_d, qw_d, kw_d, m_d = bf16(e), f32(qw), f32(kw), u8(mask)
    h_f = bf16(h)
    g_f = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    st = status()
    eg.engram_project_gate(e_d, wp, h_f, qw_d, kw_d, m_d, gate_out=g_f, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    gf = g_f.cpu().numpy()
    assert np.abs(gf - g).max() <= GATE_ATOL
    assert (gf[mask] == 0).all()
    hb = bits(h_f)
    assert (hb[mask] == h[mask]).all()
    r = residual_close(bf16_bits_to_f64(hb), out, hf, g, v, v_err)
    assert r.ok, r
    # unfused kernels on the same inputs: gates agree to fp32 summation order
    h_u = bf16(h)
    g_u = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    partials, v_d = eg.engram_project(e_d, wp, h_u, qw_d, kw_d)
    eg.engram_gate_add(partials, v_d, h_u, m_d, gate_out=g_u)
    assert np.abs(g_u.cpu().numpy() - gf).max() <= 1e-5
    _assert_same_update(bits(h_u), hb, g_u, v_d)


def test_project_gate_fused_many_groups():
    """4133 tokens (33 M-blocks, three raster groups, ragged tail) at hidden 5120: sampled rows."""
    T, H, hc = 4133, 5120, 4
    e, w, h, qw, kw = _inputs(T, H, hc, seed=77)
    mask = np.zeros(T, dtype=bool)
    mask[[3, 2048, 4132]] = True
    h_d = bf16(h)
    gate = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    st = status()
    eg.engram_project_gate(bf16(e), eg.engram_pack_wkv(bf16(w)), h_d, f32(qw), f32(kw), u8(mask), gate_out=gate,
                           status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx = np.array([0, 3, 127, 128, 2047, 2048, 2049, 4095, 4096, 4131, 4132])
    k, v, hf, g, out, k_err, v_err = _oracle(e[idx], w, h[idx], qw, kw, mask[idx], len(idx), H, hc)
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v, v_err)
    assert r.ok, r
    assert (bits(h_d)[mask] == h[mask]).all()


@pytest.mark.parametrize("T,H", [(256, 5120), (200, 5120), (37, 5120), (256, 6400)])
def test_project_gate_decode_shape(T, H):
    """Decode-size batches through engram_project_gate's two-kernel path: 256
    and 200 tokens at hidden 5120 (100 column tiles) and 256 at hidden 6400
    (125 tiles) on the CTA-pair kernel, 37 tokens on the single-CTA kernel.
    Sampled rows against the oracle; every row against engram_project +
    engram_gate_add to fp32 summation order."""
    hc = 4
    e, w, h, qw, kw = _inputs(T, H, hc, seed=500 + T)
    mask = np.zeros(T, dtype=bool)
    mask[[1, T - 2]] = True
    wp = eg.engram_pack_wkv(bf16(w))
    e_d, qw_d, kw_d, m_d = bf16(e), f32(qw), f32(kw), u8(mask)
    h_d = bf16(h)
    gate = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    st = status()
    eg.engram_project_gate(e_d, wp, h_d, qw_d, kw_d, m_d, gate_out=gate, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx = np.unique(np.concatenate([np.arange(0, T, 16), [1, T - 2, T - 1]]))
    k, v, hf, g, out, k_err, v_err = _oracle(e[idx], w, h[idx], qw, kw, mask[idx], len(idx), H, hc)
    assert np.abs(gate.cpu().numpy()[idx] - g).max() <= GATE_ATOL
    r = residual_close(bf16_bits_to_f64(bits(h_d)[idx]), out, hf, g, v, v_err)
    assert r.ok, r
    assert (bits(h_d)[mask] == h[mask]).all()
    h_u = bf16(h)
    g_u = torch.empty((T, hc), dtype=torch.float32, device=DEV)
    partials, v_u = eg.engram_project(e_d, wp, h_u, qw_d, kw_d)
    eg.engram_gate_add(partials, v_u, h_u, m_d, gate_out=g_u)
    # the gate kernel's partial sums are reduced in another order: fp32 rounding
    assert np.abs(g_u.cpu().numpy() - gate.cpu().numpy()).max() <= 1e-4
    v_err_all = dot_error_bound(bf16_bits_to_f64(e), bf16_bits_to_f64(w)[:, hc * H:])
    _assert_same_update(bits(h_u), bits(h_d), g_u, v_u, gate, v_err_all)
