"""Degenerate sizes on the GPU: every compute entry point accepts an empty
batch (0 tokens), launches nothing that writes, and leaves its status word
clear; the projection epilogue's path for more than four residual streams
(hc 5..8) is covered in test_gpu_project."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import DEV, device_table, f32, i64, require_gpu, setup, status, u8
from workloads import mxfp8_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


H, HC, K = 256, 4, 6144


def _empty_common():
    e = torch.empty((0, K), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((0, HC, H), dtype=torch.bfloat16, device=DEV)
    qw = torch.ones((H, HC), dtype=torch.float32, device=DEV)
    kw = torch.ones((H, HC), dtype=torch.float32, device=DEV)
    mask = torch.empty(0, dtype=torch.uint8, device=DEV)
    return e, h, qw, kw, mask


def test_empty_projection_gate_and_residual():
    e, h, qw, kw, mask = _empty_common()
    w = torch.zeros((K, (HC + 1) * H), dtype=torch.bfloat16, device=DEV)
    wp = eg.engram_pack_wkv(w)
    st = status()
    partials, v = eg.engram_project(e, wp, h, qw, kw, status=st)
    assert partials.shape[0] == 0 and v.shape[0] == 0
    gate = torch.empty((0, HC), dtype=torch.float32, device=DEV)
    eg.engram_gate_add(partials, v, h, mask, gate_out=gate)
    eg.engram_project_gate(e, wp, h, qw, kw, mask, gate_out=gate, status=st)
    g = eg.engram_gates(partials, 0, H, HC, mask)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and g.shape == (0, HC)


def test_empty_fp8_projection():
    _, h, qw, kw, mask = _empty_common()
    w8, sf = mxfp8_weights(K, (HC + 1) * H, 1)
    w8p, sfb = eg.engram_pack_wkv_fp8(u8(w8), u8(sf))
    e8 = torch.empty((0, K), dtype=torch.uint8, device=DEV)
    sfa = torch.empty((48, 0), dtype=torch.int32, device=DEV)
    st = status()
    eg.engram_project_gate_fp8(e8, sfa, w8p, sfb, h, qw, kw, mask, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_empty_gather_and_short_conv():
    w, tm, lay_o, lay = setup("tiny")
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    st = status()
    rows = torch.empty((0, 24), dtype=torch.int32, device=DEV)
    e = eg.engram_gather_dequant(table, total, rows, status=st)
    e8, sf = eg.engram_gather_fp8(table, total, rows, status=st)
    assert e.shape[0] == 0 and e8.shape[0] == 0
    hc, hid = 4, 512
    h = torch.empty((0, hc, hid), dtype=torch.bfloat16, device=DEV)
    v = torch.empty((0, hid), dtype=torch.bfloat16, device=DEV)
    gate = torch.empty((0, hc), dtype=torch.float32, device=DEV)
    cw = f32(np.ones((4, hc, hid), dtype=np.float32))
    gamma = f32(np.ones((hc, hid), dtype=np.float32))
    eg.engram_short_conv_add(gate, v, h, torch.empty(0, dtype=torch.uint8, device=DEV), cw, gamma, 3,
                             cu_seqlens=i64(np.array([0, 0])), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
