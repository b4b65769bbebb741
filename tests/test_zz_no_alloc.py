"""The allocation-free projection + gate entry point.

engram_project_gate_add_noalloc serves callers that cannot allocate device
memory where they run this stage (a serving engine that reserved all of HBM
for its own pools, a plugin inside a framework whose allocator it does not
own): its two intermediates live in the library's static device array.  This
test calls it through the C ABI and checks it against the allocating entry
points (engram_project + engram_gate_add) on the same inputs.  Both run the
same kernels at the same sizes, so gates and residuals must agree bit for
bit.  Calls come in a row, so that a call cannot lean on scratch contents
left by another, and one call sits exactly at the array's capacity.  The file
sorts last so that a run stopping at the first failure has run every other
test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import DEV, bf16, bits, f32, require_gpu, status, u8
from workloads import normal_bf16_bits, uniform_f32

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
SCRATCH_BYTES = 8 << 20      # ENGRAM_STAGE_STATIC_SCRATCH_BYTES
E_RANGE = -5                 # ENGRAM_E_RANGE


def _fn():
    lib = eg.lib()
    fn = lib.engram_project_gate_add_noalloc
    fn.argtypes = [P, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int32, ctypes.c_int32, P, P, P, P,
                   ctypes.c_float, ctypes.c_float, ctypes.c_float, P, P, P]
    fn.restype = ctypes.c_int
    return lib, fn


def _ptr(t):
    return None if t is None else P(t.data_ptr())


def _need_bytes(lib, T, H, hc):
    """Scratch one call needs: the partials rounded up to 256 bytes, then bf16 v."""
    partials = lib.engram_project_partials_bytes(T, H, hc)
    return (partials + 255) // 256 * 256 + T * H * 2


def _max_tokens(lib, H, hc):
    T = 1
    while _need_bytes(lib, T + 1, H, hc) <= SCRATCH_BYTES:
        T += 1
    return T


def _inputs(T, H, hc, seed):
    e = normal_bf16_bits((T, 6144), 1.0, seed, 1)
    w = normal_bf16_bits((6144, (hc + 1) * H), 0.02, seed, 2)
    h = normal_bf16_bits((T, hc, H), 1.0, seed, 3)
    qw = uniform_f32((H, hc), 0.5, 1.5, seed, 4)
    kw = uniform_f32((H, hc), 0.5, 1.5, seed, 5)
    mask = np.zeros(T, dtype=np.uint8)
    mask[::13] = 1
    return e, w, h, qw, kw, mask


def test_noalloc_matches_allocating_path_on_consecutive_calls():
    require_gpu()
    lib, fn = _fn()
    H, hc = 5120, 4
    t_max = _max_tokens(lib, H, hc)
    assert 700 < t_max < 760, t_max
    w = normal_bf16_bits((6144, (hc + 1) * H), 0.02, 7, 2)
    wp = eg.engram_pack_wkv(bf16(w))
    # a full call, a smaller one after it, one at the exact capacity, and a
    # small one last: every call must stand on its own scratch writes
    for call, (T, seed) in enumerate([(256, 101), (200, 202), (t_max, 303), (37, 404)]):
        e, _, h, qw, kw, mask = _inputs(T, H, hc, seed)
        e_d, qw_d, kw_d, m_d = bf16(e), f32(qw), f32(kw), u8(mask)
        scale = H ** -0.5
        # existing path, caller-allocated intermediates
        h_ref = bf16(h)
        g_ref = torch.empty((T, hc), dtype=torch.float32, device=DEV)
        partials, v = eg.engram_project(e_d, wp, h_ref, qw_d, kw_d)
        eg.engram_gate_add(partials, v, h_ref, m_d, 1e-6, 1e-6, scale, g_ref)
        # allocation-free path
        h_new = bf16(h)
        g_new = torch.empty((T, hc), dtype=torch.float32, device=DEV)
        st = status()
        rc = fn(_ptr(e_d), T, 6144, _ptr(wp), H, hc, _ptr(h_new), _ptr(qw_d), _ptr(kw_d), _ptr(m_d), 1e-6, 1e-6,
                scale, _ptr(g_new), _ptr(st), P(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, lib.engram_last_error()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # the same kernels on the same inputs: identical bits
        assert np.array_equal(g_ref.cpu().numpy().view(np.uint32), g_new.cpu().numpy().view(np.uint32)), call
        assert np.array_equal(bits(h_ref), bits(h_new)), call
        assert (bits(h_new)[mask.astype(bool)] == h[mask.astype(bool)]).all()


def test_noalloc_rejects_oversized_requests():
    require_gpu()
    lib, fn = _fn()
    H, hc = 5120, 4
    t_max = _max_tokens(lib, H, hc)
    # one token past the capacity, and a far larger request: rejected on the
    # host before any device work (the pointers are never dereferenced)
    for T in (t_max + 1, 4096):
        assert _need_bytes(lib, T, H, hc) > SCRATCH_BYTES
        rc = fn(P(256), T, 6144, P(256), H, hc, P(256), P(256), P(256), None, 1e-6, 1e-6, 0.01, None, None, None)
        assert rc == E_RANGE, T
        msg = lib.engram_last_error().decode()
        assert "static scratch" in msg and str(SCRATCH_BYTES) in msg
