"""GPU parity of the gather + dequantise stage: bit-exact bf16 rows."""
import numpy as np
import pytest
import torch

import hashed_gram_conditional_gb300 as eg
from gpu_util import DEV, bits, device_table, i32, i64, require_gpu, setup, status, u8
from oracle import dequant as OD
from oracle import hashing as OH
from workloads import ROW_BYTES, prefill_batch, table_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()


def _compare_bits(got_bits: np.ndarray, ref_vals: np.ndarray):
    ref_bits = OD.bf16_bits(ref_vals)
    nan_ref = np.isnan(ref_vals)
    got_nan = (got_bits & 0x7F80) == 0x7F80
    got_nan &= (got_bits & 0x7F) != 0
    assert (got_nan == nan_ref).all()
    assert (got_bits[~nan_ref] == ref_bits[~nan_ref]).all()


def test_synthetic_table_generator_agrees():
    """The device filler and the host generator produce the same bytes."""
    n = 100_003
    t = device_table(n, 5)
    host = table_rows(5, np.arange(n))
    assert (t.cpu().numpy().reshape(n, ROW_BYTES) == host).all()


def test_all_codes_all_scales():
    """Every E4M3 code under every E8M0 scale (incl. NaN codes, subnormals, overflow)."""
    codes = np.arange(256, dtype=np.uint8)
    rows = np.zeros((256, ROW_BYTES), dtype=np.uint8)
    rows[:, :256] = codes[None, :]
    rows[:, 256:] = np.arange(256, dtype=np.uint8)[:, None]       # row s: all blocks scale s
    # second set: per-block distinct scales, rolled codes
    rows2 = np.zeros((64, ROW_BYTES), dtype=np.uint8)
    rng = np.random.default_rng(0)
    rows2[:, :256] = rng.integers(0, 256, size=(64, 256))
    rows2[:, 256:] = rng.integers(0, 256, size=(64, 8))
    table = np.concatenate([rows, rows2])
    n = len(table)
    ids = np.arange(n, dtype=np.int32)
    ids = np.concatenate([ids, ids[::-1]])                        # odd and even rows in both parities
    T = len(ids) // 24
    ids = ids[: T * 24].reshape(T, 24)
    e = eg.engram_gather_dequant(u8(table.reshape(-1)), n, i32(ids))
    ref = OD.gather_dequant(ids, lambda r: table[r])
    _compare_bits(bits(e), ref)


def _gather_vs_oracle(name, sample=None):
    w, tm, lay_o, lay = setup(name)
    b = prefill_batch(w)
    rows_o, _, _ = OH.hash_prefill(b.raw_ids, b.cu_seqlens, tm, lay_o, 0)
    total = lay_o.layers[0].total_rows
    table = device_table(total, w.seed)
    st = status()
    rows_d = i32(rows_o)
    e = eg.engram_gather_dequant(table, total, rows_d, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    idx = np.arange(len(rows_o)) if sample is None else sample(len(rows_o))
    e_s = bits(e[torch.from_numpy(idx).to(DEV)])
    ref = OD.gather_dequant(rows_o[idx], lambda r: table_rows(w.seed, r))
    _compare_bits(e_s, ref)


def test_gather_tiny_all_tokens():
    _gather_vs_oracle("tiny")


def test_gather_microbench_sampled():
    """65536 tokens over a 12.7 GB table; 1024 sampled tokens plus both ends."""
    def sample(n):
        rng = np.random.default_rng(11)
        return np.unique(np.concatenate([rng.integers(0, n, 1024), [0, 1, n - 2, n - 1]]))
    _gather_vs_oracle("microbench", sample)


def test_gather_bad_rows_zero_and_flag():
    n = 1000
    table = device_table(n, 1)
    ids = np.arange(48, dtype=np.int32).reshape(2, 24)
    ids[0, 3] = n
    ids[1, 7] = -4
    st = status()
    e = eg.engram_gather_dequant(table, n, i32(ids), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & eg.ST_BAD_ROW
    eb = bits(e).reshape(2, 24, 256)
    assert (eb[0, 3] == 0).all() and (eb[1, 7] == 0).all()
    good = ids.copy()
    good[0, 3] = 0
    good[1, 7] = 0
    ref = OD.gather_dequant(good, lambda r: table_rows(1, r)).reshape(2, 24, 256)
    keep = np.ones((2, 24), bool)
    keep[0, 3] = keep[1, 7] = False
    _compare_bits(eb[keep], ref[keep])


@pytest.mark.parametrize("n", [1001, 1000])
def test_gather_last_row_exact_allocation(n):
    """The last row of an exactly sized table (even and odd last index)."""
    table = device_table(n, 2)
    ids = np.full((3, 24), n - 1, dtype=np.int32)
    ids[1] = np.arange(n - 24, n)
    ids[2, ::2] = 0
    e = eg.engram_gather_dequant(table, n, i32(ids))
    ref = OD.gather_dequant(ids, lambda r: table_rows(2, r))
    _compare_bits(bits(e), ref)


def test_gather_ragged_token_counts():
    n = 5000
    table = device_table(n, 3)
    rng = np.random.default_rng(4)
    for T in [1, 7, 8, 9, 1215, 1217, 5000]:
        ids = rng.integers(0, n, size=(T, 24)).astype(np.int32)
        e = eg.engram_gather_dequant(table, n, i32(ids))
        ref = OD.gather_dequant(ids, lambda r: table_rows(3, r))
        _compare_bits(bits(e), ref)
