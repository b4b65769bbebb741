"""Pins of the oracle's E4M3 x E8M0 row decode and bf16 rounding."""
import numpy as np
import pytest
import torch

from oracle import dequant as D
from workloads import table_rows


def test_known_e4m3_points():
    v = D.e4m3_value(np.array([0x7E, 0x38, 0x08, 0x01, 0x80, 0x00, 0xFE, 0x07]))
    assert v[0] == 448.0
    assert v[1] == 1.0
    assert v[2] == 2.0 ** -6
    assert v[3] == 2.0 ** -9
    assert v[4] == 0.0 and np.signbit(v[4])
    assert v[5] == 0.0 and not np.signbit(v[5])
    assert v[6] == -448.0
    assert v[7] == 7 * 2.0 ** -9   # largest subnormal
    assert np.isnan(D.e4m3_value(np.array([0x7F, 0xFF]))).all()


def test_all_e4m3_codes_match_library_decode():
    """All 256 codes against torch.float8_e4m3fn widened to float64."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = D.e4m3_value(codes)
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert (mine[~nan] == ref[~nan]).all()
    assert (np.signbit(mine[~nan]) == np.signbit(ref[~nan])).all()


def test_e8m0_points():
    v = D.e8m0_value(np.array([127, 0, 254, 128, 120, 130, 255]))
    assert list(v[:6]) == [1.0, 2.0 ** -127, 2.0 ** 127, 2.0, 2.0 ** -7, 2.0 ** 3]
    assert np.isnan(v[6])


def test_bf16_round_matches_library_on_fp32_values():
    """Round-to-nearest-even into bf16 against torch's float32 -> bfloat16 cast."""
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # add halfway cases, subnormals, the overflow boundary and zeros
    extra = np.array([0x3F808000, 0x3F818000, 0x00008000, 0x00018000, 0x00000001,
                      0x7F7F8000, 0x7F7FFFFF, 0x7F7F7FFF, 0x80000000, 0x00000000,
                      0x807FFFFF, 0x00400000], dtype=np.uint32)
    bits = np.concatenate([bits, extra])
    f32 = bits.view(np.float32)
    fin = np.isfinite(f32)
    f32 = f32[fin]
    ref = torch.from_numpy(f32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    mine = D.bf16_round(f32.astype(np.float64))
    assert (mine == ref).all()
    assert (np.signbit(mine) == np.signbit(ref)).all()


def test_all_codes_times_all_scales():
    """Closed form over 256 codes x 255 finite scales equals library decode, scale, round."""
    codes = np.arange(256, dtype=np.uint8)
    scales = np.arange(255)
    rows = np.zeros((255, 264), dtype=np.uint8)   # one row per scale, holding all 256 codes
    rows[:, :256] = codes[None, :]
    rows[:, 256:] = scales[:, None].astype(np.uint8)  # all 8 blocks share the scale
    mine = D.dequant_rows(rows)                         # [255][256]
    w = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
    s = torch.pow(torch.tensor(2.0, dtype=torch.float64), torch.from_numpy(scales - 127.0))
    prod = (w.to(torch.float64)[None, :] * s[:, None])
    # every finite product is exact in fp32 (4 significant bits, exponent >= -136);
    # rounding to bf16 from fp32 is then a single rounding
    ref = prod.to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert (mine[~nan] == ref[~nan]).all()
    assert (np.signbit(mine[~nan]) == np.signbit(ref[~nan])).all()


def test_block_scale_per_32_elements():
    row = np.zeros((1, 264), dtype=np.uint8)
    row[0, :256] = 0x38                     # 1.0
    row[0, 256:] = np.arange(120, 128)      # block b scale 2^(b-7)
    v = D.dequant_rows(row)[0]
    for c in range(256):
        assert v[c] == 2.0 ** (c // 32 - 7)


def test_synthetic_rows_have_no_nan_and_scales_in_range():
    r = table_rows(0, np.arange(5000))
    assert not ((r[:, :256] & 0x7F) == 0x7F).any()
    assert r[:, 256:].min() >= 120 and r[:, 256:].max() <= 130
    assert len(np.unique(r[:, 256:])) == 11
    v = D.dequant_rows(r)
    assert np.isfinite(v).all()


def test_dequant_mx_weights_blocks_along_k():
    """Row k of column n takes scale row k // 32 of that column."""
    from oracle.dequant import dequant_mx_weights
    codes = np.full((64, 2), 0x38, dtype=np.uint8)          # E4M3 1.0
    codes[31, 1] = 0x7E                                       # 448
    scales = np.array([[127, 130], [120, 125]], dtype=np.uint8)
    w = dequant_mx_weights(codes, scales)
    assert w[0, 0] == 1.0 and w[31, 0] == 1.0 and w[32, 0] == 2.0 ** -7 and w[63, 0] == 2.0 ** -7
    assert w[31, 1] == 448.0 * 8 and w[32, 1] == 0.25 and w[0, 1] == 8.0


def test_bf16_row_generator_layout_and_range():
    """The synthetic bf16-row table: element c of row r comes from 16-bit piece
    c mod 4 (little-endian) of SplitMix64 output r*(row_dim/4) + c/4, with the
    exponent field forced into 120..130; every value is finite."""
    from workloads import splitmix64_at, table_rows_bf16
    row_dim = 80
    rows = np.array([0, 1, 12345, 2 ** 30 + 7])
    got = table_rows_bf16(7, rows, row_dim)
    assert got.shape == (4, row_dim) and got.dtype == np.uint16
    for i, r in enumerate(rows):
        for c in (0, 1, 3, 4, 77, 79):
            word = int(splitmix64_at(7, np.array([r * (row_dim // 4) + c // 4]))[0])
            b = (word >> (16 * (c % 4))) & 0xFFFF
            want = (b & 0x807F) | ((120 + ((b >> 7) & 0xFF) % 11) << 7)
            assert int(got[i, c]) == want
    ex = (got >> 7) & 0xFF
    assert ex.min() >= 120 and ex.max() <= 130
    from workloads import bf16_bits_to_f64
    vals = np.abs(bf16_bits_to_f64(table_rows_bf16(3, np.arange(500), row_dim)))
    assert np.isfinite(vals).all() and vals.min() >= 2.0 ** -7 and vals.max() < 16.0


def test_gather_rows_concatenates_in_column_order():
    rows = {5: np.full(8, 1.0), 9: np.full(8, 2.0), 11: np.full(8, 3.0)}
    e = D.gather_rows(np.array([[9, 5, 11]]), lambda ids: np.stack([rows[int(i)] for i in ids]))
    assert (e[0] == np.repeat([2.0, 1.0, 3.0], 8)).all()
