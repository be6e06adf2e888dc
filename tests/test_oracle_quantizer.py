"""Pins of the oracle's quantized write (NVFP4 two-level scaling, FP8).

Each check is fixed by the pages or by the mathematics rather than by the
oracle's own code: the 9-byte ledger, exact round trips of values built on
the grid, the max element landing on code 7, the half-gap error bound, the
zero and signed-zero cases, the nibble order and the page placement.
"""
import numpy as np
import pytest

from conftest import read_golden

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e4m3_table():
    """E4M3 values of bytes 0..126 from the bit fields (independent of the oracle)."""
    v = []
    for c in range(127):
        e, m = c >> 3, c & 7
        v.append(2.0 ** (e - 7) * (1 + m / 8) if e else 2.0 ** -6 * m / 8)
    return np.array(v)


def _cache(orc, prec, num_pages, Hkv, P, D, g):
    return orc.Cache(prec, num_pages, Hkv, P, D, g)


def _unpack(codes):
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], -1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def _decode_nvfp4(codes, scales, g):
    c = _unpack(codes)
    mag = E2M1[c & 7] * np.where(c & 8, -1.0, 1.0)
    s = _e4m3_table()[scales]
    return mag * np.repeat(s, 16, axis=-1) * float(g)


def test_ledger_bytes_per_16_values(orc):
    led = {k: float(v) for k, v in read_golden("ledger.txt")}
    T, Hkv, D, P = 7, 3, 128, 4
    c = _cache(orc, orc.PREC_NVFP4, 8, Hkv, P, D, [1.0, 1.0])
    f = _cache(orc, orc.PREC_FP8, 8, Hkv, P, D, [1.0, 1.0])
    nv = c.k_data.nbytes + c.k_scale.nbytes
    f8 = f.k_data.nbytes
    values = 8 * Hkv * P * D
    assert nv * led["values_per_block"] == values * led["nvfp4_bytes_per_block"]
    assert f8 * led["values_per_block"] == values * led["fp8_bytes_per_block"]
    assert 100.0 * nv / f8 == led["footprint_vs_fp8_percent"]
    assert round(f8 / nv, 2) == led["capacity_ratio_approx"]
    del T


def test_global_scale_closed_form(orc):
    x = np.array([0.5, -2688.0, 3.0], np.float32)
    assert orc.global_scale(x) == np.float32(1.0)
    assert orc.global_scale(np.array([-448.0, 1.0], np.float32), orc.FP8_GLOBAL_DIVISOR) == np.float32(1.0)
    assert orc.global_scale(np.zeros(5, np.float32)) == 0.0
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert orc.global_scale(x) == np.float32(np.abs(x).max()) / np.float32(2688.0)


def _write_one(orc, x, g, P=4, page=2, off=1):
    """Write one token-head vector x[D] at (page, off); return (codes, scales)."""
    D = x.shape[-1]
    c = _cache(orc, orc.PREC_NVFP4, 4, 1, P, D, [g, g])
    k = x.reshape(1, 1, D).astype(np.float32)
    orc.quantize_write(c, k, k, np.array([page * P + off], np.int64))
    return c.k_data[page, 0, off], c.k_scale[page, 0, off], c


def test_round_trip_of_grid_values(orc):
    """x built as e2m1 * S * g, with each block's max at 6*S, requantizes to the same bytes."""
    rng = np.random.default_rng(1)
    tab = _e4m3_table()
    for g in (1.0, 0.37109375, 2.0 ** -20):
        codes = rng.integers(0, 16, 128)
        codes[::16] = 7  # block max magnitude 6
        sidx = rng.integers(8, 120, 8)  # normal scales away from saturation
        S = tab[sidx]
        x = (E2M1[codes & 7] * np.where(codes & 8, -1, 1)) * np.repeat(S, 16) * g
        assert np.all(x.astype(np.float32) == x)
        got_c, got_s, _ = _write_one(orc, x, np.float32(g))
        want = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)  # -0 (code 8) kept
        assert np.array_equal(got_s, sidx.astype(np.uint8)), g
        assert np.array_equal(got_c, want), g


def test_nibble_order_low_is_even_index(orc):
    x = np.zeros(16, np.float32)
    x[0], x[1] = 6.0, 0.5  # code 7 at even index, code 1 at odd index
    codes, scales, _ = _write_one(orc, x, np.float32(1.0))
    # g = 1: d = 6, sf = 1 -> S = 1, den = 1
    assert scales[0] == 0x38
    assert codes[0] == (7 | (1 << 4))


def test_block_max_gets_code_7_and_error_bound(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 128)).astype(np.float32) * np.float32(3.0)
    g = orc.global_scale(x)
    c = _cache(orc, orc.PREC_NVFP4, 16, 1, 4, 128, [g, g])
    xs = x.reshape(64, 1, 128)
    orc.quantize_write(c, xs, xs, np.arange(64, dtype=np.int64))
    codes = c.k_data.reshape(64, 64)
    scales = c.k_scale.reshape(64, 8)
    xh = _decode_nvfp4(codes, scales, g)
    cod = _unpack(codes)
    tab = _e4m3_table()
    for t in range(64):
        for b in range(8):
            blk = x[t, 16 * b:16 * b + 16].astype(np.float64)
            S = tab[scales[t, b]]
            assert 0 < scales[t, b] <= 0x7E  # the tensor-max block reaches 448 exactly
            i = np.argmax(np.abs(blk))
            assert (cod[t, 16 * b + i] & 7) == 7
            den = S * float(g)
            y = np.abs(blk) / den
            # half-gap bound of the E2M1 grid at |y| (y <= 6.4 by scale rounding)
            gap = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0))
            err = np.abs(blk - xh[t, 16 * b:16 * b + 16])
            sat = y > 6
            assert np.all(err[~sat] <= 0.5 * gap[~sat] * den * (1 + 1e-6))
            assert np.all(np.abs(xh[t, 16 * b:16 * b + 16][sat]) == 6 * den)


def test_zero_cases(orc):
    x = np.zeros(128, np.float32)
    x[3] = -0.0
    codes, scales, _ = _write_one(orc, x, np.float32(0.0))
    assert not codes.any() and not scales.any()
    # an all-zero block (with negative zeros) under a nonzero global scale
    x = np.full(128, 1.0, np.float32)
    x[:16] = -0.0
    codes, scales, _ = _write_one(orc, x, np.float32(1.0 / 2688))
    assert scales[0] == 0 and not codes[:8].any()
    assert scales[1] != 0


def test_signed_zero_in_nonzero_block(orc):
    x = np.zeros(16, np.float32)
    x[0] = 6.0
    x[2] = -0.0
    x[4] = -1e-3  # rounds to magnitude 0, keeps its sign
    codes, _, _ = _write_one(orc, x, np.float32(1.0))
    cod = _unpack(codes)
    assert cod[0] == 7 and cod[1] == 0 and cod[2] == 8 and cod[4] == 8


def test_slot_mapping_placement_and_skip(orc):
    Hkv, P, D = 2, 4, 32
    c = _cache(orc, orc.PREC_NVFP4, 5, Hkv, P, D, [1.0, 1.0])
    x = np.full((3, Hkv, D), 6.0, np.float32)
    x[:, 1] = 3.0
    orc.quantize_write(c, x, -x, np.array([9, -1, 0], np.int64))
    # token 0 -> page 2 offset 1; token 2 -> page 0 offset 0; token 1 skipped
    written = np.argwhere(c.k_scale.any(-1))
    assert sorted(map(tuple, written)) == [(0, 0, 0), (0, 1, 0), (2, 0, 1), (2, 1, 1)]
    assert np.all(_unpack(c.v_data[2, 0, 1]) == 15)  # -6 everywhere
    with pytest.raises(ValueError):
        orc.quantize_write(c, x[:1], x[:1], np.array([5 * P], np.int64))


def test_fp8_write_round_trip_and_scale(orc):
    tab = _e4m3_table()
    rng = np.random.default_rng(3)
    b = rng.integers(0, 127, (6, 2, 64))
    sign = rng.integers(0, 2, b.shape)
    s8 = np.float32(0.25)
    x = (tab[b] * np.where(sign, -1, 1) * 0.25).astype(np.float32)
    c = _cache(orc, orc.PREC_FP8, 3, 2, 2, 64, [s8, s8])
    orc.quantize_write(c, x, x, np.arange(6, dtype=np.int64))
    want = (b | (sign << 7)).astype(np.uint8)
    want[(b == 0) & (sign == 1)] = 0x80
    assert np.array_equal(c.k_data.transpose(0, 2, 1, 3).reshape(6, 2, 64), want)  # [page][head][slot] order
    # per-tensor scale convention: amax / 448
    assert orc.global_scale(x, orc.FP8_GLOBAL_DIVISOR) == np.float32(np.abs(x).max()) / np.float32(448)
    c0 = _cache(orc, orc.PREC_FP8, 3, 2, 2, 64, [0.0, 0.0])
    orc.quantize_write(c0, -np.abs(x), x, np.arange(6, dtype=np.int64))
    assert not c0.k_data.any()


def test_planted_mistakes_are_caught(orc):
    """A wrong operation order (x * (1/den)) or a dropped global scale would
    break the round trip above; check that these alternatives really differ
    from the oracle on the grid, so the pins have teeth."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal(4096).astype(np.float32)
    g = np.float32(0.0123)
    den = np.float32(np.float32(1.75) * g)
    a = (x / den)
    b = (x * (np.float32(1) / den)).astype(np.float32)
    assert np.any(a != b)  # operation order matters in FP32


def test_block_layout_offsets(orc):
    """Byte positions of one written slot, stated here independently of the
    oracle: one contiguous block per (page, KV head); groups of R slots (R = 8
    when the page size is a multiple of 8, else the page size); per group
    NVFP4 [K codes | K scales | V codes | V scales], FP8 [K | V]; K bytes in
    16-byte chunks, chunk-major; in an 8-row group V is stored by row pairs
    (2c, 2c+1): NVFP4 code of value d at byte (d//16)*64 + c*16 + d%16, row
    2c in the low nibble and 2c+1 in the high one, V scales block-major
    (block b of row r at b*8 + r); FP8 V byte at ((d%16)//8)*512 +
    (d//16)*64 + c*16 + (d%8)*2 + r%2.  Smaller groups keep V row-major."""
    # page size 4 (one group of 4 rows), D = 32: K codes 16 B per row (one chunk)
    Hkv, P, D = 2, 4, 32
    c = orc.Cache(orc.PREC_NVFP4, 3, Hkv, P, D, [1.0, 1.0])
    x = np.zeros((1, Hkv, D), np.float32)
    x[0, 1, 0] = 6.0  # head 1, element 0 -> code 7, scale 1.0 (0x38)
    orc.quantize_write(c, x, 0.5 * x, np.array([2 * P + 3], np.int64))  # page 2, offset 3
    blk = c.data[2, 1]
    # K codes [0,64): row 3 at 48; K scales [64,72): row 3 at 70; V codes [72,136): row 3 at 120; V scales at 142
    assert blk[48] == 0x07 and blk[70] == 0x38
    assert blk[120] == 0x07 and blk[142] == 0x30  # V: 3 = 6 x 0.5 -> scale 0.5
    assert np.count_nonzero(c.data) == 4
    f = orc.Cache(orc.PREC_FP8, 3, Hkv, P, D, [1.0, 1.0])
    orc.quantize_write(f, x, 0.5 * x, np.array([2 * P + 3], np.int64))
    # FP8: K [0,128): row 3 byte 0 at 48; V [128,256): row 3 at 128 + 3*32
    assert f.data[2, 1, 48] == 0x4C and f.data[2, 1, 128 + 96] == 0x44  # E4M3(6), E4M3(3)
    assert np.count_nonzero(f.data) == 2
    # page size 16, D = 128: slot 11 = group 1 (1152 bytes in), row 3
    c = orc.Cache(orc.PREC_NVFP4, 1, 1, 16, 128, [1.0, 1.0])
    x = np.zeros((1, 1, 128), np.float32)
    x[0, 0, 0] = 6.0    # K byte 0 (chunk 0) and block 0
    x[0, 0, 35] = 6.0   # byte 17 (chunk 1, high nibble), block 2
    orc.quantize_write(c, x, 0.5 * x, np.array([11], np.int64))
    blk = c.data[0, 0]
    g0 = 1152
    assert blk[g0 + 3 * 16] == 0x07 and blk[g0 + 128 + 3 * 16 + 1] == 0x70       # K chunks 0 and 1 of row 3
    assert blk[g0 + 512 + 3 * 8] == 0x38 and blk[g0 + 512 + 3 * 8 + 2] == 0x38   # K scales of blocks 0, 2
    # V: row 3 = pair 1, high nibble; value 0 -> byte 16, value 35 (block 2, j 3) -> byte 128 + 16 + 3
    assert blk[g0 + 576 + 16] == 0x70 and blk[g0 + 576 + 2 * 64 + 16 + 3] == 0x70
    assert blk[g0 + 1088 + 3] == 0x30 and blk[g0 + 1088 + 2 * 8 + 3] == 0x30      # V scales of blocks 0, 2
    assert np.count_nonzero(c.data) == 8
    f = orc.Cache(orc.PREC_FP8, 1, 1, 16, 128, [1.0, 1.0])
    orc.quantize_write(f, x, 0.5 * x, np.array([11], np.int64))
    fb = f.data[0, 0]
    g0 = 2048
    assert fb[g0 + 3 * 16] == 0x4C and fb[g0 + 2 * 128 + 3 * 16 + 3] == 0x4C   # K bytes 0 and 35
    # V: value 0 -> 0*512 + 0*64 + 16 + 0 + 1; value 35 (block 2, j 3) -> 0*512 + 128 + 16 + 6 + 1
    assert fb[g0 + 1024 + 17] == 0x44 and fb[g0 + 1024 + 151] == 0x44
    assert np.count_nonzero(f.data) == 4
