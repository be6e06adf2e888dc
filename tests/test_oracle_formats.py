"""Pins of the oracle's element formats (E2M1 codes, E4M3 scales).

The oracle's encoders are checked against (a) the code tables fixed by the
bit-field definitions (golden fixtures, with citations) and (b) a brute-force
nearest-value search over every FP32 bit pattern, a different algorithm from
the oracle's own rounding.
"""
import ctypes
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from conftest import read_golden

CHUNK = 1 << 24


def _golden_e2m1():
    return {int(c): float(v) for c, v in read_golden("e2m1_codes.txt")}


def test_e2m1_table_matches_pages(orc):
    table = _golden_e2m1()
    assert len(table) == 16
    for code, want in table.items():
        got = orc.e2m1_value(code)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e2m1_round_trip_of_representable_values(orc):
    for code, v in _golden_e2m1().items():
        assert orc.e2m1_encode(v) == code


@pytest.mark.parametrize("y,code", [
    (0.25, 0), (0.2500001, 1), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    (5.0000005, 7), (6.0, 7), (1e30, 7), (float("inf"), 7), (-0.1, 8), (-0.0, 8), (-5.5, 15),
])
def test_e2m1_ties_to_even_and_saturation(orc, y, code):
    assert orc.e2m1_encode(y) == code


def test_e4m3_golden_points(orc):
    for hx, v in read_golden("e4m3_points.txt"):
        got = orc.e4m3_value(int(hx, 16))
        if v == "nan":
            assert math.isnan(got)
        else:
            assert got == float(v) and math.copysign(1.0, got) == math.copysign(1.0, float(v)), hx


def test_e4m3_round_trip_all_finite_codes(orc):
    n = 0
    for b in range(256):
        v = orc.e4m3_value(b)
        if math.isnan(v):
            continue
        assert orc.e4m3_encode(v) == b, hex(b)
        n += 1
    assert n == 254


@pytest.mark.parametrize("y,b", [
    (2.0 ** -10, 0x00), (2.0 ** -10 * 1.0000001, 0x01), (3 * 2.0 ** -10, 0x02), (449.0, 0x7E), (464.0, 0x7E),
    (1e9, 0x7E), (float("inf"), 0x7E), (-float("inf"), 0xFE), (1.0625, 0x38), (1.1875, 0x3A), (-0.0, 0x80),
    (-1e-30, 0x80),
])
def test_e4m3_ties_to_even_and_saturation(orc, y, b):
    assert orc.e4m3_encode(y) == b


def _sweep(orc, bruteforce, which):
    enc = orc.e2m1_encode_bits if which == 2 else orc.e4m3_encode_bits

    def one(start):
        got = enc(start, CHUNK)
        bad = ctypes.c_uint32(0)
        n = bruteforce.bf_compare(which, start, CHUNK, got.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                  ctypes.byref(bad))
        return n, bad.value

    starts = list(range(0, 1 << 32, CHUNK))
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        res = list(ex.map(one, starts))
    total = sum(n for n, _ in res)
    first = [b for n, b in res if n]
    assert total == 0, f"{total} mismatches, first at bit pattern {first[0]:#010x}"


def test_e2m1_exhaustive_against_brute_force(orc, bruteforce):
    """Every non-NaN FP32 bit pattern (2^32 - NaNs) rounds like the brute force."""
    _sweep(orc, bruteforce, 2)


def test_e4m3_exhaustive_against_brute_force(orc, bruteforce):
    """Every non-NaN FP32 bit pattern rounds like the brute force."""
    _sweep(orc, bruteforce, 4)


def test_brute_force_checker_is_not_vacuous(bruteforce):
    """The checker itself distinguishes wrong codes (guards a silent pass)."""
    assert bruteforce.bf_e2m1(0.75) == 2 and bruteforce.bf_e2m1(0.74) == 1
    assert bruteforce.bf_e4m3(1.0625) == 0x38 and bruteforce.bf_e4m3(1.07) == 0x39
    buf = np.array([1], np.uint8)  # encode(0.0) is 0, so 1 must be reported
    bad = ctypes.c_uint32(0)
    n = bruteforce.bf_compare(2, 0, 1, buf.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), ctypes.byref(bad))
    assert n == 1
