"""The prefill write's threshold method, held against the oracle's write.

The CUDA prefill write (FP8 K/V into the NVFP4 cache) does not divide per
value: for each scale byte it finds the seven magnitudes T_1..T_7 at which the
E2M1 code of fl(x / den) steps up, by bisection, and then counts, four bytes at
a time, how many of them a value's magnitude reaches (a byte-lane subtraction
with a guard bit: bit 7 of (e | 0x80) - T is set exactly when e >= T; the seven
flags are monotone, so the code's bits are f4, f2^f4^f6 and f1^...^f7).  This
rests on the code being monotone in the byte's magnitude and odd in its sign.
Here the method is restated in Python (thresholds by bisection with the
oracle's own encoder on FP32 quotients, the flag arithmetic on 32-bit words) and
must reproduce the oracle's requantize write for every (largest magnitude,
byte) pair a block can hold, at several input and global scales.
"""
import numpy as np
import pytest


def _e4m3(b):
    b = np.asarray(b, np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * m / 8)
    return np.where(b & 0x80, -v, v)


def _blocks():
    """Blocks of 16 E4M3 bytes: for every largest magnitude m (1..126), the
    block leads with +m and the other 15 values run through every byte whose
    magnitude is <= m (both signs)."""
    out = []
    for m in range(1, 127):
        rest = [s | e for e in range(m + 1) for s in (0, 0x80)]
        for i in range(0, len(rest), 15):
            chunk = rest[i:i + 15]
            chunk += [0] * (15 - len(chunk))
            out.append([m] + chunk)
    return np.array(out, np.uint8)


def _thresholds(orc, xs, den):
    """T_1..T_7: the least magnitude e in [0, 127) whose code magnitude is >= k
    (128 when none), by bisection, codes from the oracle's encoder."""
    def mag(e):
        return orc.e2m1_encode(float(np.float32(xs[e]) / np.float32(den))) & 7
    ts = []
    for k in range(1, 8):
        lo, hi = 0, 127
        while lo < hi:
            mid = (lo + hi) // 2
            if mag(mid) >= k:
                hi = mid
            else:
                lo = mid + 1
        ts.append(128 if lo == 127 else lo)
    return ts


def _codes_by_flags(block, ts):
    """The 16 codes of a block by the byte-lane flag arithmetic."""
    codes = []
    for q in range(4):
        w = int.from_bytes(bytes(block[4 * q:4 * q + 4]), "little")
        a = w | 0x80808080
        f = [(a - t * 0x01010101) & 0xFFFFFFFF for t in ts]
        b1 = f[1] ^ f[3] ^ f[5]
        b0 = b1 ^ f[0] ^ f[2] ^ f[4] ^ f[6]
        for j in range(4):
            bit = lambda x: (x >> (8 * j + 7)) & 1
            codes.append(bit(w) << 3 | bit(f[3]) << 2 | bit(b1) << 1 | bit(b0))
    return codes


@pytest.mark.parametrize("s8,g", [(0.0137, None), (1.0, 448.0 / 2688.0), (3.3e-3, 1.7e-5), (2.5, 0.9)])
def test_thresholds_reproduce_the_oracle_write(orc, s8, g):
    blocks = _blocks()
    D, Hkv, P = 128, 1, 16
    nb = -(-len(blocks) // (D // 16)) * (D // 16)
    padded = np.zeros((nb, 16), np.uint8)
    padded[:len(blocks)] = blocks
    T = nb // (D // 16)
    k8 = padded.reshape(T, Hkv, D)
    s = np.array([s8, s8], np.float32)
    if g is None:
        g = orc.global_scale((_e4m3(k8).astype(np.float32) * s[0]).astype(np.float32))
    g = np.float32(g)
    pages = -(-T // P)
    c = orc.Cache(orc.PREC_NVFP4, pages, Hkv, P, D, [g, g])
    orc.requantize_write_fp8(c, k8, k8, s, np.arange(T, dtype=np.int64))
    xs = [np.float32(np.float32(_e4m3(e)) * s[0]) for e in range(128)]
    data, scale = c.k_data, c.k_scale
    cache_thr = {}
    for t in range(T):
        page, off = t // P, t % P
        got = data[page, 0, off]
        got_codes = np.stack([got & 15, got >> 4], -1).reshape(D)
        for blk in range(D // 16):
            block = k8[t, 0, 16 * blk:16 * blk + 16]
            sb = int(scale[page, 0, off, blk])
            den = np.float32(np.float32(_e4m3(sb)) * g)
            want = got_codes[16 * blk:16 * blk + 16]
            if den == 0:
                assert not want.any()
                continue
            if sb not in cache_thr:
                cache_thr[sb] = _thresholds(orc, xs, den)
            assert _codes_by_flags(block, cache_thr[sb]) == [int(v) for v in want], (t, blk, sb)
