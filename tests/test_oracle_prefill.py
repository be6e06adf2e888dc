"""Pins of the oracle's initial-prefill write from FP8 K/V into the NVFP4 cache.

Closed form: FP8 bytes that encode NVFP4 grid values (every 16-block holds a
+-6 * 2^e element, the block's scale is the E4M3 power of two 2^e, s8 = g) must
requantize to exactly those E2M1 codes and scale bytes.  Decode identity: the
requantized cache equals the plain quantized write of the FP32 values
E4M3(byte) * s8, decoded here with numpy from the E4M3 bit fields.
"""
import numpy as np

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e4m3(b):
    b = np.asarray(b, np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * m / 8)
    return np.where(b & 0x80, -v, v)


def _e4m3_byte_of(x):
    """E4M3 byte of an exactly representable value (lookup over all finite bytes)."""
    table = {float(_e4m3(b)): b for b in range(256) if (b & 0x7F) != 0x7F}
    table[0.0] = 0
    return np.vectorize(lambda v: table[float(v)])(x).astype(np.uint8)


def test_requantize_of_grid_values_is_exact(orc):
    rng = np.random.default_rng(1)
    T, Hkv, D, P = 5, 2, 128, 16
    g = np.float32(0.125)
    codes = rng.integers(0, 8, (2, T, Hkv, D // 16, 16))
    codes[..., 3] = 7  # the block max: 6 * 2^e
    signs = rng.integers(0, 2, codes.shape)
    e = rng.integers(-6, 5, (2, T, Hkv, D // 16))
    vals = E2M1[codes] * np.where(signs == 1, -1, 1) * 2.0 ** e[..., None]  # E4M3-exact
    k8 = _e4m3_byte_of(vals[0].reshape(T, Hkv, D))
    v8 = _e4m3_byte_of(vals[1].reshape(T, Hkv, D))
    c = orc.Cache(orc.PREC_NVFP4, 2, Hkv, P, D, [g, g])
    slots = np.array([3, 17, -1, 0, 31], np.int64)
    orc.requantize_write_fp8(c, k8, v8, [g, g], slots)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, off = slot // P, slot % P
        for kind, (data, scale) in enumerate(((c.k_data, c.k_scale), (c.v_data, c.v_scale))):
            got = data[page, :, off]  # [Hkv, D/2]
            got_codes = np.stack([got & 15, got >> 4], -1).reshape(Hkv, D)
            want = (codes[kind, t] | (signs[kind, t] << 3)).reshape(Hkv, D)
            np.testing.assert_array_equal(got_codes & 7, want & 7)
            nz = (want & 7) != 0  # the sign of a zero code is not fixed by the value (E4M3 +0 input)
            np.testing.assert_array_equal((got_codes >> 3)[nz], (want >> 3)[nz])
            np.testing.assert_array_equal(scale[page, :, off], _e4m3_byte_of(2.0 ** e[kind, t]))


def test_requantize_equals_write_of_decoded_values(orc):
    rng = np.random.default_rng(2)
    T, Hkv, D, P = 9, 2, 128, 8
    k8 = rng.integers(0, 0x7F, (T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (T, Hkv, D), dtype=np.uint8) << 7)
    v8 = rng.integers(0, 0x7F, (T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (T, Hkv, D), dtype=np.uint8) << 7)
    s8 = np.array([0.0137, 0.51], np.float32)
    kx = (_e4m3(k8).astype(np.float32) * s8[0]).astype(np.float32)  # one FP32 multiply each
    vx = (_e4m3(v8).astype(np.float32) * s8[1]).astype(np.float32)
    g = np.array([orc.global_scale(kx), orc.global_scale(vx)], np.float32)
    slots = rng.permutation(3 * P)[:T].astype(np.int64)
    a = orc.Cache(orc.PREC_NVFP4, 3, Hkv, P, D, g)
    b = orc.Cache(orc.PREC_NVFP4, 3, Hkv, P, D, g)
    orc.requantize_write_fp8(a, k8, v8, s8, slots)
    orc.quantize_write(b, kx, vx, slots)
    np.testing.assert_array_equal(a.data, b.data)
