"""GPU parity of the initial-prefill write from FP8 K/V into the NVFP4 cache:
cache bytes (codes and E4M3 scales) bit-exact against the oracle on the same
FP8 bytes, per-tensor FP8 scales and NVFP4 global scales, the global scales
themselves computed by the library and matched bit for bit to the oracle's."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("P,T", [(64, 300), (16, 77), (32, 1)])
def test_requantize_write_fp8_matches_oracle(orc, P, T):
    import nvfp4_quantized_paged_gb300 as nv
    rng = np.random.default_rng(P * 1000 + T)
    Hkv, D = 8, 128
    npages = (T + P - 1) // P + 2
    k8 = rng.integers(0, 0x7F, (T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (T, Hkv, D), dtype=np.uint8) << 7)
    v8 = rng.integers(0, 0x7F, (T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (T, Hkv, D), dtype=np.uint8) << 7)
    s8 = np.array([0.0173, 2.5], np.float32)
    slots = rng.permutation(npages * P)[:T].astype(np.int64)
    if T > 3:
        slots[3] = -1  # skipped token
    # global scales of the decoded values, by the library (decode by torch for the amax input)
    dk8, dv8 = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    sc = torch.from_numpy(s8).cuda()
    g = torch.zeros(2, dtype=torch.float32, device="cuda")
    for kind, x8 in enumerate((dk8, dv8)):
        xf = (x8.view(torch.float8_e4m3fn).float() * sc[kind]).contiguous()
        nv.nvkv_global_scale(xf, g[kind:kind + 1], nv.NVFP4_GLOBAL_DIVISOR)
    kx = (orc_decode(k8) * s8[0]).astype(np.float32)
    vx = (orc_decode(v8) * s8[1]).astype(np.float32)
    g_orc = np.array([orc.global_scale(kx), orc.global_scale(vx)], np.float32)
    assert np.array_equal(g.cpu().numpy(), g_orc)
    cache = nv.Cache(nv.PREC_NVFP4, npages, Hkv, P, device="cuda", kv_scale=g)
    nv.nvfp4_kv_requantize_write_fp8(dk8, dv8, sc, torch.from_numpy(slots).cuda(), g, cache)
    torch.cuda.synchronize()
    assert cache.err.item() == 0
    oc = orc.Cache(orc.PREC_NVFP4, npages, Hkv, P, D, g_orc)
    orc.requantize_write_fp8(oc, k8, v8, s8, slots)
    assert np.array_equal(cache.data.cpu().numpy(), oc.data)


def orc_decode(b):
    """Exact values of E4M3 bytes from their bit fields (float64)."""
    b = np.asarray(b, np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * m / 8)
    return np.where(b & 0x80, -v, v)


def test_quantizer_division_at_every_e2m1_rounding_boundary(orc):
    """Blocks whose scale is exactly 1 (element 0 = 6 g) so den = g, and whose
    other values sit on and one or two ulps around den * t for every E2M1
    rounding boundary t (0.25, 0.75, ..., 5) and a few interior values:
    codes must equal the oracle's, which divides x / den exactly once."""
    import nvfp4_quantized_paged_gb300 as nv
    Hkv, D, P = 2, 128, 16
    rows = []
    for g in (np.float32(0.0137), np.float32(3.1e-5), np.float32(1.7), np.float32(2.0 ** -20)):
        d6 = np.float32(6.0) * g
        bounds = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 3.0]
        vals = []
        for t in bounds:
            c = np.float32(g) * np.float32(t)
            for k in (-2, -1, 0, 1, 2):
                v = c
                for _ in range(abs(k)):
                    v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(-np.inf), dtype=np.float32)
                vals.append(v)
                vals.append(-v)
        vals = np.array(vals, np.float32)
        for i in range(0, len(vals), 15):
            blk = np.zeros(16, np.float32)
            blk[0] = d6
            part = vals[i:i + 15]
            blk[1:1 + len(part)] = part
            rows.append((g, blk))
    # one token-head row per (g, 8 blocks): pack blocks of the same g into rows of 128 values
    by_g = {}
    for g, blk in rows:
        by_g.setdefault(float(g), []).append(blk)
    for g, blks in by_g.items():
        n_rows = (len(blks) + 7) // 8
        data = np.zeros((n_rows * Hkv, D), np.float32)
        flat = np.concatenate(blks + [np.zeros(16, np.float32)] * (n_rows * 8 - len(blks)))
        data[:n_rows].reshape(-1)[:flat.size] = flat
        data[n_rows:] = data[:n_rows]
        T = n_rows
        k = data.reshape(Hkv, T, D).transpose(1, 0, 2).copy()
        gs = np.array([g, g], np.float32)
        slots = np.arange(T, dtype=np.int64)
        npages = (T + P - 1) // P
        cache = nv.Cache(nv.PREC_NVFP4, npages, Hkv, P, device="cuda")
        nv.nvfp4_kv_quantize_write(torch.from_numpy(k).cuda(), torch.from_numpy(k).cuda(),
                                   torch.from_numpy(slots).cuda(), torch.from_numpy(gs).cuda(), cache)
        torch.cuda.synchronize()
        oc = orc.Cache(orc.PREC_NVFP4, npages, Hkv, P, D, gs)
        orc.quantize_write(oc, k, k, slots)
        assert np.array_equal(cache.data.cpu().numpy(), oc.data), g


E4M3_SCALES = np.array([2.0 ** e * (1 + m / 8) for e in range(-6, 9) for m in range(8)] +
                       [2.0 ** -6 * m / 8 for m in range(1, 8)], np.float64)
E4M3_SCALES = E4M3_SCALES[E4M3_SCALES <= 448.0]
E2M1_POINTS = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _near_boundary_blocks(rng, g, n_blocks):
    """Blocks whose element 0 fixes an E4M3-representable scale s (so den =
    fl(s g)) and whose other elements sit a few ulps around den * t for E2M1
    rounding boundaries and grid points t, plus plain random values."""
    blks = np.zeros((n_blocks, 16), np.float32)
    for i in range(n_blocks):
        s = np.float32(rng.choice(E4M3_SCALES))
        blks[i, 0] = np.float32(6.0) * g * s if rng.random() < 0.5 else -(np.float32(6.0) * g * s)
        den = np.float32(s * np.float32(g))
        for j in range(1, 16):
            if rng.random() < 0.8:
                v = np.float32(den * np.float32(rng.choice(E2M1_POINTS)))
                for _ in range(int(rng.integers(0, 3))):
                    v = np.nextafter(v, np.float32(np.inf) if rng.random() < 0.5 else np.float32(0), dtype=np.float32)
            else:
                v = np.float32(rng.normal() * 6.0 * float(den))
            blks[i, j] = -v if rng.random() < 0.5 else v
    return blks


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_quantizer_random_scales_near_boundaries(orc, seed):
    """Random global scales over 60 decades and values placed on and a few ulps
    around every E2M1 rounding boundary of random E4M3 block scales: the NVFP4
    and FP8 writes must give the oracle's bytes (one exact division per value
    there).  Covers the reciprocal-bracket code selection and its fallback."""
    import nvfp4_quantized_paged_gb300 as nv
    rng = np.random.default_rng(seed)
    Hkv, D, P = 2, 128, 16
    for g in [np.float32(10.0 ** rng.uniform(-30, 30)) for _ in range(6)] + [np.float32(1.0)]:
        n_rows = 24
        blks = _near_boundary_blocks(rng, g, n_rows * Hkv * (D // 16))
        k = blks.reshape(n_rows, Hkv, D)
        v = np.ascontiguousarray(k[::-1])
        slots = rng.permutation(n_rows * 2)[:n_rows].astype(np.int64)
        npages = (2 * n_rows + P - 1) // P
        for prec, gs in ((nv.PREC_NVFP4, np.array([g, g], np.float32)),
                         (nv.PREC_FP8, np.array([g * 7, g * 7], np.float32))):
            cache = nv.Cache(prec, npages, Hkv, P, device="cuda")
            write = nv.nvfp4_kv_quantize_write if prec == nv.PREC_NVFP4 else nv.fp8_kv_quantize_write
            write(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda(),
                  torch.from_numpy(gs).cuda(), cache)
            torch.cuda.synchronize()
            oc = orc.Cache(orc.PREC_NVFP4 if prec == nv.PREC_NVFP4 else orc.PREC_FP8, npages, Hkv, P, D, gs)
            orc.quantize_write(oc, k, v, slots)
            assert np.array_equal(cache.data.cpu().numpy(), oc.data), (prec, float(g))
