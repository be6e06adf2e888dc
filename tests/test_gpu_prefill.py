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
