"""Pins of the oracle's paged GQA decode attention and workspace dequant.

The brute force here dequantizes the raw cache bytes itself (code table and
E4M3 bit fields written independently of the oracle), gathers the tokens of
each sequence contiguously and runs a dense FP64 softmax with numpy.  The
oracle walks pages through the block table; both must agree to 1e-12 for
contiguous and permuted tables and for page sizes 1, 16 and 64.
"""
import numpy as np
import pytest

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _e4m3(b):
    b = np.asarray(b, np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * m / 8)
    return np.where(b & 0x80, -v, v)


def _bf16_bits(x):
    """Round FP32 to BF16 bit patterns (ties to even)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def _bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _brute_dense(cache, q_bits, block_table, seq_lens):
    B, Hq, D = q_bits.shape
    G = Hq // cache.Hkv
    out = np.zeros((B, Hq, D))
    q = _bf16_value(q_bits)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        t = np.arange(L)
        pages = block_table[b, t // cache.P]
        offs = t % cache.P
        for h in range(cache.Hkv):
            def deq(data, scale, g):
                rows = data[pages, h, offs]  # [L, D/2] or [L, D]
                if cache.prec == 0:
                    c = np.stack([rows & 15, rows >> 4], -1).reshape(L, D)
                    val = E2M1[c & 7] * np.where(c & 8, -1, 1)
                    s = _e4m3(scale[pages, h, offs])
                    return val * np.repeat(s, 16, axis=1) * float(g)
                return _e4m3(rows) * float(g)
            K = deq(cache.k_data, cache.k_scale, cache.g[0])
            V = deq(cache.v_data, cache.v_scale, cache.g[1])
            for j in range(G):
                s = K @ q[b, h * G + j] / np.sqrt(D)
                p = np.exp(s - s.max())
                out[b, h * G + j] = p @ V / p.sum()
    return out


def _random_cache(orc, prec, B, Hkv, P, D, lens, table, seed):
    rng = np.random.default_rng(seed)
    maxp = max(1, int(max((l + P - 1) // P for l in lens)))
    npages = B * maxp + 3
    perm = rng.permutation(npages) if table == "permuted" else np.arange(npages)
    bt = perm[:B * maxp].reshape(B, maxp).astype(np.int32)
    k = (rng.standard_normal((B, maxp * P, Hkv, D)) * rng.uniform(0.5, 4, (1, 1, Hkv, D))).astype(np.float32)
    v = rng.standard_normal((B, maxp * P, Hkv, D)).astype(np.float32)
    div = orc.NVFP4_GLOBAL_DIVISOR if prec == 0 else orc.FP8_GLOBAL_DIVISOR
    g = [orc.global_scale(k, div), orc.global_scale(v, div)]
    c = orc.Cache(prec, npages, Hkv, P, D, g, fill=0x77)
    for b in range(B):
        t = np.arange(lens[b])
        slots = bt[b, t // P].astype(np.int64) * P + t % P
        orc.quantize_write(c, k[b, :lens[b]], v[b, :lens[b]], slots)
    return c, bt


@pytest.mark.parametrize("prec", [0, 1])
@pytest.mark.parametrize("P,table", [(16, "contiguous"), (16, "permuted"), (1, "permuted"), (64, "permuted")])
def test_paged_equals_brute_force_dense(orc, prec, P, table):
    B, Hq, Hkv, D = 3, 8, 2, 128
    lens = [37, 64, 5] if P != 64 else [130, 64, 1]
    c, bt = _random_cache(orc, prec, B, Hkv, P, D, lens, table, seed=P + prec)
    q = _bf16_bits(np.random.default_rng(9).standard_normal((B, Hq, D)))
    sl = np.array(lens, np.int32)
    got = orc.paged_decode_attention(c, q, bt, sl)
    want = _brute_dense(c, q, bt, sl)
    assert np.max(np.abs(got - want)) <= 1e-12 * max(1.0, np.abs(want).max())


@pytest.mark.parametrize("splits", [1, 7, 64])
def test_split_lse_merge_equals_single_softmax(orc, splits):
    B, Hq, Hkv, D, P = 2, 8, 2, 128, 16
    lens = [200, 33]
    c, bt = _random_cache(orc, 0, B, Hkv, P, D, lens, "permuted", seed=5)
    q = _bf16_bits(np.random.default_rng(1).standard_normal((B, Hq, D)) * 3)
    sl = np.array(lens, np.int32)
    a = orc.paged_decode_attention(c, q, bt, sl, num_splits=0)
    b = orc.paged_decode_attention(c, q, bt, sl, num_splits=splits)
    assert np.max(np.abs(a - b)) <= 1e-12 * max(1.0, np.abs(a).max())


def test_gqa_head_mapping(orc):
    """Query head h reads KV head h // G: with V constant per KV head, the
    output of head h is that constant."""
    B, Hq, Hkv, D, P = 1, 8, 4, 32, 4
    c = orc.Cache(0, 4, Hkv, P, D, [1.0, 1.0])
    L = 10
    rng = np.random.default_rng(0)
    k = rng.standard_normal((L, Hkv, D)).astype(np.float32)
    v = np.zeros((L, Hkv, D), np.float32)
    for h in range(Hkv):
        v[:, h, :] = [1.0, 2.0, 3.0, 4.0][h]  # exact on the grid with g = 1, S = 1 or 2/3..
    orc.quantize_write(c, k, v, np.arange(L, dtype=np.int64))
    bt = np.arange(4, dtype=np.int32).reshape(1, 4)
    out = orc.paged_decode_attention(c, _bf16_bits(rng.standard_normal((B, Hq, D))), bt, np.array([L], np.int32))
    vh = [orc.gather_dequant(c, "v", bt[0], L, h)[0, 0] for h in range(Hkv)]
    for h in range(Hq):
        assert np.allclose(out[0, h], vh[h // 2], rtol=0, atol=1e-12)


def test_closed_forms(orc):
    """One visible token returns its value row exactly; identical keys give the
    mean of the values; L = 0 gives zeros."""
    Hq, Hkv, D, P = 4, 1, 32, 8
    rng = np.random.default_rng(2)
    c = orc.Cache(0, 2, Hkv, P, D, [0.01, 0.02])
    k = np.tile(rng.standard_normal((1, Hkv, D)), (P, 1, 1)).astype(np.float32)
    v = rng.standard_normal((P, Hkv, D)).astype(np.float32)
    orc.quantize_write(c, k, v, np.arange(P, dtype=np.int64))
    bt = np.array([[0, 1], [0, 1], [0, 1]], np.int32)
    q = _bf16_bits(rng.standard_normal((3, Hq, D)))
    out = orc.paged_decode_attention(c, q, bt, np.array([1, P, 0], np.int32))
    V = orc.gather_dequant(c, "v", bt[0], P, 0)
    for h in range(Hq):
        assert np.array_equal(out[0, h], V[0])
        assert np.allclose(out[1, h], V.mean(0), rtol=0, atol=1e-13)
        assert not out[2, h].any()


def test_workspace_dequant_error_bound_and_exact_cases(orc):
    """Workspace bytes decode (times ws_scale) to the cached value within half
    an E4M3 step, and exactly when the value is representable."""
    Hkv, D, P = 2, 64, 16
    rng = np.random.default_rng(7)
    lens = [40, 17]
    c, bt = _random_cache(orc, 0, 2, Hkv, P, D, lens, "permuted", seed=11)
    ws = np.array([6 * c.g[0], 6 * c.g[1]], np.float32)
    wk, wv = orc.dequant_to_fp8_workspace(c, bt, [1, 0], [17, 40], ws)
    assert wk.shape == (57, Hkv, D)
    for which, w, g, s in (("k", wk, c.g[0], ws[0]), ("v", wv, c.g[1], ws[1])):
        rows = np.concatenate([orc.gather_dequant(c, which, bt[1], 17, h)[:, None] for h in range(Hkv)], 1)
        rows = np.concatenate([rows, np.concatenate(
            [orc.gather_dequant(c, which, bt[0], 40, h)[:, None] for h in range(Hkv)], 1)], 0)
        got = _e4m3(w) * float(s)
        y = np.abs(rows) / float(s)
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
        half_step = 0.5 * 2.0 ** (e - 3) * float(s)
        assert np.all(np.abs(got - rows) <= half_step * (1 + 1e-6) + 1e-30)
    del rng


def test_workspace_exact_when_representable(orc):
    """With ws_scale = g the ratio r is 1 and every e2m1 * S product that is an
    E4M3 value maps to exactly that byte."""
    Hkv, D, P = 1, 16, 4
    c = orc.Cache(0, 1, Hkv, P, D, [1.0, 1.0])
    c.data[0, 0, c.positions("k_data")[0]] = np.array([0x21, 0x43, 0x65, 0x07, 0x98, 0xBA, 0xDC, 0x0F], np.uint8)
    c.data[0, 0, c.positions("k_scale")[0, 0]] = 0x38  # S = 1
    bt = np.zeros((1, 1), np.int32)
    wk, _ = orc.dequant_to_fp8_workspace(c, bt, [0], [1], np.array([1.0, 1.0], np.float32))
    vals = _e4m3(wk[0, 0])
    codes = np.stack([c.k_data[0, 0, 0] & 15, c.k_data[0, 0, 0] >> 4], -1).reshape(16)
    want = E2M1[codes & 7] * np.where(codes & 8, -1, 1)
    assert np.array_equal(vals, want)
