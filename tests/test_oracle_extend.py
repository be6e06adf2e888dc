"""Pins of the oracle's chunked-extend path: the chunk's FP8 workspace append
and the causal FP8 attention over [prefix || chunk].

The brute force decodes E4M3 from its bit fields here (independently of the
oracle), builds each sequence's dense causal mask with numpy and runs a FP64
softmax; closed forms (one visible key, identical keys), causality, and the
decode oracle on an FP8 cache holding the same bytes pin the rest.
"""
import numpy as np
import pytest


def _e4m3(b):
    b = np.asarray(b, np.int64)
    e, m = (b >> 3) & 15, b & 7
    v = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * m / 8)
    return np.where(b & 0x80, -v, v)


def _bf16_value(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_bits(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + ((u >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint16)


def _problem(rng, q_lens, kv_lens, Hq, Hkv, D, gap=3):
    """Random workspace bytes (finite E4M3, both signs) with a gap of unused
    rows between sequences, and BF16 queries."""
    n = len(kv_lens)
    cu_kv = np.zeros(n, np.int64)
    r = 0
    for i in range(n):
        cu_kv[i] = r
        r += kv_lens[i] + gap
    rows = r
    codes = rng.integers(0, 0x7F, (rows, Hkv, D), dtype=np.uint8)  # no NaN (0x7F)
    signs = rng.integers(0, 2, (rows, Hkv, D), dtype=np.uint8) << 7
    ws_k = (codes | signs).astype(np.uint8)
    ws_v = (rng.integers(0, 0x7F, (rows, Hkv, D), dtype=np.uint8) | signs[::-1]).astype(np.uint8)
    cu_q = np.zeros(n + 1, np.int64)
    cu_q[1:] = np.cumsum(q_lens)
    q = _bf16_bits(rng.standard_normal((int(cu_q[-1]), Hq, D)) * 0.3)
    return q, cu_q, ws_k, ws_v, cu_kv, np.asarray(kv_lens, np.int32)


def _brute(q, cu_q, ws_k, ws_v, cu_kv, kv_lens, ws_scale, sm_scale):
    Tq, Hq, D = q.shape
    Hkv = ws_k.shape[1]
    G = Hq // Hkv
    out = np.zeros((Tq, Hq, D))
    for i in range(len(kv_lens)):
        L, nq = int(kv_lens[i]), int(cu_q[i + 1] - cu_q[i])
        if nq == 0:
            continue
        K = _e4m3(ws_k[cu_kv[i]:cu_kv[i] + L]) * float(np.float32(ws_scale[0]))  # [L, Hkv, D]
        V = _e4m3(ws_v[cu_kv[i]:cu_kv[i] + L]) * float(np.float32(ws_scale[1]))
        qpos = L - nq + np.arange(nq)
        mask = np.arange(L)[None, :] <= qpos[:, None]  # [nq, L]
        Q = _bf16_value(q[cu_q[i]:cu_q[i + 1]])  # [nq, Hq, D]
        for qh in range(Hq):
            s = Q[:, qh] @ K[:, qh // G].T * sm_scale  # [nq, L]
            s = np.where(mask, s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            out[cu_q[i]:cu_q[i + 1], qh] = p @ V[:, qh // G] / p.sum(axis=1, keepdims=True)
    return out


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (16, 2)])
def test_extend_equals_dense_causal_brute_force(orc, Hq, Hkv):
    rng = np.random.default_rng(Hq * 7 + Hkv)
    D = 32
    q_lens, kv_lens = [5, 1, 9, 0], [12, 1, 9, 4]  # prefixes 7, 0, 0, 4
    q, cu_q, wk, wv, cu_kv, kl = _problem(rng, q_lens, kv_lens, Hq, Hkv, D)
    ws_scale = np.array([0.03125, 0.0078125], np.float32)
    got = orc.fp8_extend_attention(q, cu_q, wk, wv, cu_kv, kl, ws_scale, 0.0)
    ref = _brute(q, cu_q, wk, wv, cu_kv, kl, ws_scale, 1.0 / np.sqrt(D))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_closed_forms(orc):
    rng = np.random.default_rng(5)
    Hq, Hkv, D = 4, 2, 16
    ws_scale = np.array([0.5, 0.25], np.float32)
    # (a) no prefix: the chunk's first query sees only its own key -> V row 0
    q, cu_q, wk, wv, cu_kv, kl = _problem(rng, [6], [6], Hq, Hkv, D, gap=0)
    got = orc.fp8_extend_attention(q, cu_q, wk, wv, cu_kv, kl, ws_scale)
    for qh in range(Hq):
        np.testing.assert_array_equal(got[0, qh], _e4m3(wv[0, qh // 2]) * 0.25)
    # (b) identical keys: uniform weights, query j (position p + j) averages V[0 .. p + j]
    q, cu_q, wk, wv, cu_kv, kl = _problem(rng, [5], [11], Hq, Hkv, D, gap=0)
    wk[:] = wk[0]
    got = orc.fp8_extend_attention(q, cu_q, wk, wv, cu_kv, kl, ws_scale)
    Vd = _e4m3(wv) * 0.25
    for j in range(5):
        pos = 11 - 5 + j
        for qh in range(Hq):
            np.testing.assert_allclose(got[j, qh], Vd[:pos + 1, qh // 2].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_causality(orc):
    """Keys and values after a query's position never change its output."""
    rng = np.random.default_rng(9)
    Hq, Hkv, D = 8, 2, 16
    q, cu_q, wk, wv, cu_kv, kl = _problem(rng, [8], [20], Hq, Hkv, D, gap=0)
    ws_scale = np.array([0.125, 0.125], np.float32)
    a = orc.fp8_extend_attention(q, cu_q, wk, wv, cu_kv, kl, ws_scale)
    wk2, wv2 = wk.copy(), wv.copy()
    wk2[16:] = rng.integers(0, 0x7F, wk2[16:].shape, dtype=np.uint8)  # positions 16..19 = queries 4..7
    wv2[16:] = rng.integers(0, 0x7F, wv2[16:].shape, dtype=np.uint8)
    b = orc.fp8_extend_attention(q, cu_q, wk2, wv2, cu_kv, kl, ws_scale)
    np.testing.assert_array_equal(a[:4], b[:4])
    assert np.all(np.abs(a[4:] - b[4:]).max(axis=(1, 2)) > 0)


def test_last_query_equals_decode_over_an_fp8_cache(orc):
    """The chunk's last query sees every position: it equals the decode
    oracle over an FP8 paged cache that holds the same bytes (s8 = ws_scale)."""
    rng = np.random.default_rng(11)
    Hq, Hkv, D, P = 8, 2, 32, 16
    L, nq = 45, 7
    q, cu_q, wk, wv, cu_kv, kl = _problem(rng, [nq], [L], Hq, Hkv, D, gap=0)
    ws_scale = np.array([0.0625, 0.03125], np.float32)
    got = orc.fp8_extend_attention(q, cu_q, wk, wv, cu_kv, kl, ws_scale)
    npages = (L + P - 1) // P
    c = orc.Cache(orc.PREC_FP8, npages, Hkv, P, D, [ws_scale[0], ws_scale[1]], fill=0)
    k = (_e4m3(wk[:L]) * float(ws_scale[0])).astype(np.float32)  # exact: x / s8 is the E4M3 value again
    v = (_e4m3(wv[:L]) * float(ws_scale[1])).astype(np.float32)
    orc.quantize_write(c, k, v, np.arange(L, dtype=np.int64))
    bt = np.arange(npages, dtype=np.int32)[None]
    dec = orc.paged_decode_attention(c, q[nq - 1:nq], bt, np.array([L], np.int32))
    np.testing.assert_allclose(got[nq - 1], dec[0], rtol=1e-12, atol=1e-14)


def test_workspace_append(orc):
    rng = np.random.default_rng(3)
    Hkv, D, T = 2, 16, 6
    s = np.array([0.5, 0.03125], np.float32)
    codes = rng.integers(0, 0x7F, (T, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (T, Hkv, D), dtype=np.uint8) << 7)
    k = (_e4m3(codes) * float(s[0])).astype(np.float32)  # exactly representable: round trip
    v = (_e4m3(codes) * float(s[1])).astype(np.float32)
    k[0, 0, :2] = [1e6, -1e6]  # saturate to +-448
    rows = np.array([4, -1, 0, 7, 2, 5], np.int64)
    wk = np.full((9, Hkv, D), 0xAA, np.uint8)
    wv = np.full((9, Hkv, D), 0xAA, np.uint8)
    orc.fp8_workspace_append(wk, wv, k, v, rows, s)
    want = codes.copy()
    want[0, 0, :2] = [0x7E, 0xFE]
    for t, r in enumerate(rows):
        if r >= 0:
            np.testing.assert_array_equal(wk[r], want[t])
            np.testing.assert_array_equal(wv[r], codes[t])
    for r in (1, 3, 6, 8):  # rows nobody wrote
        assert np.all(wk[r] == 0xAA) and np.all(wv[r] == 0xAA)
    with pytest.raises(ValueError):
        orc.fp8_workspace_append(wk, wv, k, v, np.array([0, 1, 2, 3, 4, 9]), s)
