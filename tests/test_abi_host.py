"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function the header declares, and rejects bad arguments with the
documented status before touching the device."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def nv():
    import nvfp4_quantized_paged_gb300 as nv
    return nv


def test_library_exports_every_header_function(nv):
    L = nv.lib()
    names = nv.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(nv.SIGNATURES)


def _desc(nv, **kw):
    d = nv.nvkv_cache()
    d.prec, d.num_pages, d.page_size, d.num_kv_heads, d.head_dim = 0, 4, 16, 2, 128
    d.data = 0x10000
    d.kv_scale = 0x20000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def _write(nv, d, fn="nvfp4_kv_quantize_write", n=1):
    return getattr(nv.lib(), fn)(0x30000, 0x30000, 0, n, 0x40000, None, ctypes.byref(d), None)


def test_write_argument_checks(nv):
    L = nv.lib()
    assert L.nvfp4_kv_quantize_write(None, None, 0, 1, None, None, None, None) == nv.NVKV_ERR_INVALID_ARG
    assert _write(nv, _desc(nv, head_dim=64)) == nv.NVKV_ERR_UNSUPPORTED
    assert _write(nv, _desc(nv, page_size=48)) == nv.NVKV_ERR_UNSUPPORTED
    assert _write(nv, _desc(nv, page_size=128)) == nv.NVKV_ERR_UNSUPPORTED
    assert _write(nv, _desc(nv, prec=1)) == nv.NVKV_ERR_INVALID_ARG           # precision mismatch
    assert _write(nv, _desc(nv, prec=0), "fp8_kv_quantize_write") == nv.NVKV_ERR_INVALID_ARG
    assert _write(nv, _desc(nv, data=None)) == nv.NVKV_ERR_INVALID_ARG
    assert _write(nv, _desc(nv, data=0x10008)) == nv.NVKV_ERR_UNSUPPORTED     # 16-byte alignment
    assert _write(nv, _desc(nv), n=0) == nv.NVKV_OK                           # nothing to do
    assert _write(nv, _desc(nv), n=-1) == nv.NVKV_ERR_INVALID_ARG


def test_decode_argument_checks(nv):
    L = nv.lib()
    d = _desc(nv)
    args = lambda **kw: dict(dict(q=0x50000, bt=0x60000, mp=4, sl=0x70000, B=2, Hq=8, prec=0, sm=0.0, ns=0,
                                  ws=0x80000, wsb=1 << 20, out=0x90000), **kw)

    def call(**kw):
        a = args(**kw)
        return L.nvfp4_paged_decode_attention(a["q"], ctypes.byref(d), a["bt"], a["mp"], a["sl"], a["B"], a["Hq"],
                                              a["prec"], a["sm"], a["ns"], a["ws"], a["wsb"], a["out"], None)
    assert call(prec=1) == nv.NVKV_ERR_INVALID_ARG          # layer_precision != cache->prec
    assert call(Hq=7) == nv.NVKV_ERR_INVALID_ARG            # Hq not a multiple of Hkv
    assert call(Hq=32) == nv.NVKV_ERR_UNSUPPORTED           # group of 16 > 8
    assert call(B=2000) == nv.NVKV_ERR_UNSUPPORTED          # batch above 1024
    assert call(ns=4, wsb=16) == nv.NVKV_ERR_WORKSPACE_TOO_SMALL
    assert call(out=0x90004) == nv.NVKV_ERR_UNSUPPORTED     # alignment
    assert call(B=0) == nv.NVKV_OK


def test_workspace_size_arithmetic(nv):
    # explicit splits need no device: one 4-byte arrival counter per (sequence,
    # KV head), rounded up to 256 B, then 2 partial slots per CTA
    slot = (8 * 128 + 16) * 4
    assert nv.nvkv_decode_workspace_size(16, 32, 8, 128, 4) == 512 + 16 * 8 * 4 * 2 * slot
    assert nv.nvkv_decode_workspace_size(3, 16, 2, 128, 1) == 256 + 3 * 2 * 1 * 2 * slot
    assert nv.nvkv_decode_workspace_size(16, 32, 8, 64, 4) == 0
    assert nv.nvkv_decode_workspace_size(16, 32, 2, 128, 4) == 0  # group of 16


def test_noalloc_refuses_problems_beyond_its_scratch(nv):
    # batch x Hkv arrival counters (4 B each) plus one CTA's two partial slots
    # must fit in the fixed array; larger problems are refused on the host,
    # before any CUDA call (so this runs without a GPU)
    L = nv.lib()
    cap = nv.NVKV_NOALLOC_SCRATCH_BYTES
    slot = (8 * 128 + 16) * 4
    hkv = 2048                                   # 1024 x 2048 x 4 B = the whole array
    assert 1024 * hkv * 4 + 2 * slot > cap
    d = _desc(nv, num_kv_heads=hkv)
    st = L.nvfp4_paged_decode_attention_noalloc(0x50000, ctypes.byref(d), 0x60000, 4, 0x70000, 1024, hkv, 0, 0.0,
                                                0, 0x90000, None)
    assert st == nv.NVKV_ERR_WORKSPACE_TOO_SMALL


def test_other_entry_points_reject_bad_arguments(nv):
    L = nv.lib()
    assert L.nvkv_global_scale(None, 0, 5, 2688.0, None, None) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvkv_global_scale(0x10000, 0, 5, 0.0, 0x20000, None) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvkv_amax_update(0x10000, 3, 5, 0x20000, None) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvkv_encode_e2m1(None, 4, None, None) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvkv_encode_e4m3(None, 0, None, None) == nv.NVKV_OK
    d = _desc(nv, prec=1)
    assert L.nvfp4_kv_dequant_to_fp8_workspace(0x1000, 4, 0x1000, 0x1000, 0x1000, 2, ctypes.byref(d), 0x1000,
                                               0x2000, 0x3000, 10, None) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvkv_status_string(4) == b"workspace too small"


def test_extend_and_prefill_argument_checks(nv):
    L = nv.lib()
    # scratch size: 2 (K, V) x Hkv x (ceil(rows / 8) + 16 groups) x 2 KB; 0 for a bad head_dim
    assert nv.fp8_extend_scratch_size(100, 8, 128) == 2 * 8 * (13 + 16) * 2048
    assert nv.fp8_extend_scratch_size(0, 2, 128) == 2 * 2 * 16 * 2048
    assert nv.fp8_extend_scratch_size(100, 8, 64) == 0

    def ext(**kw):
        a = dict(q=0x10000, cu_q=0x20000, n=2, maxq=64, Hq=32, wk=0x30000, wv=0x40000, cu_kv=0x50000,
                 kl=0x60000, Hkv=8, D=128, rows=100, s=0x70000, sm=0.0, scr=0x80000,
                 scrb=nv.fp8_extend_scratch_size(100, 8, 128), out=0x90000)
        a.update(kw)
        return L.fp8_chunked_extend_attention(a["q"], a["cu_q"], a["n"], a["maxq"], a["Hq"], a["wk"], a["wv"],
                                              a["cu_kv"], a["kl"], a["Hkv"], a["D"], a["rows"], a["s"], a["sm"],
                                              a["scr"], a["scrb"], a["out"], None, None)
    assert ext(D=64) == nv.NVKV_ERR_UNSUPPORTED                 # head_dim 128 only
    assert ext(Hq=24) == nv.NVKV_ERR_UNSUPPORTED                # group of 3: not a power of two
    assert ext(Hq=30) == nv.NVKV_ERR_INVALID_ARG                # Hq not a multiple of Hkv
    assert ext(scrb=1024) == nv.NVKV_ERR_WORKSPACE_TOO_SMALL
    assert ext(scr=None) == nv.NVKV_ERR_INVALID_ARG
    assert ext(out=0x90008) == nv.NVKV_ERR_UNSUPPORTED          # 16-byte alignment
    assert ext(n=-1) == nv.NVKV_ERR_INVALID_ARG
    assert ext(n=0) == nv.NVKV_OK and ext(maxq=0) == nv.NVKV_OK  # nothing to do

    def app(**kw):
        a = dict(k=0x10000, v=0x20000, dt=0, T=5, rows=0x30000, Hkv=8, D=128, s=0x40000, wk=0x50000,
                 wv=0x60000, wr=100)
        a.update(kw)
        return L.fp8_workspace_append_chunk(a["k"], a["v"], a["dt"], a["T"], a["rows"], a["Hkv"], a["D"], a["s"],
                                            a["wk"], a["wv"], a["wr"], None, None)
    assert app(D=100) == nv.NVKV_ERR_UNSUPPORTED
    assert app(dt=5) == nv.NVKV_ERR_INVALID_ARG
    assert app(k=None) == nv.NVKV_ERR_INVALID_ARG
    assert app(wk=0x50004) == nv.NVKV_ERR_UNSUPPORTED
    assert app(T=0) == nv.NVKV_OK

    d = _desc(nv)
    assert L.nvfp4_kv_requantize_write_fp8(0x10000, 0x20000, None, 3, 0x30000, None, ctypes.byref(d),
                                           None) == nv.NVKV_ERR_INVALID_ARG   # no FP8 scales
    assert L.nvfp4_kv_requantize_write_fp8(0x10004, 0x20000, 0x40000, 3, 0x30000, None, ctypes.byref(d),
                                           None) == nv.NVKV_ERR_UNSUPPORTED   # alignment
    d8 = _desc(nv, prec=1)
    assert L.nvfp4_kv_requantize_write_fp8(0x10000, 0x20000, 0x40000, 3, 0x30000, None, ctypes.byref(d8),
                                           None) == nv.NVKV_ERR_INVALID_ARG   # the cache must be NVFP4
    assert L.nvfp4_kv_requantize_write_fp8(0x10000, 0x20000, 0x40000, 0, 0x30000, None, ctypes.byref(d),
                                           None) == nv.NVKV_OK
