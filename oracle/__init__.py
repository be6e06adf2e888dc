"""CPU oracle for the NVFP4 / FP8 paged KV cache (numpy front end).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
CUDA library never loads it and shares no code with it; the two meet only
through the seeded input generators, which hold none of the method's
arithmetic.

The arithmetic lives in ``nvfp4kv_oracle.c`` (scalar C, one thread, FP32
quantizer steps without FMA contraction, FP64 attention); this module only
marshals numpy arrays.  Every function cites the page passage it follows:

  [P1] "SOAR Weekly Champion Notes 05 | Zhisuan Team One: NVFP4 KV Cache and
       Mixed-Precision Practice", sections 02 and 03.
  [P2] "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache Breaks
       Long-Context and Agentic Inference Bottlenecks", sections "The Core of
       the Ledger: 4-bit Does Not Equal 2x" and "Three Paths".

Parity pins live in ``tests/test_oracle_*.py``.  Functions whose result the
pages' throughput figures would pin (end-to-end serving speed-ups) are not
implemented: parity unpinned, out of scope.
"""
import ctypes
import numpy as np

from . import build as _build

_LIB = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)

PREC_NVFP4 = 0
PREC_FP8 = 1

NVFP4_GLOBAL_DIVISOR = 6.0 * 448.0  # largest E2M1 magnitude x largest E4M3 value
FP8_GLOBAL_DIVISOR = 448.0


def lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build.build())
        L.orc_e2m1_value.restype = ctypes.c_double
        L.orc_e2m1_value.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_value.restype = ctypes.c_double
        L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        L.orc_e2m1_encode.restype = ctypes.c_uint8
        L.orc_e2m1_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        for n in ("orc_e2m1_encode_bits", "orc_e4m3_encode_bits"):
            f = getattr(L, n)
            f.restype = None
            f.argtypes = [ctypes.c_uint32, ctypes.c_uint32, _u8p]
        L.orc_global_scale.restype = ctypes.c_float
        L.orc_global_scale.argtypes = [_f32p, ctypes.c_int64, ctypes.c_float]
        L.orc_nvfp4_quantize_write.restype = ctypes.c_int
        L.orc_nvfp4_quantize_write.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i64p,
                                               _f32p, ctypes.c_int, ctypes.c_int64, _u8p]
        L.orc_fp8_quantize_write.restype = ctypes.c_int
        L.orc_fp8_quantize_write.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i64p,
                                             _f32p, ctypes.c_int, ctypes.c_int64, _u8p]
        L.orc_slot_bytes.restype = ctypes.c_int
        L.orc_slot_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64p]
        L.orc_v_code_layout.restype = ctypes.c_int
        L.orc_v_code_layout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64p, _i32p]
        L.orc_gather_dequant.restype = ctypes.c_int
        L.orc_gather_dequant.argtypes = [ctypes.c_int, _u8p, ctypes.c_int, ctypes.c_float, _i32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                         _f64p]
        L.orc_paged_decode_attention.restype = ctypes.c_int
        L.orc_paged_decode_attention.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.c_int, ctypes.c_int, _u8p, _f32p, _i32p,
                                                 ctypes.c_int, _i32p, ctypes.c_int64, ctypes.c_double,
                                                 ctypes.c_int, _f64p]
        L.orc_dequant_to_fp8_workspace.restype = ctypes.c_int
        L.orc_dequant_to_fp8_workspace.argtypes = [_i32p, ctypes.c_int, _i32p, _i32p, _i64p, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                   _u8p, _f32p, _f32p, _u8p, _u8p]
        L.orc_fp8_workspace_append.restype = ctypes.c_int
        L.orc_fp8_workspace_append.argtypes = [_f32p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i64p,
                                               _f32p, ctypes.c_int64, _u8p, _u8p]
        L.orc_fp8_extend_attention.restype = ctypes.c_int
        L.orc_fp8_extend_attention.argtypes = [_u16p, _i64p, _u8p, _u8p, _i64p, _i32p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_double, _f64p]
        L.orc_nvfp4_requantize_write_fp8.restype = ctypes.c_int
        L.orc_nvfp4_requantize_write_fp8.argtypes = [_u8p, _u8p, _f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                     _i64p, _f32p, ctypes.c_int, ctypes.c_int64, _u8p]
        _LIB = L
    return _LIB


def _p(a, t):
    return a.ctypes.data_as(t)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# --------------------------------------------------------------------------
# Element formats ([P1] 02; [P2] Core of the Ledger)
# --------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (1 sign, 2 exponent, 1 mantissa bit)."""
    return lib().orc_e2m1_value(code)


def e4m3_value(b: int) -> float:
    """Value of an E4M3 byte (OCP 'fn' variant); NaN for 0x7F / 0xFF."""
    return lib().orc_e4m3_value(b)


def e2m1_encode(y: float) -> int:
    """Round-to-nearest-even E2M1 code of an FP32 value, saturating at 6."""
    return lib().orc_e2m1_encode(y)


def e4m3_encode(y: float) -> int:
    """Round-to-nearest-even E4M3 byte of an FP32 value, saturating at 448."""
    return lib().orc_e4m3_encode(y)


def e2m1_encode_bits(start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint8)
    lib().orc_e2m1_encode_bits(start, count, _p(out, _u8p))
    return out


def e4m3_encode_bits(start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint8)
    lib().orc_e4m3_encode_bits(start, count, _p(out, _u8p))
    return out


def e2m1_encode_array(y: np.ndarray) -> np.ndarray:
    y = _c(y, np.float32).ravel()
    return np.array([lib().orc_e2m1_encode(float(v)) for v in y], np.uint8)


def e4m3_encode_array(y: np.ndarray) -> np.ndarray:
    y = _c(y, np.float32).ravel()
    bits = y.view(np.uint32)
    out = np.empty(y.size, np.uint8)
    L = lib()
    for i, u in enumerate(bits):
        L.orc_e4m3_encode_bits(int(u), 1, _p(out[i:i + 1], _u8p))
    return out


# --------------------------------------------------------------------------
# Global scale ([P2] Core of the Ledger: one FP32 global scale per tensor)
# --------------------------------------------------------------------------

def global_scale(x: np.ndarray, divisor: float = NVFP4_GLOBAL_DIVISOR) -> np.float32:
    x = _c(x, np.float32)
    return np.float32(lib().orc_global_scale(_p(x, _f32p), x.size, divisor))


# --------------------------------------------------------------------------
# Paged cache ([P1] 02, the FP4 memory pool; [P2] Three Paths, paged KV cache)
# --------------------------------------------------------------------------

class Cache:
    """One layer's paged cache: one contiguous block per (page, KV head).

    ``data`` uint8 [num_pages, Hkv, block] holds the bytes in the cache layout
    stated in nvfp4kv_oracle.c (groups of 8 slots; K bytes chunk-major; V rows
    reordered); the block is P*144 bytes at D = 128 for NVFP4 and P*256 for
    FP8.  ``k_data``/``k_scale``/``v_data``/``v_scale`` return copies of the
    logical planes, shaped [num_pages, Hkv, P, D/2] and [num_pages, Hkv, P,
    D/16] (FP8: [num_pages, Hkv, P, D], no scales); ``positions(name)`` gives
    the [P, n] byte positions of a plane inside a block, for writes.
    ``g`` = float32[2] (K, V) global (NVFP4) or per-tensor (FP8) scale.
    """

    def __init__(self, prec, num_pages, Hkv, P, D, g, fill=0):
        self.prec, self.num_pages, self.Hkv, self.P, self.D = prec, num_pages, Hkv, P, D
        self.g = np.asarray(g, np.float32).reshape(2).copy()
        block = P * 2 * (D // 2 + D // 16) if prec == PREC_NVFP4 else 2 * P * D
        self.data = np.full((num_pages, Hkv, block), fill, np.uint8)
        self._slot_pos = None

    def slot_positions(self) -> np.ndarray:
        """int64 [P, n]: positions of the bytes each slot occupies in a block (K
        codes, K scales, V codes, V scales; FP8: K, V).  NVFP4 V codes of paired
        rows share bytes with the partner row: the slot's entries are the D
        bytes holding its D nibbles."""
        if self._slot_pos is None:
            rows = []
            for off in range(self.P):
                row = np.empty(2 * self.D + self.D // 8, np.int64)
                n = lib().orc_slot_bytes(self.prec, self.P, self.D, off, _p(row, _i64p))
                assert n > 0
                rows.append(row[:n])
            self._slot_pos = np.stack(rows)
        return self._slot_pos

    def positions(self, name: str) -> np.ndarray:
        """[P, n] byte positions of a byte plane (k_data, k_scale, v_scale; FP8:
        k_data, v_data).  NVFP4 v_data is not a byte plane (see v_data)."""
        D, pos = self.D, self.slot_positions()
        if self.prec == PREC_NVFP4:
            c, s = D // 2, D // 16
            cuts = {"k_data": (0, c), "k_scale": (c, c + s), "v_scale": (pos.shape[1] - s, pos.shape[1])}
        else:
            cuts = {"k_data": (0, D), "v_data": (D, 2 * D)}
        a, b = cuts[name]
        return pos[:, a:b]

    def _v_codes(self):
        """NVFP4 V as the logical [pages, Hkv, P, D/2] code bytes (value 2j in
        the low nibble, 2j+1 in the high), gathered nibble by nibble."""
        P, D = self.P, self.D
        pos = np.empty((P, D), np.int64)
        sh = np.empty((P, D), np.int32)
        for off in range(P):
            assert lib().orc_v_code_layout(P, D, off, _p(pos[off], _i64p), _p(sh[off], _i32p)) == 0
        nib = (self.data[:, :, pos] >> sh.astype(np.uint8)) & 15
        return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)

    def _plane(self, name):
        if self.prec != PREC_NVFP4 and name.endswith("scale"):
            return None
        if self.prec == PREC_NVFP4 and name == "v_data":
            return self._v_codes()
        return self.data[:, :, self.positions(name)]

    k_data = property(lambda self: self._plane("k_data"))
    k_scale = property(lambda self: self._plane("k_scale"))
    v_data = property(lambda self: self._plane("v_data"))
    v_scale = property(lambda self: self._plane("v_scale"))

    @property
    def nbytes(self):
        return self.data.nbytes


def quantize_write(cache: Cache, k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray) -> None:
    """Quantized write of new K/V [T, Hkv, D] into the cache slots.

    NVFP4 follows [P2] Core of the Ledger (two-level scaling) and [P1] 02
    (two codes per byte); FP8 follows [P1] 01/03 (FP8 KV cache layers).
    """
    k = _c(k, np.float32)
    v = _c(v, np.float32)
    assert np.isfinite(k).all() and np.isfinite(v).all()
    sm = _c(slot_mapping, np.int64)
    T = sm.shape[0]
    assert k.shape == (T, cache.Hkv, cache.D) and v.shape == k.shape
    L = lib()
    if cache.prec == PREC_NVFP4:
        rc = L.orc_nvfp4_quantize_write(_p(k, _f32p), _p(v, _f32p), T, cache.Hkv, cache.D, _p(sm, _i64p),
                                        _p(cache.g, _f32p), cache.P, cache.num_pages, _p(cache.data, _u8p))
    else:
        rc = L.orc_fp8_quantize_write(_p(k, _f32p), _p(v, _f32p), T, cache.Hkv, cache.D, _p(sm, _i64p),
                                      _p(cache.g, _f32p), cache.P, cache.num_pages, _p(cache.data, _u8p))
    if rc != 0:
        raise ValueError("slot out of range")


def requantize_write_fp8(cache: Cache, k8: np.ndarray, v8: np.ndarray, s8, slot_mapping: np.ndarray) -> None:
    """Initial-prefill write from FP8 K/V ([P2] Three Paths: the prefill's FP8
    KV is requantized into the NVFP4 cache): x = E4M3(byte) * s8 (one FP32
    multiply), then the NVFP4 quantized write with the cache's global scales."""
    assert cache.prec == PREC_NVFP4
    kk = _c(k8, np.uint8)
    vv = _c(v8, np.uint8)
    T, Hkv, D = kk.shape
    sc = _c(s8, np.float32).reshape(2)
    sm = _c(slot_mapping, np.int64)
    rc = lib().orc_nvfp4_requantize_write_fp8(_p(kk, _u8p), _p(vv, _u8p), _p(sc, _f32p), T, Hkv, D, _p(sm, _i64p),
                                              _p(cache.g, _f32p), cache.P, cache.num_pages, _p(cache.data, _u8p))
    if rc != 0:
        raise ValueError("slot out of range")


def gather_dequant(cache: Cache, which: str, block_row: np.ndarray, L: int, h: int) -> np.ndarray:
    """Exact FP64 values of tokens [0, L) of one (sequence, KV head)."""
    br = _c(block_row, np.int32)
    out = np.empty((L, cache.D), np.float64)
    kind = 0 if which == "k" else 1
    rc = lib().orc_gather_dequant(cache.prec, _p(cache.data, _u8p), kind, float(cache.g[kind]), _p(br, _i32p), L,
                                  cache.Hkv, h, cache.D, cache.P, cache.num_pages, _p(out, _f64p))
    if rc != 0:
        raise ValueError("page out of range")
    return out


def paged_decode_attention(cache: Cache, q_bf16_bits: np.ndarray, block_table: np.ndarray,
                           seq_lens: np.ndarray, sm_scale: float = 0.0, num_splits: int = 0) -> np.ndarray:
    """Paged GQA decode attention in FP64 ([P2] Three Paths, decode).

    ``q_bf16_bits``: uint16 [B, Hq, D] BF16 bit patterns.  Returns FP64
    [B, Hq, D].  ``num_splits > 1`` evaluates the split / log-sum-exp merge
    form, which must equal the plain softmax.
    """
    q = _c(q_bf16_bits, np.uint16)
    B, Hq, D = q.shape
    bt = _c(block_table, np.int32)
    sl = _c(seq_lens, np.int32)
    if sm_scale == 0.0:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.empty((B, Hq, D), np.float64)
    rc = lib().orc_paged_decode_attention(_p(q, _u16p), B, Hq, cache.Hkv, D, cache.P, cache.prec,
                                          _p(cache.data, _u8p), _p(cache.g, _f32p), _p(bt, _i32p), bt.shape[1],
                                          _p(sl, _i32p), cache.num_pages, float(sm_scale), int(num_splits),
                                          _p(out, _f64p))
    if rc != 0:
        raise ValueError("bad block table / sequence length")
    return out


def dequant_to_fp8_workspace(cache: Cache, block_table: np.ndarray, seq_ids, prefix_lens,
                             ws_scale, row_start=None, ws_rows=None) -> tuple:
    """Chunked-extend prefix dequant into the FP8 workspace ([P2] Three Paths).

    Token t of sequence i goes to row ``row_start[i] + t`` (default: the
    sequences back to back, row_start = exclusive sums of prefix_lens).
    Returns (ws_k, ws_v), uint8 [ws_rows, Hkv, D] E4M3 (default ws_rows: the
    last prefix's end); rows no prefix token lands on stay 0.
    """
    assert cache.prec == PREC_NVFP4
    bt = _c(block_table, np.int32)
    ids = _c(seq_ids, np.int32)
    pl = _c(prefix_lens, np.int32)
    cu = np.zeros(len(pl) + 1, np.int64)
    if row_start is None:
        cu[1:] = np.cumsum(pl)
    else:
        cu[:-1] = np.asarray(row_start, np.int64)
        cu[-1] = cu[-2] + pl[-1] if len(pl) else 0
    ws = _c(ws_scale, np.float32).reshape(2)
    rows = max([int(cu[i]) + int(pl[i]) for i in range(len(pl))] + [0])
    if ws_rows is not None:
        assert ws_rows >= rows
        rows = int(ws_rows)
    wk = np.zeros((rows, cache.Hkv, cache.D), np.uint8)
    wv = np.zeros((rows, cache.Hkv, cache.D), np.uint8)
    rc = lib().orc_dequant_to_fp8_workspace(_p(bt, _i32p), bt.shape[1], _p(ids, _i32p), _p(pl, _i32p),
                                            _p(cu, _i64p), len(pl), cache.Hkv, cache.D, cache.P, cache.num_pages,
                                            _p(cache.data, _u8p), _p(cache.g, _f32p),
                                            _p(ws, _f32p), _p(wk, _u8p), _p(wv, _u8p))
    if rc != 0:
        raise ValueError("bad arguments")
    return wk, wv


def fp8_workspace_append(ws_k: np.ndarray, ws_v: np.ndarray, k: np.ndarray, v: np.ndarray, rows: np.ndarray,
                         ws_scale) -> None:
    """The current chunk's K/V into FP8 workspace rows ([P2] Three Paths: the
    chunk's KV is appended to the dequantized prefix for FP8 attention).

    ``k``, ``v``: [T, Hkv, D] (FP32 or BF16-exact values); token t goes to row
    ``rows[t]`` (negative: skipped) as E4M3_RNE_sat(x / ws_scale) per tensor.
    ``ws_k`` / ``ws_v`` (uint8 [rows, Hkv, D]) are updated in place.
    """
    T, Hkv, D = k.shape
    kk = _c(k, np.float32)
    vv = _c(v, np.float32)
    r = _c(rows, np.int64)
    ws = _c(ws_scale, np.float32).reshape(2)
    assert ws_k.flags.c_contiguous and ws_v.flags.c_contiguous and ws_k.dtype == np.uint8
    rc = lib().orc_fp8_workspace_append(_p(kk, _f32p), _p(vv, _f32p), T, Hkv, D, _p(r, _i64p), _p(ws, _f32p),
                                        ws_k.shape[0], _p(ws_k, _u8p), _p(ws_v, _u8p))
    if rc != 0:
        raise ValueError("bad row or scale")


def fp8_extend_attention(q_bf16_bits: np.ndarray, cu_q, ws_k: np.ndarray, ws_v: np.ndarray, cu_kv, kv_lens,
                         ws_scale, sm_scale: float = 0.0) -> np.ndarray:
    """Chunked-extend attention over the FP8 workspace in FP64 ([P2] Three
    Paths, chunked prefill / extend).

    Sequence i's keys and values are workspace rows [cu_kv[i], cu_kv[i] +
    kv_lens[i]) (prefix, then the chunk); its queries ``q_bf16_bits[cu_q[i]:
    cu_q[i+1]]`` (uint16 BF16 bits, [Tq, Hq, D]) are the last positions of the
    sequence and see every position up to their own.  Returns FP64 [Tq, Hq, D].
    """
    q = _c(q_bf16_bits, np.uint16)
    Tq, Hq, D = q.shape
    Hkv = ws_k.shape[1]
    cq = _c(cu_q, np.int64)
    ck = _c(cu_kv, np.int64)
    kl = _c(kv_lens, np.int32)
    ws = _c(ws_scale, np.float32).reshape(2)
    wk = _c(ws_k, np.uint8)
    wv = _c(ws_v, np.uint8)
    if sm_scale == 0.0:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.zeros((Tq, Hq, D), np.float64)
    rc = lib().orc_fp8_extend_attention(_p(q, _u16p), _p(cq, _i64p), _p(wk, _u8p), _p(wv, _u8p), _p(ck, _i64p),
                                        _p(kl, _i32p), len(kl), Hq, Hkv, D, _p(ws, _f32p), float(sm_scale),
                                        _p(out, _f64p))
    if rc != 0:
        raise ValueError("bad arguments")
    return out
