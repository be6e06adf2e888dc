"""nvfp4_quantized_paged_gb300: NVFP4 paged KV cache for LLM decode on GB300.

Thin Python binding of the C ABI in ``include/nvfp4kv.h`` (library
``_build/libnvfp4kv.so``, CUDA for sm_103a).  Every function here only
marshals arguments: torch tensors give device pointers and the current CUDA
stream; the work runs in the library's kernels.  There is no CPU fallback:
if the library is missing, loading it raises.

Functions keep the C names:
  nvkv_global_scale, nvkv_amax_update, nvfp4_kv_quantize_write,
  fp8_kv_quantize_write, nvfp4_kv_requantize_write_fp8, nvkv_decode_workspace_size,
  nvkv_decode_workspace_init, nvfp4_paged_decode_attention,
  fp8_paged_decode_attention, nvfp4_kv_dequant_to_fp8_workspace,
  fp8_workspace_append_chunk, fp8_extend_scratch_size,
  fp8_chunked_extend_attention,
  nvkv_encode_e2m1, nvkv_encode_e4m3.
``Cache`` allocates one layer's paged planes with torch and builds the
``nvkv_cache`` descriptor.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libnvfp4kv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "nvfp4kv.h")

NVKV_OK = 0
NVKV_ERR_INVALID_ARG = 1
NVKV_ERR_UNSUPPORTED = 2
NVKV_ERR_CUDA = 3
NVKV_ERR_WORKSPACE_TOO_SMALL = 4
NVKV_NOALLOC_SCRATCH_BYTES = 8 << 20  # the header's fixed scratch array of the no-alloc decode

PREC_NVFP4 = 0
PREC_FP8 = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1

NVFP4_GLOBAL_DIVISOR = 2688.0  # 6 (largest E2M1) * 448 (largest E4M3)
FP8_GLOBAL_DIVISOR = 448.0
HEAD_DIM = 128


class NvkvError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: status {status} ({_status_string(status)})")


class nvkv_cache(ctypes.Structure):
    _fields_ = [
        ("prec", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("data", ctypes.c_void_p),
        ("kv_scale", ctypes.c_void_p),
        ("err_flag", ctypes.c_void_p),
    ]


_LIB = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t
_cachep = ctypes.POINTER(nvkv_cache)

SIGNATURES = {
    "nvkv_status_string": (ctypes.c_char_p, [_i32]),
    "nvkv_global_scale": (_i32, [_vp, _i32, _i64, _f32, _vp, _vp]),
    "nvkv_amax_update": (_i32, [_vp, _i32, _i64, _vp, _vp]),
    "nvfp4_kv_quantize_write": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _cachep, _vp]),
    "fp8_kv_quantize_write": (_i32, [_vp, _vp, _i32, _i64, _vp, _vp, _cachep, _vp]),
    "nvfp4_kv_requantize_write_fp8": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp, _cachep, _vp]),
    "nvkv_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "nvkv_decode_workspace_init": (_i32, [_vp, _sz, _vp]),
    "nvfp4_paged_decode_attention": (_i32, [_vp, _cachep, _vp, _i32, _vp, _i32, _i32, _i32, _f32, _i32, _vp, _sz,
                                            _vp, _vp]),
    "fp8_paged_decode_attention": (_i32, [_vp, _cachep, _vp, _i32, _vp, _i32, _i32, _f32, _i32, _vp, _sz, _vp,
                                          _vp]),
    "nvfp4_paged_decode_step": (_i32, [_vp, _vp, _vp, _i32, _cachep, _vp, _i32, _vp, _i32, _i32, _i32, _f32, _i32,
                                       _vp, _sz, _vp, _vp]),
    "nvfp4_paged_decode_attention_noalloc": (_i32, [_vp, _cachep, _vp, _i32, _vp, _i32, _i32, _i32, _f32, _i32,
                                                    _vp, _vp]),
    "nvfp4_kv_dequant_to_fp8_workspace": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _cachep, _vp, _vp, _vp, _i64,
                                                 _vp]),
    "fp8_workspace_append_chunk": (_i32, [_vp, _vp, _i32, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _i64, _vp, _vp]),
    "fp8_extend_scratch_size": (_sz, [_i64, _i32, _i32]),
    "fp8_chunked_extend_attention": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i64, _vp,
                                            _f32, _vp, _sz, _vp, _vp, _vp]),
    "nvkv_cache_page_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "nvkv_pool_pages_for_budget": (_i32, [_sz, _vp, _i32, _i32, _i32, _i32]),
    "nvkv_pool_create": (_vp, [_i32]),
    "nvkv_pool_destroy": (None, [_vp]),
    "nvkv_pool_num_free": (_i32, [_vp]),
    "nvkv_pool_alloc": (_i32, [_vp, _i32, _vp]),
    "nvkv_pool_release": (_i32, [_vp, _vp, _i32]),
    "nvkv_encode_e2m1": (_i32, [_vp, _i64, _vp, _vp]),
    "nvkv_encode_e4m3": (_i32, [_vp, _i64, _vp, _vp]),
}


def lib():
    """The loaded C library (raises if it was not built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def header_functions():
    """Names of the functions declared in include/nvfp4kv.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def _status_string(s):
    try:
        return lib().nvkv_status_string(s).decode()
    except Exception:  # pragma: no cover - message only
        return "?"


def _check(fn, status):
    if status != NVKV_OK:
        raise NvkvError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


class Cache:
    """One layer's paged cache in device memory: one contiguous block per
    (page, KV head), ``data`` uint8 [num_pages, Hkv, block], block = P * 144
    bytes (NVFP4) or P * 256 (FP8).  Inside a block the page's slots form
    groups of eight (the byte positions are stated in include/nvfp4kv.h).
    ``kv_scale`` float32[2] (K, V): the NVFP4 global scales or FP8 per-tensor
    scales.  ``err`` int32[1]: device error word (0 = none).
    """

    def __init__(self, prec: int, num_pages: int, num_kv_heads: int, page_size: int, device="cuda",
                 head_dim: int = HEAD_DIM, kv_scale: Optional[torch.Tensor] = None):
        self.prec, self.num_pages, self.Hkv, self.P, self.D = prec, num_pages, num_kv_heads, page_size, head_dim
        P, D = page_size, head_dim
        block = P * 2 * (D // 2 + D // 16) if prec == PREC_NVFP4 else 2 * P * D
        self.data = torch.zeros(num_pages, num_kv_heads, block, dtype=torch.uint8, device=device)
        self.kv_scale = kv_scale if kv_scale is not None else torch.zeros(2, dtype=torch.float32, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def desc(self) -> nvkv_cache:
        d = nvkv_cache()
        d.prec, d.num_pages, d.page_size, d.num_kv_heads, d.head_dim = (self.prec, self.num_pages, self.P, self.Hkv,
                                                                         self.D)
        d.data = self.data.data_ptr()
        d.kv_scale = self.kv_scale.data_ptr()
        d.err_flag = self.err.data_ptr()
        return d

    @property
    def nbytes(self) -> int:
        return self.data.numel()


# ---------------------------------------------------------------------------
# C entry points (same names)
# ---------------------------------------------------------------------------

def nvkv_global_scale(x: torch.Tensor, out: torch.Tensor, divisor: float = NVFP4_GLOBAL_DIVISOR, stream=None):
    """out[0] = max|x| / divisor (one FP32 per tensor)."""
    _check("nvkv_global_scale", lib().nvkv_global_scale(_ptr(x), _dtype_code(x), x.numel(), divisor, _ptr(out),
                                                        _stream(stream)))


def nvkv_amax_update(x: torch.Tensor, amax: torch.Tensor, stream=None):
    """amax[0] = max(amax[0], max|x|)."""
    _check("nvkv_amax_update", lib().nvkv_amax_update(_ptr(x), _dtype_code(x), x.numel(), _ptr(amax),
                                                      _stream(stream)))


def nvfp4_kv_quantize_write(k, v, slot_mapping, global_scale, cache: Cache, stream=None):
    d = cache.desc()
    _check("nvfp4_kv_quantize_write",
           lib().nvfp4_kv_quantize_write(_ptr(k), _ptr(v), _dtype_code(k), slot_mapping.numel(), _ptr(slot_mapping),
                                         _ptr(global_scale), ctypes.byref(d), _stream(stream)))


def fp8_kv_quantize_write(k, v, slot_mapping, global_scale, cache: Cache, stream=None):
    d = cache.desc()
    _check("fp8_kv_quantize_write",
           lib().fp8_kv_quantize_write(_ptr(k), _ptr(v), _dtype_code(k), slot_mapping.numel(), _ptr(slot_mapping),
                                       _ptr(global_scale), ctypes.byref(d), _stream(stream)))


def nvfp4_kv_requantize_write_fp8(k8, v8, in_scale, slot_mapping, global_scale, cache: Cache, stream=None):
    """Initial-prefill write: FP8 K/V bytes (uint8 [T, Hkv, D]) with their
    per-tensor scales ``in_scale`` (float32[2]) requantized into the NVFP4 cache."""
    d = cache.desc()
    _check("nvfp4_kv_requantize_write_fp8",
           lib().nvfp4_kv_requantize_write_fp8(_ptr(k8), _ptr(v8), _ptr(in_scale), slot_mapping.numel(),
                                               _ptr(slot_mapping), _ptr(global_scale), ctypes.byref(d),
                                               _stream(stream)))


def nvkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim=HEAD_DIM, num_splits=0) -> int:
    return int(lib().nvkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, num_splits))


def nvkv_decode_workspace_init(workspace: torch.Tensor, stream=None):
    _check("nvkv_decode_workspace_init",
           lib().nvkv_decode_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _stream(stream)))


def alloc_decode_workspace(batch, num_q_heads, num_kv_heads, num_splits=0, device="cuda") -> torch.Tensor:
    """Allocate (torch) and zero a decode workspace of the required size."""
    n = nvkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, HEAD_DIM, num_splits)
    if n == 0:
        raise NvkvError("nvkv_decode_workspace_size", NVKV_ERR_INVALID_ARG)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    nvkv_decode_workspace_init(ws)
    return ws


def nvfp4_paged_decode_attention(q, cache: Cache, block_table, seq_lens, layer_precision, out, workspace,
                                 sm_scale=0.0, num_splits=0, stream=None):
    d = cache.desc()
    _check("nvfp4_paged_decode_attention",
           lib().nvfp4_paged_decode_attention(_ptr(q), ctypes.byref(d), _ptr(block_table), block_table.shape[1],
                                              _ptr(seq_lens), q.shape[0], q.shape[1], layer_precision, sm_scale,
                                              num_splits, _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _ptr(out),
                                              _stream(stream)))


def fp8_paged_decode_attention(q, cache: Cache, block_table, seq_lens, out, workspace, sm_scale=0.0,
                               num_splits=0, stream=None):
    d = cache.desc()
    _check("fp8_paged_decode_attention",
           lib().fp8_paged_decode_attention(_ptr(q), ctypes.byref(d), _ptr(block_table), block_table.shape[1],
                                            _ptr(seq_lens), q.shape[0], q.shape[1], sm_scale, num_splits,
                                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                                            _ptr(out), _stream(stream)))


def nvfp4_paged_decode_step(q, k_new, v_new, cache: Cache, block_table, seq_lens, layer_precision, out, workspace,
                            sm_scale=0.0, num_splits=0, stream=None):
    """One decode step in one launch: each sequence's newest token (row b of
    k_new / v_new, [B, Hkv, 128] FP32 or BF16) quantized into the cache at
    position seq_lens[b] - 1, then decode attention over the cache."""
    d = cache.desc()
    _check("nvfp4_paged_decode_step",
           lib().nvfp4_paged_decode_step(_ptr(q), _ptr(k_new), _ptr(v_new), _dtype_code(k_new), ctypes.byref(d),
                                         _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0],
                                         q.shape[1], layer_precision, sm_scale, num_splits, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _ptr(out), _stream(stream)))


def nvfp4_paged_decode_attention_noalloc(q, cache: Cache, block_table, seq_lens, layer_precision, out,
                                         sm_scale=0.0, num_splits=0, stream=None):
    """Decode attention with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory)."""
    d = cache.desc()
    _check("nvfp4_paged_decode_attention_noalloc",
           lib().nvfp4_paged_decode_attention_noalloc(_ptr(q), ctypes.byref(d), _ptr(block_table),
                                                      block_table.shape[1], _ptr(seq_lens), q.shape[0], q.shape[1],
                                                      layer_precision, sm_scale, num_splits, _ptr(out),
                                                      _stream(stream)))


def nvfp4_kv_dequant_to_fp8_workspace(block_table, seq_ids, prefix_lens, cu_prefix, cache: Cache, ws_scale, ws_k,
                                      ws_v, stream=None):
    d = cache.desc()
    _check("nvfp4_kv_dequant_to_fp8_workspace",
           lib().nvfp4_kv_dequant_to_fp8_workspace(_ptr(block_table), block_table.shape[1], _ptr(seq_ids),
                                                   _ptr(prefix_lens), _ptr(cu_prefix), seq_ids.numel(),
                                                   ctypes.byref(d), _ptr(ws_scale), _ptr(ws_k), _ptr(ws_v),
                                                   ws_k.shape[0], _stream(stream)))


def fp8_workspace_append_chunk(k, v, rows, ws_scale, ws_k, ws_v, err=None, stream=None):
    """The chunk's K/V ([T, Hkv, D] FP32 or BF16) into workspace rows ``rows``
    (int64 [T]) as E4M3(x / ws_scale)."""
    _check("fp8_workspace_append_chunk",
           lib().fp8_workspace_append_chunk(_ptr(k), _ptr(v), _dtype_code(k), k.shape[0], _ptr(rows), k.shape[1],
                                            k.shape[2], _ptr(ws_scale), _ptr(ws_k), _ptr(ws_v), ws_k.shape[0],
                                            _ptr(err), _stream(stream)))


def fp8_extend_scratch_size(ws_rows, num_kv_heads, head_dim=HEAD_DIM) -> int:
    return int(lib().fp8_extend_scratch_size(ws_rows, num_kv_heads, head_dim))


def alloc_extend_scratch(ws_k: torch.Tensor) -> torch.Tensor:
    """Scratch (torch) for fp8_chunked_extend_attention over workspace ws_k."""
    n = fp8_extend_scratch_size(ws_k.shape[0], ws_k.shape[1], ws_k.shape[2])
    if n == 0:
        raise NvkvError("fp8_extend_scratch_size", NVKV_ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=ws_k.device)


def fp8_chunked_extend_attention(q, cu_q, max_q_len, ws_k, ws_v, cu_kv, kv_lens, ws_scale, out, scratch,
                                 sm_scale=0.0, err=None, stream=None):
    """Causal FP8 attention of the chunk queries ``q`` (BF16 [Tq, Hq, 128],
    sequence i owns rows cu_q[i]:cu_q[i+1]) over workspace rows
    [cu_kv[i], cu_kv[i] + kv_lens[i]) (prefix, then the chunk; cu_kv[i] a
    multiple of 8).  ``scratch``: see alloc_extend_scratch."""
    _check("fp8_chunked_extend_attention",
           lib().fp8_chunked_extend_attention(_ptr(q), _ptr(cu_q), kv_lens.numel(), int(max_q_len), q.shape[1],
                                              _ptr(ws_k), _ptr(ws_v), _ptr(cu_kv), _ptr(kv_lens), ws_k.shape[1],
                                              q.shape[2], ws_k.shape[0], _ptr(ws_scale), sm_scale, _ptr(scratch),
                                              scratch.numel(), _ptr(out), _ptr(err), _stream(stream)))


def nvkv_encode_e2m1(x, out, stream=None):
    _check("nvkv_encode_e2m1", lib().nvkv_encode_e2m1(_ptr(x), x.numel(), _ptr(out), _stream(stream)))


def nvkv_encode_e4m3(x, out, stream=None):
    _check("nvkv_encode_e4m3", lib().nvkv_encode_e4m3(_ptr(x), x.numel(), _ptr(out), _stream(stream)))


# ---------------------------------------------------------------------------
# Page ledger and page pool (host side of the C ABI)
# ---------------------------------------------------------------------------

def nvkv_cache_page_bytes(prec, page_size, num_kv_heads, head_dim=HEAD_DIM) -> int:
    return int(lib().nvkv_cache_page_bytes(prec, page_size, num_kv_heads, head_dim))


def nvkv_pool_pages_for_budget(budget_bytes, layer_prec, page_size, num_kv_heads, head_dim=HEAD_DIM) -> int:
    arr = (ctypes.c_int32 * len(layer_prec))(*layer_prec)
    n = lib().nvkv_pool_pages_for_budget(int(budget_bytes), ctypes.cast(arr, ctypes.c_void_p), len(layer_prec),
                                         page_size, num_kv_heads, head_dim)
    if n < 0:
        raise NvkvError("nvkv_pool_pages_for_budget", NVKV_ERR_INVALID_ARG)
    return int(n)


class PagePool:
    """The library's page pool (nvkv_pool_*): page ids shared by every layer's cache."""

    def __init__(self, num_pages: int):
        self._p = lib().nvkv_pool_create(num_pages)
        if not self._p:
            raise NvkvError("nvkv_pool_create", NVKV_ERR_INVALID_ARG)
        self.num_pages = num_pages

    def close(self):
        if self._p:
            lib().nvkv_pool_destroy(self._p)
            self._p = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass

    @property
    def num_free(self) -> int:
        return int(lib().nvkv_pool_num_free(self._p))

    def alloc(self, n: int):
        """n page ids (list) or None when fewer than n are free (nothing taken)."""
        out = (ctypes.c_int32 * max(n, 1))()
        r = lib().nvkv_pool_alloc(self._p, n, ctypes.cast(out, ctypes.c_void_p))
        return None if r < 0 else list(out[:n])

    def release(self, pages):
        arr = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        _check("nvkv_pool_release", lib().nvkv_pool_release(self._p, ctypes.cast(arr, ctypes.c_void_p), len(pages)))
