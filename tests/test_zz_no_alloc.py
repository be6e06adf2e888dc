"""The allocation-free decode entry point.

Some callers cannot give this library device memory for scratch: serving
engines that hand all free HBM to their KV page pool at start-up and keep no
allocator for per-call buffers, and plugin hosts that pass a kernel only its
inputs and outputs.  For them nvfp4_paged_decode_attention_noalloc uses a
fixed scratch array inside the library.  These tests call it through the C
ABI on problems in a row and check each output bit for bit against the
regular entry point (caller workspace), check that a call leaves the device's
free memory unchanged, and check that a split request far larger than the
device holds at once is capped to one resident wave, whose partials fit the
array.  The file is collected last so that a stop-at-first-failure run has
already run every other test.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _layer(name, lens, P, Hq, Hkv, prec, seed):
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Spec, Workload
    spec = Spec(name, B=len(lens), Hq=Hq, Hkv=Hkv, D=128, P=P, lens=tuple(lens), dist="element_outliers",
                outlier_scale=20.0, outlier_p=0.01, step_write=0)
    return Layer(Workload(spec, seed=seed, device="cuda"), 0, prec=prec)


def _noalloc(nv, lay, out):
    d = lay.cache.desc()
    return nv.lib().nvfp4_paged_decode_attention_noalloc(
        ctypes.c_void_p(lay.q.data_ptr()), ctypes.byref(d), ctypes.c_void_p(lay.block_table.data_ptr()),
        lay.block_table.shape[1], ctypes.c_void_p(lay.seq_lens.data_ptr()), lay.q.shape[0], lay.q.shape[1],
        lay.prec, 0.0, 0, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_on_calls_in_a_row():
    # b, then the larger a, then b again: whatever a call leaves in the shared
    # scratch (counters, partial slots) must not leak into the next.  Both
    # paths run the same kernels on the same schedule, so the bits agree.
    import nvfp4_quantized_paged_gb300 as nv
    a = _layer("noalloc_a", [3000, 1, 700, 64], 64, 32, 8, nv.PREC_NVFP4, 11)
    b = _layer("noalloc_b", [129, 5000], 16, 16, 2, nv.PREC_FP8, 12)
    for lay in (b, a, b):
        lay.decode()  # regular entry point, caller-owned workspace
        want = lay.out.float().clone()
        out = torch.full_like(lay.out, float("nan"))
        assert _noalloc(nv, lay, out) == nv.NVKV_OK
        torch.cuda.synchronize()
        assert lay.cache.err.item() == 0
        assert torch.equal(out.float(), want)


def test_noalloc_allocates_no_device_memory():
    # after one warm-up call (module and scratch lookup done), a call leaves the
    # device's free memory unchanged
    import nvfp4_quantized_paged_gb300 as nv
    lay = _layer("noalloc_m", [4096, 2048, 17], 64, 32, 8, nv.PREC_NVFP4, 14)
    out = torch.empty_like(lay.out)
    assert _noalloc(nv, lay, out) == nv.NVKV_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _noalloc(nv, lay, out) == nv.NVKV_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert lay.cache.err.item() == 0


def test_noalloc_caps_a_large_split_request_and_matches_the_workspace_entry():
    import nvfp4_quantized_paged_gb300 as nv
    lay = _layer("noalloc_c", [8192, 8192], 64, 32, 8, nv.PREC_NVFP4, 13)
    lay.num_splits = 100
    lay.workspace = nv.alloc_decode_workspace(2, 32, 8, 100)
    lay.decode()
    want = lay.out.float().clone()
    d = lay.cache.desc()
    out = torch.full_like(lay.out, float("nan"))
    # 2 sequences x 8 KV heads x 100 splits asks for 1600 shares; the library runs
    # one resident wave, whose partials fit the fixed scratch
    st = nv.lib().nvfp4_paged_decode_attention_noalloc(
        ctypes.c_void_p(lay.q.data_ptr()), ctypes.byref(d), ctypes.c_void_p(lay.block_table.data_ptr()),
        lay.block_table.shape[1], ctypes.c_void_p(lay.seq_lens.data_ptr()), 2, 32, nv.PREC_NVFP4, 0.0, 100,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == nv.NVKV_OK
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    got = out.float()
    assert torch.equal(got, want)  # same schedule, same kernels: same bits
