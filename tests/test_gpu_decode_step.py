"""The one-launch decode step (nvfp4_paged_decode_step): the quantized write
of each sequence's newest token and the decode attention in one kernel.

Its result must be exactly that of the two separate calls (the write kernel,
then the decode kernel): the same cache bytes and the same output bits.  To
make the step's own write observable, the new tokens' slots are first
overwritten with other values (the written slot pairs' V bytes included), so
the expected bytes come back only if the step rewrites every byte of the
token and keeps the partner slot's nibbles.  One case is also checked against
the CPU oracle directly.
"""
import zlib

import numpy as np
import pytest
import torch

from _oracle_side import OracleLayer, within_tol

pytestmark = pytest.mark.gpu

LENS = (0, 1, 2, 17, 127, 128, 129, 300, 1001, 64)


def _layer(prec, P, seed, lens=LENS, Hq=32, Hkv=8):
    import nvfp4_quantized_paged_gb300 as nv
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Spec, Workload
    spec = Spec("decode_step", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, P=P, lens=tuple(lens), dist="element_outliers",
                outlier_scale=20.0, outlier_p=0.01, step_write=1)
    wl = Workload(spec, seed=seed, device="cuda")
    return nv, wl, Layer(wl, 0, prec=nv.PREC_FP8 if prec == "fp8" else nv.PREC_NVFP4)


@pytest.mark.parametrize("prec", ["nvfp4", "fp8"])
@pytest.mark.parametrize("P", [16, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_equals_write_then_decode(prec, P, dtype):
    nv, wl, lay = _layer(prec, P, zlib.crc32(f"{prec}{P}{dtype}".encode()) % 1000)
    assert lay.fused and lay.k_step is not None
    cast = (lambda t: t.to(torch.bfloat16).contiguous()) if dtype == "bf16" else (lambda t: t)
    pristine = lay.cache.data.clone()
    # the separate calls
    lay.write(cast(lay.k_new), cast(lay.v_new), lay.slots_new)
    lay.decode()
    torch.cuda.synchronize()
    want_bytes, want_out = lay.cache.data.clone(), lay.out.clone()
    # other bytes in the new tokens' slots, then the one-launch step
    lay.cache.data.copy_(pristine)
    lay.write(lay.k_new * -3.0 + 0.5, lay.v_new * 2.5 - 1.0, lay.slots_new)
    torch.cuda.synchronize()
    assert not torch.equal(lay.cache.data, want_bytes)
    out = torch.full_like(lay.out, float("nan"))
    nv.nvfp4_paged_decode_step(lay.q, cast(lay.k_step), cast(lay.v_step), lay.cache, lay.block_table, lay.seq_lens,
                               lay.prec, out, lay.workspace)
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    assert torch.equal(lay.cache.data, want_bytes)
    assert torch.equal(out, want_out)


@pytest.mark.parametrize("prec", ["nvfp4", "fp8"])
@pytest.mark.parametrize("Hq,Hkv,P", [(16, 2, 32), (4, 4, 64), (64, 8, 16)])
def test_decode_step_other_groups_and_pages(prec, Hq, Hkv, P):
    """The same equality for 8 query heads per KV head (the kernel's second
    instantiation), one head per KV head and page size 32."""
    nv, wl, lay = _layer(prec, P, zlib.crc32(f"{prec}{Hq}{Hkv}{P}".encode()) % 1000, lens=(5, 128, 700, 1, 257),
                         Hq=Hq, Hkv=Hkv)
    pristine = lay.cache.data.clone()
    lay.write(lay.k_new, lay.v_new, lay.slots_new)
    lay.decode()
    torch.cuda.synchronize()
    want_bytes, want_out = lay.cache.data.clone(), lay.out.clone()
    lay.cache.data.copy_(pristine)
    lay.write(lay.k_new * 1.5 - 2.0, lay.v_new * -0.75, lay.slots_new)
    out = torch.full_like(lay.out, float("nan"))
    nv.nvfp4_paged_decode_step(lay.q, lay.k_step, lay.v_step, lay.cache, lay.block_table, lay.seq_lens, lay.prec,
                               out, lay.workspace)
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    assert torch.equal(lay.cache.data, want_bytes)
    assert torch.equal(out, want_out)


@pytest.mark.parametrize("prec", ["nvfp4", "fp8"])
def test_decode_step_against_the_oracle(prec):
    nv, wl, lay = _layer(prec, 64, 321)
    lay.write(lay.k_new * 4.0, lay.v_new * -4.0, lay.slots_new)  # stale bytes the step must replace
    lay.step()
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    orc = OracleLayer(wl, 0, range(wl.spec.B), prec == "fp8")
    orc.compare_bytes(lay.cache.data)
    ok, worst = within_tol(lay.out.float().cpu().numpy(), orc.attention())
    assert ok, f"max excess over tolerance {worst}"


def test_decode_step_rejects_bad_arguments():
    nv, wl, lay = _layer("nvfp4", 64, 5, lens=(10, 20), Hq=8, Hkv=2)
    d = lay.cache.desc()
    L = nv.lib()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    args = lambda k, v, dt, prec: (p(lay.q), k, v, dt, ctypes.byref(d), p(lay.block_table), lay.block_table.shape[1],
                                   p(lay.seq_lens), 2, 8, prec, 0.0, 0, p(lay.workspace), lay.workspace.numel(),
                                   p(lay.out), None)
    assert L.nvfp4_paged_decode_step(*args(None, p(lay.v_step), 0, 0)) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvfp4_paged_decode_step(*args(p(lay.k_step), p(lay.v_step), 7, 0)) == nv.NVKV_ERR_INVALID_ARG
    assert L.nvfp4_paged_decode_step(*args(p(lay.k_step), p(lay.v_step), 0, 1)) == nv.NVKV_ERR_INVALID_ARG
    off = ctypes.c_void_p(lay.k_step.data_ptr() + 4)
    assert L.nvfp4_paged_decode_step(*args(off, p(lay.v_step), 0, 0)) == nv.NVKV_ERR_UNSUPPORTED
