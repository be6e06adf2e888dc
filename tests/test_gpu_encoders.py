"""Exhaustive GPU-vs-oracle sweep of the element encoders: every FP32 bit
pattern (NaNs excluded: undefined) through the device E2M1 and E4M3
conversions must give the oracle's code bit for bit."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28
SUB = 1 << 24


def _oracle_chunk(fn, start):
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        parts = list(ex.map(lambda s: fn(s, SUB), range(start, start + CHUNK, SUB)))
    return np.concatenate(parts)


@pytest.mark.parametrize("which", ["e2m1", "e4m3"])
def test_encoder_exhaustive(which):
    import oracle
    import nvfp4_quantized_paged_gb300 as nv
    enc = nv.nvkv_encode_e2m1 if which == "e2m1" else nv.nvkv_encode_e4m3
    ofn = oracle.e2m1_encode_bits if which == "e2m1" else oracle.e4m3_encode_bits
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    bad = 0
    for start in range(0, 1 << 32, CHUNK):
        u = torch.arange(start, start + CHUNK, dtype=torch.int64, device="cuda")
        u = torch.where(u >= (1 << 31), u - (1 << 32), u).to(torch.int32)
        enc(u.view(torch.float32), out)
        got = out.cpu().numpy()
        want = _oracle_chunk(ofn, start)
        bits = np.arange(start, start + CHUNK, dtype=np.uint64)
        nan = ((bits & 0x7F800000) == 0x7F800000) & ((bits & 0x7FFFFF) != 0)
        diff = (got != want) & ~nan
        if diff.any():
            i = int(np.argmax(diff))
            bad += int(diff.sum())
            pytest.fail(f"{which}: {int(diff.sum())} mismatches in chunk {start:#x}; first bits "
                        f"{int(bits[i]):#010x}: gpu {got[i]:#04x} oracle {want[i]:#04x}")
    assert bad == 0
