"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Bytes (codes, E4M3 scales, FP8 bytes, workspace, global scales) must match
bit for bit; attention outputs (BF16) must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| element by element, the oracle being
FP64 attention over the identical quantized bytes.  Cases are small enough for
the oracle to finish in seconds yet span several 128-token tiles, ragged tails,
empty sequences, page sizes 16, 32 and 64, GQA groups 1..8 and forced splits.
"""
import zlib

import numpy as np
import pytest
import torch

from _oracle_side import OracleLayer, within_tol

pytestmark = pytest.mark.gpu


def _nv():
    import nvfp4_quantized_paged_gb300 as nv
    nv.lib()
    return nv


def _spec(**kw):
    from nvfp4_quantized_paged_gb300.workloads import Spec
    base = dict(name="case", B=1, Hq=32, Hkv=8, D=128, P=64, dist="element_outliers", outlier_scale=20.0,
                outlier_p=0.01, table="permuted", step_write=1)
    base.update(kw)
    return Spec(**base)


CASES = {
    "b1_ctx1k_p16_g4": dict(B=1, Hq=8, Hkv=2, P=16, L=1024, dist="channel_outliers", outlier_channels=4,
                            table="contiguous", step_write=1024),
    "ragged_p64": dict(B=6, lens=(1, 63, 64, 65, 200, 1000)),
    "ragged_p16": dict(B=5, P=16, lens=(5, 16, 17, 100, 300)),
    "ragged_p32": dict(B=3, P=32, lens=(31, 33, 700)),
    "empty_seqs": dict(B=4, lens=(0, 100, 0, 64)),
    "gqa8": dict(B=3, Hq=16, Hkv=2, lens=(70, 300, 129)),
    "gqa1": dict(B=2, Hq=4, Hkv=4, lens=(90, 257)),
    "gqa2": dict(B=2, Hq=8, Hkv=4, lens=(200, 33)),
    "splits7": dict(B=2, lens=(5000, 1300), num_splits=7),
    "splits64": dict(B=2, lens=(5000, 4096), num_splits=64),
    # CTA shares that run through many one-tile (sequence, head) segments in a row
    "short_segments": dict(B=9, lens=(2000, 64, 1, 100, 64, 128, 5, 64, 700), num_splits=1),
    "lognormal_channels": dict(B=3, lens=(600, 333, 64), dist="lognormal_channels", channel_sigma=0.5),
    # at least four (sequence, KV head) pairs per CTA: the launch weighs shares by
    # pairs (88 of 96 sequences hold tiles) ...
    "many_pairs_weighted": dict(B=96, lens=(1, 64, 65, 129, 200, 300, 511, 0, 700, 128, 127, 40) * 8),
    # ... and the same launch with too few non-empty sequences for the weight
    # (16 of 96), which then splits the tiles equally
    "many_pairs_mostly_empty": dict(B=96, lens=(0, 0, 0, 0, 0, 300) * 16),
}


def _run_case(name, fp8=False, check_bytes=True):
    nv = _nv()
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Workload
    spec = _spec(name=name, **CASES[name])
    wl = Workload(spec, seed=zlib.crc32(name.encode()) % 1000, device="cuda")
    lay = Layer(wl, 0, prec=nv.PREC_FP8 if fp8 else nv.PREC_NVFP4)
    lay.step()
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    orc = OracleLayer(wl, 0, range(spec.B), fp8)
    assert np.array_equal(lay.scale.cpu().numpy(), orc.g), (lay.scale.cpu().numpy(), orc.g)
    if check_bytes:  # written slots only: tokens [0, L) of each sequence
        orc.compare_bytes(lay.cache.data)
    want = orc.attention()
    got = lay.out.float().cpu().numpy()
    ok, worst = within_tol(got, want)
    assert ok, f"max excess over tolerance {worst}"
    return got, want


@pytest.mark.parametrize("name", list(CASES))
def test_nvfp4_write_and_decode(name):
    _run_case(name, fp8=False)


@pytest.mark.parametrize("name", ["ragged_p64", "ragged_p16", "empty_seqs", "gqa8", "splits7", "many_pairs_weighted"])
def test_fp8_write_and_decode(name):
    _run_case(name, fp8=True)


@pytest.mark.parametrize("fp8", [False, True])
def test_query_with_outliers(fp8):
    """The score MMA takes the BF16 query as a sum of four NVFP4 (or E4M3)
    terms; a query whose 16-value blocks hold one large outlier each (the
    case that leaves the largest residual on the small values beside it)
    still meets the tolerance."""
    nv = _nv()
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Workload
    spec = _spec(name="q_outliers", B=3, lens=(900, 130, 64))
    wl = Workload(spec, seed=21, device="cuda")
    lay = Layer(wl, 0, prec=nv.PREC_FP8 if fp8 else nv.PREC_NVFP4)
    gen = torch.Generator().manual_seed(22)
    q = torch.randn(spec.B, spec.Hq, 128, generator=gen)
    pos = torch.randint(0, 16, (spec.B, spec.Hq, 8), generator=gen) + 16 * torch.arange(8)
    q.scatter_(2, pos, 40.0 * torch.sign(torch.randn(spec.B, spec.Hq, 8, generator=gen)))
    q[:, :, 5] = 300.0  # one channel far above the rest
    qb = q.to(torch.bfloat16)
    lay.step()
    lay.decode(q=qb.cuda())
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    orc = OracleLayer(wl, 0, range(spec.B), fp8)
    orc.q_bits = qb.view(torch.int16).numpy().view(np.uint16)
    ok, worst = within_tol(lay.out.float().cpu().numpy(), orc.attention())
    assert ok, f"max excess over tolerance {worst}"


@pytest.mark.parametrize("fp8", [False, True])
def test_every_split_count_matches_the_oracle(fp8):
    """The automatic schedule, one partition per sequence and many partitions
    per sequence each give the oracle's attention within the parity
    tolerance (the split-KV merge changes only the order of the FP32 sums),
    and a fixed schedule gives the same bits on a second call."""
    nv = _nv()
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Workload
    spec = _spec(B=3, lens=(3000, 777, 64))
    wl = Workload(spec, seed=3, device="cuda")
    orc = None
    for ns in (0, 1, 5, 40):
        lay = Layer(wl, 0, num_splits=ns, prec=1 if fp8 else 0)
        lay.decode()
        first = lay.out.clone()
        lay.decode()
        torch.cuda.synchronize()
        assert lay.cache.err.item() == 0
        assert torch.equal(first, lay.out), f"num_splits={ns}: two calls differ"
        if orc is None:
            orc = OracleLayer(wl, 0, range(spec.B), fp8)
            want = orc.attention()
        ok, worst = within_tol(lay.out.float().cpu().numpy(), want)
        assert ok, f"num_splits={ns}: max excess over tolerance {worst}"
    del nv


def test_bf16_input_write_matches_oracle():
    """BF16 K/V widen exactly: the write of BF16 values equals the oracle's
    write of the same values in FP32."""
    nv = _nv()
    import oracle
    T, Hkv, P = 37, 8, 16
    g = torch.Generator(device="cuda").manual_seed(5)
    k = (torch.randn(T, Hkv, 128, generator=g, device="cuda") * 3).to(torch.bfloat16)
    v = torch.randn(T, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    slots = torch.randperm(8 * P, generator=torch.Generator().manual_seed(1))[:T].to(torch.int64)
    slots[3] = -1
    for prec in (nv.PREC_NVFP4, nv.PREC_FP8):
        div = nv.NVFP4_GLOBAL_DIVISOR if prec == nv.PREC_NVFP4 else nv.FP8_GLOBAL_DIVISOR
        scale = torch.zeros(2, device="cuda")
        nv.nvkv_global_scale(k, scale[0:1], div)
        nv.nvkv_global_scale(v, scale[1:2], div)
        c = nv.Cache(prec, 8, Hkv, P, kv_scale=scale)
        (nv.nvfp4_kv_quantize_write if prec == nv.PREC_NVFP4 else nv.fp8_kv_quantize_write)(
            k, v, slots.cuda(), scale, c)
        torch.cuda.synchronize()
        kf, vf = k.float().cpu().numpy(), v.float().cpu().numpy()
        gs = np.array([oracle.global_scale(kf, div), oracle.global_scale(vf, div)], np.float32)
        assert np.array_equal(scale.cpu().numpy(), gs)
        oc = oracle.Cache(prec, 8, Hkv, P, 128, gs)
        oracle.quantize_write(oc, kf, vf, slots.numpy())
        np.testing.assert_array_equal(c.data.cpu().numpy(), oc.data)  # whole cache: both start at zero


def test_workspace_dequant_matches_oracle():
    nv = _nv()
    import oracle
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Workload
    spec = _spec(B=5, lens=(700, 65, 1, 300, 128), extend_seqs=(0, 1, 3), extend_tokens=100, step_write=0)
    wl = Workload(spec, seed=9, device="cuda")
    lay = Layer(wl, 0)
    lay.extend()
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    orc = OracleLayer(wl, 0, [0, 1, 3], fp8=False, with_extend=False)
    # workspace scale = amax / 448 per K and V, computed on the oracle side from the inputs
    amax = [oracle.global_scale(np.concatenate([wl.kv(0, kind, b).cpu().numpy().ravel()
                                                for b in range(spec.B)]), 1.0) for kind in (0, 1)]
    ws_scale = np.array([oracle.global_scale(np.array([a], np.float32), 448.0) for a in amax], np.float32)
    assert np.array_equal(lay.ext["ws_scale"].cpu().numpy(), ws_scale)
    wk, wv = oracle.dequant_to_fp8_workspace(orc.cache, orc.block_table, [0, 1, 2], [700, 65, 300], ws_scale)
    np.testing.assert_array_equal(lay.ext["ws_k"].cpu().numpy(), wk)
    np.testing.assert_array_equal(lay.ext["ws_v"].cpu().numpy(), wv)
    # the extend chunk was written after the prefix: check those bytes too
    orc2 = OracleLayer(wl, 0, [0, 1, 3], fp8=False, with_extend=True)
    orc2.compare_bytes(lay.cache.data)
    del nv


def test_device_error_word_on_bad_slot_and_page():
    """Out-of-range slots and block-table entries are skipped and reported in
    the error word; nothing faults."""
    nv = _nv()
    c = nv.Cache(nv.PREC_NVFP4, 4, 2, 16, kv_scale=torch.ones(2, device="cuda"))
    k = torch.randn(2, 2, 128, device="cuda")
    nv.nvfp4_kv_quantize_write(k, k, torch.tensor([3, 4 * 16], dtype=torch.int64, device="cuda"), None, c)
    torch.cuda.synchronize()
    assert c.err.item() == 1  # NVKV_DEVERR_SLOT
    c.err.zero_()
    q = torch.randn(1, 8, 128, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    bt = torch.tensor([[0, 99]], dtype=torch.int32, device="cuda")
    ws = nv.alloc_decode_workspace(1, 8, 2)
    nv.nvfp4_paged_decode_attention(q, c, bt, torch.tensor([20], dtype=torch.int32, device="cuda"), nv.PREC_NVFP4,
                                    out, ws)
    torch.cuda.synchronize()
    assert c.err.item() == 2  # NVKV_DEVERR_PAGE
