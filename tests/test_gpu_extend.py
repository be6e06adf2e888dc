"""GPU parity of the chunked-extend path: the chunk's append into the FP8
workspace (bytes bit-exact against the oracle) and the causal FP8 extend
attention (|gpu - oracle| <= 2e-3 + 1e-2 |oracle| element by element, the
oracle being FP64 attention over the identical workspace bytes).

Cases span several 128-row M-tiles and 128-key tiles, ragged chunk ends, an
empty prefix, GQA groups 1, 2, 4 and 8, workspace gaps between sequences, and
a full-size serving chunk (4 sequences x 2048 new tokens over 1k-12k token
prefixes) checked on sampled queries: query j depends only on positions
[0, p + j], so the oracle evaluates it alone as a one-query problem.
"""
import zlib

import numpy as np
import pytest
import torch

from _oracle_side import within_tol

pytestmark = pytest.mark.gpu


def _nv():
    import nvfp4_quantized_paged_gb300 as nv
    nv.lib()
    return nv


def _inputs(seed, prefixes, chunks, Hq, Hkv):
    """The seeded chunked-extend generator plus a workspace scale per K and V
    (amax / 448, the FP8 per-tensor convention) chosen here as an input."""
    from nvfp4_quantized_paged_gb300.workloads import extend_inputs
    x = extend_inputs(seed, prefixes, chunks, Hq, Hkv)
    x["q"] = x["q"].float().numpy()
    x["ws_scale"] = np.array([np.abs(x["k"]).max() / 448.0, np.abs(x["v"]).max() / 448.0], np.float32)
    return x


def _device(x):
    nv = _nv()
    d = {}
    d["k"] = torch.from_numpy(x["k"]).cuda()
    d["v"] = torch.from_numpy(x["v"]).cuda()
    d["rows"] = torch.from_numpy(x["rows"]).cuda()
    d["ws_scale"] = torch.from_numpy(x["ws_scale"]).cuda()
    Hkv = x["k"].shape[1]
    d["ws_k"] = torch.zeros(x["ws_rows"], Hkv, 128, dtype=torch.uint8, device="cuda")
    d["ws_v"] = torch.zeros(x["ws_rows"], Hkv, 128, dtype=torch.uint8, device="cuda")
    d["err"] = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.fp8_workspace_append_chunk(d["k"], d["v"], d["rows"], d["ws_scale"], d["ws_k"], d["ws_v"], err=d["err"])
    d["q"] = torch.from_numpy(x["q"]).cuda().to(torch.bfloat16)
    d["cu_q"] = torch.from_numpy(x["cu_q"]).cuda()
    d["cu_kv"] = torch.from_numpy(x["cu_kv"]).cuda()
    d["kv_lens"] = torch.from_numpy(x["kv_lens"]).cuda()
    d["out"] = torch.full_like(d["q"], float("nan"))
    d["scratch"] = nv.alloc_extend_scratch(d["ws_k"])
    return d


def _attend(d, max_q_len):
    nv = _nv()
    nv.fp8_chunked_extend_attention(d["q"], d["cu_q"], max_q_len, d["ws_k"], d["ws_v"], d["cu_kv"], d["kv_lens"],
                                    d["ws_scale"], d["out"], d["scratch"], err=d["err"])
    torch.cuda.synchronize()


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


CASES = {
    "g4_three_seqs": dict(prefixes=(0, 200, 1000), chunks=(77, 130, 5), Hq=32, Hkv=8),
    "g1": dict(prefixes=(129,), chunks=(200,), Hq=4, Hkv=4),
    "g2_ragged": dict(prefixes=(31, 500), chunks=(129, 63), Hq=8, Hkv=4),
    "g8": dict(prefixes=(300, 0), chunks=(64, 17), Hq=16, Hkv=2),
    "one_token_no_prefix": dict(prefixes=(0, 0), chunks=(1, 2), Hq=8, Hkv=2),
}


@pytest.mark.parametrize("name", list(CASES))
def test_append_and_extend_attention_match_oracle(orc, name):
    c = CASES[name]
    x = _inputs(zlib.crc32(name.encode()) % 1000, c["prefixes"], c["chunks"], c["Hq"], c["Hkv"])
    d = _device(x)
    _attend(d, max(c["chunks"]) + 37)  # extra M-tiles past every chunk exit at once
    assert d["err"].item() == 0
    # workspace bytes: bit-exact against the oracle's append of the same values
    Hkv = c["Hkv"]
    wk = np.zeros((x["ws_rows"], Hkv, 128), np.uint8)
    wv = np.zeros((x["ws_rows"], Hkv, 128), np.uint8)
    orc.fp8_workspace_append(wk, wv, x["k"], x["v"], x["rows"], x["ws_scale"])
    assert np.array_equal(d["ws_k"].cpu().numpy(), wk)
    assert np.array_equal(d["ws_v"].cpu().numpy(), wv)
    want = orc.fp8_extend_attention(_bits(d["q"]), x["cu_q"], wk, wv, x["cu_kv"], x["kv_lens"], x["ws_scale"])
    got = d["out"].float().cpu().numpy()
    ok, worst = within_tol(got, want)
    assert ok, f"max excess over tolerance {worst}"


def test_bf16_chunk_append_matches_oracle(orc):
    x = _inputs(7, (40,), (90,), 8, 2)
    nv = _nv()
    kb = torch.from_numpy(x["k"]).cuda().to(torch.bfloat16)
    vb = torch.from_numpy(x["v"]).cuda().to(torch.bfloat16)
    rows = torch.from_numpy(x["rows"]).cuda()
    rows[3] = -1  # skipped
    s = torch.from_numpy(x["ws_scale"]).cuda()
    wk = torch.zeros(x["ws_rows"], 2, 128, dtype=torch.uint8, device="cuda")
    wv = torch.zeros_like(wk)
    nv.fp8_workspace_append_chunk(kb, vb, rows, s, wk, wv)
    ok_k = np.zeros((x["ws_rows"], 2, 128), np.uint8)
    ok_v = np.zeros_like(ok_k)
    orc.fp8_workspace_append(ok_k, ok_v, kb.float().cpu().numpy(), vb.float().cpu().numpy(), rows.cpu().numpy(),
                             x["ws_scale"])
    assert np.array_equal(wk.cpu().numpy(), ok_k) and np.array_equal(wv.cpu().numpy(), ok_v)


def test_full_size_serving_chunk_sampled(orc):
    """4 sequences x 2048 chunk tokens over long prefixes, 32 query / 8 KV
    heads: every output finite, sampled queries (first, last, tile edges,
    random) equal to the oracle's one-query problems."""
    prefixes, chunks = (1024, 5000, 7000, 12000), (2048,) * 4
    x = _inputs(11, prefixes, chunks, 32, 8)
    d = _device(x)
    _attend(d, 2048)
    assert d["err"].item() == 0
    got = d["out"].float().cpu().numpy()
    assert np.isfinite(got).all()
    wk = d["ws_k"].cpu().numpy()
    wv = d["ws_v"].cpu().numpy()
    qbits = _bits(d["q"])
    rng = np.random.default_rng(5)
    for i in range(4):
        for j in sorted({0, 31, 32, 2047, int(rng.integers(0, 2048))}):
            pos = prefixes[i] + j
            row = int(x["cu_q"][i]) + j
            want = orc.fp8_extend_attention(qbits[row:row + 1], [0, 1], wk, wv, [int(x["cu_kv"][i])], [pos + 1],
                                            x["ws_scale"])
            ok, worst = within_tol(got[row:row + 1], want)
            assert ok, f"sequence {i} query {j}: max excess {worst}"


def test_error_flag_for_unaligned_workspace_offset():
    x = _inputs(4, (10, 20), (30, 5), 8, 2)
    d = _device(x)
    d["cu_kv"][1] += 1  # a sequence must start on a multiple of 8 rows
    _attend(d, 30)
    assert d["err"].item() == 6  # NVKV_DEVERR_ALIGN; that sequence is skipped
    out = d["out"].float()
    assert torch.isfinite(out[:30]).all() and torch.isnan(out[30:]).all()


def test_error_flag_for_more_queries_than_keys():
    x = _inputs(3, (0,), (40,), 8, 2)
    d = _device(x)
    d["kv_lens"][0] = 20  # 40 queries cannot be the last positions of 20
    _attend(d, 40)
    assert d["err"].item() == 3  # NVKV_DEVERR_SEQLEN; the sequence is skipped
    assert torch.isnan(d["out"].float()).all()


def test_chunked_extend_chain_from_the_nvfp4_cache(orc):
    """The whole chunked-extend path ("SGLang x Qwen x NVIDIA ...", Three
    Paths): the cached NVFP4 prefix is dequantized into the shared FP8
    workspace, the chunk's K/V are appended behind it, FP8 attention of the
    chunk's queries runs over [prefix || chunk], and the chunk is then
    quantized into the NVFP4 cache.  The workspace is laid out as the
    attention reads it: each sequence starts on a multiple of 8 rows with its
    chunk's rows reserved right behind its prefix (cu_prefix = cu_kv).  Every
    byte (workspace, cache) matches the oracle's chain bit for bit and the
    attention is within the parity tolerance of the oracle's."""
    nv = _nv()
    prefixes, chunks, Hq, Hkv, P = (300, 1000, 64, 0), (130, 77, 200, 9), 32, 8, 64
    x = _inputs(11, prefixes, chunks, Hq, Hkv)
    n = len(prefixes)
    lens = [p + c for p, c in zip(prefixes, chunks)]
    pages_per = [(L + P - 1) // P for L in lens]
    max_pages = max(pages_per)
    num_pages = sum(pages_per) + 3
    perm = np.random.default_rng(4).permutation(num_pages).astype(np.int32)
    bt = np.full((n, max_pages), -1, np.int32)
    off = 0
    for i in range(n):
        bt[i, :pages_per[i]] = perm[off:off + pages_per[i]]
        off += pages_per[i]
    first = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)  # row of sequence i in x["k"]

    def slots(i, t0, t1):
        t = np.arange(t0, t1)
        return bt[i, t // P].astype(np.int64) * P + t % P

    pre_idx = np.concatenate([first[i] + np.arange(prefixes[i]) for i in range(n)]).astype(np.int64)
    pre_slots = np.concatenate([slots(i, 0, prefixes[i]) for i in range(n)])
    ch_slots = np.concatenate([slots(i, prefixes[i], lens[i]) for i in range(n)])
    ci = x["chunk_idx"]

    # ---- GPU chain, through the C ABI
    dev = "cuda"
    k_all, v_all = torch.from_numpy(x["k"]).to(dev), torch.from_numpy(x["v"]).to(dev)
    g = torch.zeros(2, dtype=torch.float32, device=dev)
    ws_scale = torch.zeros(2, dtype=torch.float32, device=dev)
    for kind, t in ((0, k_all), (1, v_all)):  # every token the layer holds, prefix and chunk
        nv.nvkv_global_scale(t, g[kind:kind + 1], nv.NVFP4_GLOBAL_DIVISOR)
        nv.nvkv_global_scale(t, ws_scale[kind:kind + 1], nv.FP8_GLOBAL_DIVISOR)
    cache = nv.Cache(nv.PREC_NVFP4, num_pages, Hkv, P, device=dev, kv_scale=g)
    pi = torch.from_numpy(pre_idx).to(dev)
    nv.nvfp4_kv_quantize_write(k_all[pi].contiguous(), v_all[pi].contiguous(), torch.from_numpy(pre_slots).to(dev),
                               g, cache)
    bt_d = torch.from_numpy(bt).to(dev)
    cu_prefix = np.concatenate([x["cu_kv"], [x["ws_rows"]]]).astype(np.int64)
    ws_k = torch.full((x["ws_rows"], Hkv, 128), 0x7F, dtype=torch.uint8, device=dev)  # NaN: rows never read
    ws_v = torch.full_like(ws_k, 0x7F)
    nv.nvfp4_kv_dequant_to_fp8_workspace(bt_d, torch.arange(n, dtype=torch.int32, device=dev),
                                         torch.tensor(prefixes, dtype=torch.int32, device=dev),
                                         torch.from_numpy(cu_prefix).to(dev), cache, ws_scale, ws_k, ws_v)
    cidx = torch.from_numpy(ci).to(dev)
    k_ch, v_ch = k_all[cidx].contiguous(), v_all[cidx].contiguous()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    nv.fp8_workspace_append_chunk(k_ch, v_ch, torch.from_numpy(x["chunk_rows"]).to(dev), ws_scale, ws_k, ws_v,
                                  err=err)
    q = x["q"].to(dev) if isinstance(x["q"], torch.Tensor) else torch.from_numpy(x["q"]).to(dev).to(torch.bfloat16)
    out = torch.full_like(q, float("nan"))
    scratch = nv.alloc_extend_scratch(ws_k)
    nv.fp8_chunked_extend_attention(q, torch.from_numpy(x["cu_q"]).to(dev), max(chunks), ws_k, ws_v,
                                    torch.from_numpy(x["cu_kv"]).to(dev), torch.from_numpy(x["kv_lens"]).to(dev),
                                    ws_scale, out, scratch, err=err)
    nv.nvfp4_kv_quantize_write(k_ch, v_ch, torch.from_numpy(ch_slots).to(dev), g, cache)
    torch.cuda.synchronize()
    assert err.item() == 0 and cache.err.item() == 0

    # ---- oracle chain on the same inputs
    g_o = np.array([orc.global_scale(x["k"], orc.NVFP4_GLOBAL_DIVISOR),
                    orc.global_scale(x["v"], orc.NVFP4_GLOBAL_DIVISOR)], np.float32)
    ws_o = np.array([orc.global_scale(x["k"], orc.FP8_GLOBAL_DIVISOR),
                     orc.global_scale(x["v"], orc.FP8_GLOBAL_DIVISOR)], np.float32)
    assert np.array_equal(g.cpu().numpy(), g_o) and np.array_equal(ws_scale.cpu().numpy(), ws_o)
    oc = orc.Cache(orc.PREC_NVFP4, num_pages, Hkv, P, 128, g_o)
    orc.quantize_write(oc, x["k"][pre_idx], x["v"][pre_idx], pre_slots)
    wk, wv = orc.dequant_to_fp8_workspace(oc, bt, np.arange(n), prefixes, ws_o, row_start=x["cu_kv"],
                                          ws_rows=x["ws_rows"])
    orc.fp8_workspace_append(wk, wv, x["k"][ci], x["v"][ci], x["chunk_rows"], ws_o)
    used = np.zeros(x["ws_rows"], bool)
    used[x["rows"]] = True  # every prefix and chunk row; gap rows were never written
    np.testing.assert_array_equal(ws_k.cpu().numpy()[used], wk[used])
    np.testing.assert_array_equal(ws_v.cpu().numpy()[used], wv[used])
    assert np.all(ws_k.cpu().numpy()[~used] == 0x7F)  # the dequant left the reserved gaps alone
    want = orc.fp8_extend_attention(_bits(q), x["cu_q"], wk, wv, x["cu_kv"], x["kv_lens"], ws_o)
    ok, worst = within_tol(out.float().cpu().numpy(), want)
    assert ok, f"max excess over tolerance {worst}"
    orc.quantize_write(oc, x["k"][ci], x["v"][ci], ch_slots)
    assert np.array_equal(cache.data.cpu().numpy(), oc.data)


def test_serving_mix_layer_runs_the_extend_attention(orc):
    """The serving-mix layer driver with the extend attention on: each extend
    sequence's cached NVFP4 prefix is dequantized into the workspace, its
    chunk appended behind it (rows reserved per sequence on 8-row starts), the
    chunk's queries attend over [prefix || chunk], and the chunk is written
    into the cache.  The attention output matches the oracle's chain on the
    same inputs within the parity tolerance, and the workspace rows it read
    match the oracle's bytes."""
    from _oracle_side import OracleLayer, oracle_global_scales
    from nvfp4_quantized_paged_gb300.runner import Layer
    from nvfp4_quantized_paged_gb300.workloads import Spec, Workload
    nv = _nv()
    spec = Spec("mix_extend", B=3, Hq=32, Hkv=8, D=128, P=64, lens=(700, 90, 1300), dist="normal", step_write=1,
                extend_seqs=(0, 2), extend_tokens=150)
    wl = Workload(spec, seed=17, device="cuda")
    lay = Layer(wl, 0, extend_attention=True)
    lay.extend()
    torch.cuda.synchronize()
    e = lay.ext
    assert e["err"].item() == 0 and lay.cache.err.item() == 0
    # oracle chain: prefix cache -> workspace rows at the same starts -> chunk append -> attention
    ids = [0, 2]
    orl = OracleLayer(wl, 0, ids, False)
    ws_o = oracle_global_scales(wl, 0, True)
    assert np.array_equal(e["ws_scale"].cpu().numpy(), ws_o)
    cu = e["cu_prefix"].cpu().numpy()
    prefixes = [int(wl.seq_lens[b]) for b in ids]
    wk, wv = orc.dequant_to_fp8_workspace(orl.cache, orl.block_table, np.arange(len(ids)), prefixes, ws_o,
                                          row_start=cu[:-1], ws_rows=int(cu[-1]))
    kc = np.concatenate([wl.kv(0, 0, b, p, p + 150).cpu().numpy() for b, p in zip(ids, prefixes)])
    vc = np.concatenate([wl.kv(0, 1, b, p, p + 150).cpu().numpy() for b, p in zip(ids, prefixes)])
    rows = e["rows"].cpu().numpy()
    orc.fp8_workspace_append(wk, wv, kc, vc, rows, ws_o)
    for i, p in enumerate(prefixes):
        r = slice(int(cu[i]), int(cu[i]) + p + 150)
        np.testing.assert_array_equal(e["ws_k"].cpu().numpy()[r], wk[r])
        np.testing.assert_array_equal(e["ws_v"].cpu().numpy()[r], wv[r])
    want = orc.fp8_extend_attention(_bits(e["q"].cpu()), e["cu_q"].cpu().numpy(), wk, wv, cu[:-1],
                                    e["kv_lens"].cpu().numpy(), ws_o)
    ok, worst = within_tol(e["out"].float().cpu().numpy(), want)
    assert ok, f"max excess over tolerance {worst}"
