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
