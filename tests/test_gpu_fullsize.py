"""Full-size parity on sampled outputs.

Each workload runs at its real size, in the launch configuration bench.py
times.  The oracle recomputes the global scales from every token of the layer
(amax per sequence, then one divide) and quantizes and attends only sampled
sequences: their cache bytes must match bit for bit and their attention
outputs must be within 2e-3 + 1e-2 * |oracle| of the FP64 oracle.
"""
import numpy as np
import pytest
import torch

from _oracle_side import OracleLayer, within_tol

pytestmark = pytest.mark.gpu


def _check_layer(lay, wl, seqs, fp8, with_extend=False):
    spec = wl.spec
    torch.cuda.synchronize()
    assert lay.cache.err.item() == 0
    orc = OracleLayer(wl, lay.layer, seqs, fp8, with_extend=with_extend)
    assert np.array_equal(lay.scale.cpu().numpy(), orc.g)
    orc.compare_bytes(lay.cache.data)
    if with_extend:
        return orc
    want = orc.attention()
    got = lay.out.float().cpu().numpy()[seqs]
    ok, worst = within_tol(got, want)
    assert ok, f"max excess over tolerance {worst}"
    return orc


def _wl(name):
    from nvfp4_quantized_paged_gb300.workloads import SPECS, Workload
    return Workload(SPECS[name], seed=0, device="cuda")


def test_decode_b16_ctx8k_full():
    from nvfp4_quantized_paged_gb300.runner import Layer
    wl = _wl("decode_b16_ctx8k")
    lay = Layer(wl, 0)
    lay.step()
    _check_layer(lay, wl, [0, 7, 15], fp8=False)


@pytest.mark.parametrize("num_splits", [64, 0])
def test_longctx_b2_ctx128k_full(num_splits):
    from nvfp4_quantized_paged_gb300.runner import Layer
    wl = _wl("longctx_b2_ctx128k")
    lay = Layer(wl, 0, num_splits=num_splits)
    lay.step()
    _check_layer(lay, wl, [1], fp8=False)


# Both batches of the 28-layer mixed-precision workload, on the FP8 layers at
# either end of the map (0, 25, 26, 27) and NVFP4 layers beside and between
# them (1, 13), each checked on its first, a middle and its last sequence.
@pytest.mark.parametrize("layer", [0, 1, 13, 25, 26, 27])
@pytest.mark.parametrize("name,seqs", [("mixed28_b44", [0, 22, 43]), ("mixed28_b70", [0, 35, 69])])
def test_mixed28_sampled_layers(name, seqs, layer):
    from nvfp4_quantized_paged_gb300.runner import Layer
    wl = _wl(name)
    lay = Layer(wl, layer)
    assert wl.spec.fp8_layers == (0, 25, 26, 27)
    assert (lay.prec == 1) == (layer in (0, 25, 26, 27))
    lay.step()
    _check_layer(lay, wl, seqs, fp8=layer in (0, 25, 26, 27))


def test_serving_mix_b256_decode_and_extend():
    import oracle
    from nvfp4_quantized_paged_gb300.runner import Layer
    wl = _wl("serving_mix_b256")
    lay = Layer(wl, 0)
    lay.decode()
    torch.cuda.synchronize()
    longest = int(np.argmax(wl.seq_lens))
    seqs = sorted({5, 200, longest})
    _check_layer(lay, wl, seqs, fp8=False)
    # chunked-extend pass: prefix dequant of sequences 0..3, then the new chunk's write
    lay.extend()
    torch.cuda.synchronize()
    orc = _check_layer(lay, wl, [0, 1], fp8=False, with_extend=True)
    amax = [max(oracle.global_scale(wl.kv(0, kind, b).cpu().numpy(), 1.0) for b in range(wl.spec.B))
            for kind in (0, 1)]
    ws_scale = np.array([oracle.global_scale(np.array([a], np.float32), 448.0) for a in amax], np.float32)
    assert np.array_equal(lay.ext["ws_scale"].cpu().numpy(), ws_scale)
    pl = [int(wl.seq_lens[0]), int(wl.seq_lens[1])]
    wk, wv = oracle.dequant_to_fp8_workspace(orc.cache, orc.block_table, [0, 1], pl, ws_scale)
    np.testing.assert_array_equal(lay.ext["ws_k"][:sum(pl)].cpu().numpy(), wk)
    np.testing.assert_array_equal(lay.ext["ws_v"][:sum(pl)].cpu().numpy(), wv)
