"""Oracle side of the GPU parity tests: the expected bytes and attention of a
workload's layer, computed by the CPU oracle from the same seeded inputs the
GPU receives (the inputs are copied to the host; nothing comes from the CUDA
path).  Only the sequences under test are quantized and attended, in a compact
cache whose pages are renumbered 0..n-1 (test plumbing, not method arithmetic).
"""
import numpy as np

import oracle


def oracle_global_scales(wl, layer, fp8):
    """(g_K, g_V) over every token of the layer: amax per piece, then one divide."""
    div = oracle.FP8_GLOBAL_DIVISOR if fp8 else oracle.NVFP4_GLOBAL_DIVISOR
    g = []
    for kind in (0, 1):
        amax = [oracle.global_scale(wl.kv(layer, kind, b).cpu().numpy(), 1.0) for b in range(wl.spec.B)]
        g.append(oracle.global_scale(np.array(amax, np.float32), div))
    return np.array(g, np.float32)


class OracleLayer:
    def __init__(self, wl, layer, seqs, fp8, with_extend=False):
        s = wl.spec
        self.seqs = list(seqs)
        self.g = oracle_global_scales(wl, layer, fp8)
        self.ext = {b: (int(wl.ext[b]) if with_extend else 0) for b in self.seqs}
        pages = []
        for b in self.seqs:
            n = (int(wl.seq_lens[b]) + self.ext[b] + s.P - 1) // s.P
            pages.extend(int(p) for p in wl.block_table[b, :n])
        self.global_pages = np.array(pages, np.int64)
        remap = {p: i for i, p in enumerate(pages)}
        self.block_table = np.full((len(self.seqs), wl.max_pages), -1, np.int32)
        for i, b in enumerate(self.seqs):
            n = (int(wl.seq_lens[b]) + self.ext[b] + s.P - 1) // s.P
            self.block_table[i, :n] = [remap[int(p)] for p in wl.block_table[b, :n]]
        prec = oracle.PREC_FP8 if fp8 else oracle.PREC_NVFP4
        self.cache = oracle.Cache(prec, max(1, len(pages)), s.Hkv, s.P, s.D, self.g)
        self.lens = {b: int(wl.seq_lens[b]) + self.ext[b] for b in self.seqs}
        for i, b in enumerate(self.seqs):
            L = self.lens[b]
            if L == 0:
                continue
            t = np.arange(L)
            slots = self.block_table[i, t // s.P].astype(np.int64) * s.P + t % s.P
            oracle.quantize_write(self.cache, wl.kv(layer, 0, b, 0, L).cpu().numpy(),
                                  wl.kv(layer, 1, b, 0, L).cpu().numpy(), slots)
        self.seq_lens = np.array([int(wl.seq_lens[b]) for b in self.seqs], np.int32)
        self.q_bits = wl.q_bf16(layer).cpu().view(__import__("torch").int16).numpy().view(np.uint16)[self.seqs]

    def attention(self, num_splits=0):
        return oracle.paged_decode_attention(self.cache, self.q_bits, self.block_table, self.seq_lens,
                                             num_splits=num_splits)

    def compare_bytes(self, gpu_data):
        """Assert that every byte of every slot the oracle wrote equals the
        GPU cache's byte at the same position (GPU pages gathered in the
        compact order; slot byte positions from the oracle's layout)."""
        import torch
        c = self.cache
        P, pos = c.P, c.slot_positions()
        blocks = gpu_data[torch.from_numpy(self.global_pages).to(gpu_data.device)].cpu().numpy()
        hh = np.arange(c.Hkv)[None, :, None]
        for i, b in enumerate(self.seqs):
            L = self.lens[b]
            for t0 in range(0, L, 4096):
                t = np.arange(t0, min(L, t0 + 4096))
                lp = self.block_table[i, t // P][:, None, None]
                idx = pos[t % P][:, None, :]
                got, want = blocks[lp, hh, idx], c.data[lp, hh, idx]
                if not np.array_equal(got, want):
                    bad = np.argwhere(got != want)[0]
                    raise AssertionError(f"cache bytes differ: sequence {b}, token {t0 + bad[0]}, head {bad[1]}, "
                                         f"byte {bad[2]} of the slot: gpu {got[tuple(bad)]:#x} oracle "
                                         f"{want[tuple(bad)]:#x}")


def within_tol(got, want, atol=2e-3, rtol=1e-2):
    """Elementwise |got - want| <= atol + rtol*|want|; returns (ok, worst excess)."""
    err = np.abs(got - want) - (atol + rtol * np.abs(want))
    return bool(np.all(err <= 0)), float(err.max())
