"""Seeded synthetic inputs for the NVFP4 paged-KV decode path.

This module only draws random numbers and builds index tables (block tables,
slot mappings, sequence lengths).  It holds none of the method's arithmetic:
no scale, no rounding, no attention.  Both the CUDA path and the CPU oracle
receive the very same tensors from here.

Random numbers come from ``torch.Generator`` (Philox on CUDA, MT19937 on the
CPU), one generator per (seed, layer, sequence, K/V) stream, so any one
sequence's values can be regenerated alone on the same device.  The tensors
are the same for a given device; CPU and CUDA streams differ, which no test
relies on.

Workloads (shapes and value distributions follow the long-context decode
settings that the NVFP4 KV-cache pages describe: GQA decode over a paged
cache, outlier channels, a per-layer FP8/NVFP4 map with the first and last
layers in FP8):

  decode_b1_ctx1k      B=1, 8 q / 2 KV heads, D=128, L=1024, page 16,
                       contiguous block table, N(0,1) with 4 outlier
                       channels per KV head scaled x20
  decode_b16_ctx8k     B=16, 32/8 heads, L=8192, page 64, permuted table,
                       N(0,1) with 1% of elements x20; one new token per
                       sequence written in the step
  mixed28_b44 / _b70   28 layers, FP8 on layers {0, 25, 26, 27}, B=44 / 70,
                       L=4096, page 64, N(0,1) x per-channel std
                       lognormal(0, 0.5)
  longctx_b2_ctx128k   B=2, L=131072, page 64, 64 split-KV partitions,
                       N(0,1) with 0.5% of elements x30
  serving_mix_b256     256 sequences, L ~ round(lognormal(ln 6000, 1)) clipped
                       to [1024, 65536], page 64, N(0,1); chunked-extend pass
                       on sequences 0..3 (2048 new tokens each)
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    L: int = 0                      # fixed length (0: drawn, see lens_lognormal)
    lens: Optional[Tuple[int, ...]] = None  # explicit per-sequence lengths (ragged test cases)
    lens_lognormal: Optional[Tuple[float, float, int, int]] = None  # median, sigma, lo, hi
    dist: str = "normal"            # normal | channel_outliers | element_outliers | lognormal_channels
    outlier_scale: float = 1.0
    outlier_p: float = 0.0
    outlier_channels: int = 0
    channel_sigma: float = 0.0
    table: str = "permuted"         # contiguous | permuted
    step_write: int = 0             # tokens per sequence re-written inside the step (the last ones)
    layers: int = 1
    fp8_layers: Tuple[int, ...] = ()
    num_splits: int = 0             # 0: automatic
    extend_seqs: Tuple[int, ...] = ()
    extend_tokens: int = 0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


SPECS = {
    "decode_b1_ctx1k": Spec("decode_b1_ctx1k", B=1, Hq=8, Hkv=2, D=128, P=16, L=1024, dist="channel_outliers",
                            outlier_scale=20.0, outlier_channels=4, table="contiguous", step_write=1024),
    "decode_b16_ctx8k": Spec("decode_b16_ctx8k", B=16, Hq=32, Hkv=8, D=128, P=64, L=8192,
                             dist="element_outliers", outlier_scale=20.0, outlier_p=0.01, step_write=1),
    "mixed28_b44": Spec("mixed28_b44", B=44, Hq=32, Hkv=8, D=128, P=64, L=4096, dist="lognormal_channels",
                        channel_sigma=0.5, step_write=1, layers=28, fp8_layers=(0, 25, 26, 27)),
    "mixed28_b70": Spec("mixed28_b70", B=70, Hq=32, Hkv=8, D=128, P=64, L=4096, dist="lognormal_channels",
                        channel_sigma=0.5, step_write=1, layers=28, fp8_layers=(0, 25, 26, 27)),
    "longctx_b2_ctx128k": Spec("longctx_b2_ctx128k", B=2, Hq=32, Hkv=8, D=128, P=64, L=131072,
                               dist="element_outliers", outlier_scale=30.0, outlier_p=0.005, num_splits=64),
    "serving_mix_b256": Spec("serving_mix_b256", B=256, Hq=32, Hkv=8, D=128, P=64,
                             lens_lognormal=(6000.0, 1.0, 1024, 65536), dist="normal",
                             extend_seqs=(0, 1, 2, 3), extend_tokens=2048),
}


def scaled(spec: Spec, **kw) -> Spec:
    """A smaller copy of a workload (same distribution and structure)."""
    return dataclasses.replace(spec, **kw)


def _gen(device, *key) -> torch.Generator:
    s = 0x9E3779B97F4A7C15
    for k in key:
        s = (s * 0x100000001B3 + int(k) + 0x632BE59BD9B4E019) & ((1 << 63) - 1)
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


class Workload:
    """Index tables and value streams of one workload on one device."""

    def __init__(self, spec: Spec, seed: int = 0, device="cpu"):
        self.spec, self.seed, self.device = spec, seed, torch.device(device)
        s = spec
        if s.lens is not None:
            self.seq_lens = np.array(s.lens, np.int32)
        elif s.lens_lognormal is not None:
            med, sig, lo, hi = s.lens_lognormal
            g = _gen("cpu", seed, 1, 0xA11)
            z = torch.randn(s.B, generator=g, dtype=torch.float64)
            lens = torch.clamp(torch.round(torch.exp(math.log(med) + sig * z)), lo, hi).to(torch.int64)
            self.seq_lens = lens.numpy().astype(np.int32)
        else:
            self.seq_lens = np.full(s.B, s.L, np.int32)
        # pages each sequence owns: its tokens plus any extend tokens
        self.ext = np.zeros(s.B, np.int32)
        for b in s.extend_seqs:
            if b < s.B:
                self.ext[b] = s.extend_tokens
        need = (self.seq_lens + self.ext + s.P - 1) // s.P
        self.max_pages = max(1, int(need.max())) if s.B else 1
        self.num_pages = int(need.sum())
        if s.table == "contiguous":
            order = np.arange(self.num_pages, dtype=np.int64)
        else:
            g = _gen("cpu", seed, 2, 0xB7)
            order = torch.randperm(self.num_pages, generator=g).numpy()
        self.block_table = np.full((s.B, self.max_pages), -1, np.int32)
        pos = 0
        for b in range(s.B):
            self.block_table[b, :need[b]] = order[pos:pos + need[b]]
            pos += need[b]

    # ------------------------------------------------------------------ tables
    def slots(self, b: int, t0: int, t1: int) -> np.ndarray:
        """Cache slot (page * P + offset) of tokens [t0, t1) of sequence b."""
        t = np.arange(t0, t1, dtype=np.int64)
        return self.block_table[b, t // self.spec.P].astype(np.int64) * self.spec.P + t % self.spec.P

    def step_slots(self) -> np.ndarray:
        """Slots of the tokens re-written inside one step, sequence-major."""
        s = self.spec
        return np.concatenate([self.slots(b, int(self.seq_lens[b]) - s.step_write, int(self.seq_lens[b]))
                               for b in self.step_seqs()] + [np.zeros(0, np.int64)])

    def step_seqs(self):
        """Sequences that re-write their last tokens inside a step."""
        s = self.spec
        return [b for b in range(s.B) if s.step_write and self.seq_lens[b] >= s.step_write]

    def is_fp8(self, layer: int) -> bool:
        return layer in self.spec.fp8_layers

    # ------------------------------------------------------------------ values
    def _channel_std(self, layer, kind):
        s = self.spec
        if s.dist == "lognormal_channels":
            g = _gen(self.device, self.seed, 3, layer, kind)
            z = torch.randn(s.Hkv, s.D, generator=g, device=self.device)
            return torch.exp(s.channel_sigma * z)
        if s.dist == "channel_outliers":
            g = _gen("cpu", self.seed, 4, layer, kind)
            std = torch.ones(s.Hkv, s.D)
            for h in range(s.Hkv):
                ch = torch.randperm(s.D, generator=g)[:s.outlier_channels]
                std[h, ch] = s.outlier_scale
            return std.to(self.device)
        return None

    def kv(self, layer: int, kind: int, b: int, t0: int = 0, t1: Optional[int] = None) -> torch.Tensor:
        """FP32 values [t1 - t0, Hkv, D] of K (kind 0) or V (kind 1) for
        positions [t0, t1) of sequence b (extend positions included)."""
        s = self.spec
        total = int(self.seq_lens[b] + self.ext[b])
        if t1 is None:
            t1 = total
        g = _gen(self.device, self.seed, 5, layer, kind, b)
        x = torch.randn(total, s.Hkv, s.D, generator=g, device=self.device, dtype=torch.float32)
        if s.dist == "element_outliers":
            u = torch.rand(total, s.Hkv, s.D, generator=g, device=self.device)
            x = torch.where(u < s.outlier_p, x * s.outlier_scale, x)
        std = self._channel_std(layer, kind)
        if std is not None:
            x = x * std
        return x[t0:t1].contiguous()

    def ext_q_bf16(self, layer: int, n: int) -> torch.Tensor:
        """BF16 queries [n, Hq, D] of the chunked-extend tokens (N(0,1) drawn in FP32, cast by torch)."""
        s = self.spec
        g = _gen(self.device, self.seed, 7, layer)
        return torch.randn(n, s.Hq, s.D, generator=g, device=self.device).to(torch.bfloat16)

    def q_bf16(self, layer: int = 0) -> torch.Tensor:
        """BF16 queries [B, Hq, D] (N(0,1) drawn in FP32, cast by torch)."""
        s = self.spec
        g = _gen(self.device, self.seed, 6, layer)
        return torch.randn(s.B, s.Hq, s.D, generator=g, device=self.device).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Chunked-extend workloads: a batch of sequences, each a cached prefix plus a
# chunk of new tokens whose queries attend over [prefix || chunk].
# ---------------------------------------------------------------------------
EXTEND_SPECS = {
    # four serving sequences (1k-12k token prefixes) extended by 2048 tokens each
    "extend_b4_chunk2k": dict(prefixes=(1024, 5000, 7000, 12000), chunks=(2048, 2048, 2048, 2048), Hq=32, Hkv=8),
}


def extend_inputs(seed, prefixes, chunks, Hq, Hkv, D=128, gap=16, outlier_p=0.01, outlier_scale=20.0):
    """Seeded host arrays of one chunked-extend batch: K/V for every position
    (prefix and chunk) N(0,1) with a fraction `outlier_p` of elements scaled
    by `outlier_scale` (the element-outlier recipe of the decode workloads),
    BF16-representable queries N(0,1) for the chunk tokens, and the workspace
    row layout: sequence i owns rows cu_kv[i] .. cu_kv[i] + prefix + chunk
    (cu_kv[i] a multiple of 8), with at least `gap` unused rows between
    sequences."""
    rng = np.random.default_rng(seed)
    n = len(prefixes)
    kv_lens = np.array([p + c for p, c in zip(prefixes, chunks)], np.int32)
    cu_kv = np.zeros(n, np.int64)
    r = 0
    for i in range(n):
        cu_kv[i] = r
        r = (r + int(kv_lens[i]) + gap + 7) // 8 * 8  # each sequence starts on a multiple of 8 rows
    T = int(kv_lens.sum())
    k = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    for x in (k, v):
        m = rng.random(x.shape) < outlier_p
        x[m] *= outlier_scale
    rows = np.concatenate([cu_kv[i] + np.arange(kv_lens[i]) for i in range(n)]).astype(np.int64)
    chunk_rows = np.concatenate([cu_kv[i] + prefixes[i] + np.arange(chunks[i]) for i in range(n)]).astype(np.int64)
    chunk_idx = np.concatenate([int(kv_lens[:i].sum()) + prefixes[i] + np.arange(chunks[i])
                                for i in range(n)]).astype(np.int64)
    cu_q = np.zeros(n + 1, np.int64)
    cu_q[1:] = np.cumsum(chunks)
    q = torch.from_numpy(rng.standard_normal((int(cu_q[-1]), Hq, D)).astype(np.float32)).to(torch.bfloat16)
    return dict(k=k, v=v, rows=rows, ws_rows=r, cu_kv=cu_kv, kv_lens=kv_lens, cu_q=cu_q, q=q,
                chunk_rows=chunk_rows, chunk_idx=chunk_idx, prefixes=tuple(prefixes), chunks=tuple(chunks))
