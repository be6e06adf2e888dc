"""Device-side driver of the decode hot path for one workload.

Builds a layer's paged cache on the GPU from a seeded workload, using only
this library's kernels for every step of the method (global scale, quantized
write, decode attention, workspace dequant), and exposes ``step()``: the work
of one serving step for that layer, i.e. the quantized write of the step's new
tokens, the paged decode attention over the batch and, for workloads with a
chunked-extend pass, the prefix dequant into the shared FP8 workspace plus the
write of the new chunk.  With one new token per sequence the write and the
attention run as one launch (nvfp4_paged_decode_step).  PyTorch only
allocates memory and orders streams.
"""
from __future__ import annotations

from typing import List, Optional

import numpy as np
import torch

from . import (Cache, FP8_GLOBAL_DIVISOR, NVFP4_GLOBAL_DIVISOR, PREC_FP8, PREC_NVFP4, alloc_decode_workspace,
               alloc_extend_scratch, fp8_chunked_extend_attention, fp8_kv_quantize_write,
               fp8_workspace_append_chunk, nvfp4_kv_dequant_to_fp8_workspace, nvfp4_kv_quantize_write,
               nvfp4_paged_decode_attention, nvfp4_paged_decode_step, nvkv_amax_update, nvkv_global_scale)
from .workloads import Workload


class Layer:
    """One layer of a workload: cache, scales and step inputs on the device.

    ``prec`` overrides the workload's precision map (the FP8 comparator runs
    the same workload with every layer in FP8).  ``fused`` chooses the
    one-launch decode step where the workload writes one new token per
    sequence (default) or the separate write and decode calls.
    ``extend_attention`` adds, to a workload's chunked-extend pass, the chunk's
    append to the FP8 workspace and the FP8 attention of its queries over
    [prefix || chunk] (the workspace then reserves each chunk's rows behind its
    prefix, every sequence starting on a multiple of 8 rows).
    """

    def __init__(self, wl: Workload, layer: int, device="cuda", prec: Optional[int] = None,
                 num_splits: Optional[int] = None, fused: Optional[bool] = None, extend_attention: bool = False):
        s = wl.spec
        self.wl, self.layer, self.device = wl, layer, torch.device(device)
        self.prec = prec if prec is not None else (PREC_FP8 if wl.is_fp8(layer) else PREC_NVFP4)
        self.num_splits = s.num_splits if num_splits is None else num_splits
        div = FP8_GLOBAL_DIVISOR if self.prec == PREC_FP8 else NVFP4_GLOBAL_DIVISOR
        # global scale over every token the layer will hold (prefix, step and
        # extend tokens), K and V separately
        self.amax = torch.zeros(2, dtype=torch.float32, device=self.device)
        for b in range(s.B):
            for kind in (0, 1):
                nvkv_amax_update(wl.kv(layer, kind, b), self.amax[kind:kind + 1])
        self.scale = torch.zeros(2, dtype=torch.float32, device=self.device)
        for kind in (0, 1):
            nvkv_global_scale(self.amax[kind:kind + 1], self.scale[kind:kind + 1], div)
        self.cache = Cache(self.prec, wl.num_pages, s.Hkv, s.P, device=self.device, kv_scale=self.scale)
        for b in range(s.B):  # initial fill of each sequence's visible prefix
            L = int(wl.seq_lens[b])
            if L:
                self.write(wl.kv(layer, 0, b, 0, L), wl.kv(layer, 1, b, 0, L),
                           torch.from_numpy(wl.slots(b, 0, L)).to(self.device))
        self.block_table = torch.from_numpy(wl.block_table).to(self.device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(self.device)
        self.q = wl.q_bf16(layer)
        self.k_new = self.v_new = self.slots_new = None
        if wl.step_seqs():  # tokens re-written inside each step (the last ones of each sequence)
            ks, vs = [], []
            for b in wl.step_seqs():
                L = int(wl.seq_lens[b])
                ks.append(wl.kv(layer, 0, b, L - s.step_write, L))
                vs.append(wl.kv(layer, 1, b, L - s.step_write, L))
            self.k_new, self.v_new = torch.cat(ks).contiguous(), torch.cat(vs).contiguous()
            self.slots_new = torch.from_numpy(wl.step_slots()).to(self.device)
        # the one-launch step's inputs: row b = the newest token of sequence b
        self.k_step = self.v_step = None
        if s.step_write == 1 and wl.step_seqs():
            self.k_step = torch.zeros(s.B, s.Hkv, s.D, dtype=torch.float32, device=self.device)
            self.v_step = torch.zeros_like(self.k_step)
            rows = torch.tensor(wl.step_seqs(), dtype=torch.int64, device=self.device)
            self.k_step[rows] = self.k_new
            self.v_step[rows] = self.v_new
        self.fused = (self.k_step is not None) if fused is None else (fused and self.k_step is not None)
        self.ext = None
        if s.extend_seqs and self.prec == PREC_NVFP4:
            ids = [b for b in s.extend_seqs if b < s.B]
            pref = [int(wl.seq_lens[b]) for b in ids]
            n_ext = s.extend_tokens
            cu = np.zeros(len(ids) + 1, np.int64)
            if extend_attention:  # [prefix || chunk] per sequence, starts on multiples of 8 rows
                for i, p in enumerate(pref):
                    cu[i + 1] = cu[i] + (p + n_ext + 7) // 8 * 8
            else:  # the prefixes back to back
                cu[1:] = np.cumsum(pref)
            ws_scale = torch.zeros(2, dtype=torch.float32, device=self.device)
            for kind in (0, 1):  # FP8 per-tensor convention: amax / 448
                nvkv_global_scale(self.amax[kind:kind + 1], ws_scale[kind:kind + 1], FP8_GLOBAL_DIVISOR)
            self.ext = dict(
                seq_ids=torch.tensor(ids, dtype=torch.int32, device=self.device),
                prefix_lens=torch.tensor(pref, dtype=torch.int32, device=self.device),
                cu_prefix=torch.from_numpy(cu).to(self.device),
                ws_scale=ws_scale,
                ws_k=torch.empty(int(cu[-1]), s.Hkv, s.D, dtype=torch.uint8, device=self.device),
                ws_v=torch.empty(int(cu[-1]), s.Hkv, s.D, dtype=torch.uint8, device=self.device),
                k=torch.cat([wl.kv(layer, 0, b, pref[i], pref[i] + n_ext) for i, b in enumerate(ids)]).contiguous(),
                v=torch.cat([wl.kv(layer, 1, b, pref[i], pref[i] + n_ext) for i, b in enumerate(ids)]).contiguous(),
                slots=torch.from_numpy(np.concatenate([wl.slots(b, pref[i], pref[i] + n_ext)
                                                       for i, b in enumerate(ids)])).to(self.device),
            )
            if extend_attention:
                e = self.ext
                nq = len(ids) * n_ext
                e.update(
                    rows=torch.from_numpy(np.concatenate([cu[i] + pref[i] + np.arange(n_ext) for i in range(len(ids))])
                                          .astype(np.int64)).to(self.device),
                    q=wl.ext_q_bf16(layer, nq),
                    cu_q=torch.arange(0, nq + 1, max(n_ext, 1), dtype=torch.int64, device=self.device)[:len(ids) + 1],
                    cu_kv=torch.from_numpy(cu[:-1].copy()).to(self.device),
                    kv_lens=torch.tensor([p + n_ext for p in pref], dtype=torch.int32, device=self.device),
                    max_q=n_ext,
                    out=torch.empty(nq, s.Hq, s.D, dtype=torch.bfloat16, device=self.device),
                    scratch=alloc_extend_scratch(e["ws_k"]),
                    err=torch.zeros(1, dtype=torch.int32, device=self.device))
        self.out = torch.empty(s.B, s.Hq, s.D, dtype=torch.bfloat16, device=self.device)
        self.workspace = alloc_decode_workspace(s.B, s.Hq, s.Hkv, self.num_splits, device=self.device)

    # ------------------------------------------------------------------ steps
    def write(self, k, v, slots):
        if self.prec == PREC_NVFP4:
            nvfp4_kv_quantize_write(k, v, slots, self.scale, self.cache)
        else:
            fp8_kv_quantize_write(k, v, slots, self.scale, self.cache)

    def decode(self, q=None, out=None):
        nvfp4_paged_decode_attention(q if q is not None else self.q, self.cache, self.block_table, self.seq_lens,
                                     self.prec, out if out is not None else self.out, self.workspace,
                                     num_splits=self.num_splits)

    def extend(self):
        """The chunked-extend pass: the cached prefix into the FP8 workspace,
        (with extend_attention) the chunk behind it and the chunk's attention,
        then the chunk quantized into the cache."""
        e = self.ext
        nvfp4_kv_dequant_to_fp8_workspace(self.block_table, e["seq_ids"], e["prefix_lens"], e["cu_prefix"],
                                          self.cache, e["ws_scale"], e["ws_k"], e["ws_v"])
        if "q" in e:
            fp8_workspace_append_chunk(e["k"], e["v"], e["rows"], e["ws_scale"], e["ws_k"], e["ws_v"], err=e["err"])
            fp8_chunked_extend_attention(e["q"], e["cu_q"], e["max_q"], e["ws_k"], e["ws_v"], e["cu_kv"],
                                         e["kv_lens"], e["ws_scale"], e["out"], e["scratch"], err=e["err"])
        self.write(e["k"], e["v"], e["slots"])

    def step(self):
        if self.fused:
            nvfp4_paged_decode_step(self.q, self.k_step, self.v_step, self.cache, self.block_table, self.seq_lens,
                                    self.prec, self.out, self.workspace, num_splits=self.num_splits)
        else:
            if self.k_new is not None:
                self.write(self.k_new, self.v_new, self.slots_new)
            self.decode()
        if self.ext is not None:
            self.extend()

    def step_inputs(self) -> List[torch.Tensor]:
        """The tensors a step reads that come from the host each step: the
        queries and the new tokens (with their slots for the separate write)."""
        if self.fused:
            return [self.q, self.k_step, self.v_step]
        return [self.q] + ([self.k_new, self.v_new, self.slots_new] if self.k_new is not None else [])

    def set_step_inputs(self, ts: List[torch.Tensor]):
        """Rebind the step inputs (same order as step_inputs) to other tensors."""
        self.q = ts[0]
        if self.fused:
            self.k_step, self.v_step = ts[1], ts[2]
        elif self.k_new is not None:
            self.k_new, self.v_new, self.slots_new = ts[1], ts[2], ts[3]

    def launches_per_step(self) -> int:
        n = 1 if self.fused else (1 if self.k_new is not None else 0) + 1
        if self.ext is not None:
            n += 2 + (3 if "q" in self.ext else 0)  # dequant, chunk write (+ append, tile expansion, attention)
        return n

    # ------------------------------------------------------------ bookkeeping
    def kv_bytes_read(self) -> int:
        """Algorithmic bytes decode reads: K/V codes and scales of every visible token."""
        per_tok = 144 if self.prec == PREC_NVFP4 else 256
        return int(self.wl.seq_lens.astype(np.int64).sum()) * self.wl.spec.Hkv * per_tok

    def qo_bytes(self) -> int:
        s = self.wl.spec
        return 2 * s.B * s.Hq * s.D * 2


def build_layers(wl: Workload, device="cuda", layers: Optional[List[int]] = None, prec=None) -> List[Layer]:
    idx = layers if layers is not None else list(range(wl.spec.layers))
    return [Layer(wl, l, device, prec=prec) for l in idx]
