"""Synthetic calibration study of the quantized KV cache.

The pages report that the NVFP4 KV cache costs accuracy on small models and
that its global scale is not calibrated yet ("SGLang x Qwen x NVIDIA ...",
opening summary; "SOAR Weekly Champion Notes 05", 03 on keeping sensitive
layers in FP8).  Without weights or datasets, this study measures what the
cache does to one attention layer: the decode output of the library's kernels
over an NVFP4 or FP8 cache against FP32 attention over the unquantized K/V,
for the synthetic distributions of the workloads (normal, sparse element
outliers, outlier channels, log-normal channel scales), and, for NVFP4, with
the global scale moved by a factor away from the amax / (6 * 448) rule (a
smaller scale saturates the largest values at 6 * 448 * g, a larger one pushes
small block scales into E4M3's subnormal range).

The reference is plain PyTorch FP32 attention (a measurement reference, not
the parity oracle: parity of the kernels is tested against the oracle
elsewhere).
"""
from __future__ import annotations

import math
from typing import Dict, List

import torch

from . import PREC_FP8, PREC_NVFP4
from .runner import Layer
from .workloads import Spec, Workload

DISTS: Dict[str, dict] = {
    "normal": {},
    "element_outliers": dict(outlier_scale=20.0, outlier_p=0.01),
    "channel_outliers": dict(outlier_scale=20.0, outlier_channels=4),
    "lognormal_channels": dict(channel_sigma=1.0),
}
FACTORS = (0.25, 0.5, 1.0, 2.0, 4.0)


def fp32_attention(wl: Workload) -> torch.Tensor:
    """Decode attention in FP32 over the unquantized K/V of layer 0: [B, Hq, D]."""
    s = wl.spec
    G = s.Hq // s.Hkv
    q = wl.q_bf16(0).float()
    out = torch.empty(s.B, s.Hq, s.D, dtype=torch.float32, device=q.device)
    for b in range(s.B):
        L = int(wl.seq_lens[b])
        k = wl.kv(0, 0, b, 0, L)
        v = wl.kv(0, 1, b, 0, L)
        for h in range(s.Hkv):
            sc = q[b, h * G:(h + 1) * G] @ k[:, h].T / math.sqrt(s.D)
            out[b, h * G:(h + 1) * G] = torch.softmax(sc, dim=-1) @ v[:, h]
    return out


def _rewrite(lay: Layer, wl: Workload):
    for b in range(wl.spec.B):
        L = int(wl.seq_lens[b])
        slots = torch.from_numpy(wl.slots(b, 0, L)).to(lay.device)
        lay.write(wl.kv(0, 0, b, 0, L), wl.kv(0, 1, b, 0, L), slots)


def study(device="cuda", B=4, L=4096, Hq=32, Hkv=8, factors=FACTORS, seed=0) -> List[dict]:
    """Rows {dist, prec, factor, rel_l2, max_abs, ref_rms} of output error vs FP32."""
    rows = []
    for dist, kw in DISTS.items():
        spec = Spec(name=f"calibration_{dist}", B=B, Hq=Hq, Hkv=Hkv, D=128, P=64, L=L, dist=dist, **kw)
        wl = Workload(spec, seed=seed, device=device)
        ref = fp32_attention(wl)
        for prec in (PREC_FP8, PREC_NVFP4):
            for f in (factors if prec == PREC_NVFP4 else (1.0,)):
                lay = Layer(wl, 0, device, prec=prec)
                if f != 1.0:
                    lay.scale.mul_(f)  # the cache's global scales (shared tensor)
                    _rewrite(lay, wl)
                lay.decode()
                torch.cuda.synchronize()
                got = lay.out.float()
                err = got - ref
                rows.append(dict(dist=dist, prec="fp8" if prec == PREC_FP8 else "nvfp4", factor=f,
                                 rel_l2=float(err.norm() / ref.norm()), max_abs=float(err.abs().max()),
                                 ref_rms=float(ref.pow(2).mean().sqrt()), cache_err=int(lay.cache.err.item())))
                del lay
    return rows
