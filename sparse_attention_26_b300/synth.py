"""Seeded synthetic inputs for the hybrid attention layer.

This module holds no arithmetic of the method: it only draws random numbers
and lays them out in the shapes the layer consumes.  Both the CUDA path and
the CPU oracle read the bytes it produces.

Recipe: seed s (default 0); tensor number i of a workload draws from a
generator seeded with s + i.  Values are N(0,1) rounded to bf16 (torch's
round-to-nearest-even), except the indexer head weights w and the sink logits
(N(0,1) fp32) and the positions (int32).  The tiny workload projects bf16
hidden states x [B, L, 256] through bf16 weights N(0,1)/sqrt(256) in fp64 and
rounds the projections to bf16; the large workloads sample the projected
tensors directly, which is the distribution such projections produce.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int            # sequences
    L: int            # cached tokens per sequence
    T: int            # queries per sequence, at positions [L - T, L)
    H: int            # query heads
    D: int            # head dim = shared KV latent dim
    r: int            # RoPE dims (the last r of each vector)
    HI: int           # indexer heads
    dI: int           # indexer dim
    k: int            # top-k
    W: int = 128      # SWA window
    m_csa: int = 4
    w_csa: int = 8
    m_hca: int = 128
    w_hca: int = 128
    branches: tuple = ("csa", "hca", "swa")
    d_model: int = 0  # >0: project from hidden states (tiny workload)
    base: float = 10000.0
    eps: float = 1e-6

    @property
    def n_csa(self) -> int:
        return self.L // self.m_csa

    @property
    def n_hca(self) -> int:
        return self.L // self.m_hca

    def cfg(self) -> dict:
        return dict(m_csa=self.m_csa, w_csa=self.w_csa, m_hca=self.m_hca, w_hca=self.w_hca,
                    k=self.k, W=self.W, r=self.r, base=self.base, eps=self.eps)


# The workloads (sizes from the layer shapes of V4-Flash / V4-Pro).
WORKLOADS = {
    "tiny": Workload("tiny", B=1, L=256, T=256, H=4, D=64, r=16, HI=2, dI=32, k=16,
                     d_model=256),
    "flash_csa_prefill": Workload("flash_csa_prefill", B=1, L=8192, T=8192, H=64, D=512, r=64,
                                  HI=64, dI=128, k=512, branches=("csa", "swa")),
    "pro_csa_decode": Workload("pro_csa_decode", B=32, L=131072, T=1, H=128, D=512, r=64, HI=64,
                               dI=128, k=1024, branches=("csa", "swa")),
    "hca_decode": Workload("hca_decode", B=16, L=1 << 20, T=1, H=128, D=512, r=64, HI=64,
                           dI=128, k=1024, branches=("hca",)),
    "hca_prefill": Workload("hca_prefill", B=1, L=1 << 20, T=4096, H=128, D=512, r=64, HI=64,
                            dI=128, k=1024, branches=("hca",)),
    "hybrid_decode_1m": Workload("hybrid_decode_1m", B=8, L=1 << 20, T=1, H=128, D=512, r=64,
                                 HI=64, dI=128, k=1024),
    # speculative decode with one multi-token-prediction draft: the accepted
    # token and the draft, two queries per sequence over the same caches
    "hybrid_decode_1m_mtp2": Workload("hybrid_decode_1m_mtp2", B=8, L=1 << 20, T=2, H=128,
                                      D=512, r=64, HI=64, dI=128, k=1024),
}


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some sizes replaced (for small parity cases)."""
    return dataclasses.replace(wl, **kw)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, seed, device, dtype=torch.bfloat16):
    g = _gen(device, seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    """Raw token caches and queries for one batch of the workload.

    Returns torch tensors on `device`:
      q [B,T,H,D] bf16, kv_raw [B,L,D] bf16, ik_raw [B,L,dI] bf16,
      gate_csa [B,L] bf16, gate_hca [B,L] bf16, iq [B,T,HI,dI] bf16,
      w [B,T,HI] fp32, sink [H] fp32, pos [B,T] int32.
    """
    B, L, T = wl.B, wl.L, wl.T
    out = {}
    if wl.d_model:
        dm = wl.d_model
        x = _randn((B, L, dm), seed + 0, device)
        s = 1.0 / math.sqrt(dm)

        def proj(n_out, i):
            Wt = (_randn((dm, n_out), seed + i, device).to(torch.float64) * s).to(torch.bfloat16)
            return x.to(torch.float64) @ Wt.to(torch.float64)

        out["kv_raw"] = proj(wl.D, 1).to(torch.bfloat16)
        out["ik_raw"] = proj(wl.dI, 2).to(torch.bfloat16)
        xq = x[:, L - T:]
        Wq = (_randn((dm, wl.H * wl.D), seed + 3, device).to(torch.float64) * s).to(torch.bfloat16)
        out["q"] = (xq.to(torch.float64) @ Wq.to(torch.float64)).to(torch.bfloat16).reshape(
            B, T, wl.H, wl.D)
        Wiq = (_randn((dm, wl.HI * wl.dI), seed + 4, device).to(torch.float64) * s).to(
            torch.bfloat16)
        out["iq"] = (xq.to(torch.float64) @ Wiq.to(torch.float64)).to(torch.bfloat16).reshape(
            B, T, wl.HI, wl.dI)
        Ww = (_randn((dm, wl.HI), seed + 5, device).to(torch.float64) * s).to(torch.bfloat16)
        out["w"] = (xq.to(torch.float64) @ Ww.to(torch.float64)).to(torch.float32)
    else:
        out["kv_raw"] = _randn((B, L, wl.D), seed + 1, device)
        out["ik_raw"] = _randn((B, L, wl.dI), seed + 2, device)
        out["q"] = _randn((B, T, wl.H, wl.D), seed + 3, device)
        out["iq"] = _randn((B, T, wl.HI, wl.dI), seed + 4, device)
        out["w"] = _randn((B, T, wl.HI), seed + 5, device, torch.float32)
    out["gate_csa"] = _randn((B, L), seed + 6, device)
    out["gate_hca"] = _randn((B, L), seed + 7, device)
    out["sink"] = _randn((wl.H,), seed + 8, device, torch.float32)
    out["pos"] = (torch.arange(L - T, L, dtype=torch.int32, device=device)
                  .unsqueeze(0).expand(B, T).contiguous())
    return out


def random_idx(B, T, k, n_visible, seed, device="cpu", n_valid=None):
    """Seeded distinct entry indices per query (a synthetic top-k result).

    n_visible: [B, T] visible entry counts.  Each row gets min(k, n_visible)
    (or n_valid) distinct indices in random order, padded with -1.
    """
    g = np.random.default_rng(seed)
    nv = np.asarray(n_visible).reshape(B, T)
    idx = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            n = int(nv[b, t])
            c = min(k, n) if n_valid is None else min(n_valid, n, k)
            if c > 0:
                idx[b, t, :c] = g.choice(n, size=c, replace=False).astype(np.int32)
    return torch.from_numpy(idx).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy); others -> numpy."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def to_numpy(inp: dict) -> dict:
    return {k: bits(v) for k, v in inp.items()}
