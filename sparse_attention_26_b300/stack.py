"""The attention layers of a DeepSeek-V4 model in decode, through the C ABI.

"DeepSeek-V4" atlas spec sheet, "Design overview" and "Core block": the first
two layers are pure sliding-window (window 128); the remaining layers
interleave CSA (4:1 overlapping compression, lightning-indexer top-k) and HCA
(128:1 compression, dense attention).  Here every layer keeps the 128-token
window beside its compressed branch, so the layer kinds are

    swa: SWA only;  csa: CSA + SWA;  hca: HCA + SWA,

and each runs as one fused attention (hattn_hybrid_attn with the matching
segment mask) followed by the sink merge with inverse RoPE.

A decode step appends one token per sequence to every layer.  A layer keeps
its raw tokens only in a ring of the last `ring` tokens (the 128-token window
and the 8- and 128-token compression windows all fit in 256), and its
compressed caches in full: a CSA entry is compressed when the token that
completes it arrives (every 4th token), an HCA entry every 128th.  This module
sequences the calls and owns the buffers; every step of the computation runs
in libhattn's kernels (the append of a token's rows into the rings is a
device-to-device copy).
"""
from __future__ import annotations

import torch

from . import hattn

SWA, CSA, HCA = "swa", "csa", "hca"


def layer_pattern(n_layers: int, n_swa: int = 2) -> list:
    """The first n_swa layers sliding-window only, then CSA and HCA alternating."""
    return [SWA] * min(n_swa, n_layers) + [CSA if i % 2 == 0 else HCA
                                           for i in range(max(0, n_layers - n_swa))]


class DecodeStack:
    """Caches and step buffers of the attention layers of one model.

    shape: B sequences, H heads of dim D (RoPE on the last r), an HI x dI
    indexer with top-k, window W, compression (m_csa, w_csa) and m_hca, room
    for contexts up to L_max tokens.  Token rows of layer l live in
    kv_ring[l] [B][ring][D] (and ik_ring, gate rings for its compressor)."""

    def __init__(self, kinds, *, B, H, D, r, HI, dI, k, L_max, W=128, m_csa=4, w_csa=8,
                 m_hca=128, ring=256, device="cuda", eps=1e-6):
        if ring & (ring - 1) or ring < max(W, w_csa, m_hca):
            raise ValueError("ring must be a power of two holding the window and both "
                             "compression windows")
        self.kinds = list(kinds)
        self.B, self.H, self.D, self.r = B, H, D, r
        self.HI, self.dI, self.k, self.W = HI, dI, k, W
        self.m_csa, self.w_csa, self.m_hca = m_csa, w_csa, m_hca
        self.ring, self.L_max, self.dev, self.eps = ring, L_max, device, eps
        self.N_csa = L_max // m_csa
        self.N_hca = max(1, L_max // m_hca)
        bf = torch.bfloat16
        self.layers = []
        for kind in self.kinds:
            st = {"kind": kind,
                  "kv_ring": torch.zeros((B, ring, D), dtype=bf, device=device)}
            if kind == CSA:
                st["ik_ring"] = torch.zeros((B, ring, dI), dtype=bf, device=device)
                st["gate_ring"] = torch.zeros((B, ring), dtype=bf, device=device)
                st["kv_c"] = torch.zeros((B, self.N_csa, D), dtype=bf, device=device)
                st["ik_c"] = torch.zeros((B, self.N_csa, dI), dtype=bf, device=device)
            elif kind == HCA:
                st["gate_ring"] = torch.zeros((B, ring), dtype=bf, device=device)
                st["kv_h"] = torch.zeros((B, self.N_hca, D), dtype=bf, device=device)
            self.layers.append(st)
        T = 1
        self.qt = torch.empty((B, T, H, D), dtype=bf, device=device)
        self.kv_w = torch.empty((B, T, W, D), dtype=bf, device=device)
        self.scores = torch.empty((B, T, self.N_csa), dtype=torch.float32, device=device)
        self.idx = torch.empty((B, T, k), dtype=torch.int32, device=device)
        ws = hattn.indexer_topk_workspace_bytes(B, T, self.N_csa, k, True)
        self.ws_topk = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        self.topk_launches = hattn.topk_launches(B, T, self.N_csa, k)
        self.out = torch.empty((len(self.kinds), B, T, H, D), dtype=bf, device=device)
        self.lse = torch.empty((len(self.kinds), B, T, H), dtype=torch.float32, device=device)
        self.ws = {}
        for kind in set(self.kinds):
            need = hattn.hybrid_attn_workspace_bytes(B, T, H, D, k, self.N_hca, W, q_prepped=True,
                                                     partials=True, segments=self.segments(kind))
            self.ws[kind] = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.dependent_launch = True

    @staticmethod
    def segments(kind):
        return {SWA: hattn.SEG_SWA, CSA: hattn.SEG_CSA | hattn.SEG_SWA,
                HCA: hattn.SEG_HCA | hattn.SEG_SWA}[kind]

    # ------------------------------------------------------------ cache setup
    def prefill(self, l, kv_raw, ik_raw=None, gate=None, n_tokens=None):
        """Layer l from full raw token rows [B][L0][...] (the prompt): compress
        every entry the L0 tokens complete, and keep the last `ring` tokens."""
        st, r = self.layers[l], self.r
        L0 = kv_raw.shape[1] if n_tokens is None else n_tokens
        if st["kind"] == CSA and L0 // self.m_csa > 0:
            hattn.csa_compress(kv_raw, ik_raw, gate, r=r, j_begin=0, j_end=L0 // self.m_csa,
                               m=self.m_csa, w=self.w_csa, kv_c=st["kv_c"], ik_c=st["ik_c"],
                               eps=self.eps)
        elif st["kind"] == HCA and L0 // self.m_hca > 0:
            hattn.hca_compress(kv_raw, gate, r=r, j_begin=0, j_end=L0 // self.m_hca,
                               m=self.m_hca, kv_h=st["kv_h"], eps=self.eps)
        u0 = max(0, L0 - self.ring)
        slots = torch.arange(u0, L0, device=kv_raw.device) % self.ring
        st["kv_ring"][:, slots] = kv_raw[:, u0:L0]
        if "ik_ring" in st and ik_raw is not None:
            st["ik_ring"][:, slots] = ik_raw[:, u0:L0]
        if "gate_ring" in st and gate is not None:
            st["gate_ring"][:, slots] = gate[:, u0:L0]

    def fill_random(self, l, seed):
        """Layer l's caches and ring drawn directly as seeded N(0,1) bf16
        (a stand-in for a built context, for timing: the kernels' work does
        not depend on the values)."""
        st = self.layers[l]
        g = torch.Generator(device=self.dev)
        g.manual_seed(int(seed))
        for name in ("kv_ring", "ik_ring", "gate_ring", "kv_c", "ik_c", "kv_h"):
            if name in st:
                t = st[name]
                for c in range(0, t.shape[1], 16384):  # chunks keep the fp32 temporary small
                    blk = t[:, c:c + 16384]
                    blk.copy_(torch.randn(blk.shape, generator=g, device=self.dev))

    def _put(self, st, u, kv, ik, gate):
        slot = u % self.ring
        st["kv_ring"][:, slot].copy_(kv)
        if "ik_ring" in st and ik is not None:
            st["ik_ring"][:, slot].copy_(ik)
        if "gate_ring" in st and gate is not None:
            st["gate_ring"][:, slot].copy_(gate)

    # ------------------------------------------------------------ one step
    def append(self, l, t, kv, ik=None, gate=None):
        """Token t's rows of layer l ([B][D], [B][dI], [B]) into its ring."""
        self._put(self.layers[l], t, kv, ik, gate)

    def step(self, t, q, iq, w, sinks, pos):
        """Attention of every layer for the query at position t (its token
        already appended): q [L][B][1][H][D], iq [L][B][1][HI][dI],
        w [L][B][1][HI], sinks [L][H], pos [B][1] (all t).  Outputs land in
        self.out[l], self.lse[l]."""
        for l, st in enumerate(self.layers):
            self._layer(l, st, t, q[l], iq[l], w[l], sinks[l], pos)

    def _layer(self, l, st, t, q, iq, w, sink, pos):
        r, kind = self.r, st["kind"]
        dep = self.dependent_launch
        # Launch order keeps every dependent launch after a kernel it may
        # overlap: compress (plain) -> indexer, top-k (dependent) -> query
        # prep, window keys (plain) -> attention, merge (dependent).
        if kind == CSA:
            if (t + 1) % self.m_csa == 0:
                j = (t + 1) // self.m_csa - 1
                hattn.csa_compress_ring(st["kv_ring"], st["ik_ring"], st["gate_ring"], r=r,
                                        j_begin=j, j_end=j + 1, kv_c=st["kv_c"], ik_c=st["ik_c"],
                                        m=self.m_csa, w=self.w_csa, eps=self.eps)
            fresh = (t + 1) // self.m_csa - 1 if (t + 1) % self.m_csa == 0 else -1
            hattn.indexer_topk(iq, w, st["ik_c"], pos, k=self.k, m=self.m_csa, idx_out=self.idx,
                               score_out=self.scores, workspace=self.ws_topk, fresh_from=fresh,
                               dependent=dep)
        elif kind == HCA and (t + 1) % self.m_hca == 0:
            j = (t + 1) // self.m_hca - 1
            hattn.hca_compress_ring(st["kv_ring"], st["gate_ring"], r=r, j_begin=j, j_end=j + 1,
                                    kv_h=st["kv_h"], m=self.m_hca, eps=self.eps)
        hattn.query_prep(q, pos, r=r, q_out=self.qt, eps=self.eps)
        hattn.swa_keys_ring(st["kv_ring"], pos, r=r, W=self.W, kv_w=self.kv_w, eps=self.eps)
        part = hattn.hybrid_attn(self.qt, st.get("kv_c"), self.idx if kind == CSA else None,
                                 st.get("kv_h"), self.kv_w, pos, r=r, m=self.m_hca, k=self.k,
                                 W=self.W, eps=self.eps, workspace=self.ws[kind], q_prepped=True,
                                 partials=True, segments=self.segments(kind), dependent=dep)
        hattn.lse_merge_splits([part], pos, r=r, H=self.H, sink=sink, out=self.out[l],
                               lse_out=self.lse[l], dependent=dep)

    def launches_per_step(self, t):
        """Kernels one step at position t launches."""
        n = 0
        for st in self.layers:
            n += 4  # query prep, window keys, attention, merge
            if st["kind"] == CSA:
                n += 1 + self.topk_launches + int((t + 1) % self.m_csa == 0)
            elif st["kind"] == HCA:
                n += int((t + 1) % self.m_hca == 0)
        return n
