"""One hybrid attention layer (CSA + HCA + SWA, sink merge) driven through the
C ABI.  This module only sequences the calls and owns the device buffers
(caches, workspaces, outputs); every step of the computation runs in
libhattn's kernels.

Decode step at query position t (its own token already written to the raw
cache), for every sequence of the batch:
  1. csa_compress / hca_compress of the entry that the token at t completes
     (when (t+1) is a multiple of m), so the caches are current;
  2. query preparation (RMSNorm + RoPE), shared by the three branches;
  3. indexer scores over the visible CSA entries, then top-k selection;
  4. sparse attention over the selected entries, dense attention over the
     visible HCA entries, sliding-window attention over the last W tokens
     (HCA and SWA optionally on a second stream, concurrent with 3);
  5. sink-augmented LSE merge of the three branches with inverse RoPE.

When a layer runs all three branches with one query per row block, steps 4
and 5 can also run fused: the window tokens are normalised and roped once
(hattn_swa_keys, on the second stream with the HCA compression), then one
attention covers the selected CSA entries, the HCA entries and the window
under a single softmax, and the merge adds the sink and inverse RoPE.
"""
from __future__ import annotations

import torch

from . import hattn


class HybridLayer:
    def __init__(self, wl, raw: dict, device="cuda", build_caches=True):
        self.wl = wl
        self.dev = device
        self.raw = raw  # kv_raw, ik_raw, gate_csa, gate_hca on device
        B, L, D = raw["kv_raw"].shape
        self.B, self.L, self.D = B, L, D
        self.N_csa = L // wl.m_csa
        self.N_hca = max(1, L // wl.m_hca)
        bf = torch.bfloat16
        # only the caches of the branches this layer runs
        n_c = self.N_csa if "csa" in wl.branches else 1
        n_h = self.N_hca if "hca" in wl.branches else 1
        self.kv_c = torch.zeros((B, n_c, D), dtype=bf, device=device)
        self.ik_c = torch.zeros((B, n_c, wl.dI), dtype=bf, device=device)
        self.kv_h = torch.zeros((B, n_h, D), dtype=bf, device=device)
        if build_caches:
            self.build_caches()
        self._bufs = {}

    def build_caches(self, n_tokens=None):
        """Compress every complete entry of the raw caches (cache build)."""
        wl, r = self.wl, self.raw
        L = self.L if n_tokens is None else n_tokens
        if "csa" in wl.branches:
            hattn.csa_compress(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=0,
                               j_end=L // wl.m_csa, m=wl.m_csa, w=wl.w_csa, kv_c=self.kv_c,
                               ik_c=self.ik_c)
        if "hca" in wl.branches and L // wl.m_hca > 0:
            hattn.hca_compress(r["kv_raw"], r["gate_hca"], r=wl.r, j_begin=0, j_end=L // wl.m_hca,
                               m=wl.m_hca, kv_h=self.kv_h)

    def buffers(self, T):
        """Outputs and workspaces for T queries per sequence (allocated once)."""
        if T in self._bufs:
            return self._bufs[T]
        wl, B, D, dev = self.wl, self.B, self.D, self.dev
        H = wl.H
        bf = torch.bfloat16
        b = dict(
            scores=torch.empty((B, T, self.N_csa if "csa" in wl.branches else 1),
                               dtype=torch.float32, device=dev),
            idx=torch.empty((B, T, wl.k), dtype=torch.int32, device=dev),
            out=torch.empty((B, T, H, D), dtype=bf, device=dev),
            lse=torch.empty((B, T, H), dtype=torch.float32, device=dev),
        )
        b["qt"] = torch.empty((B, T, H, D), dtype=bf, device=dev)  # prepared queries
        if self.can_fuse(T):
            b["kv_w"] = torch.empty((B, T, wl.W, D), dtype=bf, device=dev)  # SWA keys
            ws = hattn.hybrid_attn_workspace_bytes(B, T, H, D, wl.k, self.N_hca, wl.W,
                                                   q_prepped=True, partials=True)
            b["ws_fused"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        for name, kind, nk in self._branch_kinds():
            b["o_" + name] = torch.empty((B, T, H, D), dtype=torch.float32, device=dev)
            b["l_" + name] = torch.empty((B, T, H), dtype=torch.float32, device=dev)
            ws = max(hattn.attn_workspace_bytes(kind, B, T, H, D, nk, q_prepped=True),
                     hattn.attn_workspace_bytes(kind, B, T, H, D, nk, q_prepped=True,
                                                partials=True))
            b["ws_" + name] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self._bufs[T] = b
        return b

    def can_fuse(self, T):
        """The fused attention serves layers with all three branches, one query
        per row block (H = 128, or single-token decode) and a window buffer
        of at most 256 MB."""
        wl = self.wl
        return (set(wl.branches) == {"csa", "hca", "swa"} and (wl.H == 128 or T == 1)
                and self.B * T * wl.W * self.D * 2 <= (256 << 20))

    def _branch_kinds(self):
        wl = self.wl
        return [(n, k, nk) for n, k, nk in [("csa", hattn.KIND_SPARSE, wl.k),
                                            ("hca", hattn.KIND_HCA, self.N_hca),
                                            ("swa", hattn.KIND_SWA, wl.W)]
                if n in wl.branches]

    def step(self, q, iq, w, pos, sink, t_new=None, events=None, side_stream=None,
             branch_outputs=False, fused=None):
        """One pass of the hot path for queries q [B,T,H,D] at positions pos.

        t_new: position of the newest token (compresses the entries it
        completes); None skips the incremental compression.  events: optional
        dict name -> (start, end) torch.cuda.Event pairs recorded around the
        calls.  side_stream: a second CUDA stream; when given, the HCA and
        SWA branches run on it, concurrently with the indexer, top-k and CSA
        branch, joined before the merge.  branch_outputs: combine each
        branch's key splits into its own (o, lse) (kept in the buffers) and
        merge those; by default the branches leave their split partials and
        one merge weighs all of them.  fused: run the three branches as one
        attention (default: whenever can_fuse and no branch outputs are
        asked for).  Returns (out bf16 [B,T,H,D], lse fp32 [B,T,H])."""
        wl, r = self.wl, self.raw
        B, T = q.shape[0], q.shape[1]
        b = self.buffers(T)
        main = torch.cuda.current_stream()
        if fused is None:
            fused = self.can_fuse(T) and not branch_outputs
        if fused:
            return self._step_fused(q, iq, w, pos, sink, t_new, events, side_stream)

        def ev(name, i):
            if events is not None and name in events:
                events[name][i].record(torch.cuda.current_stream())

        def compress(kind):
            if t_new is None or kind not in wl.branches:
                return
            m, w_ = (wl.m_csa, wl.w_csa) if kind == "csa" else (wl.m_hca, wl.m_hca)
            if (t_new + 1) % m:
                return
            j = (t_new + 1) // m - 1
            if kind == "csa":
                hattn.csa_compress(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=j,
                                   j_end=j + 1, m=m, w=w_, kv_c=self.kv_c, ik_c=self.ik_c)
            else:
                hattn.hca_compress(r["kv_raw"], r["gate_hca"], r=wl.r, j_begin=j, j_end=j + 1,
                                   m=m, kv_h=self.kv_h)

        ev("compress", 0)
        compress("csa")
        if side_stream is None:
            compress("hca")
        ev("compress", 1)
        ev("qprep", 0)
        hattn.query_prep(q, pos, r=wl.r, q_out=b["qt"])
        ev("qprep", 1)
        qt = b["qt"]
        parts = {}

        def outs(name):
            if branch_outputs:
                return dict(o=b["o_" + name], lse=b["l_" + name])
            return dict(partials=True)

        def dense_branches():
            if "hca" in wl.branches:
                ev("hca", 0)
                parts["hca"] = hattn.hca_attn(qt, self.kv_h, pos, r=wl.r, m=wl.m_hca,
                                              workspace=b["ws_hca"], q_prepped=True,
                                              **outs("hca"))
                ev("hca", 1)
            if "swa" in wl.branches:
                ev("swa", 0)
                parts["swa"] = hattn.swa_attn(qt, r["kv_raw"], pos, r=wl.r, W=wl.W,
                                              workspace=b["ws_swa"], q_prepped=True,
                                              **outs("swa"))
                ev("swa", 1)

        joined = None
        if side_stream is not None:
            side_stream.wait_stream(main)
            with torch.cuda.stream(side_stream):
                compress("hca")
                dense_branches()
            joined = side_stream
        if "csa" in wl.branches:
            ev("indexer", 0)
            hattn.indexer_scores(iq, w, self.ik_c, pos, m=wl.m_csa, score_out=b["scores"])
            ev("indexer", 1)
            ev("topk", 0)
            hattn.topk_select(b["scores"], pos, k=wl.k, m=wl.m_csa, idx_out=b["idx"])
            ev("topk", 1)
            ev("sparse", 0)
            parts["csa"] = hattn.sparse_attn(qt, self.kv_c, b["idx"], pos, r=wl.r,
                                             workspace=b["ws_csa"], q_prepped=True,
                                             **outs("csa"))
            ev("sparse", 1)
        if joined is None:
            dense_branches()
        else:
            main.wait_stream(joined)
        ev("merge", 0)
        if branch_outputs:
            o_list = [b["o_" + n] for n, _, _ in self._branch_kinds()]
            l_list = [b["l_" + n] for n, _, _ in self._branch_kinds()]
            hattn.lse_merge(o_list, l_list, pos, r=wl.r, sink=sink, out=b["out"],
                            lse_out=b["lse"])
        else:
            hattn.lse_merge_splits([parts[n] for n, _, _ in self._branch_kinds()], pos, r=wl.r,
                                   H=wl.H, sink=sink, out=b["out"], lse_out=b["lse"])
        ev("merge", 1)
        return b["out"], b["lse"]

    def _step_fused(self, q, iq, w, pos, sink, t_new, events, side_stream):
        wl, r = self.wl, self.raw
        T = q.shape[1]
        b = self.buffers(T)
        main = torch.cuda.current_stream()

        def ev(name, i):
            if events is not None and name in events:
                events[name][i].record(torch.cuda.current_stream())

        def compress(kind):
            if t_new is None:
                return
            m = wl.m_csa if kind == "csa" else wl.m_hca
            if (t_new + 1) % m:
                return
            j = (t_new + 1) // m - 1
            if kind == "csa":
                hattn.csa_compress(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=j,
                                   j_end=j + 1, m=m, w=wl.w_csa, kv_c=self.kv_c, ik_c=self.ik_c)
            else:
                hattn.hca_compress(r["kv_raw"], r["gate_hca"], r=wl.r, j_begin=j, j_end=j + 1,
                                   m=m, kv_h=self.kv_h)

        def side_work():
            compress("hca")
            ev("swa_keys", 0)
            hattn.swa_keys(r["kv_raw"], pos, r=wl.r, W=wl.W, kv_w=b["kv_w"])
            ev("swa_keys", 1)

        ev("compress", 0)
        compress("csa")
        if side_stream is None:
            side_work()
        ev("compress", 1)
        joined = None
        if side_stream is not None:
            side_stream.wait_stream(main)
            with torch.cuda.stream(side_stream):
                side_work()
            joined = side_stream
        ev("qprep", 0)
        hattn.query_prep(q, pos, r=wl.r, q_out=b["qt"])
        ev("qprep", 1)
        ev("indexer", 0)
        hattn.indexer_scores(iq, w, self.ik_c, pos, m=wl.m_csa, score_out=b["scores"])
        ev("indexer", 1)
        ev("topk", 0)
        hattn.topk_select(b["scores"], pos, k=wl.k, m=wl.m_csa, idx_out=b["idx"])
        ev("topk", 1)
        if joined is not None:
            main.wait_stream(joined)
        ev("attn", 0)
        part = hattn.hybrid_attn(b["qt"], self.kv_c, b["idx"], self.kv_h, b["kv_w"], pos, r=wl.r,
                                 m=wl.m_hca, workspace=b["ws_fused"], q_prepped=True,
                                 partials=True)
        ev("attn", 1)
        ev("merge", 0)
        hattn.lse_merge_splits([part], pos, r=wl.r, H=wl.H, sink=sink, out=b["out"],
                               lse_out=b["lse"])
        ev("merge", 1)
        return b["out"], b["lse"]

    def event_names(self, T, branch_outputs=False, fused=None):
        """The call spans step() records when given events of these names."""
        if fused is None:
            fused = self.can_fuse(T) and not branch_outputs
        if fused:
            return ["compress", "swa_keys", "qprep", "indexer", "topk", "attn", "merge"]
        return ["compress", "qprep", "indexer", "topk", "sparse", "hca", "swa", "merge"]

    def launches_per_step(self, T, t_new=None, branch_outputs=False, fused=None):
        """Kernels one step launches: the query preparation, each branch's
        attention kernel (plus its combine with split-KV when branch outputs
        are formed), the indexer and top-k of CSA, the merge, and the
        compressions the new token needs."""
        wl, B, D, H = self.wl, self.B, self.D, self.wl.H
        n = 2  # query preparation, merge
        if t_new is not None:
            n += int("csa" in wl.branches and (t_new + 1) % wl.m_csa == 0)
            n += int("hca" in wl.branches and (t_new + 1) % wl.m_hca == 0)
        if fused is None:
            fused = self.can_fuse(T) and not branch_outputs
        if fused:
            return n + 4  # SWA keys, indexer scores, top-k, fused attention
        for name, kind, nk in self._branch_kinds():
            n += 1 + int(branch_outputs and hattn.attn_splits(kind, B, T, H, D, nk) > 1)
            if name == "csa":
                n += 2  # indexer scores + top-k select
        return n
