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
    def __init__(self, wl, raw: dict, device="cuda", build_caches=True, indexer_keys="bf16"):
        """indexer_keys: "bf16"; "fp8" to keep the indexer keys as E4M3 codes
        with a row scale (ik8, ik_scale) and score them on the FP8
        tensor-core path; or "mxfp4" to keep them as MXFP4 codes and block
        scales (ik4, ik4_scale, quantised from the bf16 keys as each entry is
        compressed) and score them from those."""
        if indexer_keys not in ("bf16", "fp8", "mxfp4"):
            raise ValueError(f"indexer_keys must be 'bf16', 'fp8' or 'mxfp4', "
                             f"got {indexer_keys!r}")
        self.wl = wl
        self.dev = device
        self.raw = raw  # kv_raw, ik_raw, gate_csa, gate_hca on device
        self.fp8 = indexer_keys == "fp8"
        self.mx4 = indexer_keys == "mxfp4"
        B, L, D = raw["kv_raw"].shape
        self.B, self.L, self.D = B, L, D
        self.N_csa = L // wl.m_csa
        self.N_hca = max(1, L // wl.m_hca)
        bf = torch.bfloat16
        # only the caches of the branches this layer runs
        n_c = self.N_csa if "csa" in wl.branches else 1
        n_h = self.N_hca if "hca" in wl.branches else 1
        self.kv_c = torch.zeros((B, n_c, D), dtype=bf, device=device)
        self.ik_c = torch.zeros((B, 1 if self.fp8 else n_c, wl.dI), dtype=bf, device=device)
        if self.fp8:
            self.ik8 = torch.zeros((B, n_c, wl.dI), dtype=torch.uint8, device=device)
            self.ik_scale = torch.zeros((B, n_c), dtype=torch.float32, device=device)
        if self.mx4:
            self.ik4 = torch.zeros((B, n_c, wl.dI // 2), dtype=torch.uint8, device=device)
            self.ik4_scale = torch.zeros((B, n_c, wl.dI // 32), dtype=torch.uint8, device=device)
        self.kv_h = torch.zeros((B, n_h, D), dtype=bf, device=device)
        self.override_dense_sms = 0  # > 0: HCA + SWA attention on that many SMs beside the indexer
        # fused step with a side stream: the indexer, top-k, attention and
        # merge start as dependent launches of their predecessors
        self.dependent_launch = True
        self._split_event = None  # marks the end of the score kernel in each step
        self._final = {}  # T -> the fused call writes the layer output itself
        if build_caches:
            self.build_caches()
        self._bufs = {}

    def build_caches(self, n_tokens=None):
        """Compress every complete entry of the raw caches (cache build)."""
        wl, r = self.wl, self.raw
        L = self.L if n_tokens is None else n_tokens
        if "csa" in wl.branches:
            self._csa_compress(0, L // wl.m_csa)
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
        # out and lse are adjacent in one buffer (one copy returns both)
        n_out, n_lse = B * T * H * D * 2, B * T * H * 4
        res = torch.empty(n_out + n_lse, dtype=torch.uint8, device=dev)
        n_sc = self.N_csa if "csa" in wl.branches else 1
        b = dict(
            scores=torch.empty((B, T, n_sc), dtype=torch.float32, device=dev),
            idx=torch.empty((B, T, wl.k), dtype=torch.int32, device=dev),
            ws_topk=torch.empty(max(hattn.indexer_topk_workspace_bytes(B, T, n_sc, wl.k, True),
                                    16), dtype=torch.uint8, device=dev),
            out=res[:n_out].view(bf).view(B, T, H, D),
            lse=res[n_out:].view(torch.float32).view(B, T, H),
            result=res,
        )
        b["qt"] = torch.empty((B, T, H, D), dtype=bf, device=dev)  # prepared queries
        if self.can_fuse(T):
            if "swa" in wl.branches:
                b["kv_w"] = torch.empty((B, T, wl.W, D), dtype=bf, device=dev)  # SWA keys
            for name, segs, n_sms in [("fused", self.segments(), 0),
                                      ("dense", hattn.SEG_HCA | hattn.SEG_SWA,
                                       self.override_dense_sms),
                                      ("sparse", hattn.SEG_CSA, 0)]:
                ws = hattn.hybrid_attn_workspace_bytes(B, T, H, D, wl.k, self.N_hca, wl.W,
                                                       q_prepped=True, partials=True,
                                                       segments=segs, n_sms=n_sms)
                b["ws_" + name] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        for name, kind, nk in self._branch_kinds():
            b["o_" + name] = torch.empty((B, T, H, D), dtype=torch.float32, device=dev)
            b["l_" + name] = torch.empty((B, T, H), dtype=torch.float32, device=dev)
            ws = max(hattn.attn_workspace_bytes(kind, B, T, H, D, nk, q_prepped=True),
                     hattn.attn_workspace_bytes(kind, B, T, H, D, nk, q_prepped=True,
                                                partials=True))
            b["ws_" + name] = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self._bufs[T] = b
        return b

    # SMs of this GPU and a cost model of the two concurrent chains (B300,
    # measured): a streamed 64-key tile of one output half costs ~2.25 us of
    # one SM, plus ~24 us for the HCA compression, the window keys and the
    # attention's own prologue/epilogue; the indexer streams at ~5.2 TB/s
    # when it has the SMs for it (~40 GB/s each: capped at 100 SMs it took
    # 138 us instead of 100), and top-k takes ~27 us.
    NUM_SMS = 148
    TILE_US, DENSE_FIXED_US, TOPK_US = 2.25, 24.0, 27.0
    IDX_BW, IDX_SM_BW = 5.2e12, 40e9

    def dense_sms(self, T):
        """A suggestion for override_dense_sms: the SMs to give the HCA + SWA
        attention while the indexer (on the rest) and top-k run, from the
        cost model -- the split that makes the two chains end together."""
        wl, B = self.wl, self.B
        # the attention's CTAs: nsplit key splits x 2 output halves x B*T queries
        per_split = 2 * B * T
        tiles = (self.N_hca + 63) // 64 + (wl.W + 63) // 64  # per query
        idx_bytes = B * T * (self.N_csa * (wl.dI * 2 + 4))
        best, best_t = per_split, None
        nsplit = 1
        while nsplit * per_split <= self.NUM_SMS - 32:
            x = nsplit * per_split
            dense = self.DENSE_FIXED_US + -(-tiles // nsplit) * self.TILE_US
            idx = idx_bytes / min(self.IDX_BW, (self.NUM_SMS - x) * self.IDX_SM_BW) * 1e6
            t = max(dense, idx + self.TOPK_US)
            if best_t is None or t < best_t:
                best, best_t = x, t
            nsplit += 1
        return best

    def result_buffer(self, T):
        """The one device buffer holding out (bf16) then lse (fp32) of step()."""
        return self.buffers(T)["result"]

    def segments(self):
        """The fused attention's segment mask for this layer's branches."""
        m = {"csa": hattn.SEG_CSA, "hca": hattn.SEG_HCA, "swa": hattn.SEG_SWA}
        seg = 0
        for name in self.wl.branches:
            seg |= m[name]
        return seg

    def can_fuse(self, T):
        """The fused attention serves one query per row block: it takes every
        step where that costs no MMA rows over the branch calls (H = 128,
        single-token decode, or a CSA layer, whose sparse branch runs one
        query per row block anyway), with a window buffer of at most 2 GB.
        In prefill that also removes the merge: one split per query, so the
        attention writes the layer output itself."""
        wl = self.wl
        fits = "swa" not in wl.branches or self.B * T * wl.W * self.D * 2 <= (2 << 30)
        return (wl.H == 128 or T == 1 or "csa" in wl.branches) and fits

    def fused_final(self, T):
        """Whether the fused call finalises the output itself (each query's
        keys in one split, so no merge follows)."""
        if T not in self._final:
            wl = self.wl
            self._final[T] = hattn.hybrid_attn_splits(self.B, T, wl.H, self.D, wl.k, self.N_hca,
                                                      wl.W, segments=self.segments()) == 1
        return self._final[T]

    def _branch_kinds(self):
        wl = self.wl
        return [(n, k, nk) for n, k, nk in [("csa", hattn.KIND_SPARSE, wl.k),
                                            ("hca", hattn.KIND_HCA, self.N_hca),
                                            ("swa", hattn.KIND_SWA, wl.W)]
                if n in wl.branches]

    def new_entries(self, kind, t_new, n_new=1):
        """[j0, j1): the entries of the CSA or HCA cache that the n_new tokens
        at positions t_new-n_new+1 .. t_new complete (entry j is complete once
        the token at m*(j+1)-1 is cached)."""
        if t_new is None:
            return 0, 0
        m = self.wl.m_csa if kind == "csa" else self.wl.m_hca
        j1 = (t_new + 1) // m
        return min(max(0, (t_new - n_new + 1) // m), j1), j1

    def _csa_compress(self, j0, j1):
        wl, r = self.wl, self.raw
        if self.fp8:
            hattn.csa_compress_fp8(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=j0,
                                   j_end=j1, m=wl.m_csa, w=wl.w_csa, kv_c=self.kv_c,
                                   ik8=self.ik8, ik_scale=self.ik_scale)
        elif self.mx4:
            # one launch: the entries and their MXFP4 indexer keys
            hattn.csa_compress_mxfp4(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=j0,
                                     j_end=j1, m=wl.m_csa, w=wl.w_csa, kv_c=self.kv_c,
                                     ik_c=self.ik_c, ik4=self.ik4, ik4_scale=self.ik4_scale)
        else:
            hattn.csa_compress(r["kv_raw"], r["ik_raw"], r["gate_csa"], r=wl.r, j_begin=j0,
                               j_end=j1, m=wl.m_csa, w=wl.w_csa, kv_c=self.kv_c, ik_c=self.ik_c)

    def _indexer_topk(self, iq, w, pos, b, events=None, n_sms=0, fresh_from=-1, dependent=False):
        """Indexer scores and top-k as one call (the score kernel counts the
        selection's first pass as it writes the scores).  Returns an event
        recorded between the two kernels, for other streams to wait on the
        scores alone.  With events, "indexer" spans the score kernel and
        "topk" the selection."""
        wl = self.wl
        cur = torch.cuda.current_stream()
        timed = events is not None and "indexer" in events
        if timed:
            events["indexer"][0].record(cur)
            split = events["indexer"][1]
            split.record(cur)  # creates its CUDA event; recorded again between the kernels
            events["topk"] = (split, events["topk"][1])
        else:
            if self._split_event is None:
                self._split_event = torch.cuda.Event()
                self._split_event.record(cur)  # creates its CUDA event
            split = self._split_event
        if self.mx4:
            hattn.indexer_topk_mxfp4(iq, w, self.ik4, self.ik4_scale, pos, k=wl.k, m=wl.m_csa,
                                     idx_out=b["idx"], score_out=b["scores"],
                                     workspace=b["ws_topk"], n_sms=n_sms, fresh_from=fresh_from,
                                     dependent=dependent, split_event=split,
                                     split_external=timed)
        else:
            keys = self.ik8 if self.fp8 else self.ik_c
            hattn.indexer_topk(iq, w, keys, pos, k=wl.k, m=wl.m_csa, idx_out=b["idx"],
                               score_out=b["scores"], workspace=b["ws_topk"],
                               ik_scale=self.ik_scale if self.fp8 else None, n_sms=n_sms,
                               fresh_from=fresh_from, dependent=dependent, split_event=split,
                               split_external=timed)
        if timed:
            events["topk"][1].record(cur)
        return split

    def _compress_new(self, kind, t_new, n_new):
        """Compress the entries that the step's new tokens complete."""
        wl, r = self.wl, self.raw
        j0, j1 = self.new_entries(kind, t_new, n_new)
        if j1 <= j0 or kind not in wl.branches:
            return
        if kind == "csa":
            self._csa_compress(j0, j1)
        else:
            hattn.hca_compress(r["kv_raw"], r["gate_hca"], r=wl.r, j_begin=j0, j_end=j1,
                               m=wl.m_hca, kv_h=self.kv_h)

    def step(self, q, iq, w, pos, sink, t_new=None, events=None, side_stream=None,
             branch_outputs=False, fused=None):
        """One pass of the hot path for queries q [B,T,H,D] at positions pos.

        t_new: position of the newest token; the T newest tokens (positions
        t_new-T+1 .. t_new, one per query) are new this step, and the entries
        they complete are compressed first.  None skips the incremental
        compression.  events: optional
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
            if kind in wl.branches:
                self._compress_new(kind, t_new, T)

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
            self._indexer_topk(iq, w, pos, b, events)
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
        """Fused step.  Without a side stream: one attention over all three key
        sets after top-k.  With one: the HCA + SWA key sets need no top-k, so
        their attention runs on the side stream on dense_sms() SMs while the
        indexer runs on the others; the CSA key set follows top-k, and one
        merge weighs the partials of both."""
        wl, r = self.wl, self.raw
        T = q.shape[1]
        b = self.buffers(T)
        main = torch.cuda.current_stream()

        def ev(name, i):
            if events is not None and name in events:
                events[name][i].record(torch.cuda.current_stream())

        def compress(kind):
            self._compress_new(kind, t_new, T)

        has = set(wl.branches)

        def attn(name, segments, n_sms, dependent=False):
            ev("attn_" + name, 0)
            part = hattn.hybrid_attn(b["qt"], self.kv_c if "csa" in has else None,
                                     b["idx"] if "csa" in has else None,
                                     self.kv_h if "hca" in has else None, b.get("kv_w"), pos,
                                     r=wl.r, m=wl.m_hca, k=wl.k, W=wl.W,
                                     workspace=b["ws_" + name], q_prepped=True, partials=True,
                                     segments=segments, n_sms=n_sms, dependent=dependent)
            ev("attn_" + name, 1)
            return part

        def swa_keys():
            if "swa" in has:
                ev("swa_keys", 0)
                hattn.swa_keys(r["kv_raw"], pos, r=wl.r, W=wl.W, kv_w=b["kv_w"])
                ev("swa_keys", 1)

        def qprep():
            ev("qprep", 0)
            hattn.query_prep(q, pos, r=wl.r, q_out=b["qt"])
            ev("qprep", 1)

        # Running the HCA + SWA key sets beside the indexer only pays when the
        # indexer still reaches full HBM bandwidth on the SMs left to it; on
        # B300 it needs all of them (capped at 100 SMs it runs ~40% longer),
        # so the split is opt-in (override_dense_sms) and the default runs the
        # three key sets as one attention after top-k.
        all_three = has == {"csa", "hca", "swa"}
        n_dense = self.override_dense_sms if (side_stream is not None and all_three) else 0
        overlap = n_dense > 0
        # dependent launches when the caller runs the step as the benchmark
        # does (with a side stream, without per-call events)
        pdl = side_stream is not None and self.dependent_launch and events is None
        if "csa" not in has:
            # no indexer to run beside: the layer's calls follow one another
            side_stream = None
        ev("compress", 0)
        compress("csa")
        if side_stream is None:
            compress("hca")
        ev("compress", 1)
        # from here on each main-stream call consumes what the one before it
        # produced, so its kernel may start as a dependent launch (its setup
        # overlaps the predecessor's tail; it waits before reading inputs)
        if side_stream is not None and overlap:
            qprep()
            side_stream.wait_stream(main)
            with torch.cuda.stream(side_stream):
                compress("hca")
                swa_keys()
                dense = attn("dense", hattn.SEG_HCA | hattn.SEG_SWA, n_dense)
        elif side_stream is None:
            qprep()
            swa_keys()
        scores_done = None
        if "csa" in has:
            # the entries the compression above writes are the newest ones
            j0, j1 = self.new_entries("csa", t_new, T)
            scores_done = self._indexer_topk(iq, w, pos, b, events,
                                             n_sms=(self.NUM_SMS - n_dense) if n_dense else 0,
                                             fresh_from=j0 if j1 > j0 else -1, dependent=pdl)
        if side_stream is not None and not overlap:
            # The query preparation, the HCA compression and the window keys
            # (needed only by the attention) run beside top-k, which leaves
            # SMs free.  Beside the indexer they would hold SMs its
            # persistent grid needs from the start, and its statically split
            # work would end later by as much.  (With per-call events they
            # follow the whole call.)
            if scores_done is not None and (events is None or "indexer" not in events):
                side_stream.wait_event(scores_done)
            else:
                side_stream.wait_stream(main)
            with torch.cuda.stream(side_stream):
                qprep()
                compress("hca")
                swa_keys()
        if overlap:
            parts = [attn("sparse", hattn.SEG_CSA, 0, dependent=pdl)]
            main.wait_stream(side_stream)
            parts.append(dense)
        else:
            if side_stream is not None:
                main.wait_stream(side_stream)
            if self.fused_final(T):
                # one split per query: the attention applies the sink merge
                # and the inverse RoPE itself
                ev("attn_fused", 0)
                hattn.hybrid_attn_out(b["qt"], self.kv_c if "csa" in has else None,
                                      b["idx"] if "csa" in has else None,
                                      self.kv_h if "hca" in has else None, b.get("kv_w"), pos,
                                      r=wl.r, m=wl.m_hca, k=wl.k, W=wl.W, sink=sink,
                                      out=b["out"], lse_out=b["lse"], workspace=b["ws_fused"],
                                      q_prepped=True, segments=self.segments(), dependent=pdl)
                ev("attn_fused", 1)
                return b["out"], b["lse"]
            parts = [attn("fused", self.segments(), 0, dependent=pdl)]
        ev("merge", 0)
        hattn.lse_merge_splits(parts, pos, r=wl.r, H=wl.H, sink=sink, out=b["out"],
                               lse_out=b["lse"], dependent=pdl)
        ev("merge", 1)
        return b["out"], b["lse"]

    def event_names(self, T, branch_outputs=False, fused=None, side_stream=True):
        """The call spans step() records when given events of these names."""
        if fused is None:
            fused = self.can_fuse(T) and not branch_outputs
        if fused:
            has = set(self.wl.branches)
            split = side_stream and self.override_dense_sms > 0 and has == {"csa", "hca", "swa"}
            attn = ["attn_dense", "attn_sparse"] if split else ["attn_fused"]
            names = ["compress"] + (["swa_keys"] if "swa" in has else []) + ["qprep"]
            names += ["indexer", "topk"] if "csa" in has else []
            merge = [] if (not split and self.fused_final(T)) else ["merge"]
            return names + attn + merge
        names = ["compress", "qprep"]
        if "csa" in self.wl.branches:
            names += ["indexer", "topk", "sparse"]
        names += [n for n in ("hca", "swa") if n in self.wl.branches]
        return names + ["merge"]

    def launches_per_step(self, T, t_new=None, branch_outputs=False, fused=None,
                          side_stream=False):
        """Kernels one step launches: the query preparation, each branch's
        attention kernel (plus its combine with split-KV when branch outputs
        are formed), the indexer and top-k of CSA, the merge, and the
        compressions the new token needs."""
        wl, B, D, H = self.wl, self.B, self.D, self.wl.H
        n = 2  # query preparation, merge
        for kind in ("csa", "hca"):
            j0, j1 = self.new_entries(kind, t_new, T)
            n += int(kind in wl.branches and j1 > j0)
        if fused is None:
            fused = self.can_fuse(T) and not branch_outputs
        if fused:
            # SWA keys, indexer scores, top-k, and the attention: one call, or
            # the dense and the sparse key sets when a side stream is used
            has = set(wl.branches)
            split = side_stream and self.override_dense_sms > 0 and has == {"csa", "hca", "swa"}
            topk = hattn.topk_launches(B, T, self.N_csa, wl.k) if "csa" in has else 0
            # (no merge when the attention writes the layer output itself)
            final = not split and self.fused_final(T)
            return n - int(final) + int("swa" in has) + int("csa" in has) + topk + 1 + int(split)
        for name, kind, nk in self._branch_kinds():
            n += 1 + int(branch_outputs and hattn.attn_splits(kind, B, T, H, D, nk) > 1)
            if name == "csa":
                n += 1 + hattn.topk_launches(B, T, self.N_csa, wl.k)  # indexer + top-k
        return n
