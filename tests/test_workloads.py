"""The synthetic workloads carry the structural constants printed on the
pages, and the layer and stack plan their steps (entries completed, launch
counts, fused or branch attention) as the recorded runs did: host logic,
checked on meta tensors without a device."""
import json
import os

import numpy as np
import pytest
import torch

from sparse_attention_26_b300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_constants.json")))


def v(key):
    return GOLD[key]["value"]


def test_workloads_match_page_constants():
    W = synth.WORKLOADS
    for wl in W.values():
        assert wl.m_csa == v("csa_m") and wl.m_hca == v("hca_ratio") and wl.W == v("swa_window")
    for name in ["pro_csa_decode", "hybrid_decode_1m", "hca_decode", "hca_prefill"]:
        assert W[name].H == v("heads_pro") and W[name].D == v("head_dim")
        assert W[name].r == v("rope_dims")
    assert W["flash_csa_prefill"].H == v("heads_flash") and W["flash_csa_prefill"].k == v(
        "csa_topk_flash")
    assert W["hybrid_decode_1m"].k == v("csa_topk_pro") and W["hybrid_decode_1m"].L == v(
        "context")
    assert W["hybrid_decode_1m"].n_csa == 262144 and W["hybrid_decode_1m"].n_hca == 8192


def test_generator_is_seeded_and_deterministic():
    wl = synth.scaled(synth.WORKLOADS["hybrid_decode_1m"], B=2, L=512, T=1)
    a = synth.make_inputs(wl, 0)
    b = synth.make_inputs(wl, 0)
    c = synth.make_inputs(wl, 1)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["kv_raw"], c["kv_raw"])
    assert a["q"].dtype == torch.bfloat16 and a["w"].dtype == torch.float32
    assert a["pos"].tolist() == [[511], [511]]
    # N(0,1) moments
    x = a["kv_raw"].float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1) < 0.02


def test_random_idx_distinct():
    idx = synth.random_idx(2, 3, 16, np.array([[5, 40, 100], [0, 16, 17]]), seed=3).numpy()
    for b in range(2):
        for t in range(3):
            row = idx[b, t]
            vals = row[row >= 0]
            assert len(set(vals.tolist())) == len(vals)
    assert (idx[1, 0] == -1).all() and (idx[0, 0, 5:] == -1).all()


def test_layer_pattern_of_the_pages():
    """Two sliding-window layers, then CSA and HCA alternating: V4-Pro's 61
    layers are 2 + 30 + 29, V4-Flash's 43 are 2 + 21 + 20."""
    from sparse_attention_26_b300.stack import CSA, HCA, SWA, layer_pattern
    pro = layer_pattern(61)
    assert pro[:2] == [SWA, SWA] and pro[2:6] == [CSA, HCA, CSA, HCA]
    assert (pro.count(SWA), pro.count(CSA), pro.count(HCA)) == (2, 30, 29)
    flash = layer_pattern(43)
    assert (flash.count(SWA), flash.count(CSA), flash.count(HCA)) == (2, 21, 20)
    assert layer_pattern(1) == [SWA]


def test_new_entries_of_a_step():
    """The entries a step's new tokens complete: entry j is complete once the
    token at m(j+1)-1 is cached."""
    from sparse_attention_26_b300.layer import HybridLayer

    class Shapes(HybridLayer):
        def __init__(self, wl):
            self.wl = wl

    layer = Shapes(synth.WORKLOADS["hybrid_decode_1m"])
    assert layer.new_entries("csa", 7, 1) == (1, 2)      # token 7 completes entry 1
    assert layer.new_entries("csa", 8, 1) == (2, 2)      # token 8 completes nothing
    assert layer.new_entries("csa", 11, 8) == (1, 3)     # tokens 4..11: entries 1 and 2
    assert layer.new_entries("hca", 255, 2) == (1, 2)    # tokens 254, 255: HCA entry 1
    assert layer.new_entries("hca", 257, 2) == (2, 2)      # tokens 256, 257: none
    L = 1 << 20
    assert layer.new_entries("csa", L - 1, 2) == (L // 4 - 1, L // 4)
    assert layer.new_entries("csa", None, 1) == (0, 0)
    # brute force against the definition
    for m in (4, 128):
        kind = "csa" if m == 4 else "hca"
        for t in range(0, 600, 7):
            for n in (1, 2, 5):
                done = [j for j in range(t // m + 2) if t - n + 1 <= m * (j + 1) - 1 <= t]
                j0, j1 = layer.new_entries(kind, t, n)
                assert list(range(j0, j1)) == done, (kind, t, n)


def _meta_layer(name):
    """A layer of the workload's shapes whose buffers are meta tensors (no
    memory, no device): enough for its host-side step planning."""
    from sparse_attention_26_b300.layer import HybridLayer
    wl = synth.WORKLOADS[name]
    raw = {"kv_raw": torch.empty((wl.B, wl.L, wl.D), dtype=torch.bfloat16, device="meta")}
    return wl, HybridLayer(wl, raw, device="meta", build_caches=False)


def test_launch_counts_match_the_recorded_launch_lists():
    """The kernels one decode step launches, as the bench counts them for
    gpu_launches, equal the ncu launch lists of the same steps (80 launches
    over 10 steps in profiles/launches_hybrid_decode_1m.md and
    profiles/launches_hybrid_decode_1m_mtp2.md): two compressions, window
    keys, query prep, the indexer, the top-k kernel (a cluster of CTAs per
    row of 262,144 scores), the fused attention and the merge."""
    for name, T in (("hybrid_decode_1m", 1), ("hybrid_decode_1m_mtp2", 2)):
        wl, layer = _meta_layer(name)
        n = layer.launches_per_step(T, wl.L - 1, side_stream=True)
        assert n == 80 // 10 == 8, (name, n)
        assert len(layer.event_names(T)) == 7  # one span covers both compressions
    # a step whose token completes no entry skips both compressions
    wl, layer = _meta_layer("hybrid_decode_1m")
    assert layer.launches_per_step(1, wl.L - 2, side_stream=True) == 6


def test_stack_launch_count_at_1m():
    """The 61-layer decode step at t = 2^20 - 1 launches 363 kernels: every
    layer query prep, window keys, attention and merge; a CSA layer adds the
    indexer, the top-k kernel and its new entry's compression, an HCA layer
    its new entry's compression (t + 1 is a multiple of 4 and of 128)."""
    from sparse_attention_26_b300.stack import DecodeStack, layer_pattern
    wl = synth.WORKLOADS["hybrid_decode_1m"]
    st = DecodeStack(layer_pattern(61), B=wl.B, H=wl.H, D=wl.D, r=wl.r, HI=wl.HI, dI=wl.dI,
                     k=wl.k, L_max=wl.L, device="meta")
    assert st.launches_per_step(wl.L - 1) == 2 * 4 + 30 * 7 + 29 * 5 == 363
    assert st.launches_per_step(wl.L - 2) == 2 * 4 + 30 * 6 + 29 * 4


def test_which_steps_take_the_fused_attention():
    """Every configured workload takes the fused attention: decode steps of
    any branch subset, the H = 128 HCA prefill, and the CSA prefill (its
    sparse branch runs one query per row block anyway; the 1 GB window
    buffer fits the 2 GB bound).  The prefills' queries each take one key
    split, so the attention writes the layer output and no merge follows;
    the decode steps split each query's keys and merge.  The segment mask
    names the branches."""
    from sparse_attention_26_b300 import hattn
    want = {"hybrid_decode_1m": (True, False), "hybrid_decode_1m_mtp2": (True, False),
            "pro_csa_decode": (True, False), "hca_decode": (True, False),
            "hca_prefill": (True, True), "flash_csa_prefill": (True, True)}
    seg = {"csa": hattn.SEG_CSA, "hca": hattn.SEG_HCA, "swa": hattn.SEG_SWA}
    for name, (fused, final) in want.items():
        wl, layer = _meta_layer(name)
        assert layer.can_fuse(wl.T) == fused, name
        assert layer.fused_final(wl.T) == final, name
        assert layer.segments() == sum(seg[b] for b in wl.branches), name
        names = layer.event_names(wl.T)
        assert ("attn_fused" in names) == fused, (name, names)
        assert ("merge" in names) == (not final), (name, names)
        assert ("indexer" in names) == ("csa" in wl.branches), (name, names)


def test_stack_ring_must_hold_every_window():
    from sparse_attention_26_b300.stack import DecodeStack, layer_pattern
    kw = dict(B=1, H=128, D=512, r=64, HI=64, dI=128, k=1024, L_max=4096, device="meta")
    for ring in (192, 64):   # not a power of two; smaller than the HCA window
        with pytest.raises(ValueError, match="ring"):
            DecodeStack(layer_pattern(4), ring=ring, **kw)
    assert DecodeStack(layer_pattern(4), ring=128, **kw).ring == 128
