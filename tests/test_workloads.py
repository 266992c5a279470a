"""The synthetic workloads carry the structural constants printed on the pages."""
import json
import os

import numpy as np
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
