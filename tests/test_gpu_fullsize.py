"""GPU parity at the five workloads' full sizes, on sampled outputs.

Each test runs one pass of the layer exactly as the benchmark launches it
(HybridLayer.step over the whole batch), then checks sampled sequences and
queries stage by stage against the fp64 oracle.  To keep the oracle to
seconds, each downstream stage is fed the GPU's own upstream tensors (its
compressed caches and its top-k indices), and the compressor is checked on
sampled entries; near-tie swaps in top-k are decided by the tolerance rule,
not by the attention comparison.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_26_b300 import hattn, synth
from sparse_attention_26_b300.layer import HybridLayer

from _util import KV_REL_L2, check_attn, check_topk, f64, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_26_b300 import build
    build.build()
    hattn.lib()
    orc.lib()
    yield
    torch.cuda.empty_cache()


def _bits(t):
    return synth.bits(t)


def _host_rows(t, b, rows):
    """[1, rows-of-t, ...] uint16 host array that holds only the listed rows of
    sequence b (the others stay zero and are never read by the oracle)."""
    shape = (1,) + tuple(t.shape[1:])
    out = np.zeros(shape, np.uint16)
    rows = np.asarray(sorted(set(int(x) for x in rows)), np.int64)
    if rows.size:
        out[0, rows] = _bits(t[b, torch.as_tensor(rows, device=t.device)])
    return out


def _run(wl, t_new=None, side=False, indexer_keys="bf16"):
    """The layer step twice on the same inputs: first forming each branch's
    output (kept for the stage checks), then as the benchmark runs it (split
    partials merged in one pass, HCA and SWA on a second stream when `side`).
    Returns the inputs, the layer and both (out, lse) results."""
    inp = synth.make_inputs(wl, 0, device=DEV)
    raw = {k: inp[k] for k in ["kv_raw", "ik_raw", "gate_csa", "gate_hca"]}
    layer = HybridLayer(wl, raw, device=DEV, indexer_keys=indexer_keys)
    args = (inp["q"], inp["iq"], inp["w"], inp["pos"], inp["sink"])
    out_b, lse_b = layer.step(*args, t_new=t_new, branch_outputs=True)
    out_b, lse_b = out_b.clone(), lse_b.clone()
    side_stream = torch.cuda.Stream() if side else None
    out, lse = layer.step(*args, t_new=t_new, side_stream=side_stream)
    torch.cuda.synchronize()
    hattn.check_status()
    return inp, layer, (out_b, lse_b), (out, lse)


def _check_compress(wl, inp, layer, b, entries, kind):
    m, w = (wl.m_csa, wl.w_csa) if kind == "csa" else (wl.m_hca, wl.w_hca)
    rows = [u for j in entries for u in range(max(0, m * (j + 1) - w), m * (j + 1))]
    kv = _host_rows(inp["kv_raw"], b, rows)
    gate = np.zeros((1, wl.L), np.uint16)
    gate[0] = _bits(inp["gate_" + kind][b])
    ik = _host_rows(inp["ik_raw"], b, rows) if kind == "csa" else None
    got_kv = layer.kv_c if kind == "csa" else layer.kv_h
    for j in entries:
        rk, ri, _ = orc.compress(kv, gate, m, w, wl.r, j, j + 1, ik_raw=ik)
        assert rel_l2(got_kv[b, j], rk[0, 0]) <= KV_REL_L2, f"{kind} entry {j}"
        if kind == "csa" and layer.fp8:
            # the E4M3 key decodes to within half a step of the fp64 key
            # (plus the bf16 rounding it is quantised from)
            sc = float(layer.ik_scale[b, j])
            deq = orc.dequantize_e4m3(layer.ik8[b, j].cpu().numpy(), np.float64(sc))
            ref = ri[0, 0]
            bound = (np.maximum(np.abs(ref) * 2.0 ** -4, 2.0 ** -10 * sc)
                     + np.abs(ref) * 2.0 ** -8) * 1.01 + 1e-6
            assert (np.abs(deq - ref) <= bound).all(), f"FP8 indexer key {j}"
        elif kind == "csa":
            assert rel_l2(layer.ik_c[b, j], ri[0, 0]) <= KV_REL_L2, f"indexer key {j}"
            if layer.mx4:
                # the MXFP4 key is, byte for byte, the oracle's quantisation
                # of the bf16 key beside it
                rc, rs = orc.quantize_mxfp4(_bits(layer.ik_c[b, j:j + 1]))
                np.testing.assert_array_equal(layer.ik4[b, j].cpu().numpy(), rc[0])
                np.testing.assert_array_equal(layer.ik4_scale[b, j].cpu().numpy(), rs[0])


def _check_sequence(wl, inp, layer, res_b, res, b, ts):
    """Stage-by-stage parity of queries ts of sequence b: every branch, the
    merge of the branch outputs, and the benchmark's merge of split
    partials."""
    T = inp["q"].shape[1]
    bufs = layer.buffers(T)
    tsel = torch.as_tensor(ts, device=DEV)
    q = _bits(inp["q"][b:b + 1, tsel])
    pos = inp["pos"][b:b + 1, tsel].cpu().numpy()
    sink = inp["sink"].cpu().numpy()
    o_list, l_list = [], []
    if "csa" in wl.branches:
        iq = _bits(inp["iq"][b:b + 1, tsel])
        w = inp["w"][b:b + 1, tsel].cpu().numpy()
        if layer.fp8:
            ref_sc = orc.indexer_scores_e4m3(iq, w, layer.ik8[b:b + 1].cpu().numpy(),
                                             layer.ik_scale[b:b + 1].cpu().numpy(), pos, wl.m_csa)
        elif layer.mx4:
            ref_sc = orc.indexer_scores_mxfp4(iq, w, layer.ik4[b:b + 1].cpu().numpy(),
                                              layer.ik4_scale[b:b + 1].cpu().numpy(), pos,
                                              wl.m_csa)
        else:
            ref_sc = orc.indexer_scores(iq, w, _bits(layer.ik_c[b:b + 1]), pos, wl.m_csa)
        got_sc = f64(bufs["scores"][b:b + 1, tsel])
        vis = ~np.isnan(ref_sc)
        err = np.abs(got_sc[vis] - ref_sc[vis])
        tol = 2e-3 * (np.abs(ref_sc[vis]) + np.sqrt(wl.HI * wl.dI) * 0.05)
        assert (err <= tol).all(), f"indexer score error {err.max():.3e}"
        idx = bufs["idx"][b:b + 1, tsel].cpu().numpy()
        check_topk(idx, ref_sc, pos, wl.m_csa, wl.k, "top-k")
        ro, rl = orc.attention(orc.KIND_SPARSE, q, _bits(layer.kv_c[b:b + 1]), pos, idx=idx,
                               r=wl.r)
        check_attn(bufs["o_csa"][b:b + 1, tsel], bufs["l_csa"][b:b + 1, tsel], ro, rl, "csa")
        o_list.append(ro)
        l_list.append(rl)
    if "hca" in wl.branches:
        ro, rl = orc.attention(orc.KIND_HCA, q, _bits(layer.kv_h[b:b + 1]), pos, m=wl.m_hca,
                               r=wl.r)
        check_attn(bufs["o_hca"][b:b + 1, tsel], bufs["l_hca"][b:b + 1, tsel], ro, rl, "hca")
        o_list.append(ro)
        l_list.append(rl)
    if "swa" in wl.branches:
        rows = [u for t in pos.ravel() for u in range(max(0, int(t) - wl.W + 1), int(t) + 1)]
        raw = _host_rows(inp["kv_raw"], b, rows)
        ro, rl = orc.attention(orc.KIND_SWA, q, raw, pos, W=wl.W, r=wl.r)
        check_attn(bufs["o_swa"][b:b + 1, tsel], bufs["l_swa"][b:b + 1, tsel], ro, rl, "swa")
        o_list.append(ro)
        l_list.append(rl)
    ref_out, ref_lse = orc.merge(o_list, l_list, sink, pos, wl.r)
    for (out, lse), what in [(res_b, "layer output (branch outputs)"), (res, "layer output")]:
        check_attn(out[b:b + 1, tsel], lse[b:b + 1, tsel], ref_out, ref_lse, what)


def test_hybrid_decode_1m():
    """Batch 8 at 1,048,576 cached tokens: 262,144 CSA entries (top-1024),
    8,192 HCA entries, 128 SWA tokens; the benchmark's step, with the HCA and
    SWA branches on a second stream as the benchmark runs them."""
    wl = synth.WORKLOADS["hybrid_decode_1m"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1, side=True)
    n = wl.L // wl.m_csa
    _check_compress(wl, inp, layer, 5, [0, 1, 77777, n - 1], "csa")
    _check_compress(wl, inp, layer, 2, [0, 4095, wl.L // wl.m_hca - 1], "hca")
    _check_sequence(wl, inp, layer, res_b, res, 5, [0])
    assert torch.isfinite(res[0].float()).all()


def test_hybrid_decode_1m_mtp2():
    """Two queries per sequence (the accepted token at 1,048,574 and one
    multi-token-prediction draft at 1,048,575) over the 1M caches, the
    benchmark's step; the entry both new tokens complete is compressed once."""
    wl = synth.WORKLOADS["hybrid_decode_1m_mtp2"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1, side=True)
    _check_compress(wl, inp, layer, 6, [wl.L // wl.m_csa - 1], "csa")
    _check_compress(wl, inp, layer, 6, [wl.L // wl.m_hca - 1], "hca")
    _check_sequence(wl, inp, layer, res_b, res, 6, [0, 1])
    assert torch.isfinite(res[0].float()).all()


def test_hybrid_decode_1m_fp8_keys():
    """The 1M decode step with the indexer keys held as E4M3 codes and row
    scales: the compressor's FP8 keys, the FP8 indexer scores (against the
    oracle's dequantised definition), top-k, and the attention and merge."""
    wl = synth.WORKLOADS["hybrid_decode_1m"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1, side=True, indexer_keys="fp8")
    n = wl.L // wl.m_csa
    _check_compress(wl, inp, layer, 3, [0, 1, 123457, n - 1], "csa")
    _check_sequence(wl, inp, layer, res_b, res, 3, [0])
    assert torch.isfinite(res[0].float()).all()


def test_hybrid_decode_1m_mxfp4_keys():
    """The 1M decode step with the indexer keys held as MXFP4 codes and block
    scales: the compressor's MXFP4 keys (bit for bit the oracle's
    quantisation of its bf16 keys), the block-scaled indexer scores (against
    the oracle's decoded definition), top-k, and the attention and merge."""
    wl = synth.WORKLOADS["hybrid_decode_1m"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1, side=True, indexer_keys="mxfp4")
    n = wl.L // wl.m_csa
    _check_compress(wl, inp, layer, 5, [0, 1, 123457, n - 1], "csa")
    _check_sequence(wl, inp, layer, res_b, res, 5, [0])
    assert torch.isfinite(res[0].float()).all()


def test_pro_csa_decode():
    """Batch 32, each query against its own 131,072-token context (32,768
    entries, top-1024) plus SWA."""
    wl = synth.WORKLOADS["pro_csa_decode"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1)
    _check_compress(wl, inp, layer, 31, [3, wl.L // wl.m_csa - 1], "csa")
    for b in (0, 31):
        _check_sequence(wl, inp, layer, res_b, res, b, [0])


def test_hca_decode_1m():
    """Batch 16 at 1M context: dense attention over 8,192 HCA entries."""
    wl = synth.WORKLOADS["hca_decode"]
    inp, layer, res_b, res = _run(wl, t_new=wl.L - 1)
    _check_compress(wl, inp, layer, 9, [0, 8191], "hca")
    for b in (0, 15):
        _check_sequence(wl, inp, layer, res_b, res, b, [0])


def test_hca_prefill_chunk():
    """A 4,096-query prefill chunk at the end of a 1M context, causal over
    the 128-token compressed blocks."""
    wl = synth.WORKLOADS["hca_prefill"]
    inp, layer, res_b, res = _run(wl)
    _check_sequence(wl, inp, layer, res_b, res, 0, [0, 126, 127, 2048, 4095])


def test_flash_csa_prefill():
    """Flash-shaped causal prefill, 8,192 queries (64 heads, top-512 of up to
    2,048 entries) plus SWA; samples the first queries, a ragged middle and
    the end."""
    wl = synth.WORKLOADS["flash_csa_prefill"]
    inp, layer, res_b, res = _run(wl)
    _check_compress(wl, inp, layer, 0, [0, 1, 1000, 2047], "csa")
    _check_sequence(wl, inp, layer, res_b, res, 0, [0, 3, 2051, 4097, 8191])
