"""The benchmark's roofline arithmetic on CPU: algorithmic bytes and flops of
every workload kind, derived here term by term from the workload shapes, and
the roofline object bench.py builds from per-call times (fake times, no GPU).

Every figure the bench reports as `achieved` or `frac` divides by one of
these, so each function is called here for each workload kind it serves."""
import os

import pytest

import bench
from sparse_attention_26_b300 import synth
from sparse_attention_26_b300.stack import layer_pattern

W = synth.WORKLOADS


def test_indexer_bytes_decode_1m():
    """One indexer launch at 1M context, batch 8: per (sequence, entry) a
    256 B bf16 key (or 128 B of E4M3 codes plus a 4 B scale); per sequence
    the 64 x 128 bf16 query rows and 64 fp32 weights.  The 4 B score written
    per (query, entry) is implementation overhead, counted apart."""
    wl = W["hybrid_decode_1m"]
    entries = 8 * 262144
    queries = 8 * (64 * 128 * 2 + 64 * 4)
    assert queries == 133_120
    assert bench.indexer_bytes(wl, "bf16") == entries * 256 + queries == 536_870_912 + 133_120
    assert bench.indexer_bytes(wl, "fp8") == entries * (128 + 4) + queries == 276_957_184
    assert bench.indexer_overhead_bytes(wl) == entries * 4
    # two queries per sequence: one key scan, the query rows twice, a score per query
    wl2 = W["hybrid_decode_1m_mtp2"]
    assert bench.indexer_bytes(wl2, "bf16") == entries * 256 + 2 * queries
    assert bench.indexer_overhead_bytes(wl2) == entries * 8


def test_step_bytes_decode_1m():
    """One decode step of the 1M hybrid layer (617 MB), read by read."""
    D, dI, H, HI = 512, 128, 128, 64
    per_seq = (
        262144 * dI * 2              # every CSA indexer key
        + 1024 * D * 2               # the k gathered CSA entries
        + HI * dI * 2 + HI * 4       # indexer query rows and weights
        + 8 * (D + dI + 1) * 2       # the newest CSA entry's 8-token window (kv, key, gate)
        + D * 2 + dI * 2             # ... and its entry and indexer key written
        + 8192 * D * 2               # every HCA entry
        + 128 * (D + 1) * 2          # the newest HCA entry's 128-token window
        + D * 2                      # ... and its entry written
        + 128 * D * 2                # the 128 window tokens
        + 2 * H * D * 2 + H * 4      # q in, output and lse out
    )
    assert bench.step_bytes(W["hybrid_decode_1m"], "bf16") == 8 * per_seq == 616_802_432


def _sum(f, n):
    return sum(f(u) for u in range(1, n + 1))


def test_step_flops_prefill():
    """Causal-exact flops: the query at position t sees (t+1)//m compressed
    entries; 2*HI*dI per (query, entry) for the indexer and 4*H*D per
    (query, key) for each attention branch."""
    fl = bench.step_flops(W["flash_csa_prefill"])
    L, H, D = 8192, 64, 512
    assert fl["indexer"] == 2 * 64 * 128 * _sum(lambda u: u // 4, L)
    assert fl["sparse"] == 4 * H * D * _sum(lambda u: min(u // 4, 512), L)
    assert fl["swa"] == 4 * H * D * _sum(lambda u: min(u, 128), L)
    assert "hca" not in fl
    assert abs(sum(fl.values()) - 754.7e9) < 0.05e9
    # HCA prefill: 4,096 queries ending at 1M, 8,160..8,192 visible entries each
    fh = bench.step_flops(W["hca_prefill"])
    L = 1 << 20
    n = sum((t + 1) // 128 for t in range(L - 4096, L))
    assert fh == {"hca": 4 * 128 * 512 * n}
    assert abs(fh["hca"] - 8.778e12) < 0.001e12


def test_stack_bytes_61_layers():
    """The 61-layer V4-Pro decode step: 18.5 GB, almost all of it the 30 CSA
    layers' indexer keys; each layer kind adds exactly its own reads."""
    wl = W["hybrid_decode_1m"]
    kinds = layer_pattern(61)
    total = bench.stack_bytes(wl, kinds)
    assert abs(total - 18.5e9) < 0.05e9
    swa = bench.stack_bytes(wl, ["swa"])
    csa = bench.stack_bytes(wl, ["csa"])
    hca = bench.stack_bytes(wl, ["hca"])
    assert total == (kinds.count("swa") * swa + kinds.count("csa") * csa
                     + kinds.count("hca") * hca)
    assert csa - swa > 8 * 262144 * 256       # at least the indexer keys
    assert hca - swa > 8 * 8192 * 512 * 2     # at least the HCA entries


def test_roofline_decode_indexer():
    wl = W["hybrid_decode_1m"]
    for keys in ("bf16", "fp8"):
        rf = bench.kernel_roofline(wl, keys, {"indexer": 0.1, "topk": 0.02}, 6482.7, "measured")
        ib = bench.indexer_bytes(wl, keys)
        assert rf["bound"] == "hbm" and rf["kernel"] == "indexer_score_kernel"
        assert rf["unit"] == "GB/s" and rf["peak"] == 6482.7
        assert rf["achieved"] == pytest.approx(ib / 1e-4 / 1e9)
        assert rf["frac"] == pytest.approx(rf["achieved"] / 6482.7)
        assert rf["overhead_bytes_per_launch"] == bench.indexer_overhead_bytes(wl)
        if rf["traffic"] is not None:  # scaled from the recorded capture (scores included)
            tot = ib + rf["overhead_bytes_per_launch"]
            assert 0.95 < rf["traffic"] / tot < 1.05
    # the capture is of one query per sequence: none for two
    rf2 = bench.kernel_roofline(W["hybrid_decode_1m_mtp2"], "bf16", {"indexer": 0.1}, 6482.7,
                                "measured")
    assert rf2["traffic"] is None


def test_roofline_hca_decode_reports_both_fractions():
    wl = W["hca_decode"]
    rf = bench.kernel_roofline(wl, "bf16", {"attn_fused": 0.085}, 6482.7, "measured")
    by = 16 * (8192 * 512 * 2 + (2 * 128 * 512 * 2 + 128 * 4))
    assert rf["bound"] == "hbm" and rf["algorithmic_bytes_per_launch"] == by
    assert rf["achieved"] == pytest.approx(by / 0.085e-3 / 1e9)
    t = rf["tensor"]
    # a decode step lasts microseconds: the burst peak
    assert t["unit"] == "TFLOP/s" and t["peak"] == bench.measured_bf16_burst()[0]
    assert t["flops_per_launch"] == 16 * 4 * 128 * 512 * 8192


def test_roofline_prefill_takes_the_slowest_call():
    wl = W["flash_csa_prefill"]
    times = {"indexer": 2.5, "sparse": 3.0, "swa": 2.1, "merge": 1.2}
    rf = bench.kernel_roofline(wl, "bf16", times, 6482.7, "measured")
    fl = bench.step_flops(wl)
    assert rf["bound"] == "tensor" and rf["kernel"] == "attn_kernel<kSparse>"
    assert rf["achieved"] == pytest.approx(fl["sparse"] / 3.0e-3 / 1e12)
    # a prefill pass lasts milliseconds: the burst peak, not the seconds-long sustained one
    assert rf["peak"] == bench.measured_bf16_burst()[0]
    assert set(rf["by_call"]) == {"indexer", "sparse", "swa"}
    rh = bench.kernel_roofline(W["hca_prefill"], "bf16", {"hca": 14.7}, 6482.7, "measured")
    assert rh["kernel"] == "attn_kernel<kHca>"
    # the fused call: one launch carries the flops of every attention branch
    rf = bench.kernel_roofline(wl, "bf16", {"indexer": 0.4, "attn_fused": 4.0}, 6482.7,
                               "measured")
    assert rf["kernel"].startswith("attn_kernel<kFused>")
    assert rf["flops_per_launch"] == pytest.approx(fl["sparse"] + fl["swa"])
    assert rf["achieved"] == pytest.approx((fl["sparse"] + fl["swa"]) / 4.0e-3 / 1e12)


def test_l2_note_is_true_per_workload():
    """Decode: the step's algorithmic input exceeds L2.  Prefill: the
    streamed queries exceed L2 while the compressed caches are L2-resident
    by design, and the note says so rather than calling the input larger."""
    assert "> 126 MB L2 (no flush)" in bench.l2_note(W["hybrid_decode_1m"])
    for name, cache_mb in (("flash_csa_prefill", 2.6), ("hca_prefill", 8.4)):
        note = bench.l2_note(W[name])
        assert "L2-resident" in note and f"({cache_mb:.1f} MB)" in note, note


def test_timed_replays_split_the_steps():
    """The K timed steps run as R separately timed replays of one graph of
    K / R steps (R up to 10), so the line carries a median and a spread."""
    assert bench.timed_replays(50) == (10, 5)
    assert bench.timed_replays(20) == (10, 2)
    assert bench.timed_replays(7) == (7, 1)
    assert bench.timed_replays(1) == (1, 1)
    for k in range(1, 101):
        r, g = bench.timed_replays(k)
        assert r * g == k and 1 <= r <= 10


def test_traffic_profile_is_committed():
    path = os.path.join(bench.ROOT, bench.INDEXER_TRAFFIC["profile"])
    assert os.path.isfile(path)


def test_default_run_keeps_the_timing_contract(monkeypatch):
    """With no flags: one GPU, at least 3 warm-up steps, a short timed run,
    the 1M decode workload, the oracle baseline and the end-to-end leg on."""
    monkeypatch.setattr("sys.argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.warmup >= 3 and 1 <= a.steps <= 100
    assert a.impl == "ours" and a.workload == "hybrid_decode_1m"
    assert not a.no_cpu_baseline and not a.no_e2e and a.indexer_keys == "bf16"
    assert not a.stack and not a.cache_build and not a.quantize_keys


def test_cpu_baseline_runs_on_the_host():
    """The oracle legs of the bench at reduced sizes, on CPU: a decode step
    and a sampled prefill pass, each a single-threaded oracle time with the
    host's CPU model and core count."""
    dec = bench.cpu_baseline(synth.scaled(W["hybrid_decode_1m"], L=8192))
    assert dec["kind"] == "oracle" and dec["cores"] == 1 and dec["value"] > 0
    assert dec["host"]["nproc"] >= 1 and dec["host"]["cpu_model"]
    pre = bench.cpu_baseline(synth.scaled(W["flash_csa_prefill"], L=512, T=512))
    assert pre["value"] > 0 and pre["sample"].startswith("extrapolated")
