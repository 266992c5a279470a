"""How much the low-precision indexer formats change the selection, by the
oracle, on the workloads' input distribution: N(0,1) bf16 queries and keys,
N(0,1) weights, one query per row over 8,192 visible entries, top-1024.

This measures the readings (E4M3 rows with an fp32 scale; MXFP4 blocks of 32
with E8M0 scales) rather than pinning them.  The pages train the indexer QK
path for FP4, so a trained model's scores need not lose as much as these
random inputs do; the floors below sit a little under what the oracle gives
(0.975 and 0.875 of the bf16 set kept) so that a change to either
quantisation which costs selection quality shows here."""
import numpy as np
import torch

import oracle as orc


def _b16(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def test_low_precision_formats_keep_most_of_the_bf16_selection():
    rng = np.random.default_rng(5)
    B, T, HI, dI, N, m, k = 1, 4, 64, 128, 8192, 4, 1024
    iq = _b16(rng.standard_normal((B, T, HI, dI)))
    ik = _b16(rng.standard_normal((B, N, dI)))
    w = rng.standard_normal((B, T, HI)).astype(np.float32)
    pos = np.full((B, T), N * m - 1, np.int32)
    s_bf = orc.indexer_scores(iq, w, ik, pos, m)
    c8, s8 = orc.quantize_e4m3(ik)
    s_e4 = orc.indexer_scores_e4m3(iq, w, c8, s8, pos, m)
    c4, s4 = orc.quantize_mxfp4(ik)
    s_mx = orc.indexer_scores_mxfp4(iq, w, c4, s4, pos, m)

    def kept(s):
        got = orc.topk(s, pos, m, k)[0]
        ref = orc.topk(s_bf, pos, m, k)[0]
        return np.mean([len(set(a.tolist()) & set(b.tolist())) / k for a, b in zip(got, ref)])

    def rel(s):
        return np.sqrt(np.mean((s - s_bf) ** 2) / np.mean(s_bf ** 2))

    assert kept(s_e4) >= 0.96 and rel(s_e4) <= 0.05
    assert kept(s_mx) >= 0.85 and rel(s_mx) <= 0.2
    assert kept(s_e4) > kept(s_mx)
