"""GPU parity of every C-ABI call against the fp64 CPU oracle, at sizes the
oracle finishes in seconds that still span several tiles and a ragged tail,
plus the edge cases (empty / short key sets, padding, uninitialised cache
tails, ties, the lazy-rescale path, the bounded-wait timeout)."""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_26_b300 import hattn, synth

from _util import (KV_REL_L2, check_attn, check_topk, f64, rel_l2)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def bits(t):
    return synth.bits(t)


def randn_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def randn_f32(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).float()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_26_b300 import build
    build.build()
    hattn.lib()
    orc.lib()
    torch.cuda.init()
    yield
    hattn.check_status()


# ------------------------------------------------------------------ status
def test_bounded_wait_times_out_and_reports():
    hattn.check_status()  # clear
    hattn.selftest_wait_timeout(2_000_000)  # 2 ms, nothing ever arrives
    assert hattn.check_status_code() == hattn.TIMEOUT
    assert hattn.check_status_code() == hattn.OK  # read clears it


# ------------------------------------------------------------------ compression
@pytest.mark.parametrize("B,L,D,dI,r,j0,j1", [
    (2, 64, 64, 32, 16, 0, 16),
    (1, 1030, 512, 128, 64, 0, 257),
    (2, 1024, 512, 128, 64, 100, 131),   # incremental range
    (2, 4096, 64, 32, 16, 0, 1024),      # many entries: the grid-stride kernel, not the small one
])
def test_csa_compress(B, L, D, dI, r, j0, j1):
    kv = randn_bf16((B, L, D), 1)
    ik = randn_bf16((B, L, dI), 2)
    gate = randn_bf16((B, L), 3)
    gamma = (1.0 + 0.1 * randn_f32((D,), 4))
    N_cap = L // 4
    kv_c = torch.full((B, N_cap, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ik_c = torch.full((B, N_cap, dI), float("nan"), dtype=torch.bfloat16, device=DEV)
    hattn.csa_compress(kv.to(DEV), ik.to(DEV), gate.to(DEV), r=r, j_begin=j0, j_end=j1,
                       kv_c=kv_c, ik_c=ik_c, gamma_kv=gamma.to(DEV))
    hattn.check_status()
    ref_kv, ref_ik, _ = orc.compress(bits(kv), bits(gate), 4, 8, r, j0, j1, ik_raw=bits(ik),
                                     gamma=gamma.numpy())
    assert rel_l2(kv_c[:, j0:j1], ref_kv) <= KV_REL_L2
    assert rel_l2(ik_c[:, j0:j1], ref_ik) <= KV_REL_L2
    # rows outside the range are untouched
    assert torch.isnan(kv_c[:, :j0].float()).all() and torch.isnan(kv_c[:, j1:].float()).all()


@pytest.mark.parametrize("B,L,dm,D,dI,m,w,r,j0,j1", [
    (2, 1024, 512, 512, 128, 4, 8, 64, 0, 256),      # a CSA cache build
    (1, 1030, 1024, 512, 128, 4, 8, 64, 200, 257),   # an entry range, ragged length
    (2, 1024, 512, 512, 0, 128, 128, 64, 0, 8),      # HCA: no indexer key
    (1, 600, 200, 64, 32, 4, 8, 16, 0, 150),         # a ragged last K block; a narrow key group
    (1, 520, 128, 256, 64, 4, 8, 32, 3, 130),        # mid-size D: one 256-column product
])
def test_compress_hidden(B, L, dm, D, dI, m, w, r, j0, j1):
    """Entries from hidden states (pooled, then projected once) against the
    oracle, which projects every token in fp64 and then compresses."""
    x = randn_bf16((B, L, dm), 70)
    W = (randn_f32((dm, D + dI), 71) / math.sqrt(dm)).to(torch.bfloat16)
    gate = randn_bf16((B, L), 72)
    N_cap = L // m
    kv = torch.full((B, N_cap, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ik = torch.full((B, N_cap, dI), float("nan"), dtype=torch.bfloat16, device=DEV) if dI else None
    hattn.compress_hidden(x.to(DEV), W.to(DEV), gate.to(DEV), D=D, r=r, m=m, w=w, j_begin=j0,
                          j_end=j1, kv_out=kv, ik_out=ik)
    hattn.check_status()
    ref_kv, ref_ik = orc.compress_hidden(bits(x), bits(W), bits(gate), m, w, r, j0, j1, D)
    assert rel_l2(kv[:, j0:j1], ref_kv) <= KV_REL_L2
    if dI:
        assert rel_l2(ik[:, j0:j1], ref_ik) <= KV_REL_L2
    assert torch.isnan(kv[:, :j0].float()).all() and torch.isnan(kv[:, j1:].float()).all()


def test_compress_hidden_across_chunks():
    """17,500 entries: two passes of pooling and projection; sampled entries
    on both sides of the chunk boundary and at the ends."""
    B, L, dm, D, dI, r = 1, 70000, 256, 512, 128, 64
    x = randn_bf16((B, L, dm), 73)
    W = (randn_f32((dm, D + dI), 74) / math.sqrt(dm)).to(torch.bfloat16)
    gate = randn_bf16((B, L), 75)
    kv, ik = hattn.compress_hidden(x.to(DEV), W.to(DEV), gate.to(DEV), D=D, r=r)
    hattn.check_status()
    for j0, j1 in [(0, 3), (16382, 16386), (L // 4 - 2, L // 4)]:
        ref_kv, ref_ik = orc.compress_hidden(bits(x), bits(W), bits(gate), 4, 8, r, j0, j1, D)
        assert rel_l2(kv[:, j0:j1], ref_kv) <= KV_REL_L2, (j0, j1)
        assert rel_l2(ik[:, j0:j1], ref_ik) <= KV_REL_L2, (j0, j1)


@pytest.mark.parametrize("B,L,L_cap,dm,D,dI,r", [
    (2, 1024, 1024, 512, 512, 128, 64),   # whole blocks: 256 CSA and 8 HCA entries each
    (1, 1000, 1030, 200, 64, 32, 16),     # a ragged tail block (no HCA entry), ragged K
])
def test_compress_hidden_pair(B, L, L_cap, dm, D, dI, r):
    """Both caches from one read of the hidden states equal the oracle's two
    compressions (the same as two hattn_compress_hidden calls)."""
    x = randn_bf16((B, L_cap, dm), 76)
    W_c = (randn_f32((dm, D + dI), 77) / math.sqrt(dm)).to(torch.bfloat16)
    W_h = (randn_f32((dm, D), 78) / math.sqrt(dm)).to(torch.bfloat16)
    g_c = randn_bf16((B, L_cap), 79)
    g_h = randn_bf16((B, L_cap), 80)
    gamma = 1.0 + 0.1 * randn_f32((D,), 81)
    N_c, N_h = L_cap // 4, max(1, L_cap // 128)
    kv_c = torch.full((B, N_c, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kv_h = torch.full((B, N_h, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    kv_c, ik_c, kv_h = hattn.compress_hidden_pair(x.to(DEV), W_c.to(DEV), g_c.to(DEV),
                                                  W_h.to(DEV), g_h.to(DEV), D=D, r=r, L=L,
                                                  kv_c=kv_c, kv_h=kv_h, gamma_kv=gamma.to(DEV))
    hattn.check_status()
    nc, nh = L // 4, L // 128
    ref_kv, ref_ik = orc.compress_hidden(bits(x), bits(W_c), bits(g_c), 4, 8, r, 0, nc, D,
                                         gamma=gamma.numpy())
    assert rel_l2(kv_c[:, :nc], ref_kv) <= KV_REL_L2
    assert rel_l2(ik_c[:, :nc], ref_ik) <= KV_REL_L2
    ref_h, _ = orc.compress_hidden(bits(x), bits(W_h), bits(g_h), 128, 128, r, 0, nh, D,
                                   gamma=gamma.numpy())
    assert rel_l2(kv_h[:, :nh], ref_h) <= KV_REL_L2
    # entries past L are untouched
    assert torch.isnan(kv_c[:, nc:].float()).all() and torch.isnan(kv_h[:, nh:].float()).all()


@pytest.mark.parametrize("B,L,D,r", [(2, 1024, 512, 64), (1, 300, 64, 16)])
def test_hca_compress(B, L, D, r):
    kv = randn_bf16((B, L, D), 5)
    gate = randn_bf16((B, L), 6)
    n = L // 128
    if n == 0:
        pytest.skip("no complete entry")
    kv_h = hattn.hca_compress(kv.to(DEV), gate.to(DEV), r=r)
    hattn.check_status()
    ref, _, _ = orc.compress(bits(kv), bits(gate), 128, 128, r, 0, n)
    assert rel_l2(kv_h[:, :n], ref) <= KV_REL_L2


# ------------------------------------------------------------------ indexer + top-k
def _indexer_case(B, T, HI, dI, N_cap, k, pos, seed, m=4):
    iq = randn_bf16((B, T, HI, dI), seed)
    w = randn_f32((B, T, HI), seed + 1)
    ik = randn_bf16((B, N_cap, dI), seed + 2)
    pos_t = torch.tensor(pos, dtype=torch.int32).reshape(B, T)
    scores = torch.full((B, T, N_cap), float("nan"), device=DEV)
    idx = hattn.indexer_topk(iq.to(DEV), w.to(DEV), ik.to(DEV), pos_t.to(DEV), k=k, m=m,
                             score_out=scores)
    hattn.check_status()
    ref = orc.indexer_scores(bits(iq), w.numpy(), bits(ik), pos_t.numpy(), m)
    vis = ~np.isnan(ref)
    got = f64(scores)
    assert np.isfinite(got[vis]).all()
    err = np.abs(got[vis] - ref[vis])
    tol = 2e-3 * (np.abs(ref[vis]) + np.sqrt(HI * dI) * 0.05)
    assert (err <= tol).all(), f"score error {err.max():.3e}"
    check_topk(idx.cpu().numpy(), ref, pos_t.numpy(), m, k)
    return idx


def test_indexer_decode_ragged():
    # visible counts 0, 10 (< k), 150 (spans two 128-blocks), 600 (ragged tail)
    _indexer_case(4, 1, 64, 128, 600, 16, [2, 41, 603, 2399], 10)


def test_indexer_prefill_groups():
    # 64 heads -> 4 queries per group; T=7 leaves a ragged group
    T = 7
    _indexer_case(2, T, 64, 128, 520, 32, [[4 * j + 3 + 40 * t for t in range(T)]
                                           for j in range(2)], 20)


def test_indexer_tiny_shape():
    # 2 heads x 32 dims, causal prefill over 256 positions
    _indexer_case(1, 256, 2, 32, 64, 16, [list(range(256))], 30)


# ------------------------------------------------------------------ FP8 indexer keys
def _u8(t):
    return t.cpu().numpy().astype(np.uint8)


@pytest.mark.parametrize("rows,n", [(1003, 128), (37, 64), (5, 4)])
def test_quantize_e4m3_bit_exact(rows, n):
    """Codes and row scales equal the oracle's bit for bit: row magnitudes
    from 1e-4 to 1e4 (subnormal codes included), one all-zero row, rows
    whose largest element is negative; 1003 rows of 128 leave a partial
    group of eight for the 128-wide kernel."""
    g = torch.Generator().manual_seed(50)
    mag = 10.0 ** torch.randint(-4, 5, (rows, 1), generator=g).float()
    x = (torch.randn((rows, n), generator=g) * mag).to(torch.bfloat16)
    x[0] = 0
    if rows > 3:
        x[3, 1] = -4 * x[3].float().abs().max()
    codes, scales = hattn.quantize_e4m3(x.to(DEV))
    hattn.check_status()
    rc, rs = orc.quantize_e4m3(bits(x))
    np.testing.assert_array_equal(_u8(codes), rc)
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)


@pytest.mark.parametrize("rows,n", [(1003, 128), (37, 96), (5, 32), (3, 512)])
def test_quantize_mxfp4_bit_exact(rows, n):
    """E2M1 codes and E8M0 block scales equal the oracle's bit for bit.
    Block magnitudes span 1e-30..1e30 and include subnormal blocks (scale
    exponent clamped at -127); one block is all zeros, another holds -0 and
    small negatives (stored as +0), another puts every element on a tie
    between two E2M1 values, another saturates (amax / X = 7).  n = 96 leaves
    a partial 128-element span, 1003 rows a partial group of eight (the
    128-wide kernel); rows = 0 launches nothing."""
    g = torch.Generator().manual_seed(54)
    nb = n // 32
    mag = 10.0 ** torch.randint(-30, 31, (rows, nb, 1), generator=g).float()
    x = torch.randn((rows, nb, 32), generator=g) * mag
    x[0, 0] = torch.randn(32, generator=g) * 1e-39            # subnormal block
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5, -5.0] * 3 + [6.0, 1.0])
    x[1 % rows, nb - 1] = ties * 2.0 ** -3
    if rows > 2:
        x[2, 0] = 0.0
        x[2, nb - 1] = torch.tensor([-0.0, -1e-3, 7.0, -7.0] * 8) * 2.0 ** 10   # -0, saturation
    x = x.reshape(rows, n).to(torch.bfloat16)
    codes, scales = hattn.quantize_mxfp4(x.to(DEV))
    hattn.check_status()
    rc, rs = orc.quantize_mxfp4(bits(x))
    np.testing.assert_array_equal(_u8(scales), rs)
    np.testing.assert_array_equal(_u8(codes), rc)
    e_codes, e_scales = hattn.quantize_mxfp4(torch.empty((0, n), dtype=torch.bfloat16,
                                                         device=DEV))
    assert e_codes.shape == (0, n // 2) and e_scales.shape == (0, n // 32)


# ------------------------------------------------------------------ MXFP4 indexer keys
def _mx(x):
    """MXFP4 codes [.., 64] and scales [.., 4] of bf16 rows [.., 128] (the
    library's quantiser, bit-exact against the oracle's)."""
    lead = x.shape[:-1]
    c, s = hattn.quantize_mxfp4(x.reshape(-1, 128).to(DEV))
    return c.reshape(*lead, 64), s.reshape(*lead, 4)


@pytest.mark.parametrize("B,T,N_cap,k,pos", [
    (3, 1, 600, 16, [2, 599 * 4 + 3, 4 * 300 + 1]),          # nothing visible, full, ragged
    (2, 5, 1300, 64, [[4 * 1000 + t for t in range(5)], [4 * 77 + 3 * t for t in range(5)]]),
])
def test_indexer_mxfp4(B, T, N_cap, k, pos):
    """Scores over MXFP4 keys, per entry, against the oracle's definition over
    the decoded keys and the decoded query round trip; top-k by the 1e-3
    rule.  T = 5 runs groups of 4 queries (256 columns, a ragged group)."""
    HI, dI = 64, 128
    iq = randn_bf16((B, T, HI, dI), 140)
    w = randn_f32((B, T, HI), 141)
    ik = randn_bf16((B, N_cap, dI), 142)
    ik4, iks = _mx(ik)
    pos_t = torch.tensor(pos, dtype=torch.int32).reshape(B, T)
    scores = torch.full((B, T, N_cap), float("nan"), device=DEV)
    hattn.indexer_scores_mxfp4(iq.to(DEV), w.to(DEV), ik4, iks, pos_t.to(DEV), score_out=scores)
    idx = hattn.indexer_topk_mxfp4(iq.to(DEV), w.to(DEV), ik4, iks, pos_t.to(DEV), k=k)
    hattn.check_status()
    ref = orc.indexer_scores_mxfp4(bits(iq), w.numpy(), _u8(ik4), _u8(iks), pos_t.numpy(), 4)
    vis = ~np.isnan(ref)
    got = f64(scores)
    assert np.isfinite(got[vis]).all()
    err = np.abs(got[vis] - ref[vis])
    tol = 2e-3 * (np.abs(ref[vis]) + np.sqrt(HI * dI) * 0.05)
    assert (err <= tol).all(), f"score error {err.max():.3e}"
    check_topk(idx.cpu().numpy(), ref, pos_t.numpy(), 4, k)


@pytest.mark.parametrize("N_cap,k", [(40000, 1024), (3000, 512)])
def test_indexer_mxfp4_lossless_exact(N_cap, k):
    """Rows on the E2M1 grid with a 4 in every block lose nothing to MXFP4
    (block scale 1), and their products sum exactly in fp32: scores equal
    the oracle's bit for bit and the selected sets (ties to the smaller
    index) are identical.  40,000 entries take the cluster selection with
    the folded first pass."""
    B, T, HI, dI = 2, 1, 64, 128
    g = torch.Generator().manual_seed(143)
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def rows(*shape):
        v = grid[torch.randint(0, 8, shape + (dI,), generator=g)]
        v = v * (torch.randint(0, 2, v.shape, generator=g) * 2 - 1)
        v.view(-1, dI // 32, 32)[:, :, 0] = 6.0   # each block's amax in [4, 8): scale 1
        return v.to(torch.bfloat16)

    iq, ik = rows(B, T, HI), rows(B, N_cap)
    w = torch.ones((B, T, HI)) * 0.5
    ik4, iks = _mx(ik)
    assert (_u8(iks) == 127).all()
    pos = torch.tensor([[4 * N_cap - 1], [4 * (N_cap // 2) + 1]], dtype=torch.int32)
    scores = torch.zeros((B, T, N_cap), device=DEV)
    idx = hattn.indexer_topk_mxfp4(iq.to(DEV), w.to(DEV), ik4, iks, pos.to(DEV), k=k,
                                   score_out=scores)
    hattn.check_status()
    ref = orc.indexer_scores_mxfp4(bits(iq), w.numpy(), _u8(ik4), _u8(iks), pos.numpy(), 4)
    vis = ~np.isnan(ref)
    np.testing.assert_array_equal(f64(scores)[vis], ref[vis])
    ref_idx = orc.topk(ref, pos.numpy(), 4, k)
    got = idx.cpu().numpy()
    for b in range(B):
        assert sorted(got[b, 0][got[b, 0] >= 0].tolist()) == sorted(
            ref_idx[b, 0][ref_idx[b, 0] >= 0].tolist())
        assert (got[b, 0] == -1).sum() == (ref_idx[b, 0] == -1).sum()


@pytest.mark.parametrize("B,N_cap,j0,j1", [(3, 700, 0, 700), (2, 1000, 37, 613), (2, 64, 5, 5)])
def test_quantize_mxfp4_entries(B, N_cap, j0, j1):
    """Entries [j0, j1) of every sequence of a cache, bit-exact against the
    oracle's quantiser; the codes and scales outside the range keep their
    bytes (an empty range writes nothing)."""
    x = (randn_bf16((B, N_cap, 128), 150).float() * 3.0).to(torch.bfloat16)
    codes = torch.full((B, N_cap, 64), 0xA5, dtype=torch.uint8, device=DEV)
    scales = torch.full((B, N_cap, 4), 0x5A, dtype=torch.uint8, device=DEV)
    hattn.quantize_mxfp4_entries(x.to(DEV), codes, scales, j_begin=j0, j_end=j1)
    hattn.check_status()
    rc, rs = orc.quantize_mxfp4(bits(x[:, j0:j1].reshape(-1, 128)))
    c, s = _u8(codes), _u8(scales)
    np.testing.assert_array_equal(c[:, j0:j1].reshape(-1, 64), rc)
    np.testing.assert_array_equal(s[:, j0:j1].reshape(-1, 4), rs)
    assert (c[:, :j0] == 0xA5).all() and (c[:, j1:] == 0xA5).all()
    assert (s[:, :j0] == 0x5A).all() and (s[:, j1:] == 0x5A).all()


@pytest.mark.parametrize("B,L,D,dI,r,j0,j1", [
    (2, 1024, 512, 128, 64, 255, 256),   # one new entry per sequence: the small kernel
    (2, 4096, 512, 128, 64, 0, 1024),    # cache build: the grid-stride kernel
])
def test_csa_compress_fp8(B, L, D, dI, r, j0, j1):
    """The FP8 indexer key the compressor writes is the oracle's quantisation
    of the bf16 key it writes beside it, and decodes to within half an E4M3
    step of the oracle's fp64 key; the KV entries are those of the bf16
    call."""
    kv = randn_bf16((B, L, D), 51)
    ik = randn_bf16((B, L, dI), 52)
    gate = randn_bf16((B, L), 53)
    N_cap = L // 4
    d = dict(kv=kv.to(DEV), ik=ik.to(DEV), gate=gate.to(DEV))
    kv_c, ik_c = hattn.csa_compress(d["kv"], d["ik"], d["gate"], r=r, j_begin=j0, j_end=j1)
    kv_c8 = torch.zeros_like(kv_c)
    ik_c8 = torch.zeros_like(ik_c)
    _, ik8, iks = hattn.csa_compress_fp8(d["kv"], d["ik"], d["gate"], r=r, j_begin=j0, j_end=j1,
                                         kv_c=kv_c8, ik_c=ik_c8)
    # the FP8 key alone (no bf16 key output)
    _, ik8b, iksb = hattn.csa_compress_fp8(d["kv"], d["ik"], d["gate"], r=r, j_begin=j0,
                                           j_end=j1)
    hattn.check_status()
    assert torch.equal(kv_c8, kv_c) and torch.equal(ik_c8, ik_c)
    assert torch.equal(ik8b, ik8) and torch.equal(iksb, iks)
    rc, rs = orc.quantize_e4m3(bits(ik_c[:, j0:j1].cpu()))
    np.testing.assert_array_equal(_u8(ik8[:, j0:j1]), rc)
    np.testing.assert_array_equal(iks[:, j0:j1].cpu().numpy(), rs)
    _, ref_ik, _ = orc.compress(bits(kv), bits(gate), 4, 8, r, j0, j1, ik_raw=bits(ik))
    deq = orc.dequantize_e4m3(_u8(ik8[:, j0:j1]), iks[:, j0:j1].cpu().numpy())
    sc = iks[:, j0:j1].cpu().numpy().astype(np.float64)[..., None]
    # half an E4M3 step of the bf16 key plus the bf16 rounding of the key
    bound = (np.maximum(np.abs(ref_ik) * 2.0 ** -4, 2.0 ** -10 * sc) + np.abs(ref_ik) * 2.0 ** -8
             ) * 1.01 + 1e-6
    assert (np.abs(deq - ref_ik) <= bound).all()
    assert (ik8[:, :j0] == 0).all() and (ik8[:, j1:] == 0).all()


@pytest.mark.parametrize("B,L,D,dI,r,j0,j1", [
    (2, 1024, 512, 128, 64, 255, 256),   # one new entry per sequence: the small kernel
    (2, 4096, 512, 128, 64, 0, 1024),    # cache build: the grid-stride kernel
])
def test_csa_compress_mxfp4(B, L, D, dI, r, j0, j1):
    """The MXFP4 indexer key the compressor writes is, byte for byte, the
    oracle's quantisation of the bf16 key it writes beside it; the KV entries
    and bf16 keys are those of the plain call, the other entries untouched."""
    kv = randn_bf16((B, L, D), 51)
    ik = randn_bf16((B, L, dI), 52)
    gate = randn_bf16((B, L), 53)
    N_cap = L // 4
    d = dict(kv=kv.to(DEV), ik=ik.to(DEV), gate=gate.to(DEV))
    kv_c, ik_c = hattn.csa_compress(d["kv"], d["ik"], d["gate"], r=r, j_begin=j0, j_end=j1)
    kv_c4 = torch.zeros_like(kv_c)
    ik_c4 = torch.zeros_like(ik_c)
    ik4 = torch.full((B, N_cap, dI // 2), 0xA5, dtype=torch.uint8, device=DEV)
    ik4s = torch.full((B, N_cap, dI // 32), 0x5A, dtype=torch.uint8, device=DEV)
    hattn.csa_compress_mxfp4(d["kv"], d["ik"], d["gate"], r=r, j_begin=j0, j_end=j1, kv_c=kv_c4,
                             ik_c=ik_c4, ik4=ik4, ik4_scale=ik4s)
    hattn.check_status()
    assert torch.equal(kv_c4, kv_c) and torch.equal(ik_c4, ik_c)
    rc, rs = orc.quantize_mxfp4(bits(ik_c[:, j0:j1].reshape(-1, dI).cpu()))
    np.testing.assert_array_equal(_u8(ik4[:, j0:j1]).reshape(-1, dI // 2), rc)
    np.testing.assert_array_equal(_u8(ik4s[:, j0:j1]).reshape(-1, dI // 32), rs)
    assert (ik4[:, :j0] == 0xA5).all() and (ik4[:, j1:] == 0xA5).all()
    assert (ik4s[:, :j0] == 0x5A).all() and (ik4s[:, j1:] == 0x5A).all()


def _indexer_fp8_case(B, T, HI, N_cap, k, pos, seed, m=4):
    dI = 128
    iq = randn_bf16((B, T, HI, dI), seed)
    w = randn_f32((B, T, HI), seed + 1)
    ik = randn_bf16((B, N_cap, dI), seed + 2)
    ik8, iks = orc.quantize_e4m3(bits(ik))
    pos_t = torch.tensor(pos, dtype=torch.int32).reshape(B, T)
    scores = torch.full((B, T, N_cap), float("nan"), device=DEV)
    hattn.indexer_scores_fp8(iq.to(DEV), w.to(DEV), torch.from_numpy(ik8).to(DEV),
                             torch.from_numpy(iks).to(DEV), pos_t.to(DEV), m=m,
                             score_out=scores)
    idx = hattn.topk_select(scores, pos_t.to(DEV), k=k, m=m)
    hattn.check_status()
    ref = orc.indexer_scores_e4m3(bits(iq), w.numpy(), ik8, iks, pos_t.numpy(), m)
    vis = ~np.isnan(ref)
    got = f64(scores)
    assert np.isnan(got[~vis]).all()  # entries past the visible count untouched
    err = np.abs(got[vis] - ref[vis])
    tol = 2e-3 * (np.abs(ref[vis]) + np.sqrt(HI * dI) * 0.05)
    assert (err <= tol).all(), f"score error {err.max():.3e}"
    check_topk(idx.cpu().numpy(), ref, pos_t.numpy(), m, k)


def test_indexer_fp8_decode_ragged():
    # visible counts 0, 10 (< k), 150 (two 128-blocks), 600 (ragged tail)
    _indexer_fp8_case(4, 1, 64, 600, 16, [2, 41, 603, 2399], 60)


def test_indexer_fp8_multi_query():
    # two queries per sequence (the multi-token-prediction decode), and T=7
    # with 64 heads: 4 queries per group and a ragged group
    _indexer_fp8_case(3, 2, 64, 1000, 64, [3998, 3999, 1500, 1501, 17, 18], 61)
    T = 7
    _indexer_fp8_case(2, T, 64, 520, 32, [[4 * j + 3 + 40 * t for t in range(T)]
                                          for j in range(2)], 62)


def test_indexer_fp8_exact_scores_and_ties():
    """Keys and queries of multiples of 1/2 with largest magnitude 3.5
    quantise without loss (scale 2^-7), and with weights 1 and 1/2 every
    product, head sum and scale is exact in fp32: the scores equal the
    oracle's bit for bit and the selected sets agree, ties included."""
    B, T, HI, dI, N_cap, k = 2, 1, 64, 128, 20000, 1024
    g = torch.Generator().manual_seed(63)

    def rows(shape):
        v = torch.randint(-7, 8, shape, generator=g).float() / 2
        v[..., 5] = 3.5
        return v.to(torch.bfloat16)

    iq, ik = rows((B, T, HI, dI)), rows((B, N_cap, dI))
    w = torch.where(torch.arange(HI) % 2 == 0, 1.0, 0.5).repeat(B, T, 1).float()
    pos = torch.tensor([[4 * N_cap - 1], [4 * 7777 + 2]], dtype=torch.int32)
    ik8, iks = hattn.quantize_e4m3(ik.to(DEV))
    scores = torch.zeros((B, T, N_cap), device=DEV)
    hattn.indexer_scores_fp8(iq.to(DEV), w.to(DEV), ik8, iks, pos.to(DEV), score_out=scores)
    idx = hattn.topk_select(scores, pos.to(DEV), k=k)
    hattn.check_status()
    assert (iks == 2.0 ** -7).all()
    ref = orc.indexer_scores_e4m3(bits(iq), w.numpy(), _u8(ik8), iks.cpu().numpy(), pos.numpy(),
                                  4)
    vis = ~np.isnan(ref)
    np.testing.assert_array_equal(f64(scores)[vis], ref[vis])
    ref_idx = orc.topk(ref, pos.numpy(), 4, k)
    got = idx.cpu().numpy()
    for b in range(B):
        assert sorted(got[b, 0][got[b, 0] >= 0].tolist()) == sorted(
            ref_idx[b, 0][ref_idx[b, 0] >= 0].tolist())


@pytest.mark.parametrize("N_cap,k", [(40000, 1024), (262144, 1024), (3000, 512)])
def test_topk_exact_with_ties(N_cap, k):
    """Integer-valued scores are exact in fp32 on both sides, so the selected
    sets must agree bit for bit, ties included (ties go to the smaller j)."""
    B, T, HI, dI = 2, 1, 2, 32
    g = torch.Generator().manual_seed(7)
    iq = torch.randint(-2, 3, (B, T, HI, dI), generator=g).to(torch.bfloat16)
    ik = torch.randint(-2, 3, (B, N_cap, dI), generator=g).to(torch.bfloat16)
    w = torch.tensor([1.0, 0.5]).repeat(B, T, 1).float()
    pos = torch.tensor([[4 * N_cap - 1], [4 * (N_cap // 2) + 1]], dtype=torch.int32)
    scores = torch.zeros((B, T, N_cap), device=DEV)
    idx = hattn.indexer_topk(iq.to(DEV), w.to(DEV), ik.to(DEV), pos.to(DEV), k=k, m=4,
                             score_out=scores)
    hattn.check_status()
    ref = orc.indexer_scores(bits(iq), w.numpy(), bits(ik), pos.numpy(), 4)
    vis = ~np.isnan(ref)
    np.testing.assert_array_equal(f64(scores)[vis], ref[vis])
    ref_idx = orc.topk(ref, pos.numpy(), 4, k)
    got = idx.cpu().numpy()
    for b in range(B):
        assert sorted(got[b, 0][got[b, 0] >= 0].tolist()) == sorted(
            ref_idx[b, 0][ref_idx[b, 0] >= 0].tolist())
        assert (got[b, 0] == -1).sum() == (ref_idx[b, 0] == -1).sum()


def _topk_ref_check(scores, pos, k, m, idx):
    """The oracle's selection over the same fp32 scores: identical sets."""
    ref_idx = orc.topk(scores.cpu().numpy().astype(np.float64), pos.cpu().numpy(), m, k)
    got = idx.cpu().numpy()
    for r in range(got.shape[0] * got.shape[1]):
        g, rf = got.reshape(-1, k)[r], ref_idx.reshape(-1, k)[r]
        assert sorted(g[g >= 0].tolist()) == sorted(rf[rf >= 0].tolist()), r
        n_pad = int((rf == -1).sum())
        assert (g == -1).sum() == n_pad, r
        assert (g[len(g) - n_pad:] == -1).all(), r


@pytest.mark.parametrize("B,N_cap,k", [(4, 100000, 1024), (3, 40000, 2048), (300, 3000, 512)])
def test_topk_select_edge_cases(B, N_cap, k):
    """Both selection paths (few long rows spread over many CTAs; many rows
    one CTA each) on scores built to hit their corners, against the oracle's
    selection over the same fp32 values: a row of one repeated value (every
    entry ties, the smallest indices win), a row with fewer visible entries
    than k (all of them, then -1), ties straddling the threshold, signed
    zeros, and a row of distinct random values."""
    g = torch.Generator().manual_seed(31)
    sc = torch.randn((B, 1, N_cap), generator=g)
    sc[0, 0] = 1.5                                   # all tie
    if B > 1:
        sc[1, 0, : 2 * k] = torch.randint(0, 3, (2 * k,), generator=g).float()  # few values
        sc[1, 0, 2 * k:] = -1.0
    if B > 2:
        v = torch.randn((N_cap,), generator=g)
        top = v.topk(k).values[-1]
        v[v.abs() < 0.01] = -0.0                     # signed zeros
        v[: 3 * k: 3] = top                          # ties at the threshold
        sc[2, 0] = v
    pos = torch.full((B, 1), 4 * N_cap - 1, dtype=torch.int32)
    if B > 3:
        pos[3, 0] = 4 * (k // 2) + 2                 # k // 2 visible entries
    d_sc, d_pos = sc.to(DEV), pos.to(DEV)
    idx = hattn.topk_select(d_sc, d_pos, k=k, m=4)
    idx2 = hattn.topk_select(d_sc, d_pos, k=k, m=4, dependent=True)  # twice: reused scratch
    hattn.check_status()
    _topk_ref_check(sc, pos, k, 4, idx)
    assert torch.equal(idx.sort(dim=-1).values, idx2.sort(dim=-1).values)


def test_topk_without_score_output_uses_workspace():
    B, T, HI, dI, N = 1, 1, 64, 128, 2048
    iq = randn_bf16((B, T, HI, dI), 40).to(DEV)
    w = randn_f32((B, T, HI), 41).to(DEV)
    ik = randn_bf16((B, N, dI), 42).to(DEV)
    pos = torch.tensor([[4 * N - 1]], dtype=torch.int32, device=DEV)
    a = hattn.indexer_topk(iq, w, ik, pos, k=64)
    s = torch.empty((B, T, N), device=DEV)
    b = hattn.indexer_topk(iq, w, ik, pos, k=64, score_out=s)
    assert sorted(a.cpu().flatten().tolist()) == sorted(b.cpu().flatten().tolist())


# ------------------------------------------------------------------ query preparation
@pytest.mark.parametrize("B,T,H,D,r", [(2, 3, 128, 512, 64), (1, 5, 4, 64, 16)])
def test_query_prep(B, T, H, D, r):
    q = randn_bf16((B, T, H, D), 45)
    gq = 1.0 + 0.1 * randn_f32((D,), 46)
    pos = _pos(B, T, [(7919 * i + 3) % (1 << 21) for i in range(B * T)])
    qt = hattn.query_prep(q.to(DEV), pos.to(DEV), r=r, gamma_q=gq.to(DEV))
    hattn.check_status()
    qf = f64(q)
    ref = np.empty_like(qf)
    for bb in range(B):
        for t in range(T):
            for hh in range(H):
                ref[bb, t, hh] = orc.rope(orc.rmsnorm(qf[bb, t, hh], gq.numpy()), r,
                                          int(pos[bb, t]))
    assert rel_l2(qt, ref) <= KV_REL_L2
    check_attn(qt, None, ref, None, "query prep")


# ------------------------------------------------------------------ attention branches
def _pos(B, T, values):
    return torch.tensor(values, dtype=torch.int32).reshape(B, T)


@pytest.mark.parametrize("B,T,H,D,r,N_cap,k", [
    (2, 2, 128, 512, 64, 300, 100),
    (1, 3, 4, 64, 16, 40, 16),
    (1, 2, 64, 512, 64, 2048, 512),
    (3, 1, 128, 512, 64, 5000, 1024),
])
def test_sparse_attn(B, T, H, D, r, N_cap, k):
    q = randn_bf16((B, T, H, D), 50)
    cache = randn_bf16((B, N_cap, D), 51)
    pos = _pos(B, T, [4 * N_cap - 1] * (B * T))
    nvis = np.full((B, T), N_cap)
    idx = synth.random_idx(B, T, k, nvis, seed=52, n_valid=max(1, k - 7))
    o, lse = hattn.sparse_attn(q.to(DEV), cache.to(DEV), idx.to(DEV), pos.to(DEV), r=r)
    hattn.check_status()
    ro, rl = orc.attention(orc.KIND_SPARSE, bits(q), bits(cache), pos.numpy(), idx=idx.numpy(),
                           r=r)
    check_attn(o, lse, ro, rl, "sparse")


def test_sparse_attn_all_padding_and_bad_index():
    B, T, H, D, N_cap, k = 1, 2, 8, 64, 50, 16
    q = randn_bf16((B, T, H, D), 53)
    cache = randn_bf16((B, N_cap, D), 54)
    idx = torch.full((B, T, k), -1, dtype=torch.int32)
    idx[0, 1, :3] = torch.tensor([5, 7, 9])
    pos = _pos(B, T, [199, 199])
    o, lse = hattn.sparse_attn(q.to(DEV), cache.to(DEV), idx.to(DEV), pos.to(DEV), r=16)
    hattn.check_status()
    assert torch.isinf(lse[0, 0]).all() and (lse[0, 0] < 0).all()
    assert (o[0, 0].float() == 0).all()
    ro, rl = orc.attention(orc.KIND_SPARSE, bits(q), bits(cache), pos.numpy(), idx=idx.numpy(),
                           r=16)
    check_attn(o[0, 1], lse[0, 1], ro[0, 1], rl[0, 1], "sparse short")
    idx[0, 1, 4] = N_cap + 3  # out of range: skipped and reported
    hattn.sparse_attn(q.to(DEV), cache.to(DEV), idx.to(DEV), pos.to(DEV), r=16)
    assert hattn.check_status_code() == hattn.DEVICE_INDEX


@pytest.mark.parametrize("B,T,H,D,r,N_cap,pos_list", [
    (2, 1, 128, 512, 64, 1000, [128 * 1000 - 1, 128 * 613 + 5]),   # ragged tail
    (1, 200, 4, 64, 16, 6, list(range(800 - 200, 800))),           # prefill, 32 q per block
    (1, 5, 128, 512, 64, 64, [100, 127, 128, 4000, 8191]),          # empty and short rows
])
def test_hca_attn(B, T, H, D, r, N_cap, pos_list):
    q = randn_bf16((B, T, H, D), 60)
    cache = randn_bf16((B, N_cap, D), 61)
    pos = _pos(B, T, pos_list)
    # entries that are not visible may hold anything, even NaN
    cdev = cache.to(DEV)
    nvis = [min((p + 1) // 128, N_cap) for p in pos_list]
    if B == 2:
        cdev[1, nvis[1]:] = float("nan")
    o, lse = hattn.hca_attn(q.to(DEV), cdev, pos.to(DEV), r=r, m=128)
    hattn.check_status()
    ro, rl = orc.attention(orc.KIND_HCA, bits(q), bits(cache), pos.numpy(), m=128, r=r)
    check_attn(o, lse, ro, rl, "hca")


@pytest.mark.parametrize("B,T,H,D,r,L,W,pos_list", [
    (2, 1, 128, 512, 64, 300, 128, [299, 150]),
    (1, 256, 4, 64, 16, 256, 128, list(range(256))),
    (1, 3, 64, 512, 64, 700, 128, [0, 64, 699]),
])
def test_swa_attn(B, T, H, D, r, L, W, pos_list):
    q = randn_bf16((B, T, H, D), 70)
    raw = randn_bf16((B, L, D), 71)
    gq = 1.0 + 0.1 * randn_f32((D,), 72)
    gk = 1.0 + 0.1 * randn_f32((D,), 73)
    pos = _pos(B, T, pos_list)
    o, lse = hattn.swa_attn(q.to(DEV), raw.to(DEV), pos.to(DEV), r=r, W=W, gamma_q=gq.to(DEV),
                            gamma_kv=gk.to(DEV))
    hattn.check_status()
    ro, rl = orc.attention(orc.KIND_SWA, bits(q), bits(raw), pos.numpy(), W=W, r=r,
                           gamma_q=gq.numpy(), gamma_kv=gk.numpy())
    check_attn(o, lse, ro, rl, "swa")


def test_lazy_rescale_path():
    """Keys ordered so the running max keeps growing across the tiles of one
    CTA (forces the tensor-memory rescale of O).  D=64 bounds the logits by 8;
    query and keys are spread over all dims, so values stay O(1) like real
    normalised latents.  150 sequences fill the SMs, so every row keeps all 10
    tiles in one split."""
    B, T, H, D, N = 150, 1, 4, 64, 640
    assert hattn.attn_workspace_bytes(hattn.KIND_HCA, B, T, H, D, N, q_prepped=True) == 0  # one split
    u = torch.zeros(D)
    u[: D // 2] = 1.0 / math.sqrt(D // 2)
    v = torch.zeros(D)
    v[D // 2:] = 1.0 / math.sqrt(D // 2)
    t = torch.linspace(-1.0, 1.0, N)
    keys = 8.0 * (t[:, None] * u[None] + torch.sqrt(1.0 - t ** 2)[:, None] * v[None])
    cache = keys[None].expand(B, N, D).contiguous().to(torch.bfloat16)
    q = u.expand(B, T, H, D).contiguous().to(torch.bfloat16)
    pos = _pos(B, T, [128 * N - 1] * B)
    o, lse = hattn.hca_attn(q.to(DEV), cache.to(DEV), pos.to(DEV), r=0, m=128)
    hattn.check_status()
    ro, rl = orc.attention(orc.KIND_HCA, bits(q[:2]), bits(cache[:2]), pos[:2].numpy(), m=128,
                           r=0)
    check_attn(o[:2], lse[:2], ro, rl, "rescale")


# ------------------------------------------------------------------ merge
@pytest.mark.parametrize("nb,with_sink,pos_list", [
    (3, True, [5, 77, 1 << 20, 3, 9, 123456]),
    (2, False, [5, 77, 1 << 20, 3, 9, 123456]),
    (1, True, [5, 77, 1 << 20, 3, 9, 123456]),
    # inverse RoPE at positions far beyond the cached context: the angle
    # reduction must stay exact up to the largest int32 position
    (2, True, [(1 << 31) - 1, (1 << 30) + 12345, (1 << 24) + 1, 4095, 4096, (1 << 28) - 3]),
])
def test_lse_merge(nb, with_sink, pos_list):
    B, T, H, D, r = 2, 3, 16, 512, 64
    os_ = [randn_f32((B, T, H, D), 80 + i) for i in range(nb)]
    ls = [randn_f32((B, T, H), 90 + i) * 3 for i in range(nb)]
    ls[0][0, 0, 0] = -float("inf")  # an empty branch row
    sink = randn_f32((H,), 99) if with_sink else None
    pos = _pos(B, T, pos_list)
    out, lse = hattn.lse_merge([o.to(DEV) for o in os_], [l.to(DEV) for l in ls], pos.to(DEV),
                               r=r, sink=sink.to(DEV) if sink is not None else None)
    ro, rl = orc.merge([f64(o) for o in os_], [f64(l) for l in ls],
                       sink.numpy() if sink is not None else None, pos.numpy(), r)
    check_attn(out, lse, ro, rl, "merge")


@pytest.mark.parametrize("B,H,D,r,N_hca,k,N_c,L", [
    (3, 128, 512, 64, 900, 300, 5000, 20480),     # decode: every branch split across SMs
    (1, 4, 64, 16, 40, 16, 60, 300),              # one split each
])
def test_merge_of_split_partials(B, H, D, r, N_hca, k, N_c, L):
    """Branches left as split partials (o = lse = NULL) and merged in one pass
    equal the oracle's merge of the branch outputs, and the combined path."""
    T = 1
    q = randn_bf16((B, T, H, D), 85)
    kv_h = randn_bf16((B, N_hca, D), 86)
    kv_c = randn_bf16((B, N_c, D), 87)
    raw = randn_bf16((B, L, D), 88)
    sink = randn_f32((H,), 89)
    pos = _pos(B, T, [min(128 * N_hca, 4 * N_c, L) - 1 - 7 * i for i in range(B)])
    nvis = np.array([[min((int(p) + 1) // 4, N_c)] for p in pos.ravel()]).reshape(B, T)
    idx = synth.random_idx(B, T, k, nvis, seed=90)
    d = dict(q=q.to(DEV), pos=pos.to(DEV))
    qt = hattn.query_prep(d["q"], d["pos"], r=r)
    parts = [hattn.sparse_attn(qt, kv_c.to(DEV), idx.to(DEV), d["pos"], r=r, q_prepped=True,
                               partials=True),
             hattn.hca_attn(qt, kv_h.to(DEV), d["pos"], r=r, q_prepped=True, partials=True),
             hattn.swa_attn(qt, raw.to(DEV), d["pos"], r=r, q_prepped=True, partials=True)]
    assert all(p.nsplit >= 1 for p in parts)
    out, lse = hattn.lse_merge_splits(parts, d["pos"], r=r, H=H, sink=sink.to(DEV))
    branches = [hattn.sparse_attn(qt, kv_c.to(DEV), idx.to(DEV), d["pos"], r=r, q_prepped=True),
                hattn.hca_attn(qt, kv_h.to(DEV), d["pos"], r=r, q_prepped=True),
                hattn.swa_attn(qt, raw.to(DEV), d["pos"], r=r, q_prepped=True)]
    out2, lse2 = hattn.lse_merge([o for o, _ in branches], [l for _, l in branches], d["pos"],
                                 r=r, sink=sink.to(DEV))
    hattn.check_status()
    qb, pn = bits(q), pos.numpy()
    ro = [orc.attention(orc.KIND_SPARSE, qb, bits(kv_c), pn, idx=idx.numpy(), r=r),
          orc.attention(orc.KIND_HCA, qb, bits(kv_h), pn, m=128, r=r),
          orc.attention(orc.KIND_SWA, qb, bits(raw), pn, W=128, r=r)]
    ref, rl = orc.merge([x[0] for x in ro], [x[1] for x in ro], sink.numpy(), pn, r)
    check_attn(out, lse, ref, rl, "merge of split partials")
    check_attn(out2, lse2, ref, rl, "merge of combined branches")


# ------------------------------------------------------------------ fused branches
@pytest.mark.parametrize("B,T,H,D,r,L,W", [
    (2, 3, 128, 512, 64, 300, 128),
    (1, 2, 4, 64, 16, 40, 96),
])
def test_swa_keys(B, T, H, D, r, L, W):
    """Each window row is the oracle's normalised, roped raw token (zero rows
    before token 0)."""
    raw = randn_bf16((B, L, D), 101)
    gk = 1.0 + 0.1 * randn_f32((D,), 102)
    pl = [L - 1, 5, L // 2][:T] * B
    pos = _pos(B, T, pl[:B * T])
    kv_w = hattn.swa_keys(raw.to(DEV), pos.to(DEV), r=r, W=W, gamma_kv=gk.to(DEV))
    hattn.check_status()
    got = f64(kv_w)
    for b in range(B):
        for t in range(T):
            p = int(pos[b, t])
            for j in range(W):
                u = p - W + 1 + j
                if u < 0:
                    assert (got[b, t, j] == 0).all()
                    continue
                if j % 17 and j != W - 1:
                    continue  # a sample of the rows
                ref = orc.rope(orc.rmsnorm(orc.bf16_to_f64(bits(raw[b, u])), gk.numpy()), r, u)
                assert rel_l2(got[b, t, j], ref) <= KV_REL_L2, (b, t, j)


@pytest.mark.parametrize("B,T,H,D,r,N_hca,k,N_c,L,pos_list", [
    # decode at full head width: every segment split across SMs, a ragged HCA tail
    (3, 1, 128, 512, 64, 900, 300, 5000, 20480, [20479, 20479 - 7 * 129, 11111]),
    # queries before the window is full, short HCA prefixes, one with none
    (2, 2, 128, 512, 64, 40, 64, 100, 400, [100, 127, 130, 399]),
    # fewer heads than MMA rows (one query per row block)
    (2, 1, 64, 512, 64, 100, 128, 300, 1300, [1299, 700]),
    # prefill-like: 96 queries, one key split each (the attention writes the
    # layer output itself), ragged windows and HCA prefixes
    (1, 96, 64, 512, 64, 40, 64, 1300, 5200, [5199 - 53 * i for i in range(96)]),
    (1, 80, 128, 512, 64, 30, 32, 1000, 4000, [3999 - 47 * i for i in range(80)]),
])
def test_hybrid_attn(B, T, H, D, r, N_hca, k, N_c, L, pos_list):
    """One softmax over the selected CSA entries, the HCA entries and the SWA
    window, merged with the sink, equals the oracle's merge of the three
    branches -- through the direct output, through the split partials, and
    straight to the layer output (hybrid_attn_out: written by the attention
    kernel when each query's keys take one split, else by a merge)."""
    q = randn_bf16((B, T, H, D), 91)
    kv_h = randn_bf16((B, N_hca, D), 92)
    kv_c = randn_bf16((B, N_c, D), 93)
    raw = randn_bf16((B, L, D), 94)
    sink = randn_f32((H,), 95)
    pos = _pos(B, T, pos_list)
    nvis = np.array([min((int(p) + 1) // 4, N_c) for p in pos.ravel()]).reshape(B, T)
    idx = synth.random_idx(B, T, k, nvis, seed=96)
    kvh_dev = kv_h.to(DEV)
    # HCA entries that are not visible to any query may hold anything
    nh = [min((int(p) + 1) // 128, N_hca) for p in pos.ravel()]
    for bb in range(B):
        top = max(nh[bb * T:(bb + 1) * T])
        kvh_dev[bb, top:] = float("nan")
    d = dict(q=q.to(DEV), pos=pos.to(DEV))
    qt = hattn.query_prep(d["q"], d["pos"], r=r)
    kv_w = hattn.swa_keys(raw.to(DEV), d["pos"], r=r, W=128)
    o, l = hattn.hybrid_attn(qt, kv_c.to(DEV), idx.to(DEV), kvh_dev, kv_w, d["pos"], r=r,
                             q_prepped=True)
    out, lse = hattn.lse_merge([o], [l], d["pos"], r=r, sink=sink.to(DEV))
    part = hattn.hybrid_attn(qt, kv_c.to(DEV), idx.to(DEV), kvh_dev, kv_w, d["pos"], r=r,
                             q_prepped=True, partials=True)
    out2, lse2 = hattn.lse_merge_splits([part], d["pos"], r=r, H=H, sink=sink.to(DEV))
    # the key sets in two calls (as the layer runs them beside the indexer):
    # HCA + SWA planned for a share of the SMs, then CSA; one merge of both
    dense = hattn.hybrid_attn(qt, None, None, kvh_dev, kv_w, d["pos"], r=r, k=k, q_prepped=True,
                              partials=True, segments=hattn.SEG_HCA | hattn.SEG_SWA, n_sms=40)
    sparse = hattn.hybrid_attn(qt, kv_c.to(DEV), idx.to(DEV), None, None, d["pos"], r=r, W=128,
                               q_prepped=True, partials=True, segments=hattn.SEG_CSA)
    out3, lse3 = hattn.lse_merge_splits([dense, sparse], d["pos"], r=r, H=H, sink=sink.to(DEV))
    out4, lse4 = hattn.hybrid_attn_out(qt, kv_c.to(DEV), idx.to(DEV), kvh_dev, kv_w, d["pos"],
                                       r=r, sink=sink.to(DEV), q_prepped=True)
    out5, lse5 = hattn.hybrid_attn_out(d["q"], kv_c.to(DEV), idx.to(DEV), kvh_dev, kv_w,
                                       d["pos"], r=r, dependent=True)
    # one key set alone (the branch kernels, finalised the same way)
    out6, lse6 = hattn.hybrid_attn_out(qt, None, None, kvh_dev, None, d["pos"], r=r, k=k, W=128,
                                       sink=sink.to(DEV), q_prepped=True,
                                       segments=hattn.SEG_HCA)
    out7, lse7 = hattn.hybrid_attn_out(qt, kv_c.to(DEV), idx.to(DEV), None, None, d["pos"], r=r,
                                       W=128, sink=sink.to(DEV), q_prepped=True,
                                       segments=hattn.SEG_CSA)
    hattn.check_status()
    qb, pn = bits(q), pos.numpy()
    ro = [orc.attention(orc.KIND_SPARSE, qb, bits(kv_c), pn, idx=idx.numpy(), r=r),
          orc.attention(orc.KIND_HCA, qb, bits(kv_h), pn, m=128, r=r),
          orc.attention(orc.KIND_SWA, qb, bits(raw), pn, W=128, r=r)]
    ref, rl = orc.merge([x[0] for x in ro], [x[1] for x in ro], sink.numpy(), pn, r)
    check_attn(out, lse, ref, rl, "fused, direct output")
    check_attn(out2, lse2, ref, rl, "fused, split partials")
    check_attn(out3, lse3, ref, rl, "fused, key sets in two calls")
    check_attn(out4, lse4, ref, rl, "fused, layer output")
    ref5, rl5 = orc.merge([x[0] for x in ro], [x[1] for x in ro], None, pn, r)
    check_attn(out5, lse5, ref5, rl5, "fused, layer output without a sink, raw queries")
    ref6, rl6 = orc.merge([ro[1][0]], [ro[1][1]], sink.numpy(), pn, r)
    check_attn(out6, lse6, ref6, rl6, "HCA alone, layer output")
    ref7, rl7 = orc.merge([ro[0][0]], [ro[0][1]], sink.numpy(), pn, r)
    check_attn(out7, lse7, ref7, rl7, "CSA alone, layer output")


def test_hybrid_attn_bad_index_is_reported():
    """An index past the CSA cache is skipped and reported, not read."""
    B, T, H, D, r = 1, 1, 128, 512, 64
    q = randn_bf16((B, T, H, D), 97).to(DEV)
    kv_c = randn_bf16((B, 64, D), 98).to(DEV)
    kv_h = randn_bf16((B, 8, D), 99).to(DEV)
    pos = _pos(B, T, [255]).to(DEV)
    idx = torch.full((B, T, 64), -1, dtype=torch.int32)
    idx[0, 0, :3] = torch.tensor([1, 64, 5])
    kv_w = hattn.swa_keys(randn_bf16((B, 256, D), 100).to(DEV), pos, r=r, W=128)
    hattn.hybrid_attn(q, kv_c, idx.to(DEV), kv_h, kv_w, pos, r=r)
    assert hattn.check_status_code() == hattn.DEVICE_INDEX


# ------------------------------------------------------------------ whole tiny layer
def test_tiny_layer_end_to_end():
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, 0)
    ref = orc.layer(synth.to_numpy(inp), wl.cfg(), keep=True)
    d = {k: v.to(DEV) for k, v in inp.items()}
    L = wl.L
    kv_c, ik_c = hattn.csa_compress(d["kv_raw"], d["ik_raw"], d["gate_csa"], r=wl.r)
    kv_h = hattn.hca_compress(d["kv_raw"], d["gate_hca"], r=wl.r)
    assert rel_l2(kv_c, ref["kv_c64"]) <= KV_REL_L2
    idx = hattn.indexer_topk(d["iq"], d["w"], ik_c, d["pos"], k=wl.k)
    o1, l1 = hattn.sparse_attn(d["q"], kv_c, idx, d["pos"], r=wl.r)
    o2, l2 = hattn.hca_attn(d["q"], kv_h, d["pos"], r=wl.r)
    o3, l3 = hattn.swa_attn(d["q"], d["kv_raw"], d["pos"], r=wl.r, W=wl.W)
    out, lse = hattn.lse_merge([o1, o2, o3], [l1, l2, l3], d["pos"], r=wl.r, sink=d["sink"])
    hattn.check_status()
    check_topk(idx.cpu().numpy(), ref["scores"], inp["pos"].numpy(), 4, wl.k, "tiny")
    check_attn(o3, l3, ref["o_swa"], ref["lse_swa"], "tiny swa")
    check_attn(o2, l2, ref["o_hca"], ref["lse_hca"], "tiny hca")
    check_attn(out, lse, ref["out"], ref["lse"], "tiny layer")
    assert L == 256


# ------------------------------------------------------------------ dependent launches
def test_dependent_launch_chain_matches_plain_launch():
    """The indexer -> top-k -> fused attention -> merge chain launched as
    programmatic dependents gives bit-identical results to plain launches
    (each kernel waits for its predecessor before reading its outputs)."""
    B, T, H, D, r, HI, dI, N_c, N_h, L, k = 2, 1, 128, 512, 64, 64, 128, 3000, 90, 12000, 256
    iq = randn_bf16((B, T, HI, dI), 111).to(DEV)
    w = randn_f32((B, T, HI), 112).to(DEV)
    ik = randn_bf16((B, N_c, dI), 113).to(DEV)
    kv_c = randn_bf16((B, N_c, D), 114).to(DEV)
    kv_h = randn_bf16((B, N_h, D), 115).to(DEV)
    raw = randn_bf16((B, L, D), 116).to(DEV)
    q = randn_bf16((B, T, H, D), 117).to(DEV)
    sink = randn_f32((H,), 118).to(DEV)
    pos = _pos(B, T, [11999, 9000]).to(DEV)
    qt = hattn.query_prep(q, pos, r=r)
    kv_w = hattn.swa_keys(raw, pos, r=r, W=128)
    torch.cuda.synchronize()

    def chain(dep):
        sc = hattn.indexer_scores(iq, w, ik, pos, m=4, dependent=dep)
        idx = hattn.topk_select(sc, pos, k=k, m=4, dependent=dep)
        # the selection comes in no fixed order; sorted, both runs attend to
        # the entries in the same order (and the attention waits for the sort)
        idx_s = idx.sort(dim=-1).values
        part = hattn.hybrid_attn(qt, kv_c, idx_s, kv_h, kv_w, pos, r=r, q_prepped=True,
                                 partials=True, dependent=dep)
        out, lse = hattn.lse_merge_splits([part], pos, r=r, H=H, sink=sink, dependent=dep)
        return sc, idx_s, out, lse

    plain = [t.clone() for t in chain(False)]
    torch.cuda.synchronize()
    dep = [t.clone() for t in chain(True)]
    torch.cuda.synchronize()
    hattn.check_status()
    sc0, idx0, out0, lse0 = plain
    sc1, idx1, out1, lse1 = dep
    vis = [min((int(p) + 1) // 4, N_c) for p in pos.cpu().ravel()]
    for bb in range(B):
        assert torch.equal(sc0[bb, 0, :vis[bb]], sc1[bb, 0, :vis[bb]])
    assert torch.equal(idx0, idx1)
    assert torch.equal(out0, out1)
    assert torch.equal(lse0, lse1)
