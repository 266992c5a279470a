"""Pins of the fp64 CPU oracle against things other than itself.

Each pin is a closed form, a special case that reduces to a library routine
(torch rms_norm / scaled_dot_product_attention / logsumexp), an invariant of
the definitions, or brute force on tiny inputs.  They are chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore")


def b16(x):
    """fp64 array -> bf16 bit patterns via torch's round-to-nearest-even."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(
        torch.float64).numpy()


# --------------------------------------------------------------------- bf16
def test_bf16_widening_exact(orc):
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000, 0x3EAB], np.uint16)
    ref = np.array([1.0, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -0.0,
                    0.333984375], np.float64)
    np.testing.assert_array_equal(orc.bf16_to_f64(bits), ref)


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [1.00390625, 1.01171875, -1.00390625, 3e-39, 1e-45]])
    x32 = x.astype(np.float32).astype(np.float64)  # torch rounds from fp32
    np.testing.assert_array_equal(orc.f64_to_bf16(x32), b16(x32))


# --------------------------------------------------------------------- RMSNorm
def test_rmsnorm_matches_torch(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 64))
    g = rng.standard_normal(64).astype(np.float32)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,),
                                       torch.from_numpy(g.astype(np.float64)), eps=1e-6).numpy()
    np.testing.assert_allclose(orc.rmsnorm(x, g, 1e-6), ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------- RoPE
def test_rope_hand_cases(orc):
    # pair 0 has theta = 1: e_{d0} at position 1 -> (cos 1, sin 1)
    x = orc.rope(np.array([0.0, 0.0, 1.0, 0.0]), 2, 1)
    np.testing.assert_allclose(x, [0, 0, math.cos(1), math.sin(1)], atol=1e-15)
    # interleaved pairing: e_{d0+1} -> (-sin p, cos p) in dims (d0, d0+1)
    x = orc.rope(np.array([5.0, 0.0, 1.0]), 2, 3)
    np.testing.assert_allclose(x, [5.0, -math.sin(3), math.cos(3)], atol=1e-15)
    # pair 1 of r=4 has theta = 10000^(-2/4) = 0.01: position 100 -> angle 1
    x = orc.rope(np.array([0.0, 0.0, 1.0, 0.0]), 4, 100)
    np.testing.assert_allclose(x, [0.0, 0.0, math.cos(1), math.sin(1)], atol=1e-13)


def test_rope_invariants(orc):
    rng = np.random.default_rng(3)
    D, r = 64, 16
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for p in [0, 1, 77, 1 << 20]:
        y = orc.rope(q, r, p)
        np.testing.assert_array_equal(y[:D - r], q[:D - r])          # untouched head
        assert abs(np.linalg.norm(y[D - r:]) - np.linalg.norm(q[D - r:])) < 1e-12
        np.testing.assert_allclose(orc.rope(y, r, p, sign=-1), q, atol=1e-9)
    # relative position: <R_a q, R_b k> depends only on a - b
    d1 = orc.rope(q, r, 1000) @ orc.rope(k, r, 990)
    d2 = orc.rope(q, r, 10) @ orc.rope(k, r, 0)
    assert abs(d1 - d2) < 1e-10


# --------------------------------------------------------------------- compressor
def test_compressor_hand_case(orc):
    # C(1,2), gates (0, g) over c0=(1,0), c1=(0,1): entry 1 = (a0, a1), then RMSNorm
    g = f64(b16([math.log(3.0)]))[0]
    kv = b16([[[1.0, 0.0], [0.0, 1.0]]])
    gate = b16([[0.0, g]])
    out, _, alpha = orc.compress(kv, gate, m=1, w=2, r=0, j_begin=1, j_end=2, eps=0.0)
    a1 = math.exp(g) / (1 + math.exp(g))
    a0 = 1 - a1
    rms = math.sqrt((a0 * a0 + a1 * a1) / 2)
    np.testing.assert_allclose(out[0, 0], [a0 / rms, a1 / rms], rtol=1e-14)
    np.testing.assert_allclose(alpha[0, 0], [a0, a1], rtol=1e-14)
    # with exact ln 3 these are the hand values 0.4472135955, 1.3416407865
    assert abs(a0 / rms - 0.4472135955) < 3e-3 and abs(a1 / rms - 1.3416407865) < 3e-3


def test_compressor_window_membership_brute_force(orc):
    """One-hot tokens + uniform gates: entry j = mean of exactly the tokens in
    [m(j+1)-w, m(j+1)-1] that exist (CSA: the 8 tokens [4j-4, 4j+4))."""
    for (m, w) in [(4, 8), (4, 4), (2, 6), (1, 1), (3, 3)]:
        L = 24
        kv = b16(np.eye(L)[None])          # token u = e_u, D = L
        ik = b16(np.eye(L)[None] * 2.0)
        gate = b16(np.zeros((1, L)))
        nj = L // m
        kvc, ikc, alpha = orc.compress(kv, gate, m, w, 0, 0, nj, ik_raw=ik, eps=0.0)
        for j in range(nj):
            members = [u for u in range(m * (j + 1) - w, m * (j + 1)) if u >= 0]
            pre = np.zeros(L)
            pre[members] = 1.0 / len(members)
            # RMSNorm of the mean: members get 1/len / rms
            rms = math.sqrt(np.mean(pre ** 2))
            np.testing.assert_allclose(kvc[0, j], pre / rms, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(ikc[0, j], 2 * pre, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(alpha[0, j].sum(), 1.0, rtol=1e-14)
            dropped = [s for s in range(w) if m * (j + 1) - w + s < 0]
            assert all(alpha[0, j, s] == 0 for s in dropped)


def test_compressor_gate_limits_and_constants(orc):
    rng = np.random.default_rng(4)
    L, D, dI = 16, 32, 8
    kv = b16(rng.standard_normal((1, L, D)))
    ik = b16(rng.standard_normal((1, L, dI)))
    # one dominating gate selects that token (softmax -> one-hot)
    gate = np.zeros((1, L))
    gate[0, 6] = 80.0
    kvc, ikc, _ = orc.compress(kv, b16(gate), 4, 8, 0, 1, 2, ik_raw=ik, eps=0.0)
    tok = f64(kv)[0, 6]
    np.testing.assert_allclose(kvc[0, 0], tok / math.sqrt(np.mean(tok ** 2)), rtol=1e-12)
    np.testing.assert_allclose(ikc[0, 0], f64(ik)[0, 6], rtol=1e-12)
    # constant tokens give the normalised constant, for any gates
    c = b16(np.tile(rng.standard_normal(D), (1, L, 1)))
    kvc, _, _ = orc.compress(c, b16(rng.standard_normal((1, L))), 4, 8, 0, 0, 4, eps=0.0)
    cv = f64(c)[0, 0]
    for j in range(4):
        np.testing.assert_allclose(kvc[0, j], cv / math.sqrt(np.mean(cv ** 2)), rtol=1e-12)


def test_compressor_rope_position_and_identity(orc):
    """C(1,1) is the identity before norm; entries are roped at m(j+1)-1."""
    rng = np.random.default_rng(5)
    L, D, r = 12, 16, 8
    kv = b16(rng.standard_normal((1, L, D)))
    gate = b16(rng.standard_normal((1, L)))
    c11, _, _ = orc.compress(kv, gate, 1, 1, r, 0, L)
    for u in range(L):
        ref = orc.rope(orc.rmsnorm(f64(kv)[0, u], None, 1e-6), r, u)
        np.testing.assert_allclose(c11[0, u], ref, rtol=1e-13, atol=1e-13)
    const = b16(np.tile(rng.standard_normal(D), (1, L, 1)))
    c4, _, _ = orc.compress(const, gate, 4, 8, r, 0, 3)
    base = orc.rmsnorm(f64(const)[0, 0], None, 1e-6)
    for j in range(3):
        np.testing.assert_allclose(c4[0, j], orc.rope(base, r, 4 * (j + 1) - 1), atol=1e-13)


# --------------------------------------------------------------------- indexer
def test_indexer_special_cases(orc):
    rng = np.random.default_rng(6)
    B, T, HI, dI, N, m = 1, 3, 3, 8, 5, 4
    iq = b16(rng.standard_normal((B, T, HI, dI)))
    ik = b16(rng.standard_normal((B, N, dI)))
    pos = np.array([[2, 3, 19]], np.int32)     # visible: 0, 1, 5
    q, k = f64(iq), f64(ik)
    for h in range(HI):                         # one-hot w picks relu(q_h . k_j)
        w = np.zeros((B, T, HI), np.float32)
        w[..., h] = 1.0
        s = orc.indexer_scores(iq, w, ik, pos, m)
        assert np.isnan(s[0, 0]).all()                       # t=2: nothing visible
        assert np.isnan(s[0, 1, 1:]).all()                   # t=3: only entry 0
        for t, nv in [(1, 1), (2, 5)]:
            ref = np.maximum(np.dot(k[0, :nv], q[0, t, h]), 0.0)
            np.testing.assert_allclose(s[0, t, :nv], ref, rtol=1e-14, atol=1e-14)
    # linear in w (including negative weights)
    w1 = rng.standard_normal((B, T, HI)).astype(np.float32)
    w2 = rng.standard_normal((B, T, HI)).astype(np.float32)
    s1 = orc.indexer_scores(iq, w1, ik, pos, m)
    s2 = orc.indexer_scores(iq, w2, ik, pos, m)
    s12 = orc.indexer_scores(iq, (w1.astype(np.float64) + w2).astype(np.float32), ik, pos, m)
    ok = ~np.isnan(s1)
    np.testing.assert_allclose(s12[ok], (s1 + s2)[ok], rtol=1e-5, atol=1e-5)


# --------------------------------------------------------------------- compressor from hidden states
def test_compress_hidden_with_identity_projection_is_compress(orc):
    """W = [I 0; 0 I] makes each projected row the hidden state itself, so the
    result equals the compressor over those rows exactly."""
    rng = np.random.default_rng(31)
    B, L, D, dI, r = 2, 40, 16, 8, 4
    x = b16(rng.standard_normal((B, L, D + dI)))
    gate = b16(rng.standard_normal((B, L)))
    W = b16(np.eye(D + dI))
    kv, ik = orc.compress_hidden(x, W, gate, 4, 8, r, 0, L // 4, D)
    rk, ri, _ = orc.compress(np.ascontiguousarray(x[..., :D]), gate, 4, 8, r, 0, L // 4,
                             ik_raw=np.ascontiguousarray(x[..., D:]))
    np.testing.assert_array_equal(kv, rk)
    np.testing.assert_array_equal(ik, ri)


def test_compress_hidden_single_token_window_is_norm_of_projection(orc):
    """With m = w = 1 the entry of token u is RMSNorm(x_u . W_kv), roped at
    u, and its indexer key x_u . W_ik: compared with torch's fp64 matmul and
    rms_norm and the (separately pinned) RoPE."""
    rng = np.random.default_rng(32)
    B, L, dm, D, dI, r = 1, 6, 24, 16, 8, 4
    x = b16(rng.standard_normal((B, L, dm)))
    W = b16(rng.standard_normal((dm, D + dI)) / np.sqrt(dm))
    gate = b16(rng.standard_normal((B, L)))
    kv, ik = orc.compress_hidden(x, W, gate, 1, 1, r, 0, L, D)
    y = torch.from_numpy(f64(x)) @ torch.from_numpy(f64(W))
    ref_kv = torch.nn.functional.rms_norm(y[..., :D], (D,), eps=1e-6).numpy()
    for u in range(L):
        np.testing.assert_allclose(kv[0, u], orc.rope(ref_kv[0, u], r, u), rtol=1e-12,
                                   atol=1e-12)
    np.testing.assert_allclose(ik, y[..., D:].numpy(), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------- FP8 (E4M3) keys
def _torch_e4m3(x32):
    """torch's float8_e4m3fn cast (nearest even, NaN past 464) as uint8 codes."""
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_table():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_and_rounding_match_torch(orc):
    """Decoding of every finite code, and nearest-even encoding of the code
    values, of the midpoints between neighbouring codes (the ties), and of
    random magnitudes over the whole range, against torch's float8_e4m3fn
    (an independent implementation), where torch does not overflow."""
    table = _e4m3_table()
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    np.testing.assert_array_equal(orc.e4m3_to_f64(finite), table[finite])
    mags = np.unique(np.abs(table[finite]))
    mids = (mags[1:] + mags[:-1]) / 2
    rng = np.random.default_rng(21)
    rnd = rng.standard_normal(20000) * 2.0 ** rng.integers(-14, 10, 20000)
    x = np.concatenate([table[finite], mids, -mids, rnd])
    x32 = x.astype(np.float32)
    x32 = x32[np.abs(x32) <= 464]
    np.testing.assert_array_equal(orc.f32_to_e4m3(x32), _torch_e4m3(x32))


def test_e4m3_hand_cases(orc):
    cases = [(448.0, 0x7E), (1.0, 0x38), (-1.0, 0xB8), (2.0 ** -9, 0x01), (2.0 ** -6, 0x08),
             (2.0 ** -10, 0x00),            # half the smallest subnormal: tie to even 0
             (3 * 2.0 ** -10, 0x02),        # 1.5 subnormal steps: tie to even 2
             (1.0625, 0x38), (1.1875, 0x3A),  # ties between 1, 1.125 and 1.25
             (240.0, 0x77), (500.0, 0x7E), (-1e30, 0xFE), (math.inf, 0x7E)]
    for x, code in cases:
        assert int(orc.f32_to_e4m3(np.float32(x))) == code, x


def test_e4m3_row_quantisation(orc):
    """Per-row scale amax/448, the largest element on +-448, the codes of
    x * (448/amax) rounded by torch's cast, and every dequantised value
    within half an E4M3 step of the input; a zero row has scale 0."""
    rng = np.random.default_rng(22)
    xv64 = rng.standard_normal((60, 128)) * 10.0 ** rng.integers(-3, 4, (60, 1))
    x = b16(xv64)
    xv = f64(x)
    codes, scales = orc.quantize_e4m3(x)
    amax = np.abs(xv).max(-1).astype(np.float32)
    np.testing.assert_array_equal(scales, amax / np.float32(448))
    top = np.abs(xv).argmax(-1)
    assert ((codes[np.arange(60), top] & 0x7F) == 0x7E).all()
    inv = np.float32(448) / amax
    np.testing.assert_array_equal(codes, _torch_e4m3(xv.astype(np.float32) * inv[:, None]))
    deq = orc.dequantize_e4m3(codes, scales)
    bound = np.maximum(np.abs(xv) * 2.0 ** -4, 2.0 ** -10 * scales[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - xv) <= bound).all()
    c0, s0 = orc.quantize_e4m3(np.zeros((1, 128), np.uint16))
    assert (c0 == 0).all() and s0[0] == 0


def test_indexer_e4m3_exact_rows_equal_bf16_scores(orc):
    """Rows of multiples of 1/2 with largest magnitude 3.5 quantise without
    loss (scale 2^-7, codes on 64..448), so the FP8 scores equal the bf16
    scores exactly; scaling a key row by a power of two scales its scores by
    the same factor (the key scale enters once, ReLU is homogeneous)."""
    rng = np.random.default_rng(23)
    B, T, HI, dI, N, m = 2, 3, 4, 128, 9, 4

    def rows(shape):
        v = rng.integers(-7, 8, shape).astype(np.float64) / 2
        v[..., 0] = np.where(rng.random(shape[:-1]) < 0.5, 3.5, -3.5)
        return v

    iq, ik = b16(rows((B, T, HI, dI))), b16(rows((B, N, dI)))
    w = rng.standard_normal((B, T, HI)).astype(np.float32)
    pos = np.array([[3, 20, 35], [7, 11, 2]], np.int32)
    ik8, iks = orc.quantize_e4m3(ik)
    assert (iks == np.float32(2.0 ** -7)).all()
    s_bf = orc.indexer_scores(iq, w, ik, pos, m)
    s_8 = orc.indexer_scores_e4m3(iq, w, ik8, iks, pos, m)
    np.testing.assert_array_equal(np.isnan(s_8), np.isnan(s_bf))
    ok = ~np.isnan(s_bf)
    np.testing.assert_array_equal(s_8[ok], s_bf[ok])
    iks2 = iks.copy()
    iks2[1, 2] *= 8
    s_2 = orc.indexer_scores_e4m3(iq, w, ik8, iks2, pos, m)
    want = s_8.copy()
    want[1, :, 2] *= 8
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(s_2[ok], want[ok])


# --------------------------------------------------------------------- MXFP4 (E2M1) rows
# The E2M1 element magnitudes of codes 0..7 as the OCP Microscaling Formats
# specification v1.0 tabulates them (FP4 E2M1: max normal 6, min normal 1,
# max subnormal 0.5); code bit 3 is the sign.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_brute(y):
    """Nearest table value by exhaustive search: the smallest |y - v| over
    the 8 magnitudes, ties to the even code, sign from y, +0 for zero."""
    out = np.empty(np.shape(y), np.uint8)
    for idx, v in np.ndenumerate(np.asarray(y, np.float64)):
        a = min(abs(v), 6.0)
        err = [abs(a - t) for t in E2M1_MAGNITUDES]
        best = min(err)
        cands = [c for c in range(8) if err[c] == best]
        c = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out[idx] = c | (8 if (v < 0 and c) else 0)
    return out


def test_e2m1_decode_table(orc):
    codes = np.arange(16, dtype=np.uint8)
    want = np.array(E2M1_MAGNITUDES + [-v for v in E2M1_MAGNITUDES])
    np.testing.assert_array_equal(orc.e2m1_to_f64(codes), want)


def test_e2m1_rounding_brute_force(orc):
    """Every table value, every midpoint between neighbours (the ties), values
    just either side of them, saturation beyond 6, and random values, against
    the exhaustive nearest-value search."""
    mags = np.array(E2M1_MAGNITUDES)
    mids = (mags[1:] + mags[:-1]) / 2
    near = np.concatenate([mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20)])
    rng = np.random.default_rng(24)
    y = np.concatenate([mags, mids, near, [6.5, 7.0, 7.999, 1e3, 1e-30, 0.0],
                        rng.uniform(-8, 8, 3000), rng.standard_normal(500) * 1e-2])
    y = np.concatenate([y, -y])
    np.testing.assert_array_equal(orc.f64_to_e2m1(y), _e2m1_brute(y))
    # the ties by hand: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2,
    # 3.5 -> 4, 5 -> 4 (each to the code with an even low bit)
    np.testing.assert_array_equal(orc.f64_to_e2m1(mids), [0, 2, 2, 4, 4, 6, 6])
    assert int(orc.f64_to_e2m1(-0.1)) == 0 and int(orc.f64_to_e2m1(-0.3)) == 9


def test_e8m0_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = orc.e8m0_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_array_equal(got[:255], want[:255])


def test_mxfp4_row_quantisation(orc):
    """Per 32-element block: the scale exponent is floor(log2 amax) - 2 (read
    here from the fp32 exponent field), so amax / X lies in [4, 8); the codes
    are the brute-force nearest values of x / X; nibble order is element 2i
    low; every dequantised value lies within a quarter of (|x| + X) of x;
    an all-zero block takes scale code 0 and zero codes."""
    rng = np.random.default_rng(25)
    rows, n = 24, 128
    xv64 = rng.standard_normal((rows, n)) * 10.0 ** rng.integers(-6, 7, (rows, n // 32)).repeat(
        32, axis=1)
    xv64[2, 32:64] = 0.0
    x = b16(xv64)
    xv = f64(x)
    codes, scales = orc.quantize_mxfp4(x)
    assert codes.shape == (rows, n // 2) and scales.shape == (rows, n // 32)
    blocks = xv.reshape(rows, n // 32, 32)
    amax = np.abs(blocks).max(-1)
    expo = ((amax.astype(np.float32).view(np.uint32) >> 23) & 0xFF).astype(np.int64) - 127
    want_scale = np.where(amax > 0, expo - 2 + 127, 0)
    np.testing.assert_array_equal(scales, want_scale)
    X = 2.0 ** (scales.astype(np.float64) - 127)
    live = amax > 0
    ratio = amax[live] / X[live]
    assert ((ratio >= 4) & (ratio < 8)).all()
    y = blocks / X[..., None]
    want_codes = _e2m1_brute(y).reshape(rows, n)
    np.testing.assert_array_equal(codes & 15, want_codes[:, 0::2])
    np.testing.assert_array_equal(codes >> 4, want_codes[:, 1::2])
    deq = orc.dequantize_mxfp4(codes, scales)
    Xe = np.repeat(X, 32, axis=1)
    assert (np.abs(deq - xv) <= (np.abs(xv) + Xe) / 4).all()
    assert scales[2, 1] == 0 and (codes[2, 16:32] == 0).all()


def _mx_exact_rows(rng, shape):
    """Rows whose blocks are table values times a per-block power of two,
    with one element of each block at +-4 or +-6 times it: MXFP4 holds them
    exactly (amax / X is 4 or 6)."""
    n = shape[-1]
    nb = n // 32
    v = rng.choice(E2M1_MAGNITUDES, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    lead = rng.choice([4.0, 6.0], size=shape[:-1] + (nb,)) * rng.choice([-1.0, 1.0],
                                                                        size=shape[:-1] + (nb,))
    v = v.reshape(shape[:-1] + (nb, 32))
    v[..., 0] = lead
    v *= 2.0 ** rng.integers(-6, 4, size=shape[:-1] + (nb, 1))
    return v.reshape(shape)


def test_indexer_mxfp4_exact_rows_equal_bf16_scores(orc):
    """Rows that MXFP4 holds exactly (block scales differing within a row, so
    a block scale applied to the wrong elements, or swapped nibbles, changes
    the values) give MXFP4 scores equal to the bf16 scores; raising one key
    row's four block scales by 3 multiplies its scores by 8."""
    rng = np.random.default_rng(26)
    B, T, HI, dI, N, m = 2, 3, 4, 128, 9, 4
    iq = b16(_mx_exact_rows(rng, (B, T, HI, dI)))
    ik = b16(_mx_exact_rows(rng, (B, N, dI)))
    w = rng.standard_normal((B, T, HI)).astype(np.float32)
    pos = np.array([[3, 20, 35], [7, 11, 2]], np.int32)
    ik4, iks = orc.quantize_mxfp4(ik)
    np.testing.assert_array_equal(orc.dequantize_mxfp4(ik4, iks), f64(ik))
    s_bf = orc.indexer_scores(iq, w, ik, pos, m)
    s_4 = orc.indexer_scores_mxfp4(iq, w, ik4, iks, pos, m)
    np.testing.assert_array_equal(np.isnan(s_4), np.isnan(s_bf))
    ok = ~np.isnan(s_bf)
    np.testing.assert_array_equal(s_4[ok], s_bf[ok])
    iks2 = iks.copy()
    iks2[1, 2] += 3
    s_2 = orc.indexer_scores_mxfp4(iq, w, ik4, iks2, pos, m)
    want = s_4.copy()
    want[1, :, 2] *= 8
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(s_2[ok], want[ok])
    # a query MXFP4 does not hold: it is scored as its quantised value (which
    # bf16 holds exactly: two significant bits times a power of two)
    iq_r = b16(rng.standard_normal((B, T, HI, dI)))
    qc, qs = orc.quantize_mxfp4(iq_r)
    iq_d = b16(orc.dequantize_mxfp4(qc, qs))
    np.testing.assert_array_equal(f64(iq_d), orc.dequantize_mxfp4(qc, qs))
    assert not np.array_equal(iq_d, iq_r)
    s_r = orc.indexer_scores_mxfp4(iq_r, w, ik4, iks, pos, m)
    s_d = orc.indexer_scores(iq_d, w, ik, pos, m)
    ok = ~np.isnan(s_d)
    np.testing.assert_array_equal(s_r[ok], s_d[ok])


# --------------------------------------------------------------------- top-k
def _pairwise_rule_ok(sc, chosen, n):
    ch = set(chosen)
    for i in ch:
        for j in range(n):
            if j in ch:
                continue
            if not (sc[i] > sc[j] or (sc[i] == sc[j] and i < j)):
                return False
    return True


def test_topk_brute_force_with_ties(orc):
    rng = np.random.default_rng(7)
    for trial in range(300):
        n = int(rng.integers(1, 11))
        k = int(rng.integers(1, 5))
        sc = rng.integers(-3, 4, n).astype(np.float64)        # many ties
        pos = np.array([4 * n - 1], np.int32)                 # m=4: n visible
        idx = orc.topk(sc[None], pos, 4, k)[0]
        keff = min(k, n)
        assert (idx[keff:] == -1).all()
        chosen = list(idx[:keff])
        assert len(set(chosen)) == keff
        best = max(sum(sc[list(c)]) for c in itertools.combinations(range(n), keff))
        assert sum(sc[chosen]) == best
        assert _pairwise_rule_ok(sc, chosen, n)


def test_topk_planted(orc):
    N = 1000
    sc = np.linspace(-1, 1, N)[np.random.default_rng(8).permutation(N)]
    top = np.argsort(-sc)[:10]
    idx = orc.topk(sc[None], np.array([4 * N - 1], np.int32), 4, 10)[0]
    np.testing.assert_array_equal(idx, top)
    # visibility: a query at t sees only (t+1)//4 entries
    idx = orc.topk(sc[None], np.array([4 * 7 + 2], np.int32), 4, 10)[0]
    assert sorted(idx[:7]) == list(range(7)) and (idx[7:] == -1).all()


# --------------------------------------------------------------------- attention
def _sdpa(qt, keys, causal_lens=None):
    """Library reference: torch SDPA in fp64 with V = K, plus logsumexp."""
    q = torch.from_numpy(qt)[None, None]          # [1,1,1,D]
    k = torch.from_numpy(keys)[None, None]        # [1,1,n,D]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, k)[0, 0, 0].numpy()
    lg = (q @ k.transpose(-1, -2))[0, 0, 0] / math.sqrt(qt.shape[0])
    return o, torch.logsumexp(lg, 0).item()


def _prep_q(orc, q, r, t):
    return orc.rope(torch.nn.functional.rms_norm(torch.from_numpy(q), (q.shape[0],),
                                                 eps=1e-6).numpy(), r, t)


def test_csa_with_large_k_is_dense_attention(orc):
    rng = np.random.default_rng(9)
    B, T, H, D, r, N = 1, 3, 2, 32, 8, 20
    cache = b16(rng.standard_normal((B, N, D)))
    q = b16(rng.standard_normal((B, T, H, D)))
    pos = np.array([[15, 40, 83]], np.int32)          # m=4 -> 4, 10, 20 visible
    idx = np.full((B, T, 32), -1, np.int32)
    for t in range(T):
        nv = min((pos[0, t] + 1) // 4, N)
        idx[0, t, :nv] = rng.permutation(nv)
    o, l = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=idx, r=r)
    oh, lh = orc.attention(orc.KIND_HCA, q, cache, pos, m=4, r=r)
    keys = f64(cache)[0]
    for t in range(T):
        nv = min((pos[0, t] + 1) // 4, N)
        for h in range(H):
            ref_o, ref_l = _sdpa(_prep_q(orc, f64(q)[0, t, h], r, pos[0, t]), keys[:nv])
            np.testing.assert_allclose(o[0, t, h], ref_o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(oh[0, t, h], ref_o, rtol=1e-12, atol=1e-12)
            assert abs(l[0, t, h] - ref_l) < 1e-12 and abs(lh[0, t, h] - ref_l) < 1e-12


def test_m1_uniform_gates_and_large_window_are_causal_attention(orc):
    """C(1,1) + CSA with k >= visible, and SWA with W >= L, both equal standard
    causal attention over the normalised, roped tokens (torch SDPA, is_causal)."""
    rng = np.random.default_rng(10)
    B, L, H, D, r = 1, 24, 2, 32, 8
    raw = b16(rng.standard_normal((B, L, D)))
    q = b16(rng.standard_normal((B, L, H, D)))
    pos = np.arange(L, dtype=np.int32)[None]
    c11, _, _ = orc.compress(raw, b16(np.zeros((B, L))), 1, 1, r, 0, L)
    cache = orc.f64_to_bf16(c11)
    idx = np.tile(np.arange(L, dtype=np.int32), (B, L, 1))
    idx[np.arange(L)[None, :, None] < np.arange(L)[None, None, :]] = -1
    o_csa, l_csa = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=idx, r=r)
    o_swa, l_swa = orc.attention(orc.KIND_SWA, q, raw, pos, W=L + 5, r=r)
    keys_csa = f64(cache)[0]
    keys_swa = np.stack([orc.rope(orc.rmsnorm(f64(raw)[0, u], None, 1e-6), r, u)
                         for u in range(L)])
    qq = np.stack([[_prep_q(orc, f64(q)[0, t, h], r, t) for t in range(L)] for h in range(H)])
    for keys, o in [(keys_csa, o_csa), (keys_swa, o_swa)]:
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qq)[None], torch.from_numpy(keys)[None, None].expand(1, H, L, D),
            torch.from_numpy(keys)[None, None].expand(1, H, L, D), is_causal=True)[0]
        np.testing.assert_allclose(o[0].transpose(1, 0, 2), ref.numpy(), rtol=1e-11, atol=1e-11)


def test_hand_cases_two_and_three_tokens(orc):
    """D=2, r=0, eps=0, H=1, s=1/sqrt(2), sink 0 (closed forms)."""
    s2 = math.sqrt(2.0)
    raw = b16([[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]])
    q = b16([[[[1.0, 0.0]]]])
    sink = np.array([0.0], np.float32)
    # 2 tokens, query at t=1: logits (sqrt2, 0)
    o, l = orc.attention(orc.KIND_SWA, q, raw, np.array([[1]], np.int32), W=128, eps=0.0)
    out, lse = orc.merge([o], [l], sink, np.array([[1]], np.int32), 0)
    z = math.exp(s2) + 1 + 1
    w0, w1 = math.exp(s2) / z, 1 / z
    np.testing.assert_allclose(out[0, 0, 0], [w0 * s2, w1 * s2], rtol=1e-13)
    assert abs(lse[0, 0, 0] - math.log(z)) < 1e-13
    np.testing.assert_allclose([w0, w1, out[0, 0, 0, 0], out[0, 0, 0, 1], lse[0, 0, 0]],
                               [0.6728417984, 0.1635791008, 0.9515419966, 0.2313357829,
                                1.8104586086], atol=1e-9)
    out_ns, _ = orc.merge([o], [l], None, np.array([[1]], np.int32), 0)   # no sink
    np.testing.assert_allclose(out_ns[0, 0, 0], [1.1376353670, 0.2765781954], atol=1e-9)
    # 3 tokens, query at t=2: logits (sqrt2, 0, 1), keys (sqrt2,0), (0,sqrt2), (1,1)
    o, l = orc.attention(orc.KIND_SWA, q, raw, np.array([[2]], np.int32), W=128, eps=0.0)
    out, lse = orc.merge([o], [l], sink, np.array([[2]], np.int32), 0)
    z = math.exp(s2) + 1 + math.e + 1
    ref = np.array([math.exp(s2) * s2 + math.e, s2 + math.e]) / z
    np.testing.assert_allclose(out[0, 0, 0], ref, rtol=1e-13)
    np.testing.assert_allclose([out[0, 0, 0, 0], out[0, 0, 0, 1], lse[0, 0, 0]],
                               [0.9664570201, 0.4679250773, 2.1783285225], atol=1e-9)
    # window 2: only tokens 1 and 2
    o, l = orc.attention(orc.KIND_SWA, q, raw, np.array([[2]], np.int32), W=2, eps=0.0)
    out, _ = orc.merge([o], [l], sink, np.array([[2]], np.int32), 0)
    np.testing.assert_allclose(out[0, 0, 0], [0.5761168848, 0.8758475100], atol=1e-9)


def test_weights_plus_sink_sum_to_one(orc):
    rng = np.random.default_rng(11)
    D, n = 16, 9
    keys = rng.standard_normal((n, D))
    qt = rng.standard_normal(D)
    for sink in [-5.0, 0.0, 3.0]:
        w, ws = orc.weights_with_sink(qt, keys, 1 / 4.0, sink)
        assert abs(w.sum() + ws - 1.0) < 1e-12
        # the merged output agrees: sink only enlarges the denominator
        lg = keys @ qt / 4.0
        ref = (np.exp(lg)[:, None] * keys).sum(0) / (np.exp(lg).sum() + math.exp(sink))
        np.testing.assert_allclose((w[:, None] * keys).sum(0), ref, rtol=1e-12)


def test_merge_of_split_equals_union(orc):
    """LSE merge of two disjoint key sets equals attention over their union."""
    rng = np.random.default_rng(12)
    B, T, H, D, r, N = 2, 2, 3, 32, 8, 40
    cache = b16(rng.standard_normal((B, N, D)))
    q = b16(rng.standard_normal((B, T, H, D)))
    pos = np.full((B, T), 4 * N - 1, np.int32)
    sink = rng.standard_normal(H).astype(np.float32)
    for trial in range(3):
        perm = np.stack([np.stack([rng.permutation(N) for _ in range(T)]) for _ in range(B)])
        cut = int(rng.integers(1, N))
        a = np.full((B, T, N), -1, np.int32)
        b_ = np.full((B, T, N), -1, np.int32)
        a[..., :cut] = perm[..., :cut]
        b_[..., :N - cut] = perm[..., cut:]
        oa, la = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=a, r=r)
        ob, lb = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=b_, r=r)
        ou, lu = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=perm.astype(np.int32), r=r)
        m2, l2 = orc.merge([oa, ob], [la, lb], sink, pos, r)
        m1, l1 = orc.merge([ou], [lu], sink, pos, r)
        np.testing.assert_allclose(m2, m1, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(l2, l1, rtol=1e-12)


def test_merge_inverse_rope_and_empty_branch(orc):
    rng = np.random.default_rng(13)
    B, T, H, D, r = 1, 2, 2, 16, 8
    o = rng.standard_normal((B, T, H, D))
    l = rng.standard_normal((B, T, H))
    pos = np.array([[5, 1000]], np.int32)
    out, lse = orc.merge([o], [l], None, pos, r)
    for t in range(T):
        for h in range(H):
            np.testing.assert_allclose(orc.rope(out[0, t, h], r, pos[0, t]), o[0, t, h],
                                       atol=1e-12)
    np.testing.assert_allclose(lse, l, rtol=1e-14)
    # an empty branch (lse = -inf, o = 0) changes nothing
    out2, lse2 = orc.merge([o, np.zeros_like(o)], [l, np.full_like(l, -np.inf)], None, pos, r)
    np.testing.assert_allclose(out2, out, rtol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14)


def test_layer_composition_reduces_to_causal_attention(orc):
    """The whole layer (compress, bf16 storage, indexer, top-k, branches,
    sink merge, inverse RoPE) with C(1,1) for both compressors, k and W at
    least L and no sink: every branch is standard causal attention over the
    normalised, roped tokens (torch SDPA, is_causal), rotated back by the
    query position.  Two identical branches merge to the same output with
    lse + ln 2; a finite sink s scales the output by 1 / (1 + e^(s - lse))."""
    from sparse_attention_26_b300 import synth
    wl = synth.scaled(synth.WORKLOADS["tiny"], L=40, T=40, H=2, D=32, r=8, HI=2, dI=16, k=64)
    inp = synth.to_numpy(synth.make_inputs(wl, 3))
    inp.pop("sink")
    cfg = dict(wl.cfg(), m_csa=1, w_csa=1, m_hca=1, w_hca=1, k=64, W=64, r=8)
    L, H, D, r = 40, 2, 32, 8
    raw = f64(inp["kv_raw"])[0]
    keys64 = np.stack([orc.rope(orc.rmsnorm(raw[u], None, 1e-6), r, u) for u in range(L)])
    keys16 = f64(orc.f64_to_bf16(keys64))
    qq = np.stack([[_prep_q(orc, f64(inp["q"])[0, t, h], r, t) for t in range(L)]
                   for h in range(H)])

    def reference(keys):
        kt = torch.from_numpy(keys)[None, None].expand(1, H, L, D)
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qq)[None], kt, kt, is_causal=True)[0].numpy()   # [H, L, D]
        lg = torch.from_numpy(qq) @ torch.from_numpy(keys).T / math.sqrt(D)
        lg = lg.masked_fill(torch.triu(torch.ones(L, L, dtype=torch.bool), 1), -math.inf)
        lse = torch.logsumexp(lg, -1).numpy()                                # [H, L]
        out = np.stack([[orc.rope(o[h, t], r, t, sign=-1) for h in range(H)] for t in range(L)])
        return out, lse.T

    ref16, lse16 = reference(keys16)
    ref64, lse64 = reference(keys64)
    for branches, ref, lse_ref in [(("csa",), ref16, lse16), (("hca",), ref16, lse16),
                                   (("swa",), ref64, lse64)]:
        res = orc.layer(inp, cfg, branches=branches)
        np.testing.assert_allclose(res["out"][0], ref, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(res["lse"][0], lse_ref, rtol=1e-10, atol=1e-10)
    both = orc.layer(inp, cfg, branches=("csa", "hca"))
    np.testing.assert_allclose(both["out"][0], ref16, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(both["lse"][0], lse16 + math.log(2), rtol=1e-10, atol=1e-10)
    sink = np.array([0.5, -1.5], np.float32)
    sunk = orc.layer(dict(inp, sink=sink), cfg, branches=("swa",))
    factor = 1 / (1 + np.exp(sink.astype(np.float64)[None, :] - lse64))    # [L, H]
    np.testing.assert_allclose(sunk["out"][0], ref64 * factor[..., None], rtol=1e-10,
                               atol=1e-10)
    np.testing.assert_allclose(sunk["lse"][0], np.logaddexp(lse64, sink[None, :]), rtol=1e-10,
                               atol=1e-10)
    # k = 4 < visible: the CSA branch attends to the 4 best-scored entries.
    # C(1,1) leaves an indexer key as its token, so the scores are those of
    # the raw keys; numpy's sort picks the 4 (score descending, index
    # ascending) and torch SDPA attends to them.
    k = 4
    sel = orc.layer(inp, dict(cfg, k=k), branches=("csa",))
    sc = orc.indexer_scores(inp["iq"], inp["w"], inp["ik_raw"], inp["pos"], 1)[0]
    for t in range(L):
        n = t + 1
        pick = np.lexsort((np.arange(n), -sc[t, :n]))[:k]
        kt = torch.from_numpy(keys16[pick])[None]
        for h in range(H):
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(qq[h, t])[None, None], kt, kt)[0, 0].numpy()
            np.testing.assert_allclose(sel["out"][0, t, h], orc.rope(o, r, t, sign=-1),
                                       rtol=1e-10, atol=1e-10)


def test_degenerate_cases(orc):
    """Nothing to attend: an HCA query before the first entry is complete
    (t < m - 1) and a CSA query whose indices are all padding both give
    o = 0 and lse = -inf; top-k over no visible entry is all padding; a
    merge of empty branches gives 0 and lse = -inf without a sink, and 0 with
    lse = s with a sink s (the sink takes all the weight)."""
    rng = np.random.default_rng(31)
    B, T, H, D, r = 1, 2, 2, 32, 8
    q = b16(rng.standard_normal((B, T, H, D)))
    cache = b16(rng.standard_normal((B, 4, D)))
    pos = np.array([[0, 126]], np.int32)
    o, l = orc.attention(orc.KIND_HCA, q, cache, pos, m=128, r=r)
    assert (o == 0).all() and np.isneginf(l).all()
    idx = np.full((B, T, 8), -1, np.int32)
    o2, l2 = orc.attention(orc.KIND_SPARSE, q, cache, pos, idx=idx, r=r)
    assert (o2 == 0).all() and np.isneginf(l2).all()
    sc = np.full((2, 16), np.nan)
    top = orc.topk(sc, np.array([2, 0], np.int32), 4, 5)
    assert (top == -1).all()
    out, lse = orc.merge([o, o2], [l, l2], None, pos, r)
    assert (out == 0).all() and np.isneginf(lse).all()
    sink = np.array([0.25, -2.0], np.float32)
    out, lse = orc.merge([o, o2], [l, l2], sink, pos, r)
    assert (out == 0).all()
    np.testing.assert_array_equal(lse[0], np.tile(sink.astype(np.float64), (T, 1)))


def test_tiny_layer_runs(orc):
    from sparse_attention_26_b300 import synth
    wl = synth.WORKLOADS["tiny"]
    inp = synth.to_numpy(synth.make_inputs(wl, 0))
    res = orc.layer(inp, wl.cfg(), keep=True)
    assert np.isfinite(res["out"]).all()
    assert res["idx"].shape == (1, 256, 16)
    # early queries see fewer than k entries: padded with -1
    assert (res["idx"][0, 10, 2:] == -1).all() and (res["idx"][0, 10, :2] >= 0).all()
