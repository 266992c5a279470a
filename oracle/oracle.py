"""ctypes wrapper of the fp64 CPU oracle (oracle.c) and the layer composition.

TEST INFRASTRUCTURE ONLY: used by tests/, the package smoke check and the
benchmark's CPU-baseline leg.  Inputs are numpy arrays; bf16 tensors are
passed as uint16 bit patterns (the same bytes the GPU reads).

The layer composition follows the pages' description of DeepSeek-V4's hybrid
attention ("Why DeepSeek V4 Stands Apart", section "Core Architectural
Innovations"; "DeepSeek-V4" atlas spec sheet, "Design overview" and
"Provenance references" 16-18): compress (CSA m=4 w=8, HCA m=128 w=128),
indexer score, top-k, the three attention branches, then the sink merge with
inverse RoPE on the output.
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f64_to_bf16.restype = ctypes.c_uint16
        L.orc_f64_to_bf16.argtypes = [ctypes.c_double]
        L.orc_bf16_array_to_f64.argtypes = [_u16p, _f64p, ctypes.c_int64]
        L.orc_f64_array_to_bf16.argtypes = [_f64p, _u16p, ctypes.c_int64]
        L.orc_rmsnorm.argtypes = [_f64p, ctypes.c_int, _f32p, ctypes.c_double]
        L.orc_rope.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                               ctypes.c_int64, ctypes.c_int]
        L.orc_compress.restype = ctypes.c_int
        L.orc_compress.argtypes = [_u16p, _u16p, _u16p, _f32p, ctypes.c_int, ctypes.c_int64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _f64p]
        L.orc_compress_hidden.restype = ctypes.c_int
        L.orc_compress_hidden.argtypes = [_u16p, _u16p, _u16p, _f32p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_int64, ctypes.c_int64, _f64p,
                                          _f64p]
        L.orc_visible.restype = ctypes.c_int64
        L.orc_visible.argtypes = [ctypes.c_int64, ctypes.c_int]
        L.orc_indexer_scores.restype = ctypes.c_int
        L.orc_indexer_scores.argtypes = [_u16p, _f32p, _u16p, _i32p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                         _f64p]
        L.orc_e4m3_to_f64.restype = ctypes.c_double
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_f32_to_e4m3.restype = ctypes.c_uint8
        L.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.orc_quantize_e4m3_rows.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _u8p, _f32p]
        L.orc_indexer_scores_e4m3.restype = ctypes.c_int
        L.orc_indexer_scores_e4m3.argtypes = [_u16p, _f32p, _u8p, _f32p, _i32p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int64, ctypes.c_int, _f64p]
        L.orc_e2m1_to_f64.restype = ctypes.c_double
        L.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_f64_to_e2m1.restype = ctypes.c_uint8
        L.orc_f64_to_e2m1.argtypes = [ctypes.c_double]
        L.orc_e8m0_to_f64.restype = ctypes.c_double
        L.orc_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_quantize_mxfp4_rows.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, _u8p, _u8p]
        L.orc_indexer_scores_mxfp4.restype = ctypes.c_int
        L.orc_indexer_scores_mxfp4.argtypes = [_u16p, _f32p, _u8p, _u8p, _i32p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int64, ctypes.c_int, _f64p]
        L.orc_topk.restype = ctypes.c_int
        L.orc_topk.argtypes = [_f64p, _i32p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                               ctypes.c_int, _i32p]
        L.orc_attention.restype = ctypes.c_int
        L.orc_attention.argtypes = [ctypes.c_int, _u16p, _f32p, _u16p, _f32p, _i32p, _i32p,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                    ctypes.c_double, _f64p, _f64p]
        L.orc_merge.restype = ctypes.c_int
        L.orc_merge.argtypes = [ctypes.POINTER(_f64p), ctypes.POINTER(_f64p), ctypes.c_int,
                                _f32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p, _f64p]
        L.orc_weights_with_sink.restype = ctypes.c_double
        L.orc_weights_with_sink.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_double, _f64p]
        _lib = L
    return _lib


def _p(a, typ):
    if a is None:
        return ctypes.cast(None, typ)
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(typ)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 inputs are uint16 bit patterns, got {a.dtype}"
    return a


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- bf16
def bf16_to_f64(bits):
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().orc_bf16_array_to_f64(_p(bits, _u16p), _p(out, _f64p), bits.size)
    return out


def f64_to_bf16(x):
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f64_array_to_bf16(_p(x, _f64p), _p(out, _u16p), x.size)
    return out


# ---------------------------------------------------------------- primitives
def rmsnorm(x, gamma=None, eps=1e-6):
    """RMSNorm of the last axis (fp64)."""
    x = np.array(x, dtype=np.float64, copy=True)
    g = _f32(gamma)
    flat = x.reshape(-1, x.shape[-1])
    for i in range(flat.shape[0]):
        row = np.ascontiguousarray(flat[i])
        lib().orc_rmsnorm(_p(row, _f64p), row.shape[0], _p(g, _f32p), eps)
        flat[i] = row
    return flat.reshape(x.shape)


def rope(x, r, pos, base=10000.0, sign=+1):
    """Partial RoPE of the last r dims of a vector (fp64)."""
    x = np.array(x, dtype=np.float64, copy=True)
    lib().orc_rope(_p(x, _f64p), x.shape[-1], r, base, int(pos), int(sign))
    return x


def visible(t, m):
    return int(lib().orc_visible(int(t), int(m)))


# ---------------------------------------------------------------- stages
def compress(kv_raw, gate, m, w, r, j_begin, j_end, ik_raw=None, gamma=None, base=10000.0,
             eps=1e-6):
    """C(m, w) over entries [j_begin, j_end).  Returns fp64 (kv, ik or None, alpha)."""
    kv_raw = _u16(kv_raw)
    gate = _u16(gate)
    B, L, D = kv_raw.shape
    dI = 0
    if ik_raw is not None:
        ik_raw = _u16(ik_raw)
        dI = ik_raw.shape[2]
    nj = j_end - j_begin
    kv = np.zeros((B, nj, D), np.float64)
    ik = np.zeros((B, nj, dI), np.float64) if dI else None
    alpha = np.zeros((B, nj, w), np.float64)
    g = _f32(gamma)
    rc = lib().orc_compress(_p(kv_raw, _u16p), _p(ik_raw, _u16p), _p(gate, _u16p), _p(g, _f32p),
                            B, L, D, dI, m, w, r, base, eps, j_begin, j_end, _p(kv, _f64p),
                            _p(ik, _f64p), _p(alpha, _f64p))
    _check(rc, "compress")
    return kv, ik, alpha


def compress_hidden(x, W, gate, m, w, r, j_begin, j_end, D, gamma=None, base=10000.0, eps=1e-6):
    """C(m, w) of the projected hidden states x [B, L, dm] (bf16 bits) with
    W [dm, D + dI] (bf16 bits: KV columns, then indexer-key columns): every
    token projected in fp64, then pooled, normed and roped.  Returns fp64
    (kv [B, nj, D], ik [B, nj, dI] or None)."""
    x = _u16(x)
    W = _u16(W)
    gate = _u16(gate)
    B, L, dm = x.shape
    dI = W.shape[1] - D
    nj = j_end - j_begin
    kv = np.zeros((B, nj, D), np.float64)
    ik = np.zeros((B, nj, dI), np.float64) if dI else None
    g = _f32(gamma)
    rc = lib().orc_compress_hidden(_p(x, _u16p), _p(W, _u16p), _p(gate, _u16p), _p(g, _f32p), B, L,
                                   dm, D, dI, m, w, r, base, eps, j_begin, j_end, _p(kv, _f64p),
                                   _p(ik, _f64p))
    _check(rc, "compress_hidden")
    return kv, ik


def indexer_scores(iq, w, ik, pos, m):
    """fp64 scores [B, T, N_cap]; NaN where the entry is not visible."""
    iq = _u16(iq)
    ik = _u16(ik)
    w = _f32(w)
    pos = _i32(pos)
    B, T, HI, dI = iq.shape
    N = ik.shape[1]
    out = np.empty((B, T, N), np.float64)
    rc = lib().orc_indexer_scores(_p(iq, _u16p), _p(w, _f32p), _p(ik, _u16p), _p(pos, _i32p), B, T,
                                  HI, dI, N, m, _p(out, _f64p))
    _check(rc, "indexer_scores")
    return out


# ---------------------------------------------------------------- FP8 indexer keys
def e4m3_to_f64(codes):
    """Values of E4M3 codes (uint8 array), fp64."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_e4m3_to_f64
    return np.array([f(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)


def f32_to_e4m3(x):
    """Nearest E4M3 codes (ties to even, saturating at 448) of fp32 values."""
    x = np.asarray(x, dtype=np.float32)
    f = lib().orc_f32_to_e4m3
    return np.array([f(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def quantize_e4m3(x):
    """Rows of the last axis of bf16 bits to (codes uint8, scales fp32)."""
    x = _u16(x)
    n = x.shape[-1]
    rows = x.size // n if n else 0
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[:-1], np.float32)
    lib().orc_quantize_e4m3_rows(_p(x, _u16p), rows, n, _p(codes, _u8p), _p(scales, _f32p))
    return codes, scales


def dequantize_e4m3(codes, scales):
    """codes * scale per row, fp64."""
    return e4m3_to_f64(codes) * np.asarray(scales, np.float64)[..., None]


def indexer_scores_e4m3(iq, w, ik8, iks, pos, m):
    """fp64 scores [B, T, N_cap] from FP8 keys (codes ik8, row scales iks);
    the bf16 queries are quantised the same way and both sides dequantised."""
    iq = _u16(iq)
    ik8 = np.ascontiguousarray(ik8, dtype=np.uint8)
    iks = _f32(iks)
    w = _f32(w)
    pos = _i32(pos)
    B, T, HI, dI = iq.shape
    N = ik8.shape[1]
    out = np.empty((B, T, N), np.float64)
    rc = lib().orc_indexer_scores_e4m3(_p(iq, _u16p), _p(w, _f32p), _p(ik8, _u8p),
                                       _p(iks, _f32p), _p(pos, _i32p), B, T, HI, dI, N, m,
                                       _p(out, _f64p))
    _check(rc, "indexer_scores_e4m3")
    return out


# ---------------------------------------------------------------- MXFP4 indexer rows
def e2m1_to_f64(codes):
    """Values of E2M1 codes (the low 4 bits of each uint8), fp64."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_e2m1_to_f64
    return np.array([f(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)


def f64_to_e2m1(y):
    """Nearest E2M1 codes (ties to even, saturating at 6, zero as +0)."""
    y = np.asarray(y, dtype=np.float64)
    f = lib().orc_f64_to_e2m1
    return np.array([f(float(v)) for v in y.ravel()], np.uint8).reshape(y.shape)


def e8m0_to_f64(codes):
    """Values 2^(c-127) of E8M0 scale codes (255 is NaN), fp64."""
    c = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_e8m0_to_f64
    return np.array([f(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)


def quantize_mxfp4(x):
    """Rows of the last axis (n bf16 bits, n a multiple of 32) to MXFP4:
    (codes uint8 [.., n/2], element 2i in the low nibble; scales uint8
    E8M0 [.., n/32])."""
    x = _u16(x)
    n = x.shape[-1]
    rows = x.size // n if n else 0
    codes = np.empty(x.shape[:-1] + (n // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (n // 32,), np.uint8)
    lib().orc_quantize_mxfp4_rows(_p(x, _u16p), rows, n, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def dequantize_mxfp4(codes, scales):
    """fp64 values [.., n] of MXFP4 rows."""
    codes = np.asarray(codes, np.uint8)
    nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (-1,))
    n = nib.shape[-1]
    sc = np.repeat(e8m0_to_f64(scales), 32, axis=-1)[..., :n]
    return e2m1_to_f64(nib) * sc


def indexer_scores_mxfp4(iq, w, ik4, iks, pos, m):
    """fp64 scores [B, T, N_cap] from MXFP4 keys (codes ik4 [B, N_cap, dI/2],
    E8M0 scales iks [B, N_cap, dI/32]); the bf16 queries are quantised the
    same way and both sides dequantised."""
    iq = _u16(iq)
    ik4 = np.ascontiguousarray(ik4, dtype=np.uint8)
    iks = np.ascontiguousarray(iks, dtype=np.uint8)
    w = _f32(w)
    pos = _i32(pos)
    B, T, HI, dI = iq.shape
    N = ik4.shape[1]
    out = np.empty((B, T, N), np.float64)
    rc = lib().orc_indexer_scores_mxfp4(_p(iq, _u16p), _p(w, _f32p), _p(ik4, _u8p),
                                        _p(iks, _u8p), _p(pos, _i32p), B, T, HI, dI, N, m,
                                        _p(out, _f64p))
    _check(rc, "indexer_scores_mxfp4")
    return out


def topk(scores, pos, m, k):
    """Top-k indices [.., k] (score desc, index asc), padded with -1."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    pos = _i32(pos)
    lead = scores.shape[:-1]
    N = scores.shape[-1]
    rows = int(np.prod(lead))
    out = np.empty(lead + (k,), np.int32)
    rc = lib().orc_topk(_p(scores.reshape(rows, N), _f64p), _p(pos.reshape(rows), _i32p), rows, N,
                        m, k, _p(out, _i32p))
    _check(rc, "topk")
    return out


KIND_SPARSE, KIND_HCA, KIND_SWA = 0, 1, 2


def attention(kind, q, cache, pos, *, idx=None, k=0, m=0, W=0, r=0, gamma_q=None, gamma_kv=None,
              base=10000.0, eps=1e-6, scale=None):
    """One branch.  Returns fp64 (o [B,T,H,D], lse [B,T,H])."""
    q = _u16(q)
    cache = _u16(cache)
    pos = _i32(pos)
    B, T, H, D = q.shape
    N = cache.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if idx is not None:
        idx = _i32(idx)
        k = idx.shape[-1]
    o = np.empty((B, T, H, D), np.float64)
    lse = np.empty((B, T, H), np.float64)
    gq, gk = _f32(gamma_q), _f32(gamma_kv)
    rc = lib().orc_attention(kind, _p(q, _u16p), _p(gq, _f32p), _p(cache, _u16p), _p(gk, _f32p),
                             _p(idx, _i32p), _p(pos, _i32p), B, T, H, D, N, k, m, W, r, base, eps,
                             scale, _p(o, _f64p), _p(lse, _f64p))
    _check(rc, "attention")
    return o, lse


def merge(o_list, lse_list, sink, pos, r, base=10000.0):
    """Sink-augmented LSE merge + inverse RoPE.  Returns fp64 (out, lse)."""
    o_list = [np.ascontiguousarray(o, dtype=np.float64) for o in o_list]
    lse_list = [np.ascontiguousarray(x, dtype=np.float64) for x in lse_list]
    pos = _i32(pos)
    B, T = pos.shape
    if o_list:
        H, D = o_list[0].shape[2], o_list[0].shape[3]
    else:
        raise ValueError("merge needs at least one branch to know H and D")
    nb = len(o_list)
    optrs = (_f64p * max(nb, 1))(*[_p(o, _f64p) for o in o_list])
    lptrs = (_f64p * max(nb, 1))(*[_p(x, _f64p) for x in lse_list])
    s = _f32(sink)
    out = np.empty((B, T, H, D), np.float64)
    lse = np.empty((B, T, H), np.float64)
    rc = lib().orc_merge(optrs, lptrs, nb, _p(s, _f32p), _p(pos, _i32p), B, T, H, D, r, base,
                         _p(out, _f64p), _p(lse, _f64p))
    _check(rc, "merge")
    return out, lse


def weights_with_sink(q_prepped, keys_prepped, scale, sink):
    q = np.ascontiguousarray(q_prepped, dtype=np.float64)
    kk = np.ascontiguousarray(keys_prepped, dtype=np.float64)
    nk, D = kk.shape
    w = np.empty(nk, np.float64)
    ws = lib().orc_weights_with_sink(_p(q, _f64p), _p(kk, _f64p), nk, D, scale, sink, _p(w, _f64p))
    return w, ws


# ---------------------------------------------------------------- layer
def layer(inp, cfg, branches=("csa", "hca", "swa"), keep=False):
    """Full hybrid layer for the queries in `inp`, from the raw token caches.

    inp: dict of numpy arrays (uint16 bf16 bits, fp32, int32):
      q [B,T,H,D], kv_raw [B,L,D], ik_raw [B,L,dI], gate_csa [B,L], gate_hca [B,L],
      iq [B,T,HI,dI], w [B,T,HI] fp32, pos [B,T], sink [H] fp32,
      optional gamma_q [D], gamma_kv [D].
    cfg: dict with m_csa, w_csa, m_hca, w_hca, k, W, r, base, eps.
    The compressed caches are stored in bf16 (the storage format) before the
    branches read them.  Returns dict(out, lse, and intermediates if keep).
    """
    kv_raw, pos = inp["kv_raw"], inp["pos"]
    B, L, D = kv_raw.shape
    r, base, eps = cfg["r"], cfg.get("base", 10000.0), cfg.get("eps", 1e-6)
    gq, gk = inp.get("gamma_q"), inp.get("gamma_kv")
    res = {}
    o_list, l_list = [], []
    tmax = int(np.max(pos))
    if "csa" in branches:
        m, w = cfg["m_csa"], cfg["w_csa"]
        n = min(L // m, visible(tmax, m)) if L >= m else 0
        n_cap = L // m
        kv_c = np.zeros((B, n_cap, D), np.uint16)
        ik_c = np.zeros((B, n_cap, inp["ik_raw"].shape[2]), np.uint16)
        if n > 0:
            kv64, ik64, _ = compress(kv_raw, inp["gate_csa"], m, w, r, 0, n, ik_raw=inp["ik_raw"],
                                     gamma=gk, base=base, eps=eps)
            kv_c[:, :n] = f64_to_bf16(kv64)
            ik_c[:, :n] = f64_to_bf16(ik64)
            if keep:
                res["kv_c64"], res["ik_c64"] = kv64, ik64
        scores = indexer_scores(inp["iq"], inp["w"], ik_c, pos, m)
        idx = topk(scores, pos, m, cfg["k"])
        o, l = attention(KIND_SPARSE, inp["q"], kv_c, pos, idx=idx, r=r, gamma_q=gq, base=base,
                         eps=eps)
        o_list.append(o)
        l_list.append(l)
        if keep:
            res.update(kv_c=kv_c, ik_c=ik_c, scores=scores, idx=idx, o_csa=o, lse_csa=l)
    if "hca" in branches:
        m, w = cfg["m_hca"], cfg["w_hca"]
        n_cap = L // m
        n = min(n_cap, visible(tmax, m))
        kv_h = np.zeros((B, max(n_cap, 1), D), np.uint16)
        if n > 0:
            kh64, _, _ = compress(kv_raw, inp["gate_hca"], m, w, r, 0, n, gamma=gk, base=base,
                                  eps=eps)
            kv_h[:, :n] = f64_to_bf16(kh64)
            if keep:
                res["kv_h64"] = kh64
        o, l = attention(KIND_HCA, inp["q"], kv_h, pos, m=m, r=r, gamma_q=gq, base=base, eps=eps)
        o_list.append(o)
        l_list.append(l)
        if keep:
            res.update(kv_h=kv_h, o_hca=o, lse_hca=l)
    if "swa" in branches:
        o, l = attention(KIND_SWA, inp["q"], kv_raw, pos, W=cfg["W"], r=r, gamma_q=gq,
                         gamma_kv=gk, base=base, eps=eps)
        o_list.append(o)
        l_list.append(l)
        if keep:
            res.update(o_swa=o, lse_swa=l)
    out, lse = merge(o_list, l_list, inp.get("sink"), pos, r, base)
    res["out"], res["lse"] = out, lse
    return res


def library_path():
    return os.path.abspath(_build.LIB)
