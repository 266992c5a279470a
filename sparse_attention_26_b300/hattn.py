"""Thin ctypes binding of libhattn (include/hattn.h).

Each function takes torch CUDA tensors, checks dtype / contiguity / device,
allocates any output or workspace the caller did not pass (torch is the
device-memory allocator), and calls the C entry point of the same name on the
current torch stream.  All compute runs in libhattn's kernels; there is no
CPU or PyTorch fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhattn.so")

OK, INVALID_ARG, MISALIGNED, UNSUPPORTED, CUDA_ERROR, TIMEOUT, DEVICE_INDEX = range(7)
KIND_SPARSE, KIND_HCA, KIND_SWA = 0, 1, 2

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/hattn.h
_SIGS = {
    "hattn_csa_compress": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _i32,
                                  _f32, _f32, _i64, _i64, _vp, _vp, _i64, _vp]),
    "hattn_hca_compress": (_i32, [_vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _f32, _f32, _i64,
                                  _i64, _vp, _i64, _vp]),
    "hattn_csa_compress_fp8": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                      _i32, _f32, _f32, _i64, _i64, _vp, _vp, _vp, _vp, _i64,
                                      _vp]),
    "hattn_csa_compress_mxfp4": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                        _i32, _f32, _f32, _i64, _i64, _vp, _vp, _vp, _vp, _i64,
                                        _vp]),
    "hattn_quantize_e4m3": (_i32, [_vp, _i64, _i32, _vp, _vp, _vp]),
    "hattn_quantize_mxfp4": (_i32, [_vp, _i64, _i32, _vp, _vp, _vp]),
    "hattn_compress_hidden_workspace_bytes": (_sz, [_i32, _i64, _i64, _i32, _i32, _i32]),
    "hattn_compress_hidden": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                     _i32, _i32, _f32, _f32, _i64, _i64, _vp, _vp, _i64, _vp,
                                     _sz, _vp]),
    "hattn_csa_compress_ring": (_i32, [_vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                       _i32, _f32, _f32, _i64, _i64, _vp, _vp, _i64, _vp]),
    "hattn_hca_compress_ring": (_i32, [_vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _f32, _f32,
                                       _i64, _i64, _vp, _i64, _vp]),
    "hattn_swa_keys_ring": (_i32, [_vp, _vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _f32, _f32,
                                   _vp, _vp]),
    "hattn_indexer_scores_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                        _i32, _i32, _i64, _vp, _i32, _vp]),
    "hattn_quantize_mxfp4_entries": (_i32, [_vp, _i32, _i64, _i32, _i64, _i64, _vp, _vp, _vp]),
    "hattn_indexer_scores_mxfp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                          _i32, _i32, _i64, _vp, _i32, _vp]),
    "hattn_indexer_topk_mxfp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                        _i32, _i32, _i32, _i64, _vp, _vp, _vp, _sz, _i32, _vp,
                                        _vp]),
    "hattn_indexer_topk": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _i32,
                                  _vp, _vp, _vp, _sz, _vp]),
    "hattn_indexer_topk_workspace_bytes": (_sz, [_i32, _i32, _i64, _i32, _i32]),
    "hattn_indexer_topk_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32,
                                     _i32, _i32, _i64, _vp, _vp, _vp, _sz, _i32, _vp, _vp]),
    "hattn_indexer_topk_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32,
                                          _i32, _vp, _vp]),
    "hattn_indexer_scores": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _vp,
                                    _vp]),
    "hattn_topk_select": (_i32, [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _sz, _i32,
                                 _vp]),
    "hattn_topk_workspace_bytes": (_sz, [_i32, _i32, _i64, _i32]),
    "hattn_query_prep": (_i32, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _vp,
                                _vp]),
    "hattn_sparse_attn": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64,
                                 _i32, _i32, _f32, _f32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "hattn_hca_attn": (_i32, [_vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32, _i32,
                              _f32, _f32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "hattn_swa_attn": (_i32, [_vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32,
                              _i32, _f32, _f32, _f32, _vp, _vp, _vp, _sz, _vp]),
    "hattn_attn_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i64, _i32, _i32]),
    "hattn_swa_keys": (_i32, [_vp, _vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _f32, _f32, _vp,
                              _vp]),
    "hattn_hybrid_attn": (_i32, [_vp, _vp, _i32, _vp, _vp, _i64, _i32, _vp, _i64, _i32, _vp, _i32,
                                 _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32, _i32, _i32,
                                 _vp, _vp, _vp, _sz, _i32, _vp]),
    "hattn_hybrid_attn_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i64, _i32, _i32,
                                                _i32, _i32, _i32]),
    "hattn_compress_hidden_pair_workspace_bytes": (_sz, [_i32, _i64, _i64, _i64, _i32]),
    "hattn_compress_hidden_pair": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32,
                                          _i32, _i32, _i32, _f32, _f32, _vp, _vp, _i64, _vp, _i64,
                                          _vp, _sz, _vp]),
    "hattn_hybrid_attn_out": (_i32, [_vp, _vp, _i32, _vp, _vp, _i64, _i32, _vp, _i64, _i32, _vp,
                                     _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32,
                                     _i32, _i32, _vp, _vp, _vp, _vp, _sz, _i32, _vp]),
    "hattn_hybrid_attn_out_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32, _i64, _i32,
                                                    _i32, _i32, _i32]),
    "hattn_hybrid_attn_splits": (_i32, [_i32, _i32, _i32, _i32, _i32, _i64, _i32, _i32, _i32]),
    "hattn_indexer_scores_ex": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i64, _i32,
                                       _i32, _i64, _vp, _i32, _vp]),
    "hattn_attn_splits": (_i32, [_i32, _i32, _i32, _i32, _i32, _i64]),
    "hattn_lse_merge_splits": (_i32, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_i32),
                                      _i32, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp,
                                      _i32, _vp]),
    "hattn_lse_merge": (_i32, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32, _vp, _vp, _i32,
                               _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp]),
    "hattn_status_string": (ctypes.c_char_p, [_i32]),
    "hattn_last_error": (ctypes.c_char_p, []),
    "hattn_check_status": (_i32, [_vp]),
    "hattn_selftest_wait_timeout": (_i32, [ctypes.c_uint64, _vp]),
    "hattn_version": (ctypes.c_char_p, []),
}

LAUNCH_DEPENDENT = 1  # HATTN_LAUNCH_DEPENDENT
EVENT_EXTERNAL = 2  # HATTN_EVENT_EXTERNAL

_lib = None


class HattnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libhattn error {code}: {msg}")
        self.code = code


def lib():
    """Load libhattn.so (built in-tree); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_attention_26_b300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc):
    if rc != OK:
        raise HattnError(rc, lib().hattn_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _event(ev):
    """The cudaEvent_t of a torch.cuda.Event that has been recorded once (its
    CUDA event exists), or None."""
    if ev is None:
        return None
    if not ev.cuda_event:
        raise ValueError("split_event must have been recorded once (its CUDA event is created "
                         "on the first record)")
    return ctypes.c_void_p(ev.cuda_event)


def _need(t, name, dtype, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t


def _opt(t, name, dtype):
    return None if t is None else _need(t, name, dtype)


def _shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _flags(dependent):
    return LAUNCH_DEPENDENT if dependent else 0


def _indexer_inputs(iq, w, ik, pos, ik_name="ik_c", ik_dtype=torch.bfloat16):
    """Checks the indexer inputs against each other; returns B, T, HI, dI, N_cap."""
    _need(iq, "iq", torch.bfloat16, 4)
    _need(w, "w", torch.float32, 3)
    _need(ik, ik_name, ik_dtype, 3)
    _need(pos, "pos", torch.int32, 2)
    B, T, HI, dI = iq.shape
    _shape(w, "w", (B, T, HI))
    _shape(pos, "pos", (B, T))
    if ik.shape[0] != B:
        raise ValueError(f"{ik_name} holds {ik.shape[0]} sequences, iq {B}")
    if ik_dtype == torch.bfloat16 and ik.shape[2] != dI:
        raise ValueError(f"{ik_name} rows have {ik.shape[2]} dims, iq {dI}")
    return B, T, HI, dI, ik.shape[1]


# ------------------------------------------------------------------ compression
def csa_compress(kv_raw, ik_raw, gate, *, r, j_begin=0, j_end=None, m=4, w=8, kv_c=None,
                 ik_c=None, N_cap=None, gamma_kv=None, rope_base=10000.0, eps=1e-6, stream=None):
    """C(m, w) of KV + indexer keys for entries [j_begin, j_end); returns (kv_c, ik_c)."""
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(gate, "gate", torch.bfloat16, 2)
    if ik_raw is not None:
        _need(ik_raw, "ik_raw", torch.bfloat16, 3)
    B, L, D = kv_raw.shape
    dI = ik_raw.shape[2] if ik_raw is not None else 0
    if N_cap is None:
        N_cap = kv_c.shape[1] if kv_c is not None else L // m
    if j_end is None:
        j_end = min(N_cap, L // m)
    if kv_c is None:
        kv_c = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=kv_raw.device)
    if ik_c is None and ik_raw is not None:
        ik_c = torch.zeros((B, N_cap, dI), dtype=torch.bfloat16, device=kv_raw.device)
    _need(kv_c, "kv_c", torch.bfloat16, 3)
    _opt(ik_c, "ik_c", torch.bfloat16)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    _check(lib().hattn_csa_compress(_ptr(kv_raw), _ptr(ik_raw), _ptr(gate), _ptr(gamma_kv), B, L,
                                    D, dI, m, w, r, rope_base, eps, j_begin, j_end, _ptr(kv_c),
                                    _ptr(ik_c), N_cap, _stream(stream)))
    return kv_c, ik_c


def csa_compress_fp8(kv_raw, ik_raw, gate, *, r, j_begin=0, j_end=None, m=4, w=8, kv_c=None,
                     ik8=None, ik_scale=None, ik_c=None, N_cap=None, gamma_kv=None,
                     rope_base=10000.0, eps=1e-6, stream=None):
    """csa_compress that writes each entry's indexer key as E4M3 codes with a
    row scale (and, when ik_c is given, also as bf16); returns
    (kv_c, ik8 uint8 [B, N_cap, dI], ik_scale fp32 [B, N_cap])."""
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(ik_raw, "ik_raw", torch.bfloat16, 3)
    _need(gate, "gate", torch.bfloat16, 2)
    B, L, D = kv_raw.shape
    dI = ik_raw.shape[2]
    if N_cap is None:
        N_cap = kv_c.shape[1] if kv_c is not None else L // m
    if j_end is None:
        j_end = min(N_cap, L // m)
    dev = kv_raw.device
    if kv_c is None:
        kv_c = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=dev)
    if ik8 is None:
        ik8 = torch.zeros((B, N_cap, dI), dtype=torch.uint8, device=dev)
    if ik_scale is None:
        ik_scale = torch.zeros((B, N_cap), dtype=torch.float32, device=dev)
    _need(kv_c, "kv_c", torch.bfloat16, 3)
    _need(ik8, "ik8", torch.uint8, 3)
    _need(ik_scale, "ik_scale", torch.float32, 2)
    _opt(ik_c, "ik_c", torch.bfloat16)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    _check(lib().hattn_csa_compress_fp8(_ptr(kv_raw), _ptr(ik_raw), _ptr(gate), _ptr(gamma_kv), B,
                                        L, D, dI, m, w, r, rope_base, eps, j_begin, j_end,
                                        _ptr(kv_c), _ptr(ik_c), _ptr(ik8), _ptr(ik_scale), N_cap,
                                        _stream(stream)))
    return kv_c, ik8, ik_scale


def csa_compress_mxfp4(kv_raw, ik_raw, gate, *, r, kv_c, ik_c, ik4, ik4_scale, j_begin=0,
                       j_end=None, m=4, w=8, gamma_kv=None, rope_base=10000.0, eps=1e-6,
                       stream=None):
    """csa_compress that also writes each entry's indexer key as MXFP4
    (codes ik4 uint8 [B, N_cap, dI/2], E8M0 scales ik4_scale uint8
    [B, N_cap, dI/32]), bit for bit what quantize_mxfp4 makes of ik_c."""
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(ik_raw, "ik_raw", torch.bfloat16, 3)
    _need(gate, "gate", torch.bfloat16, 2)
    B, L, D = kv_raw.shape
    dI = ik_raw.shape[2]
    N_cap = kv_c.shape[1]
    if j_end is None:
        j_end = min(N_cap, L // m)
    _need(kv_c, "kv_c", torch.bfloat16, 3)
    _need(ik_c, "ik_c", torch.bfloat16, 3)
    _need(ik4, "ik4", torch.uint8, 3)
    _shape(ik4, "ik4", (B, N_cap, dI // 2))
    _need(ik4_scale, "ik4_scale", torch.uint8, 3)
    _shape(ik4_scale, "ik4_scale", (B, N_cap, dI // 32))
    _opt(gamma_kv, "gamma_kv", torch.float32)
    _check(lib().hattn_csa_compress_mxfp4(_ptr(kv_raw), _ptr(ik_raw), _ptr(gate), _ptr(gamma_kv),
                                          B, L, D, dI, m, w, r, rope_base, eps, j_begin, j_end,
                                          _ptr(kv_c), _ptr(ik_c), _ptr(ik4), _ptr(ik4_scale),
                                          N_cap, _stream(stream)))
    return kv_c, ik_c, ik4, ik4_scale


def csa_compress_ring(kv_ring, ik_ring, gate_ring, *, r, j_begin, j_end, kv_c, ik_c, m=4, w=8,
                      gamma_kv=None, rope_base=10000.0, eps=1e-6, stream=None):
    """csa_compress over ring-buffer raw caches ([B, ring, ...], token u in
    row u % ring) into kv_c / ik_c rows [j_begin, j_end)."""
    _need(kv_ring, "kv_ring", torch.bfloat16, 3)
    _need(ik_ring, "ik_ring", torch.bfloat16, 3)
    _need(gate_ring, "gate_ring", torch.bfloat16, 2)
    _need(kv_c, "kv_c", torch.bfloat16, 3)
    _need(ik_c, "ik_c", torch.bfloat16, 3)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, ring, D = kv_ring.shape
    _check(lib().hattn_csa_compress_ring(_ptr(kv_ring), _ptr(ik_ring), _ptr(gate_ring),
                                         _ptr(gamma_kv), B, ring, D, ik_ring.shape[2], m, w, r,
                                         rope_base, eps, j_begin, j_end, _ptr(kv_c), _ptr(ik_c),
                                         kv_c.shape[1], _stream(stream)))
    return kv_c, ik_c


def hca_compress_ring(kv_ring, gate_ring, *, r, j_begin, j_end, kv_h, m=128, gamma_kv=None,
                      rope_base=10000.0, eps=1e-6, stream=None):
    """hca_compress over ring-buffer raw caches into kv_h rows [j_begin, j_end)."""
    _need(kv_ring, "kv_ring", torch.bfloat16, 3)
    _need(gate_ring, "gate_ring", torch.bfloat16, 2)
    _need(kv_h, "kv_h", torch.bfloat16, 3)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, ring, D = kv_ring.shape
    _check(lib().hattn_hca_compress_ring(_ptr(kv_ring), _ptr(gate_ring), _ptr(gamma_kv), B, ring,
                                         D, m, r, rope_base, eps, j_begin, j_end, _ptr(kv_h),
                                         kv_h.shape[1], _stream(stream)))
    return kv_h


def swa_keys_ring(kv_ring, pos, *, r, W=128, gamma_kv=None, rope_base=10000.0, eps=1e-6,
                  kv_w=None, stream=None):
    """swa_keys over a ring-buffer raw cache [B, ring, D] (token u in row u % ring)."""
    _need(kv_ring, "kv_ring", torch.bfloat16, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, ring, D = kv_ring.shape
    T = pos.shape[1]
    if kv_w is None:
        kv_w = torch.empty((B, T, W, D), dtype=torch.bfloat16, device=kv_ring.device)
    _need(kv_w, "kv_w", torch.bfloat16, 4)
    _check(lib().hattn_swa_keys_ring(_ptr(kv_ring), _ptr(gamma_kv), _ptr(pos), B, T, ring, D, W, r,
                                     rope_base, eps, _ptr(kv_w), _stream(stream)))
    return kv_w


def compress_hidden(x, W, gate, *, D, r, m=4, w=8, j_begin=0, j_end=None, kv_out=None,
                    ik_out=None, N_cap=None, gamma_kv=None, rope_base=10000.0, eps=1e-6,
                    workspace=None, stream=None):
    """C(m, w) entries [j_begin, j_end) of the projected hidden states x
    [B, L, dm] with W [dm, D + dI] (KV columns, then indexer-key columns);
    returns (kv_out [B, N_cap, D], ik_out [B, N_cap, dI] or None)."""
    _need(x, "x", torch.bfloat16, 3)
    _need(W, "W", torch.bfloat16, 2)
    _need(gate, "gate", torch.bfloat16, 2)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, L, dm = x.shape
    dI = W.shape[1] - D
    if N_cap is None:
        N_cap = kv_out.shape[1] if kv_out is not None else L // m
    if j_end is None:
        j_end = min(N_cap, L // m)
    dev = x.device
    if kv_out is None:
        kv_out = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=dev)
    if ik_out is None and dI > 0:
        ik_out = torch.zeros((B, N_cap, dI), dtype=torch.bfloat16, device=dev)
    _need(kv_out, "kv_out", torch.bfloat16, 3)
    _opt(ik_out, "ik_out", torch.bfloat16)
    need = lib().hattn_compress_hidden_workspace_bytes(B, j_begin, j_end, dm, D, dI)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().hattn_compress_hidden(_ptr(x), _ptr(W), _ptr(gate), _ptr(gamma_kv), B, L, dm, D,
                                       dI, m, w, r, rope_base, eps, j_begin, j_end, _ptr(kv_out),
                                       _ptr(ik_out), N_cap, _ptr(workspace), wsb,
                                       _stream(stream)))
    return kv_out, ik_out



def compress_hidden_pair(x, W_c, gate_c, W_h, gate_h, *, D, r, L=None, kv_c=None, ik_c=None,
                         kv_h=None, N_c=None, N_h=None, gamma_kv=None, rope_base=10000.0,
                         eps=1e-6, workspace=None, stream=None):
    """Both caches of a layer from hidden states in one read of them: the CSA
    entries C(4, 8) with indexer keys (W_c [dm, D + dI]) and the HCA entries
    C(128, 128) (W_h [dm, D]) of the first L tokens; returns (kv_c, ik_c or
    None, kv_h)."""
    _need(x, "x", torch.bfloat16, 3)
    _need(W_c, "W_c", torch.bfloat16, 2)
    _need(W_h, "W_h", torch.bfloat16, 2)
    _need(gate_c, "gate_c", torch.bfloat16, 2)
    _need(gate_h, "gate_h", torch.bfloat16, 2)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, L_cap, dm = x.shape
    L = L_cap if L is None else L
    dI = W_c.shape[1] - D
    dev = x.device
    N_c = (kv_c.shape[1] if kv_c is not None else L_cap // 4) if N_c is None else N_c
    N_h = (kv_h.shape[1] if kv_h is not None else max(1, L_cap // 128)) if N_h is None else N_h
    if kv_c is None:
        kv_c = torch.zeros((B, N_c, D), dtype=torch.bfloat16, device=dev)
    if ik_c is None and dI > 0:
        ik_c = torch.zeros((B, N_c, dI), dtype=torch.bfloat16, device=dev)
    if kv_h is None:
        kv_h = torch.zeros((B, N_h, D), dtype=torch.bfloat16, device=dev)
    need = lib().hattn_compress_hidden_pair_workspace_bytes(B, L, N_c, N_h, dm)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    wsb = workspace.numel() if workspace is not None else 0
    _check(lib().hattn_compress_hidden_pair(_ptr(x), _ptr(W_c), _ptr(gate_c), _ptr(W_h),
                                            _ptr(gate_h), _ptr(gamma_kv), B, L_cap, L, dm, D, dI,
                                            r, rope_base, eps, _ptr(kv_c), _ptr(ik_c), N_c,
                                            _ptr(kv_h), N_h, _ptr(workspace), wsb,
                                            _stream(stream)))
    return kv_c, ik_c, kv_h


def quantize_e4m3(x, *, codes=None, scales=None, stream=None):
    """Rows of the last axis of a bf16 tensor to E4M3 codes (uint8, same
    shape) and fp32 row scales (shape without the last axis)."""
    _need(x, "x", torch.bfloat16)
    n = x.shape[-1]
    rows = x.numel() // n if n else 0
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.float32)
    _check(lib().hattn_quantize_e4m3(_ptr(x), rows, n, _ptr(codes), _ptr(scales),
                                     _stream(stream)))
    return codes, scales


def quantize_mxfp4(x, *, codes=None, scales=None, stream=None):
    """Rows of the last axis of a bf16 tensor (a multiple of 32 long) to
    MXFP4: E2M1 codes (uint8 [.., n/2], element 2i in the low nibble) and
    E8M0 block scales (uint8 [.., n/32])."""
    _need(x, "x", torch.bfloat16)
    n = x.shape[-1]
    rows = x.numel() // n if n else 0
    if codes is None:
        codes = torch.empty(x.shape[:-1] + (n // 2,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (n // 32,), dtype=torch.uint8, device=x.device)
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.uint8)
    if codes.numel() * 2 != x.numel() or scales.numel() * 32 != x.numel():
        raise ValueError("codes must hold n/2 bytes and scales n/32 bytes per row")
    _check(lib().hattn_quantize_mxfp4(_ptr(x), rows, n, _ptr(codes), _ptr(scales),
                                      _stream(stream)))
    return codes, scales


def hca_compress(kv_raw, gate, *, r, j_begin=0, j_end=None, m=128, kv_h=None, N_cap=None,
                 gamma_kv=None, rope_base=10000.0, eps=1e-6, stream=None):
    """C(m, m) of KV for entries [j_begin, j_end); returns kv_h."""
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(gate, "gate", torch.bfloat16, 2)
    B, L, D = kv_raw.shape
    if N_cap is None:
        N_cap = kv_h.shape[1] if kv_h is not None else max(1, L // m)
    if j_end is None:
        j_end = min(N_cap, L // m)
    if kv_h is None:
        kv_h = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=kv_raw.device)
    _need(kv_h, "kv_h", torch.bfloat16, 3)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    _check(lib().hattn_hca_compress(_ptr(kv_raw), _ptr(gate), _ptr(gamma_kv), B, L, D, m, r,
                                    rope_base, eps, j_begin, j_end, _ptr(kv_h), N_cap,
                                    _stream(stream)))
    return kv_h


# ------------------------------------------------------------------ indexer
def indexer_topk_workspace_bytes(B, T, N_cap, k, score_out_given=False):
    return int(lib().hattn_indexer_topk_workspace_bytes(B, T, N_cap, k, int(bool(score_out_given))))


def topk_workspace_bytes(B, T, N_cap, k):
    return int(lib().hattn_topk_workspace_bytes(B, T, N_cap, k))


def topk_launches(B, T, N_cap, k):
    """Kernels one top-k selection launches (one, on either path)."""
    return 1


def _idx_out(idx_out, B, T, k, device):
    if idx_out is None:
        idx_out = torch.empty((B, T, k), dtype=torch.int32, device=device)
    _need(idx_out, "idx_out", torch.int32, 3)
    return _shape(idx_out, "idx_out", (B, T, k))


def indexer_topk(iq, w, ik_c, pos, *, k, m=4, idx_out=None, score_out=None, workspace=None,
                 ik_scale=None, n_sms=0, fresh_from=-1, dependent=False, split_event=None,
                 split_external=False, stream=None):
    """Lightning-indexer scores + per-query top-k; returns idx [B, T, k] int32.
    ik_scale: given, ik_c holds E4M3 codes uint8 [B, N_cap, 128] with these
    row scales fp32 [B, N_cap].  n_sms, fresh_from, dependent: as
    indexer_scores, for the score kernel.  split_event: a torch.cuda.Event
    (recorded once before) that the call records between the score and the
    selection kernel: other streams may wait on it for the scores alone, and
    with split_external (an external event) it times the two kernels
    apart."""
    if ik_scale is None:
        B, T, HI, dI, N_cap = _indexer_inputs(iq, w, ik_c, pos)
    else:
        B, T, HI, dI, N_cap = _indexer_inputs(iq, w, ik_c, pos, "ik8", torch.uint8)
        _need(ik_scale, "ik_scale", torch.float32, 2)
        _shape(ik_scale, "ik_scale", (B, N_cap))
    idx_out = _idx_out(idx_out, B, T, k, iq.device)
    if score_out is not None:
        _need(score_out, "score_out", torch.float32, 3)
        _shape(score_out, "score_out", (B, T, N_cap))
    need = indexer_topk_workspace_bytes(B, T, N_cap, k, score_out is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=iq.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if ik_scale is None and split_event is None and not (n_sms or fresh_from >= 0 or dependent):
        _check(lib().hattn_indexer_topk(_ptr(iq), _ptr(w), _ptr(ik_c), _ptr(pos), B, T, HI, dI,
                                        N_cap, k, m, _ptr(idx_out), _ptr(score_out),
                                        _ptr(workspace), ws_bytes, _stream(stream)))
    else:
        _check(lib().hattn_indexer_topk_ex(_ptr(iq), _ptr(w), _ptr(ik_c), _ptr(ik_scale),
                                           _ptr(pos), B, T, HI, dI, N_cap, k, m, n_sms,
                                           fresh_from, _ptr(idx_out), _ptr(score_out),
                                           _ptr(workspace), ws_bytes,
                                           _flags(dependent) | (EVENT_EXTERNAL if split_external
                                                                else 0),
                                           _event(split_event), _stream(stream)))
    return idx_out


def indexer_topk_noalloc(iq, w, ik_c, pos, *, k, m=4, idx_out=None, stream=None):
    """indexer_topk with its score and selection scratch in the library's
    fixed device array (no device allocation by the library;
    B*T*N_cap <= 4,194,304).  Calls that overlap on the GPU share that array
    and race."""
    B, T, HI, dI, N_cap = _indexer_inputs(iq, w, ik_c, pos)
    idx_out = _idx_out(idx_out, B, T, k, iq.device)
    _check(lib().hattn_indexer_topk_noalloc(_ptr(iq), _ptr(w), _ptr(ik_c), _ptr(pos), B, T, HI,
                                            dI, N_cap, k, m, _ptr(idx_out), _stream(stream)))
    return idx_out


def indexer_scores(iq, w, ik_c, pos, *, m=4, score_out=None, n_sms=0, fresh_from=-1,
                   dependent=False, stream=None):
    """Lightning-indexer scores only; returns score_out [B, T, N_cap] fp32
    (entries beyond each query's visible count are left untouched).  n_sms:
    run the persistent score kernel on at most that many SMs (0 = all);
    dependent: launch as a programmatic dependent of the previous kernel in
    the stream (HATTN_LAUNCH_DEPENDENT), with fresh_from the first entry that
    kernel may write (-1 = any)."""
    B, T, HI, dI, N_cap = _indexer_inputs(iq, w, ik_c, pos)
    if score_out is None:
        score_out = torch.empty((B, T, N_cap), dtype=torch.float32, device=iq.device)
    _need(score_out, "score_out", torch.float32, 3)
    _shape(score_out, "score_out", (B, T, N_cap))
    if n_sms or fresh_from >= 0 or dependent:
        _check(lib().hattn_indexer_scores_ex(_ptr(iq), _ptr(w), _ptr(ik_c), _ptr(pos), B, T, HI,
                                             dI, N_cap, m, n_sms, fresh_from, _ptr(score_out),
                                             _flags(dependent), _stream(stream)))
    else:
        _check(lib().hattn_indexer_scores(_ptr(iq), _ptr(w), _ptr(ik_c), _ptr(pos), B, T, HI, dI,
                                          N_cap, m, _ptr(score_out), _stream(stream)))
    return score_out


def quantize_mxfp4_entries(x, codes, scales, *, j_begin, j_end, stream=None):
    """quantize_mxfp4 of the entries [j_begin, j_end) of every sequence of a
    cache x [B, N_cap, n] bf16 into codes [B, N_cap, n/2] and scales
    [B, N_cap, n/32] (uint8)."""
    _need(x, "x", torch.bfloat16, 3)
    B, N_cap, n = x.shape
    _need(codes, "codes", torch.uint8, 3)
    _shape(codes, "codes", (B, N_cap, n // 2))
    _need(scales, "scales", torch.uint8, 3)
    _shape(scales, "scales", (B, N_cap, n // 32))
    _check(lib().hattn_quantize_mxfp4_entries(_ptr(x), B, N_cap, n, j_begin, j_end, _ptr(codes),
                                              _ptr(scales), _stream(stream)))


def _mx_keys(ik4, ik4_scale, B, N_cap):
    _need(ik4, "ik4", torch.uint8, 3)
    _shape(ik4, "ik4", (B, N_cap, 64))
    _need(ik4_scale, "ik4_scale", torch.uint8, 3)
    _shape(ik4_scale, "ik4_scale", (B, N_cap, 4))


def indexer_scores_mxfp4(iq, w, ik4, ik4_scale, pos, *, m=4, score_out=None, n_sms=0,
                         fresh_from=-1, dependent=False, stream=None):
    """indexer_scores over MXFP4 keys (codes ik4 uint8 [B, N_cap, 64] and E8M0
    scales ik4_scale uint8 [B, N_cap, 4], as quantize_mxfp4 writes them); the
    kernel quantises the bf16 queries the same way, and the score is the
    definition over the decoded values (block-scaled FP4 products)."""
    _need(iq, "iq", torch.bfloat16, 4)
    B, T, HI, dI = iq.shape
    N_cap = ik4.shape[1]
    _need(w, "w", torch.float32, 3)
    _shape(w, "w", (B, T, HI))
    _need(pos, "pos", torch.int32, 2)
    _shape(pos, "pos", (B, T))
    _mx_keys(ik4, ik4_scale, B, N_cap)
    if score_out is None:
        score_out = torch.empty((B, T, N_cap), dtype=torch.float32, device=iq.device)
    _need(score_out, "score_out", torch.float32, 3)
    _shape(score_out, "score_out", (B, T, N_cap))
    _check(lib().hattn_indexer_scores_mxfp4(_ptr(iq), _ptr(w), _ptr(ik4), _ptr(ik4_scale),
                                            _ptr(pos), B, T, HI, dI, N_cap, m, n_sms, fresh_from,
                                            _ptr(score_out), _flags(dependent), _stream(stream)))
    return score_out


def indexer_topk_mxfp4(iq, w, ik4, ik4_scale, pos, *, k, m=4, idx_out=None, score_out=None,
                       workspace=None, n_sms=0, fresh_from=-1, dependent=False, split_event=None,
                       split_external=False, stream=None):
    """indexer_topk over MXFP4 keys (see indexer_scores_mxfp4)."""
    _need(iq, "iq", torch.bfloat16, 4)
    B, T, HI, dI = iq.shape
    N_cap = ik4.shape[1]
    _need(w, "w", torch.float32, 3)
    _shape(w, "w", (B, T, HI))
    _need(pos, "pos", torch.int32, 2)
    _shape(pos, "pos", (B, T))
    _mx_keys(ik4, ik4_scale, B, N_cap)
    idx_out = _idx_out(idx_out, B, T, k, iq.device)
    if score_out is not None:
        _need(score_out, "score_out", torch.float32, 3)
        _shape(score_out, "score_out", (B, T, N_cap))
    need = indexer_topk_workspace_bytes(B, T, N_cap, k, score_out is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=iq.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().hattn_indexer_topk_mxfp4(_ptr(iq), _ptr(w), _ptr(ik4), _ptr(ik4_scale),
                                          _ptr(pos), B, T, HI, dI, N_cap, k, m, n_sms,
                                          fresh_from, _ptr(idx_out), _ptr(score_out),
                                          _ptr(workspace), ws_bytes,
                                          _flags(dependent) | (EVENT_EXTERNAL if split_external
                                                               else 0),
                                          _event(split_event), _stream(stream)))
    return idx_out


def indexer_scores_fp8(iq, w, ik8, ik_scale, pos, *, m=4, score_out=None, n_sms=0,
                       fresh_from=-1, dependent=False, stream=None):
    """indexer_scores over E4M3 keys (ik8 uint8 [B, N_cap, 128] with row
    scales ik_scale fp32 [B, N_cap]); the bf16 queries are quantised the
    same way in the kernel."""
    B, T, HI, dI, N_cap = _indexer_inputs(iq, w, ik8, pos, "ik8", torch.uint8)
    _need(ik_scale, "ik_scale", torch.float32, 2)
    _shape(ik_scale, "ik_scale", (B, N_cap))
    if score_out is None:
        score_out = torch.empty((B, T, N_cap), dtype=torch.float32, device=iq.device)
    _need(score_out, "score_out", torch.float32, 3)
    _shape(score_out, "score_out", (B, T, N_cap))
    _check(lib().hattn_indexer_scores_fp8(_ptr(iq), _ptr(w), _ptr(ik8), _ptr(ik_scale), _ptr(pos),
                                          B, T, HI, dI, N_cap, m, n_sms, fresh_from,
                                          _ptr(score_out), _flags(dependent), _stream(stream)))
    return score_out


def topk_select(scores, pos, *, k, m=4, idx_out=None, workspace=None, dependent=False,
                stream=None):
    """Per-query top-k over precomputed scores; returns idx [B, T, k] int32.
    workspace: the selection's scratch (topk_workspace_bytes; allocated here
    when needed and not given)."""
    _need(scores, "scores", torch.float32, 3)
    _need(pos, "pos", torch.int32, 2)
    B, T, N_cap = scores.shape
    _shape(pos, "pos", (B, T))
    idx_out = _idx_out(idx_out, B, T, k, scores.device)
    need = topk_workspace_bytes(B, T, N_cap, k)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().hattn_topk_select(_ptr(scores), _ptr(pos), B, T, N_cap, k, m, _ptr(idx_out),
                                   _ptr(workspace), wsb, _flags(dependent), _stream(stream)))
    return idx_out


# ------------------------------------------------------------------ attention
def attn_workspace_bytes(kind, B, T, H, D, n_keys, q_prepped=False, partials=False):
    return int(lib().hattn_attn_workspace_bytes(kind, B, T, H, D, n_keys, int(bool(q_prepped)),
                                                int(bool(partials))))


def attn_splits(kind, B, T, H, D, n_keys):
    """Key splits (partials per row) of an attention call of this shape."""
    return int(lib().hattn_attn_splits(kind, B, T, H, D, n_keys))


class Partials:
    """Split partials of one branch, viewing an attention call's workspace:
    o [B*T*H, nsplit, D] fp32, lse [B*T*H, nsplit] fp32."""

    def __init__(self, workspace, q_prepped, B, T, H, D, nsplit):
        rows = B * T * H
        off = 0 if q_prepped else rows * D * 2
        n_o = rows * nsplit * D
        f = workspace[off:off + (n_o + rows * nsplit) * 4].view(torch.float32)
        self.o = f[:n_o].view(rows, nsplit, D)
        self.lse = f[n_o:].view(rows, nsplit)
        self.nsplit = nsplit


def query_prep(q, pos, *, r, gamma_q=None, rope_base=10000.0, eps=1e-6, q_out=None, stream=None):
    """q~ = RoPE_pos(RMSNorm(q)) for every head; returns q_out [B, T, H, D] bf16."""
    _need(q, "q", torch.bfloat16, 4)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    B, T, H, D = q.shape
    if q_out is None:
        q_out = torch.empty_like(q)
    _need(q_out, "q_out", torch.bfloat16)
    _check(lib().hattn_query_prep(_ptr(q), _ptr(gamma_q), _ptr(pos), B, T, H, D, r, rope_base,
                                  eps, _ptr(q_out), _stream(stream)))
    return q_out


def _attn_out(q, o, lse):
    B, T, H, D = q.shape
    if o is None:
        o = torch.empty((B, T, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _need(o, "o", torch.float32)
    _need(lse, "lse", torch.float32)
    return o, lse


def _ws(kind, q, n_keys, workspace, q_prepped, partials=False):
    B, T, H, D = q.shape
    need = attn_workspace_bytes(kind, B, T, H, D, n_keys, q_prepped, partials)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    return workspace, (workspace.numel() * workspace.element_size() if workspace is not None
                       else 0)


def _result(kind, q, n_keys, o, lse, workspace, q_prepped, partials):
    if not partials:
        return o, lse
    B, T, H, D = q.shape
    return Partials(workspace, q_prepped, B, T, H, D, attn_splits(kind, B, T, H, D, n_keys))


def sparse_attn(q, kv_c, idx, pos, *, r, gamma_q=None, rope_base=10000.0, eps=1e-6, scale=None,
                o=None, lse=None, workspace=None, q_prepped=False, partials=False, stream=None):
    """CSA branch over the selected entries; returns (o fp32, lse fp32), or a
    Partials view of the workspace when partials=True.  q_prepped: q is the
    output of query_prep."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_c, "kv_c", torch.bfloat16, 3)
    _need(idx, "idx", torch.int32, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    B, T, H, D = q.shape
    k = idx.shape[2]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if not partials:
        o, lse = _attn_out(q, o, lse)
    workspace, wsb = _ws(KIND_SPARSE, q, k, workspace, q_prepped, partials)
    _check(lib().hattn_sparse_attn(_ptr(q), _ptr(gamma_q), int(bool(q_prepped)), _ptr(kv_c), _ptr(idx), _ptr(pos), B, T,
                                   H, D, kv_c.shape[1], k, r, rope_base, eps, scale, _ptr(o),
                                   _ptr(lse), _ptr(workspace), wsb, _stream(stream)))
    return _result(KIND_SPARSE, q, k, o, lse, workspace, q_prepped, partials)


def hca_attn(q, kv_h, pos, *, r, m=128, gamma_q=None, rope_base=10000.0, eps=1e-6, scale=None,
             o=None, lse=None, workspace=None, q_prepped=False, partials=False, stream=None):
    """HCA branch, dense over the visible compressed entries; returns (o, lse)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_h, "kv_h", torch.bfloat16, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    B, T, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if not partials:
        o, lse = _attn_out(q, o, lse)
    workspace, wsb = _ws(KIND_HCA, q, kv_h.shape[1], workspace, q_prepped, partials)
    _check(lib().hattn_hca_attn(_ptr(q), _ptr(gamma_q), int(bool(q_prepped)), _ptr(kv_h), _ptr(pos), B, T, H, D,
                                kv_h.shape[1], m, r, rope_base, eps, scale, _ptr(o), _ptr(lse),
                                _ptr(workspace), wsb, _stream(stream)))
    return _result(KIND_HCA, q, kv_h.shape[1], o, lse, workspace, q_prepped, partials)


def swa_attn(q, kv_raw, pos, *, r, W=128, gamma_q=None, gamma_kv=None, rope_base=10000.0,
             eps=1e-6, scale=None, o=None, lse=None, workspace=None, q_prepped=False,
             partials=False, stream=None):
    """SWA branch over the last W raw tokens (normalised and roped on load)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, T, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if not partials:
        o, lse = _attn_out(q, o, lse)
    workspace, wsb = _ws(KIND_SWA, q, W, workspace, q_prepped, partials)
    _check(lib().hattn_swa_attn(_ptr(q), _ptr(gamma_q), int(bool(q_prepped)), _ptr(kv_raw), _ptr(gamma_kv), _ptr(pos),
                                B, T, H, D, kv_raw.shape[1], W, r, rope_base, eps, scale, _ptr(o),
                                _ptr(lse), _ptr(workspace), wsb, _stream(stream)))
    return _result(KIND_SWA, q, W, o, lse, workspace, q_prepped, partials)


def swa_keys(kv_raw, pos, *, r, W=128, gamma_kv=None, rope_base=10000.0, eps=1e-6, kv_w=None,
             stream=None):
    """The normalised, roped window tokens of every query, kv_w [B, T, W, D]
    bf16 (row j is token pos - W + 1 + j; zero rows before token 0)."""
    _need(kv_raw, "kv_raw", torch.bfloat16, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_kv, "gamma_kv", torch.float32)
    B, L, D = kv_raw.shape
    T = pos.shape[1]
    if kv_w is None:
        kv_w = torch.empty((B, T, W, D), dtype=torch.bfloat16, device=kv_raw.device)
    _need(kv_w, "kv_w", torch.bfloat16, 4)
    _check(lib().hattn_swa_keys(_ptr(kv_raw), _ptr(gamma_kv), _ptr(pos), B, T, L, D, W, r,
                                rope_base, eps, _ptr(kv_w), _stream(stream)))
    return kv_w


SEG_CSA, SEG_HCA, SEG_SWA, SEG_ALL = 1, 2, 4, 7


def hybrid_attn_workspace_bytes(B, T, H, D, k, N_h, W, q_prepped=False, partials=False,
                                segments=SEG_ALL, n_sms=0):
    return lib().hattn_hybrid_attn_workspace_bytes(B, T, H, D, k, N_h, W, segments, n_sms,
                                                   int(bool(q_prepped)), int(bool(partials)))


def hybrid_attn_splits(B, T, H, D, k, N_h, W, segments=SEG_ALL, n_sms=0):
    return lib().hattn_hybrid_attn_splits(B, T, H, D, k, N_h, W, segments, n_sms)


def hybrid_attn(q, kv_c, idx, kv_h, kv_w, pos, *, r, m=128, k=None, W=None, gamma_q=None,
                rope_base=10000.0, eps=1e-6, scale=None, o=None, lse=None, workspace=None,
                q_prepped=False, partials=False, segments=SEG_ALL, n_sms=0, dependent=False,
                stream=None):
    """CSA (selected entries), HCA (visible entries) and SWA (kv_w from
    swa_keys) keys of each query under one softmax; returns (o fp32, lse
    fp32) or, with partials=True, a Partials view of the workspace.
    segments: the key sets covered (SEG_* mask; tensors of the others may be
    None); n_sms: the SM share the split plan assumes (0 = all); dependent:
    launch as a programmatic dependent of the previous kernel in the stream."""
    _need(q, "q", torch.bfloat16, 4)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    B, T, H, D = q.shape
    if segments & SEG_CSA:
        _need(kv_c, "kv_c", torch.bfloat16, 3)
        _need(idx, "idx", torch.int32, 3)
    if segments & SEG_HCA:
        _need(kv_h, "kv_h", torch.bfloat16, 3)
    if segments & SEG_SWA:
        _need(kv_w, "kv_w", torch.bfloat16, 4)
    k = idx.shape[2] if idx is not None else (k or 1)
    N_h = kv_h.shape[1] if kv_h is not None else 1
    N_c = kv_c.shape[1] if kv_c is not None else 1
    W = kv_w.shape[2] if kv_w is not None else (W or 1)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if not partials:
        o, lse = _attn_out(q, o, lse)
    need = hybrid_attn_workspace_bytes(B, T, H, D, k, N_h, W, q_prepped, partials, segments,
                                       n_sms)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().hattn_hybrid_attn(_ptr(q), _ptr(gamma_q), int(bool(q_prepped)), _ptr(kv_c),
                                   _ptr(idx), N_c, k, _ptr(kv_h), N_h, m, _ptr(kv_w), W,
                                   _ptr(pos), B, T, H, D, r, rope_base, eps, scale, segments,
                                   n_sms, _ptr(o), _ptr(lse), _ptr(workspace), wsb,
                                   _flags(dependent), _stream(stream)))
    if not partials:
        return o, lse
    return Partials(workspace, q_prepped, B, T, H, D,
                    hybrid_attn_splits(B, T, H, D, k, N_h, W, segments, n_sms))


def hybrid_attn_out_workspace_bytes(B, T, H, D, k, N_h, W, q_prepped=False, segments=SEG_ALL,
                                    n_sms=0):
    return lib().hattn_hybrid_attn_out_workspace_bytes(B, T, H, D, k, N_h, W, segments, n_sms,
                                                       int(bool(q_prepped)))


def hybrid_attn_out(q, kv_c, idx, kv_h, kv_w, pos, *, r, m=128, k=None, W=None, gamma_q=None,
                    rope_base=10000.0, eps=1e-6, scale=None, sink=None, out=None, lse_out=None,
                    workspace=None, q_prepped=False, segments=SEG_ALL, n_sms=0,
                    dependent=False, stream=None):
    """hybrid_attn straight to the layer output: the sink merge and the
    inverse RoPE of the call's one softmax (in the attention kernel when
    every query's keys take one split, else by a merge that follows).
    Returns (out bf16 [B, T, H, D], lse fp32 [B, T, H])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(pos, "pos", torch.int32, 2)
    _opt(gamma_q, "gamma_q", torch.float32)
    B, T, H, D = q.shape
    if segments & SEG_CSA:
        _need(kv_c, "kv_c", torch.bfloat16, 3)
        _need(idx, "idx", torch.int32, 3)
    if segments & SEG_HCA:
        _need(kv_h, "kv_h", torch.bfloat16, 3)
    if segments & SEG_SWA:
        _need(kv_w, "kv_w", torch.bfloat16, 4)
    if sink is not None:
        _need(sink, "sink", torch.float32, 1)
        _shape(sink, "sink", (H,))
    k = idx.shape[2] if idx is not None else (k or 1)
    N_h = kv_h.shape[1] if kv_h is not None else 1
    N_c = kv_c.shape[1] if kv_c is not None else 1
    W = kv_w.shape[2] if kv_w is not None else (W or 1)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if out is None:
        out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    _shape(out, "out", (B, T, H, D))
    if lse_out is None:
        lse_out = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
    _need(lse_out, "lse_out", torch.float32, 3)
    _shape(lse_out, "lse_out", (B, T, H))
    need = hybrid_attn_out_workspace_bytes(B, T, H, D, k, N_h, W, q_prepped, segments, n_sms)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().hattn_hybrid_attn_out(_ptr(q), _ptr(gamma_q), int(bool(q_prepped)), _ptr(kv_c),
                                       _ptr(idx), N_c, k, _ptr(kv_h), N_h, m, _ptr(kv_w), W,
                                       _ptr(pos), B, T, H, D, r, rope_base, eps, scale, segments,
                                       n_sms, _ptr(sink), _ptr(out), _ptr(lse_out),
                                       _ptr(workspace), wsb, _flags(dependent), _stream(stream)))
    return out, lse_out


# ------------------------------------------------------------------ merge
def lse_merge(o_list, lse_list, pos, *, r, sink=None, rope_base=10000.0, out=None, lse_out=None,
              stream=None):
    """Sink-augmented LSE merge of 1..4 branches + inverse RoPE; returns (out, lse)."""
    nb = len(o_list)
    if nb < 1 or nb != len(lse_list):
        raise ValueError("need 1..4 branches with matching lse tensors")
    for i, (o, l) in enumerate(zip(o_list, lse_list)):
        _need(o, f"o_list[{i}]", torch.float32, 4)
        _need(l, f"lse_list[{i}]", torch.float32, 3)
    _need(pos, "pos", torch.int32, 2)
    _opt(sink, "sink", torch.float32)
    B, T, H, D = o_list[0].shape
    if out is None:
        out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=o_list[0].device)
    if lse_out is None:
        lse_out = torch.empty((B, T, H), dtype=torch.float32, device=o_list[0].device)
    _need(out, "out", torch.bfloat16)
    _need(lse_out, "lse_out", torch.float32)
    op = (_vp * nb)(*[o.data_ptr() for o in o_list])
    lp = (_vp * nb)(*[l.data_ptr() for l in lse_list])
    _check(lib().hattn_lse_merge(op, lp, nb, _ptr(sink), _ptr(pos), B, T, H, D, r, rope_base,
                                 _ptr(out), _ptr(lse_out), _stream(stream)))
    return out, lse_out


def lse_merge_splits(parts, pos, *, r, H, sink=None, rope_base=10000.0, out=None, lse_out=None,
                     dependent=False, stream=None):
    """Sink-augmented merge over the split partials of 1..4 branches (a list
    of Partials) + inverse RoPE; returns (out bf16 [B, T, H, D], lse)."""
    nb = len(parts)
    if nb < 1:
        raise ValueError("need 1..4 branches")
    _need(pos, "pos", torch.int32, 2)
    _opt(sink, "sink", torch.float32)
    B, T = pos.shape
    D = parts[0].o.shape[2]
    dev = parts[0].o.device
    if out is None:
        out = torch.empty((B, T, H, D), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16)
    _need(lse_out, "lse_out", torch.float32)
    op = (_vp * nb)(*[p.o.data_ptr() for p in parts])
    lp = (_vp * nb)(*[p.lse.data_ptr() for p in parts])
    ns = (_i32 * nb)(*[p.nsplit for p in parts])
    _check(lib().hattn_lse_merge_splits(op, lp, ns, nb, _ptr(sink), _ptr(pos), B, T, H, D, r,
                                        rope_base, _ptr(out), _ptr(lse_out), _flags(dependent),
                                        _stream(stream)))
    return out, lse_out


# ------------------------------------------------------------------ status
def _bounded_sync(stream=None, timeout_s=120.0):
    import time
    s = stream if stream is not None else torch.cuda.current_stream()
    t_end = time.monotonic() + timeout_s
    while not s.query():
        if time.monotonic() > t_end:
            raise TimeoutError(f"GPU work did not finish within {timeout_s} s")
        time.sleep(1e-4)


def check_status(stream=None, timeout_s=120.0):
    """Synchronise (waiting at most timeout_s) and raise if a kernel reported
    a device-side error."""
    _bounded_sync(stream, timeout_s)
    _check(lib().hattn_check_status(_stream(stream)))


def check_status_code(stream=None, timeout_s=120.0):
    _bounded_sync(stream, timeout_s)
    return int(lib().hattn_check_status(_stream(stream)))


def selftest_wait_timeout(timeout_ns, stream=None):
    _check(lib().hattn_selftest_wait_timeout(int(timeout_ns), _stream(stream)))


def status_string(code):
    return lib().hattn_status_string(code).decode()


def version():
    return lib().hattn_version().decode()
