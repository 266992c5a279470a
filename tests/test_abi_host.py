"""Host-side checks of the C ABI: the library loads on a machine without a
GPU, exports every entry point of include/hattn.h, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

from sparse_attention_26_b300 import hattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hattn.h")


@pytest.fixture(scope="module")
def L():
    from sparse_attention_26_b300 import build
    build.build()
    return hattn.lib()


def header_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"HATTN_API\s+[\w\s\*]+?\b(hattn_\w+)\s*\(", txt)))


def test_header_declares_the_seven_calls():
    syms = header_symbols()
    for name in ["csa_compress", "hca_compress", "indexer_topk", "sparse_attn", "hca_attn",
                 "swa_attn", "lse_merge"]:
        assert f"hattn_{name}" in syms


def test_library_exports_every_declared_symbol(L):
    syms = header_symbols()
    assert len(syms) >= 14
    for s in syms:
        assert hasattr(L, s), f"{s} declared in hattn.h but not exported"
        assert s in hattn._SIGS, f"{s} has no binding signature"


def test_binding_signatures_match_the_header():
    """Every ctypes signature in the binding has the header's parameter count,
    and each parameter the header's kind (pointer, int, int64, float, size_t,
    uint64), so no call passes arguments the library reads differently."""
    txt = open(os.path.join(ROOT, "include", "hattn.h")).read()
    decls = re.findall(r"HATTN_API\s+([^;]*?)\b(hattn_\w+)\s*\(([^)]*)\)\s*;", txt, re.S)
    assert len(decls) == len(header_symbols())
    ptr_array = ctypes.POINTER(ctypes.c_void_p)
    scalar = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "float": ctypes.c_float,
              "size_t": ctypes.c_size_t, "uint64_t": ctypes.c_uint64}
    ret_kind = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char*": ctypes.c_char_p}
    for ret, name, params in decls:
        restype, argtypes = hattn._SIGS[name]
        assert restype is ret_kind[" ".join(ret.split())], name
        ps = [" ".join(p.split()) for p in params.split(",")]
        ps = [p for p in ps if p and p != "void"]
        assert len(ps) == len(argtypes), f"{name}: header {len(ps)} args, binding {len(argtypes)}"
        for i, (p, a) in enumerate(zip(ps, argtypes)):
            ctype = re.sub(r"\s*\b\w+$", "", p)
            if ctype.endswith("* const*"):
                assert a is ptr_array, (name, i, p)
            elif ctype.endswith("*") or ctype == "hattn_stream_t":
                assert a is ctypes.c_void_p or issubclass(a, ctypes._Pointer), (name, i, p)
            else:
                assert a is scalar[ctype], (name, i, p, a)


def test_status_strings(L):
    assert hattn.status_string(0) == "ok"
    assert "misaligned" in hattn.status_string(2)
    assert "timed out" in hattn.status_string(5)
    assert hattn.version().startswith("hattn")


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
MISAL = ctypes.c_void_p(0x10008)


def _err(L):
    return L.hattn_last_error().decode()


def test_compress_validation(L):
    N = None
    s = None
    rc = L.hattn_csa_compress(N, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0, 4, FAKE,
                              FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "kv_raw" in _err(L)
    rc = L.hattn_csa_compress(MISAL, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0, 4,
                              FAKE, FAKE, 16, s)
    assert rc == hattn.MISALIGNED
    # w % m != 0
    rc = L.hattn_csa_compress(FAKE, FAKE, FAKE, N, 1, 64, 64, 32, 4, 6, 16, 1e4, 1e-6, 0, 4, FAKE,
                              FAKE, 16, s)
    assert rc == hattn.INVALID_ARG
    # D not a multiple of 64
    rc = L.hattn_csa_compress(FAKE, FAKE, FAKE, N, 1, 64, 96, 32, 4, 8, 16, 1e4, 1e-6, 0, 4, FAKE,
                              FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "D=96" in _err(L)
    # entries need tokens beyond L_cap
    rc = L.hattn_csa_compress(FAKE, FAKE, FAKE, N, 1, 15, 64, 32, 4, 8, 16, 1e4, 1e-6, 0, 4, FAKE,
                              FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "L_cap" in _err(L)
    # odd RoPE width
    rc = L.hattn_hca_compress(FAKE, FAKE, N, 1, 256, 64, 128, 15, 1e4, 1e-6, 0, 2, FAKE, 2, s)
    assert rc == hattn.INVALID_ARG
    # empty range is a no-op that succeeds without a device
    rc = L.hattn_hca_compress(FAKE, FAKE, N, 1, 256, 64, 128, 16, 1e4, 1e-6, 1, 1, FAKE, 2, s)
    assert rc == hattn.OK


def test_indexer_validation(L):
    N = None
    rc = L.hattn_indexer_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 128, 100, 0, 4, FAKE, N, N, 0, N)
    assert rc == hattn.INVALID_ARG and "k=0" in _err(L)
    rc = L.hattn_indexer_topk(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 120 + 3, 100, 16, 4, FAKE, N, N,
                              0, N)
    assert rc == hattn.INVALID_ARG
    rc = L.hattn_indexer_topk(FAKE, FAKE, FAKE, N, 1, 1, 64, 128, 100, 16, 4, FAKE, N, N, 0, N)
    assert rc == hattn.INVALID_ARG and "pos" in _err(L)
    # the scores, the score kernel's partial histograms (two rows of 2,048
    # 16-bit bins per CTA, one CTA per SM: 148 without a device), then the
    # selection's scratch; rows that fit one CTA need neither of the last two
    sel = L.hattn_topk_workspace_bytes(8, 1, 262144, 1024)
    assert sel == 8 * 262144 * 4  # one candidate slot per entry
    hist = 148 * 2 * 2048 * 2
    assert L.hattn_indexer_topk_workspace_bytes(8, 1, 262144, 1024, 0) == 8 * 262144 * 4 + hist + sel
    assert L.hattn_indexer_topk_workspace_bytes(8, 1, 262144, 1024, 1) == hist + sel
    # the extended call checks its own arguments before any launch
    rc = L.hattn_indexer_topk_ex(FAKE, FAKE, FAKE, N, FAKE, 8, 1, 64, 128, 262144, 1024, 4, 0, -1,
                                 FAKE, N, FAKE, hist + sel, 8, N, N)
    assert rc == hattn.INVALID_ARG and "flags" in _err(L)
    rc = L.hattn_indexer_topk_ex(FAKE, FAKE, FAKE, N, FAKE, 8, 1, 64, 128, 262144, 1024, 4, -1, -1,
                                 FAKE, N, FAKE, hist + sel, 0, N, N)
    assert rc == hattn.INVALID_ARG and "n_sms" in _err(L)
    rc = L.hattn_indexer_topk_ex(FAKE, FAKE, FAKE, N, FAKE, 8, 1, 64, 128, 262144, 1024, 4, 0, -1,
                                 FAKE, FAKE, FAKE, hist + sel - 1, 0, N, N)
    assert rc == hattn.INVALID_ARG and "workspace" in _err(L)
    assert L.hattn_topk_workspace_bytes(8192, 1, 2048, 512) == 0
    assert L.hattn_indexer_topk_workspace_bytes(1, 8192, 2048, 512, 0) == 8192 * 2048 * 4


def test_topk_validation(L):
    """Arguments of the selection are checked before any launch: unknown
    flag bits, a missing or short scratch where the plan needs one, k."""
    N = None
    s = None
    sel = L.hattn_topk_workspace_bytes(8, 1, 262144, 1024)
    # hattn_topk_select(scores, pos, B, T, N_cap, k, m, idx_out, ws, ws_bytes, flags, stream)
    rc = L.hattn_topk_select(FAKE, FAKE, 8, 1, 262144, 1024, 4, FAKE, FAKE, sel, 4, s)
    assert rc == hattn.INVALID_ARG and "flags" in _err(L)
    rc = L.hattn_topk_select(FAKE, FAKE, 8, 1, 262144, 1024, 4, FAKE, N, 0, 0, s)
    assert rc == hattn.INVALID_ARG and "workspace" in _err(L)
    rc = L.hattn_topk_select(FAKE, FAKE, 8, 1, 262144, 1024, 4, FAKE, FAKE, sel - 1, 0, s)
    assert rc == hattn.INVALID_ARG and "workspace" in _err(L)
    rc = L.hattn_topk_select(FAKE, FAKE, 8, 1, 262144, 4096, 4, FAKE, FAKE, sel, 0, s)
    assert rc == hattn.INVALID_ARG and "k=4096" in _err(L)
    rc = L.hattn_topk_select(FAKE, FAKE, 8, 1, 1 << 31, 1024, 4, FAKE, FAKE, sel, 0, s)
    assert rc == hattn.INVALID_ARG and "N_cap" in _err(L)


def test_launch_flags_are_per_call(L):
    """No launch mode is kept between calls: the dependent-launch choice is
    a flag of each call that may launch that way, and unknown bits are
    refused."""
    import re
    assert not hasattr(L, "hattn_set_dependent_launch")
    with open(HEADER) as f:
        hdr = f.read()
    assert re.search(r"#define\s+HATTN_LAUNCH_DEPENDENT\s+1\b", hdr)
    for name in ["hattn_indexer_scores_ex", "hattn_indexer_scores_fp8", "hattn_topk_select",
                 "hattn_hybrid_attn", "hattn_lse_merge_splits"]:
        decl = re.search(name + r"\(([^;]*)\);", hdr).group(1)
        params = [x.strip() for x in decl.split(",")]
        assert params[-2] == "int flags" and params[-1].startswith("hattn_stream_t"), name
    N = None
    rc = L.hattn_indexer_scores_ex(FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 128, 100, 4, 0, -1, FAKE, 4,
                                   N)
    assert rc == hattn.INVALID_ARG and "flags" in _err(L)


def test_fp8_key_validation(L):
    N = None
    s = None
    # FP8 indexer keys are one 128-byte row: dI = 64 is rejected before any launch
    rc = L.hattn_indexer_scores_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 100, 4, 0, -1,
                                    FAKE, 0, s)
    assert rc == hattn.INVALID_ARG and "dI = 128" in _err(L)
    rc = L.hattn_indexer_scores_fp8(FAKE, FAKE, FAKE, N, FAKE, 1, 1, 64, 128, 100, 4, 0, -1,
                                    FAKE, 0, s)
    assert rc == hattn.INVALID_ARG and "ik_scale" in _err(L)
    # the scales travel in 16-byte rows: N_cap a multiple of 4
    rc = L.hattn_indexer_scores_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 128, 102, 4, 0, -1,
                                    FAKE, 0, s)
    assert rc == hattn.INVALID_ARG and "N_cap % 4" in _err(L)
    rc = L.hattn_indexer_scores_fp8(FAKE, FAKE, FAKE, MISAL, FAKE, 1, 1, 64, 128, 100, 4, 0, -1,
                                    FAKE, 0, s)
    assert rc == hattn.MISALIGNED
    # the compressor's FP8 key needs both the codes and the scales
    rc = L.hattn_csa_compress_fp8(FAKE, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0, 4,
                                  FAKE, N, FAKE, N, 16, s)
    assert rc == hattn.INVALID_ARG and "ik_scale" in _err(L)
    rc = L.hattn_csa_compress_fp8(FAKE, N, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0, 4,
                                  FAKE, N, FAKE, FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "ik_raw" in _err(L)
    # an empty range succeeds without a device
    rc = L.hattn_csa_compress_fp8(FAKE, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 2, 2,
                                  FAKE, N, FAKE, FAKE, 16, s)
    assert rc == hattn.OK
    rc = L.hattn_quantize_e4m3(FAKE, 10, 6, FAKE, FAKE, s)
    assert rc == hattn.INVALID_ARG and "n=6" in _err(L)
    assert L.hattn_quantize_e4m3(FAKE, 0, 128, FAKE, FAKE, s) == hattn.OK


def test_mxfp4_validation(L):
    N = None
    s = None
    # MXFP4 rows are whole 32-element blocks
    for n in (16, 48, 0):
        rc = L.hattn_quantize_mxfp4(FAKE, 10, n, FAKE, FAKE, s)
        assert rc == hattn.INVALID_ARG and f"n={n}" in _err(L)
    rc = L.hattn_quantize_mxfp4(FAKE, -1, 128, FAKE, FAKE, s)
    assert rc == hattn.INVALID_ARG and "rows" in _err(L)
    rc = L.hattn_quantize_mxfp4(FAKE, 10, 128, FAKE, N, s)
    assert rc == hattn.INVALID_ARG and "scales" in _err(L)
    rc = L.hattn_quantize_mxfp4(FAKE, 10, 128, MISAL, FAKE, s)
    assert rc == hattn.MISALIGNED and "codes" in _err(L)
    assert L.hattn_quantize_mxfp4(FAKE, 0, 128, FAKE, FAKE, s) == hattn.OK
    # no rows: nothing is read or written, so null pointers (an empty tensor's) pass
    assert L.hattn_quantize_mxfp4(N, 0, 128, N, N, s) == hattn.OK
    assert L.hattn_quantize_e4m3(N, 0, 128, N, N, s) == hattn.OK
    # an entry range of a cache: inside [0, N_cap); an empty one touches nothing
    rc = L.hattn_quantize_mxfp4_entries(FAKE, 2, 100, 128, 90, 101, FAKE, FAKE, s)
    assert rc == hattn.INVALID_ARG and "entry range" in _err(L)
    rc = L.hattn_quantize_mxfp4_entries(FAKE, 2, 100, 48, 0, 10, FAKE, FAKE, s)
    assert rc == hattn.INVALID_ARG and "n=48" in _err(L)
    assert L.hattn_quantize_mxfp4_entries(N, 2, 100, 128, 5, 5, N, N, s) == hattn.OK
    # the compressor's MXFP4 key needs the bf16 key, the codes and the scales,
    # and whole 32-element blocks
    rc = L.hattn_csa_compress_mxfp4(FAKE, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0,
                                    4, FAKE, FAKE, FAKE, N, 16, s)
    assert rc == hattn.INVALID_ARG and "ik4_scale" in _err(L)
    rc = L.hattn_csa_compress_mxfp4(FAKE, FAKE, FAKE, N, 1, 64, 64, 32, 4, 8, 16, 1e4, 1e-6, 0,
                                    4, FAKE, N, FAKE, FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "ik_c" in _err(L)
    rc = L.hattn_csa_compress_mxfp4(FAKE, FAKE, FAKE, N, 1, 64, 64, 40, 4, 8, 16, 1e4, 1e-6, 0,
                                    4, FAKE, FAKE, FAKE, FAKE, 16, s)
    assert rc == hattn.INVALID_ARG and "multiple of 32" in _err(L)
    # MXFP4 scoring: dI = 128, and queries in groups of at most 128 rows
    rc = L.hattn_indexer_scores_mxfp4(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 64, 64, 100, 4, 0, -1,
                                      FAKE, 0, s)
    assert rc == hattn.INVALID_ARG and "dI = 128" in _err(L)


def test_ring_and_hidden_validation(L):
    N = None
    s = None
    # a ring must be a power of two equal to L_cap, and hold the entries' windows
    rc = L.hattn_csa_compress_ring(FAKE, FAKE, FAKE, N, 1, 200, 512, 128, 4, 8, 64, 1e4, 1e-6,
                                   0, 10, FAKE, FAKE, 100, s)
    assert rc == hattn.INVALID_ARG and "power of two" in _err(L)
    rc = L.hattn_csa_compress_ring(FAKE, FAKE, FAKE, N, 1, 256, 512, 128, 4, 8, 64, 1e4, 1e-6,
                                   0, 100, FAKE, FAKE, 100, s)
    assert rc == hattn.INVALID_ARG and "span more tokens" in _err(L)
    rc = L.hattn_hca_compress_ring(FAKE, FAKE, N, 1, 256, 512, 128, 64, 1e4, 1e-6, 5, 8, FAKE,
                                   10, s)  # three 128-token entries
    assert rc == hattn.INVALID_ARG and "span more tokens" in _err(L)
    rc = L.hattn_swa_keys_ring(FAKE, N, FAKE, 1, 2, 128, 512, 128, 64, 1e4, 1e-6, FAKE, s)
    assert rc == hattn.INVALID_ARG and "W + T - 1" in _err(L)
    # entries from hidden states: d_model a multiple of 8, the indexer-key
    # output exactly when dI > 0, a large enough workspace
    rc = L.hattn_compress_hidden(FAKE, FAKE, FAKE, N, 1, 1024, 100, 512, 128, 4, 8, 64, 1e4, 1e-6,
                                 0, 256, FAKE, FAKE, 256, FAKE, 1 << 30, s)
    assert rc == hattn.INVALID_ARG and "dm=100" in _err(L)
    rc = L.hattn_compress_hidden(FAKE, FAKE, FAKE, N, 1, 1024, 512, 512, 128, 4, 8, 64, 1e4, 1e-6,
                                 0, 256, FAKE, N, 256, FAKE, 1 << 30, s)
    assert rc == hattn.INVALID_ARG and "ik_out" in _err(L)
    # the two bf16 parts (hi, lo) of each pooled row; the projection keeps
    # its fp32 result in tensor memory
    need = L.hattn_compress_hidden_workspace_bytes(1, 0, 256, 512, 512, 128)
    assert need == 2 * 256 * 512 * 2
    rc = L.hattn_compress_hidden(FAKE, FAKE, FAKE, N, 1, 1024, 512, 512, 128, 4, 8, 64, 1e4, 1e-6,
                                 0, 256, FAKE, FAKE, 256, FAKE, need - 1, s)
    assert rc == hattn.INVALID_ARG and "workspace" in _err(L)
    assert L.hattn_compress_hidden_workspace_bytes(1, 5, 5, 512, 512, 128) == 0


def test_attention_validation(L):
    N = None
    rc = L.hattn_sparse_attn(FAKE, N, 0, FAKE, N, FAKE, 1, 1, 128, 512, 100, 16, 64, 1e4, 1e-6,
                             0.04, FAKE, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "idx" in _err(L)
    rc = L.hattn_hca_attn(FAKE, N, 0, FAKE, FAKE, 1, 1, 256, 512, 100, 128, 64, 1e4, 1e-6, 0.04,
                          FAKE, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "H=256" in _err(L)
    rc = L.hattn_swa_attn(FAKE, N, 1, FAKE, N, FAKE, 1, 1, 128, 512, 100, 0, 64, 1e4, 1e-6, 0.04,
                          FAKE, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG
    rc = L.hattn_hca_attn(FAKE, N, 0, FAKE, FAKE, 1, 1, 128, 512, 100, 128, 200, 1e4, 1e-6, 0.04,
                          FAKE, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "r=200" in _err(L)
    # raw queries are prepared into the workspace, which is then required
    rc = L.hattn_hca_attn(FAKE, N, 0, FAKE, FAKE, 1, 1, 128, 512, 100, 128, 64, 1e4, 1e-6, 0.04,
                          FAKE, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "workspace" in _err(L)
    # D above 256 is split in halves of whole 64-wide chunks
    rc = L.hattn_hca_attn(FAKE, N, 1, FAKE, FAKE, 1, 1, 128, 320, 100, 128, 64, 1e4, 1e-6, 0.04,
                          FAKE, FAKE, N, 0, N)
    assert rc == hattn.UNSUPPORTED
    rc = L.hattn_query_prep(FAKE, N, N, 1, 1, 4, 64, 16, 1e4, 1e-6, FAKE, N)
    assert rc == hattn.INVALID_ARG and "pos" in _err(L)
    rc = L.hattn_query_prep(MISAL, N, FAKE, 1, 1, 4, 64, 16, 1e4, 1e-6, FAKE, N)
    assert rc == hattn.MISALIGNED
    # the merge needs 1..4 branches
    arr = (ctypes.c_void_p * 1)(FAKE)
    rc = L.hattn_lse_merge(arr, arr, 0, N, FAKE, 1, 1, 1, 64, 0, 1e4, FAKE, N, N)
    assert rc == hattn.INVALID_ARG


def test_workspace_sizes_scale_with_splits(L):
    # decode at the 1M-context shape splits keys across SMs and needs partials
    part = hattn.attn_workspace_bytes(hattn.KIND_HCA, 8, 1, 128, 512, 8192, q_prepped=True)
    assert part > 0
    # raw queries add their prepared copy (B*T*H*D bf16) in front
    full = hattn.attn_workspace_bytes(hattn.KIND_HCA, 8, 1, 128, 512, 8192)
    assert full == part + 8 * 1 * 128 * 512 * 2
    # a long prefill row block has no split and needs no partials
    assert hattn.attn_workspace_bytes(hattn.KIND_SPARSE, 1, 8192, 64, 512, 512,
                                      q_prepped=True) == 0


def test_split_counts_and_partials_workspace(L):
    # the 1M decode HCA branch splits its 8192 keys across the SMs
    n = hattn.attn_splits(hattn.KIND_HCA, 8, 1, 128, 512, 8192)
    assert n > 1
    part = hattn.attn_workspace_bytes(hattn.KIND_HCA, 8, 1, 128, 512, 8192, q_prepped=True,
                                      partials=True)
    assert part == 8 * 128 * n * (512 + 1) * 4
    # partials are kept even when a call has a single split
    assert hattn.attn_splits(hattn.KIND_SPARSE, 1, 8192, 64, 512, 512) == 1
    assert hattn.attn_workspace_bytes(hattn.KIND_SPARSE, 1, 8192, 64, 512, 512, q_prepped=True,
                                      partials=True) == 8192 * 64 * 513 * 4
    assert hattn.attn_splits(7, 1, 1, 1, 64, 10) == 0


def test_merge_splits_validation(L):
    N = None
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    ns = (ctypes.c_int * 2)(100, 40)
    rc = L.hattn_lse_merge_splits(arr, arr, ns, 2, N, FAKE, 1, 1, 1, 64, 0, 1e4, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "partials" in _err(L)
    ns = (ctypes.c_int * 2)(3, 0)
    rc = L.hattn_lse_merge_splits(arr, arr, ns, 2, N, FAKE, 1, 1, 1, 64, 0, 1e4, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG and "nsplit" in _err(L)
    rc = L.hattn_lse_merge_splits(arr, arr, N, 2, N, FAKE, 1, 1, 1, 64, 0, 1e4, FAKE, N, 0, N)
    assert rc == hattn.INVALID_ARG


def test_fused_attention_validation_and_sizes(L):
    N = None
    # hattn_hybrid_attn(q, gamma_q, q_prepped, kv_c, idx, N_c, k, kv_h, N_h, m, kv_w, W, pos,
    #                   B, T, H, D, r, rope_base, eps, scale, segments, n_sms, o, lse, ws,
    #                   ws_bytes, flags, stream)
    args = [FAKE, N, 1, FAKE, FAKE, 1000, 64, FAKE, 100, 128, FAKE, 128, FAKE,
            2, 1, 128, 512, 64, 1e4, 1e-6, 0.04, 7, 0, FAKE, FAKE, FAKE, 1 << 30, 0, N]
    bad = list(args)
    bad[10] = N  # no SWA key buffer
    assert L.hattn_hybrid_attn(*bad) == hattn.INVALID_ARG and "kv_w" in _err(L)
    bad = list(args)
    bad[8] = 0  # empty HCA cache
    assert L.hattn_hybrid_attn(*bad) == hattn.INVALID_ARG and "HCA" in _err(L)
    bad = list(args)
    bad[4] = N  # no top-k indices
    assert L.hattn_hybrid_attn(*bad) == hattn.INVALID_ARG and "idx" in _err(L)
    bad = list(args)
    bad[21] = 8  # not a segment mask
    assert L.hattn_hybrid_attn(*bad) == hattn.INVALID_ARG and "segments" in _err(L)
    # without the CSA segment the top-k indices and the CSA cache are not
    # needed: validation gets as far as the (too small) workspace, so nothing
    # is ever launched on these fake pointers
    ok_args = list(args)
    ok_args[3], ok_args[4], ok_args[21], ok_args[23], ok_args[24] = N, N, 6, N, N
    ok_args[26] = 16
    assert L.hattn_hybrid_attn(*ok_args) == hattn.INVALID_ARG and "workspace" in _err(L)
    # a smaller SM share plans fewer splits
    assert (hattn.hybrid_attn_splits(8, 1, 128, 512, 1024, 8192, 128, segments=6, n_sms=48)
            < hattn.hybrid_attn_splits(8, 1, 128, 512, 1024, 8192, 128, segments=6))
    # the fused call splits its keys like the branches and keeps partials per split
    n = hattn.hybrid_attn_splits(8, 1, 128, 512, 1024, 8192, 128)
    assert n > 1
    assert hattn.hybrid_attn_workspace_bytes(8, 1, 128, 512, 1024, 8192, 128, q_prepped=True,
                                             partials=True) == 8 * 128 * n * (512 + 1) * 4
    # hattn_swa_keys(kv_raw, gamma_kv, pos, B, T, L_cap, D, W, r, rope_base, eps, kv_w, stream)
    assert L.hattn_swa_keys(FAKE, N, FAKE, 1, 1, 100, 512, 0, 64, 1e4, 1e-6, FAKE,
                            N) == hattn.INVALID_ARG
    assert L.hattn_swa_keys(FAKE, N, FAKE, 1, 1, 100, 512, 128, 64, 1e4, 1e-6, MISAL,
                            N) == hattn.MISALIGNED


def test_no_fallback_without_the_library_or_a_gpu(monkeypatch):
    """The binding has no CPU or PyTorch path: with the library missing it
    raises, and CPU tensors are refused before any call."""
    import torch
    x = torch.zeros((4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        hattn.quantize_mxfp4(x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        hattn.quantize_e4m3(x)
    monkeypatch.setattr(hattn, "_lib", None)
    monkeypatch.setattr(hattn, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libhattn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        hattn.lib()
