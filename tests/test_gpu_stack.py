"""GPU parity of the ring-buffer calls and of a multi-layer decode loop.

The ring forms read token u from row u mod ring, so on the same tokens they
must give exactly what the linear forms give.  The decode loop runs the layer
pattern of the pages (two sliding-window layers, then CSA and HCA layers)
token by token through compression boundaries, and each checked step is
compared with the fp64 oracle layer by layer.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from sparse_attention_26_b300 import hattn, synth
from sparse_attention_26_b300.stack import CSA, HCA, SWA, DecodeStack

from _util import KV_REL_L2, check_attn, check_topk, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_26_b300 import build
    build.build()
    hattn.lib()
    orc.lib()
    yield
    hattn.check_status()


def bits(t):
    return synth.bits(t)


def randn_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def to_ring(x, L, R):
    """The last R token rows of x [B][L][...] placed at rows u mod R."""
    ring = torch.zeros((x.shape[0], R) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    u = torch.arange(max(0, L - R), L, device=x.device)
    ring[:, u % R] = x[:, u]
    return ring


@pytest.mark.parametrize("L", [700, 1152])
def test_ring_forms_equal_linear_forms(L):
    """Compression of the newest entries and the window keys of the newest
    queries from a 256-row ring equal the linear calls bit for bit."""
    B, D, dI, r, R = 2, 512, 128, 64, 256
    kv = randn_bf16((B, L, D), 1).to(DEV)
    ik = randn_bf16((B, L, dI), 2).to(DEV)
    gc = randn_bf16((B, L), 3).to(DEV)
    gh = randn_bf16((B, L), 4).to(DEV)
    kv_r, ik_r, gc_r, gh_r = (to_ring(x, L, R) for x in (kv, ik, gc, gh))
    Nc, Nh = L // 4, L // 128
    j0 = Nc - 50  # the 50 newest CSA entries span 4*50 + 4 tokens
    a_kv = torch.zeros((B, Nc, D), dtype=torch.bfloat16, device=DEV)
    a_ik = torch.zeros((B, Nc, dI), dtype=torch.bfloat16, device=DEV)
    b_kv, b_ik = a_kv.clone(), a_ik.clone()
    hattn.csa_compress(kv, ik, gc, r=r, j_begin=j0, j_end=Nc, kv_c=a_kv, ik_c=a_ik)
    hattn.csa_compress_ring(kv_r, ik_r, gc_r, r=r, j_begin=j0, j_end=Nc, kv_c=b_kv, ik_c=b_ik)
    a_h = torch.zeros((B, Nh, D), dtype=torch.bfloat16, device=DEV)
    b_h = a_h.clone()
    hattn.hca_compress(kv, gh, r=r, j_begin=Nh - 1, j_end=Nh, kv_h=a_h)
    hattn.hca_compress_ring(kv_r, gh_r, r=r, j_begin=Nh - 1, j_end=Nh, kv_h=b_h)
    pos = torch.tensor([[L - 2, L - 1], [L - 2, L - 1]], dtype=torch.int32, device=DEV)
    a_w = hattn.swa_keys(kv, pos, r=r, W=128)
    b_w = hattn.swa_keys_ring(kv_r, pos, r=r, W=128)
    hattn.check_status()
    assert torch.equal(a_kv, b_kv) and torch.equal(a_ik, b_ik)
    assert torch.equal(a_h, b_h)
    assert torch.equal(a_w, b_w)


def test_ring_rejects_spans_it_cannot_hold():
    B, D, dI, R = 1, 512, 128, 256
    kv = torch.zeros((B, R, D), dtype=torch.bfloat16, device=DEV)
    ik = torch.zeros((B, R, dI), dtype=torch.bfloat16, device=DEV)
    g = torch.zeros((B, R), dtype=torch.bfloat16, device=DEV)
    kv_c = torch.zeros((B, 400, D), dtype=torch.bfloat16, device=DEV)
    ik_c = torch.zeros((B, 400, dI), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(hattn.HattnError):  # 100 entries span 404 tokens
        hattn.csa_compress_ring(kv, ik, g, r=64, j_begin=300, j_end=400, kv_c=kv_c, ik_c=ik_c)
    pos = torch.tensor([[1000, 1001]], dtype=torch.int32, device=DEV)
    with pytest.raises(hattn.HattnError):  # W + T - 1 = 257 tokens
        hattn.swa_keys_ring(kv, pos, r=64, W=256)


def _oracle_layer(kind, stack, l, inp, t):
    """fp64 oracle of layer l's output for the query at position t, fed the
    GPU's compressed caches (checked separately) and its top-k indices."""
    q = bits(inp["q"][l].cpu())
    pos = np.full((stack.B, 1), t, np.int32)
    st = stack.layers[l]
    raw = bits(inp["kv"][l][:, :t + 1].cpu())
    o_list, l_list = [], []
    if kind == CSA:
        sc = orc.indexer_scores(bits(inp["iq"][l].cpu()), inp["w"][l].cpu().numpy(),
                                bits(st["ik_c"].cpu()), pos, 4)
        idx = stack.idx.cpu().numpy()
        check_topk(idx, sc, pos, 4, stack.k, f"layer {l} top-k at {t}")
        o, ls = orc.attention(orc.KIND_SPARSE, q, bits(st["kv_c"].cpu()), pos, idx=idx, r=stack.r)
        o_list.append(o)
        l_list.append(ls)
    elif kind == HCA:
        o, ls = orc.attention(orc.KIND_HCA, q, bits(st["kv_h"].cpu()), pos, m=128, r=stack.r)
        o_list.append(o)
        l_list.append(ls)
    o, ls = orc.attention(orc.KIND_SWA, q, raw, pos, W=stack.W, r=stack.r)
    o_list.append(o)
    l_list.append(ls)
    return orc.merge(o_list, l_list, inp["sink"][l].cpu().numpy(), pos, stack.r)


def test_decode_loop_matches_oracle():
    """Four layers (SWA, SWA, CSA, HCA), batch 2, a 900-token prompt, then 260
    decode steps: CSA entries are appended every 4th token and HCA entries at
    tokens 1023 and 1151, all from 256-row rings.  Checked steps compare every
    layer's output with the oracle; at the end the entries appended during
    decode are compared with the oracle's compression of the full token
    streams."""
    kinds = [SWA, SWA, CSA, HCA]
    B, H, D, r, HI, dI, k = 2, 64, 512, 64, 64, 128, 64
    L0, steps = 900, 260
    L = L0 + steps
    stack = DecodeStack(kinds, B=B, H=H, D=D, r=r, HI=HI, dI=dI, k=k, L_max=1280, device=DEV)
    inp = {n: [] for n in ("kv", "ik", "gc", "gh", "q", "iq", "w", "sink")}
    for l in range(len(kinds)):
        s = 100 * (l + 1)
        inp["kv"].append(randn_bf16((B, L, D), s + 1).to(DEV))
        inp["ik"].append(randn_bf16((B, L, dI), s + 2).to(DEV))
        inp["gc"].append(randn_bf16((B, L), s + 3).to(DEV))
        inp["gh"].append(randn_bf16((B, L), s + 4).to(DEV))
        inp["q"].append(randn_bf16((B, 1, H, D), s + 5).to(DEV))
        inp["iq"].append(randn_bf16((B, 1, HI, dI), s + 6).to(DEV))
        g = torch.Generator().manual_seed(s + 7)
        inp["w"].append(torch.randn((B, 1, HI), generator=g).to(DEV))
        inp["sink"].append(torch.randn((H,), generator=g).to(DEV))
        gate = inp["gc"][l] if kinds[l] == CSA else inp["gh"][l]
        stack.prefill(l, inp["kv"][l][:, :L0].contiguous(), inp["ik"][l][:, :L0].contiguous(),
                      gate[:, :L0].contiguous())
    checks = sorted({L0, L0 + 3, 1023, 1024, 1151, L - 1} | set(range(L0, L, 29)))
    for t in range(L0, L):
        for l in range(len(kinds)):
            gate = inp["gc"][l] if kinds[l] == CSA else inp["gh"][l]
            stack.append(l, t, inp["kv"][l][:, t], inp["ik"][l][:, t], gate[:, t])
        pos = torch.full((B, 1), t, dtype=torch.int32, device=DEV)
        stack.step(t, inp["q"], inp["iq"], inp["w"], inp["sink"], pos)
        if t in checks:
            torch.cuda.synchronize()
            hattn.check_status()
            for l, kind in enumerate(kinds):
                ref_o, ref_l = _oracle_layer(kind, stack, l, inp, t)
                check_attn(stack.out[l], stack.lse[l], ref_o, ref_l, f"layer {l} ({kind}) at {t}")
    torch.cuda.synchronize()
    hattn.check_status()
    # entries appended during decode, against the oracle's compression
    l_c, l_h = kinds.index(CSA), kinds.index(HCA)
    for j in [L0 // 4, L0 // 4 + 1, 255, 256, L // 4 - 1]:
        for b in range(B):
            rk, ri, _ = orc.compress(bits(inp["kv"][l_c][b:b + 1].cpu()),
                                     bits(inp["gc"][l_c][b:b + 1].cpu()), 4, 8, r, j, j + 1,
                                     ik_raw=bits(inp["ik"][l_c][b:b + 1].cpu()))
            assert rel_l2(stack.layers[l_c]["kv_c"][b, j], rk[0, 0]) <= KV_REL_L2
            assert rel_l2(stack.layers[l_c]["ik_c"][b, j], ri[0, 0]) <= KV_REL_L2
    for j in [7, 8]:  # completed at tokens 1023 and 1151
        for b in range(B):
            rk, _, _ = orc.compress(bits(inp["kv"][l_h][b:b + 1].cpu()),
                                    bits(inp["gh"][l_h][b:b + 1].cpu()), 128, 128, r, j, j + 1)
            assert rel_l2(stack.layers[l_h]["kv_h"][b, j], rk[0, 0]) <= KV_REL_L2
