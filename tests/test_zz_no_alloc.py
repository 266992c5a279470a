"""hattn_indexer_topk_noalloc: the indexer top-k for callers that cannot
allocate device memory (an engine with its own fixed pool, a plugin host that
forbids device allocations).  Its score and selection scratch is an array
compiled into the library, so the call must give the same selection as
hattn_indexer_topk with a caller-provided workspace, call after call, and
refuse requests larger than that array.

This file is collected last, so a run that stops at the first failure has
already run every other test; it passes alone and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_attention_26_b300 import hattn

SCRATCH_SCORES = 1 << 22  # the fixed scratch size stated in include/hattn.h


@pytest.fixture(scope="module")
def L():
    from sparse_attention_26_b300 import build
    build.build()
    return hattn.lib()


def test_noalloc_rejects_requests_beyond_its_scratch(L):
    """B * T * N_cap above the fixed scratch is an argument error, raised on
    the host before any device work (no GPU needed)."""
    fake = ctypes.c_void_p(0x10000)
    N_cap = SCRATCH_SCORES // 8 + 1
    rc = L.hattn_indexer_topk_noalloc(fake, fake, fake, fake, 8, 1, 64, 128, N_cap, 1024, 4,
                                      fake, None)
    assert rc == hattn.INVALID_ARG
    assert "scratch" in L.hattn_last_error().decode()


def _inputs(B, T, HI, dI, N_cap, seed):
    g = torch.Generator().manual_seed(seed)
    iq = torch.randn((B, T, HI, dI), generator=g).to(torch.bfloat16).cuda()
    w = torch.randn((B, T, HI), generator=g).float().cuda()
    ik = torch.randn((B, N_cap, dI), generator=g).to(torch.bfloat16).cuda()
    pos = torch.randint(4 * N_cap // 2, 4 * N_cap, (B, T), generator=g, dtype=torch.int32).cuda()
    return iq, w, ik, pos


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice(L):
    """Two calls in a row (different shapes, so the second runs over what the
    first left in the shared scratch) select exactly what the workspace call
    selects."""
    for B, T, HI, dI, N_cap, k, seed in [(8, 1, 64, 128, 262144, 1024, 1),
                                         (3, 4, 64, 128, 50000, 512, 2)]:
        iq, w, ik, pos = _inputs(B, T, HI, dI, N_cap, seed)
        got = hattn.indexer_topk_noalloc(iq, w, ik, pos, k=k)
        ref = hattn.indexer_topk(iq, w, ik, pos, k=k)
        hattn.check_status()
        got = np.sort(got.cpu().numpy(), axis=-1)
        ref = np.sort(ref.cpu().numpy(), axis=-1)
        np.testing.assert_array_equal(got, ref)
        assert (got >= 0).all()


@pytest.mark.gpu
def test_noalloc_back_to_back_and_on_every_device(L):
    """Calls queued back to back on one stream, with no synchronisation in
    between, each see only their own scores: the second call's scores land
    in the shared scratch after the first call's selection has read it
    (stream order).  Where more than one GPU is visible, the same holds with
    each device current (each device has its own copy of the scratch)."""
    for dev in range(torch.cuda.device_count()):
        with torch.cuda.device(dev):
            runs = [_inputs(8, 1, 64, 128, 65536, 10 + i) for i in range(2)]
            runs = [tuple(t.to(f"cuda:{dev}") for t in r) for r in runs]
            got = [hattn.indexer_topk_noalloc(*r, k=1024) for r in runs]
            ref = [hattn.indexer_topk(*r, k=1024) for r in runs]
            hattn.check_status()
            for g_, r_ in zip(got, ref):
                np.testing.assert_array_equal(np.sort(g_.cpu().numpy(), axis=-1),
                                              np.sort(r_.cpu().numpy(), axis=-1))
