"""The parity check's tolerance rules on CPU: fp32 outputs face the layer
specification's max-abs 1e-2 directly; only a bf16-stored output gets the
half-ulp allowance that storing a correct fp32 value in bf16 costs."""
import numpy as np
import pytest
import torch

from _util import bf16_half_ulp, check_attn


def test_half_ulp_values():
    # 8 significant bits: a step of 2^-6 at [2, 4), 2^-7 at [1, 2)
    assert bf16_half_ulp(3.0) == 2.0 ** -7
    assert bf16_half_ulp(1.0) == 2.0 ** -8
    assert bf16_half_ulp(0.0) == 0.0


def test_fp32_output_gets_no_allowance():
    ref = np.full((4, 8), 3.0)
    got = torch.tensor(ref + 0.012, dtype=torch.float32)  # 0.012 > 1e-2, rel 4e-3
    with pytest.raises(AssertionError, match="max-abs"):
        check_attn(got, None, ref, None, "fp32 branch output")
    ok = torch.tensor(ref + 0.009, dtype=torch.float32)
    err, _ = check_attn(ok, None, ref, None, "fp32 branch output")
    assert err == pytest.approx(0.009, rel=1e-4)


def test_bf16_stored_output_gets_half_an_ulp():
    ref = np.full((4, 8), 3.0)
    got = ref + 0.012
    # the storage format decides: stated, or taken from a bf16 tensor
    err, _ = check_attn(torch.tensor(got, dtype=torch.float32), None, ref, None, "out",
                        stored_bf16=True)
    assert err == pytest.approx(0.012 - 2.0 ** -7, rel=1e-3)
    with pytest.raises(AssertionError):
        check_attn(torch.tensor(ref + 0.02, dtype=torch.float32), None, ref, None, "out",
                   stored_bf16=True)
    # a bf16 tensor takes the allowance by itself: 3 + 0.0117 rounds to the
    # next bf16 value, 3.015625, whose 0.0156 deviation is within 1e-2 plus
    # the half step (rel-L2 5.2e-3 would fail, so the reference sits between)
    ref2 = np.full((4, 8), 3.0078)
    b = torch.tensor(ref2 + 0.004, dtype=torch.bfloat16)
    assert float(b[0, 0]) == 3.015625
    check_attn(b, None, ref2, None, "bf16 out")
    with pytest.raises(AssertionError, match="max-abs"):
        check_attn(b.float(), None, ref2 - 0.0026, None, "fp32 copy of it", stored_bf16=False)
