"""The parity checker of the GPU tests, checked on the CPU: it accepts the oracle's
own result rounded to the 16-bit storage type (the size of error the arithmetic
makes) and rejects the mistakes a wrong kernel would make in a single row -- a
sign flip, a row scaled by 10 %, a row taken from the neighbouring token, one
element off -- even when the whole-tensor norms would hide them."""

import numpy as np
import pytest
import torch

import oracle
from gpu_common import assert_close, rel_cos, row_elem_check


def _case(seed=5, L=(300, 180, 77), hq=4, hkv=2, d=64):
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(L)])
    T = int(cu[-1])
    q = rng.standard_normal((T, hq, d))
    k = rng.standard_normal((T, hkv, d))
    v = rng.standard_normal((T, hkv, d))
    do = rng.standard_normal((T, hq, d))
    return oracle.attn_fwd_bwd_thd(q, k, v, do, cu, cu, cu, cu, d ** -0.5,
                                   oracle.MASK_PADDING_CAUSAL)


def _bf16(x):
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_rounded_result_passes(idx):
    ref = _case()[idx]
    assert_close("rounded", _bf16(ref), ref)
    m = row_elem_check(_bf16(ref), ref)
    assert m["row_ratio"] < 0.25 and m["elem_ratio"] < 0.5, m


@pytest.mark.parametrize("idx", [2, 3, 4])
@pytest.mark.parametrize("mistake", ["sign", "scale", "shift", "element"])
def test_single_row_mistakes_fail(idx, mistake):
    ref = _case()[idx]
    got = _bf16(ref).copy()
    flat = got.reshape(-1, got.shape[-1])
    rn = np.linalg.norm(ref.reshape(-1, ref.shape[-1]), axis=1)
    r = int(np.argsort(rn)[len(rn) // 2 + 7])  # a row of median size
    if mistake == "sign":
        flat[r] = -flat[r]
    elif mistake == "scale":
        flat[r] = 1.1 * flat[r]
    elif mistake == "shift":
        flat[r] = flat[r + 1]
    else:
        flat[r, 3] += 0.5 * np.abs(flat[r]).max() + 0.2 * rn.mean() / np.sqrt(flat.shape[1])
    if mistake == "scale":
        # the whole-tensor check alone would not see this one
        rel, cos = rel_cos(got, ref)
        assert rel <= 1e-2 and cos >= 0.9999
    with pytest.raises(AssertionError):
        assert_close(mistake, got, ref)
