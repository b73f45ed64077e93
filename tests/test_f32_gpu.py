"""GPU parity of attn_fwd_f32, the three fp32 comparison kernels of
"masked multi head attention in CUDA" section 6.1 (naive three-pass, tiled
per-element online softmax, tiled block rowmax), against the float64 oracle
on the same fp32 inputs.  fp32 arithmetic with expf: the bound used here is
|o - o_ref| <= 1e-5 + 1e-4 |o_ref| and |lse - lse_ref| <= 1e-5 (fp32 carries
24 bits; a row of up to a few hundred terms loses a few of them)."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_attn_gb300 as attn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    attn.status()


@pytest.mark.parametrize("kernel", ["naive", "tiled_element", "tiled_rowmax"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L, vl", [(200, [200, 0]), (129, [77, 129]), (64, None)])
def test_f32_kernels_match_oracle(kernel, D, causal, L, vl):
    gen = torch.Generator().manual_seed(L + D)
    B, H = 2, 3
    q = torch.randn(B, H, L, D, generator=gen) * 2.0
    k = torch.randn(B, H, L, D, generator=gen)
    v = torch.randn(B, H, L, D, generator=gen)
    dev = torch.device("cuda")
    sm = 1.0 / math.sqrt(D)
    vl_t = None if vl is None else torch.tensor(vl, dtype=torch.int32)
    o, lse = attn.attn_fwd_f32(q.to(dev), k.to(dev), v.to(dev), kernel=kernel, causal=causal,
                               sm_scale=sm, valid_len=None if vl_t is None else vl_t.to(dev))
    assert attn.status() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = oracle.attn_fwd_f64(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                         sm, causal=causal,
                                         valid_len=None if vl is None else np.array(vl, np.int32))
    o = o.cpu().double().numpy()
    lse = lse.cpu().numpy().reshape(lse_ref.shape)
    assert np.all(np.abs(o - o_ref) <= 1e-5 + 1e-4 * np.abs(o_ref)), np.abs(o - o_ref).max()
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - lse_ref[~neg]) <= 1e-5)
