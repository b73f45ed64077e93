"""Writes stay inside the caller's buffers: O and LSE are placed in larger
allocations whose guard words (before and after) hold a sentinel, for every
head dimension and entry point, with a fully masked batch first or last (the
rows of such a batch are written by a separate zero-fill path)."""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-4
GUARD = 4096          # guard elements on each side (8 KB of O, 16 KB of LSE)
SENTINEL16 = 0x7BCD   # an fp16/bf16 bit pattern no result here can have (a large finite value)
SENTINEL32 = -7.25e30


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    oracle.build()
    attn.status()


@pytest.mark.parametrize("entry", ["attn_fwd", "attn_fwd_simt", "attn_fwd_noalloc"])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("masked_batch", [0, 2])
@pytest.mark.parametrize("causal", [False, True])
def test_writes_stay_inside_o_and_lse(entry, D, masked_batch, causal):
    B, Hq, Hkv, L = 3, 4, 2, 300
    dtype = wl.BF16 if D in (32, 128) else wl.F16
    vl = [L, 131, L]
    vl[masked_batch] = 0
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=400 + D, valid_len=vl)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    vld = vl_t.to(dev)
    n_o, n_l = B * Hq * L * D, B * Hq * L
    o_buf = torch.full((n_o + 2 * GUARD,), SENTINEL16, dtype=torch.int16, device=dev)
    l_buf = torch.full((n_l + 2 * GUARD,), SENTINEL32, dtype=torch.float32, device=dev)
    sm = 1.0 / math.sqrt(D)
    st = attn.fwd_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o_buf.data_ptr() + 2 * GUARD,
                      l_buf.data_ptr() + 4 * GUARD, B, Hq, Hkv, L, D, sm, int(causal),
                      vld.data_ptr(), wl.dtype_code(dtype), None, entry=entry)
    assert st == attn.ATTN_OK
    assert attn.status() == (attn.ATTN_OK, 0)
    o_all = o_buf.cpu()
    l_all = l_buf.cpu()
    assert bool((o_all[:GUARD] == SENTINEL16).all()), "O written before its buffer"
    assert bool((o_all[GUARD + n_o:] == SENTINEL16).all()), "O written past its buffer"
    assert bool((l_all[:GUARD] == SENTINEL32).all()), "LSE written before its buffer"
    assert bool((l_all[GUARD + n_l:] == SENTINEL32).all()), "LSE written past its buffer"
    tdt = torch.bfloat16 if dtype == wl.BF16 else torch.float16
    o = o_all[GUARD:GUARD + n_o].view(tdt).float().numpy().reshape(B, Hq, L, D)
    lse = l_all[GUARD:GUARD + n_l].numpy().reshape(B * Hq, L)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v),
                                          wl.dtype_code(dtype), sm, causal=causal,
                                          valid_len=np.array(vl, dtype=np.int32))
    assert np.all(np.abs(o - o_ref.reshape(o.shape)) <= O_ATOL + O_RTOL * np.abs(o_ref.reshape(o.shape)))
    lse_ref = lse_ref.reshape(lse.shape)
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - lse_ref[~neg]) <= LSE_ATOL)
    assert np.all(o[masked_batch] == 0.0)
