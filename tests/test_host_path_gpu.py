"""attn_fwd_host: host buffers in, host buffers out, copies pipelined with the
kernels chunk by chunk.  Each chunk runs exactly attn_fwd's kernels on a
contiguous slice, so the results must equal attn_fwd's bit for bit; one small
case is also checked against the oracle directly."""
import math

import numpy as np
import pytest
import torch

import attention_forward_attn_gb300 as attn
import oracle
from attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    oracle.build()


def _device_result(q, k, v, causal, vl):
    dev = torch.device("cuda")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal,
                           valid_len=None if vl is None else vl.to(dev))
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("B, Hq, Hkv, L, D, dtype, causal, padded", [
    (2, 16, 4, 2048, 128, wl.BF16, True, True),     # 4 chunks, ragged per batch (3 + 1 heads)
    (3, 8, 8, 1000, 64, wl.F16, False, False),      # ragged key tile, whole-batch chunks
    (5, 4, 1, 1536, 128, wl.BF16, False, True),     # MQA
    (1, 2, 2, 130, 64, wl.F16, True, False),        # one small chunk
    (4, 16, 4, 4096, 32, wl.BF16, True, True),      # D = 32 (runs the D = 64 kernel), 9 chunks
    (2, 8, 2, 1000, 16, wl.F16, False, False),      # D = 16, one chunk
])
def test_host_path_equals_device_path(B, Hq, Hkv, L, D, dtype, causal, padded):
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=200 + L)
    vl = None
    if padded:
        vl = torch.tensor([(L * (i + 1)) // (B + 1) for i in range(B)], dtype=torch.int32)
        vl[0] = 0  # a fully masked batch
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o, lse = attn.attn_fwd_host(qp, kp, vp, causal=causal,
                                valid_len=None if vl is None else vl.pin_memory())
    assert attn.status() == (attn.ATTN_OK, 0)
    o_ref, lse_ref = _device_result(q, k, v, causal, vl)
    assert torch.equal(o, o_ref)
    assert torch.equal(lse, lse_ref)
    assert len(attn.host_plan(B, Hq, Hkv, L, D)) >= 1


def test_host_path_pageable_memory_and_no_lse():
    """Pageable tensors (the driver stages the copies) and lse = NULL."""
    B, Hq, Hkv, L, D = 2, 16, 4, 2048, 128
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=211)
    assert not q.is_pinned()
    o = torch.empty_like(q)
    o2, lse = attn.attn_fwd_host(q, k, v, causal=True, out=o, return_lse=False)
    assert o2 is o and lse is None
    o_ref, _ = _device_result(q, k, v, True, None)
    assert torch.equal(o, o_ref)


def test_host_path_against_oracle():
    B, Hq, Hkv, L, D = 1, 4, 2, 300, 64
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=212)
    sm = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True,
                                sm_scale=sm)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, sm, causal=True)
    o = o.float().numpy().reshape(o_ref.shape)
    lse = lse.numpy().reshape(lse_ref.shape)
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    assert np.all(np.abs(lse - lse_ref) <= LSE_ATOL)


def test_host_path_orders_with_the_callers_stream():
    """Work queued on the caller's stream before the call (filling the input
    buffers) is seen by the copies, and the output is complete once the
    stream has synchronised, with calls queued back to back on a side stream."""
    B, Hq, Hkv, L, D = 2, 16, 4, 2048, 128
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=213)
    o_ref, lse_ref = _device_result(q, k, v, True, None)
    st = torch.cuda.Stream()
    qp = torch.zeros_like(q).pin_memory()
    kp, vp = k.pin_memory(), v.pin_memory()
    outs = []
    with torch.cuda.stream(st):
        q_dev = q.cuda()  # queued on st: device -> pinned host copy before the call
        qp.copy_(q_dev, non_blocking=True)
        for _ in range(3):
            outs.append(attn.attn_fwd_host(qp, kp, vp, causal=True, stream=st,
                                           synchronize=False))
    st.synchronize()
    assert attn.status(st) == (attn.ATTN_OK, 0)
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_host_path_reuses_pool_memory():
    B, Hq, Hkv, L, D = 2, 16, 4, 2048, 128
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=214)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    attn.attn_fwd_host(qp, kp, vp, causal=True)
    free = []
    for _ in range(3):
        attn.attn_fwd_host(qp, kp, vp, causal=True)
        free.append(torch.cuda.mem_get_info()[0])
    assert len(set(free)) == 1, free
