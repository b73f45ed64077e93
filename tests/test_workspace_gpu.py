"""Workspaces.  bf16 forwards (the fp16 copy of V and its per-tile flags),
explicit masks (their packed bits) and the backward (row statistics) need
device workspace.  The *_ws entry points take it from the caller (the binding
allocates it with torch); the plain entry points take it from a
stream-ordered pool the library owns.  These tests check that *_ws calls take
nothing from the pool and leave the device's free memory unchanged while
matching the pool path bit for bit and the oracle, that undersized or
misaligned workspaces are refused, that the pool is reused, that concurrent
calls on different streams do not share a workspace, that attn_shutdown
leaves the library usable, and the range check on a ragged last key tile."""
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


def _inputs(B, Hq, Hkv, L, D, seed, dtype=wl.BF16):
    dev = torch.device("cuda")
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=seed)
    return q.to(dev), k.to(dev), v.to(dev)


def test_pool_is_reused_across_calls():
    q, k, v = _inputs(2, 8, 2, 1024, 128, seed=101)
    attn.attn_fwd(q, k, v, causal=True, workspace="pool")  # the first call may grow the pool
    torch.cuda.synchronize()
    free = []
    for _ in range(4):
        attn.attn_fwd(q, k, v, causal=True, workspace="pool")
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    assert attn.status() == (attn.ATTN_OK, 0)
    assert len(set(free)) == 1, "device free memory changed between bf16 calls: %s" % free


def test_concurrent_streams_do_not_share_a_workspace():
    shapes = [(2, 8, 2, 896, 128, 102), (1, 16, 4, 1280, 128, 103)]
    cases = [_inputs(*s) for s in shapes]
    # results of each problem alone
    alone = []
    for q, k, v in cases:
        o, lse = attn.attn_fwd(q, k, v, causal=True, workspace="pool")
        torch.cuda.synchronize()
        alone.append((o.clone(), lse.clone()))
    # both problems at once, several times, on two streams with no ordering
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for (q, k, v), st in zip(cases, streams):
            with torch.cuda.stream(st):
                outs.append(attn.attn_fwd(q, k, v, causal=True, stream=st, workspace="pool"))
    torch.cuda.synchronize()
    assert attn.status() == (attn.ATTN_OK, 0)
    for i, (o, lse) in enumerate(outs):
        o_ref, lse_ref = alone[i % 2]
        assert torch.equal(o, o_ref), "stream result %d differs from the single-stream result" % i
        assert torch.equal(lse, lse_ref)


def test_shutdown_then_call_again():
    q, k, v = _inputs(1, 4, 2, 512, 64, seed=104)
    o1, l1 = attn.attn_fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    o1, l1 = o1.clone(), l1.clone()
    attn.shutdown()  # frees the status words, destroys the workspace pools
    o2, l2 = attn.attn_fwd(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert attn.status() == (attn.ATTN_OK, 0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("D", [64, 128])
def test_out_of_range_value_in_ragged_last_tile(D):
    """L = 700: the last key tile holds 60 keys; a value beyond fp16's range
    there keeps that partial tile in bf16 (split P) while the full tiles
    before it are copied to fp16."""
    B, Hq, Hkv, L = 1, 4, 2, 700
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=105 + D)
    v = v.clone()
    v[0, 1, 690, 3] = -1.0e5
    dev = torch.device("cuda")
    sm = 1.0 / math.sqrt(D)
    for causal in (False, True):
        o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, sm_scale=sm)
        o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, sm, causal=causal)
        o = o.float().cpu().numpy().reshape(o_ref.shape)
        lse = lse.cpu().numpy().reshape(lse_ref.shape)
        assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
        assert np.all(np.abs(lse - lse_ref) <= LSE_ATOL)
    assert attn.status() == (attn.ATTN_OK, 0)


def _check_oracle(o, lse, q, k, v, causal, sm, valid_len=None, mask=None):
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q.cpu()), wl.bits(k.cpu()), wl.bits(v.cpu()),
                                          wl.dtype_code(wl.BF16 if q.dtype == torch.bfloat16
                                                        else wl.F16), sm, causal=causal,
                                          valid_len=valid_len, mask=mask)
    o = o.float().cpu().numpy().reshape(o_ref.shape)
    lse = lse.cpu().numpy().reshape(lse_ref.shape)
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - lse_ref[~neg]) <= LSE_ATOL)


def test_caller_workspaces_take_nothing_from_the_pool():
    """attn_fwd_ws, attn_fwd_masked_ws and attn_bwd_masked_ws with torch-allocated
    workspaces: the library's pool hands out nothing (high-water mark stays 0
    after a reset), the device's free memory does not move across repeated
    calls, and the results equal the pool path's bit for bit and match the
    oracle.  A pool call afterwards does register in the high-water mark."""
    dev = torch.device("cuda")
    B, Hq, Hkv, L, D = 2, 8, 2, 1152, 128      # a size no earlier test used
    q, k, v = _inputs(B, Hq, Hkv, L, D, seed=106)
    sm = 1.0 / math.sqrt(D)
    mask = torch.rand(L, L, generator=torch.Generator().manual_seed(7)) < 0.7
    mask_d = mask.to(dev)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(8)).to(q.dtype).to(dev)
    n_f = attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_BF16)
    n_m = attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_BF16, mask_batches=1)
    n_b = attn.bwd_workspace_size(B, Hq, Hkv, L, L, D)
    assert n_f >= B * Hkv * L * D * 2 and n_m > n_f and n_b > 0
    ws = torch.empty(max(n_f, n_m, n_b), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(B * Hq, L, device=dev)

    def calls():
        attn.attn_fwd(q, k, v, causal=True, sm_scale=sm, out=o, lse=lse, workspace=ws)
        o1, l1 = o.clone(), lse.clone()
        attn.attn_fwd_strided(q, k, v, causal=False, sm_scale=sm, mask=mask_d, out=o, lse=lse,
                              workspace=ws)
        o2, l2 = o.clone(), lse.clone()
        grads = attn.attn_bwd(q, k, v, o1, l1, do, causal=True, sm_scale=sm, workspace=ws)
        return o1, l1, o2, l2, grads

    calls()  # the first launch of each kernel may load its code onto the device
    torch.cuda.synchronize()
    attn.pool_stats(reset_high_water=True)
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        res = calls()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    _, high = attn.pool_stats()
    assert attn.status() == (attn.ATTN_OK, 0)
    assert high == 0, "a *_ws call took %d bytes from the library's pool" % high
    assert free1 == free0, "device free memory changed across *_ws calls"
    o1, l1, o2, l2, (dq, dk, dv) = res
    # the pool path gives the same bits
    p1, pl1 = attn.attn_fwd(q, k, v, causal=True, sm_scale=sm, workspace="pool")
    p2, pl2 = attn.attn_fwd_strided(q, k, v, causal=False, sm_scale=sm, mask=mask_d,
                                    workspace="pool")
    pg = attn.attn_bwd(q, k, v, p1, pl1, do, causal=True, sm_scale=sm, workspace="pool")
    torch.cuda.synchronize()
    assert torch.equal(o1, p1) and torch.equal(l1, pl1)
    assert torch.equal(o2, p2) and torch.equal(l2, pl2)
    for a, b in zip((dq, dk, dv), pg):
        assert torch.equal(a, b)
    _, high = attn.pool_stats()
    assert high > 0  # the pool path does use the pool
    _check_oracle(o1, l1, q, k, v, True, sm)
    _check_oracle(o2, l2, q, k, v, False, sm, mask=mask.numpy())


def test_bad_caller_workspaces_are_refused():
    dev = torch.device("cuda")
    q, k, v = _inputs(1, 4, 2, 640, 64, seed=107)
    n = attn.fwd_workspace_size(1, 4, 2, 640, 640, 64, attn.ATTN_BF16)
    ws = torch.empty(n + 512, dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    f = attn.load().attn_fwd_ws
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), None, 1, 4, 2, 640, 64, 0.125,
            0, None, attn.ATTN_BF16)
    name = lambda st: attn.binding.STATUS_NAMES[int(st)]
    assert name(f(*args, None, 0, None)) == "ATTN_ERR_WORKSPACE"
    assert name(f(*args, ws.data_ptr(), n - 1, None)) == "ATTN_ERR_WORKSPACE"
    assert name(f(*args, ws.data_ptr() + 16, n, None)) == "ATTN_ERR_WORKSPACE"
    assert name(f(*args, ws.data_ptr(), n, None)) == "ATTN_OK"
    # fp16 needs none: NULL is fine
    qh, kh, vh = (t.half() for t in (q, k, v))
    oh = torch.empty_like(qh)
    assert attn.fwd_workspace_size(1, 4, 2, 640, 640, 64, attn.ATTN_F16) == 0
    assert name(f(qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), oh.data_ptr(), None, 1, 4, 2, 640,
                  64, 0.125, 0, None, attn.ATTN_F16, None, 0, None)) == "ATTN_OK"
    assert attn.status() == (attn.ATTN_OK, 0)
