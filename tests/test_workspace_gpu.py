"""bf16 calls of attn_fwd take a stream-ordered workspace (the fp16 copy of V
and its per-tile flags) from a pool the library owns.  These tests check that
the pool is reused, that concurrent calls on different streams do not share a
workspace, that attn_shutdown leaves the library usable, and the range check
on a ragged last key tile."""
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
    attn.attn_fwd(q, k, v, causal=True)  # first call of this size may grow the pool
    torch.cuda.synchronize()
    free = []
    for _ in range(4):
        attn.attn_fwd(q, k, v, causal=True)
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
        o, lse = attn.attn_fwd(q, k, v, causal=True)
        torch.cuda.synchronize()
        alone.append((o.clone(), lse.clone()))
    # both problems at once, several times, on two streams with no ordering
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for rep in range(3):
        for (q, k, v), st in zip(cases, streams):
            with torch.cuda.stream(st):
                outs.append(attn.attn_fwd(q, k, v, causal=True, stream=st))
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
