"""attn_fwd_noalloc: the entry point for callers that must not allocate device
memory (servers that reserve all device memory at start-up, latency-bound
loops, runtimes that account only for their own allocator).

It must give the same results as attn_fwd and as the float64 oracle (within
the parity tolerance used everywhere in these tests), on two calls in a row
that share its static scratch array, must not change the device's free
memory, and must report device-side conditions through attn_status, keeping
them until attn_status reads them.  This file is collected last on purpose; it
passes alone in a fresh process and after the other tests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 2e-3, 1e-2, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    attn.status()


def _call(entry, q, k, v, o, lse, causal, vl, sm):
    B, Hq, L, D = q.shape
    return attn.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        B, Hq, k.shape[1], L, D, sm, int(causal),
                        None if vl is None else vl.data_ptr(),
                        attn.ATTN_BF16 if q.dtype == torch.bfloat16 else attn.ATTN_F16,
                        torch.cuda.current_stream().cuda_stream or None, entry=entry)


def _close_np(o, lse, o_ref, lse_ref):
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - lse_ref[~neg]) <= LSE_ATOL)


def _close(o, lse, o_ref, lse_ref):
    o, o_ref = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
    assert np.all(np.abs(o - o_ref) <= O_ATOL + O_RTOL * np.abs(o_ref))
    lse, lse_ref = lse.cpu().numpy(), lse_ref.cpu().numpy()
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg)
    assert np.all(np.abs(lse[~neg] - lse_ref[~neg]) <= LSE_ATOL)


@pytest.mark.parametrize("B, Hq, Hkv, L, D, dtype, causal, valid_len", [
    (2, 4, 2, 700, 128, wl.BF16, True, [700, 333]),
    (2, 2, 2, 300, 64, wl.F16, False, [0, 300]),
    (1, 4, 1, 333, 32, wl.BF16, True, [333]),
    (2, 2, 1, 140, 16, wl.F16, False, [140, 3]),
])
def test_noalloc_matches_attn_fwd_twice(B, Hq, Hkv, L, D, dtype, causal, valid_len):
    dev = torch.device("cuda")
    q, k, v, vl = (t.to(dev) for t in wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=L + D,
                                                     valid_len=valid_len))
    sm = 1.0 / math.sqrt(D)
    o_ref, lse_ref = torch.empty_like(q), torch.empty(B * Hq, L, device=dev)
    outs = [(torch.empty_like(q), torch.empty(B * Hq, L, device=dev)) for _ in range(2)]
    assert _call(None, q, k, v, o_ref, lse_ref, causal, vl, sm) == attn.ATTN_OK
    assert attn.status() == (attn.ATTN_OK, 0)

    # two calls in a row on the shared scratch array.  The first call on a
    # device may make the driver load the library's static device data (the
    # scratch array itself); no later call may change the device's free memory.
    free = []
    for o, lse in outs:
        assert _call("attn_fwd_noalloc", q, k, v, o, lse, causal, vl, sm) == attn.ATTN_OK
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    assert attn.status() == (attn.ATTN_OK, 0)
    assert free[1] == free[0], "device free memory changed across attn_fwd_noalloc"
    for o, lse in outs:
        _close(o, lse, o_ref, lse_ref)
    # and against the oracle itself (two results each within the bound of
    # the oracle may be twice the bound apart from each other)
    o64, lse64 = oracle.attn_fwd_bits(wl.bits(q.cpu()), wl.bits(k.cpu()), wl.bits(v.cpu()),
                                      wl.dtype_code(dtype), sm, causal=causal,
                                      valid_len=None if vl is None else vl.cpu().numpy())
    for o, lse in outs:
        _close_np(o.float().cpu().numpy().reshape(o64.shape), lse.cpu().numpy(), o64, lse64)


def test_noalloc_reports_device_status_and_clears_it():
    dev = torch.device("cuda")
    q, k, v, _ = (t.to(dev) if t is not None else None
                  for t in wl.make_inputs(2, 2, 1, 200, 128, wl.BF16, seed=3))
    vl_bad = torch.tensor([-4, 500], dtype=torch.int32, device=dev)
    vl_ok = torch.tensor([0, 200], dtype=torch.int32, device=dev)
    o1, l1 = torch.empty_like(q), torch.empty(4, 200, device=dev)
    o2, l2 = torch.empty_like(q), torch.empty(4, 200, device=dev)
    assert _call("attn_fwd_noalloc", q, k, v, o1, l1, True, vl_bad, 0.09) == attn.ATTN_OK
    st, code = attn.status()
    assert st == 11 and (code & 2)          # ATTN_ERR_VALID_LEN from the static word
    assert attn.status() == (attn.ATTN_OK, 0)  # read-and-clear
    # a condition stays in the word until attn_status reads it, even when a
    # later call on the same stream has none
    assert _call("attn_fwd_noalloc", q, k, v, o1, l1, True, vl_bad, 0.09) == attn.ATTN_OK
    assert _call("attn_fwd_noalloc", q, k, v, o1, l1, True, vl_ok, 0.09) == attn.ATTN_OK
    st, code = attn.status()
    assert st == 11 and (code & 2)
    assert attn.status() == (attn.ATTN_OK, 0)
    # the clamped call equals an in-range call with the clamped lengths
    assert _call(None, q, k, v, o2, l2, True, vl_ok, 0.09) == attn.ATTN_OK
    assert attn.status() == (attn.ATTN_OK, 0)
    _close(o1, l1, o2, l2)


def test_noalloc_rejects_bad_arguments_before_queueing():
    st = attn.fwd_raw(0x10000, 0x10000, 0x10000, 0x10000, None, 1, 3, 2, 16, 128, 0.1, 0, None,
                      attn.ATTN_BF16, None, entry="attn_fwd_noalloc")
    assert attn.binding.STATUS_NAMES[st] == "ATTN_ERR_HEADS"
