"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerance, per element (both kernels, every case):
    |o - o_ref| <= 2e-3 + 1e-2 * |o_ref|     on O,
    |lse - lse_ref| <= 1e-4                  on LSE (and -inf exactly where the oracle has -inf).
Small shapes are compared in full (several 128-row tiles, ragged tails,
every mask), and so are the five benchmark workloads: every row of every head
of C1-C5 against the oracle run over the whole workload, with the maximum
absolute and relative errors and the worst error-to-bound ratio reported.
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
    attn.status()  # clear any stale device word


def run_gpu(q, k, v, causal, vl, sm_scale, simt=False):
    dev = torch.device("cuda")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, sm_scale=sm_scale,
                           valid_len=None if vl is None else vl.to(dev), simt=simt)
    st, code = attn.status()
    assert st == attn.ATTN_OK, "device status %d (code %#x)" % (st, code)
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(o, lse, o_ref, lse_ref, what=""):
    o = o.reshape(o_ref.shape)
    lse = lse.reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)), "non-finite O " + what
    err = np.abs(o - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    bad = err > bound
    assert not bad.any(), "%s: %d O elements out of tolerance, worst %g at %s (ref %g)" % (
        what, int(bad.sum()), float(err.max()), np.unravel_index(np.argmax(err - bound), err.shape),
        float(o_ref.reshape(-1)[np.argmax((err - bound).reshape(-1))]))
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg), "LSE -inf pattern differs " + what
    lerr = np.abs(lse[~neg] - lse_ref[~neg])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, "%s: LSE err %g" % (what, lerr.max())


def full_case(B, Hq, Hkv, L, D, dtype, causal, seed, padded=False, valid_len=None, q_scale=1.0,
              sm_scale=None, simt=False):
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed, q_scale=q_scale,
                                 valid_len=valid_len, padded=padded)
    sm = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    o, lse = run_gpu(q, k, v, causal, vl, sm, simt=simt)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype),
                                          sm, causal=causal,
                                          valid_len=None if vl is None else vl.numpy())
    check(o, lse, o_ref, lse_ref, "B%d Hq%d Hkv%d L%d D%d %s causal=%s vl=%s simt=%s" % (
        B, Hq, Hkv, L, D, dtype, causal, None if vl is None else vl.tolist(), simt))


KERNELS = [pytest.param(False, id="tc"), pytest.param(True, id="simt")]


@pytest.mark.parametrize("simt", KERNELS)
@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [wl.F16, wl.BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_small_shapes_full_compare(simt, D, dtype, causal):
    # 700 rows: two full 256-row units and a ragged one whose second tile is partly past L
    full_case(2, 4, 2, 700, D, dtype, causal, seed=100 + D, simt=simt)


@pytest.mark.parametrize("D, dtype", [(128, wl.BF16), (64, wl.F16)])
@pytest.mark.parametrize("causal", [False, True])
def test_long_ragged_sequences(D, dtype, causal):
    # 3001 rows and keys: 24 key tiles, the last one key long; MQA, padding
    # that ends inside the second half of a key tile in one batch and on a
    # half-tile boundary in the other (every row compared)
    full_case(2, 4, 1, 3001, D, dtype, causal, seed=3001 + D, valid_len=[2900, 2880])


@pytest.mark.parametrize("simt", KERNELS)
@pytest.mark.parametrize("L", [1, 2, 64, 127, 128, 129, 255, 256, 257, 383, 513])
def test_sequence_lengths(simt, L):
    full_case(1, 2, 1, L, 128, wl.BF16, causal=True, seed=L, simt=simt)
    full_case(1, 2, 2, L, 64, wl.F16, causal=False, seed=L + 1, simt=simt)


@pytest.mark.parametrize("simt", KERNELS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_padding_masks(simt, causal, D):
    # 0 (fully masked rows), 1, tile edges, L
    full_case(6, 2, 2, 300, D, wl.BF16, causal, seed=7, valid_len=[0, 1, 127, 128, 129, 300],
              simt=simt)
    full_case(3, 4, 1, 520, D, wl.F16, causal, seed=8, valid_len=[520, 257, 255], simt=simt)


@pytest.mark.parametrize("simt", KERNELS)
@pytest.mark.parametrize("Hq, Hkv", [(8, 8), (8, 4), (8, 2), (8, 1)])
def test_head_grouping(simt, Hq, Hkv):
    full_case(2, Hq, Hkv, 260, 128, wl.BF16, True, seed=Hq * 10 + Hkv, simt=simt)
    full_case(2, Hq, Hkv, 260, 64, wl.F16, False, seed=Hq * 10 + Hkv + 1, simt=simt)


@pytest.mark.parametrize("simt", KERNELS)
def test_large_scores_and_rescaling(simt):
    # Q x 8: score ranges of tens of units force many running-max updates
    full_case(2, 2, 1, 1000, 128, wl.BF16, True, seed=11, q_scale=8.0, simt=simt)
    full_case(2, 2, 2, 1000, 64, wl.F16, False, seed=12, q_scale=4.0, simt=simt)


@pytest.mark.parametrize("simt", KERNELS)
def test_zero_scale_is_uniform_average(simt):
    full_case(2, 2, 2, 300, 64, wl.BF16, True, seed=13, sm_scale=0.0, valid_len=[300, 77],
              simt=simt)


def test_valid_len_out_of_range_is_clamped_and_reported():
    q, k, v, _ = wl.make_inputs(3, 2, 2, 200, 64, wl.BF16, seed=14)
    vl = torch.tensor([-5, 1000, 50], dtype=torch.int32)
    dev = torch.device("cuda")
    o, lse = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=False,
                           valid_len=vl.to(dev))
    st, code = attn.status()
    assert st == 11 and (code & 2), (st, code)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, 0.125,
                                          causal=False, valid_len=[0, 200, 50])
    check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "clamped")
    assert attn.status() == (0, 0)  # the word was cleared


def test_no_lse_output_and_mqa_3d_layout():
    q, k, v, _ = wl.make_inputs(2, 4, 1, 300, 128, wl.BF16, seed=15)
    dev = torch.device("cuda")
    o1, _ = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=True, return_lse=False)
    o2, _ = attn.attn_fwd(q.to(dev), k[:, 0].to(dev), v[:, 0].to(dev), causal=True)
    assert attn.status()[0] == 0
    assert torch.equal(o1, o2)


def test_deterministic():
    q, k, v, vl = wl.make_inputs(2, 8, 2, 1500, 128, wl.BF16, seed=16, padded=True)
    dev = torch.device("cuda")
    args = (q.to(dev), k.to(dev), v.to(dev))
    o1, l1 = attn.attn_fwd(*args, causal=True, valid_len=vl.to(dev))
    o2, l2 = attn.attn_fwd(*args, causal=True, valid_len=vl.to(dev))
    assert attn.status()[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ the five workloads

def error_summary(o, lse, o_ref, lse_ref):
    """Margins of a full comparison: max |o - o_ref|, max |o - o_ref| / |o_ref|
    over |o_ref| >= 1e-3, the worst ratio of error to the O bound, the number of
    O elements over the bound, and the max LSE error over finite rows."""
    o = o.reshape(o_ref.shape)
    err = np.abs(o - o_ref)
    aref = np.abs(o_ref)
    big = aref >= 1e-3
    neg = np.isneginf(lse_ref)
    lerr = np.abs(lse.reshape(lse_ref.shape)[~neg] - lse_ref[~neg])
    return {
        "max_abs_err_O": float(err.max()),
        "max_rel_err_O": float((err[big] / aref[big]).max()) if big.any() else 0.0,
        "worst_err_over_bound_O": float((err / (O_ATOL + O_RTOL * aref)).max()),
        "n_over_bound_O": int((err > O_ATOL + O_RTOL * aref).sum()),
        "max_err_LSE": float(lerr.max()) if lerr.size else 0.0,
    }


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5"])
def test_workload(name):
    """Every output element of the workload against the oracle run over all of it."""
    w = wl.WORKLOADS[name]
    q, k, v, vl = wl.workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.causal, vl, w.sm_scale)
    # properties at full size
    assert np.all(np.isfinite(o))
    if vl is not None:
        for b, x in enumerate(vl.tolist()):
            if x == 0:
                assert np.all(o.reshape(w.B, w.Hq, w.L, w.D)[b] == 0.0)
                assert np.all(np.isneginf(lse.reshape(w.B, w.Hq, w.L)[b]))
    assert np.isfinite(lse).sum() > 0
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v),
                                          wl.dtype_code(w.dtype), w.sm_scale, causal=w.causal,
                                          valid_len=None if vl is None else vl.numpy())
    summary = error_summary(o, lse, o_ref, lse_ref)
    print("%s parity: %s" % (name, summary))
    check(o, lse, o_ref, lse_ref, "%s %s" % (name, summary))


@pytest.mark.parametrize("name", ["C3", "C4", "C5"])
def test_workload_tc_matches_simt_everywhere(name):
    """Both CUDA kernels agree on every output element of the full workload
    (twice the oracle tolerance: each is within it of the oracle)."""
    w = wl.WORKLOADS[name]
    q, k, v, vl = wl.workload_inputs(w)
    o1, l1 = run_gpu(q, k, v, w.causal, vl, w.sm_scale)
    o2, l2 = run_gpu(q, k, v, w.causal, vl, w.sm_scale, simt=True)
    err = np.abs(o1 - o2)
    assert np.all(err <= 2 * (O_ATOL + O_RTOL * np.abs(o2)))
    neg = np.isneginf(l2)
    assert np.array_equal(np.isneginf(l1), neg)
    assert np.abs(l1[~neg] - l2[~neg]).max() <= 2 * LSE_ATOL


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_v_tiles_beyond_fp16_range(D, causal):
    """bf16 V tiles holding |v| >= 65536 keep bf16 (split P) while the other
    tiles of the same launch run P.V in fp16; both must match the oracle."""
    B, Hq, Hkv, L = 2, 4, 2, 640
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=31 + D)
    v = v.clone()
    v[0, 0, 130, 5] = 70000.0       # key tile 1 of kv head 0, batch 0
    v[1, 1, 600, :3] = -3.0e6       # key tile 4 of kv head 1, batch 1
    v[1, 0, 0, 7] = 65504.0         # still in fp16 range: this tile converts
    sm = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, None, sm)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, sm, causal=causal)
    check(o, lse, o_ref, lse_ref, "bf16 V beyond fp16 range D%d causal=%s" % (D, causal))


@pytest.mark.parametrize("L, D, dtype, causal, valid_len", [
    (128, 128, wl.BF16, True, None),
    (200, 64, wl.F16, False, [200, 0, 77, 129, 200, 1, 150, 199]),
    (300, 128, wl.BF16, True, [300, 257, 0, 128, 300, 5, 299, 255]),
    (260, 64, wl.BF16, True, None),
])
def test_many_short_units_per_cta(L, D, dtype, causal, valid_len):
    """Several units per CTA with one to three key tiles each: the unit
    boundary (O staged in the last V stage, its deferred release, the next
    unit decoded ahead, fewer score tiles than score buffers) many times per
    CTA, with empty and ragged units mixed in."""
    B, Hq, Hkv = 8, 40, 8
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=L + D + 7, valid_len=valid_len)
    sm = 1.0 / math.sqrt(D)
    o, lse = run_gpu(q, k, v, causal, vl, sm)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype), sm,
                                          causal=causal, valid_len=None if vl is None else vl.numpy())
    check(o, lse, o_ref, lse_ref, "many short units L%d D%d causal=%s" % (L, D, causal))
    # the same call again gives the same bits (the staging stages rotate)
    o2, lse2 = run_gpu(q, k, v, causal, vl, sm)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
