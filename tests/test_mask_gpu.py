"""GPU parity of attn_fwd_masked: the explicit boolean [B, Lq, Lk] mask
("masked multi head attention in CUDA", section 2.2), intersected with the
causal and padding masks.

* Small shapes compared in full with the float64 oracle (same tolerance as
  every parity test): random masks of several densities, tile-aligned block
  masks (whole 128x128 tiles with no kept position, which the kernel skips),
  fully masked rows and batches, one mask shared by every batch, Lq != Lk,
  every head dimension, both dtypes.
* Masks that restate the implicit ones (tril = causal, key < valid_len =
  padding, all ones = none) give results identical bit for bit to the
  implicit masks, also at full size (C3, C4).
* A full-size block-sparse mask on the C4 shapes, compared with the oracle on
  sampled rows (tile-boundary rows of every head group).
* At D = 128 (one accumulator shared by the two halves of each key tile):
  rows that keep one half of every tile only, with the running max growing
  through one half.
"""
import math
import zlib

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


def check(o, lse, o_ref, lse_ref, what=""):
    o = np.asarray(o, dtype=np.float64).reshape(o_ref.shape)
    lse = np.asarray(lse).reshape(lse_ref.shape)
    err = np.abs(o - o_ref)
    bad = err > O_ATOL + O_RTOL * np.abs(o_ref)
    assert not bad.any(), "%s: %d O elements out of tolerance (max err %g)" % (
        what, int(bad.sum()), float(err.max()))
    neg = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), neg), "LSE -inf pattern differs " + what
    lerr = np.abs(lse[~neg] - lse_ref[~neg])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, "%s: LSE err %g" % (what, lerr.max())


def run(q, k, v, causal, vl, sm, mask):
    dev = torch.device("cuda")
    o, lse = attn.attn_fwd_strided(q.to(dev), k.to(dev), v.to(dev), causal=causal, sm_scale=sm,
                                   valid_len=None if vl is None else vl.to(dev),
                                   mask=None if mask is None else torch.from_numpy(mask).to(dev))
    st, code = attn.status()
    assert st == attn.ATTN_OK, "device status %d (code %#x)" % (st, code)
    return o, lse


def make_mask(kind, B, Lq, Lk, rng):
    if kind.startswith("random"):
        dens = float(kind.split("_")[1])
        m = rng.random((B, Lq, Lk)) < dens
    elif kind == "blocks":  # whole 128x128 tiles kept or removed, plus a ragged edge
        tiles = rng.random((B, (Lq + 127) // 128, (Lk + 127) // 128)) < 0.5
        tiles[:, :, 0] = True
        m = np.repeat(np.repeat(tiles, 128, axis=1), 128, axis=2)[:, :Lq, :Lk].copy()
        m[:, :, Lk // 3: Lk // 3 + 5] = False
    elif kind == "empty_rows":  # random, with fully masked rows and one fully masked batch
        m = rng.random((B, Lq, Lk)) < 0.4
        m[0, 5:140, :] = False
        m[-1] = False
    elif kind == "shared":  # one [Lq, Lk] mask for every batch
        m = rng.random((1, Lq, Lk)) < 0.3
    else:
        raise ValueError(kind)
    return m.astype(np.uint8)


@pytest.mark.parametrize("kind", ["random_0.5", "random_0.05", "random_0.97", "blocks",
                                  "empty_rows", "shared"])
@pytest.mark.parametrize("D, dtype", [(128, wl.BF16), (64, wl.F16), (32, wl.BF16)])
@pytest.mark.parametrize("causal", [False, True])
def test_masks_full_compare(kind, D, dtype, causal):
    B, Hq, Hkv, Lq, Lk = 3, 4, 2, 300, 400
    rng = np.random.default_rng(zlib.crc32(("%s/%d/%d" % (kind, D, causal)).encode()) % 1000)
    vl = [400, 261, 77]
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, Lq, D, dtype, seed=700 + D, valid_len=vl, Lk=Lk)
    mk = make_mask(kind, B, Lq, Lk, rng)
    sm = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, causal, vl_t, sm, mk)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype),
                                          sm, causal=causal, valid_len=vl_t.numpy(), mask=mk)
    check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
          "%s D%d causal=%s" % (kind, D, causal))


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.mark.parametrize("dtype", [wl.BF16, wl.F16])
@pytest.mark.parametrize("causal", [False, True])
def test_half_tile_masks_and_one_sided_max_growth(dtype, causal):
    """D = 128, where the two softmax halves of a row (keys 0-63 and 64-127
    of every 128-key tile) share one accumulator and agree on the running max
    every step: rows that keep only the first half of every tile, only the
    second, or both, with the scores of the second halves growing along the
    keys (Q x 4, K rows of the second halves scaled by up to 3), so that the
    running max moves, by more than the lazy-rescale threshold, through one
    half only."""
    B, Hq, Hkv, L, D = 2, 2, 1, 520, 128
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=44 + causal, q_scale=4.0)
    j = torch.arange(L)
    ramp = torch.where(j % 128 >= 64, 1.0 + 2.0 * j.float() / L, torch.ones(L))
    k = (k.float() * ramp[None, None, :, None]).to(k.dtype)
    i = np.arange(L)[:, None]
    jj = np.arange(L)[None, :]
    first = (jj % 128) < 64
    mk = np.where(i % 3 == 0, first, np.where(i % 3 == 1, ~first, True))
    mk = np.ascontiguousarray(np.broadcast_to(mk, (B, L, L))).astype(np.uint8)
    sm = 1.0 / math.sqrt(D)
    o, lse = run(q, k, v, causal, None, sm, mk)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype),
                                          sm, causal=causal, mask=mk)
    check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
          "half-tile masks causal=%s" % causal)


@pytest.mark.parametrize("name", ["C2", "C3", "C4"])
def test_restated_masks_are_bit_identical(name):
    """tril = causal, key < valid_len = padding: the explicit mask gives the
    implicit mask's results bit for bit (same tiles skipped, same scores
    removed, same arithmetic)."""
    w = wl.WORKLOADS[name]
    q, k, v, vl = wl.workload_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    vld = None if vl is None else vl.to(dev)
    o_i, l_i = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, valid_len=vld)
    L = w.L
    keep = torch.ones(w.B, L, L, dtype=torch.bool, device=dev)
    if w.causal:
        keep &= torch.tril(torch.ones(L, L, dtype=torch.bool, device=dev))
    if vl is not None:
        keep &= (torch.arange(L, device=dev)[None, None, :] < vld[:, None, None])
    o_m, l_m = attn.attn_fwd_strided(qd, kd, vd, sm_scale=w.sm_scale, mask=keep)
    assert attn.status() == (attn.ATTN_OK, 0)
    assert _same(o_i, o_m), "%s: O differs between the implicit and the explicit mask" % name
    assert torch.equal(l_i, l_m), "%s: LSE differs" % name
    # an all-ones mask changes nothing either
    o_1, l_1 = attn.attn_fwd_strided(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale,
                                     valid_len=vld, mask=torch.ones(L, L, dtype=torch.bool,
                                                                     device=dev))
    assert attn.status() == (attn.ATTN_OK, 0)
    assert _same(o_i, o_1) and torch.equal(l_i, l_1)


def test_block_sparse_full_size_sampled_rows():
    """C4 shapes with a block-sparse mask (a local band of 512 keys plus the
    first 256 keys, the rest removed at tile granularity, and a random partial
    tile per row block), causal, compared with the oracle on sampled rows."""
    w = wl.WORKLOADS["C4"]
    q, k, v, _ = wl.workload_inputs(w)
    L = w.L
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    keep = (np.abs(i - j) < 512) | (j < 256)
    rng = np.random.default_rng(5)
    for mb in range(L // 128):
        t = rng.integers(0, L // 128)
        keep[mb * 128:(mb + 1) * 128, t * 128:(t + 1) * 128] |= rng.random((128, 128)) < 0.3
    mk = np.stack([keep, ~np.roll(keep, 1, axis=1) | (j == 0), keep, keep]).astype(np.uint8)
    o, lse = run(q, k, v, True, None, w.sm_scale, mk)
    rows_per_head = sorted({0, 1, 127, 128, 511, 512, 2047, 2048, 4095} |
                           set(rng.integers(0, L, 12).tolist()))
    heads = [0, 5, 31, 32 + 7, 64 + 12, 96 + 31]
    rows = np.array([h * L + r for h in heads for r in rows_per_head], dtype=np.int64)
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, w.sm_scale,
                                          causal=True, mask=mk, rows=rows)
    o_all = o.float().cpu().numpy().reshape(-1, w.D)
    check(o_all[rows], lse.cpu().numpy().reshape(-1)[rows], o_ref, lse_ref, "C4 block-sparse")


def test_mask_with_strided_operands_and_guards():
    """[B, L, H, D] operands, a mask with padded rows (row stride > Lk), O in
    a guarded buffer: results match the oracle and nothing outside O is
    written."""
    B, Hq, Hkv, Lq, Lk, D, dtype = 2, 4, 1, 200, 333, 128, wl.BF16
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, Lq, D, dtype, seed=91, Lk=Lk)
    rng = np.random.default_rng(91)
    mk = (rng.random((B, Lq, Lk)) < 0.5).astype(np.uint8)
    mk[1, :, :] = 0
    dev = torch.device("cuda")
    mbuf = torch.zeros(B, Lq, Lk + 29, dtype=torch.uint8, device=dev)
    mbuf[:, :, :Lk] = torch.from_numpy(mk).to(dev)
    guard = 2048
    n_o = B * Hq * Lq * D
    obuf = torch.full((n_o + 2 * guard,), 0x7BCD, dtype=torch.int16, device=dev)
    out = obuf[guard:guard + n_o].view(torch.bfloat16).view(B, Lq, Hq, D).transpose(1, 2)
    qd = q.transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    o, lse = attn.attn_fwd_strided(qd, k.to(dev), v.to(dev), sm_scale=0.09, out=out,
                                   mask=mbuf[:, :, :Lk])
    assert attn.status() == (attn.ATTN_OK, 0)
    allb = obuf.cpu()
    assert bool((allb[:guard] == 0x7BCD).all()) and bool((allb[guard + n_o:] == 0x7BCD).all())
    o_ref, lse_ref = oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), 1, 0.09, mask=mk)
    check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "strided + mask")
    assert np.all(o[1].float().cpu().numpy() == 0.0)
