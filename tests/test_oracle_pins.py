"""Pins for the float64 oracle: it is checked here against things other than itself.

* brute force at 50 significant digits (mpmath) on tiny inputs, with the full
  score matrix and an explicit mask, no max subtraction, GQA by repetition;
* PyTorch's CPU float64 ``scaled_dot_product_attention`` with an explicit
  boolean mask and ``repeat_interleave`` head expansion, and ``torch.logsumexp``
  for the log-sum-exp;
* the hand-derived examples in ``tests/golden/hand_examples.json``;
* invariants and closed forms the pages fix (L=1 gives O=V, causal row 0 gives
  V[0], identical V rows, fully masked rows give 0, scaling Q instead of the
  scores) plus closed forms of the definition (zero scale gives the mean of
  the visible V rows and LSE = ln|J|, shifting every K row, permuting keys,
  the GQA head map);
* the fp16/bf16 decoders against numpy / PyTorch on all 65536 bit patterns.

The last test compiles deliberately broken copies of the oracle (a dropped
scale, an off-by-one mask, a modulo head map, a transposed K, ...) and checks
that every one of them fails at least one of these pins.
"""
import json
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _fwd_default(*a, **kw):
    return oracle.attn_fwd_f64(*a, **kw)


# ---------------------------------------------------------------- references

def brute_force(q, k, v, sm_scale, causal, valid_len, mask=None):
    """Attention by its definition at 50 digits: explicit mask, no max shift."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = 50
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G = Hq // Hkv
    head_of = [g for g in range(Hkv) for _ in range(G)]  # repetition, as repeat_interleave
    O = np.zeros((B, Hq, Lq, D))
    LSE = np.zeros((B * Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            g = head_of[h]
            for i in range(Lq):
                keep = [(not causal or i >= j) and (valid_len is None or j < valid_len[b])
                        and (mask is None or mask[b if mask.shape[0] > 1 else 0][i][j] != 0)
                        for j in range(Lk)]
                if not any(keep):
                    LSE[b * Hq + h, i] = -math.inf
                    continue
                w = {}
                for j in range(Lk):
                    if keep[j]:
                        s = mp.mpf(sm_scale) * mp.fsum(mp.mpf(q[b, h, i, d]) * mp.mpf(k[b, g, j, d])
                                                       for d in range(D))
                        w[j] = mp.exp(s)
                Z = mp.fsum(w.values())
                for d in range(D):
                    O[b, h, i, d] = float(mp.fsum(w[j] * mp.mpf(v[b, g, j, d]) for j in w) / Z)
                LSE[b * Hq + h, i] = float(mp.log(Z))
    return O, LSE


def explicit_mask(B, Lq, Lk, causal, valid_len, mask=None):
    m = torch.ones(B, 1, Lq, Lk, dtype=torch.bool)
    if mask is not None:
        m &= torch.from_numpy(np.asarray(mask) != 0).reshape(-1, 1, Lq, Lk)
    if causal:
        # torch.tril keeps column j <= row i of the [Lq, Lk] matrix: top-left
        m &= torch.tril(torch.ones(Lq, Lk, dtype=torch.bool))
    if valid_len is not None:
        keys = torch.arange(Lk)
        for b in range(B):
            m[b, :, :, :] &= (keys < int(valid_len[b]))[None, :]
    return m


def torch_reference(q, k, v, sm_scale, causal, valid_len, mask=None):
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    B, Hq, Lq, D = qt.shape
    Lk = kt.shape[2]
    G = Hq // kt.shape[1]
    kt = kt.repeat_interleave(G, dim=1)
    vt = vt.repeat_interleave(G, dim=1)
    mask = explicit_mask(B, Lq, Lk, causal, valid_len, mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                         scale=sm_scale)
    scores = (qt @ kt.transpose(-1, -2)) * sm_scale
    lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
    empty = ~mask.any(dim=-1).expand(B, Hq, Lq)
    return o.numpy(), lse.reshape(B * Hq, Lq).numpy(), empty.numpy()


def rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


# ---------------------------------------------------------------- pin battery
# Each pin takes the oracle's float64 entry point and raises AssertionError on
# a mismatch, so the same battery can be run against broken oracle builds.

def pin_brute_force(fwd):
    rng = np.random.default_rng(1)
    cases = [
        (1, 1, 1, 1, 1, False, None),
        (1, 2, 1, 5, 3, True, None),
        (2, 2, 2, 6, 4, False, [3, 6]),
        (2, 4, 2, 7, 5, True, [0, 4]),
        (2, 3, 3, 8, 2, True, [8, 1]),
        (1, 4, 1, 6, 7, False, [5]),
        (2, 2, 1, 8, 8, True, [7, 2]),
    ]
    # query length != key length (Lq, Lk)
    cases += [
        (1, 2, 1, (3, 7), 4, True, None),
        (2, 2, 2, (7, 3), 3, True, [3, 2]),
        (2, 4, 2, (5, 8), 5, False, [6, 0]),
        (1, 3, 3, (8, 2), 2, False, None),
    ]
    for (B, Hq, Hkv, L, D, causal, vl) in cases:
        Lq, Lk = L if isinstance(L, tuple) else (L, L)
        q = rand((B, Hq, Lq, D), rng, 1.5)
        k = rand((B, Hkv, Lk, D), rng)
        v = rand((B, Hkv, Lk, D), rng)
        sm = 1.0 / math.sqrt(D) * 1.7
        o, lse = fwd(q, k, v, sm, causal=causal, valid_len=vl)
        o_ref, lse_ref = brute_force(q, k, v, sm, causal, vl)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)


def pin_torch_sdpa(fwd):
    rng = np.random.default_rng(2)
    cases = [
        (2, 6, 3, 37, 24, False, None),
        (2, 6, 3, 37, 24, True, None),
        (3, 4, 4, 41, 16, False, [41, 0, 17]),
        (2, 8, 1, 50, 32, True, [50, 23]),
        (1, 4, 2, 64, 64, True, [60]),
        (2, 4, 2, (29, 53), 16, True, [53, 11]),
        (2, 4, 4, (61, 22), 32, True, None),
        (1, 8, 2, (40, 70), 24, False, [66]),
    ]
    for (B, Hq, Hkv, L, D, causal, vl) in cases:
        Lq, Lk = L if isinstance(L, tuple) else (L, L)
        q = rand((B, Hq, Lq, D), rng, 2.0)
        k = rand((B, Hkv, Lk, D), rng)
        v = rand((B, Hkv, Lk, D), rng)
        sm = 1.0 / math.sqrt(D)
        o, lse = fwd(q, k, v, sm, causal=causal, valid_len=vl)
        o_ref, lse_ref, empty = torch_reference(q, k, v, sm, causal, vl)
        keep = ~empty
        np.testing.assert_allclose(o[keep], o_ref[keep], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse.reshape(B, Hq, Lq)[keep],
                                   lse_ref.reshape(B, Hq, Lq)[keep], rtol=1e-12, atol=1e-12)
        assert np.all(o[empty] == 0.0)
        assert np.all(np.isneginf(lse.reshape(B, Hq, Lq)[empty]))


def pin_golden(fwd):
    with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
        data = json.load(f)
    for c in data["cases"]:
        q, k, v = (np.array(c[n], dtype=np.float64) for n in ("q", "k", "v"))
        o, lse = fwd(q, k, v, c["sm_scale"], causal=c["causal"], valid_len=c["valid_len"])
        o_exp = np.array(c["o"], dtype=np.float64)
        lse_exp = np.array([[float(x) for x in row] for row in c["lse"]])
        np.testing.assert_allclose(o, o_exp, rtol=0, atol=c["tol"], err_msg=c["name"])
        fin = np.isfinite(lse_exp)
        np.testing.assert_allclose(lse[fin], lse_exp[fin], rtol=0, atol=c["tol"],
                                   err_msg=c["name"])
        assert np.array_equal(np.isneginf(lse), np.isneginf(lse_exp)), c["name"]


def pin_invariants(fwd):
    rng = np.random.default_rng(3)
    # L = 1: the only key is visible, so O = V and LSE = the single scaled score
    q, k, v = rand((2, 4, 1, 8), rng), rand((2, 2, 1, 8), rng), rand((2, 2, 1, 8), rng)
    for causal in (False, True):
        o, lse = fwd(q, k, v, 0.3, causal=causal)
        vv = np.repeat(v, 2, axis=1)
        np.testing.assert_allclose(o, vv, rtol=1e-14, atol=0)
        s = 0.3 * np.einsum("bhid,bhid->bhi", q, np.repeat(k, 2, axis=1))
        np.testing.assert_allclose(lse, s.reshape(8, 1), rtol=1e-13, atol=1e-15)
    # causal row 0 sees key 0 only
    q, k, v = rand((2, 2, 9, 5), rng), rand((2, 2, 9, 5), rng), rand((2, 2, 9, 5), rng)
    o, lse = fwd(q, k, v, 0.7, causal=True)
    np.testing.assert_allclose(o[:, :, 0, :], v[:, :, 0, :], rtol=1e-14, atol=0)
    s0 = 0.7 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(lse.reshape(2, 2, 9)[:, :, 0], s0, rtol=1e-13, atol=1e-15)
    # identical V rows: every output row is that row
    row = rand((6,), rng)
    v = np.broadcast_to(row, (1, 3, 11, 6)).copy()
    q, k = rand((1, 3, 11, 6), rng, 3.0), rand((1, 3, 11, 6), rng)
    for causal, vl in ((False, None), (True, None), (False, [7]), (True, [4])):
        o, _ = fwd(q, k, v, 0.5, causal=causal, valid_len=vl)
        np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), rtol=1e-13, atol=1e-14)
    # fully masked rows: O = 0, LSE = -inf
    q, k, v = rand((3, 2, 6, 4), rng), rand((3, 2, 6, 4), rng), rand((3, 2, 6, 4), rng)
    o, lse = fwd(q, k, v, 0.5, causal=True, valid_len=[0, 6, 0])
    assert np.all(o[0] == 0) and np.all(o[2] == 0)
    assert np.all(np.isneginf(lse.reshape(3, 2, 6)[[0, 2]]))
    assert np.all(np.isfinite(lse.reshape(3, 2, 6)[1]))
    # scaling Q by c while dividing sm_scale by c leaves O and LSE unchanged
    q, k, v = rand((2, 2, 10, 8), rng), rand((2, 2, 10, 8), rng), rand((2, 2, 10, 8), rng)
    o1, l1 = fwd(q, k, v, 0.35, causal=True, valid_len=[10, 4])
    o2, l2 = fwd(q * 2.0, k, v, 0.35 / 2.0, causal=True, valid_len=[10, 4])
    np.testing.assert_array_equal(o1, o2)  # power of two: exact
    np.testing.assert_array_equal(l1, l2)
    o3, l3 = fwd(q * 3.0, k, v, 0.35 / 3.0, causal=True, valid_len=[10, 4])
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l3, l1, rtol=1e-12, atol=1e-13)


def pin_closed_forms(fwd):
    rng = np.random.default_rng(4)
    B, Hq, Hkv, L, D = 2, 4, 2, 9, 6
    q, k, v = rand((B, Hq, L, D), rng), rand((B, Hkv, L, D), rng), rand((B, Hkv, L, D), rng)
    vl = [9, 5]
    # zero scale (or zero keys): uniform weights over the visible keys
    for scale, kk in ((0.0, k), (0.8, np.zeros_like(k))):
        for causal in (False, True):
            o, lse = fwd(q, kk, v, scale, causal=causal, valid_len=vl)
            o = o.reshape(B, Hq, L, D)
            lse = lse.reshape(B, Hq, L)
            for b in range(B):
                for h in range(Hq):
                    g = h // (Hq // Hkv)
                    for i in range(L):
                        n = min(vl[b], i + 1) if causal else vl[b]
                        np.testing.assert_allclose(o[b, h, i], v[b, g, :n].mean(axis=0),
                                                   rtol=1e-12, atol=1e-14)
                        assert abs(lse[b, h, i] - math.log(n)) < 1e-13
    # adding one vector c to every key row shifts every score of row i by
    # sm_scale*q_i.c: O unchanged, LSE shifted by that amount
    c = rand((D,), rng)
    o1, l1 = fwd(q, k, v, 0.4)
    o2, l2 = fwd(q, k + c, v, 0.4)
    np.testing.assert_allclose(o2, o1, rtol=1e-11, atol=1e-12)
    shift = 0.4 * np.einsum("bhid,d->bhi", q, c).reshape(B * Hq, L)
    np.testing.assert_allclose(l2, l1 + shift, rtol=1e-12, atol=1e-12)
    # permuting the key/value rows together changes nothing without a mask
    perm = rng.permutation(L)
    o3, l3 = fwd(q, k[:, :, perm], v[:, :, perm], 0.4)
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l3, l1, rtol=1e-12, atol=1e-13)
    # GQA head map by integer division: kv head g answers q heads g*G .. g*G+G-1
    vh = np.zeros((B, Hkv, L, D))
    for g in range(Hkv):
        vh[:, g] = 10.0 * (g + 1)
    o, _ = fwd(q, k, vh, 0.4, causal=True)
    for h in range(Hq):
        np.testing.assert_allclose(o[:, h], 10.0 * (h // (Hq // Hkv) + 1), rtol=1e-14, atol=0)
    # GQA equals MHA on explicitly repeated K/V; MQA equals GQA with Hkv = 1
    o_g, l_g = fwd(q, k, v, 0.4, causal=True, valid_len=vl)
    o_m, l_m = fwd(q, np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1), 0.4, causal=True,
                   valid_len=vl)
    np.testing.assert_array_equal(o_g, o_m)
    np.testing.assert_array_equal(l_g, l_m)
    o_q, _ = fwd(q, k[:, :1], v[:, :1], 0.4, causal=True)
    o_r, _ = fwd(q, np.repeat(k[:, :1], Hq, axis=1), np.repeat(v[:, :1], Hq, axis=1), 0.4,
                 causal=True)
    np.testing.assert_array_equal(o_q, o_r)


def pin_lengths(fwd):
    """Query length Lq != key length Lk: relations to square problems."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D = 2, 4, 2, 6
    # one key: every query row gets V[0]; LSE is that key's scaled score
    q, k, v = rand((B, Hq, 5, D), rng), rand((B, Hkv, 1, D), rng), rand((B, Hkv, 1, D), rng)
    for causal in (False, True):
        o, lse = fwd(q, k, v, 0.3, causal=causal)
        np.testing.assert_allclose(o, np.broadcast_to(np.repeat(v, 2, axis=1), o.shape),
                                   rtol=1e-14, atol=0)
        s = 0.3 * np.einsum("bhid,bhd->bhi", q, np.repeat(k[:, :, 0], 2, axis=1))
        np.testing.assert_allclose(lse, s.reshape(B * Hq, 5), rtol=1e-13, atol=1e-15)
    # causal, Lk > Lq: keys at positions >= Lq are never visible (top-left
    # alignment), so the result equals the square problem on the first Lq keys
    q = rand((B, Hq, 6, D), rng)
    k, v = rand((B, Hkv, 11, D), rng), rand((B, Hkv, 11, D), rng)
    for vl in (None, [11, 4]):
        o, lse = fwd(q, k, v, 0.45, causal=True, valid_len=vl)
        vl_sq = None if vl is None else [min(x, 6) for x in vl]
        o_sq, lse_sq = fwd(q, k[:, :, :6], v[:, :, :6], 0.45, causal=True, valid_len=vl_sq)
        np.testing.assert_array_equal(o, o_sq)
        np.testing.assert_array_equal(lse, lse_sq)
    # causal, Lq > Lk: rows i < Lk are the square problem; rows i >= Lk - 1
    # see every key, as without the causal mask
    q = rand((B, Hq, 10, D), rng)
    k, v = rand((B, Hkv, 4, D), rng), rand((B, Hkv, 4, D), rng)
    o, lse = fwd(q, k, v, 0.45, causal=True)
    o_sq, lse_sq = fwd(q[:, :, :4], k, v, 0.45, causal=True)
    np.testing.assert_array_equal(o[:, :, :4], o_sq)
    np.testing.assert_array_equal(lse.reshape(B, Hq, 10)[:, :, :4], lse_sq.reshape(B, Hq, 4))
    o_nc, lse_nc = fwd(q, k, v, 0.45, causal=False)
    np.testing.assert_array_equal(o[:, :, 3:], o_nc[:, :, 3:])
    np.testing.assert_array_equal(lse.reshape(B, Hq, 10)[:, :, 3:],
                                  lse_nc.reshape(B, Hq, 10)[:, :, 3:])
    # without the causal mask query rows are independent: the rows of a split
    # query block equal the whole block's rows
    q = rand((B, Hq, 9, D), rng)
    k, v = rand((B, Hkv, 13, D), rng), rand((B, Hkv, 13, D), rng)
    o, lse = fwd(q, k, v, 0.5, valid_len=[13, 6])
    o_a, lse_a = fwd(q[:, :, :4], k, v, 0.5, valid_len=[13, 6])
    o_b, lse_b = fwd(q[:, :, 4:], k, v, 0.5, valid_len=[13, 6])
    np.testing.assert_array_equal(o, np.concatenate([o_a, o_b], axis=2))
    np.testing.assert_array_equal(lse.reshape(B, Hq, 9),
                                  np.concatenate([lse_a.reshape(B, Hq, 4),
                                                  lse_b.reshape(B, Hq, 5)], axis=2))


def pin_explicit_mask(fwd):
    """The explicit [B, Lq, Lk] mask: brute force, torch SDPA and the masks
    it must reproduce exactly (all ones = none, tril = causal, key < valid_len
    = padding, one mask shared by every batch)."""
    rng = np.random.default_rng(8)
    # brute force, combined with causal and padding, Lq != Lk, batch-broadcast
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl, shared) in [
            (2, 2, 1, 6, 6, 3, False, None, False), (2, 4, 2, 7, 5, 4, True, [5, 3], False),
            (1, 2, 2, 5, 8, 2, False, [7], True), (3, 2, 1, 4, 4, 5, True, None, True)]:
        q, k, v = rand((B, Hq, Lq, D), rng, 1.5), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        mk = (rng.random((1 if shared else B, Lq, Lk)) < 0.6).astype(np.uint8)
        mk[0, 1, :] = 0  # one fully masked row
        o, lse = fwd(q, k, v, 0.7, causal=causal, valid_len=vl, mask=mk)
        o_ref, lse_ref = brute_force(q, k, v, 0.7, causal, vl, mk)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)
    # torch SDPA on medium shapes with random, block and empty-row masks
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl, dens) in [
            (2, 4, 2, 33, 33, 16, False, None, 0.5), (2, 4, 1, 40, 57, 8, True, [50, 21], 0.2),
            (3, 2, 2, 29, 29, 12, False, [29, 0, 11], 0.9)]:
        q, k, v = rand((B, Hq, Lq, D), rng, 2.0), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        mk = (rng.random((B, Lq, Lk)) < dens).astype(np.uint8)
        mk[1, 3:9, :] = 0
        o, lse = fwd(q, k, v, 0.3, causal=causal, valid_len=vl, mask=mk)
        o_ref, lse_ref, empty = torch_reference(q, k, v, 0.3, causal, vl, mk)
        keep = ~empty
        np.testing.assert_allclose(o[keep], o_ref[keep], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse.reshape(B, Hq, Lq)[keep],
                                   lse_ref.reshape(B, Hq, Lq)[keep], rtol=1e-12, atol=1e-12)
        assert np.all(o[empty] == 0.0)
        assert np.all(np.isneginf(lse.reshape(B, Hq, Lq)[empty]))
    # masks that restate the implicit ones give identical results
    B, Hq, Hkv, L, D = 2, 4, 2, 12, 6
    q, k, v = rand((B, Hq, L, D), rng), rand((B, Hkv, L, D), rng), rand((B, Hkv, L, D), rng)
    o0, l0 = fwd(q, k, v, 0.5)
    o1, l1 = fwd(q, k, v, 0.5, mask=np.ones((B, L, L), np.uint8))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    oc, lc = fwd(q, k, v, 0.5, causal=True)
    om, lm = fwd(q, k, v, 0.5, mask=np.tril(np.ones((L, L), np.uint8)))
    np.testing.assert_array_equal(oc, om)
    np.testing.assert_array_equal(lc, lm)
    vl = [7, 12]
    op, lp = fwd(q, k, v, 0.5, valid_len=vl)
    pm = np.stack([np.broadcast_to(np.arange(L) < x, (L, L)) for x in vl]).astype(np.uint8)
    oq, lq = fwd(q, k, v, 0.5, mask=pm)
    np.testing.assert_array_equal(op, oq)
    np.testing.assert_array_equal(lp, lq)
    # a shared mask equals the same mask repeated per batch
    sm = (rng.random((L, L)) < 0.5).astype(np.uint8)
    o2, l2 = fwd(q, k, v, 0.5, causal=True, mask=sm)
    o3, l3 = fwd(q, k, v, 0.5, causal=True, mask=np.stack([sm, sm]))
    np.testing.assert_array_equal(o2, o3)
    np.testing.assert_array_equal(l2, l3)


PINS = [pin_brute_force, pin_torch_sdpa, pin_golden, pin_invariants, pin_closed_forms,
        pin_lengths, pin_explicit_mask]


# ---------------------------------------------------------------- the tests

@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_fwd_default)


def test_decode_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bits_entry_matches_decoded_f64_entry():
    from attention_forward_attn_gb300 import workloads as wl
    for dtype in (wl.F16, wl.BF16):
        q, k, v, vl = wl.make_inputs(2, 4, 2, 70, 64, dtype, seed=5, padded=True)
        code = wl.dtype_code(dtype)
        qb, kb, vb = wl.bits(q), wl.bits(k), wl.bits(v)
        o1, l1 = oracle.attn_fwd_bits(qb, kb, vb, code, 0.125, causal=True, valid_len=vl.numpy())
        o2, l2 = oracle.attn_fwd_f64(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                     0.125, causal=True, valid_len=vl.numpy())
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_row_subset_matches_full():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, L, D = 2, 4, 1, 33, 16
    q, k, v = rand((B, Hq, L, D), rng), rand((B, Hkv, L, D), rng), rand((B, Hkv, L, D), rng)
    o, lse = oracle.attn_fwd_f64(q, k, v, 0.25, causal=True, valid_len=[20, 0])
    rows = rng.choice(B * Hq * L, size=50, replace=False)
    o_s, lse_s = oracle.attn_fwd_f64(q, k, v, 0.25, causal=True, valid_len=[20, 0], rows=rows)
    np.testing.assert_array_equal(o_s, o.reshape(-1, D)[rows])
    np.testing.assert_array_equal(lse_s, lse.reshape(-1)[rows])


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 4, 2))
    k = np.zeros((1, 2, 4, 2))
    with pytest.raises(ValueError):
        oracle.attn_fwd_f64(q, k, k, 1.0)  # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attn_fwd_f64(np.zeros((1, 2, 4, 2)), k, k, 1.0, rows=[8])  # row out of range


MUTANTS = {
    "dropped_scale": ("s[j] = sm_scale * dot;", "s[j] = dot;"),
    "causal_off_by_one": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    "causal_inverted": ("if (causal && j > i) return 0;", "if (causal && j < i) return 0;"),
    "padding_off_by_one": ("j >= (int64_t)valid_len[b]", "j > (int64_t)valid_len[b]"),
    "modulo_head_map": ("const int h_kv = h_q / G;", "const int h_kv = h_q % Hkv;"),
    "transposed_k": ("dot += q_row[d] * k_row[d];", "dot += q_row[d] * k_head[d * (int64_t)Lk + j];"),
    "key_head_stride_from_query_length": ("* Lk * (int64_t)D;", "* Lq * (int64_t)D;"),
    "row_split_by_key_length": ("const int64_t i = r % Lq;", "const int64_t i = r % Lk;"),
    "padding_on_query_index": ("j >= (int64_t)valid_len[b]", "i >= (int64_t)valid_len[b]"),
    "mask_ignored": ("mk->mask[b * mk->batch_stride + i * mk->row_stride + j] == 0) return 0;",
                     "mk->mask[b * mk->batch_stride + i * mk->row_stride + j] == 2) return 0;"),
    "mask_row_off_by_one": ("mk->mask[b * mk->batch_stride + i * mk->row_stride + j]",
                            "mk->mask[b * mk->batch_stride + (i > 0 ? i - 1 : 0) * mk->row_stride + j]"),
    "mask_batch_ignored": ("mk->mask[b * mk->batch_stride + i", "mk->mask[0 * mk->batch_stride + i"),
    "log2_lse": ("*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    "lse_without_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) o_row[d] /= l;", ""),
    "exp_sign": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "batch_index_mixup": ("const int b = (int)(bh / Hq);", "const int b = (int)(bh % B);"),
    "value_from_key": ("const double* v_row = v_head + j * (int64_t)D;",
                       "const double* v_row = k_head + j * (int64_t)D;"),
    "empty_row_not_zeroed": ("for (int d = 0; d < D; ++d) o_row[d] = 0.0;\n    *lse_out = -INFINITY;",
                             "*lse_out = -INFINITY;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    """A plausible mistake planted in a copy of the oracle must fail a pin."""
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, "mutation anchor not found: %r" % old
    path_c = tmp_path / ("mut_%s.c" % name)
    path_so = tmp_path / ("mut_%s.so" % name)
    path_c.write_text(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-fopenmp", str(path_c), "-o",
                    str(path_so), "-lm"], check=True)
    lib = oracle.load_variant(str(path_so))

    def fwd(*a, **kw):
        return oracle.attn_fwd_f64(*a, _lib_override=lib, **kw)

    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(fwd)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
