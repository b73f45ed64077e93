"""Pins for the float64 backward oracle (oracle.attn_bwd_f64), checked against
things other than its own formulas:

* central finite differences of the forward oracle: for the loss
  sum(O * dO), each gradient element is (loss(x + h) - loss(x - h)) / 2h,
  computed with the FORWARD oracle only (no backward formula involved);
* PyTorch CPU float64 autograd through scaled_dot_product_attention with an
  explicit boolean mask and repeat_interleave for the head map;
* closed forms: dO = 0 gives zero gradients; identical V rows give
  dQ = dK = 0 (every dP_ij equals the row's weighted mean); the dV rows of a
  head sum to the sum of dO over the query rows that see any key
  (each P row sums to 1).

The last test compiles broken copies of the backward (a dropped softmax
Jacobian term, a missing scale, dK from the wrong operand, GQA gradients
written to one query head only) and checks that each fails a pin.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle


def rand(shape, rng, scale=1.0):
    return rng.standard_normal(shape) * scale


def finite_differences(q, k, v, do, sm, causal, vl, h=1e-6, mask=None):
    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd_f64(qq, kk, vv, sm, causal=causal, valid_len=vl, mask=mask)
        return float(np.sum(o * do))

    grads = []
    for which in range(3):
        x = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(x[which])
        it = np.nditer(g, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = [a.copy() for a in x]
            xm = [a.copy() for a in x]
            xp[which][idx] += h
            xm[which][idx] -= h
            g[idx] = (loss(*xp) - loss(*xm)) / (2 * h)
        grads.append(g)
    return grads


def torch_grads(q, k, v, do, sm, causal, vl, explicit=None):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    B, Hq, Lq, D = q.shape
    Lk = k.shape[2]
    G = Hq // k.shape[1]
    mask = torch.ones(B, 1, Lq, Lk, dtype=torch.bool)
    if causal:  # top-left: key j visible to query i iff j <= i
        mask &= torch.tril(torch.ones(Lq, Lk, dtype=torch.bool))
    if vl is not None:
        for b in range(B):
            mask[b, :, :, :] &= (torch.arange(Lk) < int(vl[b]))[None, :]
    if explicit is not None:  # [B, Lq, Lk] or [Lq, Lk], nonzero keeps
        mask &= torch.from_numpy(np.asarray(explicit) != 0).reshape(-1, 1, Lq, Lk)
    empty = ~mask.any(dim=-1, keepdim=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1),
        attn_mask=mask | empty, scale=sm)  # rows with no key: any finite stand-in, zeroed below
    o = o.masked_fill(empty.expand(B, Hq, Lq, 1), 0.0)
    (o * torch.from_numpy(do)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def pin_finite_differences(bwd):
    rng = np.random.default_rng(11)
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl) in [
            (1, 2, 1, 4, 4, 3, True, None), (2, 2, 2, 5, 5, 2, False, [3, 5]),
            (1, 4, 2, 4, 4, 3, True, [3]),
            (1, 2, 1, 3, 6, 2, True, None),      # Lq < Lk
            (2, 2, 1, 6, 3, 2, True, [3, 2])]:   # Lq > Lk: late queries see every key
        q, k, v = rand((B, Hq, Lq, D), rng), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        do = rand((B, Hq, Lq, D), rng)
        got = bwd(q, k, v, do, 0.8, causal=causal, valid_len=vl)
        ref = finite_differences(q, k, v, do, 0.8, causal, vl)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-6, atol=1e-8)


def pin_torch_autograd(bwd):
    rng = np.random.default_rng(12)
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl) in [
            (2, 4, 2, 23, 23, 8, True, [23, 9]), (1, 6, 3, 31, 31, 16, False, None),
            (3, 2, 1, 17, 17, 4, True, [0, 17, 5]),
            (2, 4, 2, 19, 27, 8, True, [27, 9]), (1, 2, 1, 29, 12, 4, True, None),
            (2, 2, 2, 9, 21, 6, False, [21, 4])]:
        q, k, v = rand((B, Hq, Lq, D), rng, 1.5), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        do = rand((B, Hq, Lq, D), rng)
        sm = 1.0 / math.sqrt(D)
        got = bwd(q, k, v, do, sm, causal=causal, valid_len=vl)
        ref = torch_grads(q, k, v, do, sm, causal, vl)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-11)


def pin_closed_forms(bwd):
    rng = np.random.default_rng(13)
    B, Hq, Hkv, L, D = 2, 4, 2, 9, 5
    q, k, v = rand((B, Hq, L, D), rng), rand((B, Hkv, L, D), rng), rand((B, Hkv, L, D), rng)
    vl = [9, 0]
    for g in bwd(q, k, v, np.zeros((B, Hq, L, D)), 0.4, causal=True, valid_len=vl):
        assert np.all(g == 0.0)
    do = rand((B, Hq, L, D), rng)
    vc = np.broadcast_to(rand((D,), rng), v.shape).copy()
    dq, dk, dv = bwd(q, k, vc, do, 0.4, causal=True)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    np.testing.assert_allclose(dk, 0.0, atol=1e-13)
    # each P row sums to 1: the dV rows of a K/V head sum to the dO of its query heads
    dq, dk, dv = bwd(q, k, v, do, 0.4, causal=True, valid_len=vl)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hkv):
            want = do[b, h * G:(h + 1) * G].sum(axis=(0, 1)) if vl[b] > 0 else np.zeros(D)
            np.testing.assert_allclose(dv[b, h].sum(axis=0), want, rtol=1e-12, atol=1e-12)


def pin_explicit_mask(bwd):
    """An explicit [B, Lq, Lk] (or shared [Lq, Lk]) mask combined with causal
    and padding: finite differences of the masked forward oracle, and
    autograd through the masked SDPA."""
    rng = np.random.default_rng(14)
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl, shared) in [
            (2, 2, 1, 4, 5, 2, False, None, False), (1, 2, 2, 5, 5, 3, True, [4], True)]:
        q, k, v = rand((B, Hq, Lq, D), rng), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        do = rand((B, Hq, Lq, D), rng)
        mk = (rng.random((Lq, Lk) if shared else (B, Lq, Lk)) < 0.6).astype(np.uint8)
        mk[..., 0, :] = 0  # a query row that sees no key
        got = bwd(q, k, v, do, 0.8, causal=causal, valid_len=vl, mask=mk)
        ref = finite_differences(q, k, v, do, 0.8, causal, vl, mask=mk)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-6, atol=1e-8)
    for (B, Hq, Hkv, Lq, Lk, D, causal, vl) in [(2, 4, 2, 21, 27, 8, True, [27, 9]),
                                                 (3, 2, 1, 17, 13, 4, False, None)]:
        q, k, v = rand((B, Hq, Lq, D), rng, 1.5), rand((B, Hkv, Lk, D), rng), rand((B, Hkv, Lk, D), rng)
        do = rand((B, Hq, Lq, D), rng)
        mk = (rng.random((B, Lq, Lk)) < 0.5).astype(np.uint8)
        mk[0, 3:7, :] = 0
        got = bwd(q, k, v, do, 0.3, causal=causal, valid_len=vl, mask=mk)
        ref = torch_grads(q, k, v, do, 0.3, causal, vl, explicit=mk)
        for g, r in zip(got, ref):
            np.testing.assert_allclose(g, r, rtol=1e-10, atol=1e-11)


PINS = [pin_finite_differences, pin_torch_autograd, pin_closed_forms, pin_explicit_mask]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_bwd_oracle_pin(pin):
    pin(oracle.attn_bwd_f64)


MUTANTS = {
    "no_jacobian_mean": ("const double ds = p[j] * (dp[j] - pdp);", "const double ds = p[j] * dp[j];"),
    "dq_without_scale": ("dq_row[d] += sm_scale * ds * k_head[j * D + d];",
                         "dq_row[d] += ds * k_head[j * D + d];"),
    "dk_from_keys": ("dk_head[j * D + d] += sm_scale * ds * q_row[d];",
                     "dk_head[j * D + d] += sm_scale * ds * k_head[j * D + d];"),
    "dv_without_p": ("dv_head[j * D + d] += p[j] * do_row[d];", "dv_head[j * D + d] += do_row[d];"),
    "one_query_head": ("for (int g = 0; g < G; ++g) {", "for (int g = 0; g < 1; ++g) {"),
    "mask_ignored": ("const oracle_mask_t mk = {mask, mask_batch_stride, mask_row_stride};  /* explicit mask or none */",
                     "const oracle_mask_t mk = {NULL, 0, 0};"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_pins_catch_mutant(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found: %r" % old
    path_c = tmp_path / ("mut_%s.c" % name)
    path_so = tmp_path / ("mut_%s.so" % name)
    path_c.write_text(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-fopenmp", str(path_c), "-o",
                    str(path_so), "-lm"], check=True)
    lib = oracle.load_variant(str(path_so))

    def bwd(*a, **kw):
        return oracle.attn_bwd_f64(*a, _lib_override=lib, **kw)

    failed = []
    for pin in PINS:
        try:
            pin(bwd)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
