"""Pins for oracle.attn_bwd_rows_f64, the sampled-rows backward used at full
sizes:

* its dQ, dK, dV rows equal the full backward oracle's (attn_bwd_f64, itself
  pinned by finite differences and autograd in test_oracle_bwd_pins.py) on
  causal / padded (with an empty batch) / GQA / MQA cases, rows in any order;
* its magnitudes (sum |dS|, sum_d |dO O|, sum P, sum P w, visible counts)
  equal a float64 brute force over the materialised score matrix;
* broken copies of the function (delta dropped, wrong query head of a key's
  group, P not normalised, dQ from the wrong K head) fail a pin.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle

CASES = [  # B, Hq, Hkv, Lq, Lk, D, causal, valid_len
    (2, 4, 2, 37, 37, 8, True, [37, 11]),
    (1, 6, 3, 29, 29, 5, False, None),
    (2, 4, 1, 23, 23, 4, True, [0, 23]),
    (3, 2, 2, 19, 19, 6, False, [5, 19, 1]),
    (2, 4, 2, 17, 31, 8, True, [31, 6]),
    (1, 2, 1, 33, 14, 4, True, None),
]


def inputs(case, seed):
    B, Hq, Hkv, Lq, Lk, D, causal, vl = case
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, Lq, D)), rng.standard_normal((B, Hkv, Lk, D)),
            rng.standard_normal((B, Hkv, Lk, D)), rng.standard_normal((B, Hq, Lq, D)))


def pin_rows_match_full(rows_fn):
    for n, case in enumerate(CASES):
        B, Hq, Hkv, Lq, Lk, D, causal, vl = case
        q, k, v, do = inputs(case, 40 + n)
        dq, dk, dv = oracle.attn_bwd_f64(q, k, v, do, 0.6, causal=causal, valid_len=vl)
        rng = np.random.default_rng(n)
        qr = rng.permutation(B * Hq * Lq)
        kr = rng.permutation(B * Hkv * Lk)
        dq2, _, dk2, dv2, _ = rows_fn(q, k, v, do, 0.6, causal=causal, valid_len=vl, q_rows=qr,
                                      k_rows=kr)
        np.testing.assert_allclose(dq2, dq.reshape(-1, D)[qr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk2, dk.reshape(-1, D)[kr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv2, dv.reshape(-1, D)[kr], rtol=1e-11, atol=1e-12)


def brute_magnitudes(q, k, v, do, sm, causal, vl):
    B, Hq, Lq, D = q.shape
    Lk = k.shape[2]
    G = Hq // k.shape[1]
    qm = np.zeros((B, Hq, Lq, 3))
    km = np.zeros((B, k.shape[1], Lk, 4))
    for b in range(B):
        vis = np.ones((Lq, Lk), dtype=bool)
        if causal:
            vis &= np.tri(Lq, Lk, dtype=bool)
        if vl is not None:
            vis[:, vl[b]:] = False
        for h in range(Hq):
            hk = h // G
            s = np.where(vis, sm * q[b, h] @ k[b, hk].T, -np.inf)
            mx = np.max(s, axis=1, keepdims=True)
            e = np.where(vis, np.exp(s - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
            z = e.sum(axis=1, keepdims=True)
            p = np.divide(e, z, out=np.zeros_like(e), where=z > 0)
            dp = do[b, h] @ v[b, hk].T
            ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
            w = np.sum(np.abs(do[b, h] * (p @ v[b, hk])), axis=1)
            qm[b, h, :, 0] = np.abs(ds).sum(axis=1)
            qm[b, h, :, 1] = w
            qm[b, h, :, 2] = vis.sum(axis=1)
            km[b, hk, :, 0] += np.abs(ds).sum(axis=0)
            km[b, hk, :, 1] += p.sum(axis=0)
            km[b, hk, :, 2] += (p * w[:, None]).sum(axis=0)
            km[b, hk, :, 3] += (vis & (vis.sum(axis=1) > 0)[:, None]).sum(axis=0)
    return qm.reshape(-1, 3), km.reshape(-1, 4)


def pin_magnitudes(rows_fn):
    for n, case in enumerate(CASES):
        B, Hq, Hkv, Lq, Lk, D, causal, vl = case
        q, k, v, do = inputs(case, 60 + n)
        _, qm, _, _, km = rows_fn(q, k, v, do, 0.6, causal=causal, valid_len=vl,
                                  q_rows=np.arange(B * Hq * Lq), k_rows=np.arange(B * Hkv * Lk))
        qm_ref, km_ref = brute_magnitudes(q, k, v, do, 0.6, causal, vl)
        qm_ref[qm_ref[:, 2] == 0, :2] = 0.0  # rows with no key: no dS, O = 0
        np.testing.assert_allclose(qm, qm_ref, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(km, km_ref, rtol=1e-11, atol=1e-12)


def pin_rows_match_full_masked(rows_fn):
    """With an explicit mask (per batch and shared), also against the full
    backward oracle."""
    for n, (case, shared) in enumerate([(CASES[0], False), (CASES[4], True), (CASES[5], False)]):
        B, Hq, Hkv, Lq, Lk, D, causal, vl = case
        q, k, v, do = inputs(case, 80 + n)
        rng = np.random.default_rng(90 + n)
        mk = (rng.random((Lq, Lk) if shared else (B, Lq, Lk)) < 0.5).astype(np.uint8)
        dq, dk, dv = oracle.attn_bwd_f64(q, k, v, do, 0.6, causal=causal, valid_len=vl, mask=mk)
        qr = rng.permutation(B * Hq * Lq)
        kr = rng.permutation(B * Hkv * Lk)
        dq2, _, dk2, dv2, _ = rows_fn(q, k, v, do, 0.6, causal=causal, valid_len=vl, q_rows=qr,
                                      k_rows=kr, mask=mk)
        np.testing.assert_allclose(dq2, dq.reshape(-1, D)[qr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk2, dk.reshape(-1, D)[kr], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv2, dv.reshape(-1, D)[kr], rtol=1e-11, atol=1e-12)


PINS = [pin_rows_match_full, pin_magnitudes, pin_rows_match_full_masked]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_bwd_rows_oracle_pin(pin):
    pin(oracle.attn_bwd_rows_f64)


def test_bwd_rows_rejects_out_of_range_rows():
    q, k, v, do = inputs(CASES[0], 1)
    with pytest.raises(ValueError):
        oracle.attn_bwd_rows_f64(q, k, v, do, 0.6, q_rows=[q.size // q.shape[-1]])
    with pytest.raises(ValueError):
        oracle.attn_bwd_rows_f64(q, k, v, do, 0.6, k_rows=[-1])


MUTANTS = {
    "delta_dropped": ("const double ds = p * (dp - st[4 * gi + 2]);", "const double ds = p * dp;"),
    "wrong_query_head": ("const int64_t qrow = ((int64_t)b * Hq + (int64_t)h_kv * G + gi / Lq) * Lq + i;",
                         "const int64_t qrow = ((int64_t)b * Hq + gi / Lq) * Lq + i;"),
    "p_not_normalised": ("const double p = exp(sm_scale * dot - st[4 * gi]) / st[4 * gi + 1];",
                         "const double p = exp(sm_scale * dot - st[4 * gi]);"),
    "dq_wrong_kv_head": ("const int64_t kvh = (int64_t)b * Hkv + (qh % Hq) / G;",
                         "const int64_t kvh = (int64_t)b * Hkv + (qh % Hq) % Hkv;"),
    "mask_ignored": ("const oracle_mask_t mk = {mask, mask_batch_stride, mask_row_stride};  /* the rows' key sets */",
                     "const oracle_mask_t mk = {NULL, 0, 0};"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_rows_pins_catch_mutant(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, "mutation anchor not found: %r" % old
    path_c = tmp_path / ("mut_%s.c" % name)
    path_so = tmp_path / ("mut_%s.so" % name)
    path_c.write_text(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-fopenmp", str(path_c), "-o",
                    str(path_so), "-lm"], check=True)
    lib = oracle.load_variant(str(path_so))

    def rows_fn(*a, **kw):
        return oracle.attn_bwd_rows_f64(*a, _lib_override=lib, **kw)

    failed = []
    for pin in PINS:
        try:
            pin(rows_fn)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name
