"""GPU parity of attn_bwd (dQ, dK, dV) against the float64 backward oracle.

The GPU runs the forward (attn_fwd) for O and its LSE, then attn_bwd with a
seeded dO; the oracle takes the same 16-bit Q, K, V, dO values and computes
the gradients from the definition.

Tolerance, derived from the one approximation in the method:
delta_i = dO_i . O_i is formed from the forward's 16-bit O (the output
rounding, unit roundoff u = 2^-9 bf16 / 2^-12 fp16, plus the forward's own
error, taken as another u), so |d delta_i| <= 2u sum_d |dO_id O_id| =: e_i,
and every dS_ij = P_ij (dP_ij - delta_i) of row i moves by P_ij e_i:
    |d dQ_id| <= sm_scale e_i |sum_j P_ij k_jd|      (the forward with V := K)
    |d dK_jd| <= sm_scale sum_i P_ij e_i |q_id|      (dV of the backward with dO_i := e_i |q_i|)
Both sides of that are computed by the oracle (never from the GPU).  On top
of it: 1e-2 |g_ref| (the final rounding to the 16-bit dtype, 2^-9 for bf16)
and 1e-4 max|g_ref| (fp32 accumulation).  dV does not involve delta.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    attn.status()


def run_case(B, Hq, Hkv, L, D, dtype, causal, vl, seed):
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=seed, valid_len=vl)
    gen = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, Hq, L, D, generator=gen).to(wl.TORCH_DTYPE[dtype])
    dev = torch.device("cuda")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    vld = None if vl_t is None else vl_t.to(dev)
    sm = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=causal, sm_scale=sm, valid_len=vld)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, sm_scale=sm, valid_len=vld)
    st, code = attn.status()
    assert st == attn.ATTN_OK, "device status %d (code %#x)" % (st, code)
    f = lambda t: t.double().numpy()
    vl_np = None if vl is None else np.array(vl, np.int32)
    qf, kf, vf, dof = f(q), f(k), f(v), f(do)
    ref = oracle.attn_bwd_f64(qf, kf, vf, dof, sm, causal=causal, valid_len=vl_np)
    u = 2.0 ** -9 if dtype == wl.BF16 else 2.0 ** -12
    o_ref, _ = oracle.attn_fwd_f64(qf, kf, vf, sm, causal=causal, valid_len=vl_np)
    e = 2 * u * np.sum(np.abs(dof * o_ref), axis=-1, keepdims=True)   # [B, Hq, L, 1]
    pk, _ = oracle.attn_fwd_f64(qf, kf, kf, sm, causal=causal, valid_len=vl_np)
    _, _, pq = oracle.attn_bwd_f64(qf, kf, vf, e * np.abs(qf), sm, causal=causal, valid_len=vl_np)
    delta_terms = (sm * e * np.abs(pk), sm * pq, 0.0)
    for name, g, r, dt in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, delta_terms):
        g = g.float().cpu().double().numpy()
        err = np.abs(g - r)
        bound = 1e-2 * np.abs(r) + 1e-4 * np.abs(r).max() + dt
        assert np.all(err <= bound), "%s: %d elements out of tolerance (max err %g, max ref %g)" % (
            name, int((err > bound).sum()), float(err.max()), float(np.abs(r).max()))


@pytest.mark.parametrize("D, dtype", [(64, wl.F16), (128, wl.BF16), (64, wl.BF16), (128, wl.F16)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L, vl", [(200, [200, 0]), (129, [77, 129]), (64, None)])
def test_bwd_matches_oracle(D, dtype, causal, L, vl):
    run_case(2, 4, 2, L, D, dtype, causal, vl, seed=L + D)


@pytest.mark.parametrize("Hq, Hkv", [(8, 1), (8, 8)])
def test_bwd_medium_gqa_mqa(Hq, Hkv):
    run_case(1, Hq, Hkv, 512, 128, wl.BF16, True, None, seed=512 + Hkv)
