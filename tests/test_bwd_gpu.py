"""GPU parity of attn_bwd (tensor cores) and attn_bwd_simt (fp32 SIMT) -- dQ,
dK, dV -- against the float64 backward oracle.

The GPU runs the forward (attn_fwd) for O and its LSE, then the backward with
a seeded dO; the oracle takes the same 16-bit Q, K, V, dO values and computes
the gradients from the definition.

Tolerance, derived from the approximations each path makes (u = 2^-8 for
bf16, 2^-11 for fp16: the unit roundoff of rounding to nearest):

* both paths form delta_i = dO_i . O_i from the forward's 16-bit O, whose
  rounding moves every element by at most u |O_id|, so
  |d delta_i| <= u sum_d |dO_id O_id| =: e_i, and every dS_ij =
  P_ij (dP_ij - delta_i) of row i moves by P_ij e_i:
      |d dQ_id| <= sm_scale e_i |sum_j P_ij k_jd|   (the forward with V := K)
      |d dK_jd| <= sm_scale sum_i P_ij e_i |q_id|   (dV of the backward with dO_i := e_i |q_i|)
  both computed by the oracle (never from the GPU);
* the tensor-core path rounds P and dS to the input dtype as MMA operands
  (relative error <= u each; for fp16 also an absolute 2^-25 below the
  normal range):
      |d dV_jd| <= u sum_i P_ij |dO_id|        + a sum_i |dO_id|
      |d dK_jd| <= sm_scale (u sum_i |dS_ij| |q_id| + a sum_i |q_id|)
      |d dQ_id| <= sm_scale (u sum_j |dS_ij| |k_jd| + a sum_j |k_jd|)
  with P and dS materialised in float64 from the inputs and the oracle's LSE;
* on top of either: 1e-2 |g_ref| (the final rounding of each result to the
  16-bit dtype) and 1e-4 max|g_ref| (fp32 accumulation and the fp32 scores).
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


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    attn.load()
    attn.status()


def visible(B, Lq, Lk, causal, vl, mask=None):
    """[B, Lq, Lk] bool: key j visible to query i (causal: j <= i; explicit
    mask [B or 1, Lq, Lk])."""
    m = np.ones((B, Lq, Lk), dtype=bool)
    if causal:
        m &= np.tri(Lq, Lk, dtype=bool)[None]
    if mask is not None:
        m &= np.asarray(mask).reshape(-1, Lq, Lk) != 0
    if vl is not None:
        for b in range(B):
            m[b, :, int(vl[b]):] = False
    return m


def operand_terms(qf, kf, vf, dof, sm, causal, vl, lse_ref, mask=None):
    """sum_i P |dO|, sum_i |dS| |q|, sum_j |dS| |k| and the plain sums of
    |dO|, |q|, |k| over the same index sets, per gradient element (float64)."""
    B, Hq, L, D = qf.shape
    G = Hq // kf.shape[1]
    vis = visible(B, L, kf.shape[2], causal, vl, mask)
    tv, tk, tq = np.zeros_like(vf), np.zeros_like(kf), np.zeros_like(qf)
    av, ak, aq = np.zeros_like(vf), np.zeros_like(kf), np.zeros_like(qf)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            s = sm * qf[b, h] @ kf[b, hk].T
            lse = lse_ref[b, h][:, None]
            p = np.where(vis[b] & np.isfinite(lse), np.exp(np.where(vis[b], s, 0.0) - np.where(
                np.isfinite(lse), lse, 0.0)), 0.0)
            dp = dof[b, h] @ vf[b, hk].T
            delta = np.sum(p * dp, axis=1, keepdims=True)
            ds = np.abs(p * (dp - delta))
            tv[b, hk] += p.T @ np.abs(dof[b, h])
            tk[b, hk] += ds.T @ np.abs(qf[b, h])
            tq[b, h] = ds @ np.abs(kf[b, hk])
            av[b, hk] += vis[b].T.astype(np.float64) @ np.abs(dof[b, h])
            ak[b, hk] += vis[b].T.astype(np.float64) @ np.abs(qf[b, h])
            aq[b, h] = vis[b].astype(np.float64) @ np.abs(kf[b, hk])
    return (tq, tk, tv), (aq, ak, av)


def run_case(B, Hq, Hkv, L, D, dtype, causal, vl, seed, impl, Lk=None, mask=None):
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=seed, valid_len=vl, Lk=Lk)
    gen = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, Hq, L, D, generator=gen).to(wl.TORCH_DTYPE[dtype])
    dev = torch.device("cuda")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    vld = None if vl_t is None else vl_t.to(dev)
    sm = 1.0 / math.sqrt(D)
    md = None if mask is None else torch.from_numpy(mask).to(dev)
    o, lse = attn.attn_fwd_strided(qd, kd, vd, causal=causal, sm_scale=sm, valid_len=vld, mask=md)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal, sm_scale=sm, valid_len=vld,
                               impl=impl, mask=md)
    st, code = attn.status()
    assert st == attn.ATTN_OK, "device status %d (code %#x)" % (st, code)
    f = lambda t: t.double().numpy()
    vl_np = None if vl is None else np.array(vl, np.int32)
    qf, kf, vf, dof = f(q), f(k), f(v), f(do)
    ref = oracle.attn_bwd_f64(qf, kf, vf, dof, sm, causal=causal, valid_len=vl_np, mask=mask)
    u = 2.0 ** -8 if dtype == wl.BF16 else 2.0 ** -11
    o_ref, lse_ref = oracle.attn_fwd_f64(qf, kf, vf, sm, causal=causal, valid_len=vl_np, mask=mask)
    e = u * np.sum(np.abs(dof * o_ref), axis=-1, keepdims=True)   # [B, Hq, L, 1]
    pk, _ = oracle.attn_fwd_f64(qf, kf, kf, sm, causal=causal, valid_len=vl_np, mask=mask)
    _, _, pq = oracle.attn_bwd_f64(qf, kf, vf, e * np.abs(qf), sm, causal=causal, valid_len=vl_np,
                                   mask=mask)
    terms = [sm * e * np.abs(pk), sm * pq, np.zeros_like(vf)]
    if impl == "tc":
        rel, ab = operand_terms(qf, kf, vf, dof, sm, causal, vl_np,
                                lse_ref.reshape(B, Hq, L).astype(np.float64), mask)
        a = 0.0 if dtype == wl.BF16 else 2.0 ** -25
        scale = (sm, sm, 1.0)
        terms = [t + c * (u * r + a * s) for t, c, r, s in zip(terms, scale, rel, ab)]
    for name, g, r, dt in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, terms):
        g = g.float().cpu().double().numpy()
        err = np.abs(g - r)
        bound = 1e-2 * np.abs(r) + 1e-4 * np.abs(r).max() + dt
        assert np.all(err <= bound), "%s %s: %d elements out of tolerance (max err %g, max ref %g)" % (
            impl, name, int((err > bound).sum()), float(err.max()), float(np.abs(r).max()))
    return dq, dk, dv


@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("D, dtype", [(64, wl.F16), (128, wl.BF16), (64, wl.BF16), (128, wl.F16)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L, vl", [(200, [200, 0]), (129, [77, 129]), (64, None)])
def test_bwd_matches_oracle(D, dtype, causal, L, vl, impl):
    run_case(2, 4, 2, L, D, dtype, causal, vl, seed=L + D, impl=impl)


@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("Hq, Hkv", [(8, 1), (8, 8)])
def test_bwd_medium_gqa_mqa(Hq, Hkv, impl):
    run_case(1, Hq, Hkv, 512, 128, wl.BF16, True, None, seed=512 + Hkv, impl=impl)


@pytest.mark.parametrize("L, causal, vl", [(1000, True, [1000, 613]), (1280, False, [1280, 257]),
                                           (2048, True, None)])
def test_bwd_tc_many_tiles(L, causal, vl):
    """Many key and query tiles, ragged last tile, padding cutting a tile,
    a GQA group of 4."""
    B = 1 if vl is None else 2
    run_case(B, 4, 1, L, 128, wl.BF16, causal, vl, seed=L, impl="tc")


def test_bwd_tc_deterministic_and_close_to_simt():
    """C4's head shapes with a shorter L: two runs of attn_bwd give identical
    bits (no atomics), and they agree with the fp32 SIMT backward within the
    operand-rounding scale (a cross-check between the two CUDA paths)."""
    B, Hq, Hkv, L, D = 2, 32, 8, 1024, 128
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=404)
    do = torch.randn(B, Hq, L, D, generator=torch.Generator().manual_seed(405)).to(torch.bfloat16)
    dev = torch.device("cuda")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    sm = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True, sm_scale=sm)
    a = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=sm)
    b = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=sm)
    s = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=sm, impl="simt")
    assert attn.status() == (attn.ATTN_OK, 0)
    for x, y, z in zip(a, b, s):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
        diff = (x.float() - z.float()).abs()
        assert float(diff.max()) <= 0.02 * float(z.float().abs().max()), float(diff.max())


@pytest.mark.parametrize("name", ["C4", "C2", "C3"])
def test_bwd_full_size_sampled_rows(name):
    """The workload's full shapes and masks: attn_bwd against the oracle on
    sampled rows -- dQ rows on tile boundaries of several heads and batches,
    dK/dV rows of two K/V heads (the first and the last) -- from
    oracle.attn_bwd_rows_f64.  Bound: the same terms as run_case, with the
    per-element sums over keys / queries bounded through the oracle's row
    magnitudes and the largest |k|, |q|, |dO|:
        dQ: sm_scale max|k| (u w_i + u sum_j |dS_ij| + a n_i)
        dK: sm_scale max|q| (u sum_i P_ij w_i + u sum_i |dS_ij| + a n_j)
        dV: max|dO| (u sum_i P_ij + a n_j)
    plus 1e-2 |g| and 1e-4 max|g| (w_i = sum_d |dO_id O_id|)."""
    w = wl.WORKLOADS[name]
    q, k, v, vl = wl.workload_inputs(w)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 100)).to(q.dtype)
    dev = torch.device("cuda")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    vld = None if vl is None else vl.to(dev)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, valid_len=vld)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=w.causal, sm_scale=w.sm_scale,
                               valid_len=vld)
    assert attn.status() == (attn.ATTN_OK, 0)
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    rng = np.random.default_rng(w.seed)
    rows = sorted({0, 1, 127, 128, 255, L // 2, L - 129, L - 1} | set(rng.integers(0, L, 6).tolist()))
    heads = sorted({0, 5 % Hq, Hq - 1, Hq // 2 + 3})
    qr = np.array([(b * Hq + h) * L + i for b in sorted({0, B - 1}) for h in heads for i in rows])
    kr = np.array([(z * L) + j for z in (0, B * Hkv - 1) for j in rows])
    f = lambda t: t.double().numpy()
    vl_np = None if vl is None else vl.numpy()
    r_dq, qm, r_dk, r_dv, km = oracle.attn_bwd_rows_f64(f(q), f(k), f(v), f(do), w.sm_scale,
                                                        causal=w.causal, valid_len=vl_np,
                                                        q_rows=qr, k_rows=kr)
    u = 2.0 ** -8 if w.dtype == wl.BF16 else 2.0 ** -11
    a = 0.0 if w.dtype == wl.BF16 else 2.0 ** -25
    mq, mk, mdo = (float(t.float().abs().max()) for t in (q, k, do))
    sm = w.sm_scale
    extra = {
        "dq": sm * mk * (u * qm[:, 1] + u * qm[:, 0] + a * qm[:, 2]),
        "dk": sm * mq * (u * km[:, 2] + u * km[:, 0] + a * km[:, 3]),
        "dv": mdo * (u * km[:, 1] + a * km[:, 3]),
    }
    got = {"dq": dq.reshape(-1, D)[torch.from_numpy(qr).to(dev)],
           "dk": dk.reshape(-1, D)[torch.from_numpy(kr).to(dev)],
           "dv": dv.reshape(-1, D)[torch.from_numpy(kr).to(dev)]}
    for gname, ref in (("dq", r_dq), ("dk", r_dk), ("dv", r_dv)):
        g = got[gname].float().cpu().double().numpy()
        err = np.abs(g - ref)
        bound = 1e-2 * np.abs(ref) + 1e-4 * np.abs(ref).max() + extra[gname][:, None]
        assert np.all(err <= bound), "%s %s: %d of %d elements out of tolerance (max err %g, ref max %g)" % (
            name, gname, int((err > bound).sum()), err.size, float(err.max()), float(np.abs(ref).max()))
    if vl is not None and int(vl[0]) == 0:  # keys of an empty batch: exact zeros
        assert float(dk[0].abs().max()) == 0.0 and float(dv[0].abs().max()) == 0.0


@pytest.mark.parametrize("D, dtype", [(16, wl.BF16), (32, wl.F16), (32, wl.BF16), (16, wl.F16)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_tc_small_head_dims(D, dtype, causal):
    """D = 16 and 32 (the D = 64 kernels on zero-filled columns)."""
    run_case(2, 4, 2, 200, D, dtype, causal, [200, 0] if causal else [131, 200], seed=D + 7,
             impl="tc")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_bwd_tc_writes_only_its_outputs(D):
    """dQ, dK, dV written through the C ABI into buffers with guard regions on
    both sides (ragged L, an empty batch): every guard element keeps its
    sentinel, and the outputs match the binding's."""
    B, Hq, Hkv, L = 2, 4, 2, 173
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=D, valid_len=[173, 0])
    do = torch.randn(B, Hq, L, D, generator=torch.Generator().manual_seed(D + 1)).to(torch.bfloat16)
    dev = torch.device("cuda")
    qd, kd, vd, dod, vld = q.to(dev), k.to(dev), v.to(dev), do.to(dev), vl.to(dev)
    sm = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True, sm_scale=sm, valid_len=vld)
    ref = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=sm, valid_len=vld)
    guard = 4096
    bufs = []
    for t in ref:
        n = t.numel()
        bufs.append(torch.full((n + 2 * guard,), 0x7BCD, dtype=torch.int16, device=dev))
    views = [b[guard:guard + t.numel()] for b, t in zip(bufs, ref)]
    lib = attn.load()
    st = lib.attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), dod.data_ptr(),
                      lse.data_ptr(), views[0].data_ptr(), views[1].data_ptr(), views[2].data_ptr(),
                      B, Hq, Hkv, L, D, sm, 1, vld.data_ptr(), attn.ATTN_BF16, None)
    assert st == attn.ATTN_OK
    assert attn.status() == (attn.ATTN_OK, 0)
    for b, vw, t in zip(bufs, views, ref):
        hb = b.cpu()
        assert bool((hb[:guard] == 0x7BCD).all()) and bool((hb[guard + t.numel():] == 0x7BCD).all())
        assert torch.equal(vw, t.contiguous().view(torch.int16).reshape(-1))


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("layout", ["blhd", "packed_qkv"])
def test_bwd_strided_matches_contiguous(D, layout):
    """attn_bwd on strided views -- [B, L, H, D] tensors, or Q, K, V as slices
    of one packed [B, L, Hq + 2 Hkv, D] tensor -- with dQ, dK, dV written
    into [B, L, H, D + 8] buffers (padded rows): the gradients are identical
    bit for bit to the contiguous call's, and the padding keeps its
    sentinel."""
    B, Hq, Hkv, L = 2, 8, 2, 300
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, wl.BF16, seed=D + 3, valid_len=[300, 111])
    do = torch.randn(B, Hq, L, D, generator=torch.Generator().manual_seed(D + 4)).to(torch.bfloat16)
    dev = torch.device("cuda")
    qd, kd, vd, dod, vld = q.to(dev), k.to(dev), v.to(dev), do.to(dev), vl.to(dev)
    sm = 1.0 / math.sqrt(D)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True, sm_scale=sm, valid_len=vld)
    ref = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=sm, valid_len=vld)
    blhd = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)
    if layout == "blhd":
        qs, ks, vs = blhd(qd), blhd(kd), blhd(vd)
    else:
        packed = torch.cat([qd.transpose(1, 2), kd.transpose(1, 2), vd.transpose(1, 2)], dim=2).contiguous()
        qs = packed[:, :, :Hq].transpose(1, 2)
        ks = packed[:, :, Hq:Hq + Hkv].transpose(1, 2)
        vs = packed[:, :, Hq + Hkv:].transpose(1, 2)
    os_, dos = blhd(o), blhd(dod)
    sentinel = -12345.0
    bufs = [torch.full((B, L, H, D + 8), sentinel, dtype=torch.bfloat16, device=dev)
            for H in (Hq, Hkv, Hkv)]
    outs = [b[..., :D].transpose(1, 2) for b in bufs]
    got = attn.attn_bwd(qs, ks, vs, os_, lse, dos, causal=True, sm_scale=sm, valid_len=vld,
                        dq=outs[0], dk=outs[1], dv=outs[2])
    assert attn.status() == (attn.ATTN_OK, 0)
    for g, r, b in zip(got, ref, bufs):
        assert torch.equal(g.contiguous().view(torch.int16), r.contiguous().view(torch.int16))
        assert bool((b[..., D:] == sentinel).all())


@pytest.mark.parametrize("Lq, Lk, causal, vl", [(200, 333, True, [333, 77]), (333, 200, True, None),
                                                (129, 260, False, [260, 3]), (300, 129, False, None),
                                                (100, 400, True, [400, 0])])
@pytest.mark.parametrize("D, dtype", [(128, wl.BF16), (64, wl.F16)])
def test_bwd_tc_query_and_key_lengths(Lq, Lk, causal, vl, D, dtype):
    """Lq != Lk (the forward's top-left causal reading): fewer queries than keys
    (keys after the last query get zero gradients under causality), more
    queries than keys (late queries see every key), padding, an empty batch."""
    run_case(2, 4, 2, Lq, D, dtype, causal, vl, seed=Lq + Lk + D, impl="tc", Lk=Lk)


def make_mask(kind, B, Lq, Lk, rng):
    if kind.startswith("random"):
        m = rng.random((B, Lq, Lk)) < float(kind.split("_")[1])
    elif kind == "blocks":  # whole 128 x 128 tiles kept or removed, plus a ragged edge
        tiles = rng.random((B, (Lq + 127) // 128, (Lk + 127) // 128)) < 0.5
        tiles[:, :, 0] = True
        m = np.repeat(np.repeat(tiles, 128, axis=1), 128, axis=2)[:, :Lq, :Lk].copy()
        m[:, :, Lk // 3: Lk // 3 + 5] = False
    elif kind == "empty_rows":  # fully masked rows and a fully masked batch
        m = rng.random((B, Lq, Lk)) < 0.4
        m[0, 5:140, :] = False
        m[-1] = False
    elif kind == "shared":  # one [Lq, Lk] mask for every batch
        m = rng.random((Lq, Lk)) < 0.3
    else:
        raise ValueError(kind)
    return m.astype(np.uint8)


@pytest.mark.parametrize("kind", ["random_0.5", "random_0.05", "blocks", "empty_rows", "shared"])
@pytest.mark.parametrize("D, dtype", [(128, wl.BF16), (64, wl.F16), (32, wl.BF16)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_masked_matches_oracle(kind, D, dtype, causal):
    """The explicit mask of attn_fwd_masked in the backward (attn_bwd_masked),
    intersected with causal and padding, Lq != Lk."""
    B, Lq, Lk = 2, 300, 400
    rng = np.random.default_rng(zlib.crc32(("%s/%d/%d" % (kind, D, causal)).encode()) % 1000)
    mk = make_mask(kind, B, Lq, Lk, rng)
    run_case(B, 4, 2, Lq, D, dtype, causal, [400, 233], seed=900 + D, impl="tc", Lk=Lk, mask=mk)


def test_bwd_restated_causal_mask_bit_identical():
    """C4's shapes: a shared tril mask with causal=False gives the gradients of
    causal=True bit for bit (the masked pairs get P = 0 exactly, and the
    extra tiles add exact zeros)."""
    w = wl.WORKLOADS["C4"]
    q, k, v, _ = wl.workload_inputs(w)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 100)).to(q.dtype)
    dev = torch.device("cuda")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = attn.attn_fwd(qd, kd, vd, causal=True, sm_scale=w.sm_scale)
    ref = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=w.sm_scale)
    tril = torch.tril(torch.ones(w.L, w.L, dtype=torch.bool, device=dev))
    got = attn.attn_bwd(qd, kd, vd, o, lse, dod, sm_scale=w.sm_scale, mask=tril)
    assert attn.status() == (attn.ATTN_OK, 0)
    for g, r in zip(got, ref):
        assert torch.equal(g.view(torch.int16), r.view(torch.int16))


def test_bwd_masked_full_size_sampled_rows():
    """C4's shapes with the block-sparse masks of the forward's test (a local
    band plus the first keys, random partial tiles; per batch), causal:
    sampled dQ rows and the dK/dV rows of two K/V heads against the oracle,
    with the magnitude-based bound of test_bwd_full_size_sampled_rows."""
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
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(w.seed + 7)).to(q.dtype)
    dev = torch.device("cuda")
    qd, kd, vd, dod, md = q.to(dev), k.to(dev), v.to(dev), do.to(dev), torch.from_numpy(mk).to(dev)
    o, lse = attn.attn_fwd_strided(qd, kd, vd, causal=True, sm_scale=w.sm_scale, mask=md)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, lse, dod, causal=True, sm_scale=w.sm_scale, mask=md)
    assert attn.status() == (attn.ATTN_OK, 0)
    B, Hq, _, D = q.shape
    Hkv = k.shape[1]
    rows = sorted({0, 1, 127, 128, 511, 512, 2047, 2048, L - 1} | set(rng.integers(0, L, 6).tolist()))
    qr = np.array([(b * Hq + h) * L + r for b in (0, 1) for h in (0, 5, 31) for r in rows])
    kr = np.array([z * L + r for z in (0, Hkv + 3) for r in rows])  # batch 0 head 0, batch 1 head 3
    f = lambda t: t.double().numpy()
    r_dq, qm, r_dk, r_dv, km = oracle.attn_bwd_rows_f64(f(q), f(k), f(v), f(do), w.sm_scale,
                                                        causal=True, q_rows=qr, k_rows=kr, mask=mk)
    u = 2.0 ** -8
    mq, mkk, mdo = (float(t.float().abs().max()) for t in (q, k, do))
    sm = w.sm_scale
    extra = {"dq": sm * mkk * (u * qm[:, 1] + u * qm[:, 0]),
             "dk": sm * mq * (u * km[:, 2] + u * km[:, 0]),
             "dv": mdo * u * km[:, 1]}
    got = {"dq": dq.reshape(-1, D)[torch.from_numpy(qr).to(dev)],
           "dk": dk.reshape(-1, D)[torch.from_numpy(kr).to(dev)],
           "dv": dv.reshape(-1, D)[torch.from_numpy(kr).to(dev)]}
    for gname, ref in (("dq", r_dq), ("dk", r_dk), ("dv", r_dv)):
        g = got[gname].float().cpu().double().numpy()
        err = np.abs(g - ref)
        bound = 1e-2 * np.abs(ref) + 1e-4 * np.abs(ref).max() + extra[gname][:, None]
        assert np.all(err <= bound), "%s: %d of %d out of tolerance (max err %g, ref max %g)" % (
            gname, int((err > bound).sum()), err.size, float(err.max()), float(np.abs(ref).max()))
