"""GPU parity of attn_fwd_strided: strided operands read and written in place,
and query length Lq != key length Lk.

* Small shapes, compared in full with the float64 oracle (same tolerance as
  every parity test): [B, L, H, D] storage, slices of a packed QKV tensor,
  rows padded beyond D, O written into a strided view; Lq != Lk with every
  mask, GQA/MQA, D in {16, 32, 64, 128}, both dtypes.
* Guard elements around and between O's rows keep their sentinel.
* Full-size workloads (C3 and C4 shapes) in strided layouts give results
  identical, bit for bit, to attn_fwd on contiguous copies (same kernel, same
  arithmetic order); Lq != Lk at full size is compared with the oracle on
  sampled rows.
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
SENTINEL16 = 0x7BCD  # a large finite fp16/bf16 bit pattern no result here can have


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


def oracle_ref(q, k, v, dtype, sm, causal, vl, rows=None):
    return oracle.attn_fwd_bits(wl.bits(q), wl.bits(k), wl.bits(v), wl.dtype_code(dtype), sm,
                                causal=causal, valid_len=None if vl is None else vl.numpy(),
                                rows=rows)


def place(x, layout, dev, pad=8):
    """A device view of the [B, H, L, D] CPU tensor x in the given storage layout."""
    B, H, L, D = x.shape
    if layout == "bhld":
        return x.to(dev)
    if layout == "blhd":
        return x.transpose(1, 2).contiguous().to(dev).transpose(1, 2)
    if layout == "row_pad":  # rows D + pad elements apart
        buf = torch.zeros(B, H, L, D + pad, dtype=x.dtype)
        buf[..., :D] = x
        return buf.to(dev)[..., :D]
    raise ValueError(layout)


def packed_qkv(q, k, v, dev):
    """Views of one [B, L, Hq + 2*Hkv, D] device tensor holding Q, K and V."""
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    buf = torch.cat([q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)], dim=2).contiguous()
    buf = buf.to(dev)
    return (buf[:, :, :Hq].transpose(1, 2), buf[:, :, Hq:Hq + Hkv].transpose(1, 2),
            buf[:, :, Hq + Hkv:].transpose(1, 2))


def run(qd, kd, vd, causal, vl, sm, out=None):
    dev = qd.device
    o, lse = attn.attn_fwd_strided(qd, kd, vd, causal=causal, sm_scale=sm,
                                   valid_len=None if vl is None else vl.to(dev), out=out)
    st, code = attn.status()
    assert st == attn.ATTN_OK, "device status %d (code %#x)" % (st, code)
    return o, lse


LAYOUTS = ["bhld", "blhd", "row_pad", "packed"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_layouts_full_compare(layout, D, causal):
    dtype = wl.BF16 if D in (32, 128) else wl.F16
    B, Hq, Hkv, L = 2, 4, 2, 300
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=500 + D, valid_len=[300, 131])
    dev = torch.device("cuda")
    if layout == "packed":
        qd, kd, vd = packed_qkv(q, k, v, dev)
    else:
        qd, kd, vd = place(q, layout, dev), place(k, layout, dev), place(v, layout, dev)
    # O in [B, L, H, D] storage for the packed layout, like Q otherwise
    out = torch.empty(B, L, Hq, D, dtype=q.dtype, device=dev).transpose(1, 2) \
        if layout == "packed" else None
    sm = 1.0 / math.sqrt(D)
    o, lse = run(qd, kd, vd, causal, vl, sm, out=out)
    if out is not None:
        assert o.data_ptr() == out.data_ptr()
    o_ref, lse_ref = oracle_ref(q, k, v, dtype, sm, causal, vl)
    check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
          "%s D%d causal=%s" % (layout, D, causal))


@pytest.mark.parametrize("Lq, Lk", [(300, 700), (700, 300), (1, 513), (129, 1), (128, 384),
                                    (515, 260)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D, dtype, Hq, Hkv", [(128, wl.BF16, 4, 2), (64, wl.F16, 4, 1),
                                               (32, wl.BF16, 2, 2)])
def test_lengths_full_compare(Lq, Lk, causal, D, dtype, Hq, Hkv):
    B = 3
    vl = [Lk, max(0, Lk // 2 - 3), 0]
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, Lq, D, dtype, seed=Lq + 7 * Lk, valid_len=vl,
                                   Lk=Lk)
    dev = torch.device("cuda")
    sm = 1.0 / math.sqrt(D)
    for layout in ("bhld", "blhd"):
        o, lse = run(place(q, layout, dev), place(k, layout, dev), place(v, layout, dev), causal,
                     vl_t, sm)
        o_ref, lse_ref = oracle_ref(q, k, v, dtype, sm, causal, vl_t)
        check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
              "Lq%d Lk%d D%d %s causal=%s" % (Lq, Lk, D, layout, causal))
        assert np.all(o[2].float().cpu().numpy() == 0.0)  # batch 2 sees no key


@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_writes_stay_inside_strided_o(D):
    """O viewed inside a larger buffer ([B, L, H, D + 8] storage, guard rows
    before and after): every element outside the view keeps its sentinel,
    also for the fully masked batch written by the kernel's zero-fill path."""
    dtype = wl.BF16 if D in (32, 128) else wl.F16
    B, Hq, Hkv, L, pad, guard = 3, 4, 2, 300, 8, 64
    q, k, v, vl = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=600 + D, valid_len=[300, 0, 77])
    dev = torch.device("cuda")
    tdt = q.dtype
    n_row = Hq * (D + pad)
    buf = torch.full((guard * 2 + B * L * n_row,), SENTINEL16, dtype=torch.int16, device=dev)
    inner = buf[guard:guard + B * L * n_row].view(tdt).view(B, L, Hq, D + pad)
    out = inner[..., :D].transpose(1, 2)  # [B, Hq, L, D] view: rows Hq*(D+pad) apart
    sm = 1.0 / math.sqrt(D)
    for causal in (False, True):
        buf.fill_(SENTINEL16)
        o, lse = run(q.to(dev).transpose(1, 2).contiguous().transpose(1, 2), k.to(dev), v.to(dev),
                     causal, vl, sm, out=out)
        allb = buf.cpu()
        assert bool((allb[:guard] == SENTINEL16).all()), "written before O's storage"
        assert bool((allb[guard + B * L * n_row:] == SENTINEL16).all()), "written after O's storage"
        pad_cols = allb[guard:guard + B * L * n_row].view(B, L, Hq, D + pad)[..., D:]
        assert bool((pad_cols == SENTINEL16).all()), "written into the gaps between O's rows"
        o_ref, lse_ref = oracle_ref(q, k, v, dtype, sm, causal, vl)
        check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref,
              "strided O D%d causal=%s" % (D, causal))


def _same(a, b):
    return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))


@pytest.mark.parametrize("name, layout", [("C4", "blhd"), ("C3", "packed"), ("C5", "row_pad"),
                                          ("C2", "blhd")])
def test_full_size_strided_equals_contiguous(name, layout):
    """The strided path on a full-size workload gives exactly attn_fwd's
    results on contiguous copies of the same values."""
    w = wl.WORKLOADS[name]
    q, k, v, vl = wl.workload_inputs(w)
    dev = torch.device("cuda")
    vld = None if vl is None else vl.to(dev)
    o_c, lse_c = attn.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=w.causal,
                               sm_scale=w.sm_scale, valid_len=vld)
    assert attn.status() == (attn.ATTN_OK, 0)
    if layout == "packed":
        qd, kd, vd = packed_qkv(q, k, v, dev)
    else:
        qd, kd, vd = place(q, layout, dev), place(k, layout, dev), place(v, layout, dev)
    out = place(torch.zeros_like(q), layout if layout != "packed" else "blhd", dev)
    o_s, lse_s = attn.attn_fwd_strided(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale,
                                       valid_len=vld, out=out)
    assert attn.status() == (attn.ATTN_OK, 0)
    assert _same(o_s, o_c), "%s %s: O differs from the contiguous call" % (name, layout)
    assert torch.equal(lse_s, lse_c), "%s %s: LSE differs from the contiguous call" % (name, layout)


@pytest.mark.parametrize("Lq, Lk, causal, vl", [
    (2048, 6144, False, [6144, 3001]),
    (6144, 2048, True, [2048, 1500]),
    (1, 8192, False, [8192, 4097]),
])
def test_lengths_full_size_sampled_rows(Lq, Lk, causal, vl):
    B, Hq, Hkv, D, dtype = 2, 16, 4, 128, wl.BF16
    q, k, v, vl_t = wl.make_inputs(B, Hq, Hkv, Lq, D, dtype, seed=Lq + Lk, valid_len=vl, Lk=Lk)
    dev = torch.device("cuda")
    sm = 1.0 / math.sqrt(D)
    o, lse = run(place(q, "blhd", dev), place(k, "blhd", dev), place(v, "blhd", dev), causal,
                 vl_t, sm)
    rng = np.random.default_rng(Lq)
    per_head = sorted({0, Lq - 1} | {i for t in range(0, Lq, 128) for i in (t, t + 127)
                                     if i < Lq} | set(rng.integers(0, Lq, 16).tolist()))
    heads = [0, 3, Hq - 1, Hq + 5, 2 * Hq - 1]
    rows = np.array([h * Lq + i for h in heads for i in per_head], dtype=np.int64)
    o_ref, lse_ref = oracle_ref(q, k, v, dtype, sm, causal, vl_t, rows=rows)
    o_all = o.contiguous().float().cpu().numpy().reshape(-1, D)
    check(o_all[rows], lse.cpu().numpy().reshape(-1)[rows], o_ref, lse_ref,
          "Lq%d Lk%d causal=%s" % (Lq, Lk, causal))


def test_lq_one_decode_step_matches_last_row_of_square_problem():
    """One query row at position 0 of a long cache (non-causal) equals row 0 of
    the square problem whose Q rows are all that row -- a decode step."""
    B, Hq, Hkv, L, D, dtype = 2, 8, 2, 1000, 128, wl.BF16
    q, k, v, _ = wl.make_inputs(B, Hq, Hkv, L, D, dtype, seed=77)
    dev = torch.device("cuda")
    q1 = q[:, :, :1].contiguous()
    o1, l1 = run(q1.to(dev), k.to(dev), v.to(dev), False, None, 0.088)
    qs = q1.expand(B, Hq, L, D).contiguous()
    os_, ls = attn.attn_fwd(qs.to(dev), k.to(dev), v.to(dev), sm_scale=0.088)
    assert attn.status() == (attn.ATTN_OK, 0)
    assert _same(o1[:, :, 0], os_[:, :, 0])
    assert torch.equal(l1.view(B, Hq), ls.view(B, Hq, L)[:, :, 0])
