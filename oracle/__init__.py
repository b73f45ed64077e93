"""Float64 CPU oracle for the fused multi-head attention forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` (including ``bench.py --impl reference``) may
import this package.  The product package ``attention_forward_attn_gb300`` never
imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, float64, OpenMP over query
rows).  It is the plain definition of masked multi-head attention
("masked multi head attention in CUDA", wzjinhao.cn, section 2.1) computed in
the three passes of that page's naive kernel (section 3.1): scores and row max,
then the exp-sum, then the weighted sum of V.  The masks follow section 2.2 of
that page and the "Causal Attention" / "GQA" variants of the Triton-CUDA
Attention page; the log-sum-exp is the natural-log form of
tiny_flash_attn_triton.py's stored ``m + log2(l)``.

Every function here is parity-pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so next to it (gcc, OpenMP, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i = ctypes.c_int
    i64 = ctypes.c_int64
    lib.oracle_attn_fwd_f64.argtypes = [p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double,
                                        i, p, p, i64, i64, p, i64, i]
    lib.oracle_attn_fwd_f64.restype = i
    lib.oracle_attn_fwd_u16.argtypes = [p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double,
                                        i, p, p, i64, i64, i, p, i64, i]
    lib.oracle_attn_fwd_u16.restype = i
    lib.oracle_attn_bwd_f64.argtypes = [p, p, p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double,
                                        i, p, p, i64, i64, i]
    lib.oracle_attn_bwd_f64.restype = i
    lib.oracle_attn_bwd_rows_f64.argtypes = [p, p, p, p, i, i, i, i, i, i, ctypes.c_double, i,
                                             p, p, i64, i64, p, i64, p, p, p, i64, p, p, p, i]
    lib.oracle_attn_bwd_rows_f64.restype = i
    lib.oracle_decode.argtypes = [p, p, i64, i]
    lib.oracle_decode.restype = i
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    """Threads the oracle's OpenMP region uses by default on this host."""
    return int(_load().oracle_max_threads())


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode raw fp16 (dtype=0) or bf16 (dtype=1) bit patterns to float64."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().oracle_decode(_ptr(bits), _ptr(out), bits.size, int(dtype))
    if rc != 0:
        raise ValueError("oracle_decode: bad dtype %r" % (dtype,))
    return out


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, L, D]")
    B, Hq, Lq, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k, v must be [B, Hkv, Lk, D] matching q's B and D")
    return B, Hq, k.shape[1], Lq, k.shape[2], D


def _valid(valid_len, B):
    if valid_len is None:
        return None
    vl = np.ascontiguousarray(valid_len, dtype=np.int32)
    if vl.shape != (B,):
        raise ValueError("valid_len must have shape [B]")
    return vl


def _mask(mask, B, Lq, Lk):
    """(array, batch_stride, row_stride) of an explicit mask: None, or a
    [B, Lq, Lk] / [1, Lq, Lk] / [Lq, Lk] array (nonzero keeps the position;
    the last two are shared by every batch)."""
    if mask is None:
        return None, 0, 0
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    if m.ndim == 2:
        m = m[None]
    if m.shape not in ((B, Lq, Lk), (1, Lq, Lk)):
        raise ValueError("mask must be [B, Lq, Lk], [1, Lq, Lk] or [Lq, Lk]")
    return m, (0 if m.shape[0] == 1 else Lq * Lk), Lk


def _rows(rows):
    if rows is None:
        return None, 0
    r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
    return r, r.size


def attn_fwd_f64(q, k, v, sm_scale, causal=False, valid_len=None, rows=None, threads=0,
                 _lib_override=None, mask=None):
    """Oracle on float64 inputs.

    q: [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D] (Lq = Lk is the pages' case; the
    causal mask compares absolute positions, key j visible to query i iff
    j <= i).  Returns (o, lse): o is [B, Hq, Lq, D] and lse [B*Hq, Lq] when
    ``rows`` is None, else o is [len(rows), D] and lse [len(rows)] for the
    flat row indices r = (b*Hq + h_q)*Lq + i.  ``mask``: optional explicit
    mask (see ``_mask``), intersected with the causal and padding masks.
    """
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    B, Hq, Hkv, Lq, Lk, D = _shapes(q, k, v)
    vl = _valid(valid_len, B)
    mk, msb, msr = _mask(mask, B, Lq, Lk)
    r, nr = _rows(rows)
    n_out = nr if r is not None else B * Hq * Lq
    o = np.empty((n_out, D), dtype=np.float64)
    lse = np.empty((n_out,), dtype=np.float64)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_attn_fwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                 Lq, Lk, D, float(sm_scale), int(bool(causal)), _ptr(vl),
                                 _ptr(mk), msb, msr, _ptr(r), nr, int(threads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_f64 failed with code %d" % rc)
    if r is None:
        return o.reshape(B, Hq, Lq, D), lse.reshape(B * Hq, Lq)
    return o, lse


def attn_fwd_bits(q_bits, k_bits, v_bits, dtype, sm_scale, causal=False, valid_len=None,
                  rows=None, threads=0, mask=None):
    """Oracle on raw fp16 (dtype=0) / bf16 (dtype=1) bit patterns (np.uint16 arrays).

    Same shapes and return convention as :func:`attn_fwd_f64`.
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    B, Hq, Hkv, Lq, Lk, D = _shapes(q, k, v)
    vl = _valid(valid_len, B)
    mk, msb, msr = _mask(mask, B, Lq, Lk)
    r, nr = _rows(rows)
    n_out = nr if r is not None else B * Hq * Lq
    o = np.empty((n_out, D), dtype=np.float64)
    lse = np.empty((n_out,), dtype=np.float64)
    rc = _load().oracle_attn_fwd_u16(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                     Lq, Lk, D, float(sm_scale), int(bool(causal)), _ptr(vl),
                                     _ptr(mk), msb, msr, int(dtype), _ptr(r), nr, int(threads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_u16 failed with code %d" % rc)
    if r is None:
        return o.reshape(B, Hq, Lq, D), lse.reshape(B * Hq, Lq)
    return o, lse


def attn_bwd_f64(q, k, v, do, sm_scale, causal=False, valid_len=None, threads=0,
                 _lib_override=None, mask=None):
    """Gradients (dq, dk, dv) of the attention forward for an output gradient
    ``do``, from the definition (see oracle_attn_bwd_f64).  q, do:
    [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D]; float64 results of the same shapes.
    mask: an explicit mask as for :func:`attn_fwd_f64`."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    do = np.ascontiguousarray(do, dtype=np.float64)
    B, Hq, Hkv, Lq, Lk, D = _shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must be shaped like q")
    vl = _valid(valid_len, B)
    mk, msb, msr = _mask(mask, B, Lq, Lk)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_attn_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                 B, Hq, Hkv, Lq, Lk, D, float(sm_scale), int(bool(causal)),
                                 _ptr(vl), _ptr(mk), msb, msr, int(threads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_f64 failed with code %d" % rc)
    return dq, dk, dv


def attn_bwd_rows_f64(q, k, v, do, sm_scale, causal=False, valid_len=None, q_rows=(),
                      k_rows=(), threads=0, _lib_override=None, mask=None):
    """Selected rows of :func:`attn_bwd_f64`'s gradients (see
    oracle_attn_bwd_rows_f64): dQ for flat query rows ``q_rows`` (index
    (b*Hq + h_q)*Lq + i) and dK, dV for flat key rows ``k_rows`` (index
    (b*Hkv + h_kv)*Lk + j).  Returns dq [n_q, D], qmag [n_q, 3] (sum_j |dS_ij|,
    sum_d |dO_id O_id|, visible keys), dk, dv [n_k, D], kmag [n_k, 4]
    (sum_i |dS_ij|, sum_i P_ij, sum_i P_ij sum_d |dO_id O_id|, visible queries)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    do = np.ascontiguousarray(do, dtype=np.float64)
    B, Hq, Hkv, Lq, Lk, D = _shapes(q, k, v)
    if do.shape != q.shape:
        raise ValueError("do must be shaped like q")
    vl = _valid(valid_len, B)
    mk, msb, msr = _mask(mask, B, Lq, Lk)
    qr = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int64).reshape(-1))
    kr = np.ascontiguousarray(np.asarray(k_rows, dtype=np.int64).reshape(-1))
    dq = np.empty((qr.size, D))
    qmag = np.empty((qr.size, 3))
    dk, dv = np.empty((kr.size, D)), np.empty((kr.size, D))
    kmag = np.empty((kr.size, 4))
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_attn_bwd_rows_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Lq, Lk, D,
                                      float(sm_scale), int(bool(causal)), _ptr(vl), _ptr(mk), msb,
                                      msr, _ptr(qr),
                                      qr.size, _ptr(dq), _ptr(qmag), _ptr(kr), kr.size, _ptr(dk),
                                      _ptr(dv), _ptr(kmag), int(threads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_rows_f64 failed with code %d" % rc)
    return dq, qmag, dk, dv, kmag


def load_variant(path: str):
    """Bind another build of attn_oracle.c (used by the pin tests to check that
    deliberately broken copies of the oracle fail the pins)."""
    return _bind(path)
