"""ctypes binding of libattn.so: argument marshalling only.

Every computation happens inside the CUDA library.  PyTorch is used here to
hand over device pointers and streams, and to allocate outputs when the caller
does not pass them.  A missing library raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

ATTN_F16 = 0
ATTN_BF16 = 1

STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_ALIGN", 3: "ATTN_ERR_SHAPE",
    4: "ATTN_ERR_HEADS", 5: "ATTN_ERR_HEADDIM", 6: "ATTN_ERR_DTYPE", 7: "ATTN_ERR_SCALE",
    8: "ATTN_ERR_ARCH", 9: "ATTN_ERR_CUDA", 10: "ATTN_ERR_TIMEOUT", 11: "ATTN_ERR_VALID_LEN",
    12: "ATTN_ERR_ARG", 13: "ATTN_ERR_SCRATCH", 14: "ATTN_ERR_STRIDE", 15: "ATTN_ERR_WORKSPACE",
}
ATTN_OK = 0


class AttnError(RuntimeError):
    """A non-zero attn_status_t returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, "status %d" % self.status)
        msg = "%s: %s (%s)" % (where, name, strerror(self.status))
        if self.status == 9:
            msg += " [cudaError %d]" % last_cuda_error()
        super().__init__(msg)


class Caps(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "supported", "block_m", "q_tiles_per_cta", "block_n", "kv_stages", "threads",
        "smem_bytes", "tmem_cols", "num_sms", "lse_natural_log")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Strides(ctypes.Structure):
    """attn_strides_t: element strides of batch, head and sequence position."""
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("seq", ctypes.c_int64)]


class Chunk(ctypes.Structure):
    """attn_chunk_t: flattened query heads [q_head0, q_head0 + q_heads), the K/V
    heads [kv_head0, kv_head0 + kv_heads) it copies in, its attention calls."""
    _fields_ = [(n, ctypes.c_int) for n in ("q_head0", "q_heads", "kv_head0", "kv_heads",
                                            "calls")]

    def as_tuple(self):
        return (self.q_head0, self.q_heads, self.kv_head0, self.kv_heads, self.calls)


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libattn.so (built in-tree by ``build.build_library``).  Raises when absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    "libattn.so is not built (%s); build it with "
                    "attention_forward_attn_gb300.build.build_library()" % path)
            lib = ctypes.CDLL(path)
            p = ctypes.c_void_p
            i = ctypes.c_int
            fwd_args = [p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p, i, p]
            for name in ("attn_fwd", "attn_fwd_simt", "attn_fwd_noalloc", "attn_fwd_host"):
                fn = getattr(lib, name)
                fn.argtypes = fwd_args
                fn.restype = i
            sp = ctypes.POINTER(Strides)
            lib.attn_fwd_strided.argtypes = [p, sp, p, sp, p, sp, p, sp, p, i, i, i, i, i, i,
                                             ctypes.c_float, i, p, i, p]
            lib.attn_fwd_strided.restype = i
            i64 = ctypes.c_int64
            lib.attn_fwd_masked.argtypes = [p, sp, p, sp, p, sp, p, sp, p, i, i, i, i, i, i,
                                            ctypes.c_float, i, p, p, i64, i64, i, p]
            lib.attn_fwd_masked.restype = i
            lib.attn_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i, i, i, i, i, ctypes.c_float, i, p,
                                     i, p]
            lib.attn_bwd.restype = i
            lib.attn_bwd_simt.argtypes = lib.attn_bwd.argtypes
            lib.attn_bwd_simt.restype = i
            lib.attn_bwd_strided.argtypes = [p, sp, p, sp, p, sp, p, sp, p, sp, p, p, sp, p, sp, p,
                                             sp, i, i, i, i, i, i, ctypes.c_float, i, p, i, p]
            lib.attn_bwd_strided.restype = i
            lib.attn_bwd_masked.argtypes = lib.attn_bwd_strided.argtypes[:-2] + [p, i64, i64, i, p]
            lib.attn_bwd_masked.restype = i
            sz = ctypes.c_size_t
            lib.attn_fwd_ws.argtypes = fwd_args[:-1] + [p, sz, p]
            lib.attn_fwd_ws.restype = i
            lib.attn_fwd_masked_ws.argtypes = lib.attn_fwd_masked.argtypes[:-1] + [p, sz, p]
            lib.attn_fwd_masked_ws.restype = i
            lib.attn_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i, ctypes.POINTER(sz)]
            lib.attn_fwd_workspace_size.restype = i
            lib.attn_bwd_ws.argtypes = lib.attn_bwd.argtypes[:-1] + [p, sz, p]
            lib.attn_bwd_ws.restype = i
            lib.attn_bwd_masked_ws.argtypes = lib.attn_bwd_masked.argtypes[:-1] + [p, sz, p]
            lib.attn_bwd_masked_ws.restype = i
            lib.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i, ctypes.POINTER(sz)]
            lib.attn_bwd_workspace_size.restype = i
            lib.attn_workspace_pool_stats.argtypes = [i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
            lib.attn_workspace_pool_stats.restype = i
            lib.attn_fwd_f32.argtypes = [p, p, p, p, p, i, i, i, i, ctypes.c_float, i, p, i, p]
            lib.attn_fwd_f32.restype = i
            lib.attn_host_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(Chunk), i,
                                           ctypes.POINTER(ctypes.c_int)]
            lib.attn_host_plan.restype = i
            lib.attn_status.argtypes = [p, ctypes.POINTER(ctypes.c_int)]
            lib.attn_status.restype = i
            lib.attn_query.argtypes = [i, i, ctypes.POINTER(Caps)]
            lib.attn_query.restype = i
            lib.attn_strerror.argtypes = [i]
            lib.attn_strerror.restype = ctypes.c_char_p
            lib.attn_last_cuda_error.argtypes = []
            lib.attn_last_cuda_error.restype = i
            lib.attn_shutdown.argtypes = []
            lib.attn_shutdown.restype = None
            _lib = lib
    return _lib


def declared_symbols():
    """Function names declared in include/attn.h."""
    hdr = os.path.join(_build.INCLUDE, "attn.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def strerror(status: int) -> str:
    return load().attn_strerror(int(status)).decode()


def last_cuda_error() -> int:
    return int(load().attn_last_cuda_error())


# ------------------------------------------------------------------ raw C calls

def fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, Hq, Hkv, L, D, sm_scale, causal,
            valid_len_ptr, dtype, stream, simt=False, entry=None) -> int:
    """Call attn_fwd (or attn_fwd_simt, or the entry point named by ``entry``)
    with raw integer pointers; returns the status."""
    if entry is not None:
        fn = getattr(load(), entry)
    else:
        fn = load().attn_fwd_simt if simt else load().attn_fwd
    return int(fn(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(Hq), int(Hkv), int(L), int(D),
                  float(sm_scale), int(causal), valid_len_ptr, int(dtype), stream))


def _strides_arg(st):
    if st is None:
        return None
    return ctypes.byref(Strides(int(st[0]), int(st[1]), int(st[2])))


def fwd_strided_raw(q_ptr, q_strides, k_ptr, k_strides, v_ptr, v_strides, o_ptr, o_strides,
                    lse_ptr, B, Hq, Hkv, Lq, Lk, D, sm_scale, causal, valid_len_ptr, dtype,
                    stream) -> int:
    """Call attn_fwd_strided with raw integer pointers; each *_strides is a
    (batch, head, seq) element-stride triple or None (contiguous).  Returns
    the status."""
    return int(load().attn_fwd_strided(
        q_ptr, _strides_arg(q_strides), k_ptr, _strides_arg(k_strides), v_ptr,
        _strides_arg(v_strides), o_ptr, _strides_arg(o_strides), lse_ptr, int(B), int(Hq),
        int(Hkv), int(Lq), int(Lk), int(D), float(sm_scale), int(causal), valid_len_ptr,
        int(dtype), stream))


def fwd_masked_raw(q_ptr, q_strides, k_ptr, k_strides, v_ptr, v_strides, o_ptr, o_strides,
                   lse_ptr, B, Hq, Hkv, Lq, Lk, D, sm_scale, causal, valid_len_ptr, mask_ptr,
                   mask_batch_stride, mask_row_stride, dtype, stream) -> int:
    """Call attn_fwd_masked with raw integer pointers (strides as in
    fwd_strided_raw); returns the status."""
    return int(load().attn_fwd_masked(
        q_ptr, _strides_arg(q_strides), k_ptr, _strides_arg(k_strides), v_ptr,
        _strides_arg(v_strides), o_ptr, _strides_arg(o_strides), lse_ptr, int(B), int(Hq),
        int(Hkv), int(Lq), int(Lk), int(D), float(sm_scale), int(causal), valid_len_ptr, mask_ptr,
        int(mask_batch_stride), int(mask_row_stride), int(dtype), stream))


def status(stream=None):
    """attn_status: synchronise the stream, read and clear the device word -> (status, code)."""
    code = ctypes.c_int(0)
    st = int(load().attn_status(_stream_handle(stream), ctypes.byref(code)))
    return st, int(code.value)


def fwd_workspace_size(B, Hq, Hkv, Lq, Lk, D, dtype, mask_batches=0) -> int:
    """attn_fwd_workspace_size: device bytes one forward call needs."""
    n = ctypes.c_size_t(0)
    st = int(load().attn_fwd_workspace_size(int(B), int(Hq), int(Hkv), int(Lq), int(Lk), int(D),
                                            int(dtype), int(mask_batches), ctypes.byref(n)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_workspace_size")
    return int(n.value)


def bwd_workspace_size(B, Hq, Hkv, Lq, Lk, D, mask_batches=0) -> int:
    """attn_bwd_workspace_size: device bytes one tensor-core backward call needs
    on the current device."""
    n = ctypes.c_size_t(0)
    st = int(load().attn_bwd_workspace_size(int(B), int(Hq), int(Hkv), int(Lq), int(Lk), int(D),
                                            int(mask_batches), ctypes.byref(n)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_workspace_size")
    return int(n.value)


def pool_stats(reset_high_water=False):
    """attn_workspace_pool_stats -> (reserved bytes, high-water bytes) of the
    library's workspace pool on the current device."""
    r, h = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = int(load().attn_workspace_pool_stats(int(bool(reset_high_water)), ctypes.byref(r),
                                              ctypes.byref(h)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_workspace_pool_stats")
    return int(r.value), int(h.value)


def query(D: int, dtype: int = ATTN_BF16) -> dict:
    caps = Caps()
    st = int(load().attn_query(int(D), int(dtype), ctypes.byref(caps)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_query")
    return caps.as_dict()


def shutdown():
    load().attn_shutdown()


def host_plan(B: int, Hq: int, Hkv: int, L: int, D: int, dtype: int = ATTN_BF16):
    """attn_host_plan: the chunks attn_fwd_host queues, as
    (q_head0, q_heads, kv_head0, kv_heads, calls) tuples."""
    lib = load()
    n = ctypes.c_int(0)
    st = int(lib.attn_host_plan(int(B), int(Hq), int(Hkv), int(L), int(D), int(dtype), None, 0,
                                ctypes.byref(n)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_host_plan")
    arr = (Chunk * max(1, n.value))()
    st = int(lib.attn_host_plan(int(B), int(Hq), int(Hkv), int(L), int(D), int(dtype), arr,
                                n.value, ctypes.byref(n)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_host_plan")
    return [c.as_tuple() for c in arr[:n.value]]


# ------------------------------------------------------------------ torch-facing call

def _stream_handle(stream):
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _workspace(nbytes, like, stream, workspace):
    """(pointer, bytes) of the workspace for a *_ws call: the caller's uint8
    CUDA tensor, or a new one from torch's allocator (the library then
    allocates nothing for the call).  A tensor used on a stream other than
    torch's current one is recorded on it, so torch does not hand its memory
    out again before the call's kernels finish.  Returns (None, 0, None) when
    nbytes is 0; the third value keeps the tensor alive."""
    import torch
    if nbytes == 0:
        return None, 0, None
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=like.device)
        if stream is not None and not (isinstance(stream, int) and stream == 0):
            s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(
                int(stream))
            if s != torch.cuda.current_stream(like.device):
                workspace.record_stream(s)
    elif (not workspace.is_cuda or workspace.dtype != torch.uint8 or not workspace.is_contiguous()
          or workspace.numel() < nbytes):
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor of >= %d bytes" % nbytes)
    return workspace.data_ptr(), workspace.numel(), workspace


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise TypeError("q/k/v must be float16 or bfloat16, got %s" % t.dtype)


def attn_fwd(q, k, v, *, causal=False, sm_scale=None, valid_len=None, out=None, lse=None,
             return_lse=True, stream=None, simt=False, workspace=None):
    """Fused attention forward on CUDA tensors.

    q: [B, Hq, L, D]; k, v: [B, Hkv, L, D] (or [B, L, D] for MQA); fp16/bf16,
    contiguous, on the current CUDA device.  valid_len: int32 CUDA tensor [B]
    or None.  Returns (o, lse) with o like q and lse float32 [B*Hq, L]
    (lse is None when return_lse is False).  The call goes through
    attn_fwd_ws: its workspace (bf16: the fp16 copy of V) is ``workspace``, a
    uint8 CUDA tensor of at least fwd_workspace_size(...) bytes, or one torch
    allocates; workspace="pool" calls attn_fwd, which takes it from the
    library's own pool instead.
    """
    import torch
    if k.dim() == 3:
        k = k.unsqueeze(1)
    if v.dim() == 3:
        v = v.unsqueeze(1)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA tensor" % name)
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != L or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, L, D] matching q")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B * Hq, L), dtype=torch.float32, device=q.device)
    vl_ptr = None
    if valid_len is not None:
        if valid_len.dtype != torch.int32 or not valid_len.is_cuda or valid_len.numel() != B:
            raise ValueError("valid_len must be an int32 CUDA tensor of B elements")
        vl_ptr = valid_len.data_ptr()
    lse_ptr = lse.data_ptr() if (return_lse and lse is not None) else None
    if simt or (isinstance(workspace, str) and workspace == "pool"):
        st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                     B, Hq, Hkv, L, D, sm_scale, int(bool(causal)), vl_ptr, _dtype_code(q),
                     _stream_handle(stream), simt=simt)
        name = "attn_fwd_simt" if simt else "attn_fwd"
    else:
        need = fwd_workspace_size(B, Hq, Hkv, L, L, D, _dtype_code(q))
        ws_ptr, ws_bytes, _keep = _workspace(need, q, stream, workspace)
        st = int(load().attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse_ptr, B, Hq, Hkv, L, D, float(sm_scale),
                                    int(bool(causal)), vl_ptr, _dtype_code(q), ws_ptr, ws_bytes,
                                    _stream_handle(stream)))
        name = "attn_fwd_ws"
    if st != ATTN_OK:
        raise AttnError(st, name)
    return out, (lse if return_lse else None)


def attn_fwd_host(q, k, v, *, causal=False, sm_scale=None, valid_len=None, out=None, lse=None,
                  return_lse=True, stream=None, synchronize=True):
    """Fused attention forward on host (CPU) tensors through attn_fwd_host.

    Same shapes as attn_fwd, but q, k, v, valid_len and the outputs live in
    host memory; page-locked tensors (``pin_memory()``) let the library
    overlap the copies with the kernels.  Outputs that are not passed are
    allocated page-locked.  With ``synchronize`` the call waits for the
    stream before returning; otherwise o and lse are valid once the stream
    has synchronised.  Returns (o, lse).
    """
    import torch
    if k.dim() == 3:
        k = k.unsqueeze(1)
    if v.dim() == 3:
        v = v.unsqueeze(1)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous host tensor" % name)
    B, Hq, L, D = q.shape
    Hkv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != L or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, L, D] matching q")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    elif out.is_cuda or not out.is_contiguous() or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous host tensor like q")
    if return_lse and lse is None:
        lse = torch.empty((B * Hq, L), dtype=torch.float32, pin_memory=True)
    elif return_lse and (lse.is_cuda or not lse.is_contiguous() or lse.dtype != torch.float32
                         or lse.numel() != B * Hq * L):
        raise ValueError("lse must be a contiguous float32 host tensor of B*Hq*L elements")
    vl_ptr = None
    if valid_len is not None:
        if valid_len.dtype != torch.int32 or valid_len.is_cuda or valid_len.numel() != B:
            raise ValueError("valid_len must be an int32 host tensor of B elements")
        valid_len = valid_len.contiguous()
        vl_ptr = valid_len.data_ptr()
    handle = _stream_handle(stream)
    st = fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                 lse.data_ptr() if return_lse else None, B, Hq, Hkv, L, D, sm_scale,
                 int(bool(causal)), vl_ptr, _dtype_code(q), handle, entry="attn_fwd_host")
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_host")
    if synchronize:
        st, code = status(stream)
        if st != ATTN_OK:
            raise AttnError(st, "attn_fwd_host (device status %#x)" % code)
    return out, (lse if return_lse else None)


def attn_fwd_strided(q, k, v, *, causal=False, sm_scale=None, valid_len=None, out=None, lse=None,
                     return_lse=True, stream=None, mask=None, workspace=None):
    """Fused attention forward on strided CUDA tensors through attn_fwd_strided.

    q: [B, Hq, Lq, D]; k, v: [B, Hkv, Lk, D] -- any views whose last
    dimension is contiguous and whose other strides are multiples of 8
    elements, e.g. ``x.transpose(1, 2)`` of a [B, L, H, D] tensor or slices of
    a packed QKV tensor; no copy is made.  Lq may differ from Lk (the causal
    mask keeps key j <= query i).  out: optional [B, Hq, Lq, D] view to write
    (default: ``torch.empty_like(q)``).  mask: optional explicit boolean
    mask, a bool/uint8 CUDA tensor [B, Lq, Lk] or [Lq, Lk] (shared by every
    batch) whose last dimension is contiguous (attn_fwd_masked).  Returns
    (o, lse) with lse float32 [B*Hq, Lq].  The call goes through
    attn_fwd_masked_ws, with ``workspace`` as in attn_fwd (workspace="pool":
    attn_fwd_strided / attn_fwd_masked and the library's pool).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dim() != 4 or (t.shape[3] > 1 and t.stride(3) != 1):
            raise ValueError("%s must be a 4-D CUDA tensor with a contiguous last dimension"
                             % name)
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, Lk, D] matching q's B and D")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    elif (not out.is_cuda or out.shape != q.shape or out.dtype != q.dtype
          or (D > 1 and out.stride(3) != 1)):
        raise ValueError("out must be a CUDA tensor like q with a contiguous last dimension")
    if return_lse and lse is None:
        lse = torch.empty((B * Hq, Lq), dtype=torch.float32, device=q.device)
    vl_ptr = None
    if valid_len is not None:
        if valid_len.dtype != torch.int32 or not valid_len.is_cuda or valid_len.numel() != B:
            raise ValueError("valid_len must be an int32 CUDA tensor of B elements")
        vl_ptr = valid_len.data_ptr()
    msb = msr = 0
    if mask is not None:
        if mask.dtype not in (torch.bool, torch.uint8) or not mask.is_cuda:
            raise ValueError("mask must be a bool or uint8 CUDA tensor")
        if mask.dim() == 2:
            mask = mask.unsqueeze(0)
        if (mask.dim() != 3 or mask.shape[1:] != (Lq, Lk) or mask.shape[0] not in (1, B)
                or (Lk > 1 and mask.stride(2) != 1)):
            raise ValueError("mask must be [B, Lq, Lk] or [Lq, Lk] with a contiguous last dimension")
        msb = 0 if mask.shape[0] == 1 else mask.stride(0)
        msr = mask.stride(1)
    lse_ptr = lse.data_ptr() if return_lse else None
    if isinstance(workspace, str) and workspace == "pool":
        if mask is None:
            st = fwd_strided_raw(q.data_ptr(), q.stride()[:3], k.data_ptr(), k.stride()[:3],
                                 v.data_ptr(), v.stride()[:3], out.data_ptr(), out.stride()[:3],
                                 lse_ptr, B, Hq, Hkv, Lq, Lk, D, sm_scale, int(bool(causal)),
                                 vl_ptr, _dtype_code(q), _stream_handle(stream))
        else:
            st = fwd_masked_raw(q.data_ptr(), q.stride()[:3], k.data_ptr(), k.stride()[:3],
                                v.data_ptr(), v.stride()[:3], out.data_ptr(), out.stride()[:3],
                                lse_ptr, B, Hq, Hkv, Lq, Lk, D, sm_scale, int(bool(causal)),
                                vl_ptr, mask.data_ptr(), msb, msr, _dtype_code(q),
                                _stream_handle(stream))
        name = "attn_fwd_masked" if mask is not None else "attn_fwd_strided"
    else:
        mb = 0 if mask is None else (1 if msb == 0 else B)
        need = fwd_workspace_size(B, Hq, Hkv, Lq, Lk, D, _dtype_code(q), mb)
        ws_ptr, ws_bytes, _keep = _workspace(need, q, stream, workspace)
        st = int(load().attn_fwd_masked_ws(
            q.data_ptr(), _strides_arg(q.stride()[:3]), k.data_ptr(), _strides_arg(k.stride()[:3]),
            v.data_ptr(), _strides_arg(v.stride()[:3]), out.data_ptr(),
            _strides_arg(out.stride()[:3]), lse_ptr, int(B), int(Hq), int(Hkv), int(Lq), int(Lk),
            int(D), float(sm_scale), int(bool(causal)), vl_ptr,
            None if mask is None else mask.data_ptr(), int(msb), int(msr), _dtype_code(q),
            ws_ptr, ws_bytes, _stream_handle(stream)))
        name = "attn_fwd_masked_ws"
    if st != ATTN_OK:
        raise AttnError(st, name)
    return out, (lse if return_lse else None)


F32_KERNELS = {"naive": 0, "tiled_element": 1, "tiled_rowmax": 2}


def attn_fwd_f32(q, k, v, *, kernel="tiled_rowmax", causal=False, sm_scale=None, valid_len=None,
                 out=None, lse=None, return_lse=True, stream=None):
    """fp32 attention forward with one of the comparison kernels of
    attn_fwd_f32 ("naive", "tiled_element", "tiled_rowmax").  q, k, v: fp32
    contiguous CUDA tensors [B, H, L, D] (D 64 or 128).  Returns (o, lse)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError("%s must be a contiguous float32 CUDA tensor" % name)
    B, H, L, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("k and v must have q's shape [B, H, L, D]")
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B * H, L), dtype=torch.float32, device=q.device)
    vl_ptr = None
    if valid_len is not None:
        if valid_len.dtype != torch.int32 or not valid_len.is_cuda or valid_len.numel() != B:
            raise ValueError("valid_len must be an int32 CUDA tensor of B elements")
        vl_ptr = valid_len.data_ptr()
    st = int(load().attn_fwd_f32(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if return_lse else None, B, H, L, D,
                                 float(sm_scale), int(bool(causal)), vl_ptr, F32_KERNELS[kernel],
                                 _stream_handle(stream)))
    if st != ATTN_OK:
        raise AttnError(st, "attn_fwd_f32")
    return out, (lse if return_lse else None)


def attn_bwd(q, k, v, o, lse, do, *, causal=False, sm_scale=None, valid_len=None, stream=None,
             impl="tc", dq=None, dk=None, dv=None, mask=None, workspace=None):
    """Gradients (dq, dk, dv) of attn_fwd for the output gradient ``do``.

    impl="tc": attn_bwd_strided (tensor cores).  q, o, do: [B, Hq, Lq, D]; k, v:
    [B, Hkv, Lk, D] (Lq may differ from Lk) -- fp16 or bf16 CUDA views whose last dimension is
    contiguous and whose other strides are multiples of 8 elements (e.g.
    ``x.transpose(1, 2)`` of [B, L, H, D] tensors); dq, dk, dv: optional
    output views of the same shapes (default: new contiguous tensors).
    impl="simt": attn_bwd_simt (fp32 SIMT), contiguous tensors only.
    lse: the forward's [B*Hq, L] fp32 LSE.  mask: the forward's explicit
    boolean mask (a bool/uint8 CUDA tensor [B, Lq, Lk] or [Lq, Lk] with a
    contiguous last dimension; impl="tc" only, through attn_bwd_masked).
    impl="tc" goes through attn_bwd_masked_ws with ``workspace`` as in
    attn_fwd (a uint8 CUDA tensor of >= bwd_workspace_size(...) bytes, None:
    torch allocates one, "pool": the library's pool)."""
    import torch
    if impl not in ("tc", "simt"):
        raise ValueError("impl must be 'tc' or 'simt'")
    named = (("q", q), ("k", k), ("v", v), ("o", o), ("do", do))
    for name, t in named:
        if not t.is_cuda or t.dim() != 4 or (t.shape[3] > 1 and t.stride(3) != 1):
            raise ValueError("%s must be a 4-D CUDA tensor with a contiguous last dimension" % name)
        if impl == "simt" and not t.is_contiguous():
            raise ValueError("impl='simt' takes contiguous tensors (%s is not)" % name)
    B, Hq, L, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    if impl == "simt" and Lk != L:
        raise ValueError("impl='simt' takes equal query and key lengths")
    if sm_scale is None:
        sm_scale = 1.0 / float(D) ** 0.5
    dq = torch.empty_like(q, memory_format=torch.contiguous_format) if dq is None else dq
    dk = torch.empty_like(k, memory_format=torch.contiguous_format) if dk is None else dk
    dv = torch.empty_like(v, memory_format=torch.contiguous_format) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor shaped and typed like %s" % (name, name[1:]))
        if impl == "simt" and not t.is_contiguous():
            raise ValueError("impl='simt' takes contiguous tensors (%s is not)" % name)
    vl_ptr = None
    if valid_len is not None:
        vl_ptr = valid_len.data_ptr()
    lse = lse.contiguous()
    if mask is not None:
        if impl != "tc":
            raise ValueError("an explicit mask takes impl='tc'")
        if mask.dtype not in (torch.bool, torch.uint8) or not mask.is_cuda:
            raise ValueError("mask must be a bool or uint8 CUDA tensor")
        if mask.dim() == 2:
            mask = mask.unsqueeze(0)
        if (mask.dim() != 3 or mask.shape[1:] != (L, Lk) or mask.shape[0] not in (1, B)
                or (Lk > 1 and mask.stride(2) != 1)):
            raise ValueError("mask must be [B, Lq, Lk] or [Lq, Lk] with a contiguous last dimension")
    if impl == "tc":
        st3 = lambda t: _strides_arg((t.stride(0), t.stride(1), t.stride(2)))
        args = [q.data_ptr(), st3(q), k.data_ptr(), st3(k), v.data_ptr(), st3(v), o.data_ptr(),
                st3(o), do.data_ptr(), st3(do), lse.data_ptr(), dq.data_ptr(), st3(dq),
                dk.data_ptr(), st3(dk), dv.data_ptr(), st3(dv), B, Hq, Hkv, L, Lk, D,
                float(sm_scale), int(bool(causal)), vl_ptr]
        msb = 0 if (mask is None or mask.shape[0] == 1) else mask.stride(0)
        if isinstance(workspace, str) and workspace == "pool":
            if mask is None:
                name = "attn_bwd_strided"
                st = int(load().attn_bwd_strided(*args, _dtype_code(q), _stream_handle(stream)))
            else:
                name = "attn_bwd_masked"
                st = int(load().attn_bwd_masked(*args, mask.data_ptr(), msb, mask.stride(1),
                                                _dtype_code(q), _stream_handle(stream)))
        else:
            name = "attn_bwd_masked_ws"
            mb = 0 if mask is None else (1 if msb == 0 else B)
            need = bwd_workspace_size(B, Hq, Hkv, L, Lk, D, mb)
            ws_ptr, ws_bytes, _keep = _workspace(need, q, stream, workspace)
            st = int(load().attn_bwd_masked_ws(
                *args, None if mask is None else mask.data_ptr(), msb,
                0 if mask is None else mask.stride(1), _dtype_code(q), ws_ptr, ws_bytes,
                _stream_handle(stream)))
    else:
        name = "attn_bwd_simt"
        st = int(load().attn_bwd_simt(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                      dv.data_ptr(), B, Hq, Hkv, L, D, float(sm_scale),
                                      int(bool(causal)), vl_ptr, _dtype_code(q),
                                      _stream_handle(stream)))
    if st != ATTN_OK:
        raise AttnError(st, name)
    return dq, dk, dv
