"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/attn.h declares, and rejects bad arguments before
touching a device."""
import ctypes
import os

import pytest

import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import binding

A16 = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def lib(cuda_lib_path):
    return attn.load()


def test_exports_every_declared_symbol(lib):
    names = attn.declared_symbols()
    assert {"attn_fwd", "attn_fwd_simt", "attn_status", "attn_query", "attn_strerror",
            "attn_shutdown", "attn_last_cuda_error"} <= set(names)
    for n in names:
        assert hasattr(lib, n), "libattn.so does not export %s" % n


def _call(**kw):
    args = dict(q_ptr=A16, k_ptr=A16, v_ptr=A16, o_ptr=A16, lse_ptr=None, B=1, Hq=2, Hkv=1, L=16,
                D=64, sm_scale=0.125, causal=0, valid_len_ptr=None, dtype=attn.ATTN_BF16,
                stream=None)
    args.update(kw)
    return attn.fwd_raw(**args)


@pytest.mark.parametrize("simt", [False, True])
@pytest.mark.parametrize("kw, expected", [
    (dict(dtype=7), "ATTN_ERR_DTYPE"),
    (dict(q_ptr=None), "ATTN_ERR_NULL"),
    (dict(k_ptr=None), "ATTN_ERR_NULL"),
    (dict(v_ptr=None), "ATTN_ERR_NULL"),
    (dict(o_ptr=None), "ATTN_ERR_NULL"),
    (dict(B=0), "ATTN_ERR_SHAPE"),
    (dict(Hq=0), "ATTN_ERR_SHAPE"),
    (dict(Hkv=0), "ATTN_ERR_SHAPE"),
    (dict(L=0), "ATTN_ERR_SHAPE"),
    (dict(L=-5), "ATTN_ERR_SHAPE"),
    (dict(B=1 << 12, Hq=1 << 10, Hkv=1, L=1 << 10), "ATTN_ERR_SHAPE"),
    (dict(D=96), "ATTN_ERR_HEADDIM"),
    (dict(D=0), "ATTN_ERR_HEADDIM"),
    (dict(D=8), "ATTN_ERR_HEADDIM"),
    (dict(D=48), "ATTN_ERR_HEADDIM"),
    (dict(D=256), "ATTN_ERR_HEADDIM"),
    (dict(Hq=3, Hkv=2), "ATTN_ERR_HEADS"),
    (dict(causal=2), "ATTN_ERR_ARG"),
    (dict(sm_scale=-1.0), "ATTN_ERR_SCALE"),
    (dict(sm_scale=float("nan")), "ATTN_ERR_SCALE"),
    (dict(sm_scale=float("inf")), "ATTN_ERR_SCALE"),
    (dict(q_ptr=A16 + 8), "ATTN_ERR_ALIGN"),
    (dict(k_ptr=A16 + 2), "ATTN_ERR_ALIGN"),
    (dict(v_ptr=A16 + 4), "ATTN_ERR_ALIGN"),
    (dict(o_ptr=A16 + 1), "ATTN_ERR_ALIGN"),
    (dict(lse_ptr=A16 + 2), "ATTN_ERR_ALIGN"),
    (dict(valid_len_ptr=A16 + 1), "ATTN_ERR_ALIGN"),
])
def test_invalid_arguments_rejected_on_host(lib, kw, expected, simt):
    st = _call(simt=simt, **kw)
    assert binding.STATUS_NAMES[st] == expected


def test_valid_arguments_need_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    st = _call()
    assert binding.STATUS_NAMES[st] in ("ATTN_ERR_CUDA", "ATTN_ERR_ARCH")


def test_query_static_fields(lib):
    # D = 16 and 32 run the D = 64 kernel (zero-filled columns)
    for D, stages in ((16, 12), (32, 12), (64, 12), (128, 5)):
        caps = attn.query(D, attn.ATTN_BF16)
        assert caps["block_m"] == 128 and caps["block_n"] == 128
        assert caps["q_tiles_per_cta"] == 1 and caps["kv_stages"] == stages
        assert caps["threads"] == 512 and caps["tmem_cols"] == 512
        assert 0 < caps["smem_bytes"] <= 232448
        assert caps["lse_natural_log"] == 1
    with pytest.raises(attn.AttnError):
        attn.query(80)
    with pytest.raises(attn.AttnError):
        attn.query(64, 5)
    assert lib.attn_query(64, 0, None) == 12  # NULL out-pointer: ATTN_ERR_ARG


def test_strerror_covers_every_status(lib):
    for code, name in binding.STATUS_NAMES.items():
        msg = attn.strerror(code)
        assert msg and msg != "unknown status", name
    assert attn.strerror(999) == "unknown status"


def test_status_and_shutdown_without_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    code = ctypes.c_int(-1)
    st = lib.attn_status(None, ctypes.byref(code))
    assert binding.STATUS_NAMES[st] == "ATTN_ERR_CUDA"
    assert code.value == 0
    attn.shutdown()  # harmless with nothing allocated


# ------------------------------------------------------------------ attn_fwd_strided

def _scall(**kw):
    args = dict(q_ptr=A16, q_strides=None, k_ptr=A16, k_strides=None, v_ptr=A16, v_strides=None,
                o_ptr=A16, o_strides=None, lse_ptr=None, B=2, Hq=4, Hkv=2, Lq=16, Lk=24, D=64,
                sm_scale=0.125, causal=0, valid_len_ptr=None, dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    return attn.fwd_strided_raw(**args)


BLHD_Q = (16 * 4 * 64, 64, 4 * 64)    # [B, Lq, Hq, D] storage seen as [B, Hq, Lq, D]
BLHD_KV = (24 * 2 * 64, 64, 2 * 64)


@pytest.mark.parametrize("kw, expected", [
    (dict(dtype=3), "ATTN_ERR_DTYPE"),
    (dict(v_ptr=None), "ATTN_ERR_NULL"),
    (dict(Lq=0), "ATTN_ERR_SHAPE"),
    (dict(Lk=0), "ATTN_ERR_SHAPE"),
    (dict(Lk=-3), "ATTN_ERR_SHAPE"),
    (dict(B=1 << 12, Hkv=1 << 10, Hq=1 << 10, Lq=1, Lk=1 << 10), "ATTN_ERR_SHAPE"),
    (dict(D=80), "ATTN_ERR_HEADDIM"),
    (dict(Hq=5), "ATTN_ERR_HEADS"),
    (dict(causal=-1), "ATTN_ERR_ARG"),
    (dict(sm_scale=-0.5), "ATTN_ERR_SCALE"),
    (dict(o_ptr=A16 + 2), "ATTN_ERR_ALIGN"),
    # strides: positive multiples of 8 elements below 2^39 where the extent is > 1
    (dict(q_strides=(16 * 4 * 64, 64, 68)), "ATTN_ERR_STRIDE"),
    (dict(k_strides=(0, 24 * 64, 64)), "ATTN_ERR_STRIDE"),
    (dict(v_strides=(2 * 24 * 64, -24 * 64, 64)), "ATTN_ERR_STRIDE"),
    (dict(k_strides=(1 << 39, 24 * 64, 64)), "ATTN_ERR_STRIDE"),
    (dict(v_strides=(2 * 24 * 64, 24 * 64, 4)), "ATTN_ERR_STRIDE"),
    # O's elements must not overlap: rows closer than D, heads inside a row
    (dict(o_strides=(4 * 16 * 64, 16 * 64, 32)), "ATTN_ERR_STRIDE"),
    (dict(o_strides=(4 * 16 * 64, 8, 16 * 64)), "ATTN_ERR_STRIDE"),
    (dict(o_strides=(64, 16 * 64, 64 * 4)), "ATTN_ERR_STRIDE"),
])
def test_strided_invalid_arguments_rejected_on_host(lib, kw, expected):
    assert binding.STATUS_NAMES[_scall(**kw)] == expected


@pytest.mark.parametrize("kw", [
    dict(),                                                       # all contiguous
    dict(q_strides=BLHD_Q, o_strides=BLHD_Q, k_strides=BLHD_KV, v_strides=BLHD_KV),
    dict(k_strides=(999, 24 * 64, 64), B=1),                      # extent-1 batch: stride unused
    dict(q_strides=(16 * 64, 7, 64), Hq=1, Hkv=1, o_strides=(16 * 64, 3, 64)),
    dict(k_strides=(24 * 64 * 3, 64, 2 * 64 * 3)),                # a slice of packed [B, L, 3, H, D]
    dict(q_strides=(0, 0, 0), o_strides=(0, 0, 0), B=1, Hq=1, Hkv=1, Lq=1),  # one row: no stride used
    dict(v_strides=(64, 64, 64)),                                 # inputs may overlap themselves
])
def test_strided_valid_arguments_need_a_device(lib, kw):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    st = _scall(**kw)
    assert binding.STATUS_NAMES[st] in ("ATTN_ERR_CUDA", "ATTN_ERR_ARCH")


# ------------------------------------------------------------------ attn_fwd_masked

def _mcall(**kw):
    args = dict(q_ptr=A16, q_strides=None, k_ptr=A16, k_strides=None, v_ptr=A16, v_strides=None,
                o_ptr=A16, o_strides=None, lse_ptr=None, B=2, Hq=4, Hkv=2, Lq=16, Lk=24, D=64,
                sm_scale=0.125, causal=0, valid_len_ptr=None, mask_ptr=A16 + 3,
                mask_batch_stride=16 * 24, mask_row_stride=24, dtype=attn.ATTN_BF16, stream=None)
    args.update(kw)
    return attn.fwd_masked_raw(**args)


@pytest.mark.parametrize("kw, expected", [
    (dict(mask_batch_stride=-1), "ATTN_ERR_STRIDE"),
    (dict(mask_row_stride=-24), "ATTN_ERR_STRIDE"),
    (dict(Lk=0), "ATTN_ERR_SHAPE"),
    (dict(D=100), "ATTN_ERR_HEADDIM"),
    (dict(q_ptr=None), "ATTN_ERR_NULL"),
    (dict(o_strides=(4 * 16 * 64, 16 * 64, 16)), "ATTN_ERR_STRIDE"),
    (dict(B=1 << 10, Hq=1, Hkv=1, Lq=1 << 20, Lk=1 << 20), "ATTN_ERR_SHAPE"),
])
def test_masked_invalid_arguments_rejected_on_host(lib, kw, expected):
    assert binding.STATUS_NAMES[_mcall(**kw)] == expected


@pytest.mark.parametrize("kw", [
    dict(),                                     # unaligned mask pointer is fine (byte loads)
    dict(mask_batch_stride=0),                  # one mask for every batch
    dict(mask_ptr=None),                        # no mask: attn_fwd_strided
])
def test_masked_valid_arguments_need_a_device(lib, kw):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    assert binding.STATUS_NAMES[_mcall(**kw)] in ("ATTN_ERR_CUDA", "ATTN_ERR_ARCH")


# ------------------------------------------------------------------ attn_fwd_f32

@pytest.mark.parametrize("args, expected", [
    (dict(q=None), "ATTN_ERR_NULL"),
    (dict(L=0), "ATTN_ERR_SHAPE"),
    (dict(D=32), "ATTN_ERR_HEADDIM"),
    (dict(kernel=3), "ATTN_ERR_ARG"),
    (dict(causal=5), "ATTN_ERR_ARG"),
    (dict(sm_scale=float("nan")), "ATTN_ERR_SCALE"),
    (dict(B=300, H=300), "ATTN_ERR_SHAPE"),
    (dict(L=60000, kernel=0), "ATTN_ERR_SHAPE"),
    (dict(o=A16 + 2), "ATTN_ERR_ALIGN"),
])
def test_f32_invalid_arguments_rejected_on_host(lib, args, expected):
    a = dict(q=A16, k=A16, v=A16, o=A16, lse=None, B=1, H=8, L=1024, D=64, sm_scale=0.125,
             causal=1, valid_len=None, kernel=2, stream=None)
    a.update(args)
    st = lib.attn_fwd_f32(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["L"], a["D"],
                          a["sm_scale"], a["causal"], a["valid_len"], a["kernel"], a["stream"])
    assert binding.STATUS_NAMES[st] == expected


# ------------------------------------------------------------------ attn_bwd

@pytest.mark.parametrize("args, expected", [
    (dict(dtype=4), "ATTN_ERR_DTYPE"),
    (dict(lse=None), "ATTN_ERR_NULL"),
    (dict(dv=None), "ATTN_ERR_NULL"),
    (dict(L=0), "ATTN_ERR_SHAPE"),
    (dict(D=48), "ATTN_ERR_HEADDIM"),
    (dict(D=256), "ATTN_ERR_HEADDIM"),
    (dict(Hq=6, Hkv=4), "ATTN_ERR_HEADS"),
    (dict(causal=3), "ATTN_ERR_ARG"),
    (dict(sm_scale=-2.0), "ATTN_ERR_SCALE"),
    (dict(dq=A16 + 1), "ATTN_ERR_ALIGN"),
])
@pytest.mark.parametrize("entry", ["attn_bwd", "attn_bwd_simt"])
def test_bwd_invalid_arguments_rejected_on_host(lib, args, expected, entry):
    _bwd_call(lib, entry, args, expected)


@pytest.mark.parametrize("D", [16, 32])
def test_bwd_simt_rejects_small_head_dims(lib, D):
    """attn_bwd takes D = 16 and 32 (the D = 64 kernels on zero-filled
    columns); the SIMT cross-check does not."""
    _bwd_call(lib, "attn_bwd_simt", dict(D=D), "ATTN_ERR_HEADDIM")


def _bwd_call(lib, entry, args, expected):
    a = dict(q=A16, k=A16, v=A16, o=A16, do=A16, lse=A16, dq=A16, dk=A16, dv=A16, B=1, Hq=4,
             Hkv=2, L=64, D=64, sm_scale=0.125, causal=1, valid_len=None, dtype=attn.ATTN_BF16,
             stream=None)
    a.update(args)
    st = getattr(lib, entry)(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                             a["dv"], a["B"], a["Hq"], a["Hkv"], a["L"], a["D"], a["sm_scale"],
                             a["causal"], a["valid_len"], a["dtype"], a["stream"])
    assert binding.STATUS_NAMES[st] == expected


@pytest.mark.parametrize("which, strides, expected", [
    ("q", (4 * 64 * 64, 64 * 64, 63), "ATTN_ERR_STRIDE"),       # seq stride not a multiple of 8
    ("dq", (4 * 64 * 64, 64 * 64, 32), "ATTN_ERR_STRIDE"),      # rows of dq overlap (32 < D)
    ("dk", (2 * 64 * 64, 0, 64), "ATTN_ERR_STRIDE"),            # head stride 0 with Hkv = 2
    ("do", (4 * 64 * 64, 64 * 64, 1 << 40), "ATTN_ERR_STRIDE"),  # stride too large
    ("dv", (2 * 64 * 64, 64, 60), "ATTN_ERR_STRIDE"),           # rows of dv overlap
])
def test_bwd_strided_stride_validation(lib, which, strides, expected):
    """attn_bwd_strided rejects invalid strides on the host, before any
    device work (the fake addresses are never dereferenced: every case here
    fails validation)."""
    names = ["q", "k", "v", "o", "do", "dq", "dk", "dv"]
    st = {n: None for n in names}
    st[which] = ctypes.byref(binding.Strides(*strides))
    rc = lib.attn_bwd_strided(A16, st["q"], A16, st["k"], A16, st["v"], A16, st["o"], A16, st["do"],
                              A16, A16, st["dq"], A16, st["dk"], A16, st["dv"], 1, 4, 2, 64, 64, 64,
                              0.125, 1, None, attn.ATTN_BF16, None)
    assert binding.STATUS_NAMES[rc] == expected


@pytest.mark.parametrize("msb, msr", [(-1, 64), (0, -64)])
def test_bwd_masked_negative_mask_strides_rejected(lib, msb, msr):
    """attn_bwd_masked rejects negative mask strides on the host (the fake
    addresses are never dereferenced: the call fails validation)."""
    rc = lib.attn_bwd_masked(A16, None, A16, None, A16, None, A16, None, A16, None, A16, A16, None,
                             A16, None, A16, None, 1, 4, 2, 64, 64, 64, 0.125, 1, None, A16, msb,
                             msr, attn.ATTN_BF16, None)
    assert binding.STATUS_NAMES[rc] == "ATTN_ERR_STRIDE"


def test_noalloc_source_calls_no_allocator():
    """attn_fwd_noalloc's translation unit, comments stripped, calls no
    allocating routine: no cudaMalloc* / cudaFree* / pool call and not the
    library's workspace pool (a regression there would not show in free
    device memory once the pool holds memory from earlier attn_fwd calls)."""
    import re
    src = os.path.join(os.path.dirname(attn.__file__), "csrc", "attn_noalloc.cu")
    text = open(src).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    for name in ("cudaMalloc", "cudaFree", "MemPool", "device_pool", "workspace_pool", "malloc(",
                 "new ", "cuMem"):
        assert name not in text, name
    assert "cudaGetSymbolAddress" in text


def test_forward_workspace_sizes(lib):
    """attn_fwd_workspace_size (host-only): fp16 needs none; bf16 needs the
    fp16 copy of V plus one int flag per (b, h_kv, 128-key tile), rounded up
    to 256 bytes; a mask adds its packed form, once when shared."""
    B, Hq, Hkv, L, D = 3, 8, 2, 1000, 64
    assert attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_F16) == 0
    v16 = B * Hkv * L * D * 2 + B * Hkv * 8 * 4
    assert attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_BF16) == (v16 + 255) // 256 * 256
    shared = attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_F16, mask_batches=1)
    per_batch = attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_F16, mask_batches=B)
    assert 0 < shared < per_batch
    assert shared >= L * 8 * 16  # one bit per position, 16 bytes per (row, key tile)
    with pytest.raises(binding.AttnError):
        attn.fwd_workspace_size(B, Hq, Hkv, L, L, D, attn.ATTN_F16, mask_batches=2)
    with pytest.raises(binding.AttnError):
        attn.fwd_workspace_size(B, 3, 2, L, L, D, attn.ATTN_F16)


@pytest.mark.parametrize("ws, nbytes", [(None, 0), (None, 1 << 30), (A16 + 16, 1 << 30),
                                        (A16, 16)])
def test_bad_forward_workspace_rejected_on_host(lib, ws, nbytes):
    st = lib.attn_fwd_ws(A16, A16, A16, A16, None, 1, 2, 1, 16, 64, 0.125, 0, None,
                         attn.ATTN_BF16, ws, nbytes, None)
    assert binding.STATUS_NAMES[st] == "ATTN_ERR_WORKSPACE"


def test_bad_backward_workspace_pointer_rejected_on_host(lib):
    args = [A16, None, A16, None, A16, None, A16, None, A16, None, A16, A16, None, A16, None, A16,
            None, 1, 2, 1, 16, 16, 64, 0.125, 0, None, None, 0, 0, attn.ATTN_BF16]
    for ws in (None, A16 + 16):
        st = lib.attn_bwd_masked_ws(*args, ws, 1 << 20, None)
        assert binding.STATUS_NAMES[st] == "ATTN_ERR_WORKSPACE"
