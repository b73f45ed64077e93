"""Host-side checks of attn_fwd_host that need no GPU: its argument checks and
the chunk plan (attn_host_plan) that decides which slices of Q, K, V, O and
LSE each pipelined copy and kernel covers."""
import ctypes
import itertools

import pytest

import attention_forward_attn_gb300 as attn
from attention_forward_attn_gb300 import binding

A16 = 0x10000  # a fake address (never dereferenced: every case fails before use)


@pytest.fixture(scope="module")
def lib(cuda_lib_path):
    return attn.load()


def _host_call(**kw):
    args = dict(q_ptr=A16, k_ptr=A16, v_ptr=A16, o_ptr=A16, lse_ptr=None, B=1, Hq=2, Hkv=1, L=16,
                D=64, sm_scale=0.125, causal=0, valid_len_ptr=None, dtype=attn.ATTN_BF16,
                stream=None)
    args.update(kw)
    return attn.fwd_raw(entry="attn_fwd_host", **args)


@pytest.mark.parametrize("kw, expected", [
    (dict(dtype=7), "ATTN_ERR_DTYPE"),
    (dict(q_ptr=None), "ATTN_ERR_NULL"),
    (dict(o_ptr=None), "ATTN_ERR_NULL"),
    (dict(B=0), "ATTN_ERR_SHAPE"),
    (dict(L=-1), "ATTN_ERR_SHAPE"),
    (dict(D=96), "ATTN_ERR_HEADDIM"),
    (dict(Hq=3, Hkv=2), "ATTN_ERR_HEADS"),
    (dict(causal=2), "ATTN_ERR_ARG"),
    (dict(sm_scale=float("nan")), "ATTN_ERR_SCALE"),
])
def test_host_entry_rejects_invalid_arguments(lib, kw, expected):
    assert binding.STATUS_NAMES[_host_call(**kw)] == expected


@pytest.mark.parametrize("kw", [dict(q_ptr=A16 + 1), dict(o_ptr=A16 + 2), dict(lse_ptr=A16 + 2),
                                dict(valid_len_ptr=A16 + 1)])
def test_host_entry_needs_no_alignment(lib, kw):
    """Host buffers are only copied: an odd address passes the argument checks
    (without a GPU the call then stops at the device probe)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the gpu tests run the host path")
    st = _host_call(**kw)
    assert binding.STATUS_NAMES[st] in ("ATTN_ERR_CUDA", "ATTN_ERR_ARCH")


def _pieces(u, u1, Hq, Hkv):
    """Attention calls a run of flattened query heads needs when every call
    keeps the head map h_kv = h_q // (Hq' / Hkv'): part of one group, whole
    groups of one batch, or whole batches."""
    G = Hq // Hkv
    n = 0
    while u < u1:
        h, rem = u % Hq, u1 - u
        if h % G or rem < G:
            u += min(rem, G - h % G)
        elif h == 0 and rem >= Hq:
            u += (rem // Hq) * Hq
        else:
            u += min(rem // G, (Hq - h) // G) * G
        n += 1
    return n


def _check_plan(B, Hq, Hkv, L, D, chunks):
    """Query heads and K/V heads each copied exactly once, in queue order; a
    chunk's K/V heads copied by it or an earlier chunk; chunk sizes bounded;
    the call count of each chunk as the group/batch cut gives it."""
    G = Hq // Hkv
    head = L * D * 2
    total = B * (Hq + 2 * Hkv) * head
    full = max(min(max(total // 8, 8 << 20), 32 << 20), -(-total // 48))
    q_next = kv_next = 0
    for i, (q0, nq, kv0, nkv, calls) in enumerate(chunks):
        assert q0 == q_next and nq >= 1
        assert kv0 == kv_next and nkv >= 0
        q_next += nq
        kv_next += nkv
        assert (q_next - 1) // G < kv_next, "chunk computes before its K/V heads are copied"
        assert calls == _pieces(q0, q0 + nq, Hq, Hkv)
        assert len(chunks) == 1 or nq == 1 or (nq + 2 * nkv) * head <= full
        if nq >= G and i + 1 < len(chunks) and q_next % G:
            # not ending on a group boundary: rounding down would drop over a quarter
            assert 4 * (q_next % G) > nq
    assert q_next == B * Hq and kv_next == B * Hkv


SHAPES = list(itertools.product((1, 2, 3, 4, 7, 64), (1, 8, 32), (1, 2, 3, 8), (1, 700, 4096),
                                (64, 128)))


@pytest.mark.parametrize("B, Hq, Hkv, L, D", [s for s in SHAPES if s[1] % s[2] == 0])
def test_plan_covers_every_head_once(lib, B, Hq, Hkv, L, D):
    chunks = attn.host_plan(B, Hq, Hkv, L, D)
    _check_plan(B, Hq, Hkv, L, D, chunks)
    # at most 48 full chunks, each cut by at most a quarter at a group
    # boundary, plus the ramps at both ends
    assert 1 <= len(chunks) <= 48 * 4 // 3 + 8
    if B * (Hq + 2 * Hkv) * L * D * 2 < 12 << 20:
        assert len(chunks) == 1


@pytest.mark.parametrize("B, Hq, Hkv, L, D", [(4, 32, 8, 4096, 128), (2, 32, 1, 8192, 128),
                                              (8, 32, 32, 4096, 64), (1, 1, 1, 65536, 128),
                                              (3, 12, 4, 3000, 64)])
def test_plan_of_large_problems(lib, B, Hq, Hkv, L, D):
    """Sizes ramp up from 1/8 of a full chunk (or one query head with its K/V,
    if larger) and back down to it at the end."""
    chunks = attn.host_plan(B, Hq, Hkv, L, D)
    _check_plan(B, Hq, Hkv, L, D, chunks)
    head = L * D * 2
    total = B * (Hq + 2 * Hkv) * head
    full = max(min(max(total // 8, 8 << 20), 32 << 20), -(-total // 48))
    small = max(full // 8, 3 * head)
    size = [(nq + 2 * nkv) * head for _, nq, _, nkv, _ in chunks]
    if B * Hq > 8:
        assert size[0] <= small and size[-1] <= small
        assert max(size) > small


def test_plan_of_the_causal_gqa_workload(lib):
    """Q 4x32x4096x128, K/V 4x8x4096x128 (201 MB of input): 1 MiB per query
    head, 2 MiB per K/V head pair (a group of four query heads shares one);
    full chunks of 24 MiB (an eighth of the input), 3 MiB first."""
    chunks = attn.host_plan(4, 32, 8, 4096, 128)
    assert chunks[:3] == [(0, 1, 0, 1, 1), (1, 3, 1, 0, 1), (4, 8, 1, 2, 1)]
    assert max((nq + 2 * nkv) for _, nq, _, nkv, _ in chunks) <= 24
    assert len(chunks) == 14 and sum(c[4] for c in chunks) == 17


def test_plan_cap_and_errors(lib):
    n = ctypes.c_int(-1)
    arr = (binding.Chunk * 3)()
    assert lib.attn_host_plan(4, 32, 8, 4096, 128, 1, arr, 3, ctypes.byref(n)) == 0
    assert n.value == 14  # full count, first three written
    assert [c.as_tuple() for c in arr] == [(0, 1, 0, 1, 1), (1, 3, 1, 0, 1), (4, 8, 1, 2, 1)]
    assert lib.attn_host_plan(4, 32, 8, 4096, 128, 1, None, 0, ctypes.byref(n)) == 0
    assert n.value == 14
    assert lib.attn_host_plan(4, 32, 8, 4096, 128, 1, None, 0, None) == 12   # NULL n_chunks
    assert lib.attn_host_plan(4, 32, 8, 4096, 128, 1, None, 2, ctypes.byref(n)) == 12
    assert lib.attn_host_plan(4, 32, 8, 4096, 128, 1, arr, -1, ctypes.byref(n)) == 12
    for args, name in (((4, 30, 8, 4096, 128, 1), "ATTN_ERR_HEADS"),
                       ((4, 32, 8, 4096, 80, 1), "ATTN_ERR_HEADDIM"),
                       ((0, 32, 8, 4096, 128, 1), "ATTN_ERR_SHAPE"),
                       ((4, 32, 8, 4096, 128, 9), "ATTN_ERR_DTYPE")):
        st = lib.attn_host_plan(*args, arr, 3, ctypes.byref(n))
        assert binding.STATUS_NAMES[st] == name
        assert n.value == 0
