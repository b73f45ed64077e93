"""Seeded synthetic inputs for the attention forward: the five benchmark workloads
and a generic generator for test shapes.

This module holds no attention arithmetic.  It draws Q/K/V on the CPU with a
seeded ``torch.Generator`` as N(0, 1) float32 and rounds them to fp16/bf16
(round-to-nearest-even), so the CUDA path and the float64 oracle read the very
same 16-bit values.  Seeds start at 20, the seed of tiny_flash_attn_triton.py's
``causal_test``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

F16 = "f16"
BF16 = "bf16"
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, dtype, masks and input recipe."""
    name: str
    dtype: str
    B: int
    Hq: int
    Hkv: int
    L: int
    D: int
    causal: bool
    padded: bool
    seed: int
    q_scale: float = 1.0
    fixed_valid_len: Optional[Sequence[int]] = None
    description: str = ""

    @property
    def sm_scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5


WORKLOADS = {
    "C1": Workload("C1", F16, 1, 2, 2, 128, 64, False, False, 20,
                   description="non-causal MHA, fp16 [1,2,128,64], LSE out"),
    "C2": Workload("C2", F16, 8, 16, 16, 2048, 64, True, False, 21,
                   description="causal MHA, fp16 [8,16,2048,64]"),
    "C3": Workload("C3", BF16, 8, 32, 32, 4096, 64, False, True, 22,
                   description="padding-masked MHA, bf16 [8,32,4096,64], "
                               "valid_len ~ U[0,4096], valid_len[0]=0"),
    "C4": Workload("C4", BF16, 4, 32, 8, 4096, 128, True, False, 23,
                   description="causal GQA, bf16 Q [4,32,4096,128], K/V [4,8,4096,128]"),
    "C5": Workload("C5", BF16, 2, 32, 1, 8192, 128, True, True, 24, q_scale=4.0,
                   fixed_valid_len=(8192, 5000),
                   description="causal MQA + padding, bf16 Q [2,32,8192,128] (x4), "
                               "K/V [2,1,8192,128], valid_len {8192,5000}"),
}


def _normal(gen: torch.Generator, shape, dtype: str, scale: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    x = x.to(TORCH_DTYPE[dtype])
    if scale != 1.0:
        # a power-of-two scale is exact in binary floating point, so scaling
        # after rounding equals rounding after scaling
        x = x * scale
    return x.contiguous()


def make_inputs(B: int, Hq: int, Hkv: int, L: int, D: int, dtype: str, seed: int,
                q_scale: float = 1.0, valid_len=None, padded: bool = False,
                Lk: Optional[int] = None):
    """Seeded CPU tensors (q, k, v, valid_len).

    q: [B, Hq, L, D], k/v: [B, Hkv, Lk, D] in ``dtype`` (Lk = L unless
    given).  ``valid_len`` is returned as an int32 CPU tensor [B]: the given
    values, or, when ``padded`` and none are given, B draws uniform in
    [0, Lk] with valid_len[0] = 0 (one fully masked batch).  None when there
    is no padding mask.
    """
    Lk = L if Lk is None else Lk
    gen = torch.Generator().manual_seed(int(seed))
    q = _normal(gen, (B, Hq, L, D), dtype, q_scale)
    k = _normal(gen, (B, Hkv, Lk, D), dtype)
    v = _normal(gen, (B, Hkv, Lk, D), dtype)
    vl = None
    if valid_len is not None:
        vl = torch.tensor(list(valid_len), dtype=torch.int32)
    elif padded:
        vl = torch.randint(0, Lk + 1, (B,), generator=gen, dtype=torch.int32)
        vl[0] = 0
    return q, k, v, vl


def workload_inputs(w: Workload):
    """Seeded CPU inputs (q, k, v, valid_len) of a named workload."""
    return make_inputs(w.B, w.Hq, w.Hkv, w.L, w.D, w.dtype, w.seed, q_scale=w.q_scale,
                       valid_len=w.fixed_valid_len, padded=w.padded)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of an fp16/bf16 CPU tensor as np.uint16 (no copy of values)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def dtype_code(dtype: str) -> int:
    """0 for fp16, 1 for bf16: the code both the C library and the oracle take."""
    return {F16: 0, BF16: 1}[dtype]
