"""Seeded synthetic inputs for the fused RMSNorm / RoPE / FP8 path.

This module builds inputs only; it holds none of the method's arithmetic. Both the CUDA path and the
reference oracle are fed from it. Every array is drawn from ``numpy.random.Generator(PCG64)`` with an
explicit seed -- the large activation arrays as fp32 standard normals scaled by their std, weights and
tables in fp64 -- and then converted to its storage dtype by torch.

The rotary tables are inputs too: ``angle[row, p] = pos[row] * theta ** (-2p / rope_dim)`` for
``p < rope_dim / 2`` in fp64, ``cos``/``sin`` of that in fp64, then rounded to the table dtype. The
tutorial's own demo draws random angles ("rmsnorm_rope_quant.py", ``__main__``); position-derived
tables give the same kind of values with the structure a real model feeds.

Named workloads (shapes, distributions and positions of the five measured configurations):

=========================  ===========================================================================
name                       inputs
=========================  ===========================================================================
``rope_quant_tiny``        x[256,512] bf16 ~N(0,1), w[512] ~N(1,0.1), rope_dim 64, bf16 tables from
                           pos = row index, theta 1e4
``rmsnorm_8k_4k``          x, grad_y [8192,4096] bf16 ~N(0,1), w[4096] ~N(1,0.1)
``qk_prologue_4k``         qk[4096, 32+8, 128] bf16 ~N(0, std 2), wq/wk[128] ~N(1,0.1), full-head
                           rope, fp32 tables from pos 0..4095, theta 1e4
``rope_fp16_64k``          x[65536,192] fp16 ~N(0,1) (2048 tokens x 32 heads), rope_dim 64, fp16
                           tables per row from the row's token position (0..2047), theta 1e4
``qk_prologue_32k``        qk[32768, 64+8, 128] bf16 ~N(0,1) with 1% of entries (uniform, without
                           replacement) times 50, positions uniform in [0, 131072), theta 1e6, fp32 tables
=========================  ===========================================================================
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

BASE_SEED = 20261202

_TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPES[name]


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _to(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(_TORCH_DTYPES[dtype])


def _normal32(rng: np.random.Generator, std: float, size) -> np.ndarray:
    """N(0, std) activations drawn in fp32 (they are stored in bf16/fp16 anyway)."""
    v = rng.standard_normal(size=size, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return v


def _distinct_indices(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """k distinct indices in [0, n), uniform without replacement (oversample, dedupe, subsample)."""
    cand = np.unique(rng.integers(0, n, size=int(k * 1.02) + 1024, dtype=np.int64))
    while cand.size < k:
        cand = np.unique(np.concatenate([cand, rng.integers(0, n, size=k, dtype=np.int64)]))
    return cand[rng.permutation(cand.size)[:k]]


def rope_table(positions: np.ndarray, rope_dim: int, theta: float, dtype: str):
    """(cos, sin), each [len(positions), rope_dim // 2] in ``dtype``."""
    half = rope_dim // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / rope_dim)
    angle = positions.astype(np.float64)[:, None] * inv_freq[None, :]
    return _to(np.cos(angle), dtype), _to(np.sin(angle), dtype)


def norm_weight(n: int, seed: int, dtype: str) -> torch.Tensor:
    """Norm weight ~ N(1, 0.1)."""
    return _to(_rng(seed).normal(1.0, 0.1, size=n), dtype)


def rows_inputs(M: int, N: int, rope_dim: int, dtype: str = "bf16", table_dtype: str = "bf16",
                seed: int = BASE_SEED, theta: float = 1e4, heads_per_token: int = 1,
                std: float = 1.0):
    """x [M, N] ~N(0, std), w [N] ~N(1, 0.1), per-row tables [M, rope_dim/2].

    Row r takes the position of its token, ``r // heads_per_token`` (1: pos = row index).
    """
    rng = _rng(seed)
    x = _to(_normal32(rng, std, (M, N)), dtype)
    w = _to(rng.normal(1.0, 0.1, size=N), dtype)
    pos = np.arange(M, dtype=np.int64) // max(heads_per_token, 1)
    cos, sin = rope_table(pos, max(rope_dim, 2), theta, table_dtype)
    if rope_dim == 0:
        cos, sin = cos[:, :0].contiguous(), sin[:, :0].contiguous()
    return {"x": x, "w": w, "cos": cos, "sin": sin}


def rmsnorm_inputs(M: int, N: int, dtype: str = "bf16", seed: int = BASE_SEED, std: float = 1.0):
    """x, grad_y [M, N] ~N(0, std), w [N] ~N(1, 0.1)."""
    rng = _rng(seed)
    x = _to(_normal32(rng, std, (M, N)), dtype)
    g = _to(_normal32(rng, 1.0, (M, N)), dtype)
    w = _to(rng.normal(1.0, 0.1, size=N), dtype)
    return {"x": x, "g": g, "w": w}


def qk_inputs(T: int, Hq: int, Hk: int, D: int, dtype: str = "bf16", table_dtype: str = "fp32",
              seed: int = BASE_SEED, std: float = 2.0, theta: float = 1e4, rope_dim: int | None = None,
              positions: str = "arange", max_position: int = 131072, outlier_frac: float = 0.0,
              outlier_mult: float = 50.0, token_stride: int | None = None):
    """Prologue inputs.

    qk: [T, Hq+Hk, D] (or [T, token_stride] with the heads packed first and the rest of each token
    row filled with other data, like the q/k slice of a fused QKV projection). Tables [T, R/2].
    positions: "arange" (0..T-1) or "uniform" (uniform integers in [0, max_position)).
    """
    H = Hq + Hk
    R = D if rope_dim is None else rope_dim
    rng = _rng(seed)
    vals = _normal32(rng, std, T * H * D)
    if outlier_frac > 0.0:
        k = int(round(outlier_frac * vals.size))
        vals[_distinct_indices(rng, vals.size, k)] *= np.float32(outlier_mult)
    wq = _to(rng.normal(1.0, 0.1, size=D), dtype)
    wk = _to(rng.normal(1.0, 0.1, size=D), dtype)
    if positions == "arange":
        pos = np.arange(T, dtype=np.int64)
    elif positions == "uniform":
        pos = rng.integers(0, max_position, size=T, dtype=np.int64)
    else:
        raise ValueError(positions)
    cos, sin = rope_table(pos, max(R, 2), theta, table_dtype)
    if R == 0:
        cos, sin = cos[:, :0].contiguous(), sin[:, :0].contiguous()
    if token_stride is None:
        qk = _to(vals.reshape(T, H, D), dtype)
    else:
        if token_stride < H * D:
            raise ValueError("token_stride must be >= (Hq+Hk)*D")
        full = _normal32(rng, std, (T, token_stride))
        full[:, : H * D] = vals.reshape(T, H * D)
        qk = _to(full, dtype)
    return {"qk": qk, "wq": wq, "wk": wk, "cos": cos, "sin": sin, "positions": pos,
            "Hq": Hq, "Hk": Hk, "D": D, "rope_dim": R}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "rope_quant" | "rmsnorm" | "qk" | "rope"
    params: dict
    seed: int

    def make(self):
        p = self.params
        if self.kind == "rope_quant" or self.kind == "rope":
            return rows_inputs(p["M"], p["N"], p["rope_dim"], p["dtype"], p["table_dtype"], self.seed,
                               p.get("theta", 1e4), p.get("heads_per_token", 1))
        if self.kind == "rmsnorm":
            return rmsnorm_inputs(p["M"], p["N"], p["dtype"], self.seed)
        if self.kind == "qk":
            return qk_inputs(p["T"], p["Hq"], p["Hk"], p["D"], p["dtype"], p["table_dtype"], self.seed,
                             p["std"], p["theta"], positions=p["positions"],
                             outlier_frac=p.get("outlier_frac", 0.0))
        raise ValueError(self.kind)


WORKLOADS = {
    "rope_quant_tiny": Workload("rope_quant_tiny", "rope_quant",
                                dict(M=256, N=512, rope_dim=64, dtype="bf16", table_dtype="bf16"),
                                BASE_SEED + 0),
    "rmsnorm_8k_4k": Workload("rmsnorm_8k_4k", "rmsnorm", dict(M=8192, N=4096, dtype="bf16"),
                              BASE_SEED + 1),
    "qk_prologue_4k": Workload("qk_prologue_4k", "qk",
                               dict(T=4096, Hq=32, Hk=8, D=128, dtype="bf16", table_dtype="fp32",
                                    std=2.0, theta=1e4, positions="arange"), BASE_SEED + 2),
    "rope_fp16_64k": Workload("rope_fp16_64k", "rope",
                              dict(M=65536, N=192, rope_dim=64, dtype="fp16", table_dtype="fp16",
                                   heads_per_token=32), BASE_SEED + 3),
    "qk_prologue_32k": Workload("qk_prologue_32k", "qk",
                                dict(T=32768, Hq=64, Hk=8, D=128, dtype="bf16", table_dtype="fp32",
                                     std=1.0, theta=1e6, positions="uniform", outlier_frac=0.01),
                                BASE_SEED + 4),
}
