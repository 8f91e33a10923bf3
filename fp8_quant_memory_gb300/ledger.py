"""Ideal (algorithmic) byte ledger of each entry point: every input read once, every output written
once, the norm weight(s) and the rotary table counted once per call.

This follows the accounting rule of "ledger.py" (Ch.13 ledger: one read per input, one write per
output, intermediates not free) and the prologue ledger of "case_norm_rope_quant.py" (Ch.28,
``Design.payload_bytes`` + ``Design.ideal_lookup_bytes``), with one correction: the tables here are
half width ([rows, rope_dim/2] per cos and sin), so the table term is ``2 * T * (R/2) * table_bytes``
instead of the page's ``2 * T * head_dim * table_bytes``.
"""
from __future__ import annotations

ELEM_BYTES = {"fp32": 4, "fp16": 2, "bf16": 2, "e4m3": 1}


def qk_prologue_bytes(T: int, Hq: int, Hk: int, D: int, R: int | None = None, dtype: str = "bf16",
                      table_dtype: str = "fp32") -> int:
    R = D if R is None else R
    rows = T * (Hq + Hk)
    x = rows * D * ELEM_BYTES[dtype]
    q = rows * D * ELEM_BYTES["e4m3"]
    scale = rows * 4
    table = 2 * T * (R // 2) * ELEM_BYTES[table_dtype]
    weights = 2 * D * ELEM_BYTES[dtype]
    return x + q + scale + table + weights


def qk_prologue_flops(T: int, Hq: int, Hk: int, D: int) -> int:
    """The Ch.28 page's FLOP ledger of the prologue ("case_norm_rope_quant.py", ``Design.flops``): per
    row of head_dim D, 2D for the sum of squares, 3 for rsqrt and the two scalings, 2D for the
    weight multiply, 6 per RoPE pair (D/2 pairs: four products, two sums), D for the absmax and 2D
    for scale-and-convert. Reported beside the byte ledger; bytes are what bind."""
    rows = T * (Hq + Hk)
    return rows * (2 * D + 3 + 2 * D + 6 * (D // 2) + D + 2 * D)


def rope_quant_bytes(M: int, N: int, R: int, dtype: str = "bf16", table_dtype: str = "bf16",
                     write_y: bool = True, group_size: int | None = None) -> int:
    """x, w, cos/sin read; y (optional), codes and the fp32 scales written (one per row, or one per
    group_size columns)."""
    e = ELEM_BYTES[dtype]
    n_scales = M if group_size is None else M * (N // group_size)
    return (M * N * e + N * e + 2 * M * (R // 2) * ELEM_BYTES[table_dtype] + (M * N * e if write_y else 0)
            + M * N + n_scales * 4)


def rope_bytes(M: int, N: int, R: int, dtype: str = "fp16", table_dtype: str = "fp16") -> int:
    e = ELEM_BYTES[dtype]
    return 2 * M * N * e + N * e + 2 * M * (R // 2) * ELEM_BYTES[table_dtype]


def rmsnorm_fwd_bytes(M: int, N: int, dtype: str = "bf16") -> int:
    e = ELEM_BYTES[dtype]
    return 2 * M * N * e + N * e


def rmsnorm_bwd_bytes(M: int, N: int, dtype: str = "bf16") -> int:
    """x, grad_y read; dx written; w read; dw written (the fp32 partial workspace is extra)."""
    e = ELEM_BYTES[dtype]
    return 3 * M * N * e + 2 * N * e


def page_prologue_ideal_bytes(T: int, Hq: int, Hk: int, D: int, in_bytes: int = 2, out_bytes: int = 1,
                              table_bytes: int = 4) -> int:
    """The Ch.28 page's own ideal ledger (payload + ideal lookup), table counted at full head_dim width."""
    rows = T * (Hq + Hk)
    elems = rows * D
    payload = elems * in_bytes + elems * out_bytes + rows * 4
    lookup = 2 * D * in_bytes + 2 * T * D * table_bytes
    return payload + lookup


def page_unfused_norm_rope_quant_bytes(m: int, n: int, rope_dim: int, in_bytes: int = 2, out_bytes: int = 1) -> int:
    """The Ch.13 ledger's unfused plan for RMSNorm + RoPE + quantisation ("ledger.py",
    fused_norm_rope_quant, `separate`): RMSNorm reads x, w and writes normed; RoPE reads normed, cos, sin
    and writes rotated; quantisation reads rotated and writes q and one fp32 amax per row. cos and sin
    are [m, rope_dim/2] in the input dtype, as the page's Buf declarations."""
    x = m * n * in_bytes
    w = n * in_bytes
    table = 2 * m * (rope_dim // 2) * in_bytes
    normed = m * n * in_bytes
    rotated = m * n * in_bytes
    q = m * n * out_bytes
    amax = m * 4
    return (x + w + normed) + (normed + table + rotated) + (rotated + q + amax)


def page_fused_norm_rope_quant_bytes(m: int, n: int, rope_dim: int, in_bytes: int = 2, out_bytes: int = 1) -> int:
    """The same ledger's fused plan: read x, w, cos, sin once; write q and amax once."""
    return m * n * in_bytes + n * in_bytes + 2 * m * (rope_dim // 2) * in_bytes + m * n * out_bytes + m * 4
