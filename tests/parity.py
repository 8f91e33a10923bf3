"""Tolerance rules shared by the parity tests (CUDA path vs the oracle).

- bf16 outputs: |gpu - ref| <= max(2^-7 |ref|, 1e-3)   (the stated bf16 tolerance)
- fp16 outputs: |gpu - ref| <= max(2^-9 |ref|, 1e-3)   (two fp16 ulps; fp16 has 3 more bits)
- rotated columns of rmsnorm_rope(_quant): the same relative bound applied to |y| + |lo*c| + |hi*s|
  (assert_rope_close: the definition rounds the normalised row before rotating it)
- fp32 scales:  relative difference <= 1e-5
- fp8 codes:    identical, or one e4m3 step apart on at most 0.1% of the elements
- dw (fp32 sums): |gpu - ref| <= 1e-3 * max(|ref|, rms(ref)); bf16/fp16 dw within one ulp, or
  within 1e-3 * rms(ref) where the column's sum nearly cancels

The two widened rules (rotated columns, near-cancelling dw columns) also count the elements they
accept only because of the widening and bound that count: at most 1e-4 of the rotated elements
(the oracle with every row's rstd moved by 3 fp32 ulps needs the widening on 1.3e-5 of them, on a
4097 x 1536 bf16 case) and at most 0.1% of the dw columns (one column of 4096 on a 513 x 4096 fp16
case). Rows of rmsnorm_rope_quant whose scale is further than 1e-5 from the oracle's are accepted
only when codes and scale are exactly the quantiser of the kernel's own y; scale_rows_by_own_y
counts them.
"""
from __future__ import annotations

import math

import torch


def storage_tol(dtype):
    return (2.0 ** -7, 1e-3) if dtype == torch.bfloat16 else (2.0 ** -9, 1e-3)


def assert_storage_close(gpu: torch.Tensor, ref: torch.Tensor, what: str = "y"):
    rel, abs_ = storage_tol(ref.dtype)
    a = gpu.detach().cpu().double()
    b = ref.double()
    err = (a - b).abs()
    bound = torch.clamp(b.abs() * rel, min=abs_)
    bad = err > bound
    assert not bool(bad.any()), (
        f"{what}: {int(bad.sum())} of {bad.numel()} elements outside the tolerance; worst err "
        f"{float(err.max()):.3g} at ref {float(b.flatten()[int(err.flatten().argmax())]):.5g}")


def assert_rope_close(gpu: torch.Tensor, ref: torch.Tensor, normed: torch.Tensor, cos: torch.Tensor,
                      sin: torch.Tensor, what: str = "y", max_widened_frac: float = 1e-4) -> int:
    """Tolerance for rmsnorm_rope / rmsnorm_rope_quant outputs y [M, N] (cos, sin: [M, R/2]).

    Head columns: the storage rule. Rotated columns: "rmsnorm_rope_quant.py" (torch_reference_fused)
    rounds the normalised row to the storage dtype before rotating it, so a normalised value that
    lands one storage ulp away -- which a different but equally valid fp32 order of the sum of
    squares does by moving rstd an ulp -- moves y by up to one ulp of each rotation input. The bound
    there is rel * (|y| + |lo * c| + |hi * s|) (one rounding of each input and of the output), still
    far below the error of a wrong pair, sign or table row (of the order of the inputs themselves).
    `normed` is the oracle's normalised row (rmsnorm_fwd: x * rstd * w rounded to the dtype).
    """
    rel, abs_ = storage_tol(ref.dtype)
    a = gpu.detach().cpu().double()
    b = ref.double()
    M, N = b.shape
    R = 2 * cos.shape[-1]
    spread = torch.zeros_like(b)
    if R > 0:
        n = normed.double()
        lo, hi = n[:, N - R:N - R // 2], n[:, N - R // 2:]
        c, s = cos.double(), sin.double()
        spread[:, N - R:N - R // 2] = (lo * c).abs() + (hi * s).abs()
        spread[:, N - R // 2:] = (hi * c).abs() + (lo * s).abs()
    err = (a - b).abs()
    bound = torch.clamp((b.abs() + spread) * rel, min=abs_)
    bad = err > bound
    assert not bool(bad.any()), (
        f"{what}: {int(bad.sum())} of {bad.numel()} elements outside the tolerance; worst err "
        f"{float(err.max()):.3g} at ref {float(b.flatten()[int(err.flatten().argmax())]):.5g}")
    # elements that pass only because of the widening (all of them in the rotated columns)
    widened = int((err > torch.clamp(b.abs() * rel, min=abs_)).sum())
    n_rot = M * R
    allowed = max(1, math.ceil(max_widened_frac * n_rot)) if n_rot else 0
    assert widened <= allowed, (
        f"{what}: {widened} rotated elements pass only under the widened bound (limit {allowed} of {n_rot})")
    return widened


def code_order(q: torch.Tensor) -> torch.Tensor:
    """Signed position of each e4m3fn code on the number line (adjacent finite values differ by 1)."""
    q = q.to(torch.int32)
    mag = q & 0x7F
    return torch.where((q & 0x80) != 0, -mag, mag)


def assert_codes_close(gpu_q: torch.Tensor, ref_q: torch.Tensor, what: str = "q", max_frac: float = 1e-3):
    a = code_order(gpu_q.detach().cpu())
    b = code_order(ref_q)
    d = (a - b).abs()
    assert int(d.max()) <= 1 if d.numel() else True, f"{what}: codes differ by {int(d.max())} steps"
    frac = float((d != 0).float().mean()) if d.numel() else 0.0
    assert frac <= max_frac, f"{what}: {frac:.2%} of codes differ (limit {max_frac:.2%})"
    return frac


def assert_scale_close(gpu_s: torch.Tensor, ref_s: torch.Tensor, rel: float = 1e-5, what: str = "scale"):
    a = gpu_s.detach().cpu().double()
    b = ref_s.double()
    r = ((a - b).abs() / b.abs()).max() if b.numel() else torch.tensor(0.0)
    assert float(r) <= rel, f"{what}: relative difference {float(r):.3g} > {rel}"


def assert_dw_close(gpu_f32: torch.Tensor, ref_f32: torch.Tensor, rel: float = 1e-3):
    a = gpu_f32.detach().cpu().double()
    b = ref_f32.double()
    rms = b.pow(2).mean().sqrt()
    bound = rel * torch.maximum(b.abs(), rms)
    bad = (a - b).abs() > bound
    assert not bool(bad.any()), f"dw_f32: {int(bad.sum())} columns outside 1e-3 * max(|ref|, rms)"


def assert_within_one_ulp(gpu: torch.Tensor, ref: torch.Tensor, what: str = "dw", rms_floor: float = 1e-3,
                          max_floor_frac: float = 1e-3) -> int:
    """bf16/fp16 dw within one ulp of the oracle's, or within rms_floor * rms(ref) of it. A column
    whose sum over rows nearly cancels (|dw| far below the rms of dw) moves by several of its own ulps
    when rstd moves by one fp32 ulp -- which any fp32 order of the sum of squares other than the
    oracle's does -- so there the fp32 rule's rms floor applies (tests/test_parity_rules.py pins this
    on the oracle alone)."""
    gc = gpu.detach().cpu()
    a = gc.view(torch.int16).to(torch.int32)
    b = ref.view(torch.int16).to(torch.int32)
    # same-sign patterns are ordered like integers; treat +-0 as equal
    ord_a = torch.where(a < 0, -(a & 0x7FFF), a)
    ord_b = torch.where(b < 0, -(b & 0x7FFF), b)
    rb = ref.double()
    floor = rms_floor * float(rb.pow(2).mean().sqrt()) if rb.numel() else 0.0
    far = (ord_a - ord_b).abs() > 1
    bad = far & ((gc.double() - rb).abs() > floor)
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} columns more than one ulp apart and above the rms floor"
    # columns accepted only through the rms floor
    widened = int(far.sum())
    allowed = max(1, math.ceil(max_floor_frac * far.numel()))
    assert widened <= allowed, f"{what}: {widened} columns pass only under the rms floor (limit {allowed})"
    return widened


def scale_rows_by_own_y(gpu_s: torch.Tensor, ref_s: torch.Tensor, rel: float = 1e-5) -> int:
    """Rows of rmsnorm_rope_quant whose scale is further than `rel` from the oracle's. The caller has
    checked that codes and scales are exactly the quantiser of the kernel's own y (the rule that
    accepts such a row: a bf16 flip of the row's amax element moves its scale by ~2^-8)."""
    a = gpu_s.detach().cpu().double()
    b = ref_s.double()
    return int(((a - b).abs() > rel * b.abs()).sum())


def oracle_prologue_parallel(orc, d: dict, hq: int, hk: int, **kw):
    """orc.qk_norm_rope_quant over the whole batch, split into one token slice per host core and run
    on a thread pool (the oracle is a C library called through ctypes, which releases the
    interpreter lock, and keeps no global state). Same result as one call."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    T = d["qk"].shape[0]
    cores = max(1, min(os.cpu_count() or 1, 32, T))
    bounds = [(T * i // cores, T * (i + 1) // cores) for i in range(cores)]
    bounds = [(a, b) for a, b in bounds if b > a]

    def run(ab):
        a, b = ab
        return orc.qk_norm_rope_quant(d["qk"][a:b], d["wq"], d["wk"], d["cos"][a:b], d["sin"][a:b], hq, hk, **kw)

    with ThreadPoolExecutor(len(bounds)) as ex:
        parts = list(ex.map(run, bounds))
    return torch.cat([p[0] for p in parts]), torch.cat([p[1] for p in parts])


def assert_own_quantiser(q: torch.Tensor, s: torch.Tensor, q_own: torch.Tensor, s_own: torch.Tensor):
    """The kernel's codes and scales against the oracle's quantiser applied to the kernel's own y:
    scales bit for bit (the scale is RN(max(amax, 1e-4) / fp8_max) of the same rounded y), codes under
    the code rule (kernels that code y as e4m3(RN(y * RN(1/scale))) differ from the quotient y / scale
    only where it sits at an e4m3 rounding boundary)."""
    assert torch.equal(s.detach().cpu(), s_own), "scales differ from the quantiser of the kernel's own y"
    assert_codes_close(q, q_own, "codes vs the quantiser of the kernel's own y")
