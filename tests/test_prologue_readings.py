"""The two readings of the prologue's cast points, compared on the oracle (CPU).

The prologue statement ("case_norm_rope_quant.py" (Ch.28), module docstring) names no intermediate
roundings and its payload has no y; the fusion page's definition ("rmsnorm_rope_quant.py",
torch_reference_fused) rounds the normalised row and the rotated row to the storage dtype because it
writes y. The library follows the first reading (fp32 from load to quantiser). These tests pin the
oracle's second reading (composed from rmsnorm_rope_quant) and show that the choice matters: on the
benchmark's inputs the two readings' codes differ by more than the code tolerance allows, so a kernel
can match one reading, not both.
"""
import torch

from fp8_quant_memory_gb300 import workloads as wl
from parity import code_order


def test_readings_agree_where_no_rounding_is_inexact(orc):
    """eps = 0, x = +-1 (rstd = 1/sqrt(1) = 1 exactly), storage-dtype weights, angle 0 (cos 1, sin 0):
    every intermediate is exactly representable, so both readings give the same codes and scales."""
    T, Hq, Hk, D = 16, 3, 2, 128
    g = torch.Generator().manual_seed(7)
    qk = (torch.randint(0, 2, (T, Hq + Hk, D), generator=g) * 2 - 1).to(torch.bfloat16)
    wq = (1 + torch.randint(-8, 8, (D,), generator=g) / 16).to(torch.bfloat16)
    wk = (1 + torch.randint(-8, 8, (D,), generator=g) / 16).to(torch.bfloat16)
    cos, sin = torch.ones(T, D // 2), torch.zeros(T, D // 2)
    q1, s1 = orc.qk_norm_rope_quant(qk, wq, wk, cos, sin, Hq, Hk, eps=0.0)
    q2, s2 = orc.qk_norm_rope_quant_rounded(qk, wq, wk, cos, sin, Hq, Hk, eps=0.0)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
    # ... and the scale is the largest |w| over the row's head weights / 448, exactly
    expect = torch.stack([wq.float().abs().max(), wk.float().abs().max()]) / 448.0
    assert torch.equal(s1[:, :Hq], expect[0].expand(T, Hq)) and torch.equal(s1[:, Hq:], expect[1].expand(T, Hk))


def test_rounded_reading_is_the_fusion_definition_per_head(orc):
    """The composed reading is rmsnorm_rope_quant applied to one (token, head) row with its head's
    weight and its token's table row: checked against a direct call for a few rows."""
    T, Hq, Hk, D = 8, 4, 2, 128
    d = wl.qk_inputs(T, Hq, Hk, D, "bf16", "fp32", seed=31, std=2.0)
    q, s = orc.qk_norm_rope_quant_rounded(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], Hq, Hk)
    for t, h in ((0, 0), (3, Hq - 1), (5, Hq), (7, Hq + Hk - 1)):
        w = d["wq"] if h < Hq else d["wk"]
        _, qq, ss = orc.rmsnorm_rope_quant(d["qk"][t, h][None].contiguous(), w, d["cos"][t][None].contiguous(),
                                          d["sin"][t][None].contiguous(), want_y=False)
        assert torch.equal(q[t, h], qq[0]) and torch.equal(s[t, h], ss[0])


def test_the_reading_matters_on_the_benchmark_inputs(orc):
    """On the first 256 tokens of the benchmark's prologue inputs the readings' codes differ on a few
    percent of elements, some by many e4m3 steps (rotated columns that nearly cancel amplify a
    storage-dtype rounding of the normalised value), and the scales by up to about 1%: far outside
    'identical, or one step apart on at most 0.1%'. The library, its tests and its tolerances follow
    the fp32 reading."""
    d = wl.qk_inputs(4096, 32, 8, 128, "bf16", "fp32", seed=20261202 + 2, std=2.0)
    sl = {k: d[k][:256].contiguous() for k in ("qk", "cos", "sin")}
    q1, s1 = orc.qk_norm_rope_quant(sl["qk"], d["wq"], d["wk"], sl["cos"], sl["sin"], 32, 8)
    q2, s2 = orc.qk_norm_rope_quant_rounded(sl["qk"], d["wq"], d["wk"], sl["cos"], sl["sin"], 32, 8)
    steps = (code_order(q1) - code_order(q2)).abs()
    assert float((steps != 0).float().mean()) > 0.01
    assert float((steps > 1).float().mean()) > 1e-3 and int(steps.max()) > 16
    rel = ((s1.double() - s2.double()).abs() / s1.double()).max().item()
    assert 2.0 ** -9 < rel < 2e-2
