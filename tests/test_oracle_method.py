"""Pins for the oracle's method functions: RMSNorm, NeoX partial RoPE, per-row FP8 quantisation,
the QK-Norm+RoPE+FP8 prologue and the RMSNorm backward.

Every function is pinned to something other than itself: hand-derived worked examples
(tests/golden/worked_examples.json), identities that are exact in fp32 (power-of-two scaling,
angle 0, quarter turns, constant rows), invariants of the real-valued definitions checked on the
fp64 twins (unit RMS, pair norms, angle composition, orthogonality of dx to x), central finite
differences for the backward, brute force nearest-code search, and the dequantisation error bound.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from fp8_quant_memory_gb300 import workloads as wl

BF16, FP16, FP32 = torch.bfloat16, torch.float16, torch.float32


def _golden():
    with open(os.path.join(GOLDEN, "worked_examples.json")) as f:
        return json.load(f)


G = _golden()


def t(vals, dt):
    return torch.tensor(vals, dtype=torch.float64).to(dt)


def ulp_f32(x):
    x = abs(float(x))
    if x == 0:
        return 2.0 ** -149
    return 2.0 ** (math.floor(math.log2(x)) - 23)


# --------------------------------------------------------------------------- worked examples
@pytest.mark.parametrize("dt", [BF16, FP16])
@pytest.mark.parametrize("case", ["rmsnorm_3_4", "rmsnorm_weight_index"])
def test_worked_rmsnorm(orc, case, dt):
    c = G[case]
    x = t(c["x"], dt)[None]
    w = t(c["w"], dt)
    y = orc.rmsnorm_fwd(x, w, eps=float(c["eps"]))
    expect = t(c["y"], dt)[None]
    assert torch.equal(y.view(torch.int16), expect.view(torch.int16)), (y, expect)


@pytest.mark.parametrize("tdt", [BF16, FP16, FP32])
def test_worked_rope_quarter_turn(orc, tdt):
    c = G["rope_quarter_turn"]
    x = t(c["x"], FP16)[None]
    w = t(c["w"], FP16)
    cos = t(c["cos"], tdt)[None]
    sin = t(c["sin"], tdt)[None]
    y = orc.rmsnorm_rope(x, w, cos, sin, eps=float(c["eps"]))
    assert torch.equal(y.view(torch.int16), t(c["y"], FP16)[None].view(torch.int16))


@pytest.mark.parametrize("case", ["quant_row", "quant_zero_row"])
def test_worked_quant(orc, case):
    c = G[case]
    y = t(c["y_bf16"], BF16)[None]
    q, scale = orc.quant_rows(y)
    assert q[0].tolist() == c["q"]
    assert scale.item() == np.float32(c["scale"])  # scale = amax / 448 rounded once to fp32


def test_worked_backward(orc):
    c = G["backward_3_4"]
    x = t(c["x"], BF16)[None]
    w = t(c["w"], BF16)
    g = t(c["g"], BF16)[None]
    dx, dw, dw32 = orc.rmsnorm_bwd(x, w, g, eps=float(c["eps"]))
    assert torch.equal(dx.view(torch.int16), t(c["dx"], BF16)[None].view(torch.int16))
    assert torch.allclose(dw32.double(), torch.tensor(c["dw"], dtype=torch.float64), rtol=1e-6, atol=1e-7)
    dxf, dwf = orc.rmsnorm_bwd_f64(x, w, g, eps=0.0)
    assert torch.allclose(dxf[0], torch.tensor(c["dx"], dtype=torch.float64), rtol=1e-14, atol=1e-15)
    assert torch.allclose(dwf, torch.tensor(c["dw"], dtype=torch.float64), rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------------------- RMSNorm
def test_rmsnorm_f64_unit_rms(orc):
    rng = np.random.Generator(np.random.PCG64(1))
    x = torch.from_numpy(rng.normal(0, 3, size=(17, 96)))
    y = orc.rmsnorm_f64(x, torch.ones(96, dtype=torch.float64), eps=0.0)
    assert torch.allclose((y ** 2).mean(-1), torch.ones(17, dtype=torch.float64), rtol=0, atol=1e-13)


def test_rmsnorm_f64_eps_enters_under_the_root(orc):
    """x = (a, a): y = a / sqrt(a^2 + eps)."""
    a, eps = 0.01, 1e-4
    y = orc.rmsnorm_f64(torch.tensor([[a, a]], dtype=torch.float64), torch.ones(2, dtype=torch.float64), eps)
    assert abs(y[0, 0].item() - a / math.sqrt(a * a + eps)) < 1e-15


@pytest.mark.parametrize("dt", [BF16, FP16])
def test_rmsnorm_power_of_two_scale_invariance_exact(orc, dt):
    """With eps = 0 every fp32 step scales exactly by powers of two, so y(2^k x) == y(x) bitwise."""
    d = wl.rows_inputs(33, 160, 0, "bf16" if dt == BF16 else "fp16", seed=5)
    x, w = d["x"], d["w"]
    y0 = orc.rmsnorm_fwd(x, w, eps=0.0)
    ks = (-3, 2, 5) if dt == BF16 else (1, 2, 4)  # fp16: keep every input a normal number
    for k in ks:
        xs = (x.float() * 2.0 ** k).to(dt)
        assert torch.equal(xs.float() * 2.0 ** -k, x.float())  # the scaled input is exact
        y1 = orc.rmsnorm_fwd(xs, w, eps=0.0)
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_rmsnorm_constant_row(orc):
    """A constant row c = +-2^k normalises to sign(c) * w exactly (eps = 0)."""
    w = wl.norm_weight(64, 3, "bf16")
    for c in (0.25, -8.0, 1.0):
        y = orc.rmsnorm_fwd(torch.full((1, 64), c, dtype=BF16), w, eps=0.0)
        assert torch.equal(y[0].view(torch.int16), (math.copysign(1, c) * w.float()).to(BF16).view(torch.int16))


@pytest.mark.parametrize("dt", [BF16, FP16])
def test_rmsnorm_fp32_oracle_within_one_rounding_of_fp64(orc, dt):
    """The fp32 oracle is the real-valued definition up to fp32 noise plus one storage rounding."""
    name = "bf16" if dt == BF16 else "fp16"
    d = wl.rows_inputs(64, 384, 0, name, seed=9)
    y = orc.rmsnorm_fwd(d["x"], d["w"], eps=1e-6).double()
    y64 = orc.rmsnorm_f64(d["x"].double(), d["w"].double(), 1e-6)
    step = 2.0 ** -8 if dt == BF16 else 2.0 ** -11  # half an ulp, relative, for normal outputs
    sub = 0.0 if dt == BF16 else 2.0 ** -25  # half an ulp of the fp16 subnormal range
    assert ((y - y64).abs() <= step * y64.abs() * 1.001 + sub).all()


def test_rmsnorm_weight_is_per_column(orc):
    """y(x, w) / w == y(x, 1) column by column (fp64 twin)."""
    rng = np.random.Generator(np.random.PCG64(2))
    x = torch.from_numpy(rng.normal(size=(5, 24)))
    w = torch.from_numpy(rng.uniform(0.5, 2.0, size=24))
    y = orc.rmsnorm_f64(x, w, 1e-6)
    y1 = orc.rmsnorm_f64(x, torch.ones(24, dtype=torch.float64), 1e-6)
    assert torch.allclose(y / w, y1, rtol=1e-14, atol=0)


# --------------------------------------------------------------------------- RoPE
def test_rope_f64_preserves_pair_norms_and_head(orc):
    rng = np.random.Generator(np.random.PCG64(3))
    M, N, R = 9, 40, 16
    rows = torch.from_numpy(rng.normal(size=(M, N)))
    ang = torch.from_numpy(rng.uniform(-7, 7, size=(M, R // 2)))
    out = orc.rope_f64(rows, ang.cos(), ang.sin())
    assert torch.equal(out[:, : N - R], rows[:, : N - R])
    lo, hi = rows[:, N - R: N - R // 2], rows[:, N - R // 2:]
    lo2, hi2 = out[:, N - R: N - R // 2], out[:, N - R // 2:]
    assert torch.allclose(lo2 ** 2 + hi2 ** 2, lo ** 2 + hi ** 2, rtol=1e-13, atol=1e-13)


def test_rope_f64_angles_compose(orc):
    rng = np.random.Generator(np.random.PCG64(4))
    M, N, R = 6, 32, 32
    rows = torch.from_numpy(rng.normal(size=(M, N)))
    a = torch.from_numpy(rng.uniform(-3, 3, size=(M, R // 2)))
    b = torch.from_numpy(rng.uniform(-3, 3, size=(M, R // 2)))
    two = orc.rope_f64(orc.rope_f64(rows, a.cos(), a.sin()), b.cos(), b.sin())
    one = orc.rope_f64(rows, (a + b).cos(), (a + b).sin())
    assert torch.allclose(two, one, rtol=1e-12, atol=1e-12)


def test_rope_f64_quarter_turn_pairs_half_apart(orc):
    """Angle pi/2 maps (lo, hi) = (row[p], row[p + R/2]) to (-hi, lo): NeoX pairing, not adjacent."""
    M, N, R = 1, 12, 8
    rows = torch.arange(1, N + 1, dtype=torch.float64)[None]
    out = orc.rope_f64(rows, torch.zeros(1, R // 2, dtype=torch.float64), torch.ones(1, R // 2, dtype=torch.float64))
    expect = rows.clone()
    base = N - R
    expect[0, base: base + R // 2] = -rows[0, base + R // 2:]
    expect[0, base + R // 2:] = rows[0, base: base + R // 2]
    assert torch.equal(out, expect)


@pytest.mark.parametrize("dt,tdt", [(BF16, BF16), (FP16, FP16), (BF16, FP32)])
def test_rope_angle_zero_is_identity_exact(orc, dt, tdt):
    """cos = 1, sin = 0: rmsnorm_rope == rmsnorm_fwd bit for bit (the rotation and the second
    rounding are then exact), for any rope_dim."""
    name = "bf16" if dt == BF16 else "fp16"
    for R in (0, 16, 64):
        d = wl.rows_inputs(20, 64, R, name, seed=6)
        c = torch.ones(20, R // 2, dtype=tdt)
        s = torch.zeros(20, R // 2, dtype=tdt)
        y = orc.rmsnorm_rope(d["x"], d["w"], c, s)
        assert torch.equal(y.view(torch.int16), orc.rmsnorm_fwd(d["x"], d["w"]).view(torch.int16))


def test_rope_quarter_turn_exact_on_stored_rows(orc):
    """cos = 0, sin = 1: the tail's halves swap with a sign flip exactly; the head is untouched."""
    d = wl.rows_inputs(8, 96, 32, "bf16", seed=8)
    y0 = orc.rmsnorm_fwd(d["x"], d["w"])
    y = orc.rmsnorm_rope(d["x"], d["w"], torch.zeros(8, 16, dtype=BF16), torch.ones(8, 16, dtype=BF16))
    base = 96 - 32
    assert torch.equal(y[:, :base].view(torch.int16), y0[:, :base].view(torch.int16))
    assert torch.equal(y[:, base: base + 16].float(), -y0[:, base + 16:].float())
    assert torch.equal(y[:, base + 16:].float(), y0[:, base: base + 16].float())


def test_rmsnorm_rope_fp32_oracle_close_to_fp64(orc):
    d = wl.rows_inputs(32, 256, 64, "fp16", "fp32", seed=10)
    y = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"]).double()
    n64 = orc.rmsnorm_f64(d["x"].double(), d["w"].double(), 1e-6)
    # the oracle rounds the normalised row to fp16 before rotating (two roundings)
    y64 = orc.rope_f64(n64, d["cos"].double(), d["sin"].double())
    assert ((y - y64).abs() <= 2.0 ** -9 * y64.abs() + 2.0 ** -10 * n64.abs().amax(-1, keepdim=True) * 0.01 + 1e-3).all()


# --------------------------------------------------------------------------- quantisation
def _quant_inputs(seed=12):
    return wl.rows_inputs(64, 512, 64, "bf16", "bf16", seed=seed)


def test_quant_amax_element_hits_fp8_max(orc):
    d = _quant_inputs()
    y, q, scale = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    mag = (q & 0x7F)
    assert (mag.amax(-1) == 0x7E).all()  # 448 = S.1111.110 in every row
    amax = y.float().abs().amax(-1)
    assert torch.equal(scale, torch.clamp(amax, min=1e-4) / 448.0)


def test_quant_is_composition_of_steps(orc):
    """The fused oracle's codes equal the quantiser applied to its own y."""
    d = _quant_inputs(13)
    y, q, scale = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    q2, s2 = orc.quant_rows(y)
    assert torch.equal(q, q2) and torch.equal(scale, s2)
    y2 = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    _, q3, s3 = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"], want_y=False)
    assert torch.equal(q3, q) and torch.equal(s3, scale)


def test_quant_dequant_error_bound(orc):
    """|decode(q) * scale - y| <= half an e4m3 step at |y / scale| (2^-4 relative for normals,
    2^-10 * scale absolute in the subnormal range)."""
    d = _quant_inputs(14)
    y, q, scale = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    yv = y.double()
    v = orc.decode(q).double()
    ratio = yv / scale.double()[:, None]
    err = (v - ratio).abs()
    bound = torch.where(ratio.abs() >= 2.0 ** -6, ratio.abs() * 2.0 ** -4, torch.full_like(ratio, 2.0 ** -10))
    assert (err <= bound * (1 + 1e-6)).all()


def test_quant_small_amax_row(orc):
    """A row whose amax is below 1e-4: scale = 1e-4/448 and no code reaches 448."""
    y = torch.tensor([[3e-5, -5e-5, 1e-6, 0.0]], dtype=FP32).to(BF16)
    q, scale = orc.quant_rows(y)
    assert scale.item() == np.float32(np.float32(1e-4) / np.float32(448.0))
    assert ((q & 0x7F) < 0x7E).all()


def test_quant_custom_fp8_max(orc):
    """fp8_max < 448: the amax element lands on the code nearest to fp8_max."""
    y = torch.tensor([[1.0, -0.5, 0.25, 2.0]]).to(BF16)
    q, scale = orc.quant_rows(y, fp8_max=240.0)
    assert scale.item() == np.float32(2.0 / 240.0)
    assert orc.decode(q[:, 3:]).item() == 240.0


# --------------------------------------------------------------------------- LayerNorm
@pytest.mark.parametrize("case", ["layernorm_1_2_3_4", "layernorm_affine_index"])
@pytest.mark.parametrize("dt", [BF16, FP16])
def test_worked_layernorm(orc, case, dt):
    c = G[case]
    x = t(c["x"], dt)[None]
    y, mean, rstd = orc.layernorm_fwd(x, t(c["g"], dt), t(c["b"], dt), eps=float(c["eps"]))
    assert torch.equal(y.view(torch.int16), t(c["y"], dt)[None].view(torch.int16))
    if "mean" in c:
        assert mean.item() == np.float32(c["mean"]) and rstd.item() == np.float32(c["rstd"])


def test_layernorm_shift_invariance_exact(orc):
    """Adding a constant to a row changes nothing: with small integers the shifted row, its mean and
    every deviation are exact, so y is identical bit for bit."""
    gen = torch.Generator().manual_seed(51)
    x = torch.randint(-8, 9, (9, 64), generator=gen).to(BF16)
    d = wl.rmsnorm_inputs(9, 64, "bf16", seed=51)
    y1, _, _ = orc.layernorm_fwd(x, d["w"], d["w"])
    y2, _, _ = orc.layernorm_fwd((x.float() + 16).to(BF16), d["w"], d["w"])
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_layernorm_power_of_two_scale_invariance_exact(orc):
    d = wl.rmsnorm_inputs(7, 256, "bf16", seed=52)
    y1, _, _ = orc.layernorm_fwd(d["x"], d["w"], None, eps=0.0)
    y2, _, _ = orc.layernorm_fwd((d["x"].float() * 8).to(BF16), d["w"], None, eps=0.0)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_layernorm_f64_zero_mean_unit_variance(orc):
    x = torch.randn(5, 300, generator=torch.Generator().manual_seed(53), dtype=torch.float64) * 3 + 7
    y = orc.layernorm_f64(x, torch.ones(300, dtype=torch.float64), None, 0.0)
    assert y.mean(1).abs().max() < 1e-12
    assert (y.pow(2).mean(1) - 1).abs().max() < 1e-12


def test_layernorm_fp32_oracle_within_one_rounding_of_fp64(orc):
    d = wl.rmsnorm_inputs(33, 1024, "bf16", seed=54)
    b = (d["w"].float() - 1).to(BF16)
    y, _, _ = orc.layernorm_fwd(d["x"], d["w"], b)
    y64 = orc.layernorm_f64(d["x"].double(), d["w"].double(), b.double(), 1e-5)
    err = (y.double() - y64).abs()
    assert (err <= y64.abs() * 2.0 ** -8 * 1.01 + 1e-6).all()  # one bf16 rounding (plus fp32 noise)


def test_layernorm_of_a_zero_mean_row_is_rmsnorm(orc):
    """A row whose mean is exactly 0 has var = mean(x^2): LayerNorm without bias is RMSNorm (the two
    round the statistic at slightly different points, so: within one storage rounding)."""
    x = torch.randn(6, 128, generator=torch.Generator().manual_seed(55))
    x = torch.cat([x, -x], 1).to(BF16)  # exact zero mean
    w = wl.rmsnorm_inputs(1, 256, "bf16", seed=55)["w"]
    y_ln, mean, _ = orc.layernorm_fwd(x, w, None, eps=1e-6)
    assert (mean == 0).all()
    y_rms = orc.rmsnorm_fwd(x, w, eps=1e-6)
    err = (y_ln.double() - y_rms.double()).abs()
    assert (err <= y_rms.double().abs() * 2.0 ** -7).all()


# --------------------------------------------------------------------------- saved rstd
def test_worked_rstd(orc):
    """[3, 4], eps = 0: mean(x^2) = 12.5, rstd = 1 / sqrt(12.5) = sqrt(2) / 5, rounded once to fp32."""
    x = torch.tensor([[3.0, 4.0]]).to(BF16)
    w = torch.ones(2, dtype=BF16)
    y, rstd = orc.rmsnorm_fwd_rstd(x, w, eps=0.0)
    assert rstd.item() == np.float32(np.sqrt(2.0) / 5.0)
    assert torch.equal(y.view(torch.int16), orc.rmsnorm_fwd(x, w, eps=0.0).view(torch.int16))


def test_fwd_rstd_is_the_forward_plus_its_rstd(orc):
    d = wl.rmsnorm_inputs(37, 1024, "bf16", seed=41)
    y, rstd = orc.rmsnorm_fwd_rstd(d["x"], d["w"])
    assert torch.equal(y.view(torch.int16), orc.rmsnorm_fwd(d["x"], d["w"]).view(torch.int16))
    ref = 1.0 / torch.sqrt(d["x"].double().pow(2).mean(1) + 1e-6)  # fp64 definition
    assert ((rstd.double() - ref).abs() / ref).max() < 2.0 ** -22  # a few fp32 roundings


def test_bwd_with_saved_rstd_equals_recompute(orc):
    """Reusing the forward's rstd gives the recomputing backward bit for bit (same rstd, same order)."""
    d = wl.rmsnorm_inputs(53, 512, "bf16", seed=42)
    _, rstd = orc.rmsnorm_fwd_rstd(d["x"], d["w"])
    a = orc.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], rstd)
    b = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    for u, v in zip(a, b):
        assert torch.equal(u.view(torch.int16) if u.dtype == BF16 else u, v.view(torch.int16) if v.dtype == BF16 else v)


def test_bwd_rstd_is_used_not_recomputed(orc):
    """The backward uses the rstd it is given: with twice the true rstd, dx and dw follow the
    definition dx = rstd * (g*w - xn * mean(g*w*xn)), xn = x * rstd, evaluated in fp64 at that rstd
    (a recomputed rstd would be off by a factor of two)."""
    d = wl.rmsnorm_inputs(7, 64, "bf16", seed=43)
    _, rstd = orc.rmsnorm_fwd_rstd(d["x"], d["w"], eps=0.0)
    r2 = rstd * 2.0  # exact
    dx, _, dw32 = orc.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], r2)
    x, w, g = d["x"].double(), d["w"].double(), d["g"].double()
    xn = x * r2.double()[:, None]
    gw = g * w
    c = (gw * xn).mean(1, keepdim=True)
    dx64 = r2.double()[:, None] * (gw - xn * c)
    assert ((dx.double() - dx64).abs() <= torch.clamp(dx64.abs() * 2.0 ** -7, min=1e-3)).all()
    assert ((dw32.double() - (g * xn).sum(0)).abs() <= 1e-4 * (g * xn).abs().sum(0) + 1e-6).all()


# --------------------------------------------------------------------------- group-wise scales
def test_worked_quant_groups(orc):
    c = G["quant_groups"]
    y = torch.tensor(c["y_bf16"], dtype=FP32).to(BF16)
    q, scale = orc.quant_groups(y, c["group_size"])
    assert q.tolist() == c["q"]
    assert scale.tolist() == [[float(np.float32(v)) for v in row] for row in c["scale"]]
    q_row, _ = orc.quant_rows(y[:1].contiguous())
    assert q_row[0].tolist() == c["q_per_row_row0"]


def test_quant_groups_one_group_is_the_per_row_quantiser(orc):
    """group_size = N reduces to one scale per row: bit for bit the per-row oracle."""
    d = _quant_inputs(21)
    y, q, scale = orc.rmsnorm_rope_quant(d["x"], d["w"], d["cos"], d["sin"])
    N = d["x"].shape[1]
    yg, qg, sg = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], N)
    assert torch.equal(yg.view(torch.int16), y.view(torch.int16))
    assert torch.equal(qg, q) and torch.equal(sg[:, 0], scale)


@pytest.mark.parametrize("gs", [8, 64, 128])
def test_quant_groups_equal_rows_of_groups(orc, gs):
    """Each group is quantised exactly like a row of its own: the [M, N] group-wise result equals
    the per-row quantiser on the [M * N/gs, gs] view of the same y."""
    d = _quant_inputs(22)
    y, q, scale = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs)
    M, N = y.shape
    q2, s2 = orc.quant_rows(y.reshape(M * N // gs, gs).contiguous())
    assert torch.equal(q, q2.reshape(M, N)) and torch.equal(scale, s2.reshape(M, N // gs))
    y_full = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    assert torch.equal(y.view(torch.int16), y_full.view(torch.int16))


def test_quant_groups_each_group_reaches_fp8_max_and_is_local(orc):
    """Every group's amax element lands on +-448 (code 0x7E/0xFE), and changing the values of one
    group leaves every other group's codes and scales unchanged."""
    gs = 128
    y = (torch.randn(16, 512, generator=torch.Generator().manual_seed(23)) * 3).to(BF16)
    q, scale = orc.quant_groups(y, gs)
    mag = (q & 0x7F).reshape(16, 4, gs)
    assert (mag.amax(-1) == 0x7E).all()
    y2 = y.clone()
    y2[:, 128:256] *= 7
    q2, s2 = orc.quant_groups(y2, gs)
    keep = torch.ones(4, dtype=torch.bool)
    keep[1] = False
    assert torch.equal(q.reshape(16, 4, gs)[:, keep], q2.reshape(16, 4, gs)[:, keep])
    assert torch.equal(scale[:, keep], s2[:, keep])
    assert not torch.equal(scale[:, 1], s2[:, 1])


def test_quant_groups_dequant_error_bound(orc):
    """|decode(q) * scale_g - y| <= half an e4m3 step of |y / scale_g| in every group."""
    gs = 64
    d = _quant_inputs(24)
    y, q, scale = orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], gs)
    M, N = y.shape
    ratio = y.double().reshape(M, N // gs, gs) / scale.double()[:, :, None]
    v = orc.decode(q).double().reshape(M, N // gs, gs)
    err = (v - ratio).abs()
    bound = torch.where(ratio.abs() >= 2.0 ** -6, ratio.abs() * 2.0 ** -4, torch.full_like(ratio, 2.0 ** -10))
    assert (err <= bound * (1 + 1e-6)).all()


def test_quant_groups_rejects_ragged_groups(orc):
    d = _quant_inputs(25)
    with pytest.raises(ValueError):
        orc.rmsnorm_rope_quant_groups(d["x"], d["w"], d["cos"], d["sin"], 96)  # 512 % 96 != 0


# --------------------------------------------------------------------------- prologue
def _qk(T=6, Hq=4, Hk=2, D=128, seed=15, **kw):
    return wl.qk_inputs(T, Hq, Hk, D, seed=seed, **kw)


def _prologue(orc, d, **kw):
    return orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], d["Hq"], d["Hk"],
                                  rope_dim=d["rope_dim"], **kw)


def test_prologue_per_row_fp8_max(orc):
    d = _qk()
    q, scale = _prologue(orc, d)
    assert ((q & 0x7F).amax(-1) == 0x7E).all()
    assert (scale > 0).all()


def test_prologue_head_weight_selection_exact(orc):
    """Duplicate one q head into a k head; with wk = 2 * wq the k row equals the q row times 2 at
    every fp32 step, so its scale doubles exactly and its codes are identical."""
    d = _qk(seed=16)
    qk = d["qk"].clone()
    Hq = d["Hq"]
    qk[:, Hq] = qk[:, 1]
    wk = (d["wq"].float() * 2).to(BF16)
    q, scale = orc.qk_norm_rope_quant(qk, d["wq"], wk, d["cos"], d["sin"], Hq, d["Hk"])
    assert torch.equal(q[:, Hq], q[:, 1])
    assert torch.equal(scale[:, Hq], scale[:, 1] * 2)


def test_prologue_table_row_is_per_token(orc):
    """Every head of token t uses table row t: the same head vector at every head of a token gives
    identical outputs, and changing table row t changes only token t."""
    d = _qk(seed=17)
    qk = d["qk"].clone()
    qk[:, :] = qk[:, :1]  # all heads of each token equal to head 0
    wk = d["wq"]
    q, scale = orc.qk_norm_rope_quant(qk, d["wq"], wk, d["cos"], d["sin"], d["Hq"], d["Hk"])
    assert (q == q[:, :1]).all() and (scale == scale[:, :1]).all()
    cos2, sin2 = d["cos"].clone(), d["sin"].clone()
    cos2[3], sin2[3] = 1.0, 0.0
    q2, s2 = orc.qk_norm_rope_quant(qk, d["wq"], wk, cos2, sin2, d["Hq"], d["Hk"])
    changed = (q2 != q).flatten(1).any(-1)
    assert changed.tolist() == [i == 3 for i in range(qk.shape[0])]


def test_prologue_token_stride(orc):
    """A [T, S] buffer (q/k heads packed first, other data after) gives the packed result."""
    d = _qk(seed=18, token_stride=6 * 128 + 3 * 128)
    H, D = d["Hq"] + d["Hk"], d["D"]
    packed = d["qk"][:, : H * D].contiguous().view(-1, H, D)
    q1, s1 = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], d["Hq"], d["Hk"])
    q2, s2 = orc.qk_norm_rope_quant(packed, d["wq"], d["wk"], d["cos"], d["sin"], d["Hq"], d["Hk"])
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_prologue_matches_fp64_definition(orc):
    """Scale within fp32 noise of the fp64 definition; codes equal the fp64 nearest code except at
    near-ties (at most one step, rarely)."""
    d = _qk(T=32, seed=19)
    q, scale = _prologue(orc, d)
    H, D = d["Hq"] + d["Hk"], d["D"]
    x = d["qk"].double().view(-1, D)
    w = torch.cat([d["wq"].double()[None].expand(d["Hq"], D), d["wk"].double()[None].expand(d["Hk"], D)])
    w = w[None].expand(d["qk"].shape[0], H, D).reshape(-1, D)
    n = x * torch.rsqrt((x ** 2).mean(-1, keepdim=True) + 1e-6) * w  # fp64 reference for the check
    cos = d["cos"].double().repeat_interleave(H, 0)
    sin = d["sin"].double().repeat_interleave(H, 0)
    y = orc.rope_f64(n, cos, sin)
    s64 = y.abs().amax(-1).clamp(min=1e-4) / 448.0
    assert torch.allclose(scale.double().flatten(), s64, rtol=2e-6, atol=0)
    # nearest codes of the fp64 ratios, via the (pinned) encoder
    ratio = (y / s64[:, None]).clamp(-448, 448).float()
    q64 = orc.encode(ratio, "e4m3").view(q.shape)
    diff = (q.to(torch.int32) - q64.to(torch.int32)).abs()
    assert int((diff > 1).sum()) == 0
    assert float((diff != 0).float().mean()) < 1e-3


def test_prologue_partial_rope(orc):
    """rope_dim < head_dim: the first D - R columns are only normalised (quarter turn check)."""
    d = _qk(T=3, Hq=2, Hk=1, D=64, seed=20, rope_dim=32)
    T = d["qk"].shape[0]
    c0 = torch.zeros(T, 16)
    s1 = torch.ones(T, 16)
    q_id, sc_id = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], torch.ones(T, 16), torch.zeros(T, 16),
                                         d["Hq"], d["Hk"], rope_dim=32)
    q_qt, sc_qt = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], c0, s1, d["Hq"], d["Hk"], rope_dim=32)
    assert torch.equal(sc_id, sc_qt)  # a quarter turn permutes |values|, amax unchanged
    assert torch.equal(q_qt[..., :32], q_id[..., :32])
    assert torch.equal(q_qt[..., 32:48], q_id[..., 48:64] ^ 0x80)
    assert torch.equal(q_qt[..., 48:64], q_id[..., 32:48])


# --------------------------------------------------------------------------- backward
def test_backward_f64_central_differences(orc):
    rng = np.random.Generator(np.random.PCG64(21))
    M, N, eps = 3, 8, 1e-3
    x = torch.from_numpy(rng.normal(size=(M, N)))
    w = torch.from_numpy(rng.normal(1, 0.3, size=N))
    G_ = torch.from_numpy(rng.normal(size=(M, N)))
    dx, dw = orc.rmsnorm_bwd_f64(x, w, G_, eps)

    def loss(xx, ww):
        return float((G_ * orc.rmsnorm_f64(xx, ww, eps)).sum())

    h = 1e-6
    for i in range(M):
        for j in range(N):
            xp, xm = x.clone(), x.clone()
            xp[i, j] += h
            xm[i, j] -= h
            fd = (loss(xp, w) - loss(xm, w)) / (2 * h)
            assert abs(fd - dx[i, j].item()) <= 1e-7 * max(1.0, abs(fd))
    for j in range(N):
        wp, wm = w.clone(), w.clone()
        wp[j] += h
        wm[j] -= h
        fd = (loss(x, wp) - loss(x, wm)) / (2 * h)
        assert abs(fd - dw[j].item()) <= 1e-7 * max(1.0, abs(fd))


def test_backward_f64_dx_orthogonal_to_x(orc):
    """eps = 0: y is invariant to scaling a row, so sum_j dx_j * x_j = 0 for any w and g."""
    rng = np.random.Generator(np.random.PCG64(22))
    x = torch.from_numpy(rng.normal(size=(7, 50)))
    w = torch.from_numpy(rng.normal(1, 0.5, size=50))
    g = torch.from_numpy(rng.normal(size=(7, 50)))
    dx, _ = orc.rmsnorm_bwd_f64(x, w, g, 0.0)
    assert ((dx * x).sum(-1).abs() <= 1e-12 * (dx.abs() * x.abs()).sum(-1)).all()


def test_backward_fp32_oracle_close_to_fp64(orc):
    d = wl.rmsnorm_inputs(48, 512, "bf16", seed=23)
    dx, dw, dw32 = orc.rmsnorm_bwd(d["x"], d["w"], d["g"])
    dx64, dw64 = orc.rmsnorm_bwd_f64(d["x"], d["w"], d["g"], 1e-6)
    # bf16 output: one rounding (2^-8 relative) plus fp32 noise
    assert ((dx.double() - dx64).abs() <= 2.0 ** -8 * dx64.abs() + 1e-5).all()
    rms = dw64.pow(2).mean().sqrt()
    assert ((dw32.double() - dw64).abs() <= 1e-5 * torch.maximum(dw64.abs(), rms)).all()
    assert torch.equal(dw.view(torch.int16), dw32.to(BF16).view(torch.int16))


def test_backward_dw_single_row_closed_form(orc):
    """M = 1, w = 1: dw_j = g_j * x_j * rstd and dx = rstd * (g - xn * mean(g * xn)) (fp64 twin)."""
    rng = np.random.Generator(np.random.PCG64(24))
    x = torch.from_numpy(rng.normal(size=(1, 16)))
    g = torch.from_numpy(rng.normal(size=(1, 16)))
    _, dw = orc.rmsnorm_bwd_f64(x, torch.ones(16, dtype=torch.float64), g, 0.0)
    r = math.sqrt(float((x ** 2).mean()))
    assert torch.allclose(dw, (g * x / r)[0], rtol=1e-14, atol=0)


def test_parallel_prologue_oracle_equals_one_call(orc):
    """The token-sliced, thread-pooled oracle used at full size is the same computation as one call."""
    from parity import oracle_prologue_parallel

    d = wl.qk_inputs(301, 6, 2, 128, "bf16", "fp32", seed=4321, std=2.0, positions="uniform", outlier_frac=0.01)
    q1, s1 = orc.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], 6, 2)
    q2, s2 = oracle_prologue_parallel(orc, d, 6, 2)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
