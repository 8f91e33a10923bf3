"""The tolerance rules of the parity tests, checked on the CPU with the oracle alone.

The rotated-column rule (assert_rope_close) must accept what a different but valid fp32 order of the
sum of squares produces (rstd moved by a few ulps), and must reject a wrong rotation (sign, pair or
table row), which the strict storage rule would also reject.
"""
import numpy as np
import pytest
import torch

from fp8_quant_memory_gb300 import workloads as wl
from parity import assert_rope_close, assert_storage_close


def _emulate(d, rstd_ulps=0, flip_sin=False, shift_table=False):
    """The definition's cast points in torch fp32 CPU ops, with rstd moved by `rstd_ulps` fp32 ulps."""
    DT = d["x"].dtype
    x, w = d["x"].float(), d["w"].float()
    c, s = d["cos"].float(), d["sin"].float()
    if flip_sin:
        s = -s
    if shift_table:
        c, s = torch.roll(c, 1, 0), torch.roll(s, 1, 0)
    M, N = x.shape
    R = 2 * c.shape[-1]
    ss = (x.double() ** 2).sum(1).float()
    rstd = (1.0 / torch.sqrt(ss / N + 1e-6)).numpy()
    for _ in range(abs(rstd_ulps)):
        rstd = np.nextafter(rstd, np.float32(np.inf if rstd_ulps > 0 else -np.inf)).astype(np.float32)
    n = ((x * torch.from_numpy(rstd)[:, None]) * w).to(DT).float()
    lo, hi = n[:, N - R:N - R // 2], n[:, N - R // 2:]
    return torch.cat([n[:, :N - R].to(DT), (lo * c - hi * s).to(DT), (hi * c + lo * s).to(DT)], 1)


@pytest.mark.parametrize("ulps", [-3, -1, 1, 3])
def test_rope_rule_accepts_a_few_ulps_of_rstd(orc, ulps):
    d = wl.rows_inputs(4097, 1536, 256, "bf16", "fp32", seed=970 + 4097)
    y_ref = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    assert torch.equal(_emulate(d).view(torch.int16), y_ref.view(torch.int16))  # the emulation is exact
    y = _emulate(d, rstd_ulps=ulps)
    with pytest.raises(AssertionError):  # the strict rule rejects these legitimate results
        assert_storage_close(y, y_ref)
    assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])


@pytest.mark.parametrize("mistake", ["flip_sin", "shift_table"])
def test_rope_rule_rejects_a_wrong_rotation(orc, mistake):
    d = wl.rows_inputs(64, 512, 64, "bf16", "bf16", seed=31)
    y_ref = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    y = _emulate(d, **{mistake: True})
    with pytest.raises(AssertionError):
        assert_rope_close(y, y_ref, orc.rmsnorm_fwd(d["x"], d["w"]), d["cos"], d["sin"])


def test_dw_one_ulp_rule_needs_the_rms_floor(orc):
    """The dtype dw of a column whose sum over rows nearly cancels moves by more than one of its own
    ulps when rstd moves by a single fp32 ulp (a different fp32 order of the sum of squares does
    that), so 'within one ulp' alone cannot hold; with the rms floor of the fp32 rule it does, and a
    wrong dw (a dropped row) is still rejected."""
    from parity import assert_within_one_ulp

    d = wl.rmsnorm_inputs(513, 4096, "fp16", seed=580 + 513)
    _, r = orc.rmsnorm_fwd_rstd(d["x"], d["w"])
    _, dw0, dw32 = orc.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], r)
    r1 = torch.from_numpy(np.nextafter(r.numpy(), np.float32(np.inf)).astype(np.float32))
    _, dw1, _ = orc.rmsnorm_bwd_rstd(d["x"], d["w"], d["g"], r1)
    a, b = dw1.view(torch.int16).to(torch.int32), dw0.view(torch.int16).to(torch.int32)
    ulps = (torch.where(a < 0, -(a & 0x7FFF), a) - torch.where(b < 0, -(b & 0x7FFF), b)).abs()
    assert int(ulps.max()) > 1  # one fp32 ulp of rstd: several fp16 ulps on a near-zero column
    j = int(ulps.argmax())
    assert abs(float(dw32[j])) < 1e-3 * float(dw32.pow(2).mean().sqrt())  # ... which is such a column
    assert_within_one_ulp(dw1, dw0)  # the rule with the rms floor accepts it
    _, dw_bad, _ = orc.rmsnorm_bwd_rstd(d["x"][1:], d["w"], d["g"][1:], r[1:])
    with pytest.raises(AssertionError):
        assert_within_one_ulp(dw_bad, dw0)


def test_rope_rule_bounds_how_many_elements_need_the_widening(orc):
    """The widened rotated-column bound is not a blanket: it reports how many elements it accepts
    only because of the widening and rejects a result that needs it more often than the oracle's
    own rounding-order changes do (rstd moved 3 ulps on every row: a dozen of a million)."""
    d = wl.rows_inputs(4097, 1536, 256, "bf16", "fp32", seed=970 + 4097)
    y_ref = orc.rmsnorm_rope(d["x"], d["w"], d["cos"], d["sin"])
    normed = orc.rmsnorm_fwd(d["x"], d["w"])
    n = assert_rope_close(_emulate(d, rstd_ulps=3), y_ref, normed, d["cos"], d["sin"])
    assert 0 < n <= 40
    with pytest.raises(AssertionError):
        assert_rope_close(_emulate(d, rstd_ulps=3), y_ref, normed, d["cos"], d["sin"], max_widened_frac=1e-6)
    assert assert_rope_close(y_ref, y_ref, normed, d["cos"], d["sin"]) == 0
