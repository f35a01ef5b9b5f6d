"""Pins for the oracle's TrigFlow helpers.

Page "带分数正则的一致性蒸馏" (gitcode.csdn.net), section 时间步转换 (timestep
conversion): RectifiedFlow_TrigFlowWrapper maps a TrigFlow time t to
c_skip = c_in = 1/(cos t + sin t), c_out = -sin t/(cos t + sin t),
c_noise = tau sin t/(cos t + sin t), derived from the SNR match
tan t = sigma/alpha; the TrigFlow forward process is x_t = cos t x0 + sin t eps.
Pins: the rectified-flow times printed in section 推理流程 (inference), the
exact reconstruction identities the page derives the coefficients from, special
values, and finite differences for the tangent.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "trigflow_rf_timesteps.txt")


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                _, theta, rf = line.split()
                rows.append((float(theta), float(rf)))
    return rows


def test_printed_rectified_flow_times():
    rows = _golden()
    assert len(rows) == 5
    for theta, rf in rows:
        c = oracle.trigflow_coeffs(theta, 1000.0)
        assert round(c[3] / 1000.0, 4) == pytest.approx(rf, abs=1e-12)


def test_first_printed_time_is_sigma_over_sigma_plus_one():
    # The page notes the first value equals sigma/(sigma+1) with sigma = 80.
    c = oracle.trigflow_coeffs(math.atan(80.0), 1.0)
    assert c[3] == pytest.approx(80.0 / 81.0, rel=1e-14)


@pytest.mark.parametrize("t,expect", [
    (0.0, (1.0, 0.0, 1.0, 0.0)),
    (math.pi / 4, (1 / math.sqrt(2), -0.5, 1 / math.sqrt(2), 500.0)),
    (math.pi / 2, (1.0, -1.0, 1.0, 1000.0)),
])
def test_special_values(t, expect):
    c = oracle.trigflow_coeffs(t, 1000.0)
    for got, want in zip(c, expect):
        assert abs(got - want) <= 1e-12 * max(1.0, abs(want))


@pytest.mark.parametrize("t", [1e-3, 0.2, 0.7, 1.1, 1.5, math.atan(80.0), math.pi / 2 - 1e-4])
def test_reconstruction_identities(t):
    # With the exact rectified-flow velocity F_raw = eps - x0 the wrapper
    # reconstructs x0 = c_skip x_t + c_out F_raw, and the network input
    # c_in x_t equals the rectified-flow sample (1 - t_raw) x0 + t_raw eps with
    # t_raw = c_noise / tau (section 时间步转换).
    rng = np.random.default_rng(int(t * 1000))
    x0, eps = rng.standard_normal(64), rng.standard_normal(64)
    tau = 1000.0
    c_skip, c_out, c_in, c_noise = oracle.trigflow_coeffs(t, tau)
    xt = math.cos(t) * x0 + math.sin(t) * eps
    assert np.max(np.abs(c_skip * xt + c_out * (eps - x0) - x0)) < 1e-12
    t_raw = c_noise / tau
    assert np.max(np.abs(c_in * xt - ((1 - t_raw) * x0 + t_raw * eps))) < 1e-12
    assert abs(c_skip * (math.cos(t) + math.sin(t)) - 1.0) < 1e-15


def test_scaling_factor_is_linear_in_c_noise_only():
    a = oracle.trigflow_coeffs(0.9, 1.0)
    b = oracle.trigflow_coeffs(0.9, 1000.0)
    assert a[:3] == b[:3]
    assert b[3] == pytest.approx(1000.0 * a[3], rel=1e-15)


def test_outside_domain_is_rejected():
    with pytest.raises(ValueError):
        oracle.trigflow_coeffs(-math.pi / 2, 1000.0)


def test_tangent_matches_finite_difference_and_endpoints():
    rng = np.random.default_rng(3)
    B, M = 4, 300
    x0, eps = rng.standard_normal((B, M)), rng.standard_normal((B, M))
    t = np.array([0.0, 0.3, 1.2, math.pi / 2])
    out = oracle.trigflow_tangent(x0, eps, t)
    h = 1e-6
    xt = lambda tt: np.cos(tt)[:, None] * x0 + np.sin(tt)[:, None] * eps
    fd = (xt(t + h) - xt(t - h)) / (2 * h)
    assert np.max(np.abs(out - fd)) < 1e-8
    assert np.max(np.abs(out[0] - eps[0])) < 1e-15          # t = 0: dx/dt = eps
    assert np.max(np.abs(out[3] + x0[3])) < 1e-15           # t = pi/2: dx/dt = -x0
