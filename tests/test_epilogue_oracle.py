"""Pins for the oracle's output-side functions (section 一致性模型, consistency
model, of the page "带分数正则的一致性蒸馏", its 蒸馏代码 listing): the JVP of the
wrapper coefficients, the JVP of _process_output, and the tangent target with
its warm-up, NaN masks, normalisation and the sCM loss.

Each pin is something other than the oracle: central finite differences,
library autodiff (torch.func.jvp) of the page's function written in torch,
the TrigFlow velocity the wrapper must reproduce for a perfect network, and
closed forms of the target and loss for inputs that switch single terms on.
"""
import math

import numpy as np
import pytest
import torch

import oracle

TAU = 1000.0


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("t", [0.05, 0.3, math.pi / 4, 1.1, 1.5])
def test_coeff_jvp_matches_central_difference(t):
    vals, tans = oracle.trigflow_coeffs_jvp(t, 0.37, TAU)
    assert vals == oracle.trigflow_coeffs(t, TAU)
    h = 1e-6
    cp, cm = oracle.trigflow_coeffs(t + h, TAU), oracle.trigflow_coeffs(t - h, TAU)
    for k in range(4):
        fd = 0.37 * (cp[k] - cm[k]) / (2 * h)
        assert abs(tans[k] - fd) <= 1e-7 * max(1.0, abs(fd))


def test_coeff_jvp_closed_form_at_quarter_pi():
    # cos t = sin t: D' = 0, so c_skip' = c_in' = 0; c_out' = -1/D^2 = -1/2; c_noise' = tau/2.
    _, tans = oracle.trigflow_coeffs_jvp(math.pi / 4, 1.0, TAU)
    assert abs(tans[0]) < 1e-15 and abs(tans[2]) < 1e-15
    assert abs(tans[1] + 0.5) < 1e-15 and abs(tans[3] - TAU / 2) < 1e-12


def _case(B=2, C=3, T=4, HW=5, seed=0):
    rng = np.random.default_rng(seed)
    arr = lambda: rng.standard_normal((B, C, T, HW))
    t = rng.uniform(0.1, 1.5, (B, T))
    tt = rng.standard_normal((B, T))
    return arr(), arr(), arr(), arr(), t, tt


def _torch_process_output(x, n, t):
    # The page's _process_output with the wrapper coefficients as functions of t.
    tb = t[:, None, :, None]
    D = torch.cos(tb) + torch.sin(tb)
    c_skip, c_out = 1.0 / D, -torch.sin(tb) / D
    x0 = c_skip * x + c_out * n
    return (torch.cos(tb) * x - x0) / torch.sin(tb)


def test_process_output_jvp_matches_autodiff():
    x, n, tx, tn, t, tt = _case(seed=3)
    F, tF = oracle.process_output_jvp(x, n, tx, tn, t, tt)
    prim = tuple(torch.from_numpy(a) for a in (x, n, t))
    tang = tuple(torch.from_numpy(a) for a in (tx, tn, tt))
    ref_F, ref_tF = torch.func.jvp(_torch_process_output, prim, tang)
    assert _rel(F, ref_F.numpy()) < 1e-13
    assert _rel(tF, ref_tF.numpy()) < 1e-12


def test_process_output_jvp_matches_central_difference():
    x, n, tx, tn, t, tt = _case(seed=4)
    h = 1e-6
    Fp, _ = oracle.process_output_jvp(x + h * tx, n + h * tn, tx, tn, t + h * tt, tt)
    Fm, _ = oracle.process_output_jvp(x - h * tx, n - h * tn, tx, tn, t - h * tt, tt)
    _, tF = oracle.process_output_jvp(x, n, tx, tn, t, tt)
    assert _rel(tF, (Fp - Fm) / (2 * h)) < 1e-7


def test_perfect_network_gives_trigflow_velocity():
    # If the network's x0 prediction is the true x0, F is dx_t/dt = -sin t x0 + cos t eps.
    rng = np.random.default_rng(7)
    B, C, HW = 3, 2, 6
    x0, eps = rng.standard_normal((B, C, 1, HW)), rng.standard_normal((B, C, 1, HW))
    t = rng.uniform(0.2, 1.4, (B, 1))
    tb = t[:, None, :, None]
    x = np.cos(tb) * x0 + np.sin(tb) * eps
    D = np.cos(tb) + np.sin(tb)
    n = (x0 - x / D) / (-np.sin(tb) / D)  # solves c_skip x + c_out n = x0
    F, _ = oracle.process_output_jvp(x, n, x, n, t, np.zeros_like(t))
    ref = oracle.trigflow_tangent(x0.reshape(B, -1), eps.reshape(B, -1), t[:, 0]).reshape(F.shape)
    assert _rel(F, ref) < 1e-12


def _scm_inputs(B=2, C=2, T=3, HW=4, seed=0):
    rng = np.random.default_rng(seed)
    z = lambda: rng.standard_normal((B, C, T, HW))
    return z(), z(), z(), z(), z(), rng.uniform(0.1, 1.5, (B, T))


def test_scm_each_term_of_g_in_isolation():
    F, Fsg, Ftc, x, tF, t = _scm_inputs(seed=1)
    zero = np.zeros_like(F)
    tb = t[:, None, :, None]
    # only the teacher gap: g = -cos t sqrt(1 - r^2 sin^2 t) (F_sg - F_teacher)
    r = 0.6
    g, _, _, _, _ = oracle.scm_tangent_loss(zero, Fsg, Ftc, zero, zero, t, r)
    raw = -np.cos(tb) * np.sqrt(1 - r * r * np.sin(tb) ** 2) * (Fsg - Ftc)
    norms = np.sqrt((raw ** 2).sum(axis=(1, 2, 3), keepdims=True)) + 0.1
    assert _rel(g, raw / norms) < 1e-13
    # only x: g = -r cos t sin t x
    g, _, _, _, _ = oracle.scm_tangent_loss(zero, zero, zero, x, zero, t, r)
    raw = -r * np.cos(tb) * np.sin(tb) * x
    assert _rel(g, raw / (np.sqrt((raw ** 2).sum(axis=(1, 2, 3), keepdims=True)) + 0.1)) < 1e-13
    # only the student tangent: g = -t_F
    g, _, _, _, _ = oracle.scm_tangent_loss(zero, zero, zero, zero, tF, t, r)
    assert _rel(g, -tF / (np.sqrt((tF ** 2).sum(axis=(1, 2, 3), keepdims=True)) + 0.1)) < 1e-13


def test_scm_warmup_limits():
    F, Fsg, Ftc, x, tF, t = _scm_inputs(seed=2)
    tb = t[:, None, :, None]
    # r = 0: no x term and sqrt(1) = 1
    g0, dfdt, _, _, _ = oracle.scm_tangent_loss(F, Fsg, Ftc, x, tF, t, 0.0)
    raw = -np.cos(tb) * (Fsg - Ftc) - tF
    assert _rel(g0, raw / (np.sqrt((raw ** 2).sum(axis=(1, 2, 3), keepdims=True)) + 0.1)) < 1e-13
    # df_dt does not depend on r
    _, dfdt1, _, _, _ = oracle.scm_tangent_loss(F, Fsg, Ftc, x, tF, t, 1.0)
    assert np.array_equal(dfdt, dfdt1)
    assert _rel(dfdt, -np.cos(tb) * (Fsg - Ftc) - (np.sin(tb) * x + tF)) < 1e-14
    # r = 1: sqrt(1 - sin^2) = |cos| and the x term is cos sin x
    g1, _, _, _, _ = oracle.scm_tangent_loss(F, Fsg, Ftc, x, tF, t, 1.0)
    raw = -np.cos(tb) * np.abs(np.cos(tb)) * (Fsg - Ftc) - (np.cos(tb) * np.sin(tb) * x + tF)
    assert _rel(g1, raw / (np.sqrt((raw ** 2).sum(axis=(1, 2, 3), keepdims=True)) + 0.1)) < 1e-12


def test_scm_loss_closed_forms():
    B, C, T, HW = 2, 2, 3, 4
    n = C * T * HW
    zero = np.zeros((B, C, T, HW))
    t = np.full((B, T), 0.7)
    # constant g = c: ||g|| = |c| sqrt(n), loss with F_theta = F_sg is n c^2 / (|c| sqrt(n) + 0.1)^2
    c = 0.8
    tF = np.full((B, C, T, HW), -c)
    g, _, loss, _, _ = oracle.scm_tangent_loss(zero, zero, zero, zero, tF, t, 0.3)
    assert np.allclose(g, c / (c * math.sqrt(n) + 0.1), rtol=1e-14)
    assert np.allclose(loss, n * c * c / (c * math.sqrt(n) + 0.1) ** 2, rtol=1e-14)
    # g = 0 (teacher equals the stop-gradient student, no x and no tangent): the loss is
    # the squared gap between F_theta and its stop-gradient copy
    rng = np.random.default_rng(5)
    F, Fsg = rng.standard_normal((B, C, T, HW)), rng.standard_normal((B, C, T, HW))
    g, _, loss, _, _ = oracle.scm_tangent_loss(F, Fsg, Fsg, zero, zero, t, 0.3)
    assert np.all(g == 0)
    assert np.allclose(loss, ((F - Fsg) ** 2).sum(axis=(1, 2, 3)), rtol=1e-14)


def test_scm_nan_masks_zero_one_sample_only():
    F, Fsg, Ftc, x, tF, t = _scm_inputs(B=3, seed=6)
    g_ref, dfdt_ref, loss_ref, ng, nf = oracle.scm_tangent_loss(F, Fsg, Ftc, x, tF, t, 0.5)
    assert not ng.any() and not nf.any()
    F2, tF2 = F.copy(), tF.copy()
    F2[1, 0, 1, 2] = np.nan        # student output NaN in sample 1
    tF2[2, 1, 0, 0] = np.nan       # tangent NaN in sample 2 -> g NaN there
    g, dfdt, loss, ng, nf = oracle.scm_tangent_loss(F2, Fsg, Ftc, x, tF2, t, 0.5)
    assert list(nf) == [False, True, False] and list(ng) == [False, False, True]
    assert loss[1] == 0.0 and loss[2] == 0.0 and np.all(g[1] == 0) and np.all(g[2] == 0)
    assert loss[0] == loss_ref[0] and np.array_equal(g[0], g_ref[0])
    assert np.array_equal(dfdt[:2], dfdt_ref[:2])  # df_dt is not masked
