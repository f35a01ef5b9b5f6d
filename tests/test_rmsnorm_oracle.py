"""Pins of the oracle's QK normalisation and its tangent (oracle.rmsnorm_jvp).

The norm is the per-head RMSNorm of the page "Обслуживание Ideogram v4 менее чем
за секунду" (dev48.org), section on fusing RMSNorm: y = x rsqrt(mean(x^2) + eps)
weight over each head's d channels.  The student of the page "带分数正则的一致性蒸馏"
keeps its QK normalisation (section 一致性模型), so the attention's Q and K
tangents pass through this map first.  Everything here is checked against things
other than the oracle itself: torch's own rms_norm and its forward-mode autodiff,
finite differences, and properties the definition fixes (scale invariance, unit
RMS, the tangent orthogonal to x).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _case(rows=6, d=128, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, d)) * scale
    xt = rng.standard_normal((rows, d)) * 0.3
    w = 1.0 + 0.2 * rng.standard_normal(d)
    return x, xt, w


@pytest.mark.parametrize("d", [16, 64, 128, 256])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_norm_matches_torch_rms_norm(d, eps):
    x, xt, w = _case(d=d, seed=d)
    y, _ = oracle.rmsnorm_jvp(x, xt, w, eps)
    ref = F.rms_norm(torch.from_numpy(x), (d,), weight=torch.from_numpy(w), eps=eps).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("d", [16, 128, 256])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.5])
def test_tangent_matches_torch_forward_mode_autodiff(d, eps):
    x, xt, w = _case(d=d, seed=10 + d)
    _, yt = oracle.rmsnorm_jvp(x, xt, w, eps)
    wt = torch.from_numpy(w)
    _, ref = torch.func.jvp(lambda a: F.rms_norm(a, (d,), weight=wt, eps=eps), (torch.from_numpy(x),),
                            (torch.from_numpy(xt),))
    np.testing.assert_allclose(yt, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_tangent_matches_central_difference():
    x, xt, w = _case(rows=4, d=128, seed=3)
    h = 1e-6
    yp, _ = oracle.rmsnorm_jvp(x + h * xt, xt, w, 1e-6)
    ym, _ = oracle.rmsnorm_jvp(x - h * xt, xt, w, 1e-6)
    _, yt = oracle.rmsnorm_jvp(x, xt, w, 1e-6)
    fd = (yp - ym) / (2 * h)
    assert np.max(np.abs(fd - yt)) <= 1e-7 * np.max(np.abs(yt))


def test_unit_rms_and_direction_at_zero_eps():
    x, xt, w = _case(rows=5, d=64, seed=4, scale=7.0)
    y, _ = oracle.rmsnorm_jvp(x, xt, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)
    c = np.sum(y * x, axis=1) / np.sum(x * x, axis=1)  # y is a positive multiple of x
    assert np.all(c > 0)
    np.testing.assert_allclose(y, c[:, None] * x, rtol=1e-13, atol=1e-15)
    yw, _ = oracle.rmsnorm_jvp(x, xt, w, 0.0)
    np.testing.assert_allclose(yw, y * w, rtol=1e-14)


def test_scale_invariance_gives_zero_tangent_along_x():
    # y(c x) = y(x) for c > 0 at eps = 0, so moving x along itself changes nothing
    x, _, w = _case(rows=5, d=128, seed=5)
    y1, yt = oracle.rmsnorm_jvp(x, 2.5 * x, w, 0.0)
    y2, _ = oracle.rmsnorm_jvp(3.0 * x, x, w, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-13)
    assert np.max(np.abs(yt)) <= 1e-13 * np.max(np.abs(y1))


def test_tangent_orthogonal_to_x_is_only_scaled():
    # with mean(x xt) = 0 the norm does not move: yt = w rho xt
    x, xt, w = _case(rows=5, d=128, seed=6)
    xt = xt - (np.sum(xt * x, axis=1) / np.sum(x * x, axis=1))[:, None] * x
    eps = 1e-3
    _, yt = oracle.rmsnorm_jvp(x, xt, w, eps)
    rho = 1.0 / np.sqrt(np.mean(x * x, axis=1) + eps)
    np.testing.assert_allclose(yt, w * rho[:, None] * xt, rtol=1e-11, atol=1e-14)


def test_tangent_is_linear():
    x, xt, w = _case(rows=3, d=32, seed=7)
    _, a = oracle.rmsnorm_jvp(x, xt, w, 1e-6)
    _, b = oracle.rmsnorm_jvp(x, -0.5 * xt + x, w, 1e-6)
    _, c = oracle.rmsnorm_jvp(x, x, w, 1e-6)
    np.testing.assert_allclose(b, -0.5 * a + c, rtol=1e-12, atol=1e-14)


def test_rejects_rows_with_no_norm():
    x, xt, w = _case(rows=2, d=16, seed=8)
    x[1] = 0.0
    with pytest.raises(ValueError):
        oracle.rmsnorm_jvp(x, xt, w, 0.0)
    y, yt = oracle.rmsnorm_jvp(x, xt, w, 1e-6)  # eps keeps a zero row finite: y = 0, yt = w xt / sqrt(eps)
    assert np.all(y[1] == 0.0)
    np.testing.assert_allclose(yt[1], w * xt[1] / np.sqrt(1e-6), rtol=1e-12)


def test_attention_through_the_norm_matches_autodiff_of_the_composition():
    """The QK-normed attention JVP, composed from the two oracle functions (norm
    tangents first, then the attention JVP on the normed Q, K and their tangents),
    equals torch.func.jvp of SDPA(rms_norm(q), rms_norm(k), v) in FP64."""
    rng = np.random.default_rng(9)
    H, N, d = 2, 40, 32
    q, k, v, qt, kt, vt = (rng.standard_normal((H, N, d)) for _ in range(6))
    wq, wk = 1.0 + 0.1 * rng.standard_normal(d), 1.0 + 0.1 * rng.standard_normal(d)
    eps, s = 1e-6, d ** -0.5
    qn, qnt = oracle.rmsnorm_jvp(q, qt, wq, eps)
    kn, knt = oracle.rmsnorm_jvp(k, kt, wk, eps)
    o, ot, _, _ = oracle.attn_jvp(qn, kn, v, qnt, knt, vt, s)
    T = torch.from_numpy
    twq, twk = T(wq), T(wk)

    def f(q_, k_, v_):
        return F.scaled_dot_product_attention(F.rms_norm(q_, (d,), weight=twq, eps=eps),
                                              F.rms_norm(k_, (d,), weight=twk, eps=eps), v_, scale=s)

    ro, rot = torch.func.jvp(f, (T(q), T(k), T(v)), (T(qt), T(kt), T(vt)))
    np.testing.assert_allclose(o, ro.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ot, rot.numpy(), rtol=1e-10, atol=1e-11)
