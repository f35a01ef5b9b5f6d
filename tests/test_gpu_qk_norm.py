"""GPU: the QK normalisation and its tangent (qk_rmsnorm_jvp) against the FP64
oracle, element by element, and the attention JVP through it.

Per element the kernel may differ from the oracle by its output rounding to
bf16 (at most 2^-8 of the value, round to nearest) plus its fp32 arithmetic:
row sums of at most 256 products and one rsqrt, under 2^-14 of the sizes of the
terms behind each output (|w| |x| rho for y; |w| (|xt| rho + |x| rho^3 |a|)
for yt, with a = mean(x xt)).  That bound, derived from the arithmetic, is what
the tests hold each element to; the whole tensor also keeps rel-L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, host64

pytestmark = pytest.mark.gpu


def _draw(shape, d, seed, x_scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = (torch.randn(shape + (d,), generator=g, device="cuda") * x_scale).to(torch.bfloat16)
    xt = (torch.randn(shape + (d,), generator=g, device="cuda") * 0.3).to(torch.bfloat16)
    w = 1.0 + 0.2 * torch.randn(d, generator=g, device="cuda")
    return x, xt, w


def _check_rows(x, xt, w, y, yt, eps, name):
    xs, ts, ws = host64(x).reshape(-1, x.shape[-1]), host64(xt).reshape(-1, x.shape[-1]), host64(w)
    ry, ryt = oracle.rmsnorm_jvp(xs, ts, ws, eps)
    gy, gyt = host64(y).reshape(ry.shape), host64(yt).reshape(ry.shape)
    rho = 1.0 / np.sqrt(np.mean(xs * xs, axis=1, keepdims=True) + eps)
    a = np.mean(xs * ts, axis=1, keepdims=True)
    size_y = np.abs(ws) * np.abs(xs) * rho
    size_t = np.abs(ws) * (np.abs(ts) * rho + np.abs(xs) * rho ** 3 * np.abs(a))
    for got, ref, size, what in ((gy, ry, size_y, "y"), (gyt, ryt, size_t, "yt")):
        excess = np.abs(got - ref) - (2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * size + 1e-30)
        assert np.all(excess <= 0), "%s %s: %.3e over the rounding bound" % (name, what, excess.max())
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 1e-2, "%s %s: rel-L2 %.3e" % (name, what, rel)


@pytest.mark.parametrize("d", [16, 32, 64, 128, 256])
def test_qk_norm_every_row_against_oracle(cuda_lib, d):
    # ragged row counts; K has more rows than Q; raw activations of two scales
    q, q_t, wq = _draw((2, 3, 517), d, seed=d, x_scale=1.0)
    k, k_t, wk = _draw((2, 3, 700), d, seed=d + 1, x_scale=23.0)
    eps = 1e-6
    qn, qn_t, kn, kn_t = binding.qk_rmsnorm_jvp(q, q_t, k, k_t, wq, wk, eps=eps)
    torch.cuda.synchronize()
    _check_rows(q, q_t, wq, qn, qn_t, eps, "Q")
    _check_rows(k, k_t, wk, kn, kn_t, eps, "K")


def test_qk_norm_in_place_and_large_eps(cuda_lib):
    q, q_t, wq = _draw((1, 2, 129), 128, seed=5)
    k, k_t, wk = _draw((1, 2, 33), 128, seed=6, x_scale=0.05)  # eps comparable to mean(x^2)
    ref = binding.qk_rmsnorm_jvp(q, q_t, k, k_t, wq, wk, eps=1e-2)
    torch.cuda.synchronize()
    _check_rows(q, q_t, wq, ref[0], ref[1], 1e-2, "Q")
    _check_rows(k, k_t, wk, ref[2], ref[3], 1e-2, "K")
    qc, qtc, kc, ktc = (t.clone() for t in (q, q_t, k, k_t))
    binding.qk_rmsnorm_jvp(qc, qtc, kc, ktc, wq, wk, eps=1e-2, out=(qc, qtc, kc, ktc))
    torch.cuda.synchronize()
    for a, b in zip((qc, qtc, kc, ktc), ref):
        assert torch.equal(a, b)


def test_tangent_along_x_vanishes_at_zero_eps(cuda_lib):
    # the norm is scale invariant at eps = 0, so a tangent along x gives (almost) zero
    q, _, wq = _draw((1, 1, 300), 64, seed=7)
    q_t = q.clone()  # exactly parallel (xt = x)
    qn, qn_t, _, _ = binding.qk_rmsnorm_jvp(q, q_t, q, q_t, wq, wq, eps=0.0)
    torch.cuda.synchronize()
    size = np.abs(host64(qn)).max()
    assert np.max(np.abs(host64(qn_t))) <= 2.0 ** -12 * size


def test_attention_jvp_through_the_norm(cuda_lib):
    """Raw Q, K and tangents -> qk_rmsnorm_jvp -> attn_jvp_fwd, against the oracle's
    composition (rmsnorm_jvp, then attn_jvp) on the same raw bf16 values.  The GPU
    rounds the normed Q, K and tangents to bf16 before the attention, the oracle does
    not: that input rounding is inside the usual tolerances (as for fp32 inputs)."""
    B, H, N, d = 1, 2, 700, 128
    q, q_t, wq = _draw((B, H, N), d, seed=11, x_scale=3.0)
    k, k_t, wk = _draw((B, H, N), d, seed=12, x_scale=0.7)
    g = torch.Generator(device="cuda").manual_seed(13)
    v = torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16)
    v_t = (0.3 * torch.randn((B, H, N, d), generator=g, device="cuda")).to(torch.bfloat16)
    eps, s = 1e-6, d ** -0.5
    qn, qn_t, kn, kn_t = binding.qk_rmsnorm_jvp(q, q_t, k, k_t, wq, wk, eps=eps)
    o, ot, lse, mu = binding.attn_jvp_fwd(qn, kn, v, qn_t, kn_t, v_t, scale=s)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    rq, rqt = oracle.rmsnorm_jvp(host64(q), host64(q_t), host64(wq), eps)
    rk, rkt = oracle.rmsnorm_jvp(host64(k), host64(k_t), host64(wk), eps)
    ref = oracle.attn_jvp(rq, rk, host64(v), rqt, rkt, host64(v_t), s)
    assert_close(host64(o), ref[0], "O")
    assert_close(host64(ot), ref[1], "Ot")
    assert_close(host64(mu), ref[3], "mu")


def test_full_size_video_shape_sampled_rows(cuda_lib):
    # the video DiT Q and K shape (B=1, H=40, N=32760, d=128), raw activations;
    # seeded sampled rows of both against the oracle (rows are independent)
    spec = inputs.WORKLOADS["video_dit"]
    shape = (spec["B"], spec["H"], spec["N"])
    q, q_t, wq = _draw(shape, spec["d"], seed=21, x_scale=2.0)
    k, k_t, wk = _draw(shape, spec["d"], seed=22, x_scale=0.5)
    qn, qn_t, kn, kn_t = binding.qk_rmsnorm_jvp(q, q_t, k, k_t, wq, wk, eps=1e-6)
    torch.cuda.synchronize()
    rows = torch.as_tensor(np.unique(np.concatenate([
        np.random.default_rng(23).choice(q.numel() // spec["d"], 3000, replace=False),
        np.arange(q.numel() // spec["d"] - 5, q.numel() // spec["d"])])), device="cuda")
    flat = lambda t: t.reshape(-1, spec["d"])[rows]
    _check_rows(flat(q), flat(q_t), wq, flat(qn), flat(qn_t), 1e-6, "Q")
    _check_rows(flat(k), flat(k_t), wk, flat(kn), flat(kn_t), 1e-6, "K")
    del q, q_t, k, k_t, qn, qn_t, kn, kn_t
    torch.cuda.empty_cache()
