"""Pins for the FP64 oracle, each against something other than the oracle itself.

Attention and its JVP follow the page "带分数正则的一致性蒸馏" (gitcode.csdn.net),
section 注意力 (attention): O = softmax(s Q K^T) V and, by the chain rule,
t_o = P t_v + t_p V with t_p = P (.) t_s - (P t_s^T) P and t_s = (t_q K^T + Q t_k^T) s.
The pins below are library routines (FP64 SDPA, logsumexp, torch.func.jvp),
finite differences, closed forms for one and two keys, and invariants that a
dropped term, a wrong sign, a swapped operand or a mis-indexed key would break.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from attention_jvp_gb300 import inputs


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _case(B=1, H=2, N=33, d=16, seed=0, tscale=0.5):
    q, k, v = (_rand((B, H, N, d), seed + i) for i in range(3))
    qt, kt, vt = (_rand((B, H, N, d), seed + 10 + i, tscale) for i in range(3))
    return q, k, v, qt, kt, vt


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _tiny_inputs():
    x = inputs.workload_inputs("tiny", device="cpu")
    arrs = [x[n].double().numpy() for n in inputs.NAMES]
    return arrs, x["scale"]


def test_tiny_recipe_shape_and_scale():
    (q, k, v, qt, kt, vt), s = _tiny_inputs()
    assert q.shape == (1, 2, 256, 64)
    assert s == 1.0 / 8.0


@pytest.mark.parametrize("scale", [None, 0.37])
def test_o_and_lse_match_library_sdpa(scale):
    (q, k, v, qt, kt, vt), s = _tiny_inputs()
    s = s if scale is None else scale
    o, ot, lse, mu = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, scale=s).numpy()
    assert _rel(o, ref) < 1e-12
    ref_lse = torch.logsumexp(torch.matmul(tq, tk.transpose(-1, -2)) * s, dim=-1).numpy()
    assert np.max(np.abs(lse - ref_lse)) < 1e-11


def test_tangent_matches_central_finite_difference():
    # h = 1e-6 in FP64 on the tiny workload: O((h^2) + eps/h) ~ 1e-10 error.
    (q, k, v, qt, kt, vt), s = _tiny_inputs()
    h = 1e-6
    o, ot, lse, mu = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    zeros = np.zeros_like(q)
    op, _, lp, _ = oracle.attn_jvp(q + h * qt, k + h * kt, v + h * vt, zeros, zeros, zeros, s)
    om, _, lm, _ = oracle.attn_jvp(q - h * qt, k - h * kt, v - h * vt, zeros, zeros, zeros, s)
    fd_o = (op - om) / (2 * h)
    fd_lse = (lp - lm) / (2 * h)
    assert _rel(ot, fd_o) < 1e-7
    # d LSE along the tangent is sum_j P_ij St_ij = mu_i.
    assert _rel(mu, fd_lse) < 1e-7


def test_tangent_matches_autodiff_jvp():
    q, k, v, qt, kt, vt = _case(B=2, H=3, N=40, d=24, seed=3)
    s = 0.29

    def attn(q_, k_, v_):
        w = torch.softmax(torch.matmul(q_, k_.transpose(-1, -2)) * s, dim=-1)
        return torch.matmul(w, v_)

    prim = tuple(torch.from_numpy(x) for x in (q, k, v))
    tang = tuple(torch.from_numpy(x) for x in (qt, kt, vt))
    ref_o, ref_ot = torch.func.jvp(attn, prim, tang)
    o, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    assert _rel(o, ref_o.numpy()) < 1e-12
    assert _rel(ot, ref_ot.numpy()) < 1e-12


def test_tangent_is_linear_in_the_tangents():
    q, k, v, qt1, kt1, vt1 = _case(seed=5)
    _, _, _, qt2, kt2, vt2 = _case(seed=50)
    s = 0.25
    a, b = 0.7, -1.9
    _, t1, _, m1 = oracle.attn_jvp(q, k, v, qt1, kt1, vt1, s)
    _, t2, _, m2 = oracle.attn_jvp(q, k, v, qt2, kt2, vt2, s)
    _, t12, _, m12 = oracle.attn_jvp(q, k, v, a * qt1 + b * qt2, a * kt1 + b * kt2, a * vt1 + b * vt2, s)
    assert _rel(t12, a * t1 + b * t2) < 1e-12
    assert _rel(m12, a * m1 + b * m2) < 1e-12


def test_zero_tangents_give_zero():
    q, k, v, _, _, _ = _case(seed=7)
    z = np.zeros_like(q)
    _, ot, _, mu = oracle.attn_jvp(q, k, v, z, z, z, 0.3)
    assert np.all(ot == 0.0) and np.all(mu == 0.0)


def test_only_value_tangent_gives_attention_of_value_tangent():
    # t_q = t_k = 0  =>  t_s = 0, t_p = 0, t_o = P t_v = SDPA(q, k, t_v).
    q, k, v, _, _, vt = _case(seed=9)
    z = np.zeros_like(q)
    s = 0.31
    _, ot, _, mu = oracle.attn_jvp(q, k, v, z, z, vt, s)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(x) for x in (q, k, vt)), scale=s).numpy()
    assert _rel(ot, ref) < 1e-12
    assert np.all(mu == 0.0)


def test_constant_value_rows_keep_only_value_tangent():
    # Rows of t_p sum to zero, so with every v_j equal t_p V = 0 and t_o = P t_v.
    q, k, _, qt, kt, vt = _case(seed=11)
    v = np.broadcast_to(_rand((1, 2, 1, 16), 99), q.shape).copy()
    s = 0.4
    o, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    assert _rel(o, v) < 1e-13
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(x) for x in (q, k, vt)), scale=s).numpy()
    assert _rel(ot, ref) < 1e-12


def test_single_key_closed_form():
    q, k, v, qt, kt, vt = _case(N=5, seed=13)
    k, kt, v, vt = (x[:, :, :1] for x in (k, kt, v, vt))
    s = 0.6
    o, ot, lse, mu = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    assert _rel(o, np.broadcast_to(v, o.shape)) < 1e-15
    assert _rel(ot, np.broadcast_to(vt, ot.shape)) < 1e-15
    S = s * np.einsum("bhid,bhjd->bhij", q, k)[..., 0]
    St = s * (np.einsum("bhid,bhjd->bhij", qt, k) + np.einsum("bhid,bhjd->bhij", q, kt))[..., 0]
    assert _rel(lse, S) < 1e-14
    assert _rel(mu, St) < 1e-14


def test_two_key_logistic_closed_form():
    # With two keys P_1 = sigma(S_1 - S_2), so
    # t_o = sigma'(D) (St_1 - St_2) (v_1 - v_2) + P_1 vt_1 + P_2 vt_2.
    q, k, v, qt, kt, vt = _case(N=7, seed=17)
    k, kt, v, vt = (x[:, :, :2] for x in (k, kt, v, vt))
    s = 0.45
    _, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    S = s * np.einsum("bhid,bhjd->bhij", q, k)
    St = s * (np.einsum("bhid,bhjd->bhij", qt, k) + np.einsum("bhid,bhjd->bhij", q, kt))
    D = S[..., 0] - S[..., 1]
    sig = 1.0 / (1.0 + np.exp(-D))
    dsig = sig * (1.0 - sig)
    dv = (v[:, :, 0] - v[:, :, 1])[:, :, None, :]
    ref = (dsig * (St[..., 0] - St[..., 1]))[..., None] * dv \
        + sig[..., None] * vt[:, :, None, 0] + (1 - sig)[..., None] * vt[:, :, None, 1]
    assert _rel(ot, ref) < 1e-13


def test_mu_shift_leaves_output_tangent_unchanged():
    # Append a coordinate with q = 0, k = 1, t_k = 0, t_q = c / s: every St_ij of a
    # row grows by c, S is unchanged.  Then mu grows by c and t_o (which sees
    # only St - mu) is unchanged.
    q, k, v, qt, kt, vt = _case(seed=19)
    s, c = 0.35, 1.7
    pad = lambda x, val: np.concatenate([np.full(x.shape[:-1] + (1,), val), x], axis=-1)
    base = oracle.attn_jvp(pad(q, 0.0), pad(k, 1.0), v, pad(qt, 0.0), pad(kt, 0.0), vt, s)
    shift = oracle.attn_jvp(pad(q, 0.0), pad(k, 1.0), v, pad(qt, c / s), pad(kt, 0.0), vt, s)
    assert _rel(shift[0], base[0]) < 1e-15
    assert _rel(shift[1], base[1]) < 1e-12
    assert np.max(np.abs(shift[3] - (base[3] + c))) < 1e-12


def test_row_subset_is_exact():
    q, k, v, qt, kt, vt = _case(N=50, seed=23)
    full = oracle.attn_jvp(q, k, v, qt, kt, vt, 0.3)
    rows = np.array([0, 7, 31, 49])
    sub = oracle.attn_jvp(q, k, v, qt, kt, vt, 0.3, rows=rows)
    for f, s_ in zip(full, sub):
        assert np.array_equal(f[:, :, rows], s_)


def test_query_and_key_counts_may_differ():
    q, _, _, qt, _, _ = _case(N=9, seed=29)
    _, k, v, _, kt, vt = _case(N=21, seed=31)
    o, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, 0.3)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(x) for x in (q, k, v)), scale=0.3).numpy()
    assert o.shape == (1, 2, 9, 16) and _rel(o, ref) < 1e-12


@pytest.mark.parametrize("nq,nk,d", [(9, 21, 32), (40, 7, 16)])
def test_cross_attention_tangent_matches_autodiff_jvp(nq, nk, d):
    # Fewer or more keys than queries and the small head dims of the page's
    # supported set: library autodiff of naive FP64 attention.
    q, _, _, qt, _, _ = _case(B=2, H=2, N=nq, d=d, seed=41)
    _, k, v, _, kt, vt = _case(B=2, H=2, N=nk, d=d, seed=43)
    s = d ** -0.5

    def attn(q_, k_, v_):
        return torch.matmul(torch.softmax(torch.matmul(q_, k_.transpose(-1, -2)) * s, dim=-1), v_)

    prim = tuple(torch.from_numpy(x) for x in (q, k, v))
    tang = tuple(torch.from_numpy(x) for x in (qt, kt, vt))
    ref_o, ref_ot = torch.func.jvp(attn, prim, tang)
    o, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    assert o.shape == (2, 2, nq, d)
    assert _rel(o, ref_o.numpy()) < 1e-12
    assert _rel(ot, ref_ot.numpy()) < 1e-12


@pytest.mark.parametrize("d,dv", [(16, 40), (32, 8)])
def test_value_head_dim_may_differ_autodiff_jvp(d, dv):
    # The page's forward lets V have its own head dim: library autodiff of
    # naive FP64 attention with a wider and a narrower V than Q and K.
    q, k, _, qt, kt, _ = _case(B=1, H=2, N=19, d=d, seed=47)
    v, vt = _rand((1, 2, 19, dv), 51), _rand((1, 2, 19, dv), 53, 0.5)
    s = 0.4

    def attn(q_, k_, v_):
        return torch.matmul(torch.softmax(torch.matmul(q_, k_.transpose(-1, -2)) * s, dim=-1), v_)

    prim = tuple(torch.from_numpy(x) for x in (q, k, v))
    tang = tuple(torch.from_numpy(x) for x in (qt, kt, vt))
    ref_o, ref_ot = torch.func.jvp(attn, prim, tang)
    o, ot, _, _ = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    assert o.shape == (1, 2, 19, dv)
    assert _rel(o, ref_o.numpy()) < 1e-12
    assert _rel(ot, ref_ot.numpy()) < 1e-12


@pytest.mark.parametrize("chunks", [1, 2, 4, 5])
def test_key_chunk_merge_equals_unsplit(chunks):
    q, k, v, qt, kt, vt = _case(N=61, seed=37)
    s = 0.33
    full = oracle.attn_jvp(q, k, v, qt, kt, vt, s)
    bounds = np.linspace(0, 61, chunks + 1).astype(int)
    parts = [oracle.attn_jvp(q, k[:, :, a:b], v[:, :, a:b], qt, kt[:, :, a:b], vt[:, :, a:b], s)
             for a, b in zip(bounds[:-1], bounds[1:])]
    merged = oracle.merge_chunks(*(np.stack([p[i] for p in parts]) for i in range(4)))
    for m, f in zip(merged, full):
        assert _rel(m, f) < 1e-12


def test_outlier_recipe_adds_exact_logit():
    x = inputs.make_inputs(1, 2, 200, 64, seed=5, dtype=torch.bfloat16, outlier_frac=0.01)
    q, k = x["q"].double(), x["k"].double()
    s = x["scale"]
    out = (k[..., 0] != 0)
    assert int(out.sum()) == 2 * 2
    assert torch.all(k[..., 0][out] * s == 12.0)
    assert torch.all(q[..., 0] == 1.0)
    assert torch.all(x["q_t"][..., 0] == 0) and torch.all(x["k_t"][..., 0] == 0)


def test_rounding_bound_covers_a_model_with_exactly_those_roundings():
    """The per-element Ot bound of oracle.attn_jvp_rounding_bound holds for an FP64 model
    that rounds P~ and H~ = P~ St to bf16 (unit roundoff 2^-8) before the value sums, on
    rows from diffuse to one-hot, and is not vacuous (the model's error reaches a fair
    share of it somewhere)."""
    import torch
    rng = np.random.default_rng(11)
    N, d = 300, 32
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()
    for qs in (1.0, 8.0, 40.0):
        q, k, v = rng.standard_normal((N, d)) * qs, rng.standard_normal((N, d)), rng.standard_normal((N, d))
        qt, kt, vt = (rng.standard_normal((N, d)) * 0.3 for _ in range(3))
        s = d ** -0.5
        ref = oracle.attn_jvp(q, k, v, qt, kt, vt, s)[1]
        S, St = s * q @ k.T, s * (qt @ k.T + q @ kt.T)
        Pt = np.exp(S - S.max(axis=1, keepdims=True))
        l = Pt.sum(axis=1, keepdims=True)
        O = bf(Pt) @ v / l
        T = (bf(Pt) @ vt + bf(Pt * St) @ v) / l
        model = T - ((Pt * St).sum(axis=1, keepdims=True) / l) * O
        bound = oracle.attn_jvp_rounding_bound(q, k, v, qt, kt, vt, s)
        ratio = np.abs(model - ref) / bound
        assert ratio.max() <= 1.0, (qs, ratio.max())
        assert ratio.max() >= 0.05, (qs, ratio.max())
