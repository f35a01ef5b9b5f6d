"""Pins for the oracle's primal attention backward (section 反向, backward, of
the page "带分数正则的一致性蒸馏"): dV = P^T dO, dP = dO V^T,
dS = P (.) (dP - rowsum(dP (.) P)), dQ = s dS K, dK = s dS^T Q.

Pinned against library autodiff (torch.autograd of naive FP64 attention), a
central finite difference of <O, dO>, and closed forms: one key (P = 1), the
key-shift invariance of softmax (sum_j dK_j = 0), and the identity
rowsum(dP (.) P) = rowsum(dO (.) O) that the GPU path relies on.
"""
import numpy as np
import pytest
import torch

import oracle


def _rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _case(B=2, H=2, Nq=17, Nk=23, d=16, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d))
    k = rng.standard_normal((B, H, Nk, d))
    v = rng.standard_normal((B, H, Nk, d))
    dO = rng.standard_normal((B, H, Nq, d))
    return q, k, v, dO


def _torch_attn(q, k, v, s):
    return torch.matmul(torch.softmax(torch.matmul(q, k.transpose(-1, -2)) * s, dim=-1), v)


@pytest.mark.parametrize("nq,nk", [(17, 23), (23, 17), (32, 32)])
def test_backward_matches_autograd(nq, nk):
    q, k, v, dO = _case(Nq=nq, Nk=nk, seed=nq + nk)
    s = 0.31
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    _torch_attn(tq, tk, tv, s).backward(torch.from_numpy(dO))
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, s)
    assert _rel(dq, tq.grad.numpy()) < 1e-12
    assert _rel(dk, tk.grad.numpy()) < 1e-12
    assert _rel(dv, tv.grad.numpy()) < 1e-12


def test_backward_matches_central_difference():
    q, k, v, dO = _case(B=1, H=1, seed=3)
    s = 0.25
    rng = np.random.default_rng(4)
    dirs = [rng.standard_normal(x.shape) for x in (q, k, v)]
    zero = np.zeros_like(q)
    loss = lambda q_, k_, v_: float((oracle.attn_jvp(q_, k_, v_, zero, np.zeros_like(k), np.zeros_like(v), s)[0]
                                     * dO).sum())
    h = 1e-6
    fd = (loss(q + h * dirs[0], k + h * dirs[1], v + h * dirs[2])
          - loss(q - h * dirs[0], k - h * dirs[1], v - h * dirs[2])) / (2 * h)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, s)
    analytic = float((dq * dirs[0]).sum() + (dk * dirs[1]).sum() + (dv * dirs[2]).sum())
    assert abs(fd - analytic) <= 1e-7 * max(1.0, abs(analytic))


def test_single_key_closed_form():
    # One key: P = 1, so dS = 0 (dQ = dK = 0) and dV is the sum of dO over the queries.
    q, k, v, dO = _case(Nk=1, seed=5)
    dq, dk, dv = oracle.attn_bwd(q, k, v, dO, 0.4)
    assert np.all(dq == 0) and np.all(dk == 0)
    assert _rel(dv, dO.sum(axis=2, keepdims=True)) < 1e-14


def test_key_shift_invariance():
    # Adding one vector to every key shifts each score row by a constant, which
    # softmax ignores: the gradient along that shift, sum_j dK_j, vanishes.
    q, k, v, dO = _case(seed=6)
    _, dk, _ = oracle.attn_bwd(q, k, v, dO, 0.3)
    scale_ref = np.abs(dk).sum(axis=2).max()
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12 * max(scale_ref, 1.0)


def test_rowsum_identity_used_by_the_gpu_path():
    # rowsum(dP (.) P) = sum_j P_ij (dO_i . v_j) = dO_i . O_i
    q, k, v, dO = _case(seed=7)
    s = 0.27
    z = np.zeros_like
    o = oracle.attn_jvp(q, k, v, z(q), z(k), z(v), s)[0]
    P = torch.softmax(torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * s, dim=-1).numpy()
    dP = dO @ np.swapaxes(v, -1, -2)
    assert _rel((dP * P).sum(-1), (dO * o).sum(-1)) < 1e-13


@pytest.mark.parametrize("nq,nk,d", [(37, 53, 16), (64, 19, 32), (130, 130, 8)])
def test_sampled_rows_match_the_full_head(nq, nk, d):
    # The sampled-row oracle (numpy, blocked over queries) against the full-head
    # one (C) on every row; a block smaller than Nq exercises the blocking.
    q, k, v, dO = (x[0, 0] for x in _case(B=1, H=1, Nq=nq, Nk=nk, d=d, seed=nq * nk))
    s = 0.4
    rq, rk, rv = oracle.attn_bwd(q, k, v, dO, s)
    gq, gk, gv = oracle.attn_bwd_rows(q, k, v, dO, s, np.arange(nq), np.arange(nk), block=16)
    assert _rel(gq, rq) < 1e-12 and _rel(gk, rk) < 1e-12 and _rel(gv, rv) < 1e-12
    sub_q, sub_k = [nq - 1, 0, nq // 2], [nk // 3, nk - 1]
    hq, hk, hv = oracle.attn_bwd_rows(q, k, v, dO, s, sub_q, sub_k)
    assert np.allclose(hq, rq[sub_q], rtol=1e-12, atol=1e-14)
    assert np.allclose(hk, rk[sub_k], rtol=1e-12, atol=1e-14)
    assert np.allclose(hv, rv[sub_k], rtol=1e-12, atol=1e-14)
    # the size of each sum bounds the sum itself (triangle inequality)
    *_, (sq, sk, sv) = oracle.attn_bwd_rows(q, k, v, dO, s, sub_q, sub_k, with_scales=True)
    for size, val in ((sq, hq), (sk, hk), (sv, hv)):
        assert np.all(size >= np.abs(val) * (1 - 1e-12)) and np.all(size > 0)

