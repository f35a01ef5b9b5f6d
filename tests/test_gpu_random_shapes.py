"""GPU: seeded random shapes through the forward and the backward, against the
FP64 oracle.  A second seeded set draws the Q/K and the V head dims
independently from {16, 32, 64, 128, 256} (forward only); a third runs the
backward at head dim 256.

Batch, heads, query and key lengths (cross-attention included), head dims
16/32/64/128, both memory layouts and softmax scales of 0.5 to 2 times
d^-1/2 are drawn from a fixed seed.  Tile edges, ragged tails, the zero-padded
small head dims and strided layouts thus meet in combinations that the fixed
cases do not list.  Forward: relative L2 <= 1e-2 and max-abs <= 5e-2 RMS(ref)
for O, its tangent and mu; |LSE error| <= 1e-3.  Backward: relative L2 <= 1e-2
and, per element, the bound of its bf16 operands.  P and dS enter the tensor
cores rounded to bf16 (unit roundoff 2^-8), so an output element may be off by
2^-8 of the sum of its terms' sizes; the test allows 2^-7 of that sum (the
oracle's s |dS| |K|, s |dS|^T |Q| and P^T |dO|) plus 5e-2 RMS(ref).  A max-abs
bound relative to the RMS alone does not fit when few queries meet many keys.
There a handful of dK rows are 80x the RMS, and an FP64 model with only P and
dS rounded to bf16 is already 17 % of the RMS off at them.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, host64

pytestmark = pytest.mark.gpu

NAMES = inputs.NAMES


def _cases(n=16, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        nq = int(rng.integers(1, 600))
        nkv = nq if rng.random() < 0.5 else int(rng.integers(1, 900))
        d = int(rng.choice([16, 32, 64, 128]))
        layout = "bshd" if rng.random() < 0.5 else "bhsd"
        scale = float(d ** -0.5 * rng.uniform(0.5, 2.0))
        out.append((i, B, H, nq, nkv, d, layout, scale))
    return out


CASES = _cases()


def _cases_256(n=5, seed=2028):
    """Seeded backward shapes at head dim 256 (two CTAs per row tile)."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        nq = int(rng.integers(1, 500))
        nkv = nq if rng.random() < 0.5 else int(rng.integers(1, 700))
        scale = float(256 ** -0.5 * rng.uniform(0.5, 2.0))
        out.append((50 + i, B, H, nq, nkv, 256, "bhsd", scale))
    return out


def _inputs(i, B, H, nq, nkv, d):
    xq = inputs.make_inputs(B, H, nq, d, seed=100 + i, device="cuda", qk="rms", tangent_scale=0.3)
    xk = inputs.make_inputs(B, H, nkv, d, seed=200 + i, device="cuda", qk="rms", tangent_scale=0.3)
    return {"q": xq["q"], "q_t": xq["q_t"], "k": xk["k"], "v": xk["v"], "k_t": xk["k_t"], "v_t": xk["v_t"]}


def _forward(x, layout, scale):
    if layout == "bshd":
        args = [x[n].transpose(1, 2).contiguous() for n in NAMES]
        o, ot, lse, mu = binding.attn_jvp_fwd_strided(*args, layout="bshd", scale=scale)
        o, ot = o.transpose(1, 2), ot.transpose(1, 2)
    else:
        o, ot, lse, mu = binding.attn_jvp_fwd_strided(*(x[n] for n in NAMES), scale=scale)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    return o, ot, lse, mu


@pytest.mark.parametrize("case", CASES, ids=lambda c: "c%d-B%dH%d-q%d-k%d-d%d-%s" % c[:7])
def test_forward_random_shape(cuda_lib, case):
    i, B, H, nq, nkv, d, layout, scale = case
    x = _inputs(i, B, H, nq, nkv, d)
    o, ot, lse, mu = _forward(x, layout, scale)
    ref = oracle.attn_jvp(*(host64(x[n]) for n in NAMES), scale)
    assert_close(host64(o), ref[0], "O")
    assert_close(host64(ot), ref[1], "Ot")
    assert_close(host64(mu), ref[3], "mu")
    assert np.max(np.abs(host64(lse) - ref[2])) <= 1e-3


@pytest.mark.parametrize("case", CASES + _cases_256(), ids=lambda c: "c%d-B%dH%d-q%d-k%d-d%d-%s" % c[:7])
def test_backward_random_shape(cuda_lib, case):
    i, B, H, nq, nkv, d, layout, scale = case
    x = _inputs(i, B, H, nq, nkv, d)
    o, _, lse, _ = _forward(x, "bhsd", scale)
    g = torch.Generator(device="cuda").manual_seed(300 + i)
    dO = torch.randn(x["q"].shape, generator=g, device="cuda").to(torch.bfloat16)
    dq, dk, dv = binding.attn_bwd(x["q"], x["k"], x["v"], dO, o, lse, scale=scale)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for bh in range(B * H):
        b, h = divmod(bh, H)
        ref = oracle.attn_bwd_rows(host64(x["q"][b, h]), host64(x["k"][b, h]), host64(x["v"][b, h]),
                                   host64(dO[b, h]), scale, np.arange(nq), np.arange(nkv), with_scales=True)
        for name, got, want, size in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3], ref[3]):
            g = host64(got[b, h])
            rel = np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-300)
            assert rel <= 1e-2, "%s head %d: rel-L2 %.3e" % (name, bh, rel)
            excess = np.abs(g - want) - (2.0 ** -7 * size + 5e-2 * np.sqrt(np.mean(want ** 2)))
            assert np.all(excess <= 0), "%s head %d: %.3e over the operand bound" % (name, bh, excess.max())


def _dv_cases(n=12, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        nq = int(rng.integers(1, 500))
        nkv = int(rng.integers(1, 700))
        d, d_v = (int(v) for v in rng.choice([16, 32, 64, 128, 256], size=2))
        layout = "bshd" if rng.random() < 0.5 else "bhsd"
        out.append((i, B, H, nq, nkv, d, d_v, layout))
    return out


@pytest.mark.parametrize("case", _dv_cases(), ids=lambda c: "c%d-B%dH%d-q%d-k%d-d%d-dv%d-%s" % c)
def test_forward_random_value_head_dim(cuda_lib, case):
    # Q/K and V head dims drawn independently from the page's set
    i, B, H, nq, nkv, d, d_v, layout = case
    xq = inputs.make_inputs(B, H, nq, d, seed=400 + i, device="cuda", qk="rms", tangent_scale=0.3)
    xk = inputs.make_inputs(B, H, nkv, d, seed=500 + i, device="cuda", qk="rms", tangent_scale=0.3)
    xv = inputs.make_inputs(B, H, nkv, d_v, seed=600 + i, device="cuda", tangent_scale=0.3)
    args = [xq["q"], xk["k"], xv["v"], xq["q_t"], xk["k_t"], xv["v_t"]]
    if layout == "bshd":
        args = [t.transpose(1, 2).contiguous() for t in args]
    o, ot, lse, mu = binding.attn_jvp_fwd_strided(*args, layout=layout, scale=xq["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    if layout == "bshd":
        o, ot = o.transpose(1, 2), ot.transpose(1, 2)
    ref = oracle.attn_jvp(host64(xq["q"]), host64(xk["k"]), host64(xv["v"]), host64(xq["q_t"]),
                          host64(xk["k_t"]), host64(xv["v_t"]), xq["scale"])
    assert_close(host64(o), ref[0], "O")
    assert_close(host64(ot), ref[1], "Ot")
    assert_close(host64(mu), ref[3], "mu")
    assert np.max(np.abs(host64(lse) - ref[2])) <= 1e-3
