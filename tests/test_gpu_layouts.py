"""GPU: strided layouts, cross-attention (N_q != N_kv) and head dims 16/32/256
through attn_jvp_fwd_strided, against the FP64 oracle and, where the same
numbers go through the contiguous path, bit for bit against it.

The kernel computes each (batch, head, query tile) independently of where its
rows sit in memory, so a layout change must not change a single bit; cross-
attention and the small head dims (zero-padded to 64 columns on chip) are
compared with the oracle at the usual tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, host64

pytestmark = pytest.mark.gpu

NAMES = inputs.NAMES


def _sync():
    torch.cuda.synchronize()
    binding.attn_jvp_status()


def _contig(x):
    res = binding.attn_jvp_fwd(*(x[n] for n in NAMES), scale=x["scale"])
    _sync()
    return res


def _oracle(xq, xk, scale, kv=None):
    """Oracle on [B, H, N, d] tensors (queries from ``xq``, keys/values from ``xk``)."""
    k, v, kt, vt = (host64(xk[n]) for n in ("k", "v", "k_t", "v_t"))
    if kv is not None:
        a, n = kv
        k, v, kt, vt = (t[:, :, a:a + n] for t in (k, v, kt, vt))
    return oracle.attn_jvp(host64(xq["q"]), k, v, host64(xq["q_t"]), kt, vt, scale)


def _check(got, ref):
    assert_close(host64(got[0]), ref[0], "O")
    assert_close(host64(got[1]), ref[1], "Ot")
    assert_close(host64(got[3]), ref[3], "mu")
    assert np.max(np.abs(host64(got[2]) - ref[2])) <= 1e-3


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bshd_layout_is_bit_identical_to_contiguous(cuda_lib, d):
    x = inputs.make_inputs(2, 3, 300, d, seed=21, device="cuda", qk="rms", tangent_scale=0.3)
    ref = _contig(x)
    xs = {n: x[n].transpose(1, 2).contiguous() for n in NAMES}  # [B, S, H, D]
    got = binding.attn_jvp_fwd_strided(*(xs[n] for n in NAMES), layout="bshd", scale=x["scale"])
    _sync()
    assert torch.equal(got[0].transpose(1, 2), ref[0]) and torch.equal(got[1].transpose(1, 2), ref[1])
    assert torch.equal(got[2], ref[2]) and torch.equal(got[3], ref[3])


@pytest.mark.parametrize("d,d_v", [(64, 64), (128, 256), (32, 128)])
def test_fp32_strided_inputs_equal_the_bf16_path(cuda_lib, d, d_v):
    """fp32 inputs in the page's [B, S, H, D] layout (packed-QKV views for the
    queries and keys, head strides that are multiples of 4 but not 8 elements) are
    gathered and rounded to bf16 inside the library: the result equals, bit for
    bit, the bf16 path on inputs rounded beforehand, and matches the oracle."""
    B, H, Nq, Nkv = 2, 3, 200, 333
    gen = torch.Generator(device="cuda").manual_seed(27 + d + d_v)
    # [B, S, 2, H, d + 4] buffers: slot 0 holds the primal, slot 1 its tangent, so
    # both views share one set of strides; the head stride d + 4 is a multiple of 4
    # elements but not of 8.
    qk = torch.randn((B, Nq, 2, H, d + 4), generator=gen, device="cuda")
    kk = torch.randn((B, Nkv, 2, H, d + 4), generator=gen, device="cuda")
    vv = torch.randn((B, Nkv, 2, H, d_v), generator=gen, device="cuda")
    qk[:, :, 1] *= 0.3
    kk[:, :, 1] *= 0.3
    xs = [qk[:, :, 0, :, :d], kk[:, :, 0, :, :d], vv[:, :, 0], qk[:, :, 1, :, :d], kk[:, :, 1, :, :d], vv[:, :, 1]]
    scale = d ** -0.5
    got = binding.attn_jvp_fwd_strided(*xs, layout="bshd", scale=scale)
    _sync()
    ref = binding.attn_jvp_fwd_strided(*(t.to(torch.bfloat16) for t in xs), layout="bshd", scale=scale)
    _sync()
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
    to_bhsd = lambda t: t.transpose(1, 2)
    xo = {"q": to_bhsd(xs[0]), "k": to_bhsd(xs[1]), "v": to_bhsd(xs[2]), "q_t": to_bhsd(xs[3]),
          "k_t": to_bhsd(xs[4]), "v_t": to_bhsd(xs[5])}
    want = _oracle(xo, xo, scale)
    assert_close(host64(to_bhsd(got[0])), want[0], "O")
    assert_close(host64(to_bhsd(got[1])), want[1], "Ot")


def test_packed_qkv_views_are_bit_identical(cuda_lib):
    B, H, S, d = 1, 4, 257, 128
    x = inputs.make_inputs(B, H, S, d, seed=22, device="cuda", tangent_scale=0.5)
    ref = _contig(x)
    packed = torch.empty((B, S, 3, H, d), dtype=torch.bfloat16, device="cuda")
    packed_t = torch.empty_like(packed)
    for i, (p, pt) in enumerate((("q", "q_t"), ("k", "k_t"), ("v", "v_t"))):
        packed[:, :, i] = x[p].transpose(1, 2)
        packed_t[:, :, i] = x[pt].transpose(1, 2)
    views = [packed[:, :, 0], packed[:, :, 1], packed[:, :, 2], packed_t[:, :, 0], packed_t[:, :, 1],
             packed_t[:, :, 2]]
    got = binding.attn_jvp_fwd_strided(*views, layout="bshd", scale=x["scale"])
    _sync()
    assert torch.equal(got[0].transpose(1, 2), ref[0]) and torch.equal(got[1].transpose(1, 2), ref[1])


@pytest.mark.parametrize("nq,nkv,d,layout", [(300, 1000, 64, "bhsd"), (1000, 77, 128, "bhsd"),
                                              (129, 640, 128, "bshd"), (1, 5, 64, "bhsd"),
                                              (300, 1000, 256, "bshd"), (77, 130, 256, "bhsd")])
def test_cross_attention_against_oracle(cuda_lib, nq, nkv, d, layout):
    xq = inputs.make_inputs(2, 2, nq, d, seed=30 + nq, device="cuda", qk="rms", tangent_scale=0.3)
    xk = inputs.make_inputs(2, 2, nkv, d, seed=31 + nkv, device="cuda", qk="rms", tangent_scale=0.3)
    args = [xq["q"], xk["k"], xk["v"], xq["q_t"], xk["k_t"], xk["v_t"]]
    if layout == "bshd":
        args = [t.transpose(1, 2).contiguous() for t in args]
    got = binding.attn_jvp_fwd_strided(*args, layout=layout, scale=xq["scale"])
    _sync()
    if layout == "bshd":
        got = (got[0].transpose(1, 2), got[1].transpose(1, 2), got[2], got[3])
    _check(got, _oracle(xq, xk, xq["scale"]))


@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_small_head_dims_against_oracle(cuda_lib, d, layout):
    x = inputs.make_inputs(2, 3, 333, d, seed=40 + d, device="cuda", tangent_scale=0.5)
    if layout == "bhsd":
        got = binding.attn_jvp_fwd(*(x[n] for n in NAMES), scale=x["scale"])
    else:
        xs = [x[n].transpose(1, 2).contiguous() for n in NAMES]
        got = binding.attn_jvp_fwd_strided(*xs, layout="bshd", scale=x["scale"])
        got = (got[0].transpose(1, 2), got[1].transpose(1, 2), got[2], got[3])
    _sync()
    assert got[0].shape[-1] == d
    _check(got, _oracle(x, x, x["scale"]))


def test_strided_key_split_merges_to_the_full_result(cuda_lib):
    B, H, nq, nkv, d = 1, 3, 200, 700, 128
    xq = inputs.make_inputs(B, H, nq, d, seed=51, device="cuda", qk="rms", tangent_scale=0.3)
    xk = inputs.make_inputs(B, H, nkv, d, seed=52, device="cuda", qk="rms", tangent_scale=0.3)
    args = [t.transpose(1, 2).contiguous() for t in (xq["q"], xk["k"], xk["v"], xq["q_t"], xk["k_t"], xk["v_t"])]
    full = binding.attn_jvp_fwd_strided(*args, layout="bshd", scale=xq["scale"])
    bounds = binding.chunk_bounds(nkv, 3)
    ws = binding.split_workspace((B, H, nq, d), 3, "cuda")
    for c, (a, n) in enumerate(bounds):
        # partials in [B, H, N_q, d] order: views of the bshd-shaped outputs
        binding.attn_jvp_fwd_strided(*args, layout="bshd", scale=xq["scale"], out=ws[0][c].transpose(1, 2),
                                     out_t=ws[1][c].transpose(1, 2), lse=ws[2][c], mu=ws[3][c], kv_start=a,
                                     kv_len=n)
    merged = binding.attn_jvp_merge(*ws)
    _sync()
    # Each chunk normalises P~ against its own running max before rounding it to
    # bf16, so merged and unsplit results differ at bf16 level: both are held to
    # the oracle.
    ref = _oracle(xq, xk, xq["scale"])
    _check(merged, ref)
    _check((full[0].transpose(1, 2), full[1].transpose(1, 2), full[2], full[3]), ref)
    # one chunk against the oracle over its key range
    a, n = bounds[1]
    part = binding.attn_jvp_fwd_strided(*args, layout="bshd", scale=xq["scale"], kv_start=a, kv_len=n)
    _sync()
    _check((part[0].transpose(1, 2), part[1].transpose(1, 2), part[2], part[3]),
           _oracle(xq, xk, xq["scale"], kv=(a, n)))


def test_padded_output_rows_leave_the_padding_untouched(cuda_lib):
    x = inputs.make_inputs(1, 2, 150, 64, seed=61, device="cuda")
    ref = _contig(x)
    big = torch.full((1, 2, 150, 64 + 12), float("nan"), dtype=torch.float32, device="cuda")
    big_t = torch.full_like(big, float("nan"))
    got = binding.attn_jvp_fwd_strided(*(x[n] for n in NAMES), scale=x["scale"], out=big[..., :64],
                                       out_t=big_t[..., :64])
    _sync()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert torch.isnan(big[..., 64:]).all() and torch.isnan(big_t[..., 64:]).all()


@pytest.mark.parametrize("d,d_v,layout,nq,nkv", [
    (64, 128, "bhsd", 300, 700), (128, 64, "bshd", 129, 640), (32, 128, "bhsd", 200, 333),
    (128, 256, "bshd", 300, 300), (256, 64, "bhsd", 77, 200), (256, 128, "bhsd", 150, 150),
    (64, 256, "bshd", 100, 500), (16, 32, "bhsd", 333, 333), (128, 16, "bshd", 100, 260)])
def test_value_head_dim_of_its_own_against_oracle(cuda_lib, d, d_v, layout, nq, nkv):
    # The page's forward takes V with d_v columns per head: O and its tangent
    # then have d_v columns, the scores still d.
    xq = inputs.make_inputs(2, 2, nq, d, seed=50 + d, device="cuda", qk="rms", tangent_scale=0.3)
    xk = inputs.make_inputs(2, 2, nkv, d, seed=51 + nkv, device="cuda", qk="rms", tangent_scale=0.3)
    xv = inputs.make_inputs(2, 2, nkv, d_v, seed=52 + d_v, device="cuda", tangent_scale=0.3)
    args = [xq["q"], xk["k"], xv["v"], xq["q_t"], xk["k_t"], xv["v_t"]]
    if layout == "bshd":
        args = [t.transpose(1, 2).contiguous() for t in args]
    got = binding.attn_jvp_fwd_strided(*args, layout=layout, scale=xq["scale"])
    _sync()
    if layout == "bshd":
        got = (got[0].transpose(1, 2), got[1].transpose(1, 2), got[2], got[3])
    assert got[0].shape == (2, 2, nq, d_v)
    ref = oracle.attn_jvp(host64(xq["q"]), host64(xk["k"]), host64(xv["v"]), host64(xq["q_t"]),
                          host64(xk["k_t"]), host64(xv["v_t"]), xq["scale"])
    _check(got, ref)
