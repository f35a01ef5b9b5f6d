"""GPU parity: the sm_103a kernels (called through the C ABI) against the FP64 oracle.

Small cases are compared element by element on every row (they span several
query and key tiles and end in ragged tails); the full-size workloads are
compared on seeded samples of query rows (rows are independent, so the oracle
is exact on them) plus properties that hold at any size.
Tolerances (bf16 inputs, fp32 accumulation and outputs): relative L2 <= 1e-2
and max-abs <= 5e-2 x RMS(reference) for O, Ot and mu; |LSE error| <= 1e-3
(plus the derived input-rounding bound when the inputs are fp32).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_jvp_gb300 import binding, inputs
from helpers import LSE_ABS, assert_close, gpu_rows, host64, lse_tolerance, oracle_on, rel_l2

pytestmark = pytest.mark.gpu


def _run(x, **kw):
    out = binding.attn_jvp_fwd(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], scale=x["scale"], **kw)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    return out


def _check_all(x, got, heads=None, rows=None, kv=None):
    ref = oracle_on(x, heads=heads, rows=rows, kv=kv)
    B, H = x["q"].shape[:2]
    heads = list(range(B * H)) if heads is None else heads
    g = [gpu_rows(t, heads, rows) for t in got]
    errs = {}
    errs["O"] = assert_close(g[0], ref[0], "O")
    errs["Ot"] = assert_close(g[1], ref[1], "Ot")
    errs["mu"] = assert_close(g[3], ref[3], "mu")
    lse_err = np.abs(g[2] - ref[2])
    tol = lse_tolerance(x, heads, rows)
    assert np.all(lse_err <= tol), "LSE max-abs %.3e" % float(np.max(lse_err))
    errs["LSE_maxabs"] = float(np.max(lse_err))
    print("parity", tuple(x["q"].shape), {k: v for k, v in errs.items()})
    return errs


SMALL = [
    # (B, H, N, d, recipe extras)
    (1, 2, 256, 64, dict(dtype=torch.float32)),            # the tiny fp32 workload's shape
    (1, 2, 256, 128, {}),
    (2, 3, 129, 64, {}),                                   # one row past a query tile
    (1, 1, 1, 128, {}),                                    # single key and query
    (1, 1, 63, 64, {}),                                    # one partial key tile
    (1, 2, 1000, 128, dict(qk="rms", tangent_scale=0.3)),  # many key tiles, ragged tail
    (1, 1, 700, 64, dict(outlier_frac=0.01)),              # +12 logits: forces rescales
    (2, 1, 517, 128, dict(tangent="student_t3", tangent_scale=0.1)),
    # head dim 256: two CTAs per query tile, each with half of the value columns
    (1, 2, 300, 256, dict(qk="rms", tangent_scale=0.3)),
    (1, 1, 1, 256, {}),
    (2, 1, 129, 256, dict(outlier_frac=0.01)),
]


@pytest.mark.parametrize("B,H,N,d,extra", SMALL)
def test_small_cases_every_row(cuda_lib, B, H, N, d, extra):
    spec = dict(qk="normal", tangent="normal", tangent_scale=1.0, dtype=torch.bfloat16)
    spec.update(extra)
    x = inputs.make_inputs(B, H, N, d, seed=100 + N + d, device="cuda", **spec)
    got = _run(x)
    _check_all(x, got)


def test_fp32_inputs_through_the_c_abi(cuda_lib):
    """The tiny fp32 workload's device buffers go straight to attn_jvp_fwd and
    attn_jvp_fwd_chunk with ATTNJVP_FP32: the library rounds them to bf16 itself.
    Results match the oracle (on the original fp32 values, within the derived
    input-rounding bound) and equal, bit for bit, the bf16 path on inputs rounded
    to bf16 beforehand."""
    import ctypes
    lib = binding.load()
    x = inputs.workload_inputs("tiny", device="cuda")
    B, H, N, d = x["q"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
    out_t, lse, mu = torch.empty_like(out), torch.empty((B, H, N), device="cuda"), torch.empty((B, H, N), device="cuda")
    rc = lib.attn_jvp_fwd(*(p(x[n]) for n in inputs.NAMES), p(out), p(out_t), p(lse), p(mu), B, H, N, d,
                          ctypes.c_float(x["scale"]), binding.ATTNJVP_FP32, stream)
    assert rc == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    _check_all(x, (out, out_t, lse, mu))
    xb = dict(x, **{n: x[n].to(torch.bfloat16) for n in inputs.NAMES})
    ref = _run(xb)
    for got, want in zip((out, out_t, lse, mu), ref):
        assert torch.equal(got, want)
    # a key chunk, fp32 in
    a, n = 37, 150
    co, cot = torch.empty_like(out), torch.empty_like(out)
    cl, cm = torch.empty_like(lse), torch.empty_like(mu)
    rc = lib.attn_jvp_fwd_chunk(*(p(x[n_]) for n_ in inputs.NAMES), p(co), p(cot), p(cl), p(cm), B, H, N, d,
                                ctypes.c_float(x["scale"]), binding.ATTNJVP_FP32, a, n, stream)
    assert rc == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
    torch.cuda.synchronize()
    _check_all(x, (co, cot, cl, cm), kv=(a, n))
    # any other code is refused before anything runs
    assert lib.attn_jvp_fwd(*(p(x[n_]) for n_ in inputs.NAMES), p(out), p(out_t), p(lse), p(mu), B, H, N, d,
                            ctypes.c_float(x["scale"]), 5, stream) == binding.ATTNJVP_EINVAL


def test_tiny_workload_fp32_inputs(cuda_lib):
    # fp32 inputs are rounded to bf16 by the library's cast kernel; the oracle
    # sees the original fp32 values, so the error includes the input rounding.
    x = inputs.workload_inputs("tiny", device="cuda")
    assert x["q"].dtype == torch.float32
    got = _run(x)
    _check_all(x, got)


def test_scale_is_applied_to_scores_and_tangents(cuda_lib):
    x = inputs.make_inputs(1, 2, 300, 128, seed=7, device="cuda", scale=0.31)
    got = _run(x)
    _check_all(x, got)


def test_zero_tangents_give_exact_zero(cuda_lib):
    x = inputs.make_inputs(1, 3, 777, 128, seed=8, device="cuda")
    for n in ("q_t", "k_t", "v_t"):
        x[n] = torch.zeros_like(x[n])
    o, ot, lse, mu = _run(x)
    assert torch.all(ot == 0) and torch.all(mu == 0)


@pytest.mark.parametrize("d", [64, 256])
def test_deterministic(cuda_lib, d):
    x = inputs.make_inputs(1, 4, 1100, d, seed=9, device="cuda")
    a = _run(x)
    b = _run(x)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


def test_optional_row_outputs(cuda_lib):
    x = inputs.make_inputs(1, 1, 200, 128, seed=10, device="cuda")
    o, ot, lse, mu = binding.attn_jvp_fwd(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], want_rows=False)
    assert lse is None and mu is None
    o2, ot2, _, _ = _run(x)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(ot, ot2)


@pytest.mark.parametrize("N,d,chunks", [(1000, 128, 4), (611, 64, 3), (300, 128, 1), (700, 256, 3)])
def test_chunks_and_merge(cuda_lib, N, d, chunks):
    x = inputs.make_inputs(1, 2, N, d, seed=11 + chunks, device="cuda", qk="rms", tangent_scale=0.3)
    ws = binding.split_workspace(x["q"].shape, chunks, x["q"].device)
    merged = binding.attn_jvp_split(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], chunks,
                                    scale=x["scale"], workspace=ws)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    # each chunk's partials against the oracle restricted to that key range
    for c, (a, n) in enumerate(binding.chunk_bounds(N, chunks)):
        ref = oracle_on(x, kv=(a, n))
        assert_close(host64(ws[0][c].reshape(2, N, d)), ref[0], "O_c")
        assert_close(host64(ws[1][c].reshape(2, N, d)), ref[1], "Ot_c")
        assert float(np.max(np.abs(host64(ws[2][c].reshape(2, N)) - ref[2]))) <= LSE_ABS
    # the merge kernel against the oracle's merge of the same (GPU) partials: fp32 vs fp64
    om = oracle.merge_chunks(*(host64(w) for w in ws))
    for g, r, name in zip(merged, om, ("O", "Ot", "LSE", "mu")):
        assert rel_l2(host64(g), r) < 1e-5, name
    # the merged result against the unsplit oracle
    _check_all(x, merged)


def test_trigflow_tangent_matches_oracle(cuda_lib):
    gen = torch.Generator(device="cuda").manual_seed(12)
    B, M = 5, 16 * 21 * 30 * 52 + 3
    x0 = torch.randn((B, M), generator=gen, device="cuda")
    eps = torch.randn((B, M), generator=gen, device="cuda")
    t = torch.tensor([0.0, 0.25, 0.8, math.atan(80.0), math.pi / 2], dtype=torch.float64, device="cuda")
    out = binding.trigflow_tangent(x0, eps, t)
    torch.cuda.synchronize()
    ref = oracle.trigflow_tangent(host64(x0), host64(eps), host64(t))
    err = np.abs(host64(out) - ref)
    bound = 4 * 2.0 ** -24 * (np.abs(host64(x0)) + np.abs(host64(eps))) + 1e-30
    assert np.all(err <= bound)
    # in place on x0
    x0c = x0.clone()
    binding.trigflow_tangent(x0c, eps, t, out=x0c)
    torch.cuda.synchronize()
    assert torch.equal(x0c, out)


def test_cast_is_round_to_nearest_even(cuda_lib):
    gen = torch.Generator(device="cuda").manual_seed(13)
    x = torch.randn(1 << 20 | 3, generator=gen, device="cuda") * 100
    got = binding.attn_jvp_cast_f32_bf16(x)
    torch.cuda.synchronize()
    ref = x.cpu().to(torch.bfloat16)
    assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
def _sampled(name, n_heads=4, n_rows=96):
    spec = inputs.WORKLOADS[name]
    B, H, N = spec["B"], spec["H"], spec["N"]
    gen = np.random.default_rng(spec["seed"])
    heads = sorted(set([0, B * H - 1] + list(gen.choice(B * H, size=n_heads, replace=False))))
    rows = inputs.sample_rows(N, n_rows, spec["seed"]).numpy()
    # include the last query tile's ragged tail
    rows = np.unique(np.concatenate([rows, np.arange(max(0, N - 5), N)]))
    return heads, rows


@pytest.mark.parametrize("name", ["image_dit_1k", "video_dit", "stress"])
def test_full_size_workload_sampled_rows(cuda_lib, name):
    x = inputs.workload_inputs(name, device="cuda")
    got = _run(x)
    heads, rows = _sampled(name)
    _check_all(x, got, heads=heads, rows=rows)
    for t in got:
        assert bool(torch.isfinite(t).all())
    del x, got
    torch.cuda.empty_cache()


def test_long_video_split_kv_sampled_rows(cuda_lib):
    spec = inputs.WORKLOADS["long_video"]
    x = inputs.workload_inputs("long_video", device="cuda")
    got = binding.attn_jvp_split(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], spec["kv_chunks"],
                                 scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    heads, rows = _sampled("long_video", n_heads=2, n_rows=48)
    _check_all(x, got, heads=heads, rows=rows)
    del x, got
    torch.cuda.empty_cache()


def test_head_dim_256_long_sequence_sampled_rows(cuda_lib):
    # Two CTAs per query tile and the half-tile K ring over 256 key tiles: seeded
    # query rows of every head (plus the ragged last tile) against the oracle.
    x = inputs.make_inputs(1, 3, 16380, 256, seed=61, device="cuda", qk="rms", tangent_scale=0.3)
    got = _run(x)
    rng = np.random.default_rng(62)
    rows = np.unique(np.concatenate([rng.choice(16380, 40, replace=False), np.arange(16375, 16380)]))
    _check_all(x, got, heads=[0, 1, 2], rows=rows)
    for t in got:
        assert bool(torch.isfinite(t).all())
    del x, got
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# degenerate cases of the method and the largest key counts
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("d", [64, 128, 256])
def test_uniform_attention_when_queries_are_zero(cuda_lib, d):
    """Q = 0 makes every score 0: P is uniform over the N keys, so O = mean(V),
    LSE = ln N exactly, mu = mean_j St_ij = s q_t . mean(K) (q = 0), and
    Ot = mean(Vt) + mean_j (St_ij - mu) v_j."""
    x = inputs.make_inputs(1, 2, 777, d, seed=71, device="cuda", tangent_scale=0.5)
    x["q"] = torch.zeros_like(x["q"])
    got = _run(x)
    _check_all(x, got)
    N = x["q"].shape[2]
    assert np.max(np.abs(host64(got[2]) - np.log(N))) <= 1e-5 * np.log(N)
    o_ref = host64(x["v"]).mean(axis=2)
    assert np.max(np.abs(host64(got[0]) - o_ref[:, :, None, :])) <= 1e-4 * np.abs(o_ref).max() + 1e-6


@pytest.mark.parametrize("d", [64, 128])
def test_one_hot_softmax_from_huge_logits(cuda_lib, d):
    """Queries scaled by 60: scores spread over hundreds of log units, so most rows'
    softmax is one-hot up to underflow and the online rescale fires often.  Nothing
    may overflow into inf or NaN; O, mu and LSE keep the usual tolerances.

    Ot does not, and cannot: as on the page (section 前向: p and H~ are cast to the
    value dtype before the dot products), P~ and H~ = P~ (.) St enter the value GEMMs
    rounded to bf16 (unit roundoff u = 2^-8), and Ot = T / l - mu O.  In a one-hot row
    |mu| is the dominant key's |St|, far above |Ot|, so the rounding of H~ and of P~
    in O shows at its full size.  Each element of Ot is held to that arithmetic's
    bound, u sum_j P_ij (|vt_jc| + (|St_ij| + |mu_i|) |v_jc|), from exact FP64
    quantities, plus the usual 5e-2 RMS."""
    x = inputs.make_inputs(1, 2, 640, d, seed=72, device="cuda", tangent_scale=0.2)
    x["q"] = (x["q"].float() * 60.0).to(torch.bfloat16)
    got = _run(x)
    for t in got:
        assert bool(torch.isfinite(t).all())
    ref = oracle_on(x)
    g = [gpu_rows(t, [0, 1]) for t in got]
    assert_close(g[0], ref[0], "O")
    assert_close(g[3], ref[3], "mu")
    assert np.max(np.abs(g[2] - ref[2])) <= LSE_ABS
    heads = [host64(x[n])[0] for n in ("q", "k", "v", "q_t", "k_t", "v_t")]
    bound = np.stack([oracle.attn_jvp_rounding_bound(*(t[h] for t in heads), x["scale"]) for h in range(2)])
    rms = np.sqrt(np.mean(ref[1] ** 2))
    excess = np.abs(g[1] - ref[1]) - (bound + 5e-2 * rms)
    assert np.all(excess <= 0), "Ot: %.3e over the rounding bound" % excess.max()
    print("one-hot d=%d: Ot max error / bound %.3f, rel-L2 %.3e" % (
        d, float(np.max(np.abs(g[1] - ref[1]) / (bound + 5e-2 * rms))), rel_l2(g[1], ref[1])))


@pytest.mark.parametrize("d", [64, 128])
def test_quarter_million_keys_sampled_rows(cuda_lib, d):
    """One head over 262144 keys (4096 key tiles per CTA, 2048 query tiles), the
    longest sequence here: seeded sampled rows and the last rows against the oracle;
    sums over every key of a row stay within the usual tolerances."""
    N = 1 << 18
    x = inputs.make_inputs(1, 1, N, d, seed=73, device="cuda", qk="rms", tangent_scale=0.3)
    got = _run(x)
    rows = np.unique(np.concatenate([inputs.sample_rows(N, 24, 74).numpy(), np.arange(N - 3, N)]))
    _check_all(x, got, heads=[0], rows=rows)
    del x, got
    torch.cuda.empty_cache()
