"""GPU: the output side of one consistency step (trigflow_output_jvp and
scm_tangent_loss) against the FP64 oracle on the same fp32 inputs.

The GPU forms the per-frame coefficients in FP64 and does the elementwise
arithmetic in fp32 (the page's tensors are fp32), so results carry fp32
rounding: F to ~1e-6 relative; its tangent and g, which subtract nearly equal
terms, to ~1e-5.  The norms and the loss are FP64 sums of those fp32 values.
NaN masks are exact.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_jvp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _rel(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _latent(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * scale


def _times(B, T, seed, lo=0.2, hi=1.5):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.rand((B, T), generator=g, device="cuda", dtype=torch.float64) * (hi - lo) + lo)


def _np(t):
    return t.detach().cpu().double().numpy()


# (B, C, T, H, W): a video latent (21 frames of 30 x 52), a ragged small case, one frame
SHAPES = [(2, 16, 21, 30, 52), (3, 2, 5, 7, 3), (1, 4, 1, 9, 11)]


@pytest.mark.parametrize("shape", SHAPES)
def test_output_jvp_against_oracle(cuda_lib, shape):
    B, C, T = shape[:3]
    x, n, xt, nt = (_latent(shape, 10 + i) for i in range(4))
    t, tt = _times(B, T, 20), _times(B, T, 21, -1.0, 1.0)
    F, Ft = binding.trigflow_output_jvp(x, n, xt, nt, t, tt)
    torch.cuda.synchronize()
    rF, rFt = oracle.process_output_jvp(_np(x), _np(n), _np(xt), _np(nt), _np(t), _np(tt))
    assert _rel(_np(F), rF) < 2e-6
    assert _rel(_np(Ft), rFt) < 2e-5


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("r", [0.0, 0.37, 1.0])
def test_scm_tangent_loss_against_oracle(cuda_lib, shape, r):
    B, C, T = shape[:3]
    F = _latent(shape, 30)
    Fsg = F.clone()                       # the stop-gradient copy: equal values
    Ftc, x, Ft = _latent(shape, 31), _latent(shape, 32), _latent(shape, 33, 0.5)
    t = _times(B, T, 34, 0.05, 1.55)
    g, dfdt, loss, ng, nf = binding.scm_tangent_loss(F, Fsg, Ftc, x, Ft, t, r)
    torch.cuda.synchronize()
    rg, rd, rl, rng, rnf = oracle.scm_tangent_loss(_np(F), _np(Fsg), _np(Ftc), _np(x), _np(Ft), _np(t), r)
    assert _rel(_np(g), rg) < 1e-5
    assert _rel(_np(dfdt), rd) < 2e-6
    assert np.max(np.abs(_np(loss) - rl) / rl) < 2e-5
    assert not ng.any().item() and not nf.any().item()


def test_scm_loss_with_student_gap_and_nan_masks(cuda_lib):
    shape = (4, 3, 6, 10, 10)
    F, Fsg, Ftc, x, Ft = (_latent(shape, 40 + i) for i in range(5))  # F_theta != F_sg here
    t = _times(4, 6, 45)
    F[1, 2, 3, 4, 5] = float("nan")       # student NaN in sample 1
    Ft[3, 0, 0, 0, 0] = float("nan")      # tangent NaN -> g NaN in sample 3
    g, dfdt, loss, ng, nf = binding.scm_tangent_loss(F, Fsg, Ftc, x, Ft, t, 0.8)
    torch.cuda.synchronize()
    rg, rd, rl, rng, rnf = oracle.scm_tangent_loss(_np(F), _np(Fsg), _np(Ftc), _np(x), _np(Ft), _np(t), 0.8)
    assert ng.cpu().tolist() == rng.tolist() == [False, False, False, True]
    assert nf.cpu().tolist() == rnf.tolist() == [False, True, False, False]
    gl = _np(loss)
    assert gl[1] == 0.0 and gl[3] == 0.0
    assert np.all(_np(g)[[1, 3]] == 0)
    ok = [0, 2]
    assert _rel(_np(g)[ok], rg[ok]) < 1e-5
    assert np.max(np.abs(gl[ok] - rl[ok]) / rl[ok]) < 2e-5
    # df_dt is not masked: NaN only where its inputs are
    d = _np(dfdt)
    assert np.isnan(d[3, 0, 0, 0, 0]) and np.isnan(d).sum() == 1
    assert _rel(np.nan_to_num(d[:3]), rd[:3]) < 2e-6


def test_scm_tangent_loss_is_reproducible(cuda_lib):
    shape = (2, 16, 21, 30, 52)
    args = [_latent(shape, 50 + i) for i in range(5)]
    t = _times(2, 21, 55)
    a = binding.scm_tangent_loss(*args, t, 0.5)
    b = binding.scm_tangent_loss(*args, t, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2])


def test_scm_tangent_loss_with_a_dirty_reused_workspace(cuda_lib):
    # Many small samples (one item each, so most normalisation items wait on
    # their sample), a workspace holding garbage, and the same workspace twice.
    shape = (9, 1, 2, 1, 4)
    F, Fsg, Ftc, x, Ft = (_latent(shape, 60 + i) for i in range(5))
    t = _times(9, 2, 65)
    F[4, 0, 1, 0, 2] = float("nan")
    ws = binding.scm_workspace(shape[:3] + (4,), torch.device("cuda"))
    ws.fill_(float("nan"))
    rg, rd, rl, rng, rnf = oracle.scm_tangent_loss(_np(F), _np(Fsg), _np(Ftc), _np(x), _np(Ft), _np(t), 0.25)
    for _ in range(2):
        g, dfdt, loss, ng, nf = binding.scm_tangent_loss(F, Fsg, Ftc, x, Ft, t, 0.25, workspace=ws)
        torch.cuda.synchronize()
        assert nf.cpu().tolist() == rnf.tolist() and not ng.any().item()
        ok = [b for b in range(9) if b != 4]
        assert _rel(_np(g)[ok], rg[ok]) < 1e-5
        assert np.all(_np(g)[4] == 0) and _np(loss)[4] == 0.0
        assert np.max(np.abs(_np(loss)[ok] - rl[ok]) / rl[ok]) < 2e-5


def test_output_side_on_the_benchmarked_video_batch(cuda_lib):
    # The batch bench.py times: 33 video latents [33, 16, 21, 6240], 69.2 M
    # elements per tensor; scm_tangent_loss runs with the persistent grid's
    # ticket lag in its steady state (33 samples, eight ahead).
    b = inputs.epilogue_batch("video_dit", device="cuda")
    x, n, xt, nt, t, tt = (b[k] for k in ("x", "n", "x_t", "n_t", "t", "t_t"))
    F, Ft = binding.trigflow_output_jvp(x, n, xt, nt, t, tt)
    g, dfdt, loss, ng, nf = binding.scm_tangent_loss(F, x, n, xt, Ft, t, 0.5)
    torch.cuda.synchronize()
    rF, rFt = oracle.process_output_jvp(_np(x), _np(n), _np(xt), _np(nt), _np(t), _np(tt))
    assert _rel(_np(F), rF) < 2e-6
    assert _rel(_np(Ft), rFt) < 2e-5
    del rF, rFt
    rg, rd, rl, rng, rnf = oracle.scm_tangent_loss(_np(F), _np(x), _np(n), _np(xt), _np(Ft), _np(t), 0.5)
    assert not ng.any().item() and not nf.any().item() and not rng.any() and not rnf.any()
    assert _rel(_np(g), rg) < 1e-5
    assert _rel(_np(dfdt), rd) < 2e-6
    assert np.max(np.abs(_np(loss) - rl) / rl) < 2e-5


def _random_epilogue_cases(n=10, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(rng.choice([1, 2, 7, 9, 17, 50]))
        C = int(rng.integers(1, 5))
        T = int(rng.integers(1, 6))
        HW = int(rng.choice([1, 3, 4, 37, 64, 1000, 4097, 8200]))
        out.append((i, B, C, T, HW, float(rng.uniform(0, 1)), bool(rng.random() < 0.3), bool(rng.random() < 0.4)))
    return out


@pytest.mark.parametrize("case", _random_epilogue_cases(), ids=lambda c: "c%d-B%dC%dT%dHW%d" % c[:5])
def test_output_side_random_shapes(cuda_lib, case):
    # Seeded batch sizes around the fused sCM pass's eight-sample ticket lag,
    # rows that take the 16-byte path or the scalar one (HW % 4, or tensors
    # offset by one element), and scattered NaNs.
    i, B, C, T, HW, r, offset, nans = case
    shape = (B, C, T, HW)
    n = B * C * T * HW

    def lat(seed, scale=1.0):
        base = _latent((n + 1,), seed, scale)
        return (base[1:] if offset else base[:n]).view(shape)

    x, nn, xt, nt = lat(70 + i), lat(80 + i), lat(90 + i), lat(100 + i)
    t = _times(B, T, 110 + i, 0.05, 1.55)
    tt = _times(B, T, 120 + i, -1.0, 1.0)
    F, Ft = binding.trigflow_output_jvp(x, nn, xt, nt, t, tt)
    Fsg, Ftc = lat(130 + i), lat(140 + i)
    if nans:
        flat = Fsg.view(-1)
        flat[(np.arange(3) * 7919 + i) % n] = float("nan")  # F_sg NaN: g of those elements
    g, dfdt, loss, ng, nf = binding.scm_tangent_loss(F, Fsg, Ftc, x, Ft, t, r)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    rF, rFt = oracle.process_output_jvp(_np(x), _np(nn), _np(xt), _np(nt), _np(t), _np(tt))
    assert _rel(_np(F), rF) < 2e-6
    assert _rel(_np(Ft), rFt) < 2e-5
    rg, rd, rl, rng_, rnf = oracle.scm_tangent_loss(_np(F), _np(Fsg), _np(Ftc), _np(x), _np(Ft), _np(t), r)
    assert ng.cpu().tolist() == rng_.tolist() and nf.cpu().tolist() == rnf.tolist()
    ok = ~rng_ & ~rnf
    gl = _np(loss)
    assert np.all(gl[~ok] == 0.0) and np.all(_np(g)[~ok] == 0)
    if ok.any():
        assert _rel(_np(g)[ok], rg[ok]) < 1e-5
        assert np.max(np.abs(gl[ok] - rl[ok]) / rl[ok]) < 2e-5
    d = _np(dfdt)
    fin = np.isfinite(rd)
    assert np.array_equal(np.isfinite(d), fin) and _rel(d[fin], rd[fin]) < 2e-6
