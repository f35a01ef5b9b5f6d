"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds no arithmetic of the method: it only draws random tensors
and shapes them the way the workloads below prescribe.  Both sides receive the
same tensors (the oracle gets them upcast to FP64).

Workloads (DiT-shaped attention heads; the pages print no attention sizes of
their own, so head count and head dim come from the workload list, and the
token counts from the page "带分数正则的一致性蒸馏": ``state_t = 21`` latent
frames in section 训练设置 (training setup) and the 480p 16:9 (832x480) and
720p 1:1 (960x960) rows of the video resolution table in section 实验
(experiments), at 16 pixels per token side):

  tiny          B=1 H=2  N=256   d=64   fp32, all six inputs N(0,1)
  image_dit_1k  B=2 H=24 N=4096  d=128  bf16, RMS-normalised Q/K rows, V~N(0,1), tangents N(0,0.1^2)
  video_dit     B=1 H=40 N=32760 d=128  bf16, 21 x 30x52 tokens, tangents N(0,0.3^2)
  long_video    B=1 H=40 N=75600 d=128  bf16, 21 x 60x60 tokens, tangents Student-t(3) x 0.1,
                                         run as 4 key chunks of 18900
  stress        B=4 H=16 N=16384 d=64   bf16, Q/K/V/tangents N(0,1), 1% outlier keys whose
                                         logit is +12 above the rest for every query

The softmax scale is 1/sqrt(d) everywhere.
"""
import math

import torch

WORKLOADS = {
    "tiny": dict(B=1, H=2, N=256, d=64, dtype=torch.float32, seed=1,
                 qk="normal", tangent="normal", tangent_scale=1.0),
    "image_dit_1k": dict(B=2, H=24, N=4096, d=128, dtype=torch.bfloat16, seed=2,
                         qk="rms", tangent="normal", tangent_scale=0.1),
    "video_dit": dict(B=1, H=40, N=32760, d=128, dtype=torch.bfloat16, seed=3,
                      qk="rms", tangent="normal", tangent_scale=0.3),
    "long_video": dict(B=1, H=40, N=75600, d=128, dtype=torch.bfloat16, seed=4,
                       qk="rms", tangent="student_t3", tangent_scale=0.1, kv_chunks=4),
    "stress": dict(B=4, H=16, N=16384, d=64, dtype=torch.bfloat16, seed=5,
                   qk="normal", tangent="normal", tangent_scale=1.0,
                   outlier_frac=0.01, outlier_logit=12.0),
    # the largest head dim of the page's set; not one of the benchmark workloads
    "head_dim_256": dict(B=1, H=16, N=16384, d=256, dtype=torch.bfloat16, seed=6,
                         qk="rms", tangent="normal", tangent_scale=0.3),
}

NAMES = ("q", "k", "v", "q_t", "k_t", "v_t")


def default_scale(d):
    """Softmax scale used by every workload: 1/sqrt(head_dim)."""
    return 1.0 / math.sqrt(d)


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _rms_rows(x):
    # Unit root-mean-square per (b, h, token) row, as a QK-normed DiT produces.
    return x * torch.rsqrt(x.pow(2).mean(dim=-1, keepdim=True) + 1e-6)


def _student_t3(shape, gen, device):
    z = _normal(shape, gen, device)
    chi2 = sum(_normal(shape, gen, device).pow(2) for _ in range(3))
    return z / torch.sqrt(chi2 / 3.0)


def make_inputs(B, H, N, d, *, seed, device="cpu", dtype=torch.bfloat16, qk="normal",
                tangent="normal", tangent_scale=1.0, outlier_frac=0.0, outlier_logit=12.0,
                scale=None, **_unused):
    """Return a dict of the six [B, H, N, d] tensors (names in ``NAMES``) plus ``scale``.

    Draw order is fixed (q, k, v, q_t, k_t, v_t, then the outlier-key choice), so
    a (seed, device) pair always reproduces the same values.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    shape = (B, H, N, d)
    scale = default_scale(d) if scale is None else float(scale)

    q = _normal(shape, gen, device)
    k = _normal(shape, gen, device)
    v = _normal(shape, gen, device)
    if qk == "rms":
        q, k = _rms_rows(q), _rms_rows(k)
    elif qk != "normal":
        raise ValueError("unknown qk recipe %r" % qk)

    def draw_tangent():
        if tangent == "normal":
            return _normal(shape, gen, device) * tangent_scale
        if tangent == "student_t3":
            return _student_t3(shape, gen, device) * tangent_scale
        raise ValueError("unknown tangent recipe %r" % tangent)

    q_t, k_t, v_t = draw_tangent(), draw_tangent(), draw_tangent()

    if outlier_frac > 0.0:
        # Coordinate 0 is reserved: every query has q[0] = 1, outlier keys have
        # k[0] = logit/scale and the rest 0, so each query's logit to an outlier
        # key is exactly `outlier_logit` above what it would otherwise be.  The
        # tangents' coordinate 0 is zero.  With d = 64, 12/scale = 96 is exact in bf16.
        n_out = int(math.floor(outlier_frac * N))
        pick = torch.rand((B, H, N), generator=gen, device=device).topk(n_out, dim=-1).indices
        q[..., 0] = 1.0
        k[..., 0] = 0.0
        k0 = k[..., 0].contiguous()
        k0.scatter_(-1, pick, outlier_logit / scale)
        k[..., 0] = k0
        q_t[..., 0] = 0.0
        k_t[..., 0] = 0.0

    out = {n: t.to(dtype).contiguous() for n, t in zip(NAMES, (q, k, v, q_t, k_t, v_t))}
    out["scale"] = scale
    return out


def workload_inputs(name, device="cpu", **overrides):
    """Inputs for one of the named ``WORKLOADS`` (overrides replace spec fields)."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    return make_inputs(**spec, device=device)


def latent_for(name_or_spec, device="cpu", seed=None):
    """Latent batch (x0, eps, t) for the TrigFlow steps of a workload.

    Each attention token stands for a 2x2 patch of a 16-channel latent, so a
    sample holds 64 * N values (video: 16 ch x 21 frames x 60x104 for N=32760).
    TrigFlow times follow the page's sCM time sampler (section 训练设置, training
    setup): ln sigma ~ N(-0.8, 1.6^2), t = arctan(sigma), one t per sample, FP64.
    """
    spec = dict(WORKLOADS[name_or_spec]) if isinstance(name_or_spec, str) else dict(name_or_spec)
    B, N = spec["B"], spec["N"]
    seed = spec["seed"] + 1000 if seed is None else seed
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x0 = torch.randn((B, 64 * N), generator=gen, device=device, dtype=torch.float32)
    eps = torch.randn((B, 64 * N), generator=gen, device=device, dtype=torch.float32)
    log_sigma = torch.randn((B,), generator=gen, device=device, dtype=torch.float64) * 1.6 - 0.8
    t = torch.atan(torch.exp(log_sigma))
    return x0, eps, t


def epilogue_shape(name_or_spec, min_elems=64 << 20):
    """[B, C, T, H*W] of a latent batch for the output-side kernels with at least
    ``min_elems`` elements (more than L2 holds in fp32): 16 channels and 21 frames
    when the workload's tokens split into 21 frames, else one frame; a sample holds
    64 * N values (one token per 2x2 patch of a 16-channel latent)."""
    spec = dict(WORKLOADS[name_or_spec]) if isinstance(name_or_spec, str) else dict(name_or_spec)
    per = 64 * spec["N"]
    T = 21 if (4 * spec["N"]) % 21 == 0 else 1
    HW = per // (16 * T)
    B = max(1, -(-min_elems // per))
    return B, 16, T, HW


def epilogue_batch(name_or_spec, device="cpu"):
    """Seeded fp32 latent batch of ``epilogue_shape``: x, n, x_t, n_t ~ N(0,1) and the
    FP64 [B, T] times t in [0.2, 1.5) and tangents t_t in [0, 1)."""
    spec = dict(WORKLOADS[name_or_spec]) if isinstance(name_or_spec, str) else dict(name_or_spec)
    B, C, T, HW = epilogue_shape(spec)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(spec["seed"]) + 4242)
    out = {}
    for name in ("x", "n", "x_t", "n_t"):
        out[name] = torch.randn((B, C, T, HW), generator=gen, device=device, dtype=torch.float32)
    out["t"] = torch.rand((B, T), generator=gen, device=device, dtype=torch.float64) * 1.3 + 0.2
    out["t_t"] = torch.rand((B, T), generator=gen, device=device, dtype=torch.float64)
    return out


def upstream_gradient(name_or_spec, shape, device="cpu"):
    """Seeded upstream gradient dO (bf16, N(0,1)) of the backward on a workload's queries."""
    spec = dict(WORKLOADS[name_or_spec]) if isinstance(name_or_spec, str) else dict(name_or_spec)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(spec["seed"]) + 777)
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def sample_rows(N, count, seed):
    """``count`` distinct query-row indices in [0, N), seeded, always including 0 and N-1."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed) + 7919)
    count = min(count, N)
    rows = torch.randperm(N, generator=gen)[:count]
    rows = torch.unique(torch.cat([rows, torch.tensor([0, N - 1])]))
    return rows.sort().values
