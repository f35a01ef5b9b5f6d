"""Shared test helpers: error metrics and oracle evaluation on sampled rows."""
import numpy as np
import torch

import oracle

# Tolerances for bf16 inputs with fp32 accumulation and outputs (O, Ot, mu):
# relative L2 error <= 1e-2 and max-abs error <= 5e-2 x RMS(reference).
REL_L2 = 1e-2
MAX_ABS_RMS = 5e-2
LSE_ABS = 1e-3


def rel_l2(got, ref):
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs_over_rms(got, ref):
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref)) / max(rms, 1e-300))


def assert_close(got, ref, name, rel=REL_L2, mar=MAX_ABS_RMS):
    e1, e2 = rel_l2(got, ref), max_abs_over_rms(got, ref)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % name
    assert e1 <= rel and e2 <= mar, "%s: rel-L2 %.3e (<= %.1e), max-abs/RMS %.3e (<= %.1e)" % (name, e1, rel, e2, mar)
    return e1, e2


def lse_tolerance(x, heads, rows=None):
    """Allowed |LSE error| per sampled row.

    bf16 inputs: the oracle sees exactly the kernel's inputs, so only kernel
    arithmetic differs: LSE_ABS.  fp32 inputs are rounded to bf16 (unit
    roundoff u = 2^-8) before the kernel: each score moves by at most
    s (2u + u^2) sum_c |q_c| |k_c|, and LSE is 1-Lipschitz in the max-norm of the
    scores, so the bound per row is that maximum over keys plus LSE_ABS.
    """
    if x["q"].dtype != torch.float32:
        return LSE_ABS
    u = 2.0 ** -8
    B, H, N, d = x["q"].shape
    q = x["q"].reshape(B * H, N, d)[list(heads)].abs().double()
    k = x["k"].reshape(B * H, N, d)[list(heads)].abs().double()
    if rows is not None:
        q = q[:, torch.as_tensor(rows, device=q.device)]
    worst = torch.matmul(q, k.transpose(-1, -2)).amax(dim=-1)
    return (x["scale"] * (2 * u + u * u) * worst).cpu().numpy() + LSE_ABS


def host64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_on(x, heads=None, rows=None, kv=None):
    """Oracle (O, Ot, LSE, mu) for the given flat head indices and query rows.

    ``x``: dict of [B, H, N, d] tensors (any device) plus "scale"; the oracle sees
    exactly these values upcast to FP64.  ``kv``: optional (start, len) key range.
    Returns arrays [n_heads, R, d] / [n_heads, R].
    """
    B, H, N, d = x["q"].shape
    heads = list(range(B * H)) if heads is None else list(heads)
    flat = {n: x[n].reshape(B * H, N, d) for n in ("q", "k", "v", "q_t", "k_t", "v_t")}
    outs = []
    for h in heads:
        q, qt = host64(flat["q"][h]), host64(flat["q_t"][h])
        k, kt, v, vt = (host64(flat[n][h]) for n in ("k", "k_t", "v", "v_t"))
        if kv is not None:
            a, n = kv
            k, kt, v, vt = (z[a:a + n] for z in (k, kt, v, vt))
        outs.append(oracle.attn_jvp(q, k, v, qt, kt, vt, x["scale"], rows=rows))
    return tuple(np.stack([o[i] for o in outs]) for i in range(4))


def gpu_rows(t, heads, rows=None):
    """Select [heads, rows] of a [B, H, N, ...] GPU result as FP64 numpy."""
    B, H, N = t.shape[:3]
    flat = t.reshape(B * H, N, *t.shape[3:])
    sel = flat[list(heads)]
    if rows is not None:
        sel = sel[:, torch.as_tensor(rows, device=t.device)]
    return host64(sel)
