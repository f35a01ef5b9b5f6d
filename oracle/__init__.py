"""FP64 CPU oracle for attention + JVP and the TrigFlow helpers.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never imports it; its inputs are plain numpy arrays.

The arithmetic lives in ``attn_jvp_oracle.c`` (plain C, FP64, two-pass
softmax; ``attn_bwd_rows``, the backward at sampled rows of full-size heads, is
plain numpy), following the page "带分数正则的一致性蒸馏" (gitcode.csdn.net):
section 注意力 (attention) for O = softmax(s Q K^T) V and its JVP
t_o = P t_v + t_p V, t_p = P (.) t_s - (P t_s^T) P, t_s = (t_q K^T + Q t_k^T) s;
section 前向 (forward) for the natural-log LSE; section 时间步转换 (timestep
conversion) for the TrigFlow wrapper coefficients and x_t = cos t x0 + sin t eps.
The key-chunk merge is exact algebra on those definitions (the pages have no
key split).  The output side of a consistency step (coefficient JVP, the JVP of
_process_output, the tangent target with its NaN masks and normalisation, the
sCM loss) follows section 一致性模型 (consistency model), its 蒸馏代码 listing.
The primal backward (dQ, dK, dV) follows section 反向 (backward).  The QK
normalisation the student keeps (section 一致性模型) is the per-head RMSNorm of
the page "Обслуживание Ideogram v4 менее чем за секунду" (dev48.org), section
on fusing RMSNorm, y = x rsqrt(mean(x^2) + eps) weight; its tangent is the
chain rule on that definition.  ``attn_jvp_rounding_bound`` is the per-element
error bound of the forward's two bf16 roundings (P~ and H~ before the value
sums), written from the same definitions.

Parity pins for every function here are in tests/test_*oracle.py; none is unpinned.
"""
import ctypes
import os

import numpy as np

from . import _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_attn_jvp_rows.argtypes = [dp] * 6 + [i64, i64, i64, i64, ctypes.c_double] + [dp] * 4 + [ctypes.c_int]
        lib.oracle_attn_jvp_rows.restype = ctypes.c_int
        lib.oracle_merge_chunks.argtypes = [dp] * 4 + [i64, i64, i64] + [dp] * 4
        lib.oracle_merge_chunks.restype = ctypes.c_int
        lib.oracle_trigflow_coeffs.argtypes = [ctypes.c_double, ctypes.c_double, dp]
        lib.oracle_trigflow_coeffs.restype = ctypes.c_int
        lib.oracle_trigflow_tangent.argtypes = [dp, dp, dp, i64, i64, dp]
        lib.oracle_trigflow_tangent.restype = ctypes.c_int
        lib.oracle_trigflow_coeffs_jvp.argtypes = [ctypes.c_double] * 3 + [dp]
        lib.oracle_trigflow_coeffs_jvp.restype = ctypes.c_int
        lib.oracle_process_output_jvp.argtypes = [dp] * 6 + [i64] * 4 + [dp] * 2
        lib.oracle_process_output_jvp.restype = ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_scm_tangent_loss.argtypes = [dp] * 6 + [ctypes.c_double] + [i64] * 4 + [dp] * 3 + [ip] * 2
        lib.oracle_scm_tangent_loss.restype = ctypes.c_int
        lib.oracle_attn_bwd_head.argtypes = [dp] * 4 + [i64] * 3 + [ctypes.c_double] + [dp] * 3
        lib.oracle_attn_bwd_head.restype = ctypes.c_int
        lib.oracle_rmsnorm_jvp.argtypes = [dp] * 3 + [i64, i64, ctypes.c_double] + [dp] * 2
        lib.oracle_rmsnorm_jvp.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads():
    """Host threads the oracle uses by default: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def attn_jvp(q, k, v, qt, kt, vt, scale, rows=None, nthreads=None):
    """Attention output, its tangent, LSE and mu in FP64.

    q, qt: [..., Nq, d]; k, kt: [..., Nk, d]; v, vt: [..., Nk, dv] with the
    same leading dims (one independent head per leading index).  ``rows``:
    optional 1-D array of query-row indices evaluated in every head (rows are
    independent, so a subset is exact for those rows).  Returns (o, ot, lse, mu)
    with shapes [..., R, dv], [..., R, dv], [..., R], [..., R].
    """
    lib = _load()
    q, qt, k, kt, v, vt = (_f64(x) for x in (q, qt, k, kt, v, vt))
    lead = q.shape[:-2]
    d = q.shape[-1]
    dv = v.shape[-1]
    nk = k.shape[-2]
    if not (k.shape[:-2] == v.shape[:-2] == lead and kt.shape == k.shape and vt.shape == v.shape
            and qt.shape == q.shape and k.shape[-1] == d and v.shape[-2] == nk):
        raise ValueError("oracle.attn_jvp: inconsistent shapes")
    heads = int(np.prod(lead)) if lead else 1
    qf, qtf = q.reshape(heads, q.shape[-2], d), qt.reshape(heads, q.shape[-2], d)
    kf, ktf = k.reshape(heads, nk, d), kt.reshape(heads, nk, d)
    vf, vtf = v.reshape(heads, nk, dv), vt.reshape(heads, nk, dv)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        qf = np.ascontiguousarray(qf[:, rows])
        qtf = np.ascontiguousarray(qtf[:, rows])
    R = qf.shape[1]
    o = np.empty((heads, R, dv))
    ot = np.empty((heads, R, dv))
    lse = np.empty((heads, R))
    mu = np.empty((heads, R))
    nthreads = nthreads or default_threads()
    for h in range(heads):
        args = [np.ascontiguousarray(x[h]) for x in (qf, qtf, kf, ktf, vf, vtf)]
        outs = [o[h], ot[h], lse[h], mu[h]]
        rc = lib.oracle_attn_jvp_rows(*[_ptr(a) for a in args], R, nk, d, dv, float(scale),
                                      *[_ptr(a) for a in outs], int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attn_jvp_rows failed (%d)" % rc)
    shape_rows = lead + (R,)
    return (o.reshape(shape_rows + (dv,)), ot.reshape(shape_rows + (dv,)),
            lse.reshape(shape_rows), mu.reshape(shape_rows))


def merge_chunks(o_c, ot_c, lse_c, mu_c):
    """Exact merge of key-chunk partials: o_c/ot_c [C, ..., d], lse_c/mu_c [C, ...]."""
    lib = _load()
    o_c, ot_c, lse_c, mu_c = (_f64(x) for x in (o_c, ot_c, lse_c, mu_c))
    C = o_c.shape[0]
    d = o_c.shape[-1]
    rows = int(np.prod(o_c.shape[1:-1])) if o_c.ndim > 2 else 1
    o = np.empty(o_c.shape[1:])
    ot = np.empty(o_c.shape[1:])
    lse = np.empty(lse_c.shape[1:])
    mu = np.empty(lse_c.shape[1:])
    rc = lib.oracle_merge_chunks(_ptr(o_c), _ptr(ot_c), _ptr(lse_c), _ptr(mu_c), C, rows, d,
                                 _ptr(o), _ptr(ot), _ptr(lse), _ptr(mu))
    if rc != 0:
        raise RuntimeError("oracle_merge_chunks failed (%d)" % rc)
    return o, ot, lse, mu


def trigflow_coeffs(t, tau=1000.0):
    """(c_skip, c_out, c_in, c_noise) in FP64 for TrigFlow time t (scalar)."""
    lib = _load()
    out = np.empty(4)
    rc = lib.oracle_trigflow_coeffs(float(t), float(tau), _ptr(out))
    if rc != 0:
        raise ValueError("trigflow_coeffs: cos t + sin t <= 0")
    return tuple(float(x) for x in out)


def trigflow_tangent(x0, eps, t):
    """dx_t/dt = -sin t x0 + cos t eps in FP64; x0/eps [B, ...], t [B]."""
    lib = _load()
    x0, eps, t = _f64(x0), _f64(eps), _f64(t)
    B = x0.shape[0]
    M = int(np.prod(x0.shape[1:])) if x0.ndim > 1 else 1
    out = np.empty_like(x0)
    rc = lib.oracle_trigflow_tangent(_ptr(x0), _ptr(eps), _ptr(t), B, M, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_trigflow_tangent failed")
    return out


def trigflow_coeffs_jvp(t, v, tau=1000.0):
    """((c_skip, c_out, c_in, c_noise), v * d/dt of each) in FP64 at scalar time t."""
    lib = _load()
    out = np.empty(8)
    rc = lib.oracle_trigflow_coeffs_jvp(float(t), float(v), float(tau), _ptr(out))
    if rc != 0:
        raise ValueError("trigflow_coeffs_jvp: cos t + sin t <= 0")
    return tuple(float(x) for x in out[:4]), tuple(float(x) for x in out[4:])


def _bcthw(x):
    """[B, C, T, ...] -> FP64 array and its (B, C, T, HW)."""
    x = _f64(x)
    B, C, T = x.shape[:3]
    HW = int(np.prod(x.shape[3:])) if x.ndim > 3 else 1
    return x, (B, C, T, HW)


def process_output_jvp(x, n, tx, tn, t, tt):
    """F and its tangent from the network output: x, n (network output) and their
    tangents tx, tn are [B, C, T, ...]; the time t and its tangent tt are [B, T]."""
    lib = _load()
    x, dims = _bcthw(x)
    n, tx, tn = (_bcthw(a)[0] for a in (n, tx, tn))
    t, tt = _f64(t), _f64(tt)
    if not (n.shape == tx.shape == tn.shape == x.shape and t.shape == tt.shape == dims[:1] + dims[2:3]):
        raise ValueError("process_output_jvp: inconsistent shapes")
    F = np.empty_like(x)
    tF = np.empty_like(x)
    rc = lib.oracle_process_output_jvp(_ptr(x), _ptr(n), _ptr(tx), _ptr(tn), _ptr(t), _ptr(tt), *dims,
                                       _ptr(F), _ptr(tF))
    if rc != 0:
        raise ValueError("process_output_jvp: bad time (need cos t + sin t > 0 and sin t != 0)")
    return F, tF


def scm_tangent_loss(F_theta, F_sg, F_teacher, x, tF, t, r):
    """Tangent target and sCM loss: returns (g_n, df_dt, loss [B], nan_g [B], nan_F [B]).

    Tensors are [B, C, T, ...] FP64; t is [B, T]; r is the warm-up ratio."""
    lib = _load()
    F_theta, dims = _bcthw(F_theta)
    F_sg, F_teacher, x, tF = (_bcthw(a)[0] for a in (F_sg, F_teacher, x, tF))
    t = _f64(t)
    if not (F_sg.shape == F_teacher.shape == x.shape == tF.shape == F_theta.shape
            and t.shape == dims[:1] + dims[2:3]):
        raise ValueError("scm_tangent_loss: inconsistent shapes")
    g = np.empty_like(F_theta)
    dfdt = np.empty_like(F_theta)
    B = dims[0]
    loss = np.empty(B)
    ng = np.zeros(B, dtype=np.int32)
    nf = np.zeros(B, dtype=np.int32)
    ip = ctypes.POINTER(ctypes.c_int)
    rc = lib.oracle_scm_tangent_loss(_ptr(F_theta), _ptr(F_sg), _ptr(F_teacher), _ptr(x), _ptr(tF), _ptr(t),
                                     float(r), *dims, _ptr(g), _ptr(dfdt), _ptr(loss), ng.ctypes.data_as(ip),
                                     nf.ctypes.data_as(ip))
    if rc != 0:
        raise RuntimeError("oracle_scm_tangent_loss failed")
    return g, dfdt, loss, ng.astype(bool), nf.astype(bool)


def attn_bwd(q, k, v, dO, scale):
    """Primal attention backward in FP64: (dQ, dK, dV) for upstream gradient dO.

    q, dO: [..., Nq, d]; k, v: [..., Nk, d] with the same leading dims (one head each)."""
    lib = _load()
    q, k, v, dO = (_f64(x) for x in (q, k, v, dO))
    lead = q.shape[:-2]
    Nq, d = q.shape[-2:]
    Nk = k.shape[-2]
    if not (k.shape[:-2] == v.shape[:-2] == lead and dO.shape == q.shape and k.shape[-1] == d
            and v.shape == k.shape):
        raise ValueError("oracle.attn_bwd: inconsistent shapes")
    heads = int(np.prod(lead)) if lead else 1
    qf, dOf = q.reshape(heads, Nq, d), dO.reshape(heads, Nq, d)
    kf, vf = k.reshape(heads, Nk, d), v.reshape(heads, Nk, d)
    dq, dk, dv = np.empty((heads, Nq, d)), np.empty((heads, Nk, d)), np.empty((heads, Nk, d))
    for h in range(heads):
        args = [np.ascontiguousarray(x[h]) for x in (qf, kf, vf, dOf)]
        outs = [dq[h], dk[h], dv[h]]
        rc = lib.oracle_attn_bwd_head(*[_ptr(a) for a in args], Nq, Nk, d, float(scale), *[_ptr(a) for a in outs])
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd_head failed (%d)" % rc)
    return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)


def attn_bwd_rows(q, k, v, dO, scale, q_rows, k_rows, block=512, with_scales=False):
    """dQ at the query rows ``q_rows`` and dK, dV at the key rows ``k_rows``, FP64, one head.

    q, dO: [Nq, d]; k, v: [Nk, d].  Every output row is formed from the
    definition of section 反向 (backward):
        P_i = softmax_j(s q_i . k_j),  O_i = sum_j P_ij v_j,  D_i = dO_i . O_i,
        dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - D_i),
        dQ_i = s sum_j dS_ij k_j,  dV_j = sum_i P_ij dO_i,  dK_j = s sum_i dS_ij q_i.
    A key row needs every query's softmax normaliser and D_i; those are formed
    for all queries, ``block`` query rows at a time (the rows are independent),
    so full-size heads fit in memory.  Plain numpy; the full-head reference is
    ``attn_bwd``, with which this agrees on every row (tests/test_bwd_oracle.py).
    Returns (dq [len(q_rows), d], dk [len(k_rows), d], dv [len(k_rows), d]); with
    ``with_scales`` also the size of the sum behind each output element, to which
    a relative error of every term contributes: (s |dS| |K| at the query rows,
    s |dS|^T |Q| and P^T |dO| at the key rows)."""
    q, k, v, dO = (_f64(x) for x in (q, k, v, dO))
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    Nq = q.shape[0]
    m = np.empty(Nq)
    l = np.empty(Nq)
    D = np.empty(Nq)
    for a in range(0, Nq, block):
        b = min(a + block, Nq)
        S = scale * (q[a:b] @ k.T)
        m[a:b] = S.max(axis=1)
        E = np.exp(S - m[a:b, None])
        l[a:b] = E.sum(axis=1)
        O = (E @ v) / l[a:b, None]
        D[a:b] = np.einsum("ij,ij->i", dO[a:b], O)
    # query rows
    P = np.exp(scale * (q[q_rows] @ k.T) - m[q_rows, None]) / l[q_rows, None]
    dS = P * (dO[q_rows] @ v.T - D[q_rows, None])
    dq = scale * (dS @ k)
    sq = scale * (np.abs(dS) @ np.abs(k)) if with_scales else None
    # key rows (columns j of P, dP and dS over every query i)
    Pt = np.exp(scale * (q @ k[k_rows].T) - m[:, None]) / l[:, None]
    dSt = Pt * (dO @ v[k_rows].T - D[:, None])
    dv = Pt.T @ dO
    dk = scale * (dSt.T @ q)
    if with_scales:
        sk = scale * (np.abs(dSt).T @ np.abs(q))
        sv = Pt.T @ np.abs(dO)
        return dq, dk, dv, (sq, sk, sv)
    return dq, dk, dv



def rmsnorm_jvp(x, xt, w, eps):
    """QK normalisation of each row of d values and its tangent, FP64.

    x, xt: [..., d]; w: [d].  Returns (y, yt) shaped like x:
        y = x rho w,  yt = w (xt rho - x rho^3 mean(x xt)),  rho = 1 / sqrt(mean(x^2) + eps)."""
    lib = _load()
    x, xt, w = _f64(x), _f64(xt), _f64(w)
    d = x.shape[-1]
    if xt.shape != x.shape or w.shape != (d,):
        raise ValueError("oracle.rmsnorm_jvp: inconsistent shapes")
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    y, yt = np.empty(x.shape), np.empty(x.shape)
    rc = lib.oracle_rmsnorm_jvp(_ptr(x), _ptr(xt), _ptr(w), rows, d, float(eps), _ptr(y), _ptr(yt))
    if rc != 0:
        raise ValueError("oracle_rmsnorm_jvp failed (%d): rows with no norm or bad eps" % rc)
    return y, yt


def attn_jvp_rounding_bound(q, k, v, qt, kt, vt, scale, rows=None, u=2.0 ** -8, block=256):
    """Per-element bound on |Ot_kernel - Ot| for one head from the two roundings of the
    page's streaming JVP (section 前向: p and H~ = p (.) t_s are cast to the value dtype
    before the dot products): with P~ and H~ each off by at most a relative u,
        |dOt_ic| <= u sum_j P_ij (|vt_jc| + (|St_ij| + |mu_i|) |v_jc|),
    since Ot = T / l - mu O, T = sum P~ vt + sum H~ v and O = sum P~ v / l.  Plain numpy,
    FP64, from the definitions (S, St, P, mu as in attn_jvp).  q, qt: [Nq, d];
    k, kt: [Nk, d]; v, vt: [Nk, dv].  Returns [R, dv] for the query rows ``rows``."""
    q, k, v, qt, kt, vt = (_f64(x) for x in (q, k, v, qt, kt, vt))
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    av, avt = np.abs(v), np.abs(vt)
    out = np.empty((len(rows), v.shape[1]))
    for a in range(0, len(rows), block):
        r = rows[a:a + block]
        S = scale * (q[r] @ k.T)
        St = scale * (qt[r] @ k.T + q[r] @ kt.T)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        mu = np.einsum("ij,ij->i", P, St)
        out[a:a + len(r)] = u * (P @ avt + (P * (np.abs(St) + np.abs(mu)[:, None])) @ av)
    return out
