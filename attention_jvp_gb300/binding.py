"""Thin ctypes binding of ``libattnjvp.so``: argument marshalling only.

Every function has the name of the C entry point it calls (include/attnjvp.h).
Tensors are torch tensors on the current CUDA device; torch only provides the
device memory and the stream.  All arithmetic runs in the library's kernels:
if the library is missing or fails to load, every call raises — there is no
fallback path.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattnjvp.so")

ATTNJVP_OK = 0
ATTNJVP_EINVAL = -1
ATTNJVP_EUNSUPPORTED = -2
ATTNJVP_ECUDA = -3
ATTNJVP_ETIMEOUT = -4

# input dtype codes of the forward entry points
ATTNJVP_BF16 = 0
ATTNJVP_FP32 = 1
_DTYPE_CODES = {torch.bfloat16: ATTNJVP_BF16, torch.float32: ATTNJVP_FP32}

_lib = None


class AttnJvpError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__("%s failed (%d): %s" % (fn, code, msg))
        self.code = code


def load(path=None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libattnjvp.so not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    vp, i64, fp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p
    ci = ctypes.c_int
    lib.attn_jvp_fwd.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 4 + [ctypes.c_float, ci, vp]
    lib.attn_jvp_fwd_chunk.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 4 + [ctypes.c_float, ci, i64, i64, vp]
    lib.attn_jvp_merge.argtypes = [vp] * 4 + [i64] + [vp] * 4 + [i64] * 4 + [vp]
    lib.attn_jvp_cast_f32_bf16.argtypes = [vp, vp, i64, vp]
    lib.attn_jvp_fwd_split_noalloc.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 4 + [ctypes.c_float, ci, i64, vp]
    lib.attn_jvp_fwd_host.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 4 + [ctypes.c_float, i64, i64, vp, i64, vp]
    lib.attn_jvp_fwd_strided.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 5 + [ctypes.POINTER(i64), ctypes.c_float,
                                                                          ci, i64, i64, vp]
    lib.attn_jvp_fwd_ex.argtypes = [vp] * 6 + [fp] * 4 + [i64] * 6 + [ctypes.POINTER(i64), ctypes.c_float,
                                                                    ci, i64, i64, vp]
    lib.attn_jvp_fwd_host_workspace_bytes.argtypes = [i64] * 6
    lib.attn_jvp_fwd_host_workspace_bytes.restype = i64
    lib.qk_rmsnorm_jvp.argtypes = [vp] * 10 + [i64] * 3 + [ctypes.c_float, vp]
    lib.attn_jvp_fwd_last_wave_split.argtypes = [i64] * 5 + [ctypes.POINTER(i64)]
    lib.trigflow_coeffs_jvp.argtypes = [ctypes.c_double] * 3 + [ctypes.POINTER(ctypes.c_double)]
    lib.trigflow_output_jvp.argtypes = [vp] * 8 + [i64] * 4 + [vp]
    lib.scm_tangent_loss.argtypes = [vp] * 6 + [ctypes.c_double] + [vp] * 5 + [i64] * 4 + [vp, i64, vp]
    lib.scm_tangent_loss_workspace_bytes.argtypes = [i64] * 4
    lib.scm_tangent_loss_workspace_bytes.restype = i64
    lib.attn_bwd.argtypes = [vp] * 9 + [i64] * 5 + [ctypes.c_float, vp, i64, vp]
    lib.attn_bwd_workspace_bytes.argtypes = [i64] * 3
    lib.attn_bwd_workspace_bytes.restype = i64
    lib.trigflow_coeffs.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_double)]
    lib.trigflow_tangent.argtypes = [vp, vp, vp, vp, i64, i64, vp]
    lib.attn_jvp_status.argtypes = [ctypes.c_int]
    lib.attn_jvp_selftest_wait.argtypes = [i64, vp]
    lib.attn_jvp_last_error.restype = ctypes.c_char_p
    lib.attn_jvp_version.restype = ctypes.c_char_p
    for name in ("attn_jvp_fwd", "attn_jvp_fwd_chunk", "attn_jvp_merge", "attn_jvp_cast_f32_bf16",
                 "attn_jvp_fwd_split_noalloc", "attn_jvp_fwd_host", "attn_jvp_fwd_strided", "attn_jvp_fwd_ex",
                 "trigflow_coeffs_jvp", "trigflow_output_jvp", "scm_tangent_loss", "attn_bwd", "qk_rmsnorm_jvp",
                 "trigflow_coeffs", "trigflow_tangent", "attn_jvp_status", "attn_jvp_selftest_wait"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn, rc):
    if rc != ATTNJVP_OK:
        raise AttnJvpError(fn, rc, load().attn_jvp_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _req(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))
    return t


def attn_jvp_cast_f32_bf16(x, out=None, stream=None):
    """fp32 -> bf16 on the device (round to nearest even)."""
    _req(x, "x", torch.float32)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _req(out, "out", torch.bfloat16, x.shape)
    _check("attn_jvp_cast_f32_bf16", load().attn_jvp_cast_f32_bf16(_ptr(x), _ptr(out), x.numel(), _stream(stream)))
    return out


def _inputs(tensors):
    """The six contiguous [B, H, N, d] inputs and the library's dtype code for them.

    All six must share one dtype, bf16 or fp32; fp32 inputs are rounded to bf16 by
    the library itself (the ``dtype`` argument of the C entry points)."""
    dt = tensors[0].dtype if isinstance(tensors[0], torch.Tensor) else None
    if dt not in _DTYPE_CODES:
        raise ValueError("q must be torch.bfloat16 or torch.float32 (got %s)" % dt)
    res = [_req(t, n, dt) for n, t in zip(("q", "k", "v", "q_t", "k_t", "v_t"), tensors)]
    shape = tuple(res[0].shape)
    if len(shape) != 4:
        raise ValueError("q must be [B, H, N, d]")
    for n, t in zip(("k", "v", "q_t", "k_t", "v_t"), res[1:]):
        if tuple(t.shape) != shape:
            raise ValueError("%s must have q's shape %s (got %s)" % (n, shape, tuple(t.shape)))
    return res, _DTYPE_CODES[dt]


def _outputs(shape, device, out, out_t, lse, mu, need_rows):
    B, H, N, d = shape
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.float32, device=device)
    if out_t is None:
        out_t = torch.empty((B, H, N, d), dtype=torch.float32, device=device)
    if lse is None and need_rows:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    if mu is None and need_rows:
        mu = torch.empty((B, H, N), dtype=torch.float32, device=device)
    _req(out, "out", torch.float32, shape)
    _req(out_t, "out_t", torch.float32, shape)
    if lse is not None:
        _req(lse, "lse", torch.float32, (B, H, N))
    if mu is not None:
        _req(mu, "mu", torch.float32, (B, H, N))
    return out, out_t, lse, mu


def attn_jvp_fwd(q, k, v, q_t, k_t, v_t, scale=None, out=None, out_t=None, lse=None, mu=None,
                 want_rows=True, stream=None):
    """(O, Ot, LSE, mu) of softmax attention and its JVP; inputs [B, H, N, d] bf16 (or fp32)."""
    (q, k, v, q_t, k_t, v_t), code = _inputs((q, k, v, q_t, k_t, v_t))
    B, H, N, d = q.shape
    scale = d ** -0.5 if scale is None else float(scale)
    out, out_t, lse, mu = _outputs(q.shape, q.device, out, out_t, lse, mu, want_rows)
    rc = load().attn_jvp_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(q_t), _ptr(k_t), _ptr(v_t),
                             _ptr(out), _ptr(out_t), _ptr(lse), _ptr(mu), B, H, N, d,
                             ctypes.c_float(scale), code, _stream(stream))
    _check("attn_jvp_fwd", rc)
    return out, out_t, lse, mu


def attn_jvp_fwd_last_wave_split(B, H, N_q, N_kv, d_v):
    """Pieces per unit into which attn_jvp_fwd cuts the last wave of this shape on the
    current device (1: no cut; otherwise the call launches a second, merging kernel)."""
    out = ctypes.c_int64(0)
    _check("attn_jvp_fwd_last_wave_split",
           load().attn_jvp_fwd_last_wave_split(int(B), int(H), int(N_q), int(N_kv), int(d_v), ctypes.byref(out)))
    return out.value


def attn_jvp_fwd_chunk(q, k, v, q_t, k_t, v_t, kv_start, kv_len, scale=None, out=None, out_t=None,
                       lse=None, mu=None, stream=None):
    """Partials (O_c, Ot_c, LSE_c, mu_c) over keys [kv_start, kv_start + kv_len)."""
    (q, k, v, q_t, k_t, v_t), code = _inputs((q, k, v, q_t, k_t, v_t))
    B, H, N, d = q.shape
    scale = d ** -0.5 if scale is None else float(scale)
    out, out_t, lse, mu = _outputs(q.shape, q.device, out, out_t, lse, mu, True)
    rc = load().attn_jvp_fwd_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(q_t), _ptr(k_t), _ptr(v_t),
                                   _ptr(out), _ptr(out_t), _ptr(lse), _ptr(mu), B, H, N, d,
                                   ctypes.c_float(scale), code, int(kv_start), int(kv_len), _stream(stream))
    _check("attn_jvp_fwd_chunk", rc)
    return out, out_t, lse, mu


_LAYOUTS = {
    # layout -> (index of B, S, H, D in the tensor's shape)
    "bhsd": (0, 2, 1, 3),
    "bshd": (0, 1, 2, 3),
}


def _layout_view(t, name, layout, dtype=torch.bfloat16):
    """(B, S, H, D) and element strides (batch, seq, head) of a CUDA tensor in ``layout``."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("%s must be 4-D with a unit stride in the head dimension" % name)
    ib, isq, ih, _ = _LAYOUTS[layout]
    dims = (t.shape[ib], t.shape[isq], t.shape[ih], t.shape[3])
    return dims, (t.stride(ib), t.stride(isq), t.stride(ih))


def attn_jvp_fwd_strided(q, k, v, q_t, k_t, v_t, layout="bhsd", scale=None, out=None, out_t=None, lse=None,
                         mu=None, kv_start=0, kv_len=None, want_rows=True, stream=None):
    """Strided / cross-attention form.  ``layout`` names the dimension order of every
    tensor's shape: "bhsd" ([B, H, S, D]) or "bshd" ([B, S, H, D], the page's).  Any
    strides are accepted as long as the head dimension is unit-stride; tangents must
    share their primal's strides.  V (and Vt) may have a head dim of their own,
    d_v; O and Ot then have d_v columns.  Outputs O, Ot default to a new contiguous
    tensor in ``layout``; lse, mu are [B, H, N_q].  ``kv_start``/``kv_len`` select a
    key range.  Calls attn_jvp_fwd_ex."""
    if layout not in _LAYOUTS:
        raise ValueError("layout must be one of %s" % sorted(_LAYOUTS))
    dt = q.dtype if isinstance(q, torch.Tensor) else None
    if dt not in _DTYPE_CODES:
        raise ValueError("q must be torch.bfloat16 or torch.float32 (got %s)" % dt)
    (B, Nq, H, d), qs = _layout_view(q, "q", layout, dt)
    (Bk, Nkv, Hk, dk), ks = _layout_view(k, "k", layout, dt)
    if (Bk, Hk, dk) != (B, H, d):
        raise ValueError("k must match q in batch, heads and head dim")
    (Bv, Nv, Hv, d_v), vs = _layout_view(v, "v", layout, dt)
    if (Bv, Nv, Hv) != (B, Nkv, H):
        raise ValueError("v must match k in batch, sequence length and heads")
    for n, t, ref in (("q_t", q_t, q), ("k_t", k_t, k), ("v_t", v_t, v)):
        _layout_view(t, n, layout, dt)
        if tuple(t.shape) != tuple(ref.shape) or t.stride() != ref.stride():
            raise ValueError("%s must have the shape and strides of %s" % (n, n[0]))
    ib, isq, ih, _ = _LAYOUTS[layout]
    shape_o = list(q.shape)
    shape_o[3] = d_v
    shape_o = tuple(shape_o)
    if out is None:
        out = torch.empty(shape_o, dtype=torch.float32, device=q.device)
    if out_t is None:
        out_t = torch.empty(shape_o, dtype=torch.float32, device=q.device)
    for n, t in (("out", out), ("out_t", out_t)):
        if not t.is_cuda or t.dtype != torch.float32 or tuple(t.shape) != shape_o or t.stride(3) != 1:
            raise ValueError("%s must be a float32 CUDA tensor of shape %s with a unit last stride" % (n, shape_o))
    if out_t.stride() != out.stride():
        raise ValueError("out_t must have out's strides")
    os_ = (out.stride(ib), out.stride(isq), out.stride(ih))
    if lse is None and want_rows:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if mu is None and want_rows:
        mu = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _req(lse, "lse", torch.float32, (B, H, Nq))
    if mu is not None:
        _req(mu, "mu", torch.float32, (B, H, Nq))
    kv_len = Nkv - kv_start if kv_len is None else int(kv_len)
    scale = d ** -0.5 if scale is None else float(scale)
    strides = (ctypes.c_int64 * 12)(*qs, *ks, *vs, *os_)
    rc = load().attn_jvp_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(q_t), _ptr(k_t), _ptr(v_t),
                                _ptr(out), _ptr(out_t), _ptr(lse), _ptr(mu), B, H, Nq, Nkv, d, d_v, strides,
                                ctypes.c_float(scale), _DTYPE_CODES[dt], int(kv_start), kv_len, _stream(stream))
    _check("attn_jvp_fwd_ex", rc)
    return out, out_t, lse, mu


def attn_jvp_merge(o_c, ot_c, lse_c, mu_c, out=None, out_t=None, lse=None, mu=None, stream=None):
    """Exact merge of chunk partials o_c/ot_c [C, B, H, N, d], lse_c/mu_c [C, B, H, N]."""
    _req(o_c, "o_c", torch.float32)
    C, B, H, N, d = o_c.shape
    _req(ot_c, "ot_c", torch.float32, o_c.shape)
    _req(lse_c, "lse_c", torch.float32, (C, B, H, N))
    _req(mu_c, "mu_c", torch.float32, (C, B, H, N))
    out, out_t, lse, mu = _outputs((B, H, N, d), o_c.device, out, out_t, lse, mu, True)
    rc = load().attn_jvp_merge(_ptr(o_c), _ptr(ot_c), _ptr(lse_c), _ptr(mu_c), C, _ptr(out), _ptr(out_t),
                               _ptr(lse), _ptr(mu), B, H, N, d, _stream(stream))
    _check("attn_jvp_merge", rc)
    return out, out_t, lse, mu


def chunk_bounds(N, n_chunks):
    """Key ranges [(start, len), ...] splitting N keys into n_chunks near-equal chunks."""
    edges = [(N * c) // n_chunks for c in range(n_chunks + 1)]
    return [(a, b - a) for a, b in zip(edges[:-1], edges[1:])]


def attn_jvp_split(q, k, v, q_t, k_t, v_t, n_chunks, scale=None, workspace=None, out=None, out_t=None,
                   lse=None, mu=None, stream=None):
    """Split-KV path: one chunk launch per key range, then the exact merge.

    ``workspace``: optional (o_c, ot_c, lse_c, mu_c) partial buffers to reuse.
    """
    (q, k, v, q_t, k_t, v_t), _ = _inputs((q, k, v, q_t, k_t, v_t))
    B, H, N, d = q.shape
    if workspace is None:
        workspace = split_workspace(q.shape, n_chunks, q.device)
    o_c, ot_c, lse_c, mu_c = workspace
    for c, (a, n) in enumerate(chunk_bounds(N, n_chunks)):
        attn_jvp_fwd_chunk(q, k, v, q_t, k_t, v_t, a, n, scale=scale, out=o_c[c], out_t=ot_c[c],
                           lse=lse_c[c], mu=mu_c[c], stream=stream)
    return attn_jvp_merge(o_c, ot_c, lse_c, mu_c, out=out, out_t=out_t, lse=lse, mu=mu, stream=stream)


def attn_jvp_fwd_split_noalloc(q, k, v, q_t, k_t, v_t, n_chunks, out, out_t, lse=None, mu=None, scale=None,
                               stream=None):
    """Split-KV path whose chunk partials live in the library's built-in
    scratch array, for callers that cannot allocate device memory.  All
    outputs are caller-provided; this wrapper allocates nothing either.
    Inputs are bf16 or fp32 (all six alike)."""
    (q, k, v, q_t, k_t, v_t), code = _inputs((q, k, v, q_t, k_t, v_t))
    B, H, N, d = q.shape
    _req(out, "out", torch.float32, q.shape)
    _req(out_t, "out_t", torch.float32, q.shape)
    if lse is not None:
        _req(lse, "lse", torch.float32, (B, H, N))
    if mu is not None:
        _req(mu, "mu", torch.float32, (B, H, N))
    scale = d ** -0.5 if scale is None else float(scale)
    rc = load().attn_jvp_fwd_split_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(q_t), _ptr(k_t), _ptr(v_t),
                                           _ptr(out), _ptr(out_t), _ptr(lse), _ptr(mu), B, H, N, d,
                                           ctypes.c_float(scale), code, int(n_chunks), _stream(stream))
    _check("attn_jvp_fwd_split_noalloc", rc)
    return out, out_t, lse, mu


def qk_rmsnorm_jvp(q, q_t, k, k_t, w_q, w_k, eps=1e-6, out=None, stream=None):
    """QK normalisation and its tangent: (qn, qn_t, kn, kn_t), bf16, shaped like the inputs.

    q, q_t, k, k_t: contiguous bf16 tensors whose last dim is the head dim d (each
    row of d values one token of one head); w_q, w_k: fp32 [d].  ``out``: optional
    (qn, qn_t, kn, kn_t) to write into (an input may serve as its own output)."""
    _req(q, "q", torch.bfloat16)
    d = q.shape[-1]
    _req(q_t, "q_t", torch.bfloat16, q.shape)
    _req(k, "k", torch.bfloat16)
    if k.shape[-1] != d:
        raise ValueError("k must have q's head dim %d" % d)
    _req(k_t, "k_t", torch.bfloat16, k.shape)
    _req(w_q, "w_q", torch.float32, (d,))
    _req(w_k, "w_k", torch.float32, (d,))
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), torch.empty_like(k))
    for n, t, ref in zip(("qn", "qn_t", "kn", "kn_t"), out, (q, q, k, k)):
        _req(t, n, torch.bfloat16, ref.shape)
    rc = load().qk_rmsnorm_jvp(_ptr(q), _ptr(q_t), _ptr(k), _ptr(k_t), _ptr(w_q), _ptr(w_k), *(_ptr(t) for t in out),
                               q.numel() // d, k.numel() // d, d, ctypes.c_float(eps), _stream(stream))
    _check("qk_rmsnorm_jvp", rc)
    return tuple(out)


def _host(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))
    return t


def attn_jvp_fwd_host_workspace_bytes(shape, n_chunks=1, group_heads=0):
    """Device workspace bytes attn_jvp_fwd_host needs for inputs of ``shape`` [B, H, N, d]."""
    B, H, N, d = shape
    n = load().attn_jvp_fwd_host_workspace_bytes(B, H, N, d, int(n_chunks), int(group_heads))
    if n < 0:
        _check("attn_jvp_fwd_host_workspace_bytes", int(n))
    return int(n)


def host_workspace(shape, n_chunks=1, group_heads=0, device=None):
    """A device buffer sized for attn_jvp_fwd_host (torch's allocator aligns it to 256 bytes or more)."""
    n = attn_jvp_fwd_host_workspace_bytes(shape, n_chunks, group_heads)
    return torch.empty(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def attn_jvp_fwd_host(q, k, v, q_t, k_t, v_t, out, out_t, lse=None, mu=None, scale=None, n_chunks=1,
                      group_heads=0, workspace=None, stream=None):
    """The attention JVP on host tensors (bf16 [B, H, N, d] in; fp32 out), with the
    library overlapping the transfers with compute.  Use pinned host tensors for
    overlap.  Outputs are complete once ``stream`` has been synchronised."""
    shape = tuple(q.shape)
    if len(shape) != 4:
        raise ValueError("q must be [B, H, N, d]")
    for n, t in zip(("q", "k", "v", "q_t", "k_t", "v_t"), (q, k, v, q_t, k_t, v_t)):
        _host(t, n, torch.bfloat16, shape)
    B, H, N, d = shape
    _host(out, "out", torch.float32, shape)
    _host(out_t, "out_t", torch.float32, shape)
    if lse is not None:
        _host(lse, "lse", torch.float32, (B, H, N))
    if mu is not None:
        _host(mu, "mu", torch.float32, (B, H, N))
    if workspace is None:
        workspace = host_workspace(shape, n_chunks, group_heads)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    scale = d ** -0.5 if scale is None else float(scale)
    rc = load().attn_jvp_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(q_t), _ptr(k_t), _ptr(v_t),
                                  _ptr(out), _ptr(out_t), _ptr(lse), _ptr(mu), B, H, N, d,
                                  ctypes.c_float(scale), int(n_chunks), int(group_heads), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_jvp_fwd_host", rc)
    return out, out_t, lse, mu


def split_workspace(shape, n_chunks, device):
    B, H, N, d = shape
    return (torch.empty((n_chunks, B, H, N, d), dtype=torch.float32, device=device),
            torch.empty((n_chunks, B, H, N, d), dtype=torch.float32, device=device),
            torch.empty((n_chunks, B, H, N), dtype=torch.float32, device=device),
            torch.empty((n_chunks, B, H, N), dtype=torch.float32, device=device))


def trigflow_coeffs(t, tau=1000.0):
    """(c_skip, c_out, c_in, c_noise) in FP64 (host function of the library)."""
    c = (ctypes.c_double * 4)()
    _check("trigflow_coeffs", load().trigflow_coeffs(float(t), float(tau), c))
    return tuple(c)


def trigflow_tangent(x0, eps, t, out=None, stream=None):
    """dx_t/dt = -sin t x0 + cos t eps; x0/eps fp32 [B, ...], t FP64 [B] on the device."""
    _req(x0, "x0", torch.float32)
    _req(eps, "eps", torch.float32, x0.shape)
    B = x0.shape[0]
    _req(t, "t", torch.float64, (B,))
    if out is None:
        out = torch.empty_like(x0)
    _req(out, "out", torch.float32, x0.shape)
    per = x0.numel() // B
    _check("trigflow_tangent", load().trigflow_tangent(_ptr(x0), _ptr(eps), _ptr(t), _ptr(out), B, per,
                                                       _stream(stream)))
    return out


def attn_jvp_status(clear=True):
    """0 if no kernel reported a problem; raises AttnJvpError(ETIMEOUT) otherwise."""
    _check("attn_jvp_status", load().attn_jvp_status(1 if clear else 0))
    return 0


def attn_jvp_selftest_wait(limit_ns, stream=None):
    """Launch the bounded-wait self-test kernel (see include/attnjvp.h)."""
    _check("attn_jvp_selftest_wait", load().attn_jvp_selftest_wait(int(limit_ns), _stream(stream)))


def attn_jvp_version():
    return load().attn_jvp_version().decode()


# ---- output side of one consistency step ----

def trigflow_coeffs_jvp(t, v, tau=1000.0):
    """((c_skip, c_out, c_in, c_noise), v * d/dt of each) in FP64 (host function of the library)."""
    out = (ctypes.c_double * 8)()
    _check("trigflow_coeffs_jvp", load().trigflow_coeffs_jvp(float(t), float(v), float(tau), out))
    return tuple(out[:4]), tuple(out[4:])


def _latent(t, name, shape=None):
    _req(t, name, torch.float32, shape)
    if t.dim() < 3:
        raise ValueError("%s must be [B, C, T, ...]" % name)
    return t


def _bcthw_dims(x):
    B, C, T = x.shape[:3]
    HW = 1
    for s_ in x.shape[3:]:
        HW *= s_
    return B, C, T, HW


def trigflow_output_jvp(x, n, x_t, n_t, t, t_t, out=None, out_t=None, stream=None):
    """F = (cos t x - (c_skip x + c_out n)) / sin t and its tangent; x, n, x_t, n_t are
    fp32 [B, C, T, ...] on the GPU, t and t_t FP64 [B, T]."""
    _latent(x, "x")
    for nm, a in (("n", n), ("x_t", x_t), ("n_t", n_t)):
        _latent(a, nm, x.shape)
    B, C, T, HW = _bcthw_dims(x)
    _req(t, "t", torch.float64, (B, T))
    _req(t_t, "t_t", torch.float64, (B, T))
    out = torch.empty_like(x) if out is None else _latent(out, "out", x.shape)
    out_t = torch.empty_like(x) if out_t is None else _latent(out_t, "out_t", x.shape)
    rc = load().trigflow_output_jvp(_ptr(x), _ptr(n), _ptr(x_t), _ptr(n_t), _ptr(t), _ptr(t_t), _ptr(out),
                                    _ptr(out_t), B, C, T, HW, _stream(stream))
    _check("trigflow_output_jvp", rc)
    return out, out_t


def scm_workspace(shape, device=None):
    B, C, T = shape[:3]
    HW = 1
    for s_ in shape[3:]:
        HW *= s_
    n = load().scm_tangent_loss_workspace_bytes(B, C, T, HW)
    if n < 0:
        _check("scm_tangent_loss_workspace_bytes", int(n))
    return torch.empty((n + 7) // 8, dtype=torch.float64, device=device or torch.device("cuda"))


def scm_tangent_loss(F_theta, F_sg, F_teacher, x, F_t, t, r, workspace=None, stream=None):
    """Tangent target, its NaN masks and normalisation, and the sCM loss.

    Returns (g_n fp32, df_dt fp32, loss FP64 [B], nan_g bool [B], nan_F bool [B])."""
    _latent(F_theta, "F_theta")
    for nm, a in (("F_sg", F_sg), ("F_teacher", F_teacher), ("x", x), ("F_t", F_t)):
        _latent(a, nm, F_theta.shape)
    B, C, T, HW = _bcthw_dims(F_theta)
    _req(t, "t", torch.float64, (B, T))
    dev = F_theta.device
    g_n = torch.empty_like(F_theta)
    dfdt = torch.empty_like(F_theta)
    loss = torch.empty(B, dtype=torch.float64, device=dev)
    nan_g = torch.empty(B, dtype=torch.int32, device=dev)
    nan_F = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = scm_workspace(tuple(F_theta.shape), dev)
    rc = load().scm_tangent_loss(_ptr(F_theta), _ptr(F_sg), _ptr(F_teacher), _ptr(x), _ptr(F_t), _ptr(t),
                                 float(r), _ptr(g_n), _ptr(dfdt), _ptr(loss), _ptr(nan_g), _ptr(nan_F), B, C, T,
                                 HW, _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("scm_tangent_loss", rc)
    return g_n, dfdt, loss, nan_g.bool(), nan_F.bool()


# ---- primal attention backward ----

def attn_bwd(q, k, v, dout, out, lse, scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """(dQ, dK, dV) of attention for the upstream gradient ``dout``.

    q, dout bf16 [B, H, N_q, d]; k, v bf16 [B, H, N_kv, d]; ``out`` (fp32 O) and ``lse``
    are the forward's outputs for the same q, k, v and scale.  fp32 dout is rounded to
    bf16 by the library's cast kernel."""
    if isinstance(dout, torch.Tensor) and dout.dtype == torch.float32:
        _req(dout, "dout", torch.float32)
        dout = attn_jvp_cast_f32_bf16(dout, stream=stream)
    _req(q, "q", torch.bfloat16)
    B, H, Nq, d = q.shape
    _req(k, "k", torch.bfloat16)
    Nkv = k.shape[2]
    if tuple(k.shape) != (B, H, Nkv, d):
        raise ValueError("k must be [B, H, N_kv, d] with q's B, H, d")
    _req(v, "v", torch.bfloat16, k.shape)
    _req(dout, "dout", torch.bfloat16, q.shape)
    _req(out, "out", torch.float32, q.shape)
    _req(lse, "lse", torch.float32, (B, H, Nq))
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device) if dq is None else _req(dq, "dq", torch.float32,
                                                                                             q.shape)
    dk = torch.empty(k.shape, dtype=torch.float32, device=q.device) if dk is None else _req(dk, "dk", torch.float32,
                                                                                             k.shape)
    dv = torch.empty(k.shape, dtype=torch.float32, device=q.device) if dv is None else _req(dv, "dv", torch.float32,
                                                                                             k.shape)
    if workspace is None:
        n = load().attn_bwd_workspace_bytes(B, H, Nq)
        if n < 0:
            _check("attn_bwd_workspace_bytes", int(n))
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    scale = d ** -0.5 if scale is None else float(scale)
    rc = load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                         B, H, Nq, Nkv, d, ctypes.c_float(scale), _ptr(workspace),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check("attn_bwd", rc)
    return dq, dk, dv
