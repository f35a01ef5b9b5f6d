"""CPU-side checks of the C ABI: the library loads, exports every declared
symbol, validates arguments before touching CUDA, and its host-side TrigFlow
coefficients match the oracle to 1e-12."""
import ctypes
import math
import os
import re
import subprocess

import pytest
import torch

import oracle
from attention_jvp_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attnjvp.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for expected in ("attn_jvp_fwd", "attn_jvp_fwd_chunk", "attn_jvp_merge", "attn_jvp_cast_f32_bf16",
                     "trigflow_coeffs", "trigflow_tangent", "attn_jvp_status", "attn_jvp_last_error",
                     "attn_jvp_version", "attn_jvp_selftest_wait", "attn_jvp_fwd_split_noalloc",
                     "attn_jvp_fwd_host", "attn_jvp_fwd_host_workspace_bytes", "attn_jvp_fwd_strided",
                     "trigflow_coeffs_jvp", "trigflow_output_jvp", "scm_tangent_loss",
                     "scm_tangent_loss_workspace_bytes", "attn_bwd", "attn_bwd_workspace_bytes",
                     "qk_rmsnorm_jvp", "attn_jvp_fwd_last_wave_split"):
        assert expected in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_library_is_built_for_sm103a_only(monkeypatch):
    """Every translation unit and the link step get exactly one -gencode, sm_103a
    (machine code only: no PTX for a JIT to pick up on another GPU)."""
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert not any("gencode" in f or "arch" in f for f in _build.NVCC_FLAGS)
    seen = []

    class Done(Exception):
        pass

    def fake_run(cmd, **kw):
        seen.append(cmd)
        raise Done

    monkeypatch.setattr(_build.subprocess, "run", fake_run)  # record the commands, compile nothing
    with pytest.raises(Done):
        _build.build(force=True)
    assert seen, "build() ran no compiler"
    for cmd in seen:
        assert cmd.count("-gencode") == 1 and "arch=compute_103a,code=sm_103a" in cmd, cmd


def _fwd(lib, ptrs=None, B=1, H=1, N=128, d=128, scale=0.1, chunk=None, dtype=binding.ATTNJVP_BF16):
    p = [ctypes.c_void_p(256)] * 10 if ptrs is None else ptrs
    if chunk is None:
        return lib.attn_jvp_fwd(*p, B, H, N, d, ctypes.c_float(scale), dtype, None)
    return lib.attn_jvp_fwd_chunk(*p, B, H, N, d, ctypes.c_float(scale), dtype, chunk[0], chunk[1], None)


def test_argument_validation_needs_no_gpu(lib):
    E = binding
    null = [ctypes.c_void_p(0)] + [ctypes.c_void_p(256)] * 9
    assert _fwd(lib, null) == E.ATTNJVP_EINVAL
    assert b"q is NULL" in lib.attn_jvp_last_error()
    mis = [ctypes.c_void_p(256)] * 3 + [ctypes.c_void_p(258)] + [ctypes.c_void_p(256)] * 6
    assert _fwd(lib, mis) == E.ATTNJVP_EINVAL
    assert b"16-byte" in lib.attn_jvp_last_error()
    assert _fwd(lib, N=0) == E.ATTNJVP_EINVAL
    assert _fwd(lib, B=0) == E.ATTNJVP_EINVAL
    assert _fwd(lib, scale=float("nan")) == E.ATTNJVP_EINVAL
    assert _fwd(lib, scale=-1.0) == E.ATTNJVP_EINVAL
    assert _fwd(lib, scale=float("inf")) == E.ATTNJVP_EINVAL
    assert _fwd(lib, d=96) == E.ATTNJVP_EUNSUPPORTED
    assert _fwd(lib, d=512) == E.ATTNJVP_EUNSUPPORTED
    assert _fwd(lib, d=192) == E.ATTNJVP_EUNSUPPORTED
    assert _fwd(lib, chunk=(0, 0)) == E.ATTNJVP_EINVAL
    assert _fwd(lib, chunk=(100, 29)) == E.ATTNJVP_EINVAL
    assert _fwd(lib, chunk=(-1, 10)) == E.ATTNJVP_EINVAL
    no_rows = [ctypes.c_void_p(256)] * 8 + [ctypes.c_void_p(0)] * 2
    assert _fwd(lib, no_rows, chunk=(0, 64)) == E.ATTNJVP_EINVAL
    vp = ctypes.c_void_p(256)
    assert lib.attn_jvp_merge(vp, vp, vp, vp, 0, vp, vp, None, None, 1, 1, 8, 128, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_merge(vp, vp, vp, vp, 2, vp, vp, None, None, 1, 1, 8, 130, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_cast_f32_bf16(vp, vp, -1, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_cast_f32_bf16(vp, vp, 0, None) == E.ATTNJVP_OK
    assert lib.trigflow_tangent(vp, vp, vp, vp, 0, 10, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_selftest_wait(10, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_selftest_wait(5_000_000_000, None) == E.ATTNJVP_EINVAL
    assert lib.attn_jvp_fwd_split_noalloc(*[ctypes.c_void_p(256)] * 10, 1, 1, 64, 128, ctypes.c_float(0.1),
                                          E.ATTNJVP_BF16, 0, None) == E.ATTNJVP_EINVAL
    assert lib.trigflow_tangent(vp, vp, vp, vp, 2, 0, None) == E.ATTNJVP_EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_cuda_error(lib):
    assert _fwd(lib) == binding.ATTNJVP_ECUDA
    assert len(lib.attn_jvp_last_error()) > 0


@pytest.mark.parametrize("t", [0.0, 1e-3, 0.3, math.pi / 4, 1.0, 1.4, 1.5, math.atan(80.0), math.pi / 2])
def test_trigflow_coeffs_match_oracle(lib, t):
    got = binding.trigflow_coeffs(t, 1000.0)
    ref = oracle.trigflow_coeffs(t, 1000.0)
    for g, r in zip(got, ref):
        assert abs(g - r) <= 1e-12 * max(abs(r), 1e-300) or abs(g - r) <= 1e-15
    assert lib.attn_jvp_last_error() == b""


@pytest.mark.parametrize("t", [0.0, 0.2, math.pi / 4, 1.3, math.pi / 2])
def test_trigflow_coeffs_jvp_match_oracle(lib, t):
    vals, tans = binding.trigflow_coeffs_jvp(t, -0.7, 1000.0)
    rv, rt = oracle.trigflow_coeffs_jvp(t, -0.7, 1000.0)
    for g, r in zip(vals + tans, rv + rt):
        assert abs(g - r) <= 1e-12 * max(abs(r), 1.0)
    with pytest.raises(binding.AttnJvpError):
        binding.trigflow_coeffs_jvp(-math.pi / 2, 1.0)


def test_epilogue_validation_needs_no_gpu(lib):
    E = binding
    vp = ctypes.c_void_p
    p4, p8 = vp(256), vp(256)
    out8 = [p4] * 4 + [p8, p8] + [p4, p4]
    assert lib.trigflow_output_jvp(None, *out8[1:], 2, 3, 4, 5, None) == E.ATTNJVP_EINVAL
    assert lib.trigflow_output_jvp(*out8, 1 << 20, 1 << 10, 1 << 10, 5, None) == E.ATTNJVP_EINVAL
    assert lib.trigflow_output_jvp(*out8, 2, 3, 4, 1 << 41, None) == E.ATTNJVP_EINVAL
    assert lib.trigflow_output_jvp(*out8, 2, 0, 4, 5, None) == E.ATTNJVP_EINVAL
    misaligned = [p4] * 4 + [vp(260), p8] + [p4, p4]  # t must be 8-byte aligned
    assert lib.trigflow_output_jvp(*misaligned, 2, 3, 4, 5, None) == E.ATTNJVP_EINVAL
    need = lib.scm_tangent_loss_workspace_bytes(2, 3, 4, 5)
    assert need > 0 and need % 8 == 0
    assert lib.scm_tangent_loss_workspace_bytes(2, 3, 4, 0) == E.ATTNJVP_EINVAL
    scm = lambda r, ws, nbytes: lib.scm_tangent_loss(*[p4] * 5, p8, ctypes.c_double(r), p4, p4, p8, p4, p4,
                                                     2, 3, 4, 5, ws, nbytes, None)
    assert scm(1.5, p8, need) == E.ATTNJVP_EINVAL
    assert b"warm-up" in lib.attn_jvp_last_error()
    assert scm(0.5, p8, need - 8) == E.ATTNJVP_EINVAL
    assert scm(0.5, None, need) == E.ATTNJVP_EINVAL


def test_backward_validation_needs_no_gpu(lib):
    E = binding
    vp = ctypes.c_void_p
    p = vp(256)
    assert lib.attn_bwd_workspace_bytes(2, 3, 517) >= 2 * 4 * 2 * 3 * 520
    assert lib.attn_bwd_workspace_bytes(0, 3, 5) == E.ATTNJVP_EINVAL
    need = lib.attn_bwd_workspace_bytes(2, 3, 300)  # the calls below use N_q = 300
    assert need % 256 == 0
    call = lambda ptrs, d=128, nq=300, nkv=700, ws=p, nbytes=need, scale=0.1: lib.attn_bwd(
        *ptrs, 2, 3, nq, nkv, d, ctypes.c_float(scale), ws, nbytes, None)
    good = [p] * 9
    assert call([vp(0)] + good[1:]) == E.ATTNJVP_EINVAL
    assert call(good[:3] + [vp(264)] + good[4:]) == E.ATTNJVP_EINVAL  # dout not 16-byte aligned
    assert b"dout" in lib.attn_jvp_last_error()
    assert call(good, d=512) == E.ATTNJVP_EUNSUPPORTED
    assert call(good, d=96) == E.ATTNJVP_EUNSUPPORTED
    assert b"head dim 96" in lib.attn_jvp_last_error()
    if not torch.cuda.is_available():  # placeholder pointers: never launch with them
        assert call(good, d=256) == E.ATTNJVP_ECUDA  # 256 passes every argument check
    assert call(good, nkv=0) == E.ATTNJVP_EINVAL
    assert call(good, scale=float("nan")) == E.ATTNJVP_EINVAL
    assert call(good, nbytes=need - 4) == E.ATTNJVP_EINVAL
    assert call(good, ws=vp(0x1040)) == E.ATTNJVP_EINVAL  # workspace not 256-byte aligned


def test_trigflow_coeffs_domain(lib):
    with pytest.raises(binding.AttnJvpError) as e:
        binding.trigflow_coeffs(-math.pi / 2)
    assert e.value.code == binding.ATTNJVP_EINVAL
    with pytest.raises(binding.AttnJvpError):
        binding.trigflow_coeffs(float("nan"))


def _strided(lib, strides=None, d=64, nq=100, nkv=300, kv=(0, 300), scale=0.1, dtype=binding.ATTNJVP_BF16):
    vp = ctypes.c_void_p
    st = None if strides is None else (ctypes.c_int64 * 9)(*strides)
    return lib.attn_jvp_fwd_strided(*[vp(256)] * 6, vp(256), vp(256), None, None, 2, 3, nq, nkv, d, st,
                                    ctypes.c_float(scale), dtype, kv[0], kv[1], None)


def test_strided_entry_validation_needs_no_gpu(lib):
    E = binding
    bshd = [nq * 3 * 64 for nq in (100,)] + [3 * 64, 64] + [300 * 3 * 64, 3 * 64, 64] + [100 * 3 * 64, 3 * 64, 64]
    assert _strided(lib, d=512) == E.ATTNJVP_EUNSUPPORTED
    assert b"16, 32, 64, 128 or 256" in lib.attn_jvp_last_error()
    assert _strided(lib, d=48) == E.ATTNJVP_EUNSUPPORTED
    assert _strided(lib, nkv=0, kv=(0, 1)) == E.ATTNJVP_EINVAL
    assert _strided(lib, kv=(250, 51)) == E.ATTNJVP_EINVAL
    assert _strided(lib, kv=(0, 0)) == E.ATTNJVP_EINVAL
    bad = list(bshd)
    bad[1] = 3 * 64 + 4  # query sequence stride: not a multiple of 8 elements (16 bytes)
    assert _strided(lib, bad) == E.ATTNJVP_EINVAL
    assert b"q stride 1" in lib.attn_jvp_last_error()
    bad = list(bshd)
    bad[5] = -64
    assert _strided(lib, bad) == E.ATTNJVP_EINVAL
    bad = list(bshd)
    bad[7] = 3 * 64 + 2  # output stride: not a multiple of 4 (float4 stores)
    assert _strided(lib, bad) == E.ATTNJVP_EINVAL
    assert b"out stride 1" in lib.attn_jvp_last_error()
    assert _strided(lib, scale=0.0) == E.ATTNJVP_EINVAL


def _ex(lib, strides=None, d=64, d_v=128, nq=100, nkv=300, scale=0.1, dtype=binding.ATTNJVP_BF16):
    vp = ctypes.c_void_p
    st = None if strides is None else (ctypes.c_int64 * 12)(*strides)
    return lib.attn_jvp_fwd_ex(*[vp(256)] * 6, vp(256), vp(256), None, None, 2, 3, nq, nkv, d, d_v, st,
                               ctypes.c_float(scale), dtype, 0, nkv, None)


def test_value_head_dim_entry_validation_needs_no_gpu(lib):
    E = binding
    assert _ex(lib, d_v=96) == E.ATTNJVP_EUNSUPPORTED
    assert _ex(lib, d=48, d_v=64) == E.ATTNJVP_EUNSUPPORTED
    assert _ex(lib, d_v=512) == E.ATTNJVP_EUNSUPPORTED
    # [B, S, H, D] strides for q (d = 64), k (d = 64), v (d_v = 128), out (d_v = 128)
    good = [100 * 3 * 64, 3 * 64, 64, 300 * 3 * 64, 3 * 64, 64, 300 * 3 * 128, 3 * 128, 128,
            100 * 3 * 128, 3 * 128, 128]
    bad = list(good)
    bad[7] = 3 * 128 + 4  # value row stride: not a multiple of 8 elements (TMA)
    assert _ex(lib, bad) == E.ATTNJVP_EINVAL
    assert b"v stride 1" in lib.attn_jvp_last_error()
    bad = list(good)
    bad[10] = 3 * 128 + 2  # output row stride: not a multiple of 4 (float4 stores)
    assert _ex(lib, bad) == E.ATTNJVP_EINVAL
    assert b"out stride 1" in lib.attn_jvp_last_error()
    assert _ex(lib, good, nkv=0) == E.ATTNJVP_EINVAL
    assert _ex(lib, good, scale=float("nan")) == E.ATTNJVP_EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_strided_call_without_device_reports_cuda_error(lib):
    bshd = [100 * 3 * 16, 3 * 16, 16, 300 * 3 * 16, 3 * 16, 16, 100 * 3 * 16, 3 * 16, 16]
    assert _strided(lib, bshd, d=16) == binding.ATTNJVP_ECUDA


def _host_call(lib, ws=256, ws_bytes=1 << 40, d=128, n_chunks=1, group=0, first=256):
    vp = ctypes.c_void_p
    ins = [vp(first)] + [vp(256)] * 5
    return lib.attn_jvp_fwd_host(*ins, vp(256), vp(256), None, None, 1, 4, 300, d, ctypes.c_float(0.1),
                                 n_chunks, group, vp(ws) if ws else None, ws_bytes, None)


def test_host_entry_validation_needs_no_gpu(lib):
    E = binding
    assert _host_call(lib, first=0) == E.ATTNJVP_EINVAL
    assert _host_call(lib, d=96) == E.ATTNJVP_EUNSUPPORTED
    assert _host_call(lib, ws=0) == E.ATTNJVP_EINVAL
    assert b"workspace" in lib.attn_jvp_last_error()
    assert _host_call(lib, ws=512 + 16) == E.ATTNJVP_EINVAL
    assert b"256-byte" in lib.attn_jvp_last_error()
    assert _host_call(lib, ws_bytes=1024) == E.ATTNJVP_EINVAL
    assert b"needs" in lib.attn_jvp_last_error()
    assert _host_call(lib, n_chunks=0) == E.ATTNJVP_EINVAL
    assert _host_call(lib, n_chunks=301) == E.ATTNJVP_EINVAL
    assert _host_call(lib, group=-1) == E.ATTNJVP_EINVAL


def test_host_workspace_size(lib):
    size = lambda *a: lib.attn_jvp_fwd_host_workspace_bytes(*a)
    B, H, N, d = 1, 40, 32760, 128
    auto = size(B, H, N, d, 1, 0)
    # automatic grouping: ceil(608 / ceil(N / 128)) = 3 heads per item, three slots
    per_head = 6 * N * d * 2 + 2 * N * d * 4 + 2 * N * 4
    assert auto >= 3 * 3 * per_head and auto < 3 * 3 * per_head + 3 * 10 * 256
    assert size(B, H, N, d, 1, 3) == auto
    assert size(B, H, N, d, 1, 1) < auto < size(B, H, N, d, 1, 40)
    assert size(B, H, N, d, 1, 400) == size(B, H, N, d, 1, 40)  # clamped to H
    assert size(B, H, N, d, 4, 3) > auto  # chunk partials
    assert size(B, H, N, 96, 1, 0) == binding.ATTNJVP_EUNSUPPORTED
    assert size(0, H, N, d, 1, 0) == binding.ATTNJVP_EINVAL
    with pytest.raises(binding.AttnJvpError):
        binding.attn_jvp_fwd_host_workspace_bytes((1, 2, 64, 96))


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.load(str(tmp_path / "libattnjvp.so"))


def test_dtype_code_is_checked_before_any_cuda_call(lib):
    """The forward entry points take the inputs' type as a code; anything but
    ATTNJVP_BF16 or ATTNJVP_FP32 is EINVAL, reported the same with or without a GPU."""
    E = binding
    assert (E.ATTNJVP_BF16, E.ATTNJVP_FP32) == (0, 1)
    for bad in (-1, 2, 7):
        assert _fwd(lib, dtype=bad) == E.ATTNJVP_EINVAL
        assert b"dtype code" in lib.attn_jvp_last_error()
        assert _fwd(lib, chunk=(0, 64), dtype=bad) == E.ATTNJVP_EINVAL
        assert _strided(lib, dtype=bad) == E.ATTNJVP_EINVAL
        assert _ex(lib, dtype=bad) == E.ATTNJVP_EINVAL
        assert lib.attn_jvp_fwd_split_noalloc(*[ctypes.c_void_p(256)] * 10, 1, 1, 64, 128, ctypes.c_float(0.1),
                                              bad, 2, None) == E.ATTNJVP_EINVAL
    # fp32 inputs are gathered with 16-byte loads: strides need only be multiples of 4
    # elements, where bf16 inputs (read by TMA) need multiples of 8.
    st = [100 * 3 * 64, 3 * 64 + 4, 64, 300 * 3 * 64, 3 * 64, 64, 100 * 3 * 64, 3 * 64, 64]
    assert _strided(lib, st) == E.ATTNJVP_EINVAL
    if not torch.cuda.is_available():  # the pointers here are placeholders: never launch with them
        rc = _strided(lib, st, dtype=E.ATTNJVP_FP32)
        assert rc == E.ATTNJVP_ECUDA, lib.attn_jvp_last_error()
    st[1] = 3 * 64 + 2
    assert _strided(lib, st, dtype=E.ATTNJVP_FP32) == E.ATTNJVP_EINVAL


def test_noalloc_checks_every_argument_before_launching(lib):
    """Sizes that would overflow, and NULL or misaligned outputs, are refused by the
    no-alloc entry before it computes its scratch layout or launches anything."""
    E = binding
    vp = ctypes.c_void_p
    call = lambda ptrs, B=1, H=1, N=64, d=128, n=2, dtype=E.ATTNJVP_BF16: lib.attn_jvp_fwd_split_noalloc(
        *ptrs, B, H, N, d, ctypes.c_float(0.1), dtype, n, None)
    good = [vp(256)] * 8 + [None, None]
    assert call(good[:6] + [None] + good[7:]) == E.ATTNJVP_EINVAL
    assert b"out" in lib.attn_jvp_last_error()
    assert call(good[:7] + [vp(264)] + good[8:]) == E.ATTNJVP_EINVAL
    assert b"16-byte" in lib.attn_jvp_last_error()
    assert call(good, B=1 << 40, H=1 << 40) == E.ATTNJVP_EINVAL
    assert b"2^31" in lib.attn_jvp_last_error()
    assert call(good, N=1 << 33) == E.ATTNJVP_EINVAL
    assert call(good, n=65) == E.ATTNJVP_EINVAL
    # 16 MiB of scratch: 1 x 64 x 128 rows of partials fit at 4 chunks; 64 x 1024 rows do not
    assert call(good, H=64, N=1024, n=4) == E.ATTNJVP_EINVAL
    assert b"scratch" in lib.attn_jvp_last_error()
    # fp32 inputs add their bf16 copies to the same limit
    msg_bf16 = lib.attn_jvp_last_error()
    assert call(good, H=64, N=1024, n=4, dtype=E.ATTNJVP_FP32) == E.ATTNJVP_EINVAL
    assert b"bf16 input copies" in lib.attn_jvp_last_error() and msg_bf16 != lib.attn_jvp_last_error()


def test_qk_norm_validation_needs_no_gpu(lib):
    E = binding
    vp = ctypes.c_void_p
    p = vp(256)
    call = lambda ptrs, rq=10, rk=12, d=128, eps=1e-6: lib.qk_rmsnorm_jvp(*ptrs, rq, rk, d, ctypes.c_float(eps), None)
    good = [p] * 10
    assert call(good, d=96) == E.ATTNJVP_EUNSUPPORTED
    assert call(good, eps=-1.0) == E.ATTNJVP_EINVAL
    assert call(good, eps=float("nan")) == E.ATTNJVP_EINVAL
    assert call(good, rq=-1) == E.ATTNJVP_EINVAL
    assert call([None] + good[1:]) == E.ATTNJVP_EINVAL
    assert b"q is NULL" in lib.attn_jvp_last_error()
    assert call(good[:5] + [vp(264)] + good[6:]) == E.ATTNJVP_EINVAL  # w_k misaligned
    assert b"w_k" in lib.attn_jvp_last_error()
    # with no K rows the K pointers are not needed; nothing to do at all is a no-op
    assert call(good[:2] + [None, None] + good[4:5] + [None] + good[6:], rq=0, rk=0) == E.ATTNJVP_OK


def test_last_wave_query_validation_needs_no_gpu(lib):
    out = ctypes.c_int64(-7)
    for args in ((0, 1, 100, 100, 64), (1, 1, 0, 100, 64), (1, 1, 100, 0, 64), (1 << 16, 1 << 15, 10, 10, 64)):
        assert lib.attn_jvp_fwd_last_wave_split(*args, ctypes.byref(out)) == binding.ATTNJVP_EINVAL
    assert lib.attn_jvp_fwd_last_wave_split(1, 1, 100, 100, 48, ctypes.byref(out)) == binding.ATTNJVP_EUNSUPPORTED
    assert lib.attn_jvp_fwd_last_wave_split(1, 1, 100, 100, 64, None) == binding.ATTNJVP_EINVAL
    if not torch.cuda.is_available():
        assert lib.attn_jvp_fwd_last_wave_split(1, 1, 100, 100, 64, ctypes.byref(out)) == binding.ATTNJVP_ECUDA
    assert out.value == -7
