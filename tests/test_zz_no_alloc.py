"""attn_jvp_fwd_split_noalloc: the split-KV path for callers that may not
allocate device memory (their host framework owns all device memory, or
cudaMalloc/cudaFree's implicit synchronisation is not allowed where they run).
Its chunk partials live in a fixed array inside the library.

Checked through the C ABI, on calls in a row of different shapes, against the
FP64 oracle on every row and against the split path with a caller-provided
partial buffer (attn_jvp_fwd_chunk + attn_jvp_merge), within the parity
tolerances the other GPU tests use.  The cases cover head dim 256 (two CTAs
write each row's partials), one chunk, one key per chunk, fp32 inputs (their
bf16 copies share the array) and a call without LSE and mu.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from attention_jvp_gb300 import _build, binding, inputs
from helpers import assert_close, gpu_rows, host64, lse_tolerance, oracle_on

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return binding.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, x, n_chunks, out, out_t, lse, mu):
    B, H, N, d = x["q"].shape
    code = binding.ATTNJVP_FP32 if x["q"].dtype == torch.float32 else binding.ATTNJVP_BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.attn_jvp_fwd_split_noalloc(*(_p(x[n]) for n in inputs.NAMES), _p(out), _p(out_t), _p(lse), _p(mu),
                                          B, H, N, d, ctypes.c_float(x["scale"]), code, n_chunks, stream)


CASES = [
    # (B, H, N, d, n_chunks, seed, recipe extras)
    (1, 2, 1000, 128, 4, 31, dict(qk="rms", tangent_scale=0.3)),
    (2, 1, 700, 64, 3, 32, dict(qk="rms", tangent_scale=0.3)),
    (1, 1, 1000, 256, 3, 33, dict(qk="rms", tangent_scale=0.3)),   # two CTAs per query tile
    (1, 1, 300, 128, 1, 34, dict(outlier_frac=0.01)),               # a single chunk
    (1, 1, 40, 64, 40, 35, {}),                                     # one key per chunk
    (1, 2, 256, 64, 4, 36, dict(dtype=torch.float32)),              # fp32: bf16 copies in the array
]


def test_noalloc_split_matches_oracle_and_caller_buffer_split(lib):
    for B, H, N, d, chunks, seed, extra in CASES:  # calls in a row, different shapes
        x = inputs.make_inputs(B, H, N, d, seed=seed, device="cuda", **extra)
        out = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
        out_t = torch.empty_like(out)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        mu = torch.empty_like(lse)
        rc = _call_noalloc(lib, x, chunks, out, out_t, lse, mu)
        assert rc == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
        torch.cuda.synchronize()
        assert binding.attn_jvp_status() == 0
        ref = oracle_on(x)
        heads = list(range(B * H))
        for got, want, name in zip((out, out_t, mu), (ref[0], ref[1], ref[3]), ("O", "Ot", "mu")):
            assert_close(gpu_rows(got, heads), want, "%s (N=%d, d=%d, %d chunks)" % (name, N, d, chunks))
        assert np.all(np.abs(gpu_rows(lse, heads) - ref[2]) <= lse_tolerance(x, heads))
        split = binding.attn_jvp_split(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], chunks,
                                       scale=x["scale"])
        torch.cuda.synchronize()
        for got, want, name in zip((out, out_t, mu), split[:2] + split[3:], ("O", "Ot", "mu")):
            assert_close(host64(got), host64(want), name)
        assert float((lse - split[2]).abs().max()) <= 1e-3


def test_noalloc_without_lse_and_mu(lib):
    B, H, N, d, chunks = 1, 2, 600, 128, 3
    x = inputs.make_inputs(B, H, N, d, seed=37, device="cuda", qk="rms", tangent_scale=0.3)
    full = [torch.empty((B, H, N, d), dtype=torch.float32, device="cuda") for _ in range(2)]
    rows = [torch.empty((B, H, N), dtype=torch.float32, device="cuda") for _ in range(2)]
    assert _call_noalloc(lib, x, chunks, *full, *rows) == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
    only = [torch.full((B, H, N, d), float("nan"), dtype=torch.float32, device="cuda") for _ in range(2)]
    assert _call_noalloc(lib, x, chunks, *only, None, None) == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
    torch.cuda.synchronize()
    assert binding.attn_jvp_status() == 0
    # the same arithmetic with or without the per-row outputs
    assert torch.equal(only[0], full[0]) and torch.equal(only[1], full[1])
    ref = oracle_on(x)
    assert_close(host64(only[0]), ref[0].reshape(only[0].shape), "O")
    assert_close(host64(only[1]), ref[1].reshape(only[1].shape), "Ot")


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    # 4 chunks x 1 x 8 x 4096 rows x (2*128+2) x 4 bytes = 135 MB > 16 MiB
    B, H, N, d = 1, 8, 4096, 128
    x = inputs.make_inputs(1, 1, 8, d, seed=1, device="cuda")  # pointers are never dereferenced
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    rc = lib.attn_jvp_fwd_split_noalloc(*(_p(x[n]) for n in inputs.NAMES), _p(dummy), _p(dummy), None, None,
                                        B, H, N, d, ctypes.c_float(0.1), binding.ATTNJVP_BF16, 4, None)
    assert rc == binding.ATTNJVP_EINVAL
    assert b"scratch" in lib.attn_jvp_last_error()
