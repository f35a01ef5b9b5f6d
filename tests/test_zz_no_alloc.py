"""attn_jvp_fwd_split_noalloc: the split-KV path for callers that may not
allocate device memory (their host framework owns all device memory, or
cudaMalloc/cudaFree's implicit synchronisation is not allowed where they run).
Its chunk partials live in a fixed array inside the library.  Checked through
the C ABI against the split path with a caller-provided partial buffer
(attn_jvp_fwd_chunk + attn_jvp_merge), on two calls in a row of different
shapes, within the parity tolerances the other GPU tests use.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

from attention_jvp_gb300 import _build, binding, inputs
from helpers import assert_close, host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    return binding.load()


def _call_noalloc(lib, x, n_chunks, out, out_t, lse, mu):
    B, H, N, d = x["q"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.attn_jvp_fwd_split_noalloc(*(p(x[n]) for n in inputs.NAMES), p(out), p(out_t), p(lse), p(mu),
                                        B, H, N, d, ctypes.c_float(x["scale"]), n_chunks, stream)
    return rc


def test_noalloc_split_matches_caller_buffer_split(lib):
    cases = [(1, 2, 1000, 128, 4, 31), (2, 1, 700, 64, 3, 32)]  # two calls in a row, different shapes
    for B, H, N, d, chunks, seed in cases:
        x = inputs.make_inputs(B, H, N, d, seed=seed, device="cuda", qk="rms", tangent_scale=0.3)
        out = torch.empty((B, H, N, d), dtype=torch.float32, device="cuda")
        out_t = torch.empty_like(out)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        mu = torch.empty_like(lse)
        rc = _call_noalloc(lib, x, chunks, out, out_t, lse, mu)
        assert rc == binding.ATTNJVP_OK, lib.attn_jvp_last_error()
        ref = binding.attn_jvp_split(x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"], chunks,
                                     scale=x["scale"])
        torch.cuda.synchronize()
        binding.attn_jvp_status()
        for got, want, name in zip((out, out_t, mu), ref[:2] + ref[3:], ("O", "Ot", "mu")):
            assert_close(host64(got), host64(want), name)
        assert float((lse - ref[2]).abs().max()) <= 1e-3


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    # 4 chunks x 1 x 8 x 4096 rows x (2*128+2) x 4 bytes = 135 MB > 16 MiB
    B, H, N, d = 1, 8, 4096, 128
    x = inputs.make_inputs(1, 1, 8, d, seed=1, device="cuda")  # pointers are never dereferenced
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.attn_jvp_fwd_split_noalloc(*(p(x[n]) for n in inputs.NAMES), p(dummy), p(dummy), None, None,
                                        B, H, N, d, ctypes.c_float(0.1), 4, None)
    assert rc == binding.ATTNJVP_EINVAL
    assert b"scratch" in lib.attn_jvp_last_error()
