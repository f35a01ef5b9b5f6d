"""GPU: attn_jvp_fwd_host (host tensors in and out, transfers pipelined
against compute) returns exactly what the device-resident entry points
return for the same inputs, and agrees with the FP64 oracle.

Each pipelined item runs the same kernels on a [group, N, d] slice, and the
kernel's result for a head does not depend on which other heads share the
launch, so the comparison with the device path is bit for bit.
"""
import pytest
import torch

from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, gpu_rows, oracle_on

pytestmark = pytest.mark.gpu


def _device_reference(x, n_chunks):
    names = inputs.NAMES
    if n_chunks == 1:
        res = binding.attn_jvp_fwd(*(x[n] for n in names), scale=x["scale"])
    else:
        res = binding.attn_jvp_split(*(x[n] for n in names), n_chunks, scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    return [t.cpu() for t in res]


def _host_run(x, n_chunks, group_heads, pinned=True, rows=True):
    names = inputs.NAMES
    host_in = [x[n].cpu().pin_memory() if pinned else x[n].cpu() for n in names]
    B, H, N, d = x["q"].shape

    def alloc(shape):
        t = torch.full(shape, float("nan"), dtype=torch.float32)
        return t.pin_memory() if pinned else t

    out, out_t = alloc((B, H, N, d)), alloc((B, H, N, d))
    lse, mu = (alloc((B, H, N)), alloc((B, H, N))) if rows else (None, None)
    stream = torch.cuda.Stream()
    binding.attn_jvp_fwd_host(*host_in, out, out_t, lse, mu, scale=x["scale"], n_chunks=n_chunks,
                              group_heads=group_heads, stream=stream)
    stream.synchronize()
    binding.attn_jvp_status()
    return out, out_t, lse, mu


CASES = [
    # (B, H, N, d, n_chunks, group_heads)
    (2, 5, 300, 128, 1, 1),   # ten items of one head: both slots reused four times
    (1, 7, 517, 64, 1, 3),    # groups of 3, 3 and 1 heads
    (2, 3, 1000, 128, 3, 2),  # split path per item
    (1, 4, 129, 128, 1, 0),   # automatic group size (one item)
    (1, 3, 300, 256, 2, 2),   # head dim 256, split path, groups of 2 and 1 heads
]


@pytest.mark.parametrize("B,H,N,d,n_chunks,group_heads", CASES)
def test_host_path_matches_device_path_bitwise(cuda_lib, B, H, N, d, n_chunks, group_heads):
    x = inputs.make_inputs(B, H, N, d, seed=11 + N, device="cuda", qk="rms", tangent_scale=0.3)
    ref = _device_reference(x, n_chunks)
    got = _host_run(x, n_chunks, group_heads)
    for name, g, r in zip(("O", "Ot", "LSE", "mu"), got, ref):
        assert torch.equal(g, r), "%s differs from the device path" % name


def test_host_path_against_oracle(cuda_lib):
    x = inputs.make_inputs(1, 3, 700, 128, seed=5, device="cuda", qk="rms", tangent_scale=0.3)
    got = _host_run(x, 1, 1)
    ref = oracle_on(x)
    heads = list(range(3))
    assert_close(gpu_rows(got[0], heads, None), ref[0], "O")
    assert_close(gpu_rows(got[1], heads, None), ref[1], "Ot")
    assert_close(gpu_rows(got[3], heads, None), ref[3], "mu")


def test_host_path_without_row_outputs_and_pageable_memory(cuda_lib):
    x = inputs.make_inputs(1, 2, 256, 64, seed=3, device="cuda")
    ref = _device_reference(x, 1)
    got = _host_run(x, 1, 1, pinned=False, rows=False)
    assert got[2] is None and got[3] is None
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_host_path_rejects_small_workspace(cuda_lib):
    x = inputs.make_inputs(1, 2, 256, 64, seed=3, device="cuda")
    host_in = [x[n].cpu() for n in inputs.NAMES]
    out = torch.empty((1, 2, 256, 64), dtype=torch.float32)
    out_t = torch.empty_like(out)
    need = binding.attn_jvp_fwd_host_workspace_bytes((1, 2, 256, 64))
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.AttnJvpError) as e:
        binding.attn_jvp_fwd_host(*host_in, out, out_t, workspace=small)
    assert e.value.code == binding.ATTNJVP_EINVAL
