"""GPU: the entry points inside CUDA graph capture.

A caller may capture the library's calls into a CUDA graph and replay them.
Each case runs once eagerly first (the library looks up its device state on
the first call, which capture does not allow), then captures the same call on a
side stream, replays the graph on fresh inputs written into the captured input
buffers, and compares with an eager call on those inputs bit for bit.  The
shapes include a grid whose last wave the forward and the backward cut into
pieces, whose partials are then a graph memory node.
"""
import pytest
import torch

from attention_jvp_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def _cut_shape(d, N):
    per_head = (N + 127) // 128 * (2 if d == 256 else 1)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    return 1, n_sm // per_head + 1


def _capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            out = fn()
    torch.cuda.current_stream().wait_stream(s)
    return g, out


def _refill(x, seed):
    y = inputs.make_inputs(*x["q"].shape, seed=seed, device="cuda", qk="rms", tangent_scale=0.3)
    for n in inputs.NAMES:
        x[n].copy_(y[n])


@pytest.mark.parametrize("d,N,cut", [(128, 1000, True), (64, 300, False)])
def test_forward_replays_like_eager(cuda_lib, d, N, cut):
    B, H = _cut_shape(d, N) if cut else (1, 3)
    assert (binding.attn_jvp_fwd_last_wave_split(B, H, N, N, d) > 1) == cut
    x = inputs.make_inputs(B, H, N, d, seed=5, device="cuda", qk="rms", tangent_scale=0.3)
    args = [x[n] for n in inputs.NAMES]
    binding.attn_jvp_fwd(*args, scale=x["scale"])  # first call outside capture
    torch.cuda.synchronize()
    g, got = _capture(lambda: binding.attn_jvp_fwd(*args, scale=x["scale"]))
    _refill(x, 6)
    g.replay()
    torch.cuda.synchronize()
    want = binding.attn_jvp_fwd(*args, scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_split_path_and_backward_replay_like_eager(cuda_lib):
    d, N = 128, 1000
    B, H = _cut_shape(d, N)
    x = inputs.make_inputs(B, H, N, d, seed=7, device="cuda", qk="rms", tangent_scale=0.3)
    args = [x[n] for n in inputs.NAMES]
    dO = torch.randn((B, H, N, d), device="cuda").to(torch.bfloat16)
    ws = binding.split_workspace((B, H, N, d), 3, "cuda")

    def step():
        o, ot, lse, mu = binding.attn_jvp_split(*args, 3, scale=x["scale"], workspace=ws)
        dq, dk, dv = binding.attn_bwd(x["q"], x["k"], x["v"], dO, o, lse, scale=x["scale"])
        return o, ot, lse, mu, dq, dk, dv

    step()
    torch.cuda.synchronize()
    g, got = _capture(step)
    _refill(x, 8)
    g.replay()
    torch.cuda.synchronize()
    want = step()
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for a, b in zip(got, want):
        assert torch.equal(a, b)
