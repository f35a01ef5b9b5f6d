"""GPU: the cut of a short last wave into pieces over the keys.

The fused kernel runs one CTA per SM, so a grid of (query tile, value half)
units runs in waves of the SM count.  When the last wave is at most half full,
attn_jvp_fwd cuts each of its units into pieces over consecutive key ranges
(at least four key tiles each) and merges them exactly afterwards.  The shapes
here are chosen from the device's SM count so that the grid is one wave plus a
short tail; the units of the tail are then the last heads' query tiles.

The cut heads are checked against the FP64 oracle with the usual tolerances.
They are not compared bit for bit with an uncut run: each piece rounds its own
P~ = 2^(S - m) to bf16 against its own running maximum, so the roundings differ
(both runs stay within the oracle's tolerance).  Every head whose units all ran
in the first wave must equal the uncut run (the chunk entry point over the whole
key range, which never cuts) bit for bit.
"""
import numpy as np
import pytest
import torch

from attention_jvp_gb300 import binding, inputs
from helpers import assert_close, gpu_rows, oracle_on

pytestmark = pytest.mark.gpu


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _shape(d, n_qtiles):
    """(B, H) with B*H*n_qtiles*(2 if d == 256) units: one wave plus a tail of
    at most a quarter of the SMs, so the tail is cut (n_qtiles divides the
    units, so the tail is whole heads' worth of query tiles)."""
    per_head = n_qtiles * (2 if d == 256 else 1)
    n_sm = _sm_count()
    heads = n_sm // per_head + 1
    assert 0 < heads * per_head - n_sm <= n_sm // 4
    return 1, heads


def _whole_range(x):
    N = x["q"].shape[2]
    out = binding.attn_jvp_fwd_chunk(*(x[n] for n in inputs.NAMES), 0, N, scale=x["scale"])
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d,N", [(64, 1000), (128, 1000), (256, 1000), (32, 777)])
def test_cut_tail_matches_oracle_and_uncut_path(cuda_lib, d, N):
    n_qtiles = (N + 127) // 128
    B, H = _shape(d, n_qtiles)
    x = inputs.make_inputs(B, H, N, d, seed=70 + d, device="cuda", qk="rms", tangent_scale=0.3)
    got = binding.attn_jvp_fwd(*(x[n] for n in inputs.NAMES), scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    ref = _whole_range(x)
    # the cut units are those past the first wave: the last heads' query tiles
    per_head = n_qtiles * (2 if d == 256 else 1)
    first_cut = _sm_count() // per_head
    for name, g, r in zip(("O", "Ot", "LSE", "mu"), got, ref):
        assert torch.equal(g[:, :first_cut], r[:, :first_cut]), name
    heads = list(range(first_cut, B * H))
    o = oracle_on(x, heads=heads)
    assert_close(gpu_rows(got[0], heads), o[0], "O")
    assert_close(gpu_rows(got[1], heads), o[1], "Ot")
    assert_close(gpu_rows(got[3], heads), o[3], "mu")
    assert np.max(np.abs(gpu_rows(got[2], heads) - o[2])) <= 1e-3


def test_cut_tail_with_strided_outputs_and_no_row_outputs(cuda_lib):
    d, N = 128, 1000
    B, H = _shape(d, (N + 127) // 128)
    x = inputs.make_inputs(B, H, N, d, seed=81, device="cuda", qk="rms", tangent_scale=0.3)
    ref = binding.attn_jvp_fwd(*(x[n] for n in inputs.NAMES), scale=x["scale"])
    # the same values in [B, N, H, d]; outputs in that layout too
    xs = {n: x[n].transpose(1, 2).contiguous() for n in inputs.NAMES}
    got = binding.attn_jvp_fwd_strided(*(xs[n] for n in inputs.NAMES), layout="bshd", scale=x["scale"])
    only = binding.attn_jvp_fwd(*(x[n] for n in inputs.NAMES), scale=x["scale"], want_rows=False)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    assert torch.equal(got[0].transpose(1, 2), ref[0]) and torch.equal(got[1].transpose(1, 2), ref[1])
    assert torch.equal(got[2], ref[2]) and torch.equal(got[3], ref[3])
    assert only[2] is None and only[3] is None
    assert torch.equal(only[0], ref[0]) and torch.equal(only[1], ref[1])


def test_cut_tail_with_fp32_inputs(cuda_lib):
    d, N = 64, 1000
    B, H = _shape(d, (N + 127) // 128)
    x = inputs.make_inputs(B, H, N, d, seed=83, device="cuda", dtype=torch.float32)
    got = binding.attn_jvp_fwd(*(x[n] for n in inputs.NAMES), scale=x["scale"])
    xb = {n: x[n].to(torch.bfloat16) for n in inputs.NAMES}
    ref = binding.attn_jvp_fwd(*(xb[n] for n in inputs.NAMES), scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for g, r in zip(got, ref):
        assert torch.equal(g, r)



def _documented_split(grid, kv_len, n_sm):
    # the header's rule: cut only a last wave at most half full, into as many
    # pieces as spread it over the SMs, each at least four 64-key tiles, at most 16
    tail = grid % n_sm
    if grid < n_sm or tail == 0 or 2 * tail > n_sm:
        return 1
    split = min(n_sm // tail, ((kv_len + 63) // 64) // 4, 16)
    return split if split >= 2 else 1


def test_last_wave_query_follows_the_documented_rule(cuda_lib):
    n_sm = _sm_count()
    seen = set()
    for B, H, Nq, Nkv, dv in [(1, n_sm // 8 + 1, 1000, 1000, 128), (1, n_sm, 128, 1000, 128),
                              (1, 1, 128, 1000, 128), (1, n_sm + 1, 128, 100, 128),
                              (1, n_sm + 1, 128, 4096, 128), (1, n_sm + n_sm // 2 + 1, 128, 4096, 128),
                              (2, 24, 4096, 4096, 128), (1, 40, 32760, 32760, 128), (4, 16, 16384, 16384, 64),
                              (1, n_sm // 2 + 1, 128, 4096, 256), (1, 7, 777, 300, 32)]:
        grid = (Nq + 127) // 128 * B * H * (2 if dv > 128 else 1)
        want = _documented_split(grid, Nkv, n_sm)
        assert binding.attn_jvp_fwd_last_wave_split(B, H, Nq, Nkv, dv) == want, (B, H, Nq, Nkv, dv)
        seen.add(want > 1)
    assert seen == {True, False}


@pytest.mark.parametrize("d,N", [(128, 1000), (64, 777), (256, 1000)])
def test_backward_cut_tail_matches_oracle_and_uncut_heads(cuda_lib, d, N):
    """The backward's two passes cut a short last wave the same way, over their
    streamed rows (queries in the dK/dV pass, keys in the dQ pass), and add the
    pieces' partial sums.  Heads whose units all ran in the first wave equal a
    run over those heads alone (whole waves, no cut) bit for bit; the cut heads
    are checked against the FP64 oracle."""
    import oracle
    from helpers import host64
    n_qtiles = (N + 127) // 128
    B, H = _shape(d, n_qtiles)
    per_head = n_qtiles * (2 if d == 256 else 1)
    assert binding.attn_jvp_fwd_last_wave_split(B, H, N, N, d) > 1  # the backward uses the same rule
    g = torch.Generator(device="cuda").manual_seed(90 + d)
    q, k, v, dO = (torch.randn((B, H, N, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    scale = d ** -0.5
    z = torch.zeros_like(q)
    o, _, lse, _ = binding.attn_jvp_fwd_chunk(q, k, v, z, z, z, 0, N, scale=scale)
    got = binding.attn_bwd(q, k, v, dO, o, lse, scale=scale)
    first_cut = _sm_count() // per_head
    sub = lambda t: t[:, :first_cut].contiguous()  # noqa: E731
    ref = binding.attn_bwd(sub(q), sub(k), sub(v), sub(dO), sub(o), sub(lse), scale=scale)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
        assert torch.equal(a[:, :first_cut], b), name
    for h in range(first_cut, H):
        want = oracle.attn_bwd(host64(q[0, h]), host64(k[0, h]), host64(v[0, h]), host64(dO[0, h]), scale)
        for name, a, r in zip(("dQ", "dK", "dV"), got, want):
            assert_close(host64(a[0, h]), r, "%s head %d" % (name, h))


def test_cut_tail_cross_attention_with_own_value_dim(cuda_lib):
    """N_q != N_kv and d_v != d through the general entry point over the whole key
    range: the forward cuts (its units are query tiles); the backward's dQ pass cuts
    and its dK/dV pass (fewer key tiles than one wave) does not."""
    import oracle
    from helpers import host64
    d, dv, Nq, Nkv = 128, 64, 1000, 700
    B, H = _shape(128, (Nq + 127) // 128)
    assert binding.attn_jvp_fwd_last_wave_split(B, H, Nq, Nkv, dv) > 1
    g = torch.Generator(device="cuda").manual_seed(97)
    mk = lambda n, c: (torch.randn((B, H, n, c), generator=g, device="cuda") * 0.8).to(torch.bfloat16)  # noqa: E731
    q, qt, k, kt = mk(Nq, d), mk(Nq, d), mk(Nkv, d), mk(Nkv, d)
    v, vt = mk(Nkv, dv), mk(Nkv, dv)
    s = d ** -0.5
    got = binding.attn_jvp_fwd_strided(q, k, v, qt, kt, vt, scale=s)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    first_cut = _sm_count() // ((Nq + 127) // 128)
    for h in range(first_cut, H):
        o = oracle.attn_jvp(host64(q[0, h]), host64(k[0, h]), host64(v[0, h]), host64(qt[0, h]),
                            host64(kt[0, h]), host64(vt[0, h]), s)
        assert_close(host64(got[0][0, h]), o[0], "O head %d" % h)
        assert_close(host64(got[1][0, h]), o[1], "Ot head %d" % h)
        assert_close(host64(got[3][0, h]), o[3], "mu head %d" % h)
    # backward (d_v = d required): the dQ pass cuts, the dK/dV pass does not
    v2, dO = mk(Nkv, d), mk(Nq, d)
    z = torch.zeros_like
    o2, _, lse2, _ = binding.attn_jvp_fwd_strided(q, k, v2, z(q), z(k), z(v2), scale=s)
    dq, dk, dv_ = binding.attn_bwd(q, k, v2, dO, o2, lse2, scale=s)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    for h in range(first_cut, H):
        want = oracle.attn_bwd(host64(q[0, h]), host64(k[0, h]), host64(v2[0, h]), host64(dO[0, h]), s)
        for name, a, r in zip(("dQ", "dK", "dV"), (dq, dk, dv_), want):
            assert_close(host64(a[0, h]), r, "%s head %d" % (name, h))


def test_image_dit_workload_cut_rows_at_full_size(cuda_lib):
    """The image DiT 1K workload (B=2, H=24, N=4096, d=128) as the benchmark runs it: on a
    152-SM GB300 its 1536 units leave a 16-unit last wave, which is cut.  Seeded rows of
    the cut units (the last head's second half, on such a GPU) against the oracle."""
    from helpers import gpu_rows, oracle_on
    spec = inputs.WORKLOADS["image_dit_1k"]
    B, H, N, d = spec["B"], spec["H"], spec["N"], spec["d"]
    n_sm = _sm_count()
    grid = B * H * (N // 128)
    pieces = binding.attn_jvp_fwd_last_wave_split(B, H, N, N, d)
    tail = grid % n_sm
    if pieces == 1:
        pytest.skip("this GPU's SM count (%d) leaves no short last wave for this workload" % n_sm)
    x = inputs.workload_inputs("image_dit_1k", device="cuda")
    got = binding.attn_jvp_fwd(*(x[n] for n in inputs.NAMES), scale=x["scale"])
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    # cut units: the last ``tail`` (query tile) units, i.e. flat heads / tiles at the end
    first_unit = grid - tail
    units = range(first_unit, grid)
    heads = sorted(set(u // (N // 128) for u in units))
    rng = np.random.default_rng(101)
    for h in heads:
        tiles = [u % (N // 128) for u in units if u // (N // 128) == h]
        rows = np.unique(np.concatenate([rng.integers(t * 128, t * 128 + 128, 6) for t in tiles]))
        ref = oracle_on(x, heads=[h], rows=rows)
        g = [gpu_rows(t, [h], rows) for t in got]
        assert_close(g[0], ref[0], "O")
        assert_close(g[1], ref[1], "Ot")
        assert_close(g[3], ref[3], "mu")
        assert np.max(np.abs(g[2] - ref[2])) <= 1e-3


def test_cut_into_the_most_pieces(cuda_lib):
    """One unit past a whole wave, over 4096 keys: the lone unit is cut into the most
    pieces (16 of four key tiles each).  Its rows against the oracle, and a second
    identical call bit for bit (the cut and its merge are deterministic)."""
    import oracle
    from helpers import host64
    n_sm = _sm_count()
    B, H, Nq, Nkv, d = 1, n_sm + 1, 128, 4096, 64
    assert binding.attn_jvp_fwd_last_wave_split(B, H, Nq, Nkv, d) == 16
    g = torch.Generator(device="cuda").manual_seed(131)
    mk = lambda n: torch.randn((B, H, n, d), generator=g, device="cuda").to(torch.bfloat16)  # noqa: E731
    q, qt, k, kt, v, vt = mk(Nq), mk(Nq), mk(Nkv), mk(Nkv), mk(Nkv), mk(Nkv)
    s = d ** -0.5
    got = binding.attn_jvp_fwd_strided(q, k, v, qt, kt, vt, scale=s)
    ref = binding.attn_jvp_fwd_strided(q, k, v, qt, kt, vt, scale=s, kv_start=0, kv_len=Nkv)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    h = H - 1
    o = oracle.attn_jvp(host64(q[0, h]), host64(k[0, h]), host64(v[0, h]), host64(qt[0, h]), host64(kt[0, h]),
                        host64(vt[0, h]), s)
    assert_close(host64(got[0][0, h]), o[0], "O")
    assert_close(host64(got[1][0, h]), o[1], "Ot")
    assert_close(host64(got[3][0, h]), o[3], "mu")
    assert np.max(np.abs(host64(got[2][0, h]) - o[2])) <= 1e-3
    for a, b in zip(got, ref):
        assert torch.equal(a, b)  # the same call twice: the cut is deterministic
