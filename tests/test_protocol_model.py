"""Host-side race check of the fused forward kernel's mbarrier hand-offs.

compute-sanitizer is not available on the GPU pool, and a protocol race shows
on a GPU only as a rare wrong tile or a timed-out wait.  So the protocol is
run as a CPU model (``protocol_model.py``) with random completion orders, for
every ring configuration the kernel instantiates, and held to exact mbarrier
parity semantics.  Planted mistakes show that the model catches the errors it
is there for.
"""
import pytest

from protocol_model import BwdModel, FwdModel, ProtocolError, bwd_config, fwd_config

PAIRS = [(d, dv) for d in (64, 128, 256) for dv in (64, 128, 256)]


def test_configs_match_the_kernel_sizes():
    # the combinations the design notes list: 3 stages at 64, 2 at 128, one
    # tile in two units at 256 (Q/K dim), and the TMEM buffers by value dim
    assert fwd_config(64, 64) == dict(NS=1, NSt=5, KS=3, VS=3, UPT=1, KU=3)
    assert fwd_config(128, 128) == dict(NS=1, NSt=3, KS=2, VS=2, UPT=1, KU=2)
    assert fwd_config(256, 256) == dict(NS=1, NSt=3, KS=1, VS=1, UPT=2, KU=2)
    assert fwd_config(256, 64)["KS"] == 1 and fwd_config(128, 64)["KS"] == 3
    assert fwd_config(128, 256)["KS"] == 2 and fwd_config(64, 256)["KS"] == 3


@pytest.mark.parametrize("d,dv", PAIRS)
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 4, 7])
def test_protocol_is_race_free(d, dv, n_tiles):
    cfg = fwd_config(d, dv)
    for seed in range(12):
        FwdModel(cfg, n_tiles, seed=1000 * n_tiles + seed).run()


def _caught(cfg, mutate, n_tiles=6, seeds=40):
    hits = 0
    for seed in range(seeds):
        try:
            FwdModel(cfg, n_tiles, seed=seed, mutate=mutate).run()
        except ProtocolError:
            hits += 1
    return hits


@pytest.mark.parametrize("mutate", ["S_no_free_wait", "St_no_free_wait", "rescale_no_wait"])
def test_planted_mistakes_are_caught(mutate):
    assert _caught(fwd_config(128, 128), mutate) > 0


def test_one_barrier_slot_for_two_groups_is_caught():
    # Two consumers alternating on one single-slot barrier: the later one can
    # be two phases behind, which a parity test cannot see.
    from protocol_model import Bar
    m = FwdModel(fwd_config(128, 128), 1, seed=0)
    bar = Bar("shared", 1)
    bar.arrive()
    bar.arrive()  # phases 0 and 1 complete before the slow consumer looks at phase 0
    with pytest.raises(ProtocolError):
        list(m.wait(bar, 0))
    # and a waiter for a phase whose predecessor is incomplete is caught too
    bar2 = Bar("early", 1)
    with pytest.raises(ProtocolError):
        list(m.wait(bar2, 1))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dkdv", [True, False], ids=["dKdV", "dQ"])
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 9])
def test_backward_protocol_is_race_free(D, dkdv, n_tiles):
    cfg = bwd_config(D, dkdv)
    for seed in range(12):
        BwdModel(cfg, n_tiles, seed=1000 * n_tiles + seed).run()


def test_backward_shared_stage_without_the_value_release_is_caught():
    # the score ring's stage also feeds the value MMAs up to head dim 128; released
    # after the two score issuers alone, it would be reloaded under the value MMAs
    for D in (64, 128):
        hits = 0
        for seed in range(40):
            try:
                BwdModel(bwd_config(D, True), 9, seed=seed, mutate="shared_stage_two_arrivals").run()
            except ProtocolError:
                hits += 1
        assert hits > 0, D


def test_backward_two_groups_on_one_s1_slot_is_caught():
    # the reason the S1 barriers have one slot per tile parity at d = 128
    hits = 0
    for seed in range(40):
        try:
            BwdModel(bwd_config(128, True), 8, seed=seed, mutate="one_s1_slot").run()
        except ProtocolError:
            hits += 1
    assert hits > 0


# ---------------------------------------------------------------------------
# The model's ring sizes against the kernels' own compile-time configuration
# ---------------------------------------------------------------------------
CFG_HARNESS = r"""
#include <cstdint>
#include <cstdio>
constexpr int kModeDQ = 0;
constexpr int kModeDKDV = 1;
%s
%s
template <int D, int DV> void fwd() {
  using C = FwdCfg<D, DV>;
  printf("fwd %%d %%d %%d %%d %%d %%d %%d %%d\n", D, DV, C::kNS, C::kNSt, C::kKS, C::kVS, C::kUPT, C::kKU);
}
template <int D, int M> void bwd() {
  using C = BwdCfg<D, M>;
  printf("bwd %%d %%d %%d %%d %%d %%d %%d %%d %%d %%d %%d\n", D, M, C::kNS, C::kNSt, C::kSBar, C::kKS, C::kVS,
         C::kVecS, C::kUPT, C::kKU, int(C::kShared));
}
int main() {
  fwd<64, 64>(); fwd<64, 128>(); fwd<64, 256>(); fwd<128, 64>(); fwd<128, 128>(); fwd<128, 256>();
  fwd<256, 64>(); fwd<256, 128>(); fwd<256, 256>();
  bwd<64, 0>(); bwd<64, 1>(); bwd<128, 0>(); bwd<128, 1>(); bwd<256, 0>(); bwd<256, 1>();
  return 0;
}
"""


def test_model_sizes_are_the_kernels_sizes(tmp_path):
    import os
    import re
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "attention_jvp_gb300", "csrc")
    fwd_src = open(os.path.join(csrc, "attn_jvp_fwd.cu"), encoding="utf-8").read()
    bwd_src = open(os.path.join(csrc, "attn_bwd.cu"), encoding="utf-8").read()
    fcfg = re.search(r"template <int D, int DVF>\nstruct FwdCfg \{.*?\n\};\n", fwd_src, re.S)
    bcfg = re.search(r"template <int D, int kMode>\nstruct BwdCfg \{.*?\n\};\n", bwd_src, re.S)
    assert fcfg and bcfg, "FwdCfg / BwdCfg not found in the kernel sources"
    (tmp_path / "cfg.cpp").write_text(CFG_HARNESS % (fcfg.group(0), bcfg.group(0)))
    exe = tmp_path / "cfg"
    subprocess.run([cxx, "-std=c++17", str(tmp_path / "cfg.cpp"), "-o", str(exe)], check=True)
    seen = 0
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        kind, *v = line.split()
        v = [int(x) for x in v]
        if kind == "fwd":
            want = fwd_config(v[0], v[1])
            assert (want["NS"], want["NSt"], want["KS"], want["VS"], want["UPT"], want["KU"]) == tuple(v[2:]), line
        else:
            want = bwd_config(v[0], v[1] == 1)
            assert (want["NS"], want["NSt"], want["SBar"], want["KS"], want["VS"], want["VecS"], want["UPT"],
                    want["KU"], int(want["shared"])) == tuple(v[2:]), line
        seen += 1
    assert seen == 15


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (256, 256), (256, 64)])
def test_abort_path_drains_and_terminates(d, dv):
    # A bounded wait gives up at a random point; every role must still finish, and
    # nothing a role started may be in flight when the CTA releases its memory.
    from protocol_model import AbortFwdModel
    cfg = fwd_config(d, dv)
    for seed in range(60):
        AbortFwdModel(cfg, 6, seed=seed, abort_at=seed * 7).run()


def test_abort_path_catches_a_producer_that_does_not_drain():
    from protocol_model import AbortFwdModel

    class NoDrain(AbortFwdModel):
        def tma_k(self):
            c = self.c
            self.later("tmaK", self.q_full.arrive)
            for n in range(self.n * c["UPT"]):
                s = n % c["KU"]
                ok = yield from self.wait_or_abort(self.k_empty[s], n // c["KU"] - 1)
                if not ok:
                    return  # gives up without waiting for its copies
                self.later("tmaK", self.k_full[s].arrive)
                if n == self.n * c["UPT"] - 2:
                    self.aborted = True  # a wait elsewhere gives up with this copy in flight

    hits = 0
    for seed in range(100):
        try:
            NoDrain(fwd_config(128, 128), 6, seed=seed, abort_at=-1).run()
        except ProtocolError:
            hits += 1
    assert hits >= 50


def test_abort_right_after_the_last_copy():
    """Another role gives up just after the last copy was issued: the TMA threads still
    wait for their last copies, so none lands in memory the CTA has released."""
    from protocol_model import AbortFwdModel

    class AbortAfterLastCopy(AbortFwdModel):
        def tma_k(self):
            yield from super().tma_k()
            if any(q.startswith("tma") for q, _ in self.pending):
                self.aborted = True  # another role's wait gives up now

    for seed in range(100):
        AbortAfterLastCopy(fwd_config(128, 128), 6, seed=seed, abort_at=-1).run()


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("dkdv", [True, False], ids=["dKdV", "dQ"])
def test_backward_abort_path_drains_and_terminates(D, dkdv):
    from protocol_model import AbortBwdModel
    cfg = bwd_config(D, dkdv)
    for seed in range(60):
        AbortBwdModel(cfg, 7, seed=seed, abort_at=seed * 9).run()


def test_backward_abort_right_after_the_last_copy():
    from protocol_model import AbortBwdModel

    class AbortAfterLastCopy(AbortBwdModel):
        def producer(self):
            yield from super().producer()
            if any(q.startswith("tma") for q, _ in self.pending):
                self.aborted = True

    for seed in range(100):
        AbortAfterLastCopy(bwd_config(128, True), 7, seed=seed, abort_at=-1).run()


@pytest.mark.parametrize("n_items", [1, 2, 3, 4, 7, 12])
def test_host_pipeline_streams_are_race_free(n_items):
    from protocol_model import HostPipelineModel
    for seed in range(40):
        HostPipelineModel(n_items, seed).run()


@pytest.mark.parametrize("mutate", ["no_copied_wait", "no_computed_wait"])
def test_host_pipeline_missing_waits_are_caught(mutate):
    from protocol_model import HostPipelineModel
    hits = 0
    for seed in range(60):
        try:
            HostPipelineModel(9, seed, mutate=mutate).run()
        except ProtocolError:
            hits += 1
    assert hits > 0
