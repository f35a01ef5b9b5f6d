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
    assert fwd_config(64, 64) == dict(NS=3, NSt=3, KS=3, VS=3, UPT=1, KU=3)
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


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dkdv", [True, False], ids=["dKdV", "dQ"])
@pytest.mark.parametrize("n_tiles", [1, 2, 3, 5, 9])
def test_backward_protocol_is_race_free(D, dkdv, n_tiles):
    cfg = bwd_config(D, dkdv)
    for seed in range(12):
        BwdModel(cfg, n_tiles, seed=1000 * n_tiles + seed).run()


def test_backward_two_groups_on_one_s1_slot_is_caught():
    # the reason the S1 barriers have one slot per tile parity at d = 128
    hits = 0
    for seed in range(40):
        try:
            BwdModel(bwd_config(128, True), 8, seed=seed, mutate="one_s1_slot").run()
        except ProtocolError:
            hits += 1
    assert hits > 0
