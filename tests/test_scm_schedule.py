"""Host check of the sCM pass's ticket order (the persistent grid's scheduler).

The fused target / reduce / normalise pass hands out work by ticket: a block
takes the next ticket and runs the item ``unit_of`` maps it to.  A
normalisation item waits for its sample's scale, published by the last of that
sample's target items.  The wait always ends only if every target item of a
sample holds an earlier ticket than any normalisation item of that sample:
tickets are taken in order and only by running blocks, so the item with the
smallest unfinished ticket never waits on anything unfinished.

This test compiles ``unit_of`` from the kernel source itself (extracted as
text, with the device qualifiers defined away) with the host compiler, and
checks over many (items per sample, samples) that the order is a bijection
onto the 2 B n items, that the lag puts min(8, B) samples of target items
before a sample's first normalisation item, and that a simulated grid of
resident blocks taking tickets in order always finishes.
"""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "attention_jvp_gb300", "csrc", "epilogue.cu")

HARNESS = r"""
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#define __device__
#define __forceinline__ inline
%s
int main(int argc, char** argv) {
  const int64_t n = atoll(argv[1]);
  const int B = atoi(argv[2]);
  for (unsigned long long j = 0; j < 2ull * B * n; ++j) {
    const Unit u = unit_of(j, n, B);
    printf("%%d %%d %%lld\n", u.normalise ? 1 : 0, u.b, (long long)u.item);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def ticket_order(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = open(SRC, encoding="utf-8").read()
    unit = re.search(r"struct Unit \{.*?\n\};\n", src, re.S)
    fn = re.search(r"__device__ __forceinline__ Unit unit_of\(.*?\n\}\n", src, re.S)
    assert unit and fn, "unit_of / Unit not found in epilogue.cu"
    d = tmp_path_factory.mktemp("scm_schedule")
    (d / "h.cpp").write_text(HARNESS % (unit.group(0) + fn.group(0)))
    exe = d / "h"
    subprocess.run([cxx, "-O1", "-std=c++17", str(d / "h.cpp"), "-o", str(exe)], check=True)

    def run(n, B):
        out = subprocess.run([str(exe), str(n), str(B)], check=True, capture_output=True, text=True).stdout
        return [tuple(int(x) for x in ln.split()) for ln in out.splitlines()]
    return run


CASES = [(1, 1), (3, 1), (5, 2), (7, 3), (2, 8), (4, 9), (6, 17), (1, 33), (11, 33), (3, 64)]


@pytest.mark.parametrize("n,B", CASES)
def test_order_is_a_bijection_and_targets_come_first(ticket_order, n, B):
    order = ticket_order(n, B)
    assert len(order) == 2 * B * n
    assert sorted(order) == sorted((k, b, b * n + r) for k in (0, 1) for b in range(B) for r in range(n))
    last_target = {}
    first_norm = {}
    for j, (norm, b, _) in enumerate(order):
        if norm:
            first_norm.setdefault(b, j)
        else:
            last_target[b] = j
    lag = min(8, B)
    for b in range(B):
        assert last_target[b] < first_norm[b]
        # target items of min(8, B) samples in all precede sample b's first normalisation
        targets_before = sum(1 for (k, _, _) in order[:first_norm[b]] if k == 0)
        assert targets_before >= min(B, b + lag) * n


@pytest.mark.parametrize("n,B", CASES)
@pytest.mark.parametrize("blocks", [1, 2, 5, 40])
def test_grid_taking_tickets_in_order_always_finishes(ticket_order, n, B, blocks):
    # Each resident block holds one ticket; a target item finishes in one step, a
    # normalisation item only once all of its sample's target items have finished.
    order = ticket_order(n, B)
    targets_done = [0] * B
    next_ticket = 0
    held = []
    steps = 0
    while next_ticket < len(order) or held:
        while len(held) < blocks and next_ticket < len(order):
            held.append(next_ticket)
            next_ticket += 1
        progressed = False
        for j in list(held):
            norm, b, _ = order[j]
            if not norm:
                targets_done[b] += 1
            elif targets_done[b] < n:
                continue  # waits for the sample's scale
            held.remove(j)
            progressed = True
        assert progressed, "every resident block waits: the grid would hang"
        steps += 1
    assert targets_done == [n] * B
