"""CPU model of the fused forward kernel's hand-off protocol (test helper).

The kernel's roles meet only through mbarriers: a TMA thread for Q, Qt and the
K/Kt ring, a TMA thread for the V/Vt ring, the S, St and value-MMA issuing
threads, and four softmax warps.  This model runs each role as a generator,
completes the asynchronous work (TMA copies in any order, each issuing
thread's MMAs in issue order) at random points, and checks what the GPU
cannot be asked to show without faulting it:

* every wait uses the hardware's parity test (it passes when the barrier's
  current phase parity differs from the awaited phase's), and a waiter is
  never more than one phase behind: a parity test cannot tell phase k from
  phase k + 2, and passing on phase k - 1 reads data that is not there yet;
* no deadlock;
* no buffer is overwritten while an MMA or the softmax still needs it, and
  each reader finds the tile it expects (shared-memory ring units, the S and
  St TMEM buffers, the P~/H~ written back into St);
* O and T are rescaled only when no value MMA is in flight, and every tile's
  value MMAs land exactly once.

``fwd_config`` restates the kernel's compile-time ring and buffer sizes for a
pair of (Q/K, V) head dims rounded up to 64, 128 or 256.
"""
import random

SMEM = 227 * 1024


def fwd_config(D, DVF):
    """Ring and buffer counts of the fused kernel for padded head dims (D, DVF)."""
    kDC = D // 64
    kDV = 128 if DVF > 128 else DVF
    kVC = kDV // 64
    NS = 1
    NSt = 5 if kDV == 64 else 3
    chunk_q, chunk_k = 128 * 128, 64 * 128
    q_bytes = kDC * chunk_q
    k_stage, v_stage = 2 * kDC * chunk_k, 2 * kVC * chunk_k
    room = SMEM - 1280 - 2 * q_bytes
    KS = 3 if room >= 3 * (k_stage + v_stage) else (2 if room >= 2 * (k_stage + v_stage) else 1)
    UPT = 2 if (KS == 1 and kDC % 2 == 0) else 1
    return dict(NS=NS, NSt=NSt, KS=KS, VS=KS, UPT=UPT, KU=KS * UPT)


class ProtocolError(AssertionError):
    pass


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.done, self.pending = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending > self.count:
            raise ProtocolError("%s: more arrivals than its count" % self.name)
        if self.pending == self.count:
            self.pending = 0
            self.done += 1


class FwdModel:
    """One CTA's roles over ``n_tiles`` key tiles.  ``mutate`` plants a protocol
    mistake (for the test that shows the model catches it)."""

    def __init__(self, cfg, n_tiles, seed, mutate=None):
        self.c = dict(cfg)
        self.n = n_tiles
        self.rng = random.Random(seed)
        self.mutate = mutate
        c = self.c
        B = lambda nm, cnt, k: [Bar("%s%d" % (nm, i), cnt) for i in range(k)]  # noqa: E731
        self.q_full = Bar("q_full", 1)
        self.k_full, self.k_empty = B("k_full", 1, c["KU"]), B("k_empty", 2, c["KU"])
        self.v_full, self.v_empty = B("v_full", 1, c["VS"]), B("v_empty", 1, c["VS"])
        self.s_full, self.s_free = B("s_full", 1, c["NS"]), B("s_free", 4, c["NS"])
        self.st_full = B("st_full", 1, c["NSt"])
        self.p_full, self.pv_done = B("p_full", 4, c["NSt"]), B("pv_done", 1, c["NSt"])
        self.k_unit = [None] * c["KU"]      # (tile, unit) held by each ring unit
        self.k_readers = [0] * c["KU"]
        self.v_stage = [None] * c["VS"]
        self.v_readers = [0] * c["VS"]
        self.s_buf = [None] * c["NS"]       # ("S", tile) once written
        self.s_writer = [0] * c["NS"]
        self.s_loaded = [None] * c["NS"]    # last tile the softmax loaded from each S buffer
        self.st_buf = [None] * c["NSt"]     # ("St", tile), then ("P", tile)
        self.st_writer = [0] * c["NSt"]
        self.st_readers = [0] * c["NSt"]
        self.pv_in_flight = 0
        self.pv_landed = []
        self.pending = []                   # (queue, completion) of asynchronous work

    # -- parity waits ---------------------------------------------------------
    def wait(self, bar, k):
        """Wait for phase k (k = -1: the phase before the first, already passed)."""
        while True:
            if bar.done >= k + 2:
                raise ProtocolError("%s: waiter for phase %d is two phases behind (%d done)"
                                    % (bar.name, k, bar.done))
            if (bar.done & 1) != (k & 1):
                if bar.done != k + 1:
                    raise ProtocolError("%s: parity test for phase %d passed with %d done"
                                        % (bar.name, k, bar.done))
                return
            yield

    def later(self, queue, fn):
        self.pending.append((queue, fn))

    # -- roles ----------------------------------------------------------------
    def tma_k(self):
        c = self.c
        self.later("tma", self.q_full.arrive)
        for n in range(self.n * c["UPT"]):
            t, u, s = n // c["UPT"], n % c["UPT"], n % c["KU"]
            yield from self.wait(self.k_empty[s], n // c["KU"] - 1)
            if self.k_readers[s]:
                raise ProtocolError("K unit %d reloaded while an MMA reads it" % s)

            def land(s=s, t=t, u=u):
                self.k_unit[s] = (t, u)
                self.k_full[s].arrive()
            self.later("tma", land)

    def tma_v(self):
        c = self.c
        for t in range(self.n):
            s = t % c["VS"]
            yield from self.wait(self.v_empty[s], t // c["VS"] - 1)
            if self.v_readers[s]:
                raise ProtocolError("V stage %d reloaded while an MMA reads it" % s)

            def land(s=s, t=t):
                self.v_stage[s] = t
                self.v_full[s].arrive()
            self.later("tma", land)

    def _score_issuer(self, name, NB, full, free_wait, buf, writer):
        c = self.c
        yield from self.wait(self.q_full, 0)
        for t in range(self.n):
            b = t % NB
            for u in range(c["UPT"]):
                n = t * c["UPT"] + u
                s = n % c["KU"]
                yield from self.wait(self.k_full[s], n // c["KU"])
                if u == 0 and t >= NB and self.mutate != name + "_no_free_wait":
                    yield from free_wait(t - NB)
                if self.k_unit[s] != (t, u):
                    raise ProtocolError("%s MMA of tile %d reads K unit holding %s" % (name, t, self.k_unit[s]))
                if u == 0 and (writer[b] or (name == "St" and self.st_readers[b])):
                    raise ProtocolError("%s buffer %d overwritten while in use" % (name, b))
                if u == 0 and t >= NB:
                    # the buffer's previous tile must be finished with: loaded by the
                    # softmax (S), or read as P~/H~ by its value MMAs (St)
                    prev = t - NB
                    if name == "S" and self.s_loaded[b] != prev:
                        raise ProtocolError("S buffer %d overwritten before tile %d was loaded" % (b, prev))
                    if name == "St" and prev not in self.pv_landed:
                        raise ProtocolError("St buffer %d overwritten before tile %d's value MMAs" % (b, prev))
                self.k_readers[s] += 1
                writer[b] += 1

                def done(s=s, b=b):
                    self.k_readers[s] -= 1
                    writer[b] -= 1
                    self.k_empty[s].arrive()
                self.later(name, done)

            def finished(b=b, t=t):
                buf[b] = (name, t)
                full[b].arrive()
            self.later(name, finished)

    def s_issuer(self):
        c = self.c

        def free(tp):
            yield from self.wait(self.s_free[tp % c["NS"]], tp // c["NS"])
        yield from self._score_issuer("S", c["NS"], self.s_full, free, self.s_buf, self.s_writer)

    def st_issuer(self):
        c = self.c

        def free(tp):
            yield from self.wait(self.pv_done[tp % c["NSt"]], tp // c["NSt"])
        yield from self._score_issuer("St", c["NSt"], self.st_full, free, self.st_buf, self.st_writer)

    def pv_issuer(self):
        c = self.c
        for j in range(self.n):
            b, s = j % c["NSt"], j % c["VS"]
            yield from self.wait(self.p_full[b], j // c["NSt"])
            yield from self.wait(self.v_full[s], j // c["VS"])
            if self.st_buf[b] != ("P", j) or self.v_stage[s] != j:
                raise ProtocolError("value MMAs of tile %d read %s and V of tile %s"
                                    % (j, self.st_buf[b], self.v_stage[s]))
            self.st_readers[b] += 1
            self.v_readers[s] += 1
            self.pv_in_flight += 1

            def done(b=b, s=s, j=j):
                self.st_readers[b] -= 1
                self.v_readers[s] -= 1
                self.pv_in_flight -= 1
                self.pv_landed.append(j)
                self.v_empty[s].arrive()
                self.pv_done[b].arrive()
            self.later("PV", done)

    def softmax_warp(self, w):
        c = self.c
        for j in range(self.n):
            b, bt = j % c["NS"], j % c["NSt"]
            yield from self.wait(self.s_full[b], j // c["NS"])
            yield from self.wait(self.st_full[bt], j // c["NSt"])
            if w == 0 and (self.s_buf[b] != ("S", j) or self.st_buf[bt] != ("St", j)):
                raise ProtocolError("softmax of tile %d loads %s and %s" % (j, self.s_buf[b], self.st_buf[bt]))
            if w == 0:
                self.s_loaded[b] = j
            yield
            self.s_free[b].arrive()
            yield
            if j >= 1 and self.rng.random() < 0.3:  # the row max grew: rescale O and T
                if self.mutate != "rescale_no_wait":
                    yield from self.wait(self.pv_done[(j - 1) % c["NSt"]], (j - 1) // c["NSt"])
                if self.pv_in_flight:
                    raise ProtocolError("O and T rescaled while value MMAs are in flight")
            if w == 0:
                self.st_buf[bt] = ("P", j)
            yield
            self.p_full[bt].arrive()
        yield from self.wait(self.pv_done[(self.n - 1) % c["NSt"]], (self.n - 1) // c["NSt"])
        if self.pv_in_flight or sorted(self.pv_landed) != list(range(self.n)):
            raise ProtocolError("epilogue before every value MMA landed")

    # -- scheduler ------------------------------------------------------------
    def run(self, max_steps=500000):
        roles = [self.tma_k(), self.tma_v(), self.s_issuer(), self.st_issuer(), self.pv_issuer()]
        roles += [self.softmax_warp(w) for w in range(4)]
        live = list(roles)
        for _ in range(max_steps):
            if not live and not self.pending:
                return
            if self.pending and (not live or self.rng.random() < 0.4):
                # any TMA copy may land; an issuing thread's MMAs complete in order
                heads, seen = [], set()
                for i, (q, _) in enumerate(self.pending):
                    if q == "tma" or q not in seen:
                        heads.append(i)
                        seen.add(q)
                _, fn = self.pending.pop(self.rng.choice(heads))
                fn()
                continue
            if live:
                r = self.rng.choice(live)
                try:
                    next(r)
                except StopIteration:
                    live.remove(r)
        raise ProtocolError("deadlock: no progress in %d steps" % max_steps)


# ---------------------------------------------------------------------------
# The backward kernel (both passes)
# ---------------------------------------------------------------------------
def bwd_config(D, dkdv):
    """Ring and buffer counts of the backward kernel for padded head dim D and a pass."""
    DV = min(D, 128)  # gradient columns per CTA (two CTAs share a row tile at 256)
    r_tmem = (not dkdv) and D <= 128
    free = 512 - (2 if dkdv else 1) * DV - (D if r_tmem else 0) - 64 * 3
    NS = 3 if free >= 192 else 1
    # up to 128 the value MMAs read their B operands from the score ring's stage
    shared = D <= 128
    KS = 1 if D == 256 else (4 if D == 128 else 6)
    VS = 1 if shared else (1 if dkdv else 2)
    UPT = 2 if (KS == 1 and (D // 64) % 2 == 0) else 1  # score-ring units per streamed tile
    return dict(NS=NS, NSt=3, SBar=2 if NS == 1 else NS, KS=KS, VS=VS, VecS=2 if D == 256 else 4, dkdv=dkdv,
                r_tmem=r_tmem, UPT=UPT, KU=KS * UPT, shared=shared)


class BwdModel(FwdModel):
    """One CTA of a backward pass: a TMA thread polling the score, value and (dK/dV
    pass) per-query vector rings; S1, S2 and value-MMA issuers; two groups of four
    elementwise warps taking even and odd tiles.  In the dQ pass group 0 first
    copies the resident tiles into TMEM for the score MMAs.  Up to head dim 128
    (``shared``) the value MMAs take their B operands from the score ring's stage of
    the same tile, which the value issuer releases as a third arrival on k_empty.
    ``mutate``: "one_s1_slot" gives the S1 barriers a single slot (two groups on one
    slot); "shared_stage_two_arrivals" leaves the value issuer's release out of the
    shared stage's count."""

    def __init__(self, cfg, n_tiles, seed, mutate=None):
        self.c = dict(cfg)
        c = self.c
        if mutate == "one_s1_slot":
            c["SBar"] = 1
        self.n = n_tiles
        self.rng = random.Random(seed)
        self.mutate = mutate
        B = lambda nm, cnt, k: [Bar("%s%d" % (nm, i), cnt) for i in range(k)]  # noqa: E731
        self.r_full, self.r_tmem = Bar("r_full", 1), Bar("r_tmem", 4)
        self.k_full = B("k_full", 1, c["KU"])
        self.k_empty = B("k_empty", 3 if c["shared"] and mutate != "shared_stage_two_arrivals" else 2, c["KU"])
        self.v_full, self.v_empty = B("v_full", 1, c["VS"]), B("v_empty", 1, c["VS"])
        self.vec_full, self.vec_empty = B("vec_full", 1, c["VecS"]), B("vec_empty", 4, c["VecS"])
        self.s_full, self.s_free = B("s_full", 1, c["SBar"]), B("s_free", 4, c["SBar"])
        self.st_full = B("st_full", 1, c["NSt"])
        self.p_full, self.pv_done = B("p_full", 4, c["NSt"]), B("pv_done", 1, c["NSt"])
        self.acc_done = Bar("acc_done", 1)
        self.k_stage, self.k_readers = [None] * c["KU"], [0] * c["KU"]  # (tile, unit) per ring unit
        self.v_stage, self.v_readers = [None] * c["VS"], [0] * c["VS"]
        self.vec_slot, self.vec_unread = [None] * c["VecS"], [0] * c["VecS"]
        self.s1_buf, self.s1_writer, self.s1_loaded = [None] * c["NS"], [0] * c["NS"], [None] * c["NS"]
        self.s2_buf, self.s2_writer, self.s2_readers = [None] * c["NSt"], [0] * c["NSt"], [0] * c["NSt"]
        self.r_in_tmem = False
        self.pv_in_flight = 0
        self.pv_landed = []
        self.pending = []

    def test(self, bar, k):
        """Non-blocking parity test (the producer's poll), held to the same rules as a wait."""
        if bar.done >= k + 2:
            raise ProtocolError("%s: poll for phase %d is two phases behind (%d done)" % (bar.name, k, bar.done))
        if (bar.done & 1) != (k & 1):
            if bar.done != k + 1:
                raise ProtocolError("%s: parity poll for phase %d passed with %d done" % (bar.name, k, bar.done))
            return True
        return False

    def producer(self):
        c = self.c
        self.later("tma", self.r_full.arrive)
        tk = tv = tq = 0
        nq = self.n if c["dkdv"] else 0
        nv = 0 if c["shared"] else self.n
        while tk < self.n * c["UPT"] or tv < nv or tq < nq:
            if tq < nq and self.test(self.vec_empty[tq % c["VecS"]], tq // c["VecS"] - 1):
                s = tq % c["VecS"]
                if self.vec_unread[s]:
                    raise ProtocolError("vector slot %d reloaded before a group read it" % s)

                def landq(s=s, t=tq):
                    self.vec_slot[s] = t
                    self.vec_unread[s] = 4
                    self.vec_full[s].arrive()
                self.later("tma", landq)
                tq += 1
            # tk counts score-ring units: unit tk % UPT of tile tk // UPT
            if tk < self.n * c["UPT"] and self.test(self.k_empty[tk % c["KU"]], tk // c["KU"] - 1):
                s = tk % c["KU"]
                if self.k_readers[s]:
                    raise ProtocolError("score unit %d reloaded while an MMA reads it" % s)

                def landk(s=s, n=tk):
                    self.k_stage[s] = divmod(n, c["UPT"])
                    self.k_full[s].arrive()
                self.later("tma", landk)
                tk += 1
            if tv < nv and self.test(self.v_empty[tv % c["VS"]], tv // c["VS"] - 1):
                s = tv % c["VS"]
                if self.v_readers[s]:
                    raise ProtocolError("value stage %d reloaded while an MMA reads it" % s)

                def landv(s=s, t=tv):
                    self.v_stage[s] = t
                    self.v_full[s].arrive()
                self.later("tma", landv)
                tv += 1
            yield

    def score_issuer(self, first):
        c = self.c
        name = "S1" if first else "S2"
        yield from self.wait(self.r_tmem if c["r_tmem"] else self.r_full, 0)
        if c["r_tmem"] and not self.r_in_tmem:
            raise ProtocolError("score MMAs before the resident tiles are in TMEM")
        for t in range(self.n):
            b = t % (c["NS"] if first else c["NSt"])
            writer = self.s1_writer if first else self.s2_writer
            for u in range(c["UPT"]):
                n = t * c["UPT"] + u
                s = n % c["KU"]
                yield from self.wait(self.k_full[s], n // c["KU"])
                if u == 0 and first and t >= c["NS"]:
                    tp = t - c["NS"]
                    yield from self.wait(self.s_free[tp % c["SBar"]], tp // c["SBar"])
                    if self.s1_loaded[b] != tp:
                        raise ProtocolError("S1 buffer %d overwritten before tile %d was loaded" % (b, tp))
                if u == 0 and not first and t >= c["NSt"]:
                    tp = t - c["NSt"]
                    yield from self.wait(self.pv_done[b], tp // c["NSt"])
                    if tp not in self.pv_landed:
                        raise ProtocolError("S2 buffer %d overwritten before tile %d's value MMAs" % (b, tp))
                if self.k_stage[s] != (t, u):
                    raise ProtocolError("%s MMA of tile %d unit %d reads a unit holding %s"
                                        % (name, t, u, self.k_stage[s]))
                if u == 0 and (writer[b] or (not first and self.s2_readers[b])):
                    raise ProtocolError("%s buffer %d overwritten while in use" % (name, b))
                self.k_readers[s] += 1
                writer[b] += 1

                def unit_done(s=s, b=b, writer=writer):
                    self.k_readers[s] -= 1
                    writer[b] -= 1
                    self.k_empty[s].arrive()
                self.later(name, unit_done)

            def done(b=b, t=t, first=first):
                (self.s1_buf if first else self.s2_buf)[b] = (name, t)
                (self.s_full[t % c["SBar"]] if first else self.st_full[b]).arrive()
            self.later(name, done)

    def value_issuer(self):
        c = self.c
        sh = c["shared"]
        for j in range(self.n):
            b, s = j % c["NSt"], j % (c["KU"] if sh else c["VS"])
            yield from self.wait(self.p_full[b], j // c["NSt"])
            if sh:
                yield from self.wait(self.k_full[s], j // c["KU"])
                stage, readers, empty = self.k_stage[s], self.k_readers, self.k_empty
                ok = stage == (j, 0)
            else:
                yield from self.wait(self.v_full[s], j // c["VS"])
                stage, readers, empty = self.v_stage[s], self.v_readers, self.v_empty
                ok = stage == j
            if self.s2_buf[b] != ("P", j) or not ok:
                raise ProtocolError("value MMAs of tile %d read %s and stage %s" % (j, self.s2_buf[b], stage))
            self.s2_readers[b] += 1
            readers[s] += 1
            self.pv_in_flight += 1

            def done(b=b, s=s, j=j, readers=readers, empty=empty):
                self.s2_readers[b] -= 1
                readers[s] -= 1
                self.pv_in_flight -= 1
                self.pv_landed.append(j)
                empty[s].arrive()
                self.pv_done[b].arrive()
            self.later("PV", done)
        self.later("PV", self.acc_done.arrive)

    def elementwise_warp(self, group, w):
        c = self.c
        if c["r_tmem"] and group == 0:
            yield from self.wait(self.r_full, 0)
            yield
            if w == 3:
                self.r_in_tmem = True  # the last of the four copies (modelled at the last arrival)
            self.r_tmem.arrive()
        for j in range(group, self.n, 2):
            b, bs, bt, sq = j % c["NS"], j % c["SBar"], j % c["NSt"], j % c["VecS"]
            yield from self.wait(self.s_full[bs], j // c["SBar"])
            if self.s1_buf[b] != ("S1", j):
                raise ProtocolError("tile %d loads S1 buffer holding %s" % (j, self.s1_buf[b]))
            if w == 0:
                self.s1_loaded[b] = j
            yield
            self.s_free[bs].arrive()
            yield from self.wait(self.st_full[bt], j // c["NSt"])
            if c["dkdv"]:
                yield from self.wait(self.vec_full[sq], j // c["VecS"])
                if self.vec_slot[sq] != j:
                    raise ProtocolError("tile %d reads vector slot holding %s" % (j, self.vec_slot[sq]))
                self.vec_unread[sq] -= 1
            if self.s2_buf[bt] not in (("S2", j), ("P", j)):
                raise ProtocolError("tile %d loads S2 buffer holding %s" % (j, self.s2_buf[bt]))
            yield
            if w == 0:
                self.s2_buf[bt] = ("P", j)
            yield
            self.p_full[bt].arrive()
            if c["dkdv"]:
                self.vec_empty[sq].arrive()
        yield from self.wait(self.acc_done, 0)
        if self.pv_in_flight or sorted(self.pv_landed) != list(range(self.n)):
            raise ProtocolError("epilogue before every value MMA landed")

    def run(self, max_steps=500000):
        roles = [self.producer(), self.score_issuer(True), self.score_issuer(False), self.value_issuer()]
        roles += [self.elementwise_warp(g, w) for g in range(2) for w in range(4)]
        live = list(roles)
        for _ in range(max_steps):
            if not live and not self.pending:
                return
            if self.pending and (not live or self.rng.random() < 0.4):
                heads, seen = [], set()
                for i, (q, _) in enumerate(self.pending):
                    if q == "tma" or q not in seen:
                        heads.append(i)
                        seen.add(q)
                _, fn = self.pending.pop(self.rng.choice(heads))
                fn()
                continue
            if live:
                r = self.rng.choice(live)
                try:
                    next(r)
                except StopIteration:
                    live.remove(r)
        raise ProtocolError("deadlock: no progress in %d steps" % max_steps)


# ---------------------------------------------------------------------------
# The forward kernel's abort path
# ---------------------------------------------------------------------------
class AbortFwdModel(FwdModel):
    """The forward protocol with a bounded wait giving up at a random point.

    As in the kernel: waits in the main loops see the CTA's abort flag and give up;
    each role then drains what it started (the TMA thread waits for the copies it
    issued into the last ring units and for Q; each MMA issuer commits to its drain
    barrier and waits on it) with waits that ignore the flag.  After every role has
    finished, nothing may still be in flight: no copy landing in, and no MMA
    reading, memory the CTA is about to release."""

    def __init__(self, cfg, n_tiles, seed, abort_at):
        super().__init__(cfg, n_tiles, seed)
        self.abort_at = abort_at
        self.aborted = False
        self.drain = {q: Bar("drain_" + q, 1) for q in ("S", "St", "PV")}
        self.step = 0
        self.ready = []  # earliest scheduler step of each pending entry

    def later(self, queue, fn):
        # a copy takes a while to land; MMAs and arrivals are quick
        self.pending.append((queue, fn))
        self.ready.append(self.step + (self.rng.randint(20, 200) if queue.startswith("tma") else 0))

    def wait_or_abort(self, bar, k):
        """Bounded wait: returns False once the abort flag is up."""
        while True:
            if self.aborted:
                return False
            if bar.done >= k + 2:
                raise ProtocolError("%s: waiter for phase %d is two phases behind" % (bar.name, k))
            if (bar.done & 1) != (k & 1):
                if bar.done != k + 1:
                    raise ProtocolError("%s: parity test for phase %d passed with %d done" % (bar.name, k, bar.done))
                return True
            yield

    def tma_k(self):
        c = self.c
        self.later("tmaK", self.q_full.arrive)
        issued, ok = 0, True
        for n in range(self.n * c["UPT"]):
            s = n % c["KU"]
            ok = yield from self.wait_or_abort(self.k_empty[s], n // c["KU"] - 1)
            if not ok:
                break
            self.later("tmaK", self.k_full[s].arrive)
            issued = n + 1
        # as in the kernel: the last copies are waited for whether or not this thread gave up
        yield from self.wait(self.q_full, 0)
        for n in range(max(0, issued - c["KU"]), issued):
            yield from self.wait(self.k_full[n % c["KU"]], n // c["KU"])

    def tma_v(self):
        c = self.c
        issued, ok = 0, True
        for t in range(self.n):
            s = t % c["VS"]
            ok = yield from self.wait_or_abort(self.v_empty[s], t // c["VS"] - 1)
            if not ok:
                break
            self.later("tmaV", self.v_full[s].arrive)
            issued = t + 1
        for t in range(max(0, issued - c["VS"]), issued):
            yield from self.wait(self.v_full[t % c["VS"]], t // c["VS"])

    def _issuer(self, name, NB, full, free_bar):
        c = self.c
        ok = yield from self.wait_or_abort(self.q_full, 0)
        t = 0
        while ok and t < self.n:
            for u in range(c["UPT"]):
                n = t * c["UPT"] + u
                s = n % c["KU"]
                ok = yield from self.wait_or_abort(self.k_full[s], n // c["KU"])
                if ok and u == 0 and t >= NB:
                    tp = t - NB
                    ok = yield from self.wait_or_abort(free_bar[tp % NB], tp // NB)
                if not ok:
                    break
                self.later(name, self.k_empty[s].arrive)
            if not ok:
                break
            self.later(name, full[t % NB].arrive)
            t += 1
        self.later(name, self.drain[name].arrive)
        yield from self.wait(self.drain[name], 0)

    def s_issuer(self):
        yield from self._issuer("S", self.c["NS"], self.s_full, self.s_free)

    def st_issuer(self):
        yield from self._issuer("St", self.c["NSt"], self.st_full, self.pv_done)

    def pv_issuer(self):
        c = self.c
        for j in range(self.n):
            b, s = j % c["NSt"], j % c["VS"]
            ok = yield from self.wait_or_abort(self.p_full[b], j // c["NSt"])
            ok = ok and (yield from self.wait_or_abort(self.v_full[s], j // c["VS"]))
            if not ok:
                break
            self.later("PV", self.v_empty[s].arrive)
            self.later("PV", self.pv_done[b].arrive)
        self.later("PV", self.drain["PV"].arrive)
        yield from self.wait(self.drain["PV"], 0)

    def softmax_warp(self, w):
        c = self.c
        ok = True
        for j in range(self.n):
            b, bt = j % c["NS"], j % c["NSt"]
            ok = yield from self.wait_or_abort(self.s_full[b], j // c["NS"])
            ok = ok and (yield from self.wait_or_abort(self.st_full[bt], j // c["NSt"]))
            if not ok:
                break
            self.s_free[b].arrive()
            if j >= 1 and self.rng.random() < 0.3:
                ok = yield from self.wait_or_abort(self.pv_done[(j - 1) % c["NSt"]], (j - 1) // c["NSt"])
                if not ok:
                    break
            self.p_full[bt].arrive()
        if ok:
            yield from self.wait_or_abort(self.pv_done[(self.n - 1) % c["NSt"]], (self.n - 1) // c["NSt"])

    def run(self, max_steps=500000):
        roles = [self.tma_k(), self.tma_v(), self.s_issuer(), self.st_issuer(), self.pv_issuer()]
        roles += [self.softmax_warp(w) for w in range(4)]
        return self.run_roles(roles, max_steps)

    def run_roles(self, roles, max_steps):
        live = list(roles)
        for step in range(max_steps):
            self.step = step
            if step == self.abort_at:
                self.aborted = True
            if not live:
                stray = [q for q, _ in self.pending]
                if stray:
                    raise ProtocolError("teardown with %d copies or MMAs still in flight" % len(stray))
                return
            if self.pending and self.rng.random() < 0.4:
                heads, seen = [], set()
                for i, (q, _) in enumerate(self.pending):
                    if q.startswith("tma") or q not in seen:
                        seen.add(q)
                        if self.ready[i] <= step:
                            heads.append(i)
                if heads:
                    i = self.rng.choice(heads)
                    self.ready.pop(i)
                    _, fn = self.pending.pop(i)
                    fn()
                    continue
            r = self.rng.choice(live)
            try:
                next(r)
            except StopIteration:
                live.remove(r)
        raise ProtocolError("a role never finished after the abort")


class AbortBwdModel(BwdModel):
    """The backward protocol with a bounded wait giving up (see AbortFwdModel).  The
    polling TMA thread always waits for the resident tiles and the last stage of each
    ring before it leaves; each MMA issuer drains its own MMAs."""

    def __init__(self, cfg, n_tiles, seed, abort_at):
        super().__init__(cfg, n_tiles, seed)
        self.abort_at = abort_at
        self.aborted = False
        self.drain = {q: Bar("drain_" + q, 1) for q in ("S1", "S2", "PV")}
        self.step = 0
        self.ready = []

    later = AbortFwdModel.later
    wait_or_abort = AbortFwdModel.wait_or_abort

    def producer(self):
        c = self.c
        self.later("tma", self.r_full.arrive)
        tk = tv = tq = 0
        nq = self.n if c["dkdv"] else 0
        nv = 0 if c["shared"] else self.n
        ok = True
        while tk < self.n * c["UPT"] or tv < nv or tq < nq:
            if self.aborted:
                ok = False
                break
            if tq < nq and self.test(self.vec_empty[tq % c["VecS"]], tq // c["VecS"] - 1):
                self.later("tma", self.vec_full[tq % c["VecS"]].arrive)
                tq += 1
            if tk < self.n * c["UPT"] and self.test(self.k_empty[tk % c["KU"]], tk // c["KU"] - 1):
                self.later("tma", self.k_full[tk % c["KU"]].arrive)
                tk += 1
            if tv < nv and self.test(self.v_empty[tv % c["VS"]], tv // c["VS"] - 1):
                self.later("tma", self.v_full[tv % c["VS"]].arrive)
                tv += 1
            yield
        # as in the kernel: the last copies are waited for whether or not this thread gave up
        yield from self.wait(self.r_full, 0)
        for bars, n, k in ((self.k_full, tk, c["KU"]), (self.v_full, tv, c["VS"]),
                           (self.vec_full, tq, c["VecS"])):
            for t in range(max(0, n - k), n):
                yield from self.wait(bars[t % k], t // k)

    def score_issuer(self, first):
        c = self.c
        name = "S1" if first else "S2"
        ok = yield from self.wait_or_abort(self.r_tmem if c["r_tmem"] else self.r_full, 0)
        for t in range(self.n):
            if not ok:
                break
            b = t % (c["NS"] if first else c["NSt"])
            for u in range(c["UPT"]):
                n = t * c["UPT"] + u
                s = n % c["KU"]
                ok = yield from self.wait_or_abort(self.k_full[s], n // c["KU"])
                if ok and u == 0 and first and t >= c["NS"]:
                    tp = t - c["NS"]
                    ok = yield from self.wait_or_abort(self.s_free[tp % c["SBar"]], tp // c["SBar"])
                if ok and u == 0 and not first and t >= c["NSt"]:
                    ok = yield from self.wait_or_abort(self.pv_done[b], (t - c["NSt"]) // c["NSt"])
                if not ok:
                    break
                self.later(name, self.k_empty[s].arrive)
            if not ok:
                break
            self.later(name, (self.s_full[t % c["SBar"]] if first else self.st_full[b]).arrive)
        self.later(name, self.drain[name].arrive)
        yield from self.wait(self.drain[name], 0)

    def value_issuer(self):
        c = self.c
        ok = True
        sh = c["shared"]
        for j in range(self.n):
            b, s = j % c["NSt"], j % (c["KU"] if sh else c["VS"])
            ok = yield from self.wait_or_abort(self.p_full[b], j // c["NSt"])
            if sh:
                ok = ok and (yield from self.wait_or_abort(self.k_full[s], j // c["KU"]))
            else:
                ok = ok and (yield from self.wait_or_abort(self.v_full[s], j // c["VS"]))
            if not ok:
                break
            self.later("PV", (self.k_empty if sh else self.v_empty)[s].arrive)
            self.later("PV", self.pv_done[b].arrive)
        if ok:
            self.later("PV", self.acc_done.arrive)
        self.later("PV", self.drain["PV"].arrive)
        yield from self.wait(self.drain["PV"], 0)

    def elementwise_warp(self, group, w):
        c = self.c
        ok = True
        if c["r_tmem"] and group == 0:
            ok = yield from self.wait_or_abort(self.r_full, 0)
            if ok:
                self.r_tmem.arrive()
        for j in range(group, self.n, 2):
            if not ok:
                break
            bs, bt, sq = j % c["SBar"], j % c["NSt"], j % c["VecS"]
            ok = yield from self.wait_or_abort(self.s_full[bs], j // c["SBar"])
            if not ok:
                break
            self.s_free[bs].arrive()
            ok = yield from self.wait_or_abort(self.st_full[bt], j // c["NSt"])
            if ok and c["dkdv"]:
                ok = yield from self.wait_or_abort(self.vec_full[sq], j // c["VecS"])
            if not ok:
                break
            self.p_full[bt].arrive()
            if c["dkdv"]:
                self.vec_empty[sq].arrive()
        if ok:
            yield from self.wait_or_abort(self.acc_done, 0)

    def run(self, max_steps=500000):
        roles = [self.producer(), self.score_issuer(True), self.score_issuer(False), self.value_issuer()]
        roles += [self.elementwise_warp(g, w) for g in range(2) for w in range(4)]
        self._roles = roles
        return AbortFwdModel.run_roles(self, roles, max_steps)


# ---------------------------------------------------------------------------
# attn_jvp_fwd_host: items rotating through three workspace slots on streams
# ---------------------------------------------------------------------------
class HostPipelineModel:
    """The host path's stream and event order.

    Streams run their operations in order; ``cudaStreamWaitEvent`` waits for the
    most recent record of the event enqueued before the wait (none: no wait);
    copies and kernels take time and may overlap with work on other streams.
    The enqueue order below follows the host loop of ``attn_jvp_fwd_host``: per
    item i in slot s = i mod 3, copy-in on the H2D stream after the slot's
    previous compute, compute on the slot's stream after its copy-in and the
    slot's previous copy-out, copy-out on the D2H stream after the compute; the
    caller's stream finally waits for the last copy-out of every slot.  Checked:
    no copy or kernel touches a slot's buffers while a conflicting one is in
    progress, every kernel reads its own item's inputs and every copy-out its
    own item's outputs, and nothing is left when the caller's stream is done.
    ``mutate``: "no_copied_wait" drops the compute's wait for the slot's previous
    copy-out, "no_computed_wait" drops the copy-in's wait for the previous
    compute."""

    SLOTS = 3

    def __init__(self, n_items, seed, mutate=None):
        self.n = n_items
        self.rng = random.Random(seed)
        self.mutate = mutate
        self.streams = {name: [] for name in ("caller", "h2d", "d2h", "c0", "c1", "c2")}
        self.enqueued = {}   # event -> versions recorded (enqueued) so far
        self.completed = {}  # event -> versions completed
        self.inputs = [None] * self.SLOTS    # item whose inputs the slot holds
        self.outputs = [None] * self.SLOTS   # item whose outputs the slot holds
        self.busy_in = [[] for _ in range(self.SLOTS)]   # ops touching the slot's inputs now
        self.busy_out = [[] for _ in range(self.SLOTS)]
        self.delivered = set()

    def record(self, stream, ev):
        v = self.enqueued.get(ev, 0) + 1
        self.enqueued[ev] = v
        self.streams[stream].append(("record", ev, v))

    def wait_event(self, stream, ev):
        v = self.enqueued.get(ev, 0)
        if v:
            self.streams[stream].append(("wait", ev, v))

    def enqueue(self):
        S = self.SLOTS
        self.record("caller", "entry")
        for i in range(self.n):
            s = i % S
            reuse = i >= S
            if not (reuse and self.mutate == "no_computed_wait"):
                self.wait_event("h2d", ("computed", s) if reuse else "entry")
            self.streams["h2d"].append(("copy_in", s, i))
            self.record("h2d", ("in_ready", s))
            cs = "c%d" % s
            self.wait_event(cs, ("in_ready", s))
            if reuse and self.mutate != "no_copied_wait":
                self.wait_event(cs, ("copied", s))
            self.streams[cs].append(("compute", s, i))
            self.record(cs, ("computed", s))
            self.wait_event("d2h", ("computed", s))
            self.streams["d2h"].append(("copy_out", s, i))
            self.record("d2h", ("copied", s))
        for s in range(min(S, self.n)):
            self.wait_event("caller", ("copied", s))
        self.streams["caller"].append(("done",))

    def _start(self, op):
        kind, s, i = op
        if kind == "copy_in":
            if self.busy_in[s]:
                raise ProtocolError("copy-in of item %d over inputs in use by %s" % (i, self.busy_in[s]))
            self.busy_in[s].append(op)
        elif kind == "compute":
            if self.inputs[s] != i or any(o[0] == "copy_in" for o in self.busy_in[s]):
                raise ProtocolError("compute of item %d reads inputs of item %s" % (i, self.inputs[s]))
            if self.busy_out[s]:
                raise ProtocolError("compute of item %d writes outputs in use by %s" % (i, self.busy_out[s]))
            self.busy_in[s].append(op)
            self.busy_out[s].append(op)
        else:
            if self.outputs[s] != i or any(o[0] == "compute" for o in self.busy_out[s]):
                raise ProtocolError("copy-out of item %d reads outputs of item %s" % (i, self.outputs[s]))
            self.busy_out[s].append(op)

    def _finish(self, op):
        kind, s, i = op
        if kind == "copy_in":
            self.busy_in[s].remove(op)
            self.inputs[s] = i
        elif kind == "compute":
            self.busy_in[s].remove(op)
            self.busy_out[s].remove(op)
            self.outputs[s] = i
        else:
            self.busy_out[s].remove(op)
            self.delivered.add(i)

    def run(self, max_steps=200000):
        self.enqueue()
        running = {}  # stream -> data op in progress
        for _ in range(max_steps):
            ready = []
            for name, q in self.streams.items():
                if name in running:
                    ready.append(name)
                elif q:
                    head = q[0]
                    if head[0] == "wait" and self.completed.get(head[1], 0) < head[2]:
                        continue
                    ready.append(name)
            if not ready:
                if any(self.streams.values()) or running:
                    raise ProtocolError("streams deadlocked")
                break
            name = self.rng.choice(ready)
            if name in running:
                self._finish(running.pop(name))
                continue
            head = self.streams[name].pop(0)
            if head[0] == "record":
                self.completed[head[1]] = max(self.completed.get(head[1], 0), head[2])
            elif head[0] == "done":
                if self.delivered != set(range(self.n)):
                    raise ProtocolError("caller's stream done before every output reached the host")
                return
            elif head[0] in ("copy_in", "compute", "copy_out"):
                self._start(head)
                running[name] = head
        raise ProtocolError("no end in %d steps" % max_steps)
