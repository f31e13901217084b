"""Random-interleaving model of the attention forward kernel's synchronisation protocol.

Test infrastructure (not part of the library): a hand-written abstraction of the roles of
`attn_fwd_kernel` (csrc/attn_fwd.cu) for one CTA with `t + 1` key tiles -- the TMA producer, the
MMA-issuing warp, the own-block V decoder, the scale forwarder and the four softmax warps -- and of
the hardware objects they synchronise through.  A scheduler runs one step of a randomly chosen role,
the tensor pipe or an outstanding copy at a time, so that many interleavings of the same program are
explored.  It checks:

* every role finishes (no deadlock), the mbarrier waits being bounded: a wait may give up (an abort,
  raised at random), after which every later wait gives up too, as in the kernel;
* no named-barrier generation ever holds arrivals of two different tiles;
* without an abort, every read of a buffer sees the version the protocol promises and no buffer is
  written while an asynchronous reader (an MMA or a copy in flight) still uses it.

Semantics modelled:
* mbarrier: a phase counter; `wait(parity P)` passes when the completed-phase count has the other
  parity (so a wait can alias a phase two ahead, as the hardware's can);
* named barrier: a count of warps; `arrive` does not wait, `sync` waits for its generation;
* tensor pipe: MMAs and commits execute in issue order and complete at random later times; a commit
  arrives on its mbarrier when every earlier operation has completed;
* TMA: each copy completes independently; the stage's barrier completes when all its bytes landed.

`n_pids` is the number of named-barrier IDs the P hand-over (softmax -> MMA warp) rotates through:
3 as built; 2 (tile parity) is the earlier form, which the model shows can mix generations and
deadlock once a wait gives up mid-run.  `sets` is the number of softmax sets: 1 (four warps take every
key tile; the kernel with one P term) or 2 (two sets of four take alternate tiles and hand each other
the running row maximum at the NB_M barriers, set 1 its row sum at NB_L; the kernel with two P terms).
`mistake` plants a protocol error, so that the tests can show the model catches one: "no_stage_wait"
(the producer refills a K/V stage without waiting for the scores that prove its last reader
completed), "publish_before_take" (two sets: a set publishes its tile's maximum before taking the
previous tile's), "no_final_take" (two sets: the set that does not own the last tile hands over its
row sum without the final maximum).
"""
import random

NST = 4   # K/V stages


class ModelError(Exception):
    pass


class _MBar:
    def __init__(self, name):
        self.name, self.c, self.pending, self.tx = name, 0, 1, 0

    def arrive(self, tx=0):
        if self.pending == 0:
            raise ModelError("over-arrival on " + self.name)
        self.pending -= 1
        self.tx += tx
        self._check()

    def tx_done(self):
        self.tx -= 1
        if self.tx < 0:
            raise ModelError("byte-count underflow on " + self.name)
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.c += 1
            self.pending = 1

    def passed(self, parity):
        return (self.c & 1) != parity


class _World:
    def __init__(self, t, own, seed, rescale_p, abort_p, n_pids, mistake=None, sets=1):
        self.mistake, self.sets = mistake, sets
        self.rng = random.Random(seed)
        self.t, self.own, self.rescale_p, self.abort_p, self.n_pids = t, own, rescale_p, abort_p, n_pids
        self.aborted = False
        self.res, self.inflight, self.bars, self.nb = {}, {}, {}, {}
        self.pipe, self.copies = [], []

    def bar(self, name):
        if name not in self.bars:
            self.bars[name] = _MBar(name)
        return self.bars[name]

    # buffers with versions
    def write(self, r, v, who):
        if not self.aborted and self.inflight.get(r, 0):
            raise ModelError("%s writes %s while %d asynchronous readers use it" % (who, r, self.inflight[r]))
        self.res[r] = v

    def read(self, r, v, who):
        if not self.aborted and self.res.get(r) != v:
            raise ModelError("%s reads %s: holds %s, expected %s" % (who, r, self.res.get(r), v))

    # tensor pipe
    def mma(self, who, reads, writes):
        for r, v in reads:
            pending = [vv for op in self.pipe if op[0] == "op" for rr, vv in op[3] if rr == r]
            if self.aborted:
                pass
            elif pending:
                if pending[-1] != v:
                    raise ModelError("%s at issue reads %s: pending %s, expected %s" % (who, r, pending[-1], v))
            else:
                self.read(r, v, who + " at issue")
        for r, _ in reads:
            self.inflight[r] = self.inflight.get(r, 0) + 1
        self.pipe.append(("op", who, reads, writes))

    def commit(self, bar_name):
        self.pipe.append(("commit", bar_name))

    def pipe_step(self):
        op = self.pipe.pop(0)
        if op[0] == "commit":
            self.bar(op[1]).arrive()
            return
        _, who, reads, writes = op
        for r, v in reads:
            self.inflight[r] -= 1
            self.read(r, v, who + " at completion")
        for r, v in writes:
            self.res[r] = v

    # copies
    def copy(self, bar_name, r, v):
        self.write(r, ("in flight",), "copy")
        self.copies.append((bar_name, r, v))

    def copy_step(self, i):
        bar_name, r, v = self.copies.pop(i)
        self.res[r] = v
        self.bar(bar_name).tx_done()

    # named barriers
    def nb_arrive(self, name, count, tile):
        st = self.nb.setdefault(name, {"arr": [], "gen": 0})
        st["arr"].append(tile)
        gen = st["gen"]
        if len(st["arr"]) == count:
            if len(set(st["arr"])) != 1:
                raise ModelError("named barrier %s: one generation holds tiles %s" % (name, st["arr"]))
            st["arr"] = []
            st["gen"] += 1
        return gen

    def nb_sync(self, name, count, tile):
        gen = self.nb_arrive(name, count, tile)
        while self.nb[name]["gen"] <= gen:
            yield

    def pid(self, j):
        return "P%d" % (j % self.n_pids)

    def wait(self, bar_name, parity):
        """A bounded mbarrier wait (generator): True when the phase passed, False when it gave up."""
        while True:
            if self.bar(bar_name).passed(parity):
                return True
            if self.aborted:
                return False
            if self.abort_p and self.rng.random() < self.abort_p:
                self.aborted = True
                return False
            yield


def _producer(w):
    t = w.t
    w.bar("Q_FULL").arrive(2)
    w.copy("Q_FULL", "Q", 0)
    w.copy("Q_FULL", "QSC", 0)
    loaded = [0] * NST
    for j in range(t + 1):
        st = j % NST
        if j >= 2 and w.mistake != "no_stage_wait":   # tile j - 2's scores: the stage's last reader is done
            ok = yield from w.wait("S_FULL%d" % (j & 1), ((j - 2) >> 1) & 1)
            if not ok:
                break
        w.bar("FULL%d" % st).arrive(4)
        for r in ("K", "KSC", "V", "VSC"):
            w.copy("FULL%d" % st, "%s%d" % (r, st), j)
        loaded[st] += 1
        yield
    for st in range(NST):   # drain: own copies always land
        if loaded[st]:
            while not w.bar("FULL%d" % st).passed((loaded[st] - 1) & 1):
                yield
    while not w.bar("Q_FULL").passed(0):
        yield


def _forwarder(w):
    t = w.t
    ok = yield from w.wait("Q_FULL", 0)
    if ok:
        w.read("QSC", 0, "forwarder")
        w.write("QATOM", 0, "forwarder")
    for j in range(t + 1):
        st = j % NST
        if ok:
            ok = yield from w.wait("FULL%d" % st, (j // NST) & 1)
        if ok:
            w.read("KSC%d" % st, j, "forwarder")
            w.read("VSC%d" % st, j, "forwarder")
            w.write("KATOM%d" % st, j, "forwarder")
            w.write("VATOM%d" % st, j, "forwarder")
        yield
        yield from w.nb_sync("KV", 2, j)


def _decoder(w):
    yield
    w.write("VT", 1, "decoder")
    w.bar("VT_READY").arrive()


def _mma(w):
    t = w.t
    ok = [True]

    def qk(j):
        st, sb = j % NST, j & 1
        w.mma("scale copy K%d" % j, [("KATOM%d" % st, j)], [("TSFK%d" % sb, j)])
        w.mma("QK%d" % j, [("TQ", 0), ("TSFQ", 0), ("K%d" % st, j), ("TSFK%d" % sb, j)],
              [("S%d_%d" % (sb, q), ("S", j)) for q in range(4)])
        w.commit("S_FULL%d" % sb)

    def pv(j, own_tile):
        st, sb = j % NST, j & 1
        w.mma("scale copy V%d" % j, [("VATOM%d" % st, j)], [("TSFV%d" % sb, j)])
        reads = [("V%d" % st, j), ("TSFV%d" % sb, j)] + [("S%d_%d" % (sb, q), ("P", j)) for q in range(4)] \
            + [("SFP%d_%d" % (sb, q), ("P", j)) for q in range(4)] + ([("O%d" % q, j) for q in range(4)] if j > 0 else [])
        if not own_tile:
            w.mma("PV%d" % j, reads, [("O%d" % q, j + 1) for q in range(4)])
        else:
            w.mma("PV%d" % j, reads, [("O%d" % q, j + 0.5) for q in range(4)])
            ok[0] = yield from w.wait("VT_READY", 0)
            if ok[0]:
                ob = (t + 1) & 1
                w.mma("own%d" % j, [("VT", 1)] + [("S%d_%d" % (ob, q), ("OWN", t)) for q in range(4)]
                      + [("O%d" % q, j + 0.5) for q in range(4)], [("O%d" % q, j + 1) for q in range(4)])
        if j == t - 1:
            w.commit("P_DONE")

    yield from w.nb_sync("KV", 2, 0)
    w.mma("Q copy", [("QATOM", 0), ("Q", 0)], [("TSFQ", 0), ("TQ", 0)])
    qk(0)
    if t >= 1:
        yield from w.nb_sync("KV", 2, 1)
        qk(1)
    for j in range(t + 1):
        yield from w.nb_sync(w.pid(j), 5, j)
        if ok[0]:
            yield from pv(j, w.own and j == t)
        if j == t and ok[0]:
            w.commit("O_FULL")
        if j + 2 <= t:
            yield from w.nb_sync("KV", 2, j + 2)
            if ok[0]:
                qk(j + 2)
    w.commit("DRAIN")
    while not w.bar("DRAIN").passed(0):
        yield


def _softmax(w, q):
    t = w.t
    ok = True
    for j in range(t + 1):
        sb = j & 1
        arrived = False
        while True:   # one pass; break = gave up
            if ok:
                ok = yield from w.wait("S_FULL%d" % sb, (j >> 1) & 1)
            if not ok:
                break
            w.read("S%d_%d" % (sb, q), ("S", j), "softmax%d" % q)
            yield
            if j > 0 and w.rng.random() < w.rescale_p:   # O rescaled once the previous P.V completed
                if j < t:
                    ok = yield from w.wait("S_FULL%d" % ((j + 1) & 1), ((j + 1) >> 1) & 1)
                else:
                    ok = yield from w.wait("P_DONE", 0)
                if not ok:
                    break
                w.read("O%d" % q, j, "rescale%d" % q)
                w.write("O%d" % q, j, "rescale%d" % q)
            w.write("S%d_%d" % (sb, q), ("P", j), "softmax%d" % q)
            if w.own and j == t and t > 0:
                ok = yield from w.wait("P_DONE", 0)
                if not ok:
                    break
            if w.own and j == t:
                w.write("S%d_%d" % ((t + 1) & 1, q), ("OWN", t), "softmax%d" % q)
            w.write("SFP%d_%d" % (sb, q), ("P", j), "softmax%d" % q)
            w.nb_arrive(w.pid(j), 5, j)
            arrived = True
            break
        if not arrived:   # a warp that gave up blocks on the generation instead of arriving
            yield from w.nb_sync(w.pid(j), 5, j)
        yield
    if ok:
        ok = yield from w.wait("O_FULL", 0)
    if ok:
        w.read("O%d" % q, t + 1, "epilogue%d" % q)


def _softmax_set(w, x, q):
    """One softmax warp of set x (two sets): tiles j with j % 2 == x, rows of lane quarter q."""
    t = w.t
    ok = True
    seen = [-1]   # the latest tile whose maximum this warp knows

    def take(j):   # the maximum decided at tile j by the other set
        yield from w.nb_sync("M%d" % (j & 1), 8, j)
        if ok:
            w.read("M%d" % q, j, "set%d softmax%d takes" % (x, q))
        seen[0] = j

    for j in range(x, t + 1, 2):
        sb = j & 1
        arrived = published = False
        while True:   # one pass; break = gave up
            if ok:
                ok = yield from w.wait("S_FULL%d" % sb, (j >> 1) & 1)
            if not ok:
                break
            w.read("S%d_%d" % (sb, q), ("S", j), "set%d softmax%d" % (x, q))
            yield
            if w.mistake == "publish_before_take":
                w.write("M%d" % q, j, "set%d softmax%d publishes" % (x, q))
                w.nb_arrive("M%d" % (j & 1), 8, j)
                published = True
                seen[0] = j
            if j > 0:
                yield from take(j - 1)
            if not published:
                w.write("M%d" % q, j, "set%d softmax%d publishes" % (x, q))
                w.nb_arrive("M%d" % (j & 1), 8, j)
                published = True
                seen[0] = j
            if j > 0 and w.rng.random() < w.rescale_p:
                if j < t:
                    ok = yield from w.wait("S_FULL%d" % ((j + 1) & 1), ((j + 1) >> 1) & 1)
                else:
                    ok = yield from w.wait("P_DONE", 0)
                if not ok:
                    break
                w.read("O%d" % q, j, "rescale%d%d" % (x, q))
                w.write("O%d" % q, j, "rescale%d%d" % (x, q))
            w.write("S%d_%d" % (sb, q), ("P", j), "set%d softmax%d" % (x, q))
            if w.own and j == t and t > 0:
                ok = yield from w.wait("P_DONE", 0)
                if not ok:
                    break
            if w.own and j == t:
                w.write("S%d_%d" % ((t + 1) & 1, q), ("OWN", t), "set%d softmax%d" % (x, q))
            w.write("SFP%d_%d" % (sb, q), ("P", j), "set%d softmax%d" % (x, q))
            w.nb_arrive(w.pid(j), 5, j)
            arrived = True
            break
        if not published:   # gave up first: meet the maximum generations in the same order
            if j > 0:
                yield from take(j - 1)
            w.nb_arrive("M%d" % (j & 1), 8, j)
            seen[0] = j
        if not arrived:
            yield from w.nb_sync(w.pid(j), 5, j)
        yield
    if (t & 1) != x and w.mistake != "no_final_take":
        yield from take(t)
    if not w.aborted and seen[0] != t:
        raise ModelError("set%d softmax%d hands over its row sum without the final maximum" % (x, q))
    if x == 1:
        w.write("L%d" % q, 1, "set1 softmax%d" % q)
        w.nb_arrive("L", 8, 0)
    else:
        yield from w.nb_sync("L", 8, 0)
        if ok:
            w.read("L%d" % q, 1, "set0 softmax%d" % q)
        if ok:
            ok = yield from w.wait("O_FULL", 0)
        if ok:
            w.read("O%d" % q, t + 1, "epilogue%d" % q)


def run(t, own, seed, rescale_p=0.3, abort_p=0.0, n_pids=3, mistake=None, sets=1, max_idle=200000):
    """One interleaving; raises ModelError on a violation or a deadlock."""
    w = _World(t, own, seed, rescale_p, abort_p, n_pids, mistake, sets)
    roles = {"producer": _producer(w), "forwarder": _forwarder(w), "mma": _mma(w)}
    if own:
        roles["decoder"] = _decoder(w)
    for q in range(4):
        if sets == 1:
            roles["softmax%d" % q] = _softmax(w, q)
        else:
            for x in range(2):
                roles["set%d softmax%d" % (x, q)] = _softmax_set(w, x, q)
    idle = 0
    while roles or w.pipe or w.copies:
        choices = list(roles) + (["pipe"] if w.pipe else []) + ["copy%d" % i for i in range(len(w.copies))]
        c = w.rng.choice(choices)
        if c == "pipe":
            w.pipe_step()
            idle = 0
            continue
        if c.startswith("copy"):
            w.copy_step(int(c[4:]))
            idle = 0
            continue
        try:
            next(roles[c])
        except StopIteration:
            del roles[c]
        idle += 1
        if idle > max_idle:
            raise ModelError("deadlock: %s still running" % ", ".join(sorted(roles)))


def count_failures(seeds, tiles=(0, 1, 2, 3, 5, 8), abort_ps=(0.0, 0.002, 0.02), n_pids=3, mistake=None, sets=1):
    """Failures over seeds x tile counts x {own block, leaky} x abort rates; the first messages."""
    failures, first = 0, []
    for seed in range(seeds):
        for t in tiles:
            for own in (True, False):
                for ap in abort_ps:
                    try:
                        run(t, own, seed * 1000 + t, abort_p=ap, n_pids=n_pids, mistake=mistake, sets=sets)
                    except ModelError as e:
                        failures += 1
                        if len(first) < 3:
                            first.append("t=%d own=%d seed=%d abort_p=%g: %s" % (t, own, seed, ap, e))
    return failures, first
