"""Random-interleaving model of a forward protocol with P in TMEM columns of its own.

Test infrastructure (not part of the library).  The kernel as built (csrc/attn_fwd.cu, modelled in
tests/fwd_protocol_model.py) writes P over its S buffer, so QK(j + 2) waits for P(j).V and every S
buffer runs softmax pass, P.V, QK and score wait in series.  This models the alternative, with the same
semantics (imported: parity-aliasing mbarriers, bounded waits that may give up, named barriers counted
in warps, an in-order tensor pipe, independent copies, buffer versions):
* P(j) goes to P buffer j % NPB (NPB = 2 with one P term, 1 with two terms), not over S(j);
* the softmax warps of the pass of tile j arrive on SC(j) once they have loaded S(j); the MMA warp
  issues QK(j + 2) into that S buffer after SC(j), before P(j).V: order QK0 QK1 | QK2 PV0 | QK3 PV1 ...
* every P(j).V commits PF(j % 2) (by tile parity, whatever NPB): the pass of tile j waits for
  P(j - NPB).V before storing P(j), and an O rescale at tile j waits for P(j - 1).V; S_FULL(j) implies
  P(j - 3).V complete, which keeps each of these parity waits at most one phase behind;
* five K/V stages: the producer keeps the kernel's rule (tile j - 2's scores before loading tile j,
  every phase waited in order and in time, so no wait aliases), and QK(j - 2) now follows P(j - 5).V
  in issue order, the last reader of the stage tile j takes (with four stages the rule would free a
  stage P(j - 4).V may still read);
* the own block's BF16 P goes to the other S buffer, which held S(t - 1), once the pass of tile t - 1
  has loaded it (the same warp, or with two sets the maximum hand-over of tile t - 1).

`mistake` plants an error the model must catch: "no_pfree_wait" (P stored before the P.V that read
the buffer last completed), "no_rescale_wait" (O rescaled while the previous P.V may still write it),
"sc_before_load" (the scores-loaded arrival before the load); `nst=4` is the stage-count mistake.
"""
from fwd_protocol_model import ModelError, _World


def _ids(prefix, j, n=3):
    return "%s%d" % (prefix, j % n)


def run(t, own, seed, sets=1, npb=2, nst=5, rescale_p=0.3, abort_p=0.0, mistake=None, max_idle=200000):
    w = _World(t, own, seed, rescale_p, abort_p, 3, mistake, sets)

    def producer():
        w.bar("Q_FULL").arrive(2)
        w.copy("Q_FULL", "Q", 0)
        w.copy("Q_FULL", "QSC", 0)
        loaded = [0] * nst
        for j in range(t + 1):
            st = j % nst
            if j >= 2:   # tile j - 2's scores: QK(j - 2) follows P(j - 5).V, the stage's last reader
                ok = yield from w.wait("S_FULL%d" % (j & 1), ((j - 2) >> 1) & 1)
                if not ok:
                    break
            w.bar("FULL%d" % st).arrive(4)
            for r in ("K", "KSC", "V", "VSC"):
                w.copy("FULL%d" % st, "%s%d" % (r, st), j)
            loaded[st] += 1
            yield
        for st in range(nst):
            if loaded[st]:
                while not w.bar("FULL%d" % st).passed((loaded[st] - 1) & 1):
                    yield
        while not w.bar("Q_FULL").passed(0):
            yield

    def forwarder():
        ok = yield from w.wait("Q_FULL", 0)
        if ok:
            w.read("QSC", 0, "forwarder")
            w.write("QATOM", 0, "forwarder")
        for j in range(t + 1):
            st = j % nst
            if ok:
                ok = yield from w.wait("FULL%d" % st, (j // nst) & 1)
            if ok:
                w.read("KSC%d" % st, j, "forwarder")
                w.read("VSC%d" % st, j, "forwarder")
                w.write("KATOM%d" % st, j, "forwarder")
                w.write("VATOM%d" % st, j, "forwarder")
            yield
            yield from w.nb_sync("KV", 2, j)

    def decoder():
        yield
        w.write("VT", 1, "decoder")
        w.bar("VT_READY").arrive()

    def mma():
        ok = [True]

        def live():
            return ok[0] and not w.aborted

        def qk(j):
            st, sb = j % nst, j & 1
            w.mma("scale copy K%d" % j, [("KATOM%d" % st, j)], [("TSFK%d" % sb, j)])
            w.mma("QK%d" % j, [("TQ", 0), ("TSFQ", 0), ("K%d" % st, j), ("TSFK%d" % sb, j)],
                  [("S%d_%d" % (sb, q), ("S", j)) for q in range(4)])
            w.commit("S_FULL%d" % sb)

        def pv(j):
            st, pb = j % nst, j % npb
            w.mma("scale copy V%d" % j, [("VATOM%d" % st, j)], [("TSFV%d" % (j & 1), j)])
            reads = [("V%d" % st, j), ("TSFV%d" % (j & 1), j)] + [("P%d_%d" % (pb, q), j) for q in range(4)] \
                + [("SFP%d_%d" % (pb, q), j) for q in range(4)] + ([("O%d" % q, j) for q in range(4)] if j > 0 else [])
            own_tile = own and j == t
            w.mma("PV%d" % j, reads, [("O%d" % q, j + (0.5 if own_tile else 1)) for q in range(4)])
            if own_tile:
                ok[0] = yield from w.wait("VT_READY", 0)
                if live():
                    ob = (t + 1) & 1
                    w.mma("own%d" % j, [("VT", 1)] + [("S%d_%d" % (ob, q), ("OWN", t)) for q in range(4)]
                          + [("O%d" % q, j + 0.5) for q in range(4)], [("O%d" % q, j + 1) for q in range(4)])
            w.commit("PF%d" % (j & 1))

        yield from w.nb_sync("KV", 2, 0)
        w.mma("Q copy", [("QATOM", 0), ("Q", 0)], [("TSFQ", 0), ("TQ", 0)])
        qk(0)
        if t >= 1:
            yield from w.nb_sync("KV", 2, 1)
            qk(1)
        for j in range(t + 1):
            if j + 2 <= t:
                yield from w.nb_sync(_ids("SC", j), 5, j)
                yield from w.nb_sync("KV", 2, j + 2)
                if live():
                    qk(j + 2)
            yield from w.nb_sync(_ids("P", j), 5, j)
            if live():
                yield from pv(j)
            if j == t and live():
                w.commit("O_FULL")
        w.commit("DRAIN")
        while not w.bar("DRAIN").passed(0):
            yield

    def softmax(x, q):
        ok = True
        seen = [-1]

        def take(j):
            yield from w.nb_sync("M%d" % (j & 1), 8, j)
            if ok:
                w.read("M%d" % q, j, "set%d softmax%d takes" % (x, q))
            seen[0] = j

        for j in range(x, t + 1, sets):
            sb, pb = j & 1, j % npb
            loaded = arrived = published = False
            while True:   # one pass; break = gave up
                if ok:
                    ok = yield from w.wait("S_FULL%d" % sb, (j >> 1) & 1)
                if not ok:
                    break
                w.read("S%d_%d" % (sb, q), ("S", j), "set%d softmax%d" % (x, q))
                if j + 2 <= t and mistake != "sc_before_load":
                    w.nb_arrive(_ids("SC", j), 5, j)
                loaded = True
                yield
                if sets == 2:
                    if j > 0:
                        yield from take(j - 1)
                    w.write("M%d" % q, j, "set%d softmax%d publishes" % (x, q))
                    w.nb_arrive("M%d" % (j & 1), 8, j)
                    published = True
                    seen[0] = j
                if j > 0 and w.rng.random() < w.rescale_p:
                    jj = j - 1   # O's last writer
                    if mistake != "no_rescale_wait":
                        ok = yield from w.wait("PF%d" % (jj & 1), (jj >> 1) & 1)
                    if not ok:
                        break
                    w.read("O%d" % q, j, "rescale%d%d" % (x, q))
                    w.write("O%d" % q, j, "rescale%d%d" % (x, q))
                if j >= npb and mistake != "no_pfree_wait":
                    jj = j - npb   # the last reader of this P buffer
                    ok = yield from w.wait("PF%d" % (jj & 1), (jj >> 1) & 1)
                    if not ok:
                        break
                w.write("P%d_%d" % (pb, q), j, "set%d softmax%d" % (x, q))
                w.write("SFP%d_%d" % (pb, q), j, "set%d softmax%d" % (x, q))
                if own and j == t:
                    w.write("S%d_%d" % ((t + 1) & 1, q), ("OWN", t), "set%d softmax%d" % (x, q))
                w.nb_arrive(_ids("P", j), 5, j)
                arrived = True
                break
            if not loaded and j + 2 <= t:   # gave up before loading: block on the generation
                yield from w.nb_sync(_ids("SC", j), 5, j)
            if sets == 2 and not published:
                if j > 0:
                    yield from take(j - 1)
                w.nb_arrive("M%d" % (j & 1), 8, j)
                seen[0] = j
            if not arrived:
                yield from w.nb_sync(_ids("P", j), 5, j)
            yield
        if sets == 2:
            if (t & 1) != x:
                yield from take(t)
            if x == 1:
                w.write("L%d" % q, 1, "set1 softmax%d" % q)
                w.nb_arrive("L", 8, 0)
                return
            yield from w.nb_sync("L", 8, 0)
            if ok:
                w.read("L%d" % q, 1, "set0 softmax%d" % q)
        if ok:
            ok = yield from w.wait("O_FULL", 0)
        if ok:
            w.read("O%d" % q, t + 1, "epilogue%d" % q)

    roles = {"producer": producer(), "forwarder": forwarder(), "mma": mma()}
    if own:
        roles["decoder"] = decoder()
    for q in range(4):
        for x in range(sets):
            roles["set%d softmax%d" % (x, q)] = softmax(x, q)
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


def count_failures(seeds, tiles=(0, 1, 2, 3, 4, 5, 8, 13), abort_ps=(0.0, 0.002, 0.02), sets=1, npb=2, nst=5, mistake=None):
    failures, first = 0, []
    for seed in range(seeds):
        for t in tiles:
            for own in (True, False):
                for ap in abort_ps:
                    try:
                        run(t, own, seed * 1000 + t, sets=sets, npb=npb, nst=nst, abort_p=ap, mistake=mistake)
                    except ModelError as e:
                        failures += 1
                        if len(first) < 3:
                            first.append("t=%d own=%d seed=%d abort_p=%g: %s" % (t, own, seed, ap, e))
    return failures, first
