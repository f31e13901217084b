"""Random-interleaving model of the backward kernel's two CTA roles (csrc/attn_bwd.cu).

Test infrastructure, on the same semantics as tests/fwd_protocol_model.py (mbarriers with parity
aliasing, bounded waits that may give up, named barriers counted in warps, an in-order tensor pipe,
independent copies, buffer versions):

* dK/dV (`dkdv_cta`, N query-tile pairs): a copy thread with two stages for Q-hat, dO and the row
  statistics, freed by the commit after each pair's dK; the MMA warp issuing S^T(0) dP^T(0) |
  dV(n) S^T(n+1) dK(n) dP^T(n+1) | ...; eight softmax warps (four lane quarters x two query halves)
  writing P^T over S^T and dS^T over dP^T.  Named barriers: LD (a pair landed; the softmax warps'
  first generation blocking, later ones arrivals), P (arrivals), DS (blocking).
* dQ (`dq_cta`, J key tiles): Q-hat and dO arrive in stage 2 and are copied into TMEM before stage 2
  takes key tile 2; key tiles go round three stages freed by the commit after each dQ(j); the MMA
  warp issues S(0) dP(0) | S(j+1) dQ(j) dP(j+1) | ...; eight softmax warps (four lane quarters x two
  key halves) read S and write dS over dP.  Named barriers: LD, S (S(j) has been read; arrivals),
  DS (blocking).

`mistake` plants a protocol error, so that the tests can show the model catches one: "no_pd_wait"
(dK/dV: a stage refilled before the MMAs of its pair completed), "first_ld_arrive" (dK/dV: the softmax
warps' first load generation met by an arrival), "no_cp_wait" (dQ: stage 2 refilled before Q-hat and
dO were copied out of it), "dp_before_dq" (dQ: dP(j+1) issued before the dQ(j) that reads dS(j)).
"""
import random

from fwd_protocol_model import ModelError, _World

WARPS = [(q, h) for q in range(4) for h in range(2)]   # softmax warps: lane quarter, half
NB = 9                                                # eight softmax warps + the MMA warp


def _dkdv(w, N):
    def stage(n):
        return n & 1

    def producer():
        def load_pair(n):
            st = stage(n)
            w.bar("LF%d" % st).arrive(3)
            for r in ("QH", "DO", "STAT"):
                w.copy("LF%d" % st, "%s%d" % (r, st), n)
        w.bar("KV").arrive(2)
        w.copy("KV", "KH", 0)
        w.copy("KV", "VH", 0)
        loaded = [0, 0]
        for n in range(min(N, 2)):
            load_pair(n)
            loaded[n] = 1
        for n in range(N - 2):
            ok = True if w.mistake == "no_pd_wait" else (yield from w.wait("PD%d" % (n & 1), (n >> 1) & 1))
            if not ok:
                break
            load_pair(n + 2)
            loaded[n & 1] += 1
        while not w.bar("KV").passed(0):
            yield
        for st in range(2):
            if loaded[st]:
                while not w.bar("LF%d" % st).passed((loaded[st] - 1) & 1):
                    yield

    def mma():
        ok = yield from w.wait("KV", 0)

        def live():
            return ok and not w.aborted

        def issue_s(n):
            w.mma("S%d" % n, [("KH", 0), ("QH%d" % stage(n), n)], [("ST%d%d" % x, ("S", n)) for x in WARPS])
            w.commit("SF")

        def issue_dp(n):
            w.mma("dP%d" % n, [("VH", 0), ("DO%d" % stage(n), n)], [("DPT%d%d" % x, ("DP", n)) for x in WARPS])
            w.commit("DP")

        yield from w.nb_sync("LD", NB, 0)
        if live():
            issue_s(0)
            issue_dp(0)
        for n in range(N):
            yield from w.nb_sync("P", NB, n)
            if live():
                w.mma("dV%d" % n, [("ST%d%d" % x, ("P", n)) for x in WARPS] + [("DO%d" % stage(n), n)]
                      + ([("TDV", n)] if n else []), [("TDV", n + 1)])
            if n + 1 < N:
                yield from w.nb_sync("LD", NB, n + 1)
                if live():
                    issue_s(n + 1)
            yield from w.nb_sync("DS", NB, n)
            if live():
                w.mma("dK%d" % n, [("DPT%d%d" % x, ("DS", n)) for x in WARPS] + [("QH%d" % stage(n), n)]
                      + ([("TDK", n)] if n else []), [("TDK", n + 1)])
                w.commit("PD%d" % (n & 1))
                if n + 1 < N:
                    issue_dp(n + 1)
        w.commit("DRAIN")

    def softmax(x):
        ok = True

        def landed(n):
            nonlocal ok
            if ok:
                ok = yield from w.wait("LF%d" % stage(n), (n >> 1) & 1)
            if n == 0 and w.mistake != "first_ld_arrive":
                yield from w.nb_sync("LD", NB, n)
            else:
                w.nb_arrive("LD", NB, n)

        yield from landed(0)
        for n in range(N):
            if ok:
                ok = yield from w.wait("SF", n & 1)
            if ok:
                w.read("ST%d%d" % x, ("S", n), "softmax P")
                w.read("STAT%d" % stage(n), n, "softmax P")
                yield
                w.write("ST%d%d" % x, ("P", n), "softmax P")
            w.nb_arrive("P", NB, n)
            if n + 1 < N:
                yield from landed(n + 1)
            if ok:
                ok = yield from w.wait("DP", n & 1)
            if ok:
                w.read("DPT%d%d" % x, ("DP", n), "softmax dS")
                w.read("STAT%d" % stage(n), n, "softmax dS")
                yield
                w.write("DPT%d%d" % x, ("DS", n), "softmax dS")
            yield from w.nb_sync("DS", NB, n)

    roles = {"producer": producer(), "mma": mma()}
    for x in WARPS:
        roles["softmax%d%d" % x] = softmax(x)

    def epilogue():
        w.read("TDV", N, "epilogue")
        w.read("TDK", N, "epilogue")
    return roles, epilogue


def _dq(w, J):
    KST = 3

    def producer():
        def load_kv(j):
            st = j % KST
            w.bar("KF%d" % st).arrive(1)
            w.copy("KF%d" % st, "KV%d" % st, j)
        w.bar("QD").arrive(2)
        w.copy("QD", "KV2", "QD")     # Q-hat and dO arrive in stage 2
        w.copy("QD", "STAT", 0)
        loaded = [0, 0, 0]
        ok = True
        for j in range(min(J, 2)):
            load_kv(j)
            loaded[j] = 1
        if J > 2:
            ok = True if w.mistake == "no_cp_wait" else (yield from w.wait("CP", 0))   # stage 2 is free
            if ok:
                load_kv(2)
                loaded[2] = 1
        j = 0
        while ok and j + KST < J:
            ok = yield from w.wait("KD%d" % (j % KST), (j // KST) & 1)
            if not ok:
                break
            load_kv(j + KST)
            loaded[j % KST] += 1
            j += 1
        while not w.bar("QD").passed(0):
            yield
        for st in range(KST):
            if loaded[st]:
                while not w.bar("KF%d" % st).passed((loaded[st] - 1) & 1):
                    yield

    def mma():
        ok = yield from w.wait("QD", 0)
        if ok:
            w.mma("Q, dO into TMEM", [("KV2", "QD")], [("TQH", 0), ("TDOH", 0)])
            w.commit("CP")

        def live():
            return ok and not w.aborted

        def issue_s(j):
            w.mma("S%d" % j, [("TQH", 0), ("KV%d" % (j % KST), j)], [("TS%d%d" % x, ("S", j)) for x in WARPS])
            w.commit("SF")

        def issue_dp(j):
            w.mma("dP%d" % j, [("TDOH", 0), ("KV%d" % (j % KST), j)], [("TDP%d%d" % x, ("DP", j)) for x in WARPS])
            w.commit("DP")

        yield from w.nb_sync("LD", NB, 0)
        if live():
            issue_s(0)
            issue_dp(0)
        for j in range(J):
            yield from w.nb_sync("S", NB, j)
            if j + 1 < J:
                yield from w.nb_sync("LD", NB, j + 1)
                if live():
                    issue_s(j + 1)
            if w.mistake == "dp_before_dq" and live() and j + 1 < J:
                issue_dp(j + 1)
            yield from w.nb_sync("DS", NB, j)
            if live():
                w.mma("dQ%d" % j, [("TDP%d%d" % x, ("DS", j)) for x in WARPS] + [("KV%d" % (j % KST), j)]
                      + ([("TDQ", j)] if j else []), [("TDQ", j + 1)])
                w.commit("KD%d" % (j % KST))
                if j + 1 < J and w.mistake != "dp_before_dq":
                    issue_dp(j + 1)
        w.commit("DRAIN")

    def softmax(x):
        ok = yield from w.wait("QD", 0)
        if ok:
            w.read("STAT", 0, "softmax")

        def landed(j):
            nonlocal ok
            if ok:
                ok = yield from w.wait("KF%d" % (j % KST), (j // KST) & 1)
            if j == 0:
                yield from w.nb_sync("LD", NB, j)
            else:
                w.nb_arrive("LD", NB, j)

        yield from landed(0)
        for j in range(J):
            if ok:
                ok = yield from w.wait("SF", j & 1)
            if ok:
                w.read("TS%d%d" % x, ("S", j), "softmax S")
                yield
            w.nb_arrive("S", NB, j)
            if j + 1 < J:
                yield from landed(j + 1)
            if ok:
                ok = yield from w.wait("DP", j & 1)
            if ok:
                w.read("TDP%d%d" % x, ("DP", j), "softmax dS")
                yield
                w.write("TDP%d%d" % x, ("DS", j), "softmax dS")
            yield from w.nb_sync("DS", NB, j)

    roles = {"producer": producer(), "mma": mma()}
    for x in WARPS:
        roles["softmax%d%d" % x] = softmax(x)

    def epilogue():
        w.read("TDQ", J, "epilogue")
    return roles, epilogue


def run(kind, n, seed, abort_p=0.0, mistake=None, max_idle=200000):
    """One interleaving of a dK/dV CTA with n pairs or a dQ CTA with n key tiles."""
    w = _World(t=0, own=False, seed=seed, rescale_p=0.0, abort_p=abort_p, n_pids=3, mistake=mistake)
    roles, epilogue = (_dkdv if kind == "dkdv" else _dq)(w, n)
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
    if not w.bar("DRAIN").passed(0):
        raise ModelError("the MMA warp's final commit never arrived")
    if not w.aborted:
        epilogue()


def count_failures(kind, seeds, sizes=(1, 2, 3, 4, 7), abort_ps=(0.0, 0.002, 0.02), mistake=None):
    failures, first = 0, []
    for seed in range(seeds):
        for n in sizes:
            for ap in abort_ps:
                try:
                    run(kind, n, seed * 1000 + n, abort_p=ap, mistake=mistake)
                except ModelError as e:
                    failures += 1
                    if len(first) < 3:
                        first.append("%s n=%d seed=%d abort_p=%g: %s" % (kind, n, seed, ap, e))
    return failures, first
