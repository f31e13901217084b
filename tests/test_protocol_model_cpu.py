"""The attention forward kernel's synchronisation protocol, checked on a random-interleaving model
(tests/fwd_protocol_model.py) on the CPU: no deadlock, no named-barrier generation holding two tiles,
no stale or overwritten buffer, also when bounded waits give up mid-run.  The model also has to
catch the earlier two-ID form of the P hand-over and a planted ordering mistake, so that a model that
checks nothing cannot pass."""
import pytest

import fwd_protocol_model as M


def test_protocol_as_built_is_clean():
    failures, first = M.count_failures(seeds=12, n_pids=3)
    assert failures == 0, first


def test_protocol_without_aborts_is_clean_on_long_runs():
    for seed in range(6):
        for own in (True, False):
            M.run(t=21, own=own, seed=seed, rescale_p=0.5)


def test_two_p_ids_mix_generations_after_a_mid_run_abort():
    # the form the kernel had before: tile parity picks the ID; a warp that gives up at tile j can
    # join tile j - 2's generation while a slower warp has not arrived there
    failures, first = M.count_failures(seeds=40, tiles=(5, 8, 13), abort_ps=(0.002, 0.02), n_pids=2)
    assert failures > 0


def test_model_catches_a_missing_wait(monkeypatch):
    # planted mistake: the producer reuses a K/V stage without waiting for the scores that prove its
    # last reader completed
    original = M._producer

    def producer_without_wait(w):
        t = w.t
        w.bar("Q_FULL").arrive(2)
        w.copy("Q_FULL", "Q", 0)
        w.copy("Q_FULL", "QSC", 0)
        for j in range(t + 1):
            st = j % M.NST
            w.bar("FULL%d" % st).arrive(4)
            for r in ("K", "KSC", "V", "VSC"):
                w.copy("FULL%d" % st, "%s%d" % (r, st), j)
            yield
        while not w.bar("Q_FULL").passed(0):
            yield

    monkeypatch.setattr(M, "_producer", producer_without_wait)
    failures, _ = M.count_failures(seeds=4, tiles=(5, 8), abort_ps=(0.0,))
    monkeypatch.setattr(M, "_producer", original)
    assert failures > 0
