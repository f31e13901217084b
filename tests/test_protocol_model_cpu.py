"""The attention kernels' synchronisation protocols, checked on random-interleaving models
(tests/fwd_protocol_model.py for the forward, tests/bwd_protocol_model.py for the backward's dK/dV
and dQ roles, tests/fwd_own_p_protocol_model.py for a forward with P in TMEM columns of its own) on
the CPU: no deadlock, no named-barrier generation holding two tiles, no stale or
overwritten buffer, also when bounded waits give up mid-run.  Each model must also catch planted
mistakes (and the forward model the earlier two-ID form of the P hand-over), so that a model that
checks nothing cannot pass."""
import pytest

import bwd_protocol_model as BM
import fwd_own_p_protocol_model as PM
import fwd_protocol_model as FM


def test_forward_protocol_as_built_is_clean():
    failures, first = FM.count_failures(seeds=12, n_pids=3)
    assert failures == 0, first


def test_forward_protocol_without_aborts_is_clean_on_long_runs():
    for seed in range(6):
        for own in (True, False):
            FM.run(t=21, own=own, seed=seed, rescale_p=0.5)


def test_forward_two_p_ids_mix_generations_after_a_mid_run_abort():
    # the form the kernel had before: tile parity picks the ID; a warp that gives up at tile j can
    # join tile j - 2's generation while a slower warp has not arrived there
    failures, _ = FM.count_failures(seeds=40, tiles=(5, 8, 13), abort_ps=(0.002, 0.02), n_pids=2)
    assert failures > 0


def test_forward_two_softmax_sets_are_clean():
    # the kernel with two P terms: two sets of softmax warps take alternate key tiles
    failures, first = FM.count_failures(seeds=10, sets=2)
    assert failures == 0, first


@pytest.mark.parametrize("mistake", ["publish_before_take", "no_final_take"])
def test_forward_two_set_model_catches_planted_mistakes(mistake):
    failures, _ = FM.count_failures(seeds=6, tiles=(0, 1, 3, 6), abort_ps=(0.0,), sets=2, mistake=mistake)
    assert failures > 0


def test_forward_model_catches_a_missing_stage_wait():
    failures, _ = FM.count_failures(seeds=4, tiles=(5, 8), abort_ps=(0.0,), mistake="no_stage_wait")
    assert failures > 0


@pytest.mark.parametrize("kind", ["dkdv", "dq"])
def test_backward_protocols_as_built_are_clean(kind):
    failures, first = BM.count_failures(kind, seeds=15)
    assert failures == 0, first


@pytest.mark.parametrize("kind,mistake", [("dkdv", "no_pd_wait"), ("dkdv", "first_ld_arrive"),
                                          ("dq", "no_cp_wait"), ("dq", "dp_before_dq")])
def test_backward_models_catch_planted_mistakes(kind, mistake):
    failures, _ = BM.count_failures(kind, seeds=10, mistake=mistake)
    assert failures > 0


@pytest.mark.parametrize("sets,npb", [(1, 1), (1, 2), (2, 1), (2, 2)])
def test_own_p_forward_protocol_is_clean(sets, npb):
    failures, first = PM.count_failures(seeds=6, sets=sets, npb=npb)
    assert failures == 0, first


@pytest.mark.parametrize("mistake", ["no_pfree_wait", "no_rescale_wait", "sc_before_load"])
@pytest.mark.parametrize("sets,npb", [(1, 1), (2, 2)])
def test_own_p_model_catches_planted_mistakes(mistake, sets, npb):
    failures, _ = PM.count_failures(seeds=2, tiles=(3, 5), abort_ps=(0.0,), sets=sets, npb=npb, mistake=mistake)
    assert failures > 0


def test_own_p_protocol_needs_five_stages():
    # with four stages the producer's rule (tile j - 2's scores) frees a stage P(j - 4).V may still read
    failures, _ = PM.count_failures(seeds=4, abort_ps=(0.0,), sets=2, npb=2, nst=4)
    assert failures > 0
