"""The synchronisation of the parallel-to-recurrent hand-off kernel, on a model
of its barriers and buffers (`handoff_protocol_model.py`, CPU only): over unit
schedules with pieces of many units and of one, a CTA's range starting inside
a head, and two to four stages, random interleavings show no deadlock, no
parity wait that could be misread and no overlapping use of a stage or of the
accumulator; with a wait giving up at a random step, every warp still leaves
(the debt loop keeps the twelve weighting warps' barriers matched); and each
planted mistake is caught."""
import random

import pytest

import handoff_protocol_model as F

# (units in the CTA's range, chunks per head, first unit's chunk, stages)
SCHEDULES = [(20, 32, 5, 3), (7, 2, 1, 3), (1, 1, 0, 3), (12, 4, 3, 2), (30, 8, 0, 4), (9, 3, 2, 3)]


@pytest.mark.parametrize("sched", SCHEDULES, ids=lambda s: "x".join(map(str, s)))
def test_schedule_runs_clean(sched):
    for seed in range(12):
        status, errors, _ = F.run(*sched, seed)
        assert status == "ok" and not errors, (seed, status, errors[:3])


def _timeout_runs(sched, n_runs, **kw):
    _, _, length = F.run(*sched, 0, **kw)
    rng = random.Random(sum(sched) * 7919 + n_runs)
    for seed in range(n_runs):
        yield F.run(*sched, seed, give_up_at=rng.randrange(1, length), **kw)


@pytest.mark.parametrize("sched", SCHEDULES, ids=lambda s: "x".join(map(str, s)))
def test_waits_that_give_up_leave_no_warp_stranded(sched):
    for status, errors, _ in _timeout_runs(sched, 40):
        assert status == "ok", errors[-3:]


MUTATIONS = {
    "empty_count": "a stage counted empty at the MMA commit alone (the n warps may still read its K)",
    "no_debt": "a warp that left early does not make up the barriers of the units it skipped",
    "debt_no_piece": "the make-up skips the piece-end agreement",
    "acc_plain": "the piece-end meeting does not agree on the exit",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    caught = 0
    for sched in SCHEDULES[:2] + SCHEDULES[3:5]:
        if mutation == "empty_count":
            runs = (F.run(*sched, seed, mutation=mutation) for seed in range(6))
        else:
            runs = _timeout_runs(sched, 40, mutation=mutation)
        for status, errors, _ in runs:
            caught += status != "ok" or (mutation == "empty_count" and bool(errors))
    assert caught > 0, MUTATIONS[mutation]
