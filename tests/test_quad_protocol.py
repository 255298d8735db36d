"""The synchronisation of the fused forward on CTA pairs, its four-CTA form
(d_v = 512) and its two-CTA form, on a model of their barriers and buffers
(`quad_protocol_model.py`, CPU only): no
deadlock, no parity wait that could be misread, and no overlapping use of a
pair's O accumulator, an S buffer holding P or a CTA's P buffer, over the
work-item schedules of the GPU tests and of the bench's d = 512 layers and
many random interleavings; with waits that give up at random points, every
warp still leaves (no group is stranded at a named barrier); and each planted
mistake is caught."""
import random

import pytest

import quad_protocol_model as Q


def rings(dqk):
    """K granules per tile and the K/V ring split the kernel's planner gives
    the four-CTA form (16 KB granules in the shared memory left beside Q and
    the P buffer, at most 8; V takes two granules a tile, K half of its
    granules' share because it carries every other tile only)."""
    room = 232448 - 1840 - (1024 + dqk * 128 * 2 + 128 * 128 * 2)
    total = min(8, room // 16384)
    nkg = dqk // 128
    nv = max(2, round(total * 2 / (0.5 * nkg + 2)))
    nv = min(max(nv, 1), total - 1)
    return nkg, total - nv, nv


# (B, H, T, d_qk): the GPU tests' shapes and the bench's d = 512 layers
SHAPES = [(1, 1, 1, 512), (1, 1, 100, 512), (1, 2, 129, 512), (2, 1, 384, 128), (1, 1, 777, 256),
          (1, 2, 500, 384), (8, 8, 640, 512), (1, 1, 2048, 512), (4, 4, 2048, 512)]


@pytest.mark.parametrize("n_clusters", [36, 4, 1])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_schedule_runs_clean(shape, n_clusters):
    B, H, T, dqk = shape
    nkg, nk, nv = rings(dqk)
    for c in sorted({0, n_clusters // 2, n_clusters - 1}):
        items = Q.cluster_items(n_clusters, c, B, H, T)
        if not items:
            continue
        # interleavings per cluster, fewer where its schedule is long
        for seed in range(max(1, min(6, 600 // sum(n for _, n in items)))):
            status, errors, _ = Q.run(items, seed, nkg=nkg, nk=nk, nv=nv)
            assert status == "ok" and not errors, (c, seed, status, errors[:3])


def test_long_sequence_schedule_runs_clean():
    items = Q.cluster_items(36, 0, 1, 4, 16384)
    for seed in range(2):
        status, errors, _ = Q.run(items, seed)
        assert status == "ok" and not errors, (seed, status, errors[:3])


MUTATIONS = {
    "single_pfull": "one own-P barrier for both S buffers",
    "prx_count": "the other pair's P counted from one CTA's warps",
    "bx_count": "the other pair's row sums counted from two warps",
    "no_epidone": "the first P sent in an item does not wait for the receiver's epilogue",
    "no_pempty": "a P send does not wait for the receiver's O product to consume the last one",
    "no_sempty": "an S product does not wait for the O product that reads the P stored over its buffer",
}
# Two of the kernel's waits are implied by others in this protocol, and the
# model shows no hazard without them: the next item's first O product waiting
# for the epilogue's read-out of O (its P comes from warps that finished that
# epilogue, or from the other pair after it), and an item without tiles of a
# pair waiting for the other pair's previous epilogue (the row-sum exchange
# already keeps the pairs within one item).  The kernel keeps both.


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    caught = 0
    for shape, n_clusters in (((8, 8, 640, 512), 36), ((1, 2, 500, 512), 1), ((2, 1, 384, 512), 1)):
        B, H, T, dqk = shape
        for c in range(min(n_clusters, 3)):
            items = Q.cluster_items(n_clusters, c, B, H, T)
            for seed in range(12):
                status, errors, _ = Q.run(items, seed, mutation=mutation)
                caught += status != "ok" or bool(errors)
    assert caught > 0, MUTATIONS[mutation]


def _timeout_runs(items, n_runs, **kw):
    """Runs with one wait giving up at a step drawn over the length of a clean
    run (early, mid-item and at item ends alike)."""
    _, _, length = Q.run(items, 0, **kw)
    rng = random.Random(len(items) * 7919 + n_runs)
    for seed in range(n_runs):
        yield Q.run(items, seed, give_up_at=rng.randrange(1, length), **kw)


@pytest.mark.parametrize("shape", [(8, 8, 640, 512), (1, 2, 500, 512), (2, 1, 384, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_waits_that_give_up_leave_no_group_stranded(shape):
    """A wait runs out of its budget (the kernel's spin limit) at a random
    point: every role must still reach the end, through the reducing barriers
    where the gating warps agree on their exit."""
    B, H, T, dqk = shape
    nkg, nk, nv = rings(dqk)
    for n_clusters, n_runs in ((36, 40), (4, 6)):
        items = Q.cluster_items(n_clusters, 0, B, H, T)
        for status, errors, _ in _timeout_runs(items, n_runs, nkg=nkg, nk=nk, nv=nv):
            assert status == "ok", (n_clusters, errors[-3:])


EXIT_MUTATIONS = {
    "exit_early": "a gating warp whose wait gave up leaves without meeting its group",
    "exit_unreduced": "the gating warps meet before the epilogue without agreeing on the exit",
}


@pytest.mark.parametrize("mutation", sorted(EXIT_MUTATIONS))
def test_planted_exit_mistake_strands_a_group(mutation):
    stranded = 0
    for shape in ((8, 8, 640), (4, 4, 2048)):
        items = Q.cluster_items(36, 0, *shape)
        for status, _, _ in _timeout_runs(items, 60, mutation=mutation):
            stranded += status == "deadlock"
    assert stranded > 0, EXIT_MUTATIONS[mutation]


# The two-CTA form: (B, H, T, nsplit, ring planner inputs) for the 125M-scale
# layer (d = 384: one S buffer, 3 + 3 granules, three V granules a tile), the
# split form at d_v = 512 (two slices, 2 + 2), d = 256 (two S buffers, 4 + 4)
# and a one-token sequence.
PAIR_FORMS = {
    "d384": dict(nsbuf=1, nkg=3, nk=3, nv=3, vpt=3),
    "d512split": dict(nsbuf=2, nkg=4, nk=2, nv=2, vpt=2),
    "d256": dict(nsbuf=2, nkg=2, nk=4, nv=4, vpt=2),
}
PAIR_CASES = [("d384", (8, 4, 2048), 1), ("d384", (1, 1, 1), 1), ("d512split", (4, 4, 2048), 2),
              ("d256", (2, 2, 300), 1)]


@pytest.mark.parametrize("case", PAIR_CASES, ids=lambda c: c[0] + "-" + "x".join(map(str, c[1])))
def test_pair_form_runs_clean_and_leaves_on_timeouts(case):
    form, (B, H, T), nsplit = case
    kw = dict(form="pair", **PAIR_FORMS[form])
    for n_clusters, n_runs in ((76, 20), (4, 3)):
        items = Q.cluster_items(n_clusters, 0, B, H, T, nsplit)
        if not items:
            continue
        for seed in range(4):
            status, errors, _ = Q.run(items, seed, **kw)
            assert status == "ok" and not errors, (n_clusters, seed, errors[:3])
        for status, errors, _ in _timeout_runs(items, n_runs, **kw):
            assert status == "ok", (n_clusters, errors[-3:])


@pytest.mark.parametrize("mutation", ["pair_exit_early", "pair_sempty_count"])
def test_pair_form_planted_mistake_is_caught(mutation):
    kw = dict(form="pair", mutation=mutation, **PAIR_FORMS["d384"])
    caught = 0
    for c in (0, 40, 75):
        items = Q.cluster_items(76, c, 8, 4, 2048)
        for status, errors, _ in _timeout_runs(items, 60, **kw):
            caught += status != "ok"
        for seed in range(4):
            status, errors, _ = Q.run(items, seed, **kw)
            caught += status != "ok" or bool(errors)
    assert caught > 0, mutation
