"""The synchronisation of the fused forward's four-CTA form (d_v = 512), on a
model of its barriers and buffers (`quad_protocol_model.py`, CPU only): no
deadlock, no wait that could take phase k + 2 for phase k, and no overlapping
use of a pair's O accumulator or of a CTA's P buffer, over the work-item
schedules of the GPU tests and of the bench's d = 512 layers and many random
interleavings; and each planted mistake is caught."""
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
            status, errors = Q.run(items, seed, nkg=nkg, nk=nk, nv=nv)
            assert status == "ok" and not errors, (c, seed, status, errors[:3])


def test_long_sequence_schedule_runs_clean():
    items = Q.cluster_items(36, 0, 1, 4, 16384)
    for seed in range(2):
        status, errors = Q.run(items, seed)
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
                status, errors = Q.run(items, seed, mutation=mutation)
                caught += status != "ok" or bool(errors)
    assert caught > 0, MUTATIONS[mutation]
