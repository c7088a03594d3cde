"""The split-KV schedule restatement and its invariant checker (CPU only)."""
import random

import pytest

from oracle.schedule import check_schedule, expand_segments, schedule_reference


def test_hand_worked_example():
    # pages per request: 3, 5, 0, 2; two parts, per-segment cost 1
    seqlens = [3 * 64, 4 * 64 + 1, 0, 2 * 64]
    meta, ns = schedule_reference(seqlens, num_parts=2, fixed_cost=1, hbm_parts=100)
    # costs 4, 6, 0, 3 -> C = 0, 4, 10, 10, 13; T = ceil(13 / 2) = 7; pages sit at
    # positions 1-3 (request 0), 5-9 (request 1), 11-12 (request 3)
    assert meta == [(0, 0, 1, 2, 0), (1, 2, 3, 2, 1)]
    assert ns == [0, 1, 3, 3, 4]
    check_schedule(meta, ns, seqlens)


def test_hbm_parts_caps_the_spread():
    seqlens = [3 * 64, 5 * 64, 0, 2 * 64]
    meta, ns = schedule_reference(seqlens, num_parts=4, fixed_cost=1, hbm_parts=2)
    assert meta == [(0, 0, 1, 2, 0), (1, 2, 3, 2, 1), (-1, 0, 0, 0, 0), (-1, 0, 0, 0, 0)]
    assert ns == [0, 1, 3, 3, 4]
    check_schedule(meta, ns, seqlens)


def test_uniform_batch_without_splits():
    # 64 requests of 64 pages on 64 effective parts: one request per part, no split
    seqlens = [4096] * 64
    meta, ns = schedule_reference(seqlens, num_parts=76, fixed_cost=2, hbm_parts=64)
    assert ns == list(range(65))
    assert all(m == (i, 0, i, 64, 0) for i, m in enumerate(meta[:64]))
    assert all(m[0] == -1 for m in meta[64:])


def test_single_long_request_is_split_evenly():
    seqlens = [131072]                      # 2048 pages
    meta, ns = schedule_reference(seqlens, num_parts=16, fixed_cost=2, hbm_parts=64)
    segs = expand_segments(meta, seqlens)
    sizes = [ke - kb for _, _, kb, ke, _ in segs]
    assert len(segs) == 16 and ns == [0, 16]
    # cost 2048 + 2 = 2050 -> T = 129 positions per part; part 0 also holds the set-up
    assert sizes == [127] + [129] * 14 + [115]
    check_schedule(meta, ns, seqlens)


@pytest.mark.parametrize("seed", range(40))
def test_random_schedules_are_valid(seed):
    rng = random.Random(seed)
    B = rng.randint(1, 300)
    seqlens = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 20000)]) for _ in range(B)]
    P = rng.randint(1, 160)
    meta, ns = schedule_reference(seqlens, P, fixed_cost=rng.randint(0, 6), hbm_parts=rng.randint(1, 200))
    assert len(meta) == P
    check_schedule(meta, ns, seqlens)


def test_checker_rejects_broken_schedules():
    seqlens = [5 * 64, 7 * 64, 3 * 64]
    meta, ns = schedule_reference(seqlens, 3, 1, 100)
    check_schedule(meta, ns, seqlens)
    broken = {
        "gap": [list(m) for m in meta],
        "overlap": [list(m) for m in meta],
        "split index": [list(m) for m in meta],
    }
    # find a part that starts inside a request (k_first > 0)
    idx = next(i for i, m in enumerate(meta) if m[1] > 0)
    broken["gap"][idx][1] += 1
    broken["overlap"][idx][1] -= 1
    broken["split index"][idx][4] += 1
    for name, m in broken.items():
        with pytest.raises(AssertionError):
            check_schedule([tuple(x) for x in m], ns, seqlens)
    bad_ns = list(ns)
    bad_ns[-1] += 1
    with pytest.raises(AssertionError):
        check_schedule(meta, bad_ns, seqlens)


def test_split_cost_picks_the_part_count():
    # 64 equal requests: 64 parts take one request each; 76 parts would split them all
    seqlens = [4096] * 64
    meta, ns = schedule_reference(seqlens, num_parts=76, fixed_cost=2, hbm_parts=64, split_cost=12)
    assert ns == list(range(65)) and all(m[0] == -1 for m in meta[64:])
    # 4 long requests are split anyway: all 76 parts are used
    seqlens = [131072] * 4
    meta, ns = schedule_reference(seqlens, num_parts=76, fixed_cost=2, hbm_parts=64, split_cost=12)
    assert sum(1 for m in meta if m[0] >= 0) == 76
    check_schedule(meta, ns, seqlens)


@pytest.mark.parametrize("seed", range(20))
def test_random_schedules_with_split_cost_are_valid(seed):
    rng = random.Random(100 + seed)
    B = rng.randint(1, 200)
    seqlens = [rng.choice([0, rng.randint(1, 64), rng.randint(1, 20000)]) for _ in range(B)]
    P = rng.randint(1, 160)
    meta, ns = schedule_reference(seqlens, P, fixed_cost=rng.randint(0, 6), hbm_parts=rng.randint(1, 200),
                                  split_cost=rng.randint(1, 20))
    check_schedule(meta, ns, seqlens)
