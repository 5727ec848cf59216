"""The multi-round schedule of the oracle against closed forms, invariants
and its slot-by-slot second form (CPU)."""
import numpy as np
import pytest

from oracle import multiround as mr


def _check_invariants(counts, E, C, G, s):
    take, start, ro, R = s["take"], s["start"], s["round_offsets"], s["R"]
    assert take.shape == (R, E) and R >= 1
    assert np.array_equal(take.sum(axis=0), counts)          # nothing dropped
    for grp in mr.groups_of(E, G):
        assert (take[:, grp].sum(axis=1) <= C * len(grp)).all()  # group capacity per round
        n = counts[grp].sum()
        assert R >= -(-n // (C * len(grp)))
    assert (ro[:, -1] <= C * E).all()                       # the round buffer holds a round
    assert np.array_equal(start[0], np.zeros(E))
    # every expert takes its own capacity first
    rem = counts.copy()
    for r in range(R):
        assert (take[r] >= np.minimum(rem, C)).all()
        rem = rem - take[r]


def test_one_round_when_everything_fits():
    counts = np.array([3, 0, 4, 1, 2, 4, 0, 4])
    s = mr.schedule(counts, 8, 4, 4)
    assert s["R"] == 1 and np.array_equal(s["take"][0], counts)
    assert s["round_offsets"][0].tolist() == [0, 3, 3, 7, 8, 10, 14, 14, 18]


def test_borrowing_inside_a_group_avoids_a_round():
    # e0 has 6 > C = 4, but its group (e0, e1) leaves 1 + ... unused: 6 + 2 <= 8
    s = mr.schedule(np.array([6, 2, 1, 1]), 4, 4, 2)
    assert s["R"] == 1 and s["take"][0].tolist() == [6, 2, 1, 1]
    # without borrowing across groups: e0's group has 6 + 3 = 9 > 8 seats
    s = mr.schedule(np.array([6, 3, 0, 0]), 4, 4, 2)
    assert s["R"] == 2
    assert s["take"].tolist() == [[5, 3, 0, 0], [1, 0, 0, 0]]  # e1 first takes its own 3


def test_round_count_is_global():
    # only group 1 overflows; group 0 then runs an empty second round
    s = mr.schedule(np.array([1, 1, 9, 9]), 4, 4, 2)
    assert s["R"] == 3
    assert s["take"][:, :2].sum(axis=0).tolist() == [1, 1] and s["take"][1:, :2].sum() == 0


def test_lending_goes_to_the_lowest_expert_first():
    s = mr.schedule(np.array([7, 7, 0, 0]), 4, 2, 4)  # 8 seats, 4 owned, 4 lent
    assert s["take"][0].tolist() == [6, 2, 0, 0]
    assert s["take"][1].tolist() == [1, 5, 0, 0]


@pytest.mark.parametrize("seed", range(12))
def test_matches_slot_by_slot_form(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 20))
    G = int(rng.integers(1, E + 1))
    C = int(rng.integers(1, 9))
    counts = rng.zipf(1.5, size=E).clip(max=60) - 1 if seed % 2 else rng.integers(0, 12, size=E)
    counts = np.asarray(counts, dtype=np.int64)
    s = mr.schedule(counts, E, C, G)
    _check_invariants(counts, E, C, G, s)
    placed = mr.schedule_by_slots(counts, E, C, G)
    for e in range(E):
        want = np.repeat(np.arange(s["R"]), s["take"][:, e])
        assert placed[e] == want.tolist(), (e, placed[e], want)


def test_rounds_equal_the_largest_group_ceiling():
    rng = np.random.default_rng(7)
    for _ in range(50):
        E, G, C = 16, 4, 3
        counts = rng.integers(0, 20, size=E)
        s = mr.schedule(counts, E, C, G)
        need = max(-(-int(counts[g].sum()) // (C * len(g))) for g in mr.groups_of(E, G))
        assert s["R"] == max(1, need)


# ---------------------------------------------------------------- planted mistakes

def _no_borrowing(counts, E, capacity, group_size):
    counts = np.asarray(counts, dtype=np.int64)
    R = max(1, int(-(-counts.max() // capacity)))
    take = np.stack([np.clip(counts - r * capacity, 0, capacity) for r in range(R)])
    ro = np.zeros((R, E + 1), dtype=np.int64)
    ro[:, 1:] = np.cumsum(take, axis=1)
    return {"take": take, "start": np.cumsum(take, 0) - take, "round_offsets": ro, "R": R}


def _lend_highest_first(counts, E, capacity, group_size):
    rev = mr.schedule(np.asarray(counts)[::-1].copy(), E, capacity, group_size)
    return {"take": rev["take"][:, ::-1], "start": rev["start"][:, ::-1],
            "round_offsets": None, "R": rev["R"]}


def _one_group(counts, E, capacity, group_size):
    return mr.schedule(counts, E, capacity, E)


PLANTED = {"no_borrowing": _no_borrowing, "lend_highest_first": _lend_highest_first,
           "borrow_across_groups": _one_group}


@pytest.mark.parametrize("name", sorted(PLANTED))
def test_planted_schedule_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(mr, "schedule", PLANTED[name])
    caught = 0
    checks = [test_one_round_when_everything_fits, test_borrowing_inside_a_group_avoids_a_round,
              test_round_count_is_global, test_lending_goes_to_the_lowest_expert_first,
              test_rounds_equal_the_largest_group_ceiling] + \
        [lambda s=s: test_matches_slot_by_slot_form(s) for s in range(12)]
    for c in checks:
        try:
            c()
        except Exception:
            caught += 1
    assert caught, name
