"""Multi-round fixed-capacity expert schedule (test infrastructure).

Only ``tests/`` may import this module; it shares no code with the CUDA
library.

"Frontier Pre-training at Microsoft AI", section "Dropless MoE with tunable,
fixed-size memory usage", and "MAI-Base-2: Microsoft's 2.8T base model, and
whether its compute numbers add up" (the multi-round dropless passage): the
experts are put into groups; every group runs one or more rounds, each with a
fixed token capacity per expert; an expert that receives more tokens than its
capacity first uses capacity that other experts of its group leave unused in
that round, and only what still does not fit waits for another round; the
number of rounds is the same for every group (the largest any group needs).
No token is dropped, so the layer's output is that of the dropless forward.

Readings where the pages are silent:
- groups are consecutive expert ranges of ``group_size`` experts (the last
  group may be smaller);
- in each round every expert first takes up to ``capacity`` of its remaining
  slots; the group's unused capacity is then lent to experts that still have
  slots, lowest expert index first, each taking as much as it can;
- an expert's slots keep their order (token order) across rounds: round r
  takes the next ``take[r, e]`` of them;
- a round's slots are packed expert after expert into a buffer of
  E * capacity rows.
"""
from __future__ import annotations

from typing import Dict

import numpy as np


def groups_of(E: int, group_size: int):
    return [list(range(g0, min(g0 + group_size, E))) for g0 in range(0, E, group_size)]


def schedule(counts, E: int, capacity: int, group_size: int) -> Dict[str, np.ndarray]:
    """Per-round takes of every expert.

    Returns take [R, E] (slots expert e runs in round r), start [R, E] (how
    many of e's slots ran before round r), round_offsets [R, E+1] (where e's
    slots of round r begin in the round buffer) and R >= 1."""
    counts = np.asarray(counts, dtype=np.int64)
    assert counts.shape == (E,) and capacity >= 1 and group_size >= 1
    rem = counts.copy()
    takes = []
    while True:
        take = np.zeros(E, dtype=np.int64)
        for grp in groups_of(E, group_size):
            own = {e: min(int(rem[e]), capacity) for e in grp}
            pool = capacity * len(grp) - sum(own.values())
            for e in grp:  # lend the unused capacity, lowest index first
                extra = min(int(rem[e]) - own[e], pool)
                pool -= extra
                take[e] = own[e] + extra
        takes.append(take)
        rem -= take
        if not rem.any():
            break
    take = np.stack(takes)
    start = np.cumsum(take, axis=0) - take
    R = take.shape[0]
    ro = np.zeros((R, E + 1), dtype=np.int64)
    ro[:, 1:] = np.cumsum(take, axis=1)
    return {"take": take, "start": start, "round_offsets": ro, "R": R}


def schedule_by_slots(counts, E: int, capacity: int, group_size: int) -> np.ndarray:
    """Second form: the round of every slot, placing slots one at a time.

    Round by round, each group first gives every expert one seat per unit of
    its own capacity (while it has slots left), then hands the remaining seats
    of the group out one by one, to the lowest-indexed expert that still has
    slots. Returns rounds: list over experts of the round index of each of its
    slots, in slot order."""
    counts = [int(c) for c in counts]
    placed = [[] for _ in range(E)]
    r = 0
    while any(len(placed[e]) < counts[e] for e in range(E)):
        for grp in groups_of(E, group_size):
            seats = capacity * len(grp)
            for e in grp:
                for _ in range(capacity):
                    if len(placed[e]) < counts[e]:
                        placed[e].append(r)
                        seats -= 1
            while seats > 0:
                e = next((e for e in grp if len(placed[e]) < counts[e]), None)
                if e is None:
                    break
                placed[e].append(r)
                seats -= 1
        r += 1
    return placed
