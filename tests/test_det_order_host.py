"""The deterministic backward's order of dQ additions, restated and checked on
the host (FlashAttention-4 summary, section 3.2.4): key tiles start in ticket
order on a limited number of SMs, each walks its query tiles, and an addition
into query tile i waits until every key tile ahead of it in i's order has added.

Shortest-processing-time order (causal: walk up from the diagonal, additions in
descending key order) never deadlocks whatever the residency, and no key tile
waits on its first addition. The rotated walk (non-causal, equal lengths) is
deadlock-free as long as all key tiles of a (batch, head) fit on the SMs, and
keeps every query tile receiving one addition per step. The ascending order
(no mask) is deadlock-free but skews: key tile j cannot start before j - 1."""

import collections

import pytest


def run(n_heads, nk, causal, order, n_sm, max_time=100000):
    """Unit-time simulation; returns the number of steps, or None on deadlock."""
    items = []
    for t in range(n_heads * nk):
        j = nk - 1 - t % nk if order in ("spt", "rotated") else t % nk
        items.append((t // nk, j))

    def steps(j):
        if causal:
            return [(i, i - j) for i in range(j, nk)]
        if order == "rotated":
            return [((j + k) % nk, k) for k in range(nk)]
        return [(i, i) for i in range(nk)]

    def turn(j, k):
        return k if order in ("spt", "rotated") else j

    sem = collections.Counter()
    running, nxt, done, time = {}, 0, 0, 0
    first_write_waited = False
    while done < len(items):
        while len(running) < n_sm and nxt < len(items):
            running[nxt] = [steps(items[nxt][1]), 0]
            nxt += 1
        progressed, writes = False, []
        for t, st in list(running.items()):
            seq, pos = st
            if pos == len(seq):
                del running[t]
                done += 1
                progressed = True
                continue
            i, k = seq[pos]
            h, j = items[t]
            if sem[(h, i)] == turn(j, k):
                writes.append((h, i))
                st[1] += 1
                progressed = True
            elif pos == 0:
                first_write_waited = True
        for key in writes:
            sem[key] += 1
        time += 1
        if not progressed or time > max_time:
            return None, first_write_waited
    return time, first_write_waited


@pytest.mark.parametrize("n_sm", [152, 7, 1])
def test_spt_causal_is_deadlock_free_and_never_stalls_a_first_addition(n_sm):
    t, waited = run(n_heads=3, nk=12, causal=True, order="spt", n_sm=n_sm)
    assert t is not None
    assert not waited


def test_spt_causal_beats_ascending():
    spt, _ = run(n_heads=8, nk=32, causal=True, order="spt", n_sm=40)
    asc, _ = run(n_heads=8, nk=32, causal=True, order="asc", n_sm=40)
    assert spt is not None and asc is not None and spt < 0.6 * asc


def test_rotated_walk_needs_the_whole_group_resident():
    assert run(n_heads=4, nk=16, causal=False, order="rotated", n_sm=16)[0] is not None
    assert run(n_heads=4, nk=16, causal=False, order="rotated", n_sm=40)[0] is not None
    # fewer SMs than key tiles in a group: the cyclic waits cannot all be met
    assert run(n_heads=1, nk=16, causal=False, order="rotated", n_sm=8)[0] is None


def test_rotated_walk_beats_ascending_and_ascending_is_always_safe():
    rot, _ = run(n_heads=8, nk=16, causal=False, order="rotated", n_sm=64)
    asc, _ = run(n_heads=8, nk=16, causal=False, order="asc", n_sm=64)
    assert rot < asc
    assert run(n_heads=2, nk=16, causal=False, order="asc", n_sm=3)[0] is not None
