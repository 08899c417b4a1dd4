"""Randomised model of the work queue shared by the persistent main clusters and the side clusters
(csrc/flce_bwd.cu, claim_unit / launch_corun), on the CPU.

One 64-bit word holds the main units claimed (low half) and the side units claimed (high half).  A main
cluster (P pairs) takes unit a (row pair a / main_groups, the P chunks of H group a mod main_groups) while
that row pair is below every row pair the side has begun; a side cluster (S pairs) takes unit b (row pair
R - 1 - b / side_groups, the S chunks of group b mod side_groups), always when it continues a row pair
already begun and, for a new row pair, only while that row pair lies at least `reserve` row pairs above
every row pair the main launch has begun.  A single-pair cluster takes the same units as a side cluster,
from the same count, under its own reserve, and computes their S chunks one at a time.
Every update is a compare-and-swap of the whole word.

The model runs main, side and single-pair claimers in random orders (each claim reads the word, then
tries its swap, which fails when another claimer swapped in between) and asserts: every (row pair, H
chunk) is computed exactly once; no row pair is shared between the main launch and the others; neither
the side nor the single-pair launch begins a row pair within its reserve of the main launch's; every
launch stops.  Planted mistakes in the rule must be caught.
"""
import random

import pytest


def claim(word, role, R, mg, sg, reserve, mistake=None):
    """The next unit for `role` ("main", "side" or "single") given the word, and the new word; (None, word)
    when there is none."""
    a, b = word & 0xFFFFFFFF, word >> 32
    a_rows = (a + mg - 1) // mg
    b_rows = (b + sg - 1) // sg
    if role == "main":
        limit = R if mistake == "main ignores the side" else R - b_rows
        if a // mg >= limit:
            return None, word
        return a, word + 1
    check = role == "single" or b % sg == 0
    if mistake == "side opens without the reserve":
        check = False
    if mistake == "single continues without its reserve" and role == "single":
        check = b % sg == 0
    if check and (R - 1 - b // sg) - a_rows < reserve:
        return None, word
    return b, word + (1 << 32)


def run(R, H_chunks, n_main, n_side, reserve, seed, mistake=None, P=4, S=1, n_single=0, reserve_single=None):
    """P pairs per main cluster (a main unit: P chunks of one row pair), S per side cluster (S chunks);
    single-pair clusters take side units (S chunks, one at a time) under reserve_single."""
    rng = random.Random(seed)
    mg, sg = H_chunks // P, H_chunks // S
    if reserve_single is None:
        reserve_single = reserve
    reserve_single = max(reserve_single, reserve)   # (as launch_corun sets it)
    word = 0
    done = {}                       # (row pair, chunk) -> launch
    rows_of = {"main": set(), "side": set(), "single": set()}
    active = ([("main", i) for i in range(n_main)] + [("side", i) for i in range(n_side)]
              + [("single", i) for i in range(n_single)])
    stale = {c: None for c in active}   # word each claimer read before its swap
    finished = set()
    steps = 0
    while len(finished) < len(active):
        steps += 1
        assert steps < 10 ** 6, "the claimers did not stop"
        c = rng.choice([x for x in active if x not in finished])
        role = c[0]
        if stale[c] is None:
            stale[c] = word             # read the word
            continue
        seen = stale[c]
        stale[c] = None
        unit, new = claim(seen, role, R, mg, sg, reserve_single if role == "single" else reserve, mistake)
        if unit is None:
            if seen == word:
                finished.add(c)         # nothing left for this claimer
            continue
        if seen != word:
            continue                    # the swap failed: read again
        word = new
        if role == "main":
            row, chunks = unit // mg, [P * (unit % mg) + k for k in range(P)]
        else:
            row, chunks = R - 1 - unit // sg, [S * (unit % sg) + k for k in range(S)]
            a_rows = ((word & 0xFFFFFFFF) + mg - 1) // mg
            if role == "single":
                assert row - a_rows >= reserve_single, "a single-pair cluster took a unit within its reserve"
            elif unit % sg == 0:
                assert row - a_rows >= reserve or mistake, "side began a row pair within the reserve"
        assert 0 <= row < R, "claimed a row pair outside the pass"
        rows_of[role].add(row)
        for k in chunks:
            assert (row, k) not in done, f"row pair {row} chunk {k} computed twice"
            done[(row, k)] = role
    assert not (rows_of["main"] & (rows_of["side"] | rows_of["single"])), "a row pair was split between the launches"
    missing = [(r, k) for r in range(R) for k in range(H_chunks) if (r, k) not in done]
    assert not missing, f"{len(missing)} (row pair, chunk) units never computed, e.g. {missing[:3]}"
    return rows_of


@pytest.mark.parametrize("R,H_chunks,P,S,n_main,n_side,reserve", [
    (256, 4, 4, 2, 15, 8, 11),     # the long workload's grad_input pass (two-pair side clusters)
    (689, 4, 4, 2, 15, 8, 23),     # its grad_W pass
    (65, 4, 4, 2, 15, 8, 23),      # the GPU test shape
    (256, 4, 4, 1, 15, 16, 19),    # single-pair side clusters
    (47, 8, 4, 2, 15, 8, 10),      # two H groups per main unit
    (1001, 9, 3, 1, 23, 7, 40),    # the rule with three-pair main clusters and single-pair side clusters
    (40, 4, 4, 2, 3, 1, 1),        # minimal reserve
    (45, 4, 4, 2, 15, 8, 100),     # a reserve the side can never meet: main does everything
])
def test_work_queue_covers_every_unit_once(R, H_chunks, P, S, n_main, n_side, reserve):
    for seed in range(20):
        rows = run(R, H_chunks, n_main, n_side, reserve, seed, P=P, S=S)
        if reserve >= R:
            assert not rows["side"]


@pytest.mark.parametrize("R,n_side,n_single,reserve,reserve_single", [
    (256, 6, 4, 11, 38),    # the long workload's grad_input pass: side and single-pair clusters
    (689, 6, 4, 23, 75),    # its grad_W pass
    (97, 6, 4, 11, 75),     # the GPU test shape of the grad_input pass
    (80, 6, 4, 11, 75),     # single-pair clusters that can take a unit only before the main launch begins
    (60, 6, 4, 11, 75),     # single-pair clusters that never can
    (40, 6, 4, 1, 1),       # minimal reserves
])
def test_work_queue_with_single_pair_clusters(R, n_side, n_single, reserve, reserve_single):
    took = 0
    for seed in range(20):
        rows = run(R, 4, 15, n_side, reserve, seed, P=4, S=2, n_single=n_single, reserve_single=reserve_single)
        if R - 1 < reserve_single:
            assert not rows["single"]
        took += len(rows["single"])
    if R - 15 - 1 >= reserve_single + 4:
        assert took > 0, "the single-pair clusters never took a unit"


@pytest.mark.parametrize("mistake", ["main ignores the side", "side opens without the reserve"])
def test_work_queue_planted_mistakes_are_caught(mistake):
    with pytest.raises(AssertionError):
        for seed in range(20):
            run(256, 4, 15, 8, 11, seed, mistake, P=4, S=2)


@pytest.mark.parametrize("mistake", ["main ignores the side", "single continues without its reserve"])
def test_work_queue_planted_mistakes_with_single_pair_clusters(mistake):
    # the single-pair clusters share the side count: a main launch that ignored it would take their rows
    # too; and a single-pair cluster must not continue a side row pair close to the main launch's
    with pytest.raises(AssertionError):
        for seed in range(20):
            run(256, 4, 15, 6, 11, seed, mistake, P=4, S=2, n_single=4, reserve_single=38)
