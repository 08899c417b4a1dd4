"""Randomised interleaving model of the gradient passes' dS hand-over (csrc/flce_bwd.cu), on the CPU.

The kernel's actors -- each pair's MMA issuer, each CTA's receiver warp, the epilogue warp groups of
each half of each CTA -- are generators stepped in a random order, with copies between CTAs landing at
random times.  The model follows the kernel's protocol with S half-block dS slots per CTA: content
n = 2j + h (half h of column block j) sits in slot n mod S; the pair that owns block j (j mod P) writes it
into its own slot and sends it to the other pairs; before overwriting a copy it waits until the pair
holding that copy has run GEMM2 on the slot's previous content (ds_free[slot][pair], one arrival by that
pair's MMA commit, parity = the writer's earlier waited writes into the slot); receivers arm rx_full,
wait, and arrive on their pair's ds_full; GEMM2 of content n waits ds_full[slot] at parity n // S.  It
asserts that every parity wait is unambiguous (the barrier is never two phases away from the waited
one), that no copy of a slot is overwritten before its pair consumed it, that GEMM2 reads the content it
expects, and that nothing deadlocks.

The kernel uses S = 2 (two pairs or three per cluster) and S = 3 or 4 (four pairs); with S odd a slot
holds contents of either half in turn, so the writer counts its waits per slot in content order over both
halves.  Random orders are run as well as orders in which one pair's actors are starved.  Two planted protocol
mistakes must be caught: a release sent to the next block's owner instead of the slot's next writer,
and a writer that sends to the other pairs without waiting until each of them is done with the slot.
"""
import random

import pytest

import random, sys


class Bar:
    def __init__(s, name, count):
        s.name, s.count, s.pending, s.done, s.tx = name, count, count, 0, 0
    def arrive(s, tx=0):
        s.tx += tx; s.pending -= 1
        assert s.pending >= 0, f"{s.name}: too many arrivals"
        s._maybe()
    def complete_tx(s, b):
        s.tx -= b; s._maybe()
    def _maybe(s):
        if s.pending == 0 and s.tx == 0:
            s.done += 1; s.pending = s.count
    def poll(s, phase, who):
        assert s.done in (phase, phase + 1), f"{who}: alias on {s.name}: done={s.done} want={phase}"
        return s.done == phase + 1


def g1_share(s, pr, P):
    lead = P + 1
    d = (pr - (s + lead)) % P
    return s + lead + d, P - 1 - d


def run(P, S, nt, nkb, seed, mistake=None, slow_pair=None):
    rnd = random.Random(seed)
    B = {}
    for p in range(P):
        for c in range(2):
            for k in range(S):
                for q in range(P):
                    B[(p, c, "free", k, q)] = Bar(f"ds_free[{p}.{c}][{k}][{q}]", 1)
                B[(p, c, "rx", k)] = Bar(f"rx[{p}.{c}][{k}]", 1)
        for k in range(S):
            B[(p, "full", k)] = Bar(f"ds_full[{p}][{k}]", 2)
        B[(p, "s_full")] = Bar(f"s_full[{p}]", 1)
        B[(p, "s_empty")] = Bar(f"s_empty[{p}]", 4)
    slot = {(p, c, k): None for p in range(P) for c in range(2) for k in range(S)}
    consumed = {(p, k): set() for p in range(P) for k in range(S)}   # contents consumed by pair p's GEMM2
    inflight = []
    s_tile = {p: None for p in range(P)}

    def write(p, c, k, content):
        prev = slot[(p, c, k)]
        if prev is not None:
            assert prev in consumed[(p, k)], f"overwrite of {prev} in {p}.{c} slot {k} before GEMM2 consumed it"
        slot[(p, c, k)] = content

    def mma(p):
        u = 0
        for s in range(-2 * P, nt):
            blk, prog = g1_share(s, p, P)
            has = 0 <= blk < nt
            if s >= 0:
                for h in range(2):
                    n = 2 * s + h; k = n % S
                    while not B[(p, "full", k)].poll(n // S, f"mma{p} full"):
                        yield
                    for c in range(2):
                        assert slot[(p, c, k)] == (s, h), f"pair {p} slot {k} holds {slot[(p, c, k)]} want {(s, h)}"
                    consumed[(p, k)].add((s, h))
                    nx = n + S
                    if mistake == "release to the next block's owner":
                        nx = n + 2
                    if nx // 2 < nt:
                        o = (nx // 2) % P
                        for c in range(2):
                            B[(o, c, "free", k, p)].arrive()
                    yield
            if has:
                if prog == 0:
                    while u > 0 and not B[(p, "s_empty")].poll(u - 1, f"mma{p} s_empty"):
                        yield
                    s_tile[p] = ("busy", blk)
                yield
                if prog == P - 1:
                    s_tile[p] = ("ready", blk)
                    B[(p, "s_full")].arrive()
                    u += 1

    def epi(p, c, hh):
        u = 0
        waits = [0] * S
        for j in range(p, nt, P):
            while not B[(p, "s_full")].poll(u, f"epi{p}.{c}.{hh} s_full"):
                yield
            assert s_tile[p] == ("ready", j), (p, s_tile[p], j)
            B[(p, "s_empty")].arrive()
            u += 1
            yield
            n = 2 * j + hh; k = n % S
            ph = sum(1 for m in range(S, n) if m % S == k and (m // 2) % P == p)
            if n >= S:
                while not B[(p, c, "free", k, p)].poll(ph, f"epi{p}.{c}.{hh} free{k}"):
                    yield
            write(p, c, k, (j, hh))
            for q in range(P):
                if q != p:
                    if n >= S and mistake != "no wait for the other pairs":
                        while not B[(p, c, "free", k, q)].poll(ph, f"epi{p}.{c}.{hh} free{k}/{q}"):
                            yield
                    inflight.append((q, c, k, (j, hh)))
                    yield
            yield
            B[(p, "full", k)].arrive()

    def recv(p, c):
        v = [0] * S
        for j in range(nt):
            if j % P == p:
                continue
            for h in range(2):
                k = (2 * j + h) % S
                B[(p, c, "rx", k)].arrive(tx=1)
                while not B[(p, c, "rx", k)].poll(v[k], f"rx{p}.{c}"):
                    yield
                assert slot[(p, c, k)] == (j, h), (p, c, k, slot[(p, c, k)], (j, h))
                v[k] += 1
                B[(p, "full", k)].arrive()
                yield

    actors = []
    slow = set()
    for p in range(P):
        actors.append(mma(p))
        if p == slow_pair:
            slow.add(actors[-1])
        for c in range(2):
            actors.append(recv(p, c))
            if p == slow_pair:
                slow.add(actors[-1])
            for hh in range(2):
                actors.append(epi(p, c, hh))
                if p == slow_pair:
                    slow.add(actors[-1])
    live = list(actors)
    steps = 0
    while live or inflight:
        steps += 1
        assert steps < 2_000_000, "deadlock"
        if inflight and rnd.random() < 0.3:
            q, c, k, content = inflight.pop(rnd.randrange(len(inflight)))
            write(q, c, k, content)
            B[(q, c, "rx", k)].complete_tx(1)
            continue
        if not live:
            continue
        a = rnd.choice(live)
        if slow_pair is not None and a in slow and rnd.random() < 0.97:
            continue   # one pair's actors run rarely: the other pairs get as far ahead as the protocol allows
        try:
            next(a)
        except StopIteration:
            live.remove(a)
    return steps


@pytest.mark.parametrize("S", [2, 3, 4])
@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_protocol_holds(P, S):
    for nt in range(1, 14):
        for seed in range(20):
            run(P, S, nt, 16, seed * 1000 + nt)
    # one pair's actors starved, so that the others run as far ahead as the barriers let them
    for nt in (16, 30):
        for seed in range(3):
            for slow in range(P):
                run(P, S, nt, 16, seed * 7919 + nt, slow_pair=slow)


def test_send_without_waiting_for_the_peer_is_caught():
    with pytest.raises(AssertionError):
        for nt in range(3, 10):
            for seed in range(20):
                run(4, 4, nt, 16, seed * 1000 + nt, mistake="no wait for the other pairs")


def test_release_to_wrong_writer_is_caught():
    with pytest.raises(AssertionError):
        for nt in range(3, 10):
            for seed in range(20):
                run(4, 4, nt, 16, seed * 1000 + nt, mistake="release to the next block's owner")
