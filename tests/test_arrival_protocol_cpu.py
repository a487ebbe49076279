"""The split-KV kernel's per-unit arrival counter, simulated on the CPU.

Each CTA that holds part of a unit's tiles writes its partial and then
counts one arrival on the unit's 64-bit counter word, (epoch << 16) | count.
The arrival adds one; when the word already carries this call's tag, the
count it returns is exact in that one atomic. Otherwise (another call's tag,
or whatever bytes the workspace held) it retags the word with compare-and-
swap: it restarts the count at one, or counts itself once another arrival
has retagged. The arrival whose count equals the unit's contributors merges
the unit and sets the word back to (epoch << 16) | 0.

The simulation interleaves the contributors' atomic steps at random, from
every kind of starting word, and checks that exactly one arrival sees the
full count (it is the last one to start, so every partial was written
before it), that every arrival count 1..n is handed out once, and that the
word ends at (epoch << 16) | 0, which the next call, or a replay with the
same tag, counts from; also with the kernel's counter warps retagging the
word at the same time. A negative control shows that a plain add, without
the retag, miscounts on a word left by another call.
"""
import random

import pytest

MASK64 = (1 << 64) - 1


def _arrival(epoch, mem, log, name):
    """One CTA's arrival as a generator of atomic steps on mem[0]; yields
    between steps. Appends (name, count) to log when it has its count."""
    old = mem[0]
    mem[0] = (old + 1) & MASK64                  # atomicAdd
    yield
    if old >> 16 == epoch:
        log.append((name, (old & 0xFFFF) + 1))
        return
    cur = (old + 1) & MASK64
    for _ in range(1000):
        nxt = cur + 1 if cur >> 16 == epoch else (epoch << 16) | 1
        prev = mem[0]                            # atomicCAS(ctr, cur, nxt)
        if prev == cur:
            mem[0] = nxt
        yield
        if prev == cur:
            log.append((name, nxt & 0xFFFF))
            return
        cur = prev
    raise AssertionError("CAS loop did not end")


def _retagger(epoch, mem, log, name):
    """The counter warp's retag: not an arrival. It swaps a word with another
    tag for (epoch << 16) | 0 and leaves a word with this call's tag alone."""
    cur = mem[0]
    yield
    for _ in range(64):
        if cur >> 16 == epoch:
            return
        prev = mem[0]                            # atomicCAS(ctr, cur, epoch << 16)
        if prev == cur:
            mem[0] = epoch << 16
        yield
        if prev == cur:
            return
        cur = prev


def _plain_add(epoch, mem, log, name):
    old = mem[0]
    mem[0] = (old + 1) & MASK64
    yield
    log.append((name, (old & 0xFFFF) + 1))


def simulate(seed, n, start, epoch, arrival=_arrival, retaggers=0):
    rnd = random.Random(seed)
    mem = [start]
    log = []
    agents = {i: arrival(epoch, mem, log, i) for i in range(n)}
    for k in range(retaggers):
        agents[n + k] = _retagger(epoch, mem, log, n + k)
    waiting = list(agents)                       # not started yet
    running = []
    while waiting or running:
        pick = rnd.randrange(len(waiting) + len(running))
        if pick < len(waiting):
            a = waiting.pop(pick)
            running.append(a)
        else:
            a = running[pick - len(waiting)]
        try:
            next(agents[a])
        except StopIteration:
            running.remove(a)
            if log and log[-1][0] == a and log[-1][1] == n:
                mem[0] = epoch << 16             # the last arrival resets the word
    return mem[0], log


STARTS = {
    "zero": 0,
    "other call, reset": 0x1234 << 16,
    "other call, part-way": (0x1234 << 16) | 3,
    "same tag, reset (graph replay)": 0xBEEF << 16,
    "canary bytes": 0xA5A5A5A5A5A5A5A5,
    "all ones": MASK64,
    "count field about to carry": (0x77 << 16) | 0xFFFF,
}


@pytest.mark.parametrize("start", list(STARTS), ids=list(STARTS))
@pytest.mark.parametrize("n", [1, 2, 3, 19])
def test_every_count_once_and_the_word_left_clean(start, n):
    epoch = 0xBEEF
    for seed in range(200):
        end, log = simulate(seed, n, STARTS[start], epoch)
        counts = sorted(c for _, c in log)
        assert counts == list(range(1, n + 1)), (seed, log)
        assert end == epoch << 16, hex(end)
        # the next call (another tag) and a replay (same tag) count correctly
        for nxt in (epoch, epoch + 1):
            end2, log2 = simulate(seed + 7, n, end, nxt)
            assert sorted(c for _, c in log2) == list(range(1, n + 1))
            assert end2 == nxt << 16


@pytest.mark.parametrize("start", list(STARTS), ids=list(STARTS))
@pytest.mark.parametrize("n", [2, 3, 19])
def test_early_retag_races_with_arrivals(start, n):
    """The counter warp retags the word while arrivals may already be adding
    (a CTA with a one-tile share can reach its segment's end first). Each
    contributing CTA's counter warp retags, in any interleaving with the
    adds and swaps: every count 1..n is still handed out once, and the
    word ends reset."""
    epoch = 0xBEEF
    for seed in range(200):
        end, log = simulate(seed, n, STARTS[start], epoch, retaggers=min(n, 4))
        assert sorted(c for _, c in log) == list(range(1, n + 1)), (seed, log)
        assert end == epoch << 16, hex(end)


def test_plain_add_miscounts_on_another_calls_word():
    """Negative control: counting with the add alone trusts whatever the word
    holds. A word left part-way by another call gives the wrong counts (so
    some unit would merge before its partials were written, or never)."""
    bad = 0
    for seed in range(50):
        _, log = simulate(seed, 2, STARTS["other call, part-way"], 0xBEEF, arrival=_plain_add)
        if sorted(c for _, c in log) != [1, 2]:
            bad += 1
    assert bad == 50
