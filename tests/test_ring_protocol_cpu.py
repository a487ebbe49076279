"""The split-KV kernel's shared-memory ring, simulated on the CPU.

One producer issues the tiles of a CTA's share in order into a ring of
`stages` stages; every stage has a "full" mbarrier (one arrival plus the copy's
bytes) and an "empty" mbarrier (one arrival per warp that reads the tile).
With bf16 caches the four consumer warps of each 16-row tile form two groups
that take alternate tiles of each segment, and the warps of a row tile meet at
every segment end (the slice merge). A wait on an mbarrier only sees the parity
of the current phase, and the copies of different stages land in any order.

The simulation runs random interleavings of those agents and checks that no
wait passes early (a stage's last completed phase must be exactly the one
before the awaited tile's), that no copy lands while a warp reads the stage,
that no mbarrier gets more arrivals than its count, and that every tile is
read. The ring depths are the ones the library's plan reports; an odd depth
is shown to break the protocol (a warp would see the phase two loads back,
whose parity equals the awaited one, while its stage's previous copy is still
in flight).
"""
import random

import pytest

import grouped_query_decode_gb300 as gq


class _Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase, self.tx = count, count, 0, 0

    def arrive(self):
        self.pending -= 1
        if self.pending < 0:
            raise AssertionError("more arrivals than the barrier's count")
        self._complete()

    def expect(self, n):
        self.tx += n

    def land(self, n):
        self.tx -= n
        if self.tx < 0:
            raise AssertionError("more bytes than expected")
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def passed(self, parity):
        # mbarrier.try_wait.parity: true once the phase of that parity is over
        return (self.phase & 1) != parity


def simulate(seed, row_tiles, stages, segments, groups=2):
    rnd = random.Random(seed)
    readers = (4 // groups) * row_tiles
    full = [_Bar(1) for _ in range(stages)]
    empty = [_Bar(readers) for _ in range(stages)]
    held = [None] * stages                  # tile whose bytes have landed in the stage
    reading = [set() for _ in range(stages)]
    inflight = []                           # (stage, tile)
    starts, acc = [], 0
    for n in segments:
        starts.append(acc)
        acc += n
    total = acc
    warps = []
    for mt in range(row_tiles):
        for sl in range(4):
            g = sl >> 1 if groups == 2 else 0
            plan = []
            for si, n in enumerate(segments):
                plan += [("tile", si, starts[si] + i) for i in range(g, n, groups)]
                plan.append(("merge", si, None))
            warps.append({"mt": mt, "plan": plan, "pc": 0, "state": "ready"})
    met = {}
    issued = 0
    reads = [0] * total
    while True:
        choices = (["producer"] if issued < total else []) + (["copy"] if inflight else [])
        choices += [w for w in range(len(warps)) if warps[w]["pc"] < len(warps[w]["plan"])]
        if not choices:
            break
        c = rnd.choice(choices)
        if c == "producer":
            t, s = issued, issued % stages
            if empty[s].passed(((t // stages) & 1) ^ 1):
                assert empty[s].phase == t // stages, "producer's wait passed early"
                assert not reading[s], "a copy was issued into a stage being read"
                full[s].expect(1)
                full[s].arrive()
                inflight.append((s, t))
                issued += 1
        elif c == "copy":
            s, t = inflight.pop(rnd.randrange(len(inflight)))   # copies land in any order
            held[s] = t
            full[s].land(1)
        else:
            w = warps[c]
            op, si, t = w["plan"][w["pc"]]
            if op == "tile":
                s = t % stages
                if w["state"] == "ready":
                    if full[s].passed((t // stages) & 1):
                        assert full[s].phase == t // stages + 1, f"wait for tile {t} passed early"
                        assert held[s] == t
                        reading[s].add(c)
                        w["state"] = "reading"
                else:
                    assert held[s] == t, "a stage changed under its reader"
                    reading[s].discard(c)
                    reads[t] += 1
                    empty[s].arrive()
                    w["state"] = "ready"
                    w["pc"] += 1
            else:
                key = (w["mt"], si)
                if w["state"] == "ready":
                    met[key] = met.get(key, 0) + 1
                    w["state"] = "merging"
                elif met[key] == 4:
                    w["state"] = "ready"
                    w["pc"] += 1
    assert reads == [readers] * total


SEGMENTS = [[64], [300], [3, 1, 1, 1, 2, 7, 1], [1, 1, 5, 2, 9, 1, 1, 1, 3], [2, 1, 1, 1, 1, 1, 1, 6], [1], [2]]


@pytest.mark.parametrize("D,row_tiles", [(128, 1), (128, 2), (64, 1), (64, 2)])
def test_ring_protocol_with_the_plans_depth(D, row_tiles):
    H, G = (16, 1) if row_tiles == 1 else (32, 1)
    plan = gq.gqa_decode_plan(2, 1, H, G, D, 4096, 152)
    assert plan["row_tiles"] == row_tiles
    for segments in SEGMENTS:
        for seed in range(60):
            simulate(seed, row_tiles, plan["stages"], segments)


def test_an_odd_ring_lets_a_wait_pass_early():
    """The negative control: five stages with two groups. Some interleaving
    has a warp wait on tile t while tile t - 5 (the other group's) is still
    in flight; the stage then shows the phase of tile t - 10, whose parity
    equals tile t's, and the wait passes before tile t has landed."""
    failures = 0
    for seed in range(200):
        try:
            simulate(seed, 1, 5, [64])
        except AssertionError as e:
            assert "passed early" in str(e) or "under its reader" in str(e), e
            failures += 1
    assert failures > 0


def test_one_group_is_safe_at_any_depth():
    """Every warp reading every tile (one group) keeps any depth safe: the
    warp has read the stage's previous tile itself."""
    for stages in (3, 4, 5):
        for seed in range(60):
            simulate(seed, 1, stages, [64], groups=1)
