"""The decode chain's ring protocol, simulated on the CPU: producers issue a
block's items into S ring slots (item i in slot i % S) behind mbarrier-style
"full" and "empty" phases tested by parity, under a cap of F copies in
flight; consumer warps take their rows' items in order behind a layer
barrier. The rules the kernel follows -- S and F multiples of the producer
count P (each slot only ever holds one producer's items), the in-flight
cursor advanced on every item, and per-slot item tags that consumers wait
for before the parity -- must never let a slot be refilled while its item is
in use, never hand a consumer another item, and never deadlock, under
weighted-random schedules. Without the ownership rule or without the tags,
the same schedules do find violations (the checks have teeth)."""
import random

import pytest


class _Bar:
    """An mbarrier's phase bookkeeping: expected arrivals and a byte count;
    a parity test is true when the phase of that parity has completed
    (which cannot tell it from the phase two earlier)."""

    def __init__(self):
        self.pending, self.phase, self.tx = 1, 0, 0

    def done(self, parity):
        return (self.phase & 1) != parity

    def arrive(self, tx=0):
        self.tx += tx
        self.pending -= 1
        self._settle()

    def land(self, tx):
        self.tx -= tx
        assert self.tx >= 0, "byte count below zero"
        self._settle()

    def _settle(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = 1


def _run(S, P, F, PL, layers, CW, SEG, seed, tags=True):
    rnd = random.Random(seed)
    total = PL * layers
    full = [_Bar() for _ in range(S)]
    empty = [_Bar() for _ in range(S)]
    held = [None] * S          # the item a slot holds, issued and not yet consumed
    tag = [-1] * S             # the kernel's per-slot word: the last item issued into the slot
    inflight = []
    prod = []
    for g in range(P):
        su, phu = g - F, 0
        while su < 0:
            su += S
            phu ^= 1
        prod.append(dict(i=g, s=g % S, ph=(g // S) & 1, su=su, phu=phu))
    rows = PL // SEG
    cons = [dict(seq=[l * PL + j * SEG + h for l in range(layers) for j in range(w, rows, CW) for h in range(SEG)],
                 k=0) for w in range(CW)]
    done_layer = [0] * layers
    consumed = 0
    actors = [("p", g) for g in range(P)] + [("c", w) for w in range(CW)] + [("land", 0)]
    weights = [rnd.choice([0.01, 0.1, 1, 10]) for _ in actors]

    def ready(kind, a):
        if kind == "p":
            st = prod[a]
            if st["i"] >= total:
                return False
            if st["i"] >= S and not empty[st["s"]].done(st["ph"] ^ 1):
                return False
            if F < S and st["i"] >= F:
                assert st["su"] == (st["i"] - F) % S, "in-flight cursor"
                if not full[st["su"]].done(st["phu"]):
                    return False
            return True
        if kind == "land":
            return bool(inflight)
        st = cons[a]
        if st["k"] >= len(st["seq"]):
            return False
        it = st["seq"][st["k"]]
        l = it // PL
        if l > 0 and done_layer[l - 1] < PL:
            return False
        s = it % S
        if tags and S < PL and tag[s] != it:
            return False
        return full[s].done((it // S) & 1)

    while consumed < total:
        en = [(x, w) for x, w in zip(actors, weights) if ready(*x)]
        assert en, f"deadlock with {consumed} of {total} items consumed"
        kind, a = rnd.choices([x for x, _ in en], [w for _, w in en])[0]
        if kind == "p":
            st = prod[a]
            i, s = st["i"], st["s"]
            assert s == i % S
            assert held[s] is None, f"slot {s} refilled with item {i} while item {held[s]} is in use"
            held[s] = i
            tag[s] = i
            full[s].arrive(tx=1)
            inflight.append((i, s))
            st["i"] += P
            st["s"] += P
            while st["s"] >= S:
                st["s"] -= S
                st["ph"] ^= 1
            st["su"] += P
            while st["su"] >= S:
                st["su"] -= S
                st["phu"] ^= 1
        elif kind == "land":
            _, s = inflight.pop(rnd.randrange(len(inflight)))
            full[s].land(1)
        else:
            st = cons[a]
            it = st["seq"][st["k"]]
            s = it % S
            assert held[s] == it, f"a consumer waiting for item {it} was handed slot {s} holding {held[s]}"
            held[s] = None
            st["k"] += 1
            done_layer[it // PL] += 1
            consumed += 1
            empty[s].arrive()


def _caps(S, P):
    return sorted({min(S, -(-f // P) * P) for f in (1, S // 2 or 1, S)})


@pytest.mark.parametrize("S,P", [(54, 3), (33, 3), (32, 2), (9, 3), (2, 2), (1, 1)])
@pytest.mark.parametrize("PL,CW,SEG", [(54, 16, 2), (82, 16, 2), (27, 8, 1), (4, 16, 2)])
def test_ring_protocol_holds(S, P, PL, CW, SEG):
    for F in _caps(S, P):
        for seed in range(12):
            _run(S, P, F, PL, 2, CW, SEG, seed)


def test_protocol_checks_find_the_faults_they_guard_against():
    def violations(S, P, tags):
        found = 0
        for PL, CW, SEG in [(54, 16, 2), (82, 16, 2)]:
            for seed in range(40):
                try:
                    _run(S, P, S, PL, 3, CW, SEG, seed, tags=tags)
                except AssertionError:
                    found += 1
        return found
    assert violations(35, 4, tags=True) > 0    # slots shared by several producers
    assert violations(30, 3, tags=False) > 0   # a ring shorter than a layer, no tags
    assert violations(30, 3, tags=True) == 0
