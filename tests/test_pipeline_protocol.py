"""Host model of the prefill kernel's mbarrier protocol for the 16-bit ring (roles: TMA producer,
MMA thread, the two softmax warpgroups), run under random interleavings.

An mbarrier wait tests only the parity of a phase, so a waiter that the arriving side does not
wait for in turn can fall two phases behind (it then waits for a phase that already passed) or
test a phase two ahead (and pass at once).  The model records, for every wait, the phase it
means; a wait that passes on parity before that phase completed is an alias, and a state where
no role can move is a deadlock.  The protocol as built (tile 0's softmax waits for ring step
j+1 before it signals P_0(j), so the MMA thread skips that wait) must show neither, for rings
of 2 and 4 stages and work tiles whose second query tile is empty, equal, or one block longer.
A variant in which tile 1's softmax would take its S from the step's `released` commit, which
the MMA thread never waits on in work tiles without tile 1, must be caught.  The protocol with
P signalled in two halves (p_half, then p_full) is checked the same way.
"""
import random

import pytest


class _Bar:
    def __init__(self, name):
        self.name, self.phase = name, 0

    def arrive(self):  # every barrier of the model completes a phase per arrival (count 1)
        self.phase += 1


def _run(units, stages, seed, tile1_on_released=False, p_half=False):
    rnd = random.Random(seed)
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Bar(name))

    def producer():
        g, qn = 0, [0, 0]
        for nt in units:
            nb = max(nt)
            if nb == 0:
                continue
            for t in range(2):
                if nt[t] == 0:
                    continue
                if qn[t] > 0:
                    yield ("wait", bar(f"q_empty{t}"), qn[t] - 1)
                yield ("do", bar(f"q_full{t}"))
                qn[t] += 1
            for _ in range(nb + 1):
                s, r = g % stages, g // stages
                if r > 0:
                    yield ("wait", bar(f"released{s}"), r - 1)
                yield ("do", bar(f"in_full{s}"))
                g += 1

    def mma():
        g, qn, pn = 0, [0, 0], [0, 0]
        for nt in units:
            nb = max(nt)
            if nb == 0:
                continue
            for t in range(2):
                if nt[t] > 0:
                    yield ("wait", bar(f"q_full{t}"), qn[t])
            for j in range(nb + 1):
                s, r = g % stages, g // stages
                if not (j >= 1 and j - 1 < nt[0]):
                    yield ("wait", bar(f"in_full{s}"), r)
                for t in range(2):
                    if j >= 1 and j - 1 < nt[t]:
                        if j == 1 and qn[t] > 0:
                            yield ("wait", bar(f"o_empty{t}"), qn[t] - 1)
                        if p_half:  # the first half of P, for the first half of the P.V MMAs
                            yield ("wait", bar(f"p_half{t}"), pn[t])
                        yield ("wait", bar(f"p_full{t}"), pn[t])
                        pn[t] += 1
                        if j == nt[t]:
                            yield ("do", bar(f"o_full{t}"))
                    if j < nt[t]:
                        if t == 0 or not tile1_on_released:
                            yield ("do", bar(f"s_full{t}"))
                        if j == nt[t] - 1:
                            yield ("do", bar(f"q_empty{t}"))
                yield ("do", bar(f"released{s}"))
                g += 1
            for t in range(2):
                if nt[t] > 0:
                    qn[t] += 1

    def softmax(t):
        sn = on = gbase = 0
        for nt in units:
            nb = max(nt)
            g0 = gbase
            gbase += nb + 1 if nb > 0 else 0
            if nt[t] == 0:
                continue
            for j in range(nt[t]):
                if t == 1 and tile1_on_released:
                    G = g0 + j
                    yield ("wait", bar(f"released{G % stages}"), G // stages)
                else:
                    yield ("wait", bar(f"s_full{t}"), sn)
                if t == 0:
                    G = g0 + j + 1
                    yield ("wait", bar(f"in_full{G % stages}"), G // stages)
                if p_half:  # after the covering wait: the first half of P.V reads V(j) already
                    yield ("do", bar(f"p_half{t}"))
                yield ("do", bar(f"p_full{t}"))
                sn += 1
            yield ("wait", bar(f"o_full{t}"), on)
            on += 1
            yield ("do", bar(f"o_empty{t}"))

    roles = {"producer": producer(), "mma": mma(), "softmax0": softmax(0), "softmax1": softmax(1)}
    pending = {}
    for name, gen in roles.items():
        op = next(gen, None)
        if op is not None:
            pending[name] = op
    while pending:
        ready = []
        for name, op in pending.items():
            if op[0] == "do":
                ready.append(name)
                continue
            b, index = op[1], op[2]
            if (b.phase & 1) != (index & 1):  # what the hardware tests
                if b.phase < index + 1:
                    return f"alias: {name} passed {b.name} phase {index} at phase {b.phase}"
                ready.append(name)
        if not ready:
            return "deadlock: " + ", ".join(f"{n} on {op[1].name}" for n, op in pending.items())
        name = rnd.choice(ready)
        op = pending[name]
        if op[0] == "do":
            op[1].arrive()
        nxt = next(roles[name], None)
        if nxt is None:
            del pending[name]
        else:
            pending[name] = nxt
    return None


def _random_units(rnd):
    units = []
    for _ in range(rnd.randint(1, 8)):
        n, kind = rnd.randint(1, 5), rnd.random()
        if kind < 0.3:
            units.append((n, 0))       # second query tile past the rows
        elif kind < 0.6:
            units.append((n, n))       # non-causal
        elif kind < 0.9:
            units.append((n, n + 1))   # causal: the second tile sees one more block
        else:
            units.append((0, 0))       # empty packed-sequence unit
    return units


@pytest.mark.parametrize("p_half", [False, True])
@pytest.mark.parametrize("stages", [2, 4])
def test_protocol_has_no_alias_or_deadlock(stages, p_half):
    # p_half: the softmax also signals the first half of P (keys 0-63) before the second, and the
    # MMA thread issues the first half of the P.V MMAs on it
    for seed in range(1500):
        units = _random_units(random.Random(seed))
        assert _run(units, stages, seed, p_half=p_half) is None, units


def test_model_catches_a_tile_waiting_on_a_barrier_nobody_waits_for():
    failures = [_run(_random_units(random.Random(s)), 2, s, tile1_on_released=True) for s in range(300)]
    assert sum(f is not None for f in failures) > 50


def _run_e4m3(units, stages, seed, t0_covers=True, p_half=False):
    """The e4m3 ring: K(j) and raw V(j) load one step ahead of P.V(j); two converter warps turn
    raw V into f16 (v_ready), free the raw buffer themselves (vraw_free) and write the converted
    buffer only after the P.V that last read it (v_free).  With t0_covers, tile 0's softmax waits
    for V(j-1) converted and K(j) landed before it signals P_0(j-1), and the MMA thread skips both
    waits at that step."""
    rnd = random.Random(seed)
    bars = {}

    def bar(name):
        return bars.setdefault(name, _Bar(name))

    def producer():
        g, qn = 0, [0, 0]
        for nt in units:
            nb = max(nt)
            if nb == 0:
                continue
            for t in range(2):
                if nt[t] == 0:
                    continue
                if qn[t] > 0:
                    yield ("wait", bar(f"q_empty{t}"), qn[t] - 1)
                yield ("do", bar(f"q_full{t}"))
                qn[t] += 1
            for _ in range(nb):
                s, r = g % stages, g // stages
                if r > 0:
                    yield ("wait", bar(f"released{s}"), r - 1)
                yield ("do", bar(f"in_full{s}"))
                if r > 0:
                    yield ("wait", bar(f"vraw_free{s}"), r - 1)
                yield ("do", bar(f"v_full{s}"))
                g += 1

    def converter():
        g = 0
        for nt in units:
            for _ in range(max(nt)):
                s, r = g % stages, g // stages
                yield ("wait", bar(f"v_full{s}"), r)
                if r > 0:
                    yield ("wait", bar(f"v_free{s}"), r - 1)
                yield ("do", bar(f"v_ready{s}"))
                yield ("do", bar(f"vraw_free{s}"))
                g += 1

    def mma():
        g, qn, pn = 0, [0, 0], [0, 0]
        for nt in units:
            nb = max(nt)
            if nb == 0:
                continue
            for t in range(2):
                if nt[t] > 0:
                    yield ("wait", bar(f"q_full{t}"), qn[t])
            for j in range(nb + 1):
                gk, gv = g + j, g + j - 1
                covered = t0_covers and j >= 1 and j - 1 < nt[0]
                if j >= 1 and not covered:
                    yield ("wait", bar(f"v_ready{gv % stages}"), gv // stages)
                k_ready = covered
                for t in range(2):
                    if j >= 1 and j - 1 < nt[t]:
                        if j == 1 and qn[t] > 0:
                            yield ("wait", bar(f"o_empty{t}"), qn[t] - 1)
                        if p_half:  # the first half of P, for the first half of the P.V MMAs
                            yield ("wait", bar(f"p_half{t}"), pn[t])
                        yield ("wait", bar(f"p_full{t}"), pn[t])
                        pn[t] += 1
                        if j == nt[t]:
                            yield ("do", bar(f"o_full{t}"))
                    if t == 1 and j >= 1:
                        yield ("do", bar(f"v_free{gv % stages}"))
                    if j < nt[t]:
                        if not k_ready:
                            yield ("wait", bar(f"in_full{gk % stages}"), gk // stages)
                            k_ready = True
                        yield ("do", bar(f"s_full{t}"))
                        if j == nt[t] - 1:
                            yield ("do", bar(f"q_empty{t}"))
                if j < nb:
                    yield ("do", bar(f"released{gk % stages}"))
            g += nb
            for t in range(2):
                if nt[t] > 0:
                    qn[t] += 1

    def softmax(t):
        sn = on = gbase = 0
        for nt in units:
            nb = max(nt)
            g0 = gbase
            gbase += nb
            if nt[t] == 0:
                continue
            for j in range(nt[t]):
                yield ("wait", bar(f"s_full{t}"), sn)
                if t == 0 and t0_covers:
                    G = g0 + j
                    yield ("wait", bar(f"v_ready{G % stages}"), G // stages)
                    if j + 1 < nb:
                        yield ("wait", bar(f"in_full{(G + 1) % stages}"), (G + 1) // stages)
                if p_half:
                    yield ("do", bar(f"p_half{t}"))
                yield ("do", bar(f"p_full{t}"))
                sn += 1
            yield ("wait", bar(f"o_full{t}"), on)
            on += 1
            yield ("do", bar(f"o_empty{t}"))

    roles = {"producer": producer(), "converter": converter(), "mma": mma(), "softmax0": softmax(0),
             "softmax1": softmax(1)}
    pending = {}
    for name, gen in roles.items():
        op = next(gen, None)
        if op is not None:
            pending[name] = op
    while pending:
        ready = []
        for name, op in pending.items():
            if op[0] == "do":
                ready.append(name)
                continue
            b, index = op[1], op[2]
            if (b.phase & 1) != (index & 1):
                if b.phase < index + 1:
                    return f"alias: {name} passed {b.name} phase {index} at phase {b.phase}"
                ready.append(name)
        if not ready:
            return "deadlock: " + ", ".join(f"{n} on {op[1].name}" for n, op in pending.items())
        name = rnd.choice(ready)
        op = pending[name]
        if op[0] == "do":
            op[1].arrive()
        nxt = next(roles[name], None)
        if nxt is None:
            del pending[name]
        else:
            pending[name] = nxt
    return None


@pytest.mark.parametrize("p_half", [False, True])
@pytest.mark.parametrize("t0_covers", [False, True])
@pytest.mark.parametrize("stages", [2, 4])
def test_e4m3_protocol_has_no_alias_or_deadlock(stages, t0_covers, p_half):
    for seed in range(1000):
        units = _random_units(random.Random(seed))
        assert _run_e4m3(units, stages, seed, t0_covers=t0_covers, p_half=p_half) is None, units
