"""A host-side model of the hand-offs of the main backward kernel when it
stores dS with two query tiles in flight (csrc/bwd_tc.cu, the MMA, softmax,
producer and epilogue roles of the pipelined schedule).

Each role is a generator that waits on mbarrier phases by parity, as the
kernel does. TMA loads land after random delays, and tensor-core operations
complete in issue order at random times. Over many random interleavings the
model checks two things:
- no wait can block forever (a parity wait that sees a phase two behind would);
- every shared tile is overwritten only after the tensor-core operations that
  read it have completed (P tiles by dV, the dS tile by dK).

A variant with a planted mistake must fail, so the checks are known to bite.
"""
import random

import pytest


class _Bar:
    """An mbarrier: `count` arrivals complete a phase; a parity wait passes
    once the phase of that parity has completed."""

    def __init__(self, count=1):
        self.count, self.pending, self.ph = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.ph += 1
            self.pending = self.count

    def done(self, parity):
        return (self.ph & 1) != parity


class _Hazard(AssertionError):
    pass


def _run(seed, units, dos, planted=None):
    rnd = random.Random(seed)
    names = ["KV_FULL", "KV_EMPTY", "Q_FULL0", "Q_FULL1", "Q_EMPTY0", "Q_EMPTY1", "DO_FULL0", "DO_FULL1",
             "DO_EMPTY0", "DO_EMPTY1", "S_FULL0", "S_FULL1", "DP_FULL0", "DP_FULL1", "P_FULL", "DS_FULL",
             "MMA_DONE0", "MMA_DONE1", "ACC_FULL", "ACC_FREE"]
    bars = {n: _Bar() for n in names}
    events = []            # (time, callback): TMA completions
    pipe = []              # in-order tensor-core queue: ("op", id) or ("commit", barrier)
    completed = set()      # tensor-core operation ids completed
    ops = {}               # (kind, tile) -> operation id
    clock = [0]

    def tma(bar):
        events.append((clock[0] + rnd.randint(1, 30), lambda: bars[bar].arrive()))

    def mma(kind, t):
        ops[(kind, t)] = len(ops)
        pipe.append(("op", ops[(kind, t)]))

    def commit(bar):
        pipe.append(("commit", bar))

    def wait(bar, parity):
        while not bars[bar].done(parity):
            yield (bar, parity)

    def require_done(kind, t):
        if (kind, t) in ops and ops[(kind, t)] not in completed:
            raise _Hazard(f"shared tile overwritten while {kind}({t}) may still read it")

    def producer():
        t = 0
        for ne, n in enumerate(units):
            if ne > 0:
                yield from wait("KV_EMPTY", (ne - 1) & 1)
            tma("KV_FULL")
            for _ in range(n):
                s, d = t & 1, t % dos
                if t >= 2:
                    yield from wait(f"Q_EMPTY{s}", ((t >> 1) - 1) & 1)
                tma(f"Q_FULL{s}")
                if t >= dos:
                    yield from wait(f"DO_EMPTY{d}", ((t // dos) - 1) & 1)
                tma(f"DO_FULL{d}")
                t += 1

    def mma_role():
        def issue_s(t):
            yield from wait(f"Q_FULL{t & 1}", (t >> 1) & 1)
            mma("S", t)
            commit(f"S_FULL{t & 1}")

        def issue_dp(t):
            yield from wait(f"DO_FULL{t % dos}", (t // dos) & 1)
            mma("dP", t)
            commit(f"DP_FULL{t & 1}")

        t = 0
        for ne, n in enumerate(units):
            yield from wait("KV_FULL", ne & 1)
            if ne > 0:
                yield from wait("ACC_FREE", (ne - 1) & 1)
            yield from issue_s(t)
            yield from issue_dp(t)
            for i in range(n):
                s, d, more = t & 1, t % dos, i + 1 < n
                yield from wait("P_FULL", t & 1)
                mma("dV", t)
                commit(f"DO_EMPTY{d}")
                if more:
                    yield from issue_s(t + 1)
                yield from wait("DS_FULL", t & 1)
                mma("dK", t)
                commit(f"Q_EMPTY{s}")
                commit(f"MMA_DONE{s}")
                if more:
                    yield from issue_dp(t + 1)
                t += 1
            commit("ACC_FULL")
            commit("KV_EMPTY")

    def softmax():
        t = 0
        for n in units:
            for _ in range(n):
                s = t & 1
                yield from wait(f"Q_FULL{s}", (t >> 1) & 1)
                yield from wait(f"S_FULL{s}", (t >> 1) & 1)
                if t >= 2:
                    if planted == "one_done_barrier":
                        yield from wait("MMA_DONE0", (t - 2) & 1)
                    else:
                        yield from wait(f"MMA_DONE{s}", ((t >> 1) - 1) & 1)
                require_done("dV", t - 2)          # P tile t & 1
                bars["P_FULL"].arrive()
                yield from wait(f"DP_FULL{s}", (t >> 1) & 1)
                require_done("dK", t - 1)          # the one dS tile
                bars["DS_FULL"].arrive()
                t += 1

    def epilogue():
        for ne, _ in enumerate(units):
            yield from wait("ACC_FULL", ne & 1)
            bars["ACC_FREE"].arrive()

    if planted == "one_done_barrier":
        # every dK commits to one barrier that the softmax waits on two tiles back
        old_commit = commit

        def commit(bar):  # noqa: F811
            old_commit("MMA_DONE0" if bar.startswith("MMA_DONE") else bar)

    if planted == "dp_before_dk":
        # dP(t+1) issued before dK(t): the dS tile may be overwritten while dK(t) reads it
        def mma_role():  # noqa: F811
            def issue_s(t):
                yield from wait(f"Q_FULL{t & 1}", (t >> 1) & 1)
                mma("S", t)
                commit(f"S_FULL{t & 1}")

            def issue_dp(t):
                yield from wait(f"DO_FULL{t % dos}", (t // dos) & 1)
                mma("dP", t)
                commit(f"DP_FULL{t & 1}")

            t = 0
            for ne, n in enumerate(units):
                yield from wait("KV_FULL", ne & 1)
                if ne > 0:
                    yield from wait("ACC_FREE", (ne - 1) & 1)
                yield from issue_s(t)
                yield from issue_dp(t)
                for i in range(n):
                    s, d, more = t & 1, t % dos, i + 1 < n
                    yield from wait("P_FULL", t & 1)
                    mma("dV", t)
                    commit(f"DO_EMPTY{d}")
                    if more:
                        yield from issue_s(t + 1)
                        yield from issue_dp(t + 1)
                    yield from wait("DS_FULL", t & 1)
                    mma("dK", t)
                    commit(f"Q_EMPTY{s}")
                    commit(f"MMA_DONE{s}")
                    t += 1
                commit("ACC_FULL")
                commit("KV_EMPTY")

    agents = {"producer": producer(), "mma": mma_role(), "softmax": softmax(), "epilogue": epilogue()}
    blocked = {k: None for k in agents}
    for _ in range(400000):
        if not agents:
            return "ok"
        runnable = [k for k in agents if blocked[k] is None or bars[blocked[k][0]].done(blocked[k][1])]
        choices = runnable + (["tma"] if events else []) + (["pipe"] if pipe else [])
        if not choices:
            return f"deadlock: {blocked}"
        c = rnd.choice(choices)
        clock[0] += 1
        if c == "tma":
            events.sort(key=lambda e: e[0])
            events.pop(0)[1]()
        elif c == "pipe":
            kind, x = pipe.pop(0)
            if kind == "op":
                completed.add(x)
            else:
                bars[x].arrive()
        else:
            try:
                blocked[c] = next(agents[c])
            except StopIteration:
                del agents[c], blocked[c]
            except _Hazard as e:
                return f"hazard: {e}"
    return "did not finish"


def _cases(n):
    rnd = random.Random(1234)
    for seed in range(n):
        units = [rnd.randint(1, 6) for _ in range(rnd.randint(1, 5))]
        for dos in (1, 2):
            yield seed, units, dos


def test_pipelined_handoffs_never_block_or_overwrite_in_use_tiles():
    bad = [(seed, units, dos, r) for seed, units, dos in _cases(400) if (r := _run(seed, units, dos)) != "ok"]
    assert not bad, bad[:3]


@pytest.mark.parametrize("planted", ["one_done_barrier", "dp_before_dk"])
def test_the_model_catches_a_planted_mistake(planted):
    results = [_run(seed, units, dos, planted) for seed, units, dos in _cases(200)]
    assert any(r != "ok" for r in results), planted
