"""The persistent dense backward's barrier protocol, modelled on the CPU.

One CTA takes several 128-key tiles in turn; every tile has the same n query blocks, so each role
counts blocks g = T n + it across tiles and waits on barrier phases by parity.  Between tiles the
K/V tile is reloaded once the three issuing threads' last products are complete (kvdone, three
commits), the epilogue stages dK in the dS tiles and dV in the dQ staging tile (after the drain's
reductions of the tile have read it: stagefree), and the next tile's first dV and dK products wait
for the P/dS warps' first pfull of that tile, which follows their reads of the accumulators.

This model plays the producer, the three issuing threads with their in-order product queues, the
P/dS warps, the dQ drain, the TMA engine and the asynchronous bulk reads (dQ reductions, dK/dV
tensor stores) in random interleavings, with the kernel's index and parity formulas.  Every
buffer carries the version last written to it and every read checks the version it expects, so a
wait that passes early (or a buffer rewritten while a read is pending) shows up as a wrong
version; a parity wait two or more completions behind the phase it wants is reported as stuck.
Planted mistakes (K/V reloaded before the products are complete, dV staged before the drain's
reductions have read the tile, the next tile's accumulation not ordered after the epilogue's
reads, S of a block issued before dK read the dS^T that the same S columns hold) are caught."""
import random

import pytest


class Fault(Exception):
    pass


STAGES = 3


class Model:
    def __init__(self, n, ntile, rnd, plant=None):
        self.n, self.ntile, self.rnd, self.plant = n, ntile, rnd, plant
        self.arrivals = {}
        self.count = {"qempty": 2, "sfull": 2, "pfull": 1, "dsfree": 2, "kvdone": 3, "kread": 1}
        self.ver = {}        # buffer -> version last written
        self.pending = []    # asynchronous reads in flight: (owner, buffer, expected version)
        self.tma = []        # loads in flight: (buffer, version, barrier)
        self.pipes = {r: [] for r in range(3)}

    # -- barriers ------------------------------------------------------------------------
    def completions(self, bar):
        name = bar[0] if isinstance(bar, tuple) else bar
        return self.arrivals.get(bar, 0) // self.count.get(name, 1)

    def arrive(self, bar):
        self.arrivals[bar] = self.arrivals.get(bar, 0) + 1

    def wait_ok(self, bar, k):
        """Parity wait for completion #k (0-based) of bar."""
        c = self.completions(bar)
        sat = (c & 1) != (k & 1)
        if sat and c < k + 1:
            raise Fault(f"early pass on {bar}: {c} completions, wanted #{k}")
        if not sat and c >= k + 2:
            raise Fault(f"stuck on {bar}: {c} completions, wanted #{k}")
        return sat

    # -- data ------------------------------------------------------------------------------
    def write(self, buf, v):
        self.ver[buf] = v

    def read(self, buf, v, who):
        if self.ver.get(buf) != v:
            raise Fault(f"{who} read {buf} = {self.ver.get(buf)}, expected {v}")


def _programs(m):
    """Each agent is a generator yielding ('wait', bar, k), ('do', fn) or ('until', predicate)."""
    n, ntile = m.n, m.ntile
    qs = lambda g: ("q", g % STAGES)

    def prod():
        for T in range(ntile):
            if T > 0 and m.plant != "kv_early":
                yield ("wait", "kvdone", T - 1)
            yield ("do", lambda T=T: m.tma.append(("kv", T, "kv")))
            for it in range(n):
                g = T * n + it
                if g >= STAGES:
                    yield ("wait", ("qempty", g % STAGES), g // STAGES - 1)
                yield ("do", lambda g=g: m.tma.append((qs(g), g, ("qfull", g % STAGES))))

    def issuer(role):
        pipe = m.pipes[role]

        def first(g, T):
            yield ("wait", ("qfull", g % STAGES), g // STAGES)
            if role == 1 and g >= 1:
                yield ("wait", "dpfree", g - 1)
            # the S buffer also holds dS^T of block g - 2 (d = 128) until dK has read it
            if role == 0 and g >= 2 and m.plant != "kread_skipped":
                yield ("wait", ("kread", g & 1), (g - 2) >> 1)
            buf = ("S", g & 1) if role == 0 else ("dP",)
            ops = [("r", "kv", T), ("r", qs(g), g), ("w", buf, ("S" if role == 0 else "dP", g))]
            if role == 0:
                ops.append(("w", ("SdS", g & 1), ("S", g)))
            yield ("do", lambda: pipe.append(ops + [("a", ("sfull", g & 1))]))

        for T in range(ntile):
            yield ("wait", "kv", T)
            g0 = T * n
            if role < 2:
                yield from first(g0, T)
                for it in range(n):
                    g = g0 + it
                    if it + 1 < n:
                        yield from first(g + 1, T)
                    yield ("wait", ("pfull", g & 1), g >> 1)
                    acc = "dV" if role == 0 else "dK"
                    # dK reads dS^T from the S buffer's free columns (d = 128)
                    src = [("r", ("S", g & 1), ("P", g))] if role == 0 else [("r", ("SdS", g & 1), ("dS", g))]
                    ops = src + [("r", qs(g), g), ("acc", acc, T, it)]
                    if role == 1:
                        ops.append(("a", ("kread", g & 1)))
                        ops.append(("a", ("dsfree", g & 1)))
                    ops.append(("a", ("qempty", g % STAGES)))
                    yield ("do", lambda ops=ops: pipe.append(ops))
            else:
                for it in range(n):
                    g = g0 + it
                    yield ("wait", ("pfull", g & 1), g >> 1)
                    if g >= 1:
                        yield ("wait", "dqfree", g - 1)
                    ops = [("r", "kv", T), ("r", ("dS", g & 1), ("dS", g)), ("w", ("dQt",), g),
                           ("a", ("dsfree", g & 1)), ("a", "dqfull")]
                    yield ("do", lambda ops=ops: pipe.append(ops))
            yield ("do", lambda: pipe.append([("a", "kvdone")]))

    def pds():
        for T in range(ntile):
            for it in range(n):
                g = T * n + it
                yield ("wait", ("sfull", g & 1), g >> 1)
                if g >= 2:
                    yield ("wait", ("dsfree", g & 1), (g - 2) >> 1)

                def work(g=g):
                    m.read(("S", g & 1), ("S", g), "P/dS")
                    m.read(("dP",), ("dP", g), "P/dS")
                    m.arrive("dpfree")
                yield ("do", work)

                def publish(g=g, T=T, it=it):
                    m.read(qs(g), g, "P/dS row terms")
                    m.write(("S", g & 1), ("P", g))
                    m.write(("SdS", g & 1), ("dS", g))
                    m.write(("dS", g & 1), ("dS", g))
                    m.arrive(("pfull", g & 1))
                    if m.plant == "acc_unordered" and it == 0 and T > 0:
                        # planted: the previous tile's accumulator reads come after this pfull
                        def late(T=T):
                            m.read("dK", ("acc", T - 1, n), "epilogue dK")
                            m.read("dV", ("acc", T - 1, n), "epilogue dV")
                        m.late.append(late)
                yield ("do", publish)
            # epilogue of tile T: dK (warps 0-3) once the products are complete, dV (warps 4-7)
            # once the drain's reductions have also read the staging tile
            yield ("wait", "kvdone", T)

            def stage_k(T=T):
                if m.plant != "acc_unordered":
                    m.read("dK", ("acc", T, n), "epilogue dK")
                m.write(("dS", 0), ("stK", T))
                m.write(("dS", 1), ("stK", T))
                m.pending.extend([("store", ("dS", 0), ("stK", T)), ("store", ("dS", 1), ("stK", T))])
            yield ("do", stage_k)
            if m.plant != "stage_early":
                yield ("wait", "stagefree", T)

            def stage_v(T=T):
                if m.plant != "acc_unordered":
                    m.read("dV", ("acc", T, n), "epilogue dV")
                m.write(("dq", 0), ("stV", T))
                m.write(("dq", 1), ("stV", T))
                m.pending.extend([("store", ("dq", 0), ("stV", T)), ("store", ("dq", 1), ("stV", T))])
            yield ("do", stage_v)
            # the store threads wait for their stores to have read shared memory, then the eight
            # warps meet
            yield ("until", lambda: not any(p[0] == "store" for p in m.pending))

    def drain():
        red = []  # this thread's reductions in issue order
        for T in range(ntile):
            for it in range(n):
                g = T * n + it
                yield ("wait", "dqfull", g)

                def take(g=g):
                    m.read(("dQt",), g, "drain")
                    m.arrive("dqfree")
                yield ("do", take)
                for hq in (0, 1):
                    # bulk_wait_read_but_one: every reduction but the newest has read its half
                    yield ("until", lambda: not any(p[0] == "red" and p[3] in red[:-1] for p in m.pending))

                    def stage(g=g, hq=hq):
                        m.write(("dq", hq), ("dq", g, hq))
                        red.append((g, hq))
                        m.pending.append(("red", ("dq", hq), ("dq", g, hq), (g, hq)))
                    yield ("do", stage)
            yield ("until", lambda: not any(p[0] == "red" for p in m.pending))
            yield ("do", lambda: m.arrive("stagefree"))

    return {"prod": prod(), "iss0": issuer(0), "iss1": issuer(1), "iss2": issuer(2), "pds": pds(),
            "drain": drain()}


def _run_pipe_op(m, op):
    kind = op[0]
    if kind == "r":
        m.read(op[1], op[2], "MMA")
    elif kind == "w":
        m.write(op[1], op[2])
    elif kind == "a":
        m.arrive(op[1])
    elif kind == "acc":
        _, acc, T, it = op
        if it == 0:
            if m.ver.get(acc) is not None and m.ver[acc][1] != T and m.read_acc.get(m.ver[acc][1]) is None:
                raise Fault(f"{acc} of tile {m.ver[acc][1]} overwritten before the epilogue read it")
        elif m.ver.get(acc) != ("acc", T, it):
            raise Fault(f"{acc} accumulation out of order: {m.ver.get(acc)} at ({T}, {it})")
        m.write(acc, ("acc", T, it + 1))


def simulate(n, ntile, seed, plant=None):
    rnd = random.Random(seed)
    m = Model(n, ntile, rnd, plant)
    m.late, m.read_acc = [], {}
    progs = _programs(m)
    cur = {k: next(g, None) for k, g in progs.items()}
    orig_read = m.read

    def read(buf, v, who):
        orig_read(buf, v, who)
        if who.startswith("epilogue") and isinstance(v, tuple) and v[0] == "acc":
            m.read_acc[v[1]] = True
    m.read = read
    for _ in range(2_000_000):
        ready = []
        for k, step in cur.items():
            if step is None:
                continue
            if step[0] == "wait":
                if m.wait_ok(step[1], step[2]):
                    ready.append(k)
            elif step[0] == "until":
                if step[1]():
                    ready.append(k)
            else:
                ready.append(k)
        ready += [("pipe", r) for r in range(3) if m.pipes[r]]
        ready += ["tma"] * bool(m.tma) + ["async"] * bool(m.pending) + ["late"] * bool(m.late)
        if not ready:
            if all(s is None for s in cur.values()):
                return m
            raise Fault(f"deadlock: {cur}")
        who = rnd.choice(ready)
        if isinstance(who, tuple):
            ops = m.pipes[who[1]].pop(0)
            for op in ops:
                _run_pipe_op(m, op)
        elif who == "tma":
            buf, v, bar = m.tma.pop(rnd.randrange(len(m.tma)))
            m.write(buf, v)
            m.arrive(bar)
        elif who == "async":
            op = m.pending.pop(rnd.randrange(len(m.pending)))
            m.read(op[1], op[2], "bulk read")
        elif who == "late":
            m.late.pop(0)()
        else:
            step = cur[who]
            if step[0] == "do":
                step[1]()
            cur[who] = next(progs[who], None)
    raise Fault("no progress")


@pytest.mark.parametrize("n,ntile", [(2, 4), (3, 3), (4, 5), (5, 2), (8, 3)])
def test_persistent_backward_protocol(n, ntile):
    for seed in range(150):
        simulate(n, ntile, seed)


@pytest.mark.parametrize("plant", ["kv_early", "stage_early", "acc_unordered", "kread_skipped"])
def test_planted_protocol_mistakes_are_caught(plant):
    caught = 0
    for seed in range(200):
        try:
            simulate(3, 4, seed, plant)
        except Fault:
            caught += 1
    assert caught > 0, plant
