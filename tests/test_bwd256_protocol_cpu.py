"""The d = 256 backward's barrier protocols, modelled on the CPU.

At d = 256 a 128-key tile's dK and dV accumulators (128 x 256 fp32 each) fill tensor memory, and K
and V (64 KB each) leave no room for a Q/dO ring beside them, so each key tile runs two passes:

  pass A (dV):     K resident; Q_i and dO_i (with the row terms) in two-stage rings of their own,
                   Q released by S^T, dO by dV; S^T_i = K Q_i^T into one of two S buffers, P^T
                   written back over it by the P warps, dV += P^T dO_i (A from tensor memory).
                   The issuing thread puts S^T of block i + 1 before dV of block i.
  pass B (dK, dQ): K and V resident; Q_i in two 128-column halves ("units" 2i, 2i + 1) in a ring
                   of three unit slots (unit u in slot u mod 3, its row terms with unit 2i); dO_i
                   in one slot; one S, one dP, one dS and one dQ^T buffer.  Issuer 0 issues S^T of
                   block i + 1 over the first unit, then dK of block i (two N = 128 products, one
                   per unit, each releasing its unit), then S^T of block i + 1 over the second
                   unit, which can only be loaded once dK of block i has read unit 2i.  Issuer 1
                   issues dP^T, issuer 2 dQ^T, whose M half 0 four drain warps add into the fp32
                   accumulator and whose M half 1 the eight dS warps add after publishing the next
                   block's dS; the buffer is released by both.  The dK epilogue stages over the
                   unit slots and the dS tile once the last dQ^T, which reads dS, is complete.

The model plays the producer, the issuing threads with their in-order product queues, the
elementwise warps, the dQ drain, the TMA engine and the epilogue's tensor stores in random
interleavings with the kernel's index and parity formulas.  Every buffer carries the version last
written to it and every read checks the version it expects, so a wait that passes early, or a
buffer rewritten while a read is pending, shows up as a wrong version; a parity wait two or more
completions behind the phase it wants is reported as stuck; a wait that can never pass is reported
as a deadlock.  Planted mistakes are caught."""
import random

import pytest


class Fault(Exception):
    pass


class Model:
    def __init__(self, counts, plant):
        self.plant = plant
        self.arrivals = {}
        self.count = counts
        self.ver = {}
        self.pending = []    # tensor stores in flight: (buffer, expected version)
        self.tma = []        # loads in flight: ([(buffer, version)], barrier)
        self.pipes = {r: [] for r in range(3)}

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

    def write(self, buf, v):
        self.ver[buf] = v

    def read(self, buf, v, who):
        if self.ver.get(buf) != v:
            raise Fault(f"{who} read {buf} = {self.ver.get(buf)}, expected {v}")

    def load(self, items, bar):
        for buf, _ in items:
            if any(buf == p[0] for p in self.pending):
                raise Fault(f"load into {buf} while a tensor store still reads it")
        self.tma.append((items, bar))


def _run_pipe_op(m, op):
    kind = op[0]
    if kind == "r":
        m.read(op[1], op[2], "MMA")
    elif kind == "w":
        m.write(op[1], op[2])
    elif kind == "a":
        m.arrive(op[1])
    elif kind == "acc":
        _, acc, it = op
        if it == 0:
            if m.ver.get(acc) is not None:
                raise Fault(f"{acc} accumulated twice from zero")
        elif m.ver.get(acc) != ("acc", it):
            raise Fault(f"{acc} accumulation out of order: {m.ver.get(acc)} at {it}")
        m.write(acc, ("acc", it + 1))


def _run(m, progs, rnd):
    cur = {k: next(g, None) for k, g in progs.items()}
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
        ready += ["tma"] * bool(m.tma) + ["async"] * bool(m.pending)
        if not ready:
            if all(s is None for s in cur.values()):
                return m
            raise Fault(f"deadlock: {cur}")
        who = rnd.choice(ready)
        if isinstance(who, tuple):
            for op in m.pipes[who[1]].pop(0):
                _run_pipe_op(m, op)
        elif who == "tma":
            items, bar = m.tma.pop(rnd.randrange(len(m.tma)))
            for buf, v in items:
                m.write(buf, v)
            m.arrive(bar)
        elif who == "async":
            buf, v = m.pending.pop(rnd.randrange(len(m.pending)))
            m.read(buf, v, "tensor store")
        else:
            step = cur[who]
            if step[0] == "do":
                step[1]()
            cur[who] = next(progs[who], None)
    raise Fault("no progress")


# ------------------------------------------------------------------------------ pass A (dV)
def simulate_dv(n, seed, plant=None):
    rnd = random.Random(seed)
    m = Model({"qempty": 1, "qfull": 1, "dofull": 1, "doempty": 1, "sfull": 1, "pfull": 1, "kvdone": 1}, plant)
    ST = 2
    sb = lambda it: 0 if plant == "a_one_s_buffer" else it & 1

    def prod():
        yield ("do", lambda: m.load([("K", 0)], "kv"))
        for it in range(n):
            s = it % ST
            if it >= ST and plant != "a_ring_early":
                yield ("wait", ("qempty", s), it // ST - 1)
            yield ("do", lambda it=it, s=s: m.load([(("q", s), it)], ("qfull", s)))
            if it >= ST:
                yield ("wait", ("doempty", s), it // ST - 1)
            # the row terms travel with dO: the P warps read them after S^T has released Q
            yield ("do", lambda it=it, s=s: m.load([(("do", s), it), (("ld", s), it)], ("dofull", s)))

    def issuer():
        pipe = m.pipes[0]

        def first(it):
            s, b = it % ST, sb(it)
            yield ("wait", ("qfull", s), it // ST)
            yield ("do", lambda: pipe.append([("r", "K", 0), ("r", ("q", s), it), ("w", ("S", b), ("S", it)),
                                              ("a", ("sfull", b)), ("a", ("qempty", s))]))

        yield ("wait", "kv", 0)
        yield from first(0)
        for it in range(n):
            s, b = it % ST, sb(it)
            if it + 1 < n:
                yield from first(it + 1)
            yield ("wait", ("pfull", b), it >> 1)
            yield ("wait", ("dofull", s), it // ST)
            ops = [("r", ("S", b), ("P", it)), ("r", ("do", s), it), ("acc", "dV", it), ("a", ("doempty", s))]
            yield ("do", lambda ops=ops: pipe.append(ops))
        yield ("do", lambda: pipe.append([("a", "kvdone")]))

    def pwarps():
        for it in range(n):
            s, b = it % ST, sb(it)
            yield ("wait", ("sfull", b), it >> 1)
            if plant != "a_ld_unwaited":
                yield ("wait", ("dofull", s), it // ST)

            def work(it=it, s=s, b=b):
                m.read(("S", b), ("S", it), "P warps")
                m.read(("ld", s), it, "P warps row terms")
                m.write(("S", b), ("P", it))
                m.arrive(("pfull", b))
            yield ("do", work)
        if n > 0:
            yield ("wait", "kvdone", 0)

            def stage():
                m.read("dV", ("acc", n), "epilogue")
                for s in range(ST):
                    m.write(("q", s), "stage")
                    m.pending.append((("q", s), "stage"))
            yield ("do", stage)
            yield ("until", lambda: not m.pending)

    _run(m, {"prod": prod(), "iss": issuer(), "pw": pwarps()}, rnd)
    return m


# ------------------------------------------------------------------------------ pass B (dK, dQ)
U = 3  # Q unit slots


def simulate_dk(n, seed, plant=None):
    rnd = random.Random(seed)
    m = Model({"qempty": 1, "sfull": 1, "dpfull": 1, "sfree": 1, "dpfree": 1, "pfull": 1, "dsfree": 2,
               "dqfull": 1, "dqfree": 2, "dofull": 1, "doempty": 1, "kvdone": 1}, plant)
    qu = lambda u: ("qu", u % U)

    def prod():
        yield ("do", lambda: m.load([("K", 0), ("V", 0)], "kv"))
        for it in range(n):
            u0, u1 = 2 * it, 2 * it + 1
            if u0 >= U and plant != "b_ring_early":
                yield ("wait", ("qempty", u0 % U), u0 // U - 1)
            # the first unit carries the block's row terms
            yield ("do", lambda it=it, u0=u0: m.load([(qu(u0), u0), (("ld", u0 % U), it)], ("qempty_full", u0 % U)))
            if it >= 1:
                yield ("wait", "doempty", it - 1)
            yield ("do", lambda it=it: m.load([("dO", it)], "dofull"))
            if u1 >= U and plant != "b_ring_early":
                yield ("wait", ("qempty", u1 % U), u1 // U - 1)
            yield ("do", lambda u1=u1: m.load([(qu(u1), u1)], ("qempty_full", u1 % U)))

    def issuer0():
        pipe = m.pipes[0]

        def s_lo(it):
            u = 2 * it
            yield ("wait", ("qempty_full", u % U), u // U)
            if it >= 1 and plant != "b_no_sfree":
                yield ("wait", "sfree", it - 1)
            yield ("do", lambda: pipe.append([("r", "K", 0), ("r", qu(u), u), ("w", "S", ("Slo", it))]))

        def s_hi(it):
            u = 2 * it + 1
            yield ("wait", ("qempty_full", u % U), u // U)
            yield ("do", lambda: pipe.append([("r", "K", 0), ("r", qu(u), u), ("r", "S", ("Slo", it)),
                                              ("w", "S", ("S", it)), ("a", "sfull")]))

        yield ("wait", "kv", 0)
        yield from s_lo(0)
        yield from s_hi(0)
        for it in range(n):
            if it + 1 < n:
                yield from s_lo(it + 1)
            yield ("wait", "pfull", it)
            u0, u1 = 2 * it, 2 * it + 1
            ops = [("r", "dS", it), ("r", qu(u0), u0), ("acc", "dK0", it), ("a", ("qempty", u0 % U)),
                   ("r", "dS", it), ("r", qu(u1), u1), ("acc", "dK1", it), ("a", ("qempty", u1 % U)),
                   ("a", "dsfree")]
            yield ("do", lambda ops=ops: pipe.append(ops))
            if it + 1 < n:
                yield from s_hi(it + 1)
        yield ("do", lambda: pipe.append([("a", "kvdone")]))

    def issuer1():
        pipe = m.pipes[1]
        yield ("wait", "kv", 0)
        for it in range(n):
            yield ("wait", "dofull", it)
            if it >= 1:
                yield ("wait", "dpfree", it - 1)
            ops = [("r", "V", 0), ("r", "dO", it), ("w", "dP", ("dP", it)), ("a", "dpfull"), ("a", "doempty")]
            yield ("do", lambda ops=ops: pipe.append(ops))

    def issuer2():
        pipe = m.pipes[2]
        yield ("wait", "kv", 0)
        for it in range(n):
            yield ("wait", "pfull", it)
            if it >= 1 and plant != "b_no_dqfree":
                yield ("wait", "dqfree", it - 1)
            ops = [("r", "K", 0), ("r", "dS", it), ("w", "dQt", it), ("a", "dsfree"), ("a", "dqfull")]
            yield ("do", lambda ops=ops: pipe.append(ops))

    def pdswarps():
        for it in range(n):
            yield ("wait", "sfull", it)
            yield ("wait", "dpfull", it)

            def take(it=it):
                m.read("S", ("S", it), "P/dS")
                m.read("dP", ("dP", it), "P/dS")
                m.read(("ld", (2 * it) % U), it, "P/dS row terms")
                m.arrive("sfree")
                m.arrive("dpfree")
            yield ("do", take)
            if it >= 1 and plant != "b_no_dsfree":
                yield ("wait", "dsfree", it - 1)

            def publish(it=it):
                m.write("dS", it)
                m.arrive("pfull")
            yield ("do", publish)
            # then M half 1 of dQ^T of the block before (the drain warps take half 0)
            if it >= 1:
                yield ("wait", "dqfull", it - 1)

                def half(it=it):
                    m.read("dQt", it - 1, "dS warps")
                    m.arrive("dqfree")
                yield ("do", half)
        if n > 0:
            yield ("wait", "dqfull", n - 1)

            def lasthalf():
                m.read("dQt", n - 1, "dS warps")
                m.arrive("dqfree")
            yield ("do", lasthalf)
            yield ("wait", "kvdone", 0)
            # dK is staged over the unit slots and the dS tile: dQ^T of the last block reads dS
            if plant != "b_epilogue_early":
                yield ("wait", "dsfree", n - 1)

            def stage():
                m.read("dK0", ("acc", n), "epilogue")
                m.read("dK1", ("acc", n), "epilogue")
                for buf in [("qu", s) for s in range(U)] + ["dS"]:
                    m.write(buf, "stage")
                    m.pending.append((buf, "stage"))
            yield ("do", stage)
            yield ("until", lambda: not any(p[1] == "stage" for p in m.pending))

    def drain():
        # M half 0 of dQ^T of block it (atomic adds from registers follow); the buffer is handed
        # back once the dS warps have read half 1 too
        for it in range(n):
            yield ("wait", "dqfull", it)

            def take(it=it):
                m.read("dQt", it, "drain")
                m.arrive("dqfree")
            yield ("do", take)

    # the unit slots' full barriers are named apart from qempty so that counts stay per name
    m.count["qempty_full"] = 1
    _run(m, {"prod": prod(), "iss0": issuer0(), "iss1": issuer1(), "iss2": issuer2(), "pds": pdswarps(),
             "drain": drain()}, rnd)
    return m


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_dv_pass_protocol(n):
    for seed in range(150):
        simulate_dv(n, seed)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8])
def test_dk_pass_protocol(n):
    for seed in range(150):
        simulate_dk(n, seed)


@pytest.mark.parametrize("plant", ["a_ring_early", "a_one_s_buffer", "a_ld_unwaited"])
def test_dv_pass_planted_mistakes_are_caught(plant):
    caught = 0
    for seed in range(200):
        try:
            simulate_dv(4, seed, plant)
        except Fault:
            caught += 1
    assert caught > 0, plant


@pytest.mark.parametrize("plant", ["b_ring_early", "b_no_sfree", "b_no_dsfree", "b_no_dqfree"])
def test_dk_pass_planted_mistakes_are_caught(plant):
    # a drain that lags a whole block behind is a rare interleaving: run until one is caught
    for seed in range(3000):
        try:
            simulate_dk(8, seed, plant)
        except Fault:
            return
    pytest.fail(plant)
