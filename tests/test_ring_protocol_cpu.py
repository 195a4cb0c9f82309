"""The head-pair forward's tile rings, modelled on the CPU.

The kernel streams K and V tiles of two heads through two rings of shared-memory slots: K
piece 2j + x (K of head 2g + x at the j-th visited key block) into K slot (2j + x) % KS, V piece
2i + x into V slot (2i + x) % VS.  Only the S products commit a release, on the K slot's empty
barrier; V piece v counts as free once K piece v + 2 is released, because PV_x(i) precedes
S_x(i+1) in the one issuing thread's order.  Every wait is on the parity of a barrier phase, so
a waiter must never be two completions behind the phase it wants, and no slot may be reloaded
while a product still reads it.  This model plays the producer, the issuing thread, the two
softmax warpgroups, the in-order tensor pipe and the TMA engine in random interleavings, with
the kernel's index and parity formulas, and checks both properties at (KS, VS) = (3, 2) (d = 128)
and (6, 4) (d = 64).  The same model flags the single-ring scheme in which the V pieces carried
no commit (it stalls on a phase that has already been passed)."""
import random

import pytest


class Fault(Exception):
    pass


def _wait_ok(bars, b, k):
    """Wait for completion index k of barrier b by parity (k & 1)."""
    c = bars.get(b, 0)
    sat = (c & 1) != (k & 1)
    if sat and c < k + 1:
        raise Fault(f"early pass on {b}: {c} completions, wanted #{k}")
    if not sat and c >= k + 2:
        raise Fault(f"stuck on {b}: {c} completions, wanted #{k}")
    return sat


def _simulate(n, prod, iss, rnd):
    """prod: [(waits, ('K'|'V', slot))], iss: [(waits, [pipe groups])]; a pipe group is a list of
    ('free', kind, slot) and barrier names completed when the group's products finish."""
    bars = {}
    sm = {x: [([(("sfull", x), j)], x) for j in range(n)] for x in (0, 1)}
    progs = {"prod": prod, "iss": iss, "sm0": sm[0], "sm1": sm[1]}
    pcs = dict.fromkeys(progs, 0)
    pipe, tma, live = [], [("q",)], {}
    done = lambda b: bars.__setitem__(b, bars.get(b, 0) + 1)
    for _ in range(1_000_000):
        ready = [nm for nm, pg in progs.items() if pcs[nm] < len(pg)
                 and all(_wait_ok(bars, b, k) for b, k in pg[pcs[nm]][0])]
        ready += ["mma"] * bool(pipe) + ["tma"] * bool(tma)
        if not ready:
            if all(pcs[nm] >= len(pg) for nm, pg in progs.items()):
                return
            raise Fault(f"deadlock at {pcs}")
        who = rnd.choice(ready)
        if who == "mma":
            for e in pipe.pop(0):
                if e[0] == "free":
                    live[e[1:]] = None
                else:
                    done(e)
        elif who == "tma":
            done(tma.pop(rnd.randrange(len(tma))))
        else:
            act = progs[who][pcs[who]][1]
            pcs[who] += 1
            if who == "prod":
                kind, slot = act
                if live.get((kind, slot)) is not None:
                    raise Fault(f"{kind} slot {slot} reloaded while read")
                live[(kind, slot)] = True
                tma.append((kind + "full", slot))
            elif who == "iss":
                pipe.extend(act)
            else:
                done(("pfull", act))
    raise Fault("no progress")


def _head_pair(n, KS, VS):
    """Programs with the kernel's formulas (separate K and V rings)."""
    prod = []

    def load_k(kq):
        w = [] if kq < KS else [(("kempty", kq % KS), kq // KS - 1)]   # parity ((kq / KS) & 1) ^ 1
        prod.append((w, ("K", kq % KS)))

    def load_v(vq):
        r = vq - VS + 2                                                 # K piece whose release frees V piece vq - VS
        w = [] if vq < VS else [(("kempty", r % KS), r // KS)]
        prod.append((w, ("V", vq % VS)))

    load_k(0)
    load_k(1)
    for i in range(n):
        more = i + 1 < n
        load_v(2 * i)
        if more:
            load_k(2 * i + 2)
        load_v(2 * i + 1)
        if more:
            load_k(2 * i + 3)
    wk = lambda kk: (("Kfull", kk % KS), kk // KS)
    wv = lambda vv: (("Vfull", vv % VS), vv // VS)
    s_group = lambda x, kk: [("free", "K", kk % KS), ("kempty", kk % KS), ("sfull", x)]
    iss = [([(("q",), 0), wk(0)], [s_group(0, 0)]), ([wk(1)], [s_group(1, 1)])]
    for i in range(n):
        more = i + 1 < n
        for x in (0, 1):
            vv, kk = 2 * i + x, 2 * i + 2 + x
            waits = [wv(vv)] + ([wk(kk)] if more else []) + [(("pfull", x), i)]
            pv = [("free", "V", vv % VS)]
            iss.append((waits, [pv, s_group(x, kk)] if more else [pv + [("odone", x)]]))
    return prod, iss


def _single_ring_without_v_commits(n, P):
    """The earlier single ring of P pieces in load order, V pieces without a commit, a V slot's
    reuse keyed to the next piece's slot barrier."""
    order = [("K", 0, 0), ("K", 1, 0)]
    for i in range(n):
        more = i + 1 < n
        order += [("V", 0, i)] + ([("K", 0, i + 1)] if more else []) + [("V", 1, i)] + \
                 ([("K", 1, i + 1)] if more else [])
    isv = lambda r: r >= 2 and (r - 2) % 2 == 0
    prod = []
    for q, _ in enumerate(order):
        r = q - P + (1 if q >= P and isv(q - P) else 0)
        prod.append(([] if q < P else [(("empty", r % P), r // P)], ("R", q % P)))
    pos = {pc: q for q, pc in enumerate(order)}
    w = lambda q: (("Rfull", q % P), q // P)
    s_group = lambda x, q: [("free", "R", q % P), ("empty", q % P), ("sfull", x)]
    iss = [([(("q",), 0), w(0)], [s_group(0, 0)]), ([w(1)], [s_group(1, 1)])]
    for i in range(n):
        more = i + 1 < n
        for x in (0, 1):
            qv = pos[("V", x, i)]
            qk = pos[("K", x, i + 1)] if more else None
            waits = [w(qv)] + ([w(qk)] if more else []) + [(("pfull", x), i)]
            pv = [("free", "R", qv % P)]
            iss.append((waits, [pv, s_group(x, qk)] if more else [pv + [("odone", x)]]))
    return prod, iss


@pytest.mark.parametrize("KS,VS", [(3, 2), (6, 4)])
def test_head_pair_rings(KS, VS):
    for n in list(range(1, 10)) + [23]:
        for seed in range(60):
            prod, iss = _head_pair(n, KS, VS)
            _simulate(n, prod, iss, random.Random(seed * 1000 + n))


def test_model_flags_the_single_ring_without_v_commits():
    failures = 0
    for n in range(3, 9):
        for seed in range(20):
            prod, iss = _single_ring_without_v_commits(n, 5)
            try:
                _simulate(n, prod, iss, random.Random(seed))
            except Fault:
                failures += 1
    assert failures > 0
