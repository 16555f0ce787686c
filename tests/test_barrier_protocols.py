"""Deadlock check of the tensor-core kernels' mbarrier protocols, on the CPU.

Each kernel's warp roles are restated here as sequences of the waits and arrivals they
perform on their mbarriers, step by step, in the order the CUDA code issues them
(`csrc/tc_fwd.cu`, `csrc/tc_bwd.cu`).  An MMA commit or a TMA load is an arrival that may
land at any later time, so a protocol is modelled with every completion immediate and the
roles interleaved at random: one that deadlocks, or that lets a barrier run two phases
ahead of a waiter (the waiter then sees its parity unchanged and waits for ever), stops
making progress here for some interleaving.  A compute warpgroup is one role (its 128
threads arrive together); a barrier counted in threads is counted in groups.

This checks the order of waits and arrivals only, not the data each protects.  The last
test plants a known race (a single dS-ready barrier in the dQ pass, which the kernel
double-buffers) and checks that the model finds it.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.phase = count, count, 0

    def arrive(self):
        self.pending -= 1
        assert self.pending >= 0, "more arrivals than the barrier's count"
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):  # mbarrier.try_wait.parity semantics
        return (self.phase & 1) != parity


def W(b, p):
    return ("wait", b, p)


def A(b):
    return ("arrive", b)


def run(roles, bars, seed, max_stuck=20000):
    """Random interleaving until every role finishes; returns None or a deadlock report."""
    rng = random.Random(seed)
    cur = {k: None for k in roles}
    alive, stuck = set(roles), 0
    while alive:
        k = rng.choice(sorted(alive))
        if cur[k] is None:
            try:
                cur[k] = next(roles[k])
            except StopIteration:
                alive.discard(k)
                continue
        act = cur[k]
        b = bars[act[1]]
        if act[0] == "arrive":
            b.arrive()
            cur[k], stuck = None, 0
        elif b.done(act[2]):
            cur[k], stuck = None, 0
        else:
            stuck += 1
            if stuck > max_stuck:
                return "; ".join(f"{r}: {cur[r]}" for r in sorted(alive))
    return None


def steps_of(costs):
    """Steps over a CTA's whole list: item counter kv, step j, global step g."""
    out, g = [], 0
    for kv, n in enumerate(c for c in costs if c > 0):
        for j in range(n):
            out.append(dict(kv=kv, j=j, g=g, n=n, last=j == n - 1))
            g += 1
    return out


def bars_of(spec):
    return {name: Bar(count) for name, count in spec}


# The work-item ring of the claimed mode (`csrc/feed.cuh`): the claimer publishes list
# entry e + 1 when it claims entry e (entry 0 first; the entry after the last item is
# the end marker), and every other role takes the entries in order, skipping items of no
# steps, with one arrival on the slot's EMPTY barrier per role (an issuer's leading
# cursor "cs" only waits).  Roles mark where they move on: ("claim", kv) before the
# claimer's kv-th item of steps, ("take", kv, cursor) where a cursor moves to it (kv
# equal to the number of such items: the end of the list).
FEED_SLOTS = 8


def feed_bars(costs, readers):
    spec = [(("FEEDFULL", s), 1) for s in range(FEED_SLOTS)]
    spec += [(("FEEDEMPTY", s), readers) for s in range(FEED_SLOTS)]
    return bars_of(spec)


def with_feed(gen, costs, role_kind, feed):
    """Turns a role's markers into feed waits and arrivals (or drops them)."""
    li = [i for i, n in enumerate(costs) if n > 0] + [len(costs)]  # list index; last: end
    pos = {}

    def upto(cursor, last):
        e = pos.get(cursor, 0)
        while e <= last:
            s = e % FEED_SLOTS
            if role_kind == "claimer":
                yield W(("FEEDEMPTY", s), ((e // FEED_SLOTS) & 1) ^ 1)
                yield A(("FEEDFULL", s))
            else:
                yield W(("FEEDFULL", s), (e // FEED_SLOTS) & 1)
                if cursor != "cs":
                    yield A(("FEEDEMPTY", s))
            e += 1
        pos[cursor] = e

    for ev in gen:
        if ev[0] == "claim":
            if feed:
                yield from upto("main", min(li[ev[1]] + 1, len(costs)))
        elif ev[0] == "take":
            if feed:
                yield from upto(ev[2], li[ev[1]])
        else:
            yield ev
    if feed:  # the end marker: published by the claimer, taken by every cursor
        for cursor in pos or ["main"]:
            yield from upto(cursor, len(costs))


# ----------------------------------------------------------------------------- forward
def fwd_roles(costs, NQB, NK, NV, softmax, seed, feed=False, late_epilogue=False):
    """late_epilogue: drain the previous item's output after the next item's second step
    instead of its first (a variant the kernel does not use; with softmax it hangs)."""
    G = 2 if softmax else 4  # softmax warpgroups
    spec = [(("QFULL", s), 1) for s in range(NQB)] + [(("QEMPTY", s), 1) for s in range(NQB)]
    spec += [(("KFULL", s), 1) for s in range(NK)] + [(("KEMPTY", s), 1) for s in range(NK)]
    spec += [(("VFULL", s), 1) for s in range(NV)] + [(("VEMPTY", s), 1) for s in range(NV)]
    for s in range(2):
        spec += [(("SFULL", s), 1), (("PFULL", s), G), (("PEMPTY", s), 1), (("RED", s), G),
                 (("REDL", s), G)]
    spec += [("OFULL", 1), ("OEMPTY", G)]
    bars = bars_of(spec)
    items = [n for n in costs if n > 0]
    rng = random.Random(seed + 7)

    def producer_qk():
        t = 0
        for kv, n in enumerate(items):
            yield ("claim", kv)
            qs = kv % NQB
            yield W(("QEMPTY", qs), ((kv // NQB) & 1) ^ 1)
            yield A(("QFULL", qs))
            for _ in range(n):
                st = t % NK
                yield W(("KEMPTY", st), ((t // NK) & 1) ^ 1)
                yield A(("KFULL", st))
                t += 1

    def producer_v():
        t = 0
        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            for _ in range(n):
                st = t % NV
                yield W(("VEMPTY", st), ((t // NV) & 1) ^ 1)
                yield A(("VFULL", st))
                t += 1

    def s_issuer():
        gs = 0
        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            qs = kv % NQB
            yield W(("QFULL", qs), (kv // NQB) & 1)
            for i in range(n):
                b, kst = gs & 1, gs % NK
                yield W(("PFULL", b), ((gs >> 1) & 1) ^ 1)
                yield W(("KFULL", kst), (gs // NK) & 1)
                yield A(("SFULL", b))
                yield A(("KEMPTY", kst))
                if i == n - 1:
                    yield A(("QEMPTY", qs))
                gs += 1

    def pv_issuer():
        gs, o_it = 0, 0
        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            for j in range(n):
                b, vst = gs & 1, gs % NV
                yield W(("PFULL", b), (gs >> 1) & 1)
                yield W(("VFULL", vst), (gs // NV) & 1)
                if j == 0:
                    yield W("OEMPTY", (o_it & 1) ^ 1)
                yield A(("PEMPTY", b))
                yield A(("VEMPTY", vst))
                if j == n - 1:
                    yield A("OFULL")
                gs += 1
            o_it += 1

    def softmax_group():
        p_it, o_it, l_it, pend = 0, 0, 0, False

        def epilogue():
            nonlocal o_it, pend
            yield W("OFULL", o_it & 1)
            o_it += 1
            yield A("OEMPTY")
            pend = False

        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            for j in range(n):
                b = p_it & 1
                yield W(("SFULL", b), (p_it >> 1) & 1)
                rescale = False
                if softmax:
                    yield A(("RED", b))
                    yield W(("RED", b), (p_it >> 1) & 1)
                    rescale = j > 0 and rng.random() < 0.3
                yield W(("PEMPTY", b), ((p_it >> 1) & 1) ^ 1)
                if rescale:
                    yield W(("PEMPTY", b ^ 1), ((p_it - 1) >> 1) & 1)
                yield A(("PFULL", b))
                if pend and (not late_epilogue or j >= 1 or j == n - 1):  # late: after step 2
                    yield from epilogue()
                p_it += 1
            if softmax:  # row sums through the REDL pair
                yield A(("REDL", 0))
                yield W(("REDL", 0), l_it & 1)
                yield A(("REDL", 1))
                yield W(("REDL", 1), l_it & 1)
                l_it += 1
            if pend:
                yield from epilogue()
            pend = True
        if pend:
            yield from epilogue()

    roles = dict(producer_qk=producer_qk(), producer_v=producer_v(), s_issuer=s_issuer(),
                 pv_issuer=pv_issuer())
    roles.update({f"softmax{g}": softmax_group() for g in range(G)})
    bars.update(feed_bars(costs, len(roles) - 1))
    roles = {k: with_feed(g, costs, "claimer" if k == "producer_qk" else "reader", feed)
             for k, g in roles.items()}
    return roles, bars


# ----------------------------------------------------------------------------- dK/dV
def dkdv_roles(costs, NQ, NO, softmax, seed, feed=False, stage_release_by_score=False):
    """stage_release_by_score: a planted mistake; the Q and dO stages are released by the
    score products (S^T, dP^T) instead of the gradient products that read them later."""
    G = 2 if softmax else 4  # compute warpgroups
    spec = [("KFULL", 1), ("KEMPTY", 1), ("VFULL", 1), ("VEMPTY", 1)]
    # A Q stage is read by S^T(g) (issuer A) and dK(g) (issuer B), a dO stage by dP^T(g)
    # (B) and dV(g) (A).  Each is released by one commit, after the later product: dK(g)
    # is issued only once dS^T(g) exists, which the compute warps form after S^T(g) has
    # completed, and likewise dV(g) after dP^T(g).  `done` records each product's
    # completion (at its commit), and the producers check it before refilling a stage.
    spec += [(("QFULL", s), 1) for s in range(NQ)] + [(("QEMPTY", s), 1) for s in range(NQ)]
    spec += [(("OFULL", s), 1) for s in range(NO)] + [(("OEMPTY", s), 1) for s in range(NO)]
    done = set()  # (product, step)
    spec += [(("RSFULL", s), 1) for s in range(NO)]
    for s in range(2):
        spec += [(("SFULL", s), 1), (("SEMPTY", s), G), (("DPFULL", s), 1), (("PDSFULL", s), G),
                 (("KDONE", s), 1)]
    spec += [("ACCFULL", 2), ("ACCEMPTY", G)]
    bars = bars_of(spec)
    ST = steps_of(costs)
    items = [n for n in costs if n > 0]
    rng = random.Random(seed + 1000)

    def producer_kq():
        q = 0
        for kv, n in enumerate(items):
            yield ("claim", kv)
            yield W("KEMPTY", (kv & 1) ^ 1)
            yield A("KFULL")
            for _ in range(n):
                st = q % NQ
                yield W(("QEMPTY", st), ((q // NQ) & 1) ^ 1)
                if q >= NQ:  # the stage's previous readers have completed
                    assert ("S", q - NQ) in done and ("dK", q - NQ) in done, ("Q stage", q)
                yield A(("QFULL", st))
                q += 1

    def producer_vo():  # V, dO and the row terms (on the dO stage)
        q = 0
        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            yield W("VEMPTY", (kv & 1) ^ 1)
            yield A("VFULL")
            for _ in range(n):
                so = q % NO
                yield W(("OEMPTY", so), ((q // NO) & 1) ^ 1)
                if q >= NO:
                    assert ("dP", q - NO) in done and ("dV", q - NO) in done, ("dO stage", q)
                yield A(("OFULL", so))
                yield A(("RSFULL", so))
                q += 1

    def issuer(chain_p):  # issuer A: S^T and dV; issuer B: dP^T and dK
        a_it = 0

        def score(c):
            b = c["g"] & 1
            n_ring = NQ if chain_p else NO
            st, ph = c["g"] % n_ring, (c["g"] // n_ring) & 1
            if c["j"] == 0:
                yield W("KFULL" if chain_p else "VFULL", c["kv"] & 1)
            yield W(("QFULL" if chain_p else "OFULL", st), ph)
            if chain_p:
                yield W(("KDONE", b), ((c["g"] >> 1) & 1) ^ 1)
            else:
                yield W(("SEMPTY", b), (c["g"] >> 1) & 1)
            done.add(("S" if chain_p else "dP", c["g"]))
            yield A(("SFULL" if chain_p else "DPFULL", b))
            if stage_release_by_score:
                yield A(("QEMPTY" if chain_p else "OEMPTY", st))
            if c["last"]:
                yield A("KEMPTY" if chain_p else "VEMPTY")
                yield ("take", c["kv"] + 1, "cs")  # the leading cursor moves on

        yield ("take", 0, "cs")
        yield ("take", 0, "main")
        cs = 0
        if ST:
            yield from score(ST[0])
            cs = 1
        for cg in ST:
            score_first = chain_p or cg["j"] == 0
            if score_first and cs < len(ST):
                yield from score(ST[cs])
                cs += 1
            b = cg["g"] & 1
            yield W(("PDSFULL", b), (cg["g"] >> 1) & 1)
            if cg["j"] == 0:
                yield W("ACCEMPTY", (a_it & 1) ^ 1)
            done.add(("dV" if chain_p else "dK", cg["g"]))
            if chain_p:
                if not stage_release_by_score:
                    yield A(("OEMPTY", cg["g"] % NO))
            else:
                yield A(("KDONE", b))
                if not stage_release_by_score:
                    yield A(("QEMPTY", cg["g"] % NQ))
            if cg["last"]:
                yield A("ACCFULL")
                a_it += 1
                yield ("take", cg["kv"] + 1, "main")
            if not score_first and cs < len(ST):
                yield from score(ST[cs])
                cs += 1

    def compute_group():
        a_it, pend = 0, False

        def epilogue():
            nonlocal a_it, pend
            yield W("ACCFULL", a_it & 1)
            a_it += 1
            yield A("ACCEMPTY")
            pend = False

        for c in ST:
            if c["j"] == 0:
                yield ("take", c["kv"], "main")
            b = c["g"] & 1
            yield W(("SFULL", b), (c["g"] >> 1) & 1)
            skip = rng.random() < 0.2  # no valid query among this group's columns
            yield A(("SEMPTY", b))
            if not skip:
                yield W(("RSFULL", c["g"] % NO), (c["g"] // NO) & 1)
            yield W(("DPFULL", b), (c["g"] >> 1) & 1)
            yield A(("PDSFULL", b))
            if pend:
                yield from epilogue()
            if c["last"]:
                if pend:
                    yield from epilogue()
                pend = True
        if pend:
            yield from epilogue()

    roles = dict(producer_kq=producer_kq(), producer_vo=producer_vo(), issuer_a=issuer(True),
                 issuer_b=issuer(False))
    roles.update({f"compute{g}": compute_group() for g in range(G)})
    bars.update(feed_bars(costs, len(roles) - 1))
    roles = {k: with_feed(g, costs, "claimer" if k == "producer_kq" else "reader", feed)
             for k, g in roles.items()}
    return roles, bars


# ----------------------------------------------------------------------------- dQ
def dq_roles(costs, NQ, NO, NK, NV, single_ds_barrier=False, feed=False):
    G = 2  # compute warpgroups
    spec = [(("QFULL", s), 1) for s in range(NQ)] + [(("QEMPTY", s), 1) for s in range(NQ)]
    spec += [(("OFULL", s), 1) for s in range(NO)] + [(("OEMPTY", s), 1) for s in range(NO)]
    spec += [(("KFULL", s), 1) for s in range(NK)] + [(("KEMPTY", s), 1) for s in range(NK)]
    spec += [(("VFULL", s), 1) for s in range(NV)] + [(("VEMPTY", s), 1) for s in range(NV)]
    spec += [(("SFULL", s), 1) for s in range(2)] + [(("DSFULL", s), G) for s in range(2)]
    spec += [("DPFULL", 1), ("DPEMPTY", G), ("ACCFULL", 1), ("ACCEMPTY", G)]
    bars = bars_of(spec)
    ST = steps_of(costs)
    items = [n for n in costs if n > 0]

    def ds_bar(g):  # (barrier, parity) on which dS(g) is signalled
        return (("DSFULL", 0), g & 1) if single_ds_barrier else (("DSFULL", g & 1), (g >> 1) & 1)

    def producer(qk):  # Q then K(0), K(1), ...; or dO then V(0), V(1), ...
        q_it, t = 0, 0
        n_row, n_ring = (NQ, NK) if qk else (NO, NV)
        rf, re, kf, ke = ("QFULL", "QEMPTY", "KFULL", "KEMPTY") if qk else ("OFULL", "OEMPTY", "VFULL", "VEMPTY")
        for kv, n in enumerate(items):
            yield ("claim", kv) if qk else ("take", kv, "main")
            qs = q_it % n_row
            yield W((re, qs), ((q_it // n_row) & 1) ^ 1)
            yield A((rf, qs))
            q_it += 1
            for _ in range(n):
                st = t % n_ring
                yield W((ke, st), ((t // n_ring) & 1) ^ 1)
                yield A((kf, st))
                t += 1

    def issuer_a():  # S and dQ
        a_it = 0

        def issue_s(c):
            qs, kst = c["kv"] % NQ, c["g"] % NK
            if c["j"] == 0:
                yield W(("QFULL", qs), (c["kv"] // NQ) & 1)
            yield W(("KFULL", kst), (c["g"] // NK) & 1)
            yield A(("SFULL", c["g"] & 1))
            if c["last"]:
                yield A(("QEMPTY", qs))
                if NQ > 1:
                    yield ("take", c["kv"] + 1, "cs")

        def dq_step(c):
            nonlocal a_it
            yield W(*ds_bar(c["g"]))
            if c["j"] == 0:
                yield W("ACCEMPTY", (a_it & 1) ^ 1)
            yield A(("KEMPTY", c["g"] % NK))
            if c["last"]:
                yield A("ACCFULL")
                a_it += 1
                if NQ > 1:
                    yield ("take", c["kv"] + 1, "main")

        if NQ == 1:  # items one by one: S(0), S(1), then dQ(j) and S(j+2)
            i = 0
            while i < len(ST):
                yield ("take", ST[i]["kv"], "main")
                n = ST[i]["n"]
                it = ST[i:i + n]
                yield from issue_s(it[0])
                if n > 1:
                    yield from issue_s(it[1])
                for j in range(n):
                    yield from dq_step(it[j])
                    if j + 2 < n:
                        yield from issue_s(it[j + 2])
                i += n
        else:  # steps across items: S up to two steps ahead of the next dQ
            cs = 0

            def ahead(cgi):
                nonlocal cs
                while cs < len(ST) and cgi < len(ST) and ST[cs]["g"] < ST[cgi]["g"] + 2:
                    yield from issue_s(ST[cs])
                    cs += 1

            yield ("take", 0, "cs")
            yield ("take", 0, "main")
            yield from ahead(0)
            for i, c in enumerate(ST):
                yield from dq_step(c)
                yield from ahead(i + 1)

    def issuer_b():  # dP
        v_it = 0
        for kv, n in enumerate(items):
            yield ("take", kv, "main")
            qs = kv % NO
            yield W(("OFULL", qs), (kv // NO) & 1)
            for j in range(n):
                vst = v_it % NV
                yield W(("VFULL", vst), (v_it // NV) & 1)
                yield W("DPEMPTY", (v_it & 1) ^ 1)
                yield A("DPFULL")
                yield A(("VEMPTY", vst))
                if j == n - 1:
                    yield A(("OEMPTY", qs))
                v_it += 1

    def compute_group():
        a_it, pend = 0, False

        def epilogue():
            nonlocal a_it, pend
            yield W("ACCFULL", a_it & 1)
            a_it += 1
            yield A("ACCEMPTY")
            pend = False

        for c in ST:
            if c["j"] == 0:
                yield ("take", c["kv"], "main")
            yield W(("SFULL", c["g"] & 1), (c["g"] >> 1) & 1)
            yield W("DPFULL", c["g"] & 1)
            yield A("DPEMPTY")
            yield A(ds_bar(c["g"])[0])
            if pend:
                yield from epilogue()
            if c["last"]:
                if pend:
                    yield from epilogue()
                pend = True
        if pend:
            yield from epilogue()

    roles = dict(producer_qk=producer(True), producer_dov=producer(False), issuer_a=issuer_a(),
                 issuer_b=issuer_b())
    roles.update({f"compute{g}": compute_group() for g in range(G)})
    bars.update(feed_bars(costs, len(roles) - 1))
    roles = {k: with_feed(g, costs, "claimer" if k == "producer_qk" else "reader", feed)
             for k, g in roles.items()}
    return roles, bars


def item_costs(seed, n=24):
    """Steps per item of one CTA: many one- and two-step items, some long ones, a few empty."""
    rng = random.Random(seed)
    return [rng.choice([0, 1, 1, 1, 2, 2, 3, 4, 7]) for _ in range(n)]


SEEDS = range(8)


# ring depths of the head-dim variants (Dqk, Dv) = (128,128), (64,64), (128,64), (64,128)
@pytest.mark.parametrize("rings", [(2, 3, 2), (2, 6, 6), (2, 3, 4), (2, 4, 4)])
@pytest.mark.parametrize("softmax", [True, False])
def test_forward_protocol(rings, softmax):
    for seed in SEEDS:
        roles, bars = fwd_roles(item_costs(seed), *rings, softmax, seed)
        assert run(roles, bars, seed) is None, f"seed {seed}"


@pytest.mark.parametrize("rings", [(3, 2), (4, 4), (4, 2)])
@pytest.mark.parametrize("softmax", [True, False])
def test_dkdv_protocol(rings, softmax):
    for seed in SEEDS:
        roles, bars = dkdv_roles(item_costs(seed), *rings, softmax, seed)
        assert run(roles, bars, seed) is None, f"seed {seed}"


@pytest.mark.parametrize("rings", [(1, 1, 3, 2), (2, 2, 6, 4), (2, 2, 3, 2), (2, 2, 4, 2)])
def test_dq_protocol(rings):
    for seed in SEEDS:
        roles, bars = dq_roles(item_costs(seed), *rings)
        assert run(roles, bars, seed) is None, f"seed {seed}"


# The claimed mode runs only in the SiLU/L kernels (softmax=False) of the dK/dV and
# forward passes; the dQ model has the SiLU/L kernel's two-Q-tile walk for D = 64 and the
# single-tile one for D = 128.
@pytest.mark.parametrize("rings", [(2, 3, 2), (2, 6, 6)])
def test_forward_protocol_with_item_ring(rings):
    for seed in SEEDS:
        roles, bars = fwd_roles(item_costs(seed), *rings, False, seed, feed=True)
        assert run(roles, bars, seed) is None, f"seed {seed}"


@pytest.mark.parametrize("rings", [(3, 2), (4, 4)])
def test_dkdv_protocol_with_item_ring(rings):
    for seed in SEEDS:
        roles, bars = dkdv_roles(item_costs(seed), *rings, False, seed, feed=True)
        assert run(roles, bars, seed) is None, f"seed {seed}"


@pytest.mark.parametrize("rings", [(1, 1, 3, 2), (2, 2, 6, 4)])
def test_dq_protocol_with_item_ring(rings):
    for seed in SEEDS:
        roles, bars = dq_roles(item_costs(seed), *rings, feed=True)
        assert run(roles, bars, seed) is None, f"seed {seed}"


def test_item_ring_model_finds_a_missing_arrival():
    """A reader role that never releases its slots must stall the claimer once the ring
    is full; the model must report it."""
    costs = [1] * 40
    roles, bars = fwd_roles(costs, 2, 3, 2, False, 0, feed=True)
    bars[("FEEDEMPTY", 0)].count = bars[("FEEDEMPTY", 0)].pending = 99  # never completes
    assert run(roles, bars, 0) is not None


def test_model_finds_the_softmax_late_epilogue_deadlock():
    """Softmax may wait, at an item's second step, for the item's first PV product before
    rescaling O; that product waits for the previous item's output to be drained.  So the
    forward drains at the first step; drained at the second, the model must hang."""
    found = 0
    for seed in SEEDS:
        roles, bars = fwd_roles(item_costs(seed), 2, 3, 2, True, seed, late_epilogue=True)
        found += run(roles, bars, seed) is not None
    assert found > 0


def test_model_finds_a_planted_race():
    """A single dS-ready barrier lets the compute warps finish two steps before issuer A
    looks; the model must find the resulting hang for some interleaving."""
    found = 0
    for seed in SEEDS:
        roles, bars = dq_roles(item_costs(seed), 2, 2, 6, 4, single_ds_barrier=True)
        found += run(roles, bars, seed) is not None
    assert found > 0


def test_model_finds_a_stage_released_before_its_last_reader():
    """The Q and dO stages of dK/dV are released by one commit each, after the gradient
    product that reads them last.  Released instead by the score products, a producer can
    refill a stage that dK or dV still reads; the model's hazard check must catch it."""
    caught = 0
    for seed in SEEDS:
        roles, bars = dkdv_roles(item_costs(seed), 3, 2, False, seed, stage_release_by_score=True)
        try:
            run(roles, bars, seed)
        except AssertionError:
            caught += 1
    assert caught > 0
