"""Discrete-event model of the persistent prefill kernel's synchronisation.

Test infrastructure: no kernel code, no oracle.  Each role of the kernel
(TMA producer, the two QK issuers, the PV issuer, the eight softmax warps)
is a generator that performs the same mbarrier waits, arrivals and
tensor-core commits as the CUDA code, in the same order (the producer polls
its K, V and Q conditions without blocking, as the kernel does), over one CTA's
stream of KV tiles g = 0, 1, ... spanning several work items.  Asynchronous
copies and MMAs complete after random latencies and the roles interleave at
random, and the model checks:

- every wait eventually passes (no deadlock);
- a wait never runs on a phase that the barrier has already left twice, nor
  while the barrier is still two or more phases short of it (a parity wait
  cannot tell phase p from p + 2, nor from p - 2: it would pass at once);
- no buffer is read or written while a conflicting write is in flight;
- every read sees the version the reader expects (K_g for QK_g, the item's Q
  for its products, P_g for PV_g, O accumulated over exactly the item's
  earlier tiles for a rescale or the epilogue, the reference max of tile
  g-1 for tile g);
- the reference max is handed between a quadrant's two softmax warps
  through one shared slot per row tagged with the tile index (the reader
  polls for tag g-1), and a warp never overwrites a value the other warp
  has not taken.

Barrier phases are tracked as counts, so each wait states the phase it means
(`phase`); the kernel passes its parity.  A thread's tensor-core commits
arrive in the order it issued them.  `drop` removes named waits, so a
test can check that each of them is needed.
"""
import random

KK, KV = 4, 3  # K stages, V stages


class ProtocolError(Exception):
    pass


class _Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.done = name, count, count, 0, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise ProtocolError(f"too many arrivals on {self.name}")
        self._complete()

    def expect(self, nbytes):
        self.tx += nbytes

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._complete()

    def _complete(self):
        if self.pending == 0 and self.tx == 0:
            self.done += 1
            self.pending = self.count


class _Sim:
    def __init__(self, rng):
        self.rng = rng
        self.t = 0
        self.bars = {}
        self.events = []       # (time, action)
        self.version = {}      # resource -> version written by completed writes
        self.writes = {}       # resource -> [(end, version)] of issued writes
        self.inflight = {}     # resource -> [(kind, end, who)]
        self.async_ends = {}   # issuing thread -> completion times of its async ops
        self.tags = {}         # tagged shared slot -> tile index it holds
        self.last_commit = {}  # issuing thread -> time its latest commit arrives

    def bar(self, name, count):
        self.bars[name] = _Bar(name, count)

    def lat(self):
        return self.rng.randint(5, 200)

    def access(self, res, kind, dur, who, expect=None, new=None):
        now = self.t
        for (k2, end, w2) in self.inflight.get(res, []):
            if end > now and (kind == "W" or k2 == "W"):
                raise ProtocolError(f"race on {res}: {kind} by {who} while {k2} by {w2}")
        if expect is not None:
            v = self.version.get(res)
            for (end, nv) in sorted(self.writes.get(res, [])):
                if end <= now:
                    v = nv
            if v != expect:
                raise ProtocolError(f"{who} reads {res}: holds {v}, expects {expect}")
        end = now + dur
        self.inflight.setdefault(res, []).append((kind, end, who))
        if kind == "W":
            self.writes.setdefault(res, []).append((end, new))
            self.events.append((end, lambda: self.version.__setitem__(res, new)))
        return end

    def async_op(self, who, end):
        self.async_ends.setdefault(who, []).append(end)

    def commit(self, who, bar):
        # arrives once every earlier asynchronous op of this thread completed,
        # and after this thread's earlier commits (they signal in order)
        end = max(self.async_ends.get(who, []) + [self.t]) + self.rng.randint(1, 30)
        end = max(end, self.last_commit.get(who, 0) + 1)
        self.last_commit[who] = end
        self.events.append((end, lambda: self.bars[bar].arrive()))


def run(items, T, seed, drop=()):
    """items: list of (qt, nkv) for one CTA; raises ProtocolError on a
    violation, returns the number of scheduling steps otherwise."""
    rng = random.Random(seed)
    S = _Sim(rng)
    for b in range(2):
        S.bar(("QFull", b), 2)
        S.bar(("QEmpty", b), 2)
        S.bar(("SFull", b), 1)
        S.bar(("PReady", b), 4)           # one elected lane per softmax warp
    S.bar("QSf", 1)
    S.bar("Ones", 256)
    S.bar("OFree", 4)
    for s in range(KK):
        S.bar(("SRead", s), 4)
        S.bar(("KFull", s), 1)
    for s in range(KV):
        S.bar(("VFull", s), 1)
        S.bar(("ODone", s), 1)
    starts, g = [], 0
    for (_, n) in items:
        starts.append((g, n))
        g += n
    gtot = g

    def wait(name, bar, phase):
        if name in drop:
            return ("step",)
        return ("wait", bar, phase)

    def wait_tag(name, slot, tag):
        if name in drop:
            return ("step",)
        return ("tag", slot, tag)

    def wait_ge(name, slot, tag):
        if name in drop:
            return ("step",)
        return ("ge", slot, tag)

    def producer():
        def load_q(k):
            buf = k & 1
            if k >= 2:
                yield wait("q_empty", ("QEmpty", buf), (k - 2) >> 1)
            qf = S.bars[("QFull", buf)]
            qf.expect(1)
            qf.arrive()
            end = S.access(("Q", buf), "W", S.lat(), "producer", new=("Q", k))
            S.events.append((end, lambda: qf.complete_tx(1)))
            S.access(("Qb", buf), "W", 0, "producer", new=("Qb", k))
            yield ("step",)
            qf.arrive()

        item_of_tile = {}
        for k, (g0, n) in enumerate(starts):
            for j in range(n):
                item_of_tile[g0 + j] = k
        loaded = set()

        def load_k(g):
            k = item_of_tile[g]
            if k not in loaded:
                yield from load_q(k)
                loaded.add(k)
            s = g % KK
            if g >= KK:
                yield wait("k_ring", ("SRead", s), g // KK - 1)
            b = S.bars[("KFull", s)]
            b.expect(1)
            b.arrive()
            end = S.access(("K", s), "W", S.lat(), "producer", new=("K", g))
            S.events.append((end, lambda: b.complete_tx(1)))

        def load_v(g):
            s = g % KV
            if g >= KV:
                yield wait("v_ring", ("ODone", s), g // KV - 1)
            b = S.bars[("VFull", s)]
            b.expect(1)
            b.arrive()
            end = S.access(("V", s), "W", S.lat(), "producer", new=("V", g))
            S.events.append((end, lambda: b.complete_tx(1)))

        # polled: K and V each as soon as its own stage is free
        def ready(name, bar, phase):
            if name in drop:
                return True
            done = S.bars[bar].done
            if done >= phase + 2:
                raise ProtocolError(f"producer: test on {bar} phase {phase} aliased")
            if done < phase and (phase - done) % 2 == 1:
                raise ProtocolError(f"producer: test on {bar} phase {phase} would pass two "
                                    f"phases early (done {done})")
            return done >= phase + 1

        def issue_k(g):
            s = g % KK
            b = S.bars[("KFull", s)]
            b.expect(1)
            b.arrive()
            end = S.access(("K", s), "W", S.lat(), "producer", new=("K", g))
            S.events.append((end, lambda: b.complete_tx(1)))

        def issue_v(g):
            s = g % KV
            b = S.bars[("VFull", s)]
            b.expect(1)
            b.arrive()
            end = S.access(("V", s), "W", S.lat(), "producer", new=("V", g))
            S.events.append((end, lambda: b.complete_tx(1)))

        gk = gv = 0
        loaded.add(0)
        yield from load_q(0)
        while gk < gtot or gv < gtot:
            if gk < gtot:
                k = item_of_tile[gk]
                if k not in loaded:
                    if k < 2 or ready("q_empty", ("QEmpty", k & 1), (k - 2) >> 1):
                        yield from load_q(k)
                        loaded.add(k)
                elif gk < KK or ready("k_ring", ("SRead", gk % KK), gk // KK - 1):
                    issue_k(gk)
                    gk += 1
            if gv < gtot and (gv < KV or ready("v_ring", ("ODone", gv % KV), gv // KV - 1)):
                issue_v(gv)
                gv += 1
            yield ("step",)

    def issuer(par):
        who = f"qk{par}"
        cp_done = [0]   # a thread's MMAs start after its own earlier scale copies

        def issue_qk(g, buf, k):
            s, bk = g % KK, g & 1
            yield wait("k_full", ("KFull", s), g // KK)
            e = S.access(("K", s), "R", S.lat(), who, expect=("K", g))
            S.async_op(who, e)
            e = S.access(("SfK", bk), "W", S.lat(), who, new=("SfK", g))
            S.async_op(who, e)
            start = max(e, cp_done[0])
            yield ("step",)
            saved, S.t = S.t, max(S.t, start)
            d = S.lat()
            for res, v in [(("Q", buf), ("Q", k)), (("Qb", buf), ("Qb", k)), (("SfQ",), ("SfQ", k)),
                           (("SfK", bk), ("SfK", g)), (("K", s), ("K", g))]:
                S.async_op(who, S.access(res, "R", d, who, expect=v))
            S.async_op(who, S.access(("S", bk), "W", d, who, new=("S", g)))
            S.t = saved
            S.commit(who, ("SFull", bk))

        for k, (g0, n) in enumerate(starts):
            buf = k & 1
            copier = (g0 & 1) == par
            if copier:
                yield wait("q_full", ("QFull", buf), k >> 1)
                if g0 >= 1:
                    # the other issuer's products up to tile g0-1 (the last
                    # of the previous item on its bank) have completed
                    yield wait_ge("prev_item_qk", ("qkdone", par ^ 1), g0 - 1)
                if g0 >= 2:
                    yield wait("s_read", ("SRead", (g0 - 2) % KK), (g0 - 2) // KK)
                e = S.access(("SfQ",), "W", S.lat(), who, new=("SfQ", k))
                S.async_op(who, e)
                cp_done[0] = e
                S.access(("Q", buf), "R", 0, who, expect=("Q", k))
                S.commit(who, "QSf")
                yield ("step",)
                yield from issue_qk(g0, buf, k)
                first = g0 + 2
            else:
                if n > 1:
                    yield wait("q_sf", "QSf", k)
                first = g0 + 1
            for g in range(first, g0 + n, 2):
                if g >= 2:
                    yield wait("s_read", ("SRead", (g - 2) % KK), (g - 2) // KK)
                yield from issue_qk(g, buf, k)
            # the last tile this thread issued in the item: once its products
            # have landed (its own latest phase), say so to the other thread
            mine = [g for g in range(g0, g0 + n) if (g & 1) == par]
            if mine:
                last = mine[-1]
                yield wait("qk_own", ("SFull", last & 1), last >> 1)
                S.tags[("qkdone", par)] = last
            S.commit(who, ("QEmpty", buf))

    def pv():
        who = "pv"
        done = [0]   # MMAs of one thread into one accumulator run in order
        yield wait("ones", "Ones", 0)
        for k, (g0, n) in enumerate(starts):
            if k >= 1:
                yield wait("o_free", "OFree", k - 1)
            for j in range(n):
                g = g0 + j
                bp, sp = g & 1, g % KV
                yield wait("p_ready", ("PReady", bp), g >> 1)
                yield wait("v_full", ("VFull", sp), g // KV)
                d = S.lat()
                saved, S.t = S.t, max(S.t, done[0])
                S.async_op(who, S.access(("P", bp), "R", d, who, expect=("P", g)))
                S.async_op(who, S.access(("V", sp), "R", d, who, expect=("V", g)))
                for par in range(2):
                    for quad in range(4):
                        S.async_op(who, S.access(("Ones", par, quad), "R", d, who, expect="ones"))
                e = S.access(("O",), "W", d, who, expect=(("O", k, j) if j > 0 else None),
                             new=("O", k, j + 1))
                S.async_op(who, e)
                done[0] = e
                S.t = saved
                S.commit(who, ("ODone", sp))
                yield ("step",)

    epilogues = set()

    def softmax(par, quad):
        who = f"softmax{par}{quad}"
        yield ("step",)
        # this warp's share of the E4M3 ones atom that every PV reads
        S.access(("Ones", par, quad), "W", 0, who, new="ones")
        S.bars["Ones"].arrive(32)
        yield ("step",)
        for k, (g0, n) in enumerate(starts):
            qt = items[k][0]
            for j in range(0 if (g0 & 1) == par else 1, n, 2):
                g = g0 + j
                bk = par
                yield wait("s_full", ("SFull", bk), g >> 1)
                S.access(("S", bk), "R", 0, who, expect=("S", g))
                S.bars[("SRead", g % KK)].arrive(1)
                yield ("step",)
                slot = ("mslot", quad)
                if g > 0:
                    yield wait_tag("hand_over", slot, g - 1)
                    if S.tags.get(slot) != g - 1:
                        raise ProtocolError(f"{who} tile {g} reads the max of tile "
                                            f"{S.tags.get(slot)}")
                if g + 1 < gtot:
                    if S.tags.get(slot) != (g - 1 if g > 0 else None):
                        raise ProtocolError(f"{who} tile {g} overwrites the max of tile "
                                            f"{S.tags.get(slot)} before it was taken")
                    S.tags[slot] = g
                yield ("step",)
                if j > 0 and rng.random() < 0.3:   # the reference max moved: rescale O
                    yield wait("rescale_o", ("ODone", (g - 1) % KV), (g - 1) // KV)
                    S.access(("O",), "R", 0, who, expect=("O", k, j))
                    S.access(("O",), "W", 0, who, new=("O", k, j))
                if g >= 2:
                    yield wait("p_bank", ("ODone", (g - 2) % KV), (g - 2) // KV)
                S.access(("P", bk), "W", 0, who, new=("P", g))
                S.bars[("PReady", bk)].arrive(1)
                yield ("step",)
            if ((g0 + n - 1) & 1) == par:   # this parity owns the item's last tile
                g = g0 + n - 1
                yield wait("epilogue", ("ODone", g % KV), g // KV)
                S.access(("O",), "R", 0, who, expect=("O", k, n))
                S.bars["OFree"].arrive(1)
                epilogues.add((k, quad))
            del qt

    roles = {"producer": producer(), "qk0": issuer(0), "qk1": issuer(1), "pv": pv()}
    for par in range(2):
        for quad in range(4):
            roles[f"softmax{par}{quad}"] = softmax(par, quad)
    # each role runs at its own random speed in this run and is now and then
    # held back for a while, so that slow warps and stragglers occur as well
    # as even progress
    speed = {r: rng.choice([0.01, 0.1, 1.0]) * rng.random() + 1e-3 for r in roles}
    held = {r: (rng.randint(0, 3000) if rng.random() < 0.3 else 0) for r in roles}
    blocked = {r: None for r in roles}
    live = set(roles)
    steps = 0
    while live:
        steps += 1
        if steps > 5_000_000:
            raise ProtocolError("step limit")
        S.events.sort(key=lambda e: e[0])
        runnable = []
        for r in sorted(live):
            if held[r] > S.t:
                continue
            w = blocked[r]
            if w is None:
                runnable.append(r)
                continue
            if w[0] == "tag":
                if S.tags.get(w[1]) == w[2]:
                    runnable.append(r)
                continue
            if w[0] == "ge":
                if S.tags.get(w[1], -1) >= w[2]:
                    runnable.append(r)
                continue
            bar, phase = w
            done = S.bars[bar].done
            if done >= phase + 2:
                raise ProtocolError(f"{r}: wait on {bar} phase {phase} aliased (done {done})")
            if done < phase and (phase - done) % 2 == 1:
                raise ProtocolError(f"{r}: wait on {bar} phase {phase} would pass two phases "
                                    f"early (done {done})")
            if done == phase + 1:
                runnable.append(r)
        if runnable and (not S.events or rng.random() < 0.7):
            r = rng.choices(runnable, weights=[speed[x] for x in runnable])[0]
            if rng.random() < 0.01:
                held[r] = S.t + rng.randint(1, 2000)
            blocked[r] = None
            try:
                act = next(roles[r])
            except StopIteration:
                live.discard(r)
                continue
            if act[0] == "wait":
                bar, phase = act[1], act[2]
                if S.bars[bar].done >= phase + 2:
                    raise ProtocolError(f"{r}: wait on {bar} phase {phase} aliased")
                d0 = S.bars[bar].done
                if d0 < phase and (phase - d0) % 2 == 1:
                    raise ProtocolError(f"{r}: wait on {bar} phase {phase} would pass two phases "
                                        f"early (done {d0})")
                blocked[r] = (bar, phase)
            elif act[0] in ("tag", "ge"):
                blocked[r] = act
            S.t += 1
        elif S.events or any(held[r] > S.t for r in live):
            t_held = min([held[r] for r in live if held[r] > S.t], default=None)
            if S.events and (t_held is None or S.events[0][0] <= t_held):
                t, action = S.events.pop(0)
                S.t = max(S.t, t)
                action()
            else:
                S.t = t_held
        else:
            raise ProtocolError("deadlock: " + ", ".join(
                f"{r} on {blocked[r]}" for r in sorted(live) if blocked[r]))
    for k in range(len(items)):
        for quad in range(4):
            if (k, quad) not in epilogues:
                raise ProtocolError(f"item {k} quadrant {quad}: no epilogue")
    return steps


def random_items(rng, max_items=7, max_tiles=9):
    """A CTA's item list: causal-like (nkv = qt + 1) or arbitrary lengths."""
    out = []
    for _ in range(rng.randint(1, max_items)):
        qt = rng.randint(0, max_tiles - 1)
        out.append((qt, qt + 1 if rng.random() < 0.5 else rng.randint(1, max_tiles)))
    return out
