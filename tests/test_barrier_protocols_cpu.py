"""Models of the attention kernels' synchronisation protocols, checked on the CPU.

Each tcgen05 attention kernel coordinates a TMA thread, one MMA-issuing thread
and groups of element-wise warps through mbarriers. A protocol error in such a
kernel hangs or faults the GPU rather than failing a comparison, so each
protocol is modelled here as a discrete-event system and run with random
latencies:

* mbarriers complete a phase after `count` arrivals, and a wait with parity p
  returns once (completed phases & 1) != p, as on the hardware; every wait in
  a model names the phase it means, and the checker fails a wait that returns
  before that phase completed or after a later one did (a waiter two phases
  behind cannot tell them apart);
* the tensor pipe runs products in issue order; a commit arrives on its
  barrier once every product issued before it has finished;
* a TMA load into a shared-memory slot or stage that a product still reads,
  a product reading a slot that holds another tile, or an element-wise
  access to a TMEM region that a product in flight writes or reads, fails;
* a model that stops making progress fails as a deadlock.

The protocols are those of the dK/dV and dQ backward kernels
(attention_bwd_tc.cu) and of the hd-128 forward (attention_tc.cu). Each test
also runs a variant with one release moved to the wrong slot or stage and
expects the checker to catch it.
"""
import heapq
import random

import pytest


class Bar:
    def __init__(self, name, count):
        self.name, self.count, self.arrivals, self.done = name, count, 0, 0

    def arrive(self):
        self.arrivals += 1
        if self.arrivals == self.count:
            self.arrivals = 0
            self.done += 1

    def ready(self, parity):
        return (self.done & 1) != parity


class Sim:
    """Agents are generators yielding ('wait', bar, phase, what), ('do', fn)
    or ('delay', t); a phase below 0 (the first use of a free slot) passes."""

    def __init__(self, seed):
        self.rnd = random.Random(seed)
        self.t = 0.0
        self.events = []
        self.errors = []
        self.pipe = []
        self.busy = {}
        self.waiting = {}
        self.agents = {}
        self.sched(0.0, self._pipe_step)

    def sched(self, dt, fn):
        heapq.heappush(self.events, (self.t + dt, self.rnd.random(), fn))

    # tensor pipe: products (reading slots, writing / reading TMEM regions) and commits
    def product(self, name, reads=(), writes=None, tmem_reads=None):
        for holder, key, want in reads:
            if holder[key] != want:
                self.errors.append(f"{name} reads {key} holding {holder[key]}, wants {want}")
        self.pipe.append(("mma", name, reads, writes, tmem_reads, None))
        for holder, key, _ in reads:
            self.readers[key] = self.readers.get(key, 0) + 1
        for r in (writes, tmem_reads):
            if r:
                self.busy.setdefault(r, []).append(name)

    def commit(self, bar):
        self.pipe.append(("commit", None, (), None, None, bar))

    def _pipe_step(self):
        if not self.pipe:
            self.sched(0.2, self._pipe_step)
            return
        kind, name, reads, writes, tmem_reads, bar = self.pipe.pop(0)

        def finish():
            if kind == "commit":
                bar.arrive()
            else:
                for _, key, _ in reads:
                    self.readers[key] -= 1
                for r in (writes, tmem_reads):
                    if r:
                        self.busy[r].remove(name)
            self._pipe_step()

        self.sched(0.01 if kind == "commit" else self.rnd.uniform(0.5, 1.5), finish)

    def load(self, holder, key, tag, bar):
        if self.readers.get(key, 0):
            self.errors.append(f"load of {tag} into {key} while {self.readers[key]} product(s) read it")

        def land():
            holder[key] = tag
            bar.arrive()

        self.sched(self.rnd.uniform(1, 6), land)

    def touch(self, region, who):
        if self.busy.get(region):
            self.errors.append(f"{who} touched {region} under {self.busy[region]}")

    def run(self, agents, finished, limit):
        self.agents = agents
        self.readers = {}
        for name in agents:
            self.sched(self.rnd.uniform(0, 0.2), lambda n=name: self._step(n))
        while self.events:
            t, _, fn = heapq.heappop(self.events)
            self.t = t
            fn()
            if finished() and not self.waiting:
                break
            if self.t > limit:
                self.errors.append(f"deadlock: {[(k, v[2]) for k, v in self.waiting.items()]}")
                break
        return self.errors

    def _step(self, name):
        gen = self.agents[name]
        while True:
            try:
                act = next(gen)
            except StopIteration:
                return
            if act[0] == "do":
                act[1]()
                continue
            if act[0] == "delay":
                self.sched(act[1], lambda: self._step(name))
                return
            _, bar, phase, what = act
            if phase < 0:
                continue
            self.waiting[name] = (bar, phase, what)
            self.sched(0.0, lambda: self._poll(name))
            return

    def _poll(self, name):
        bar, phase, what = self.waiting[name]
        if bar.ready(phase & 1):
            if bar.done <= phase:
                self.errors.append(f"{what}: passed with {bar.name} at {bar.done} phases, wants phase {phase}")
            if bar.done > phase + 1:
                self.errors.append(f"{what}: {bar.name} ran two phases past the waiter")
            del self.waiting[name]
            self.sched(self.rnd.uniform(0.01, 0.1), lambda: self._step(name))
        else:
            self.sched(0.05, lambda: self._poll(name))


def slot_q(j):
    return (0, 2, 1, 3)[j & 3]


def slot_o(j):
    return (1, 3, 0, 2)[j & 3]


def dkdv(total, seed, misplace=False):
    """dK/dV, 128-query sub-tiles: the MMA thread issues dP^T j, dV j,
    S^T j + 1, dK j, waiting on the element-wise group's s_read / pv_full /
    d_read / ds_full and committing s_full / d_full only; one element-wise
    warp checks Q / dO landed and releases each slot once s_full j (dV j - 1
    done) or d_full j (dK j - 1 done) shows its last reader finished."""
    sim = Sim(seed)
    slots = {}
    kv = Bar("kv_full", 1)
    full = [Bar(f"slot_full{i}", 1) for i in range(4)]
    empty = [Bar(f"slot_empty{i}", 1) for i in range(4)]
    s_full, s_read, d_full, d_read = (Bar(n, 1) for n in ("s_full", "s_read", "d_full", "d_read"))
    pv_full, ds_full, done = Bar("pv_full", 1), Bar("ds_full", 1), Bar("done", 1)

    def producer():
        yield ("do", lambda: sim.sched(sim.rnd.uniform(1, 4), kv.arrive))
        for j in range(total):
            for sl, tag in ((slot_q(j), ("Q", j)), (slot_o(j), ("dO", j))):
                yield ("wait", empty[sl], (j >> 1) - 1, f"producer slot {sl} for {tag}")
                yield ("do", lambda sl=sl, tag=tag: sim.load(slots, sl, tag, full[sl]))

    def mma():
        yield ("wait", kv, 0, "mma K, V")
        yield ("wait", full[slot_q(0)], 0, "mma Q0")
        yield ("do", lambda: sim.product("S0", [(slots, slot_q(0), ("Q", 0))], writes="tA"))
        yield ("do", lambda: sim.commit(s_full))
        for j in range(total):
            yield ("wait", s_read, j, f"mma s_read {j}")
            yield ("do", lambda j=j: sim.product(f"dP{j}", [(slots, slot_o(j), ("dO", j))], writes="tA"))
            yield ("do", lambda: sim.commit(d_full))
            yield ("wait", pv_full, j, f"mma pv_full {j}")
            yield ("do", lambda j=j: sim.product(f"dV{j}", [(slots, slot_o(j), ("dO", j))], tmem_reads="tB.P"))
            if j + 1 < total:
                yield ("wait", d_read, j, f"mma d_read {j}")
                yield ("do", lambda j=j: sim.product(f"S{j + 1}", [(slots, slot_q(j + 1), ("Q", j + 1))],
                                                     writes="tA"))
                yield ("do", lambda: sim.commit(s_full))
            yield ("wait", ds_full, j, f"mma ds_full {j}")
            yield ("do", lambda j=j: sim.product(f"dK{j}", [(slots, slot_q(j), ("Q", j))], tmem_reads="tB.dS"))
        yield ("do", lambda: sim.commit(done))

    def group():
        for j in range(total):
            yield ("wait", full[slot_o(j)], j >> 1, f"loads warp dO {j}")
            yield ("wait", s_full, j, f"group s_full {j}")
            if j > 0:
                rel = slot_o(j) if misplace else slot_o(j - 1)
                yield ("do", lambda rel=rel: empty[rel].arrive())
            yield ("do", lambda j=j: sim.touch("tA", f"group load S{j}"))
            yield ("do", s_read.arrive)
            yield ("delay", sim.rnd.uniform(0.3, 1.0))
            yield ("do", lambda j=j: sim.touch("tB.P", f"group store P{j}"))
            yield ("do", pv_full.arrive)
            if j + 1 < total:
                yield ("wait", full[slot_q(j + 1)], (j + 1) >> 1, f"loads warp Q {j + 1}")
            yield ("wait", d_full, j, f"group d_full {j}")
            if j > 0:
                yield ("do", lambda j=j: empty[slot_q(j - 1)].arrive())
            yield ("do", lambda j=j: sim.touch("tA", f"group load dP{j}"))
            yield ("do", d_read.arrive)
            yield ("delay", sim.rnd.uniform(0.3, 1.0))
            yield ("do", lambda j=j: sim.touch("tB.dS", f"group store dS{j}"))
            yield ("do", ds_full.arrive)
        yield ("wait", done, 0, "group done")

    return sim.run({"producer": producer(), "mma": mma(), "group": group()},
                   lambda: done.done >= 1, 60 * (total + 5))


def dq(n, seed, ks_n=3, vs_n=2, misplace=False):
    """dQ: K and V of tile j land on one barrier (j % kVS) that one
    element-wise warp checks before the s_empty arrival; that warp frees V
    j's stage once S / dP j are done; the MMA thread commits K j's stage
    after dQ j."""
    sim = Sim(seed)
    stages = {}
    q_full = Bar("q_full", 1)
    kv_full = [Bar(f"kv_full{i}", 2) for i in range(vs_n)]   # K and V land on one barrier
    k_empty = [Bar(f"k_empty{i}", 1) for i in range(ks_n)]
    v_empty = [Bar(f"v_empty{i}", 1) for i in range(vs_n)]
    s_full, s_empty, p_full, done = (Bar(n_, 1) for n_ in ("s_full", "s_empty", "p_full", "done"))

    def producer():
        yield ("do", lambda: sim.sched(sim.rnd.uniform(1, 3), q_full.arrive))
        for j in range(n):
            yield ("wait", k_empty[j % ks_n], j // ks_n - 1, f"producer K stage for {j}")
            yield ("wait", v_empty[j % vs_n], j // vs_n - 1, f"producer V stage for {j}")

            def issue(j=j):
                sim.load(stages, ("K", j % ks_n), j, kv_full[j % vs_n])
                sim.load(stages, ("V", j % vs_n), j, kv_full[j % vs_n])
            yield ("do", issue)

    def mma():
        yield ("wait", q_full, 0, "mma Q")
        yield ("wait", kv_full[0], 0, "mma K, V 0")
        yield ("do", lambda: sim.product("SdP0", [(stages, ("K", 0), 0), (stages, ("V", 0), 0)], writes="tS"))
        yield ("do", lambda: sim.commit(s_full))
        for j in range(n):
            if j + 1 < n:
                yield ("wait", s_empty, j, f"mma s_empty {j}")
                yield ("do", lambda j=j: sim.product(
                    f"SdP{j + 1}", [(stages, ("K", (j + 1) % ks_n), j + 1), (stages, ("V", (j + 1) % vs_n), j + 1)],
                    writes="tS"))
                yield ("do", lambda: sim.commit(s_full))
            yield ("wait", p_full, j, f"mma p_full {j}")
            yield ("do", lambda j=j: sim.product(f"dQ{j}", [(stages, ("K", j % ks_n), j)], tmem_reads=f"tDS{j & 1}"))
            yield ("do", lambda j=j: sim.commit(k_empty[j % ks_n]))
        yield ("do", lambda: sim.commit(done))

    def group():
        for j in range(n):
            if j + 1 < n:
                yield ("wait", kv_full[(j + 1) % vs_n], (j + 1) // vs_n, f"loads warp K, V {j + 1}")
            yield ("wait", s_full, j, f"group s_full {j}")
            rel = (j + 1) % vs_n if misplace else j % vs_n
            yield ("do", lambda rel=rel: v_empty[rel].arrive())
            yield ("do", lambda j=j: sim.touch("tS", f"group load S, dP {j}"))
            yield ("do", s_empty.arrive)
            yield ("delay", sim.rnd.uniform(0.3, 1.0))
            yield ("do", lambda j=j: sim.touch(f"tDS{j & 1}", f"group store dS {j}"))
            yield ("do", p_full.arrive)
        yield ("wait", done, 0, "group done")

    return sim.run({"producer": producer(), "mma": mma(), "group": group()},
                   lambda: done.done >= 1, 60 * (n + 5))


def fwd(qt0, ntile, seed, misplace=False):
    """Forward at hd 128, two query tiles per CTA: the MMA thread waits only
    on p_full_t and commits s_full_t (and p_empty_t after a tile's last P V);
    each softmax group checks V j and K j + 1 landed before waiting for
    S_t(j), and on S_t(j) frees K j and V j - 1 (P_t(j-1) V ran before it)."""
    sim = Sim(seed)
    stages = {}
    nkv = [qt0 + 1, qt0 + 2 if ntile == 2 else 0]
    n_kv = max(nkv)
    q_full = Bar("q_full", 1)
    k_full = [Bar(f"k_full{i}", 1) for i in range(3)]
    v_full = [Bar(f"v_full{i}", 1) for i in range(2)]
    k_empty = [Bar(f"k_empty{i}", ntile) for i in range(3)]
    v_empty = [Bar(f"v_empty{i}", ntile) for i in range(2)]
    s_full = [Bar(f"s_full{t}", 1) for t in range(2)]
    p_full = [Bar(f"p_full{t}", 1) for t in range(2)]
    p_last = [Bar(f"p_empty{t}", 1) for t in range(2)]

    def producer():
        yield ("do", lambda: sim.sched(sim.rnd.uniform(1, 3), q_full.arrive))
        for j in range(n_kv + 1):
            if j < n_kv:
                yield ("wait", k_empty[j % 3], j // 3 - 1, f"producer K stage for {j}")
                yield ("do", lambda j=j: sim.load(stages, ("K", j % 3), j, k_full[j % 3]))
            if j > 0:
                yield ("wait", v_empty[(j - 1) % 2], (j - 1) // 2 - 1, f"producer V stage for {j - 1}")
                yield ("do", lambda j=j: sim.load(stages, ("V", (j - 1) % 2), j - 1, v_full[(j - 1) % 2]))

    def mma():
        yield ("wait", q_full, 0, "mma Q")
        yield ("wait", k_full[0], 0, "mma K0")
        for t in range(2):
            if nkv[t] > 0:
                yield ("do", lambda t=t: sim.product(f"S{t},0", [(stages, ("K", 0), 0)], writes=f"tS{t}"))
                yield ("do", lambda t=t: sim.commit(s_full[t]))
        for j in range(n_kv):
            for t in range(2):
                if j >= nkv[t]:
                    continue
                yield ("wait", p_full[t], j, f"mma p_full {t},{j}")
                yield ("do", lambda t=t, j=j: sim.product(f"PV{t},{j}", [(stages, ("V", j % 2), j)],
                                                          tmem_reads=f"tS{t}"))
                if j + 1 < nkv[t]:
                    yield ("do", lambda t=t, j=j: sim.product(f"S{t},{j + 1}", [(stages, ("K", (j + 1) % 3), j + 1)],
                                                              writes=f"tS{t}"))
                    yield ("do", lambda t=t: sim.commit(s_full[t]))
                else:
                    yield ("do", lambda t=t: sim.commit(p_last[t]))

    def group(t):
        nk = nkv[t]
        for j in range(nk):
            yield ("wait", v_full[j % 2], j // 2, f"group {t} V {j}")
            if j + 1 < nk:
                yield ("wait", k_full[(j + 1) % 3], (j + 1) // 3, f"group {t} K {j + 1}")
            yield ("wait", s_full[t], j, f"group {t} s_full {j}")
            rel = (j + 1) % 3 if misplace else j % 3
            yield ("do", lambda rel=rel: k_empty[rel].arrive())
            if j > 0:
                yield ("do", lambda j=j: v_empty[(j - 1) % 2].arrive())
            yield ("do", lambda j=j: sim.touch(f"tS{t}", f"group {t} load S{j}"))
            yield ("delay", sim.rnd.uniform(0.3, 1.2))
            yield ("do", lambda j=j: sim.touch(f"tS{t}", f"group {t} store P{j}"))
            yield ("do", p_full[t].arrive)
        if nk > 0:
            yield ("wait", p_last[t], 0, f"group {t} last P V")

    tiles = [t for t in range(2) if nkv[t] > 0]
    return sim.run({"producer": producer(), "mma": mma(), "g0": group(0), "g1": group(1)},
                   lambda: all(p_last[t].done >= 1 for t in tiles), 80 * (n_kv + 5))


@pytest.mark.parametrize("total", [1, 2, 3, 5, 8, 13])
def test_dkdv_protocol(total):
    for seed in range(40):
        assert dkdv(total, seed) == [], (total, seed)


@pytest.mark.parametrize("n,ks,vs", [(1, 3, 2), (2, 3, 2), (5, 3, 2), (13, 3, 2), (3, 4, 4), (9, 4, 4)])
def test_dq_protocol(n, ks, vs):
    for seed in range(40):
        assert dq(n, seed, ks, vs) == [], (n, ks, vs, seed)


@pytest.mark.parametrize("qt0,ntile", [(0, 1), (0, 2), (2, 1), (2, 2), (6, 2), (10, 2)])
def test_forward_protocol(qt0, ntile):
    for seed in range(40):
        assert fwd(qt0, ntile, seed) == [], (qt0, ntile, seed)


def test_misplaced_releases_are_caught():
    """Each model fails when one release goes to the wrong slot or stage."""
    assert any(dkdv(5, seed, misplace=True) for seed in range(20))
    assert any(dq(6, seed, misplace=True) for seed in range(20))
    assert any(fwd(4, 2, seed, misplace=True) for seed in range(20))
