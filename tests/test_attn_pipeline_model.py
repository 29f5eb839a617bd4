"""A CPU model of the barrier protocol of the persistent tensor-core attention
partial (csrc/attn_tree_tc.cu): its roles (the K/Q loader, the V loader, the
MMA issuer, the softmax warps), its rings (two K stages, three V stages, two S
and two P buffers, one Q tile, one O accumulator) and its mbarriers, with the
hardware's parity-wait semantics.  TMA copies and MMAs complete after random
delays; the roles interleave at random.

Checked over random unit sequences (a CTA's units of 1..16 key blocks):
  * no wait is ever two phases behind its barrier (a parity wait would then
    hang until its bound);
  * no buffer is overwritten while an MMA or a copy still reads it, and every
    consumer sees the block it expects (S_j, P_j, V_j, K_j, the unit's Q);
  * O is rescaled only when no PV product is in flight, and each unit's
    epilogue reads O after its last PV product;
  * no deadlock.
The variant with one PFULL barrier for both P buffers (a parity wait that
falls two phases behind when the softmax writes P_{j+1} before the MMA issuer
has seen P_j) must be caught.
"""
import random

import pytest


class Bar:
    """An mbarrier: `count` arrivals (plus transaction bytes) complete a phase."""

    def __init__(self, count):
        self.count = count
        self.pending = count
        self.tx = 0
        self.n = 0                     # completed phases

    def arrive(self):
        self.pending -= 1
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.n += 1
            self.pending = self.count


class Aliased(Exception):
    pass


def run(units, seed, split_pfull=True, NKS=2, NVS=3):
    rnd = random.Random(seed)
    names = (["Q", "QE", "PF0", "PF1", "PVD0", "PVD1", "SF0", "SF1", "SR0", "SR1"]
             + [f"KF{i}" for i in range(NKS)] + [f"KE{i}" for i in range(NKS)]
             + [f"VF{i}" for i in range(NVS)] + [f"VE{i}" for i in range(NVS)])
    bar = {n: Bar(1) for n in names}
    events = []                        # (time, action)
    now = [0]
    buf = {}                           # buffer -> content tag
    reading = {}                       # buffer -> in-flight async readers
    mma_queue = []                     # MMAs complete in issue order
    done_mmas = [0]
    stuck = []

    def later(fn):
        events.append((now[0] + rnd.randint(1, 30), fn))

    def wait(name, phase):
        b = bar[name]

        def ready():
            if b.n >= phase + 2 and (b.n - phase) % 2 == 0:
                stuck.append((name, phase, b.n))
            return b.n > phase and (b.n & 1) != (phase & 1)
        return ready

    def tma(name, target, tag):
        b = bar[name]
        assert reading.get(target, 0) == 0, f"copy into {target} while it is read"
        b.tx += 1
        b.pending -= 1

        def land():
            buf[target] = tag
            b.tx -= 1
            b._check()
        later(land)

    def mma(reads, writes):
        for r in reads:
            reading[r] = reading.get(r, 0) + 1

        def complete():
            for r in reads:
                reading[r] -= 1
            for w, tag in writes:
                buf[w] = tag
            done_mmas[0] += 1
        mma_queue.append(complete)

        def fire():
            mma_queue.pop(0)()
        later(fire)

    def commit(name):
        b = bar[name]
        b.pending -= 1
        target = done_mmas[0] + len(mma_queue)

        def poll():
            if done_mmas[0] >= target:
                b._check()
            else:
                events.append((now[0] + 1, poll))
        events.append((now[0] + 1, poll))

    blocks = [(k, j, nb) for k, nb in enumerate(units) for j in range(nb)]
    nj = len(blocks)
    pf = (lambda J: (f"PF{J & 1}", J >> 1)) if split_pfull else (lambda J: ("PF0", J))
    if not split_pfull:
        bar["PF0"] = Bar(1)
    vconv = [None] * NVS

    def k_loader():
        J = 0
        for k, nb in enumerate(units):
            for j in range(nb):
                s = J % NKS
                if J >= NKS:
                    yield wait(f"KE{s}", J // NKS - 1)
                tma(f"KF{s}", f"K{s}", ("K", J))
                if j == 0:
                    if k >= 1:
                        yield wait("QE", k - 1)
                    tma("Q", "Q", ("Q", k))
                J += 1

    def v_loader():
        for J in range(nj):
            s = J % NVS
            if J >= NVS:
                yield wait(f"VE{s}", J // NVS - 1)
            tma(f"VF{s}", f"V{s}", ("V", J))

    def mma_issuer():
        cur = {"JS": 0}

        def issue_s():
            JS = cur["JS"]
            k, j, nb = blocks[JS]
            s, ks = JS & 1, JS % NKS
            if j == 0:
                yield wait("Q", k)
            yield wait(f"KF{ks}", JS // NKS)
            if JS >= 2:
                yield wait(f"SR{s}", (JS >> 1) - 1)
            assert buf.get("Q") == ("Q", k) and buf.get(f"K{ks}") == ("K", JS)
            mma(["Q", f"K{ks}"], [(f"S{s}", ("S", JS))])
            commit(f"SF{s}")
            commit(f"KE{ks}")
            if j == nb - 1:
                commit("QE")
            cur["JS"] += 1

        def catch_up(done):
            while cur["JS"] < nj and cur["JS"] <= done + 2:
                if blocks[cur["JS"]][1] == 0 and cur["JS"] == done + 2:
                    break              # a unit's first S waits until the PV before it is issued
                yield from issue_s()

        yield from catch_up(-1)
        for J in range(nj):
            k, j, nb = blocks[J]
            yield wait(*pf(J))
            assert buf.get(f"P{J & 1}") == ("P", J) and vconv[J % NVS] == J
            # the accumulation reads O as well (the first product of a unit
            # overwrites it, after the previous unit's epilogue)
            mma([f"P{J & 1}", f"V{J % NVS}", "O"], [("O", ("O", k, j))])
            commit(f"PVD{J & 1}")
            commit(f"VE{J % NVS}")
            yield from catch_up(J)

    def softmax():
        J = 0
        for k, nb in enumerate(units):
            for j in range(nb):
                s = J & 1
                yield wait(f"SF{s}", J >> 1)
                assert buf.get(f"S{s}") == ("S", J)
                bar[f"SR{s}"].arrive()
                vs = J % NVS
                yield wait(f"VF{vs}", J // NVS)
                assert buf.get(f"V{vs}") == ("V", J) and reading.get(f"V{vs}", 0) == 0
                vconv[vs] = J
                if J >= 2:
                    yield wait(f"PVD{J & 1}", (J >> 1) - 1)
                if j >= 1 and rnd.random() < 0.3:       # a rescale of O
                    yield wait(f"PVD{(J - 1) & 1}", (J - 1) >> 1)
                    assert buf.get("O") == ("O", k, j - 1) and reading.get("O", 0) == 0
                assert reading.get(f"P{J & 1}", 0) == 0, "P overwritten while read"
                buf[f"P{J & 1}"] = ("P", J)
                name, _ = pf(J)
                bar[name].arrive()
                J += 1
            yield wait(f"PVD{(J - 1) & 1}", (J - 1) >> 1)
            assert buf.get("O") == ("O", k, nb - 1), "epilogue before the last PV"

    roles = [k_loader(), v_loader(), mma_issuer(), softmax()]
    conds = []
    alive = []
    for r in roles:
        try:
            conds.append(next(r))
            alive.append(True)
        except StopIteration:
            conds.append(None)
            alive.append(False)
    for _ in range(400000):
        if stuck:
            raise Aliased(stuck[0])
        if not any(alive):
            return
        order = list(range(len(roles)))
        rnd.shuffle(order)
        progressed = False
        for i in order:
            if alive[i] and conds[i]():
                try:
                    conds[i] = next(roles[i])
                except StopIteration:
                    alive[i] = False
                progressed = True
                break
        if not progressed:
            if not events:
                raise AssertionError("deadlock")
            events.sort(key=lambda e: e[0])
            t, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
    raise AssertionError("no progress")


def _cases(n):
    for seed in range(n):
        r = random.Random(seed)
        yield seed, [r.choice([1, 1, 2, 3, 5, 16]) for _ in range(r.randint(0, 8))]


def test_pipeline_protocol_holds():
    for seed, units in _cases(400):
        run(units, seed)


@pytest.mark.parametrize("nks,nvs", [(3, 2), (2, 2), (3, 3)])
def test_pipeline_protocol_holds_for_other_ring_depths(nks, nvs):
    for seed, units in _cases(150):
        run(units, seed, NKS=nks, NVS=nvs)


def test_one_pfull_barrier_for_two_p_buffers_is_caught():
    caught = 0
    for seed, units in _cases(200):
        try:
            run(units, seed, split_pfull=False)
        except Aliased:
            caught += 1
    assert caught > 0
