"""A CPU model of the barrier protocol of the GDN verify kernel
(csrc/gdn_state.cu): its two warpgroups (the state-splitting warpgroup, which
issues the copies and the state products, and the four row warps, of which
warp 0 issues the Gram and output products and warps 0/1 build the weights),
its buffers (the state staging tile, the K/Q tile, two v buffers, two P^T
buffers in tensor memory, the Gram rows, the weights, the write-vector and
output columns) and its mbarriers, with the hardware's parity-wait semantics.
Copies and MMAs complete after random delays (MMAs in issue order); every
role's work takes a random time.

Checked over random item counts and delays:
  * no wait is ever two phases behind its barrier (the parity wait would then
    hang until its bound);
  * no buffer is overwritten while a copy, an MMA or a warp still reads it;
  * no deadlock.
The earlier rule -- item k's products waiting only for item k - 2's P^T
buffer -- lets the products barrier run two phases ahead of a slow row warp,
and must be caught.
"""
import heapq
import random

import pytest


class Aliased(Exception):
    pass


class Hazard(Exception):
    pass


class Bar:
    def __init__(self, count):
        self.count, self.pending, self.n = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.n += 1
            self.pending = self.count


def run(n_items, seed, old_rule=False):
    rnd = random.Random(seed)
    bars = {b: Bar(1) for b in ("KQ", "ST", "PROD", "GRAM", "O")}
    bars["REL0"], bars["REL1"] = Bar(4), Bar(4)
    heap, seq, now = [], [0], [0.0]
    mma_done_at = [0.0]
    # buffer bookkeeping: the item each buffer holds and its pending readers
    done = {}                          # (what, item) -> True once finished

    def at(t, fn):
        seq[0] += 1
        heapq.heappush(heap, (t, seq[0], fn))

    def dly(a=0.2, b=3.0):
        return rnd.uniform(a, b)

    def mma(finish):                   # MMAs complete in issue order
        t = max(now[0] + dly(0.1, 1.0), mma_done_at[0] + 0.01)
        mma_done_at[0] = t
        at(t, finish)

    def need(key, what):
        if not done.get(key):
            raise Hazard(f"{what}: {key} not finished at t={now[0]:.2f}")

    # ---- roles as generators yielding ("wait", bar, completion), ("sleep", dt),
    # ("sync", group) -----------------------------------------------------------------
    def issue_copies(k):               # the state and K/Q/v copies of item k
        if k >= 1:
            need(("convert", k - 1), f"state copy {k}")
            need(("prod", k - 1), f"state copy {k}")
            need(("gram", k - 1), f"K/Q copy {k}")
        if k >= 2:
            for w in range(4):         # v buffer k & 1 held item k - 2's rows
                need(("uinit", k - 2, w), f"v copy {k}")

        def land_st():
            done[("st", k)] = True
            bars["ST"].arrive()

        def land_kq():
            done[("kq", k)] = True
            bars["KQ"].arrive()
        at(now[0] + dly(1.0, 4.0), land_st)
        at(now[0] + dly(0.5, 3.0), land_kq)

    def wg1():
        for k in range(n_items):
            yield ("wait", "ST", k)
            for kh in range(2):
                yield ("sleep", dly())
                if kh == 0:
                    if old_rule:
                        if k >= 2:
                            yield ("wait", f"REL{k & 1}", (k - 2) >> 1)
                    elif k >= 1:
                        yield ("wait", f"REL{(k - 1) & 1}", (k - 1) >> 1)
                    yield ("wait", "KQ", k)
                    if k >= 2:
                        for w in range(4):     # P^T buffer k & 1 held item k - 2
                            need(("ptload", k - 2, w), f"products {k}")
            done[("convert", k)] = True

            def fin(k=k):
                done[("prod", k)] = True
                bars["PROD"].arrive()
            mma(fin)
            if k + 1 < n_items:
                yield ("wait", "PROD", k)
                yield ("wait", "GRAM", k)
                if k >= 1:
                    yield ("wait", f"REL{(k - 1) & 1}", (k - 1) >> 1)
                issue_copies(k + 1)

    def row(w):
        for k in range(n_items):
            if w == 0:
                yield ("wait", "KQ", k)
                if k >= 1:
                    need(("weights", k - 1), f"Gram {k}")

                def fin(k=k):
                    done[("gram", k)] = True
                    bars["GRAM"].arrive()
                mma(fin)
            if w < 2:
                yield ("wait", "GRAM", k)
                yield ("sleep", dly(0.2, 4.0))     # weights (a slow warp at times)
                done[("weights", k)] = True
            yield ("wait", "PROD", k)
            yield ("sync", ("weights", k))
            need(("prod", k), f"rows {k}")
            need(("kq", k), f"v of {k}")
            done[("uinit", k, w)] = True
            yield ("sleep", dly())                  # recursion
            if k >= 1:
                need(("o", k - 1), f"write vectors {k}")
            done[("ptload", k, w)] = True
            bars[f"REL{k & 1}"].arrive()
            yield ("sync", ("c", k))
            if w == 0:
                for v in range(4):
                    if k >= 1:
                        need(("oread", k - 1, v), f"output products {k}")

                def fin(k=k):
                    done[("o", k)] = True
                    bars["O"].arrive()
                mma(fin)
            yield ("wait", "O", k)
            done[("oread", k, w)] = True
            yield ("sleep", dly(0.1, 1.0))
            yield ("sync", ("end", k))

    agents = {"wg1": wg1()}
    for w in range(4):
        agents[f"w{w}"] = row(w)
    state = {a: None for a in agents}          # what each agent waits for
    syncs = {}

    def step(a):
        try:
            state[a] = next(agents[a])
        except StopIteration:
            state[a] = ("exit",)

    bars["KQ"].n, bars["ST"].n = 0, 0
    issue_copies(0)
    for a in agents:
        step(a)
    for _ in range(200000):
        progressed = False
        for a in list(agents):
            s = state[a]
            if s[0] == "wait":
                n = bars[s[1]].n
                if n >= s[2] + 2:
                    raise Aliased(f"{a} waits for {s[1]} #{s[2]} but it is at {n}")
                if n >= s[2] + 1:
                    step(a)
                    progressed = True
            elif s[0] == "sync":
                members = syncs.setdefault(s[1], set())
                members.add(a)
                if len(members) == 4:
                    for m in members:
                        step(m)
                    progressed = True
            elif s[0] == "sleep":
                state[a] = ("timer",)
                at(now[0] + s[1], lambda a=a: step(a))
                progressed = True
        if all(state[a][0] == "exit" for a in agents):
            return now[0]
        if not progressed:
            if not heap:
                raise RuntimeError(f"deadlock: {state}")
            t, _, fn = heapq.heappop(heap)
            now[0] = t
            fn()
    raise RuntimeError("did not finish")


@pytest.mark.parametrize("n_items", [1, 2, 3, 5, 9])
def test_protocol_holds(n_items):
    for seed in range(300):
        run(n_items, seed)


def test_earlier_products_rule_is_caught():
    with pytest.raises(Aliased):
        for seed in range(3000):
            run(6, seed, old_rule=True)
