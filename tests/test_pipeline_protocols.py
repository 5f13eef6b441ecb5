"""Barrier protocols of the backward, Based and GEMM kernels, checked on the CPU.

Each kernel role (TMA producer, MMA issuer, elementwise warps) is replayed
as the sequence of mbarrier operations its source performs, in the same
order, under many random interleavings and completion delays:

  wait(bar, k)   block until phase k of `bar` has completed
  arrive(bar)    one arrival (phase completes when all expected arrivals are in)
  commit(bar)    asynchronous arrival when everything issued before it has
                 finished: tensor-core commits and TMA completions land later,
                 in issue order per issuing thread

Two properties are asserted:
  - every role finishes (no deadlock);
  - when a role starts waiting for phase k, the barrier has completed at most
    k + 1 phases.  A hardware wait sees only the phase parity, so a barrier
    two phases ahead of its waiter would look incomplete to it.

GPU race detection (compute-sanitizer) is not available here; this checks
the protocol design, not the hardware.
"""
import random

import pytest


class Barrier:
    def __init__(self, name, count=1):
        self.name, self.count, self.arrived, self.completed = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1


class Sim:
    def __init__(self, seed):
        self.rng = random.Random(seed)
        self.bars = {}
        self.pending = []  # (ready_time, seq, barrier) asynchronous arrivals
        self.seq = 0
        self.now = 0
        self.last_ready = {}  # issuer -> ready time of its last async op (in-order landing)

    def bar(self, name, count=1):
        if name not in self.bars:
            self.bars[name] = Barrier(name, count)
        return self.bars[name]

    def run(self, roles):
        state = {name: None for name in roles}  # pending wait per role
        live = dict(roles)
        while live or self.pending:
            choices = [n for n in live if state[n] is None or
                       self.bars[state[n][0]].completed > state[n][1]]
            if self.pending and (not choices or self.rng.random() < 0.3):
                self.pending.sort()
                _, _, b = self.pending.pop(0)
                self.bars[b].arrive()
                continue
            if not choices:
                stuck = {n: state[n] for n in live}
                raise AssertionError(f"deadlock: {stuck}")
            name = self.rng.choice(choices)
            gen = live[name]
            state[name] = None
            while True:
                try:
                    op = next(gen)
                except StopIteration:
                    del live[name]
                    break
                kind = op[0]
                self.now += 1
                if kind == "wait":
                    b, k = op[1], op[2]
                    done = self.bars[b].completed
                    assert done <= k + 1, (
                        f"{name}: waits for phase {k} of {b}, which has completed {done}")
                    if done <= k:
                        state[name] = (b, k)
                        break
                elif kind == "arrive":
                    self.bars[op[1]].arrive()
                elif kind == "commit":
                    issuer = op[2] if len(op) > 2 else name
                    t = max(self.now + self.rng.randint(1, 40), self.last_ready.get(issuer, 0))
                    self.last_ready[issuer] = t
                    self.seq += 1
                    self.pending.append((t, self.seq, op[1]))


def based_roles(sim, units, S=8, NB=3):
    """tk_based_fwd_kernel: units = list of step counts n (one CTA)."""
    sim.bar("fix_full"), sim.bar("fix_empty"), sim.bar("acc_full"), sim.bar("lsum")
    sim.bar("acc_empty")
    for s in range(S):
        sim.bar(f"kv_full{s}"), sim.bar(f"kv_empty{s}")
    for b in range(NB):
        sim.bar(f"s_full{b}"), sim.bar(f"p_full{b}")

    def producer():
        it = 0
        for uc, n in enumerate(units):
            if uc > 0:
                yield ("wait", "fix_empty", uc - 1)
            yield ("commit", "fix_full", "tma")
            for _ in range(n):
                s = it % S
                if it >= S:
                    yield ("wait", f"kv_empty{s}", it // S - 1)
                yield ("commit", f"kv_full{s}", "tma")
                it += 1

    def mma():
        it = 0
        for uc, n in enumerate(units):
            yield ("wait", "fix_full", uc)
            for j in range(min(NB, n)):
                yield ("wait", f"kv_full{(it + j) % S}", (it + j) // S)
                yield ("commit", f"s_full{(it + j) % NB}")
                if j == n - 1:
                    yield ("commit", "fix_empty")
            if uc > 0:
                yield ("wait", "acc_empty", uc - 1)
            for j in range(n):
                yield ("wait", f"p_full{it % NB}", it // NB)
                yield ("commit", f"kv_empty{it % S}")
                if j + NB < n:
                    yield ("wait", f"kv_full{(it + NB) % S}", (it + NB) // S)
                    yield ("commit", f"s_full{(it + NB) % NB}")
                    if j + NB + 1 == n:
                        yield ("commit", "fix_empty")
                it += 1
            yield ("commit", "acc_full")

    def warps():
        it = 0
        for uc, n in enumerate(units):
            for _ in range(n):
                yield ("wait", f"s_full{it % NB}", it // NB)
                yield ("arrive", f"p_full{it % NB}")
                it += 1
            yield ("arrive", "lsum")
            yield ("wait", "lsum", uc)
            yield ("wait", "acc_full", uc)
            yield ("arrive", "acc_empty")

    return {"producer": producer(), "mma": mma(), "warps": warps()}


def dq_roles(sim, units, KS=3, VS=2):
    """tk_attn_bwd_dq_kernel (second S buffer, separate K and V rings)."""
    for b in ("fix_full", "fix_empty", "s_full", "p_full", "acc_full", "acc_empty"):
        sim.bar(b)
    for s in range(KS):
        sim.bar(f"k_full{s}"), sim.bar(f"k_empty{s}")
    for s in range(VS):
        sim.bar(f"v_full{s}"), sim.bar(f"v_empty{s}")

    def producer():
        it = 0
        for uc, n in enumerate(units):
            if uc > 0:
                yield ("wait", "fix_empty", uc - 1)
            yield ("commit", "fix_full", "tma")
            for _ in range(n):
                if it >= KS:
                    yield ("wait", f"k_empty{it % KS}", it // KS - 1)
                yield ("commit", f"k_full{it % KS}", "tma")
                if it >= VS:
                    yield ("wait", f"v_empty{it % VS}", it // VS - 1)
                yield ("commit", f"v_full{it % VS}", "tma")
                it += 1

    def mma():
        it = 0
        for uc, n in enumerate(units):
            yield ("wait", "fix_full", uc)
            yield ("wait", f"k_full{it % KS}", it // KS)
            yield ("wait", f"v_full{it % VS}", it // VS)
            yield ("commit", "s_full")
            yield ("commit", f"v_empty{it % VS}")
            if n == 1:
                yield ("commit", "fix_empty")
            if uc > 0:
                yield ("wait", "acc_empty", uc - 1)
            for j in range(n):
                more = j + 1 < n
                if more:
                    yield ("wait", f"k_full{(it + 1) % KS}", (it + 1) // KS)
                yield ("wait", "p_full", it)
                yield ("commit", f"k_empty{it % KS}")
                if more:
                    yield ("wait", f"v_full{(it + 1) % VS}", (it + 1) // VS)
                    yield ("commit", "s_full")
                    yield ("commit", f"v_empty{(it + 1) % VS}")
                    if j + 2 == n:
                        yield ("commit", "fix_empty")
                it += 1
            yield ("commit", "acc_full")

    def warps():
        it = 0
        for uc, n in enumerate(units):
            for _ in range(n):
                yield ("wait", "s_full", it)
                yield ("arrive", "p_full")
                it += 1
            yield ("wait", "acc_full", uc)
            yield ("arrive", "acc_empty")

    return {"producer": producer(), "mma": mma(), "warps": warps()}


def dkdv_roles(sim, units, S=2):
    """tk_attn_bwd_dkdv_kernel (two halves per step: P^T, then dS^T)."""
    for b in ("fix_full", "fix_empty", "s_full", "p_full", "dp_full", "ds_full", "acc_full",
              "acc_empty"):
        sim.bar(b)
    for s in range(S):
        sim.bar(f"ring_full{s}"), sim.bar(f"ring_empty{s}")

    def producer():
        it = 0
        for uc, n in enumerate(units):
            if uc > 0:
                yield ("wait", "fix_empty", uc - 1)
            yield ("commit", "fix_full", "tma")
            for _ in range(n):
                if it >= S:
                    yield ("wait", f"ring_empty{it % S}", it // S - 1)
                yield ("commit", f"ring_full{it % S}", "tma")
                it += 1

    def mma():
        it = 0
        for uc, n in enumerate(units):
            yield ("wait", "fix_full", uc)
            yield ("wait", f"ring_full{it % S}", it // S)
            yield ("commit", "s_full")
            yield ("commit", "dp_full")
            if n == 1:
                yield ("commit", "fix_empty")
            if uc > 0:
                yield ("wait", "acc_empty", uc - 1)
            for st in range(n):
                yield ("wait", "p_full", it)
                more = st + 1 < n
                if more:
                    yield ("wait", f"ring_full{(it + 1) % S}", (it + 1) // S)
                    yield ("commit", "s_full")
                yield ("wait", "ds_full", it)
                yield ("commit", f"ring_empty{it % S}")
                if more:
                    yield ("commit", "dp_full")
                    if st + 2 == n:
                        yield ("commit", "fix_empty")
                it += 1
            yield ("commit", "acc_full")

    def warps():
        it = 0
        for uc, n in enumerate(units):
            for _ in range(n):
                yield ("wait", "s_full", it)
                yield ("wait", f"ring_full{it % S}", it // S)
                yield ("arrive", "p_full")
                yield ("wait", "dp_full", it)
                yield ("arrive", "ds_full")
                it += 1
            yield ("wait", "acc_full", uc)
            yield ("arrive", "acc_empty")

    return {"producer": producer(), "mma": mma(), "warps": warps()}


def gemm_pair_roles(sim, tiles, k_blocks, S=6):
    """tk_gemm_kernel, one CTA pair: both CTAs' producers, the first CTA's MMA
    thread, both CTAs' epilogues and TMEM-release waits.  `full` lives in the
    first CTA and completes on that CTA's expect-tx arrival plus both CTAs'
    copies; MMA commits multicast to both CTAs' barriers."""
    for s_ in range(S):
        sim.bar(f"full{s_}", 3)
        for r in range(2):
            sim.bar(f"empty{r}_{s_}")
    for b in range(2):
        sim.bar(f"acc_empty{b}", 2)
        for r in range(2):
            sim.bar(f"acc_full{r}_{b}")
    for r in range(2):
        sim.bar(f"mma_done{r}")

    def producer(r):
        it = 0
        for _ in range(tiles):
            for _ in range(k_blocks):
                s_ = it % S
                if it >= S:
                    yield ("wait", f"empty{r}_{s_}", it // S - 1)
                if r == 0:
                    yield ("arrive", f"full{s_}")
                yield ("commit", f"full{s_}", f"tma{r}")
                it += 1
        for s_ in range(min(S, it)):  # the last commits on this CTA's stages
            last = it - 1 - ((it - 1 - s_) % S)
            yield ("wait", f"empty{r}_{s_}", last // S)

    def mma():
        it = 0
        for tc in range(tiles):
            b = tc & 1
            if tc >= 2:
                yield ("wait", f"acc_empty{b}", (tc >> 1) - 1)
            for _ in range(k_blocks):
                yield ("wait", f"full{it % S}", it // S)
                yield ("commit", f"empty0_{it % S}")
                yield ("commit", f"empty1_{it % S}")
                it += 1
            yield ("commit", f"acc_full0_{b}")
            yield ("commit", f"acc_full1_{b}")
        for i in range(max(0, tiles - 2), tiles):
            yield ("wait", f"acc_empty{i & 1}", i >> 1)
        yield ("commit", "mma_done0")
        yield ("commit", "mma_done1")

    def epilogue(r):
        for tc in range(tiles):
            yield ("wait", f"acc_full{r}_{tc & 1}", tc >> 1)
            yield ("arrive", f"acc_empty{tc & 1}")

    def release(r):
        yield ("wait", f"mma_done{r}", 0)

    return {"prod0": producer(0), "prod1": producer(1), "mma": mma(), "epi0": epilogue(0),
            "epi1": epilogue(1), "rel0": release(0), "rel1": release(1)}


@pytest.mark.parametrize("tiles,k_blocks", [(1, 1), (1, 7), (2, 3), (3, 1), (5, 4), (4, 13)])
def test_gemm_pair_protocol(tiles, k_blocks):
    for seed in range(60):
        sim = Sim(seed)
        sim.run(gemm_pair_roles(sim, tiles, k_blocks))


UNIT_LISTS = [[1], [2], [3], [4], [1, 1, 1], [5, 1, 2, 7], [3, 3], [1, 4, 1, 9, 2]]


@pytest.mark.parametrize("units", UNIT_LISTS, ids=lambda u: "-".join(map(str, u)))
@pytest.mark.parametrize("kernel", ["based", "dq", "dkdv"])
def test_protocol_completes_without_run_ahead(kernel, units):
    build = {"based": based_roles, "dq": dq_roles, "dkdv": dkdv_roles}[kernel]
    for seed in range(60):
        sim = Sim(seed)
        sim.run(build(sim, units))


def test_single_s_barrier_for_two_buffers_runs_ahead():
    """The hazard the per-buffer barriers exist for: with one s_full/p_full
    pair for two S buffers (the next step's S issued before the current
    step's P is consumed), the warps can complete two p_full phases before
    the MMA thread waits for the first."""

    def roles(sim, n=6):
        for b in ("s_full", "p_full"):
            sim.bar(b)

        def mma():
            yield ("commit", "s_full")
            yield ("commit", "s_full")
            for j in range(n):
                yield ("wait", "p_full", j)
                if j + 2 < n:
                    yield ("commit", "s_full")

        def warps():
            for j in range(n):
                yield ("wait", "s_full", j)
                yield ("arrive", "p_full")

        return {"mma": mma(), "warps": warps()}

    failures = 0
    for seed in range(200):
        sim = Sim(seed)
        try:
            sim.run(roles(sim))
        except AssertionError:
            failures += 1
    assert failures > 0
