"""Barrier protocols of the forward, backward, Based and GEMM kernels, checked on the CPU.

Each kernel role (TMA producer, MMA issuer, elementwise warps) is replayed
as the sequence of mbarrier operations its source performs, in the same
order, under many random interleavings and completion delays:

  wait(bar, k)   block until phase k of `bar` has completed
  arrive(bar)    one arrival (phase completes when all expected arrivals are in)
  commit(bar)    asynchronous arrival when everything issued before it has
                 finished: tensor-core commits and TMA completions land later,
                 in issue order per issuing thread
  check(bar, k)  a use of data that phase k of `bar` guards, without a wait of
                 its own (the role relies on another role's wait): phase k
                 must have completed already
  write(res, v) / read(res, v)
                 a plain shared-memory buffer handed from one role to another:
                 version v may only be written once version v - 1 was read

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

    def arrive(self, phase=None):
        # an arrival tagged with the phase it belongs to must land in that
        # phase: with several arrivers, one that runs a whole phase ahead
        # would otherwise complete a phase the others have not finished
        assert phase is None or phase == self.completed, (
            f"{self.name}: an arrival for phase {phase} lands in phase {self.completed}")
        self.arrived += 1
        if self.arrived == self.count:
            self.arrived = 0
            self.completed += 1


class Sim:
    def __init__(self, seed, preempt=0.25):
        self.rng = random.Random(seed)
        self.preempt = preempt
        self.bars = {}
        self.pending = []  # (ready_time, seq, barrier) asynchronous arrivals
        self.seq = 0
        self.now = 0
        self.last_ready = {}  # issuer -> ready time of its last async op (in-order landing)

    def bar(self, name, count=1):
        if name not in self.bars:
            self.bars[name] = Barrier(name, count)
        return self.bars[name]

    versions = None  # res -> (last version written, read yet)

    def run(self, roles):
        state = {name: None for name in roles}  # pending wait per role
        live = dict(roles)
        while live or self.pending:
            choices = [n for n in live if state[n] is None or
                       self.bars[state[n][0]].completed > state[n][1]]
            if self.pending and (not choices or self.rng.random() < 0.3):
                self.pending.sort()
                _, _, b, tag = self.pending.pop(0)
                self.bars[b].arrive(tag)
                continue
            if not choices:
                stuck = {n: state[n] for n in live}
                raise AssertionError(f"deadlock: {stuck}")
            name = self.rng.choice(choices)
            gen = live[name]
            state[name] = None
            first = True
            while True:
                # a role may be descheduled between any two of its operations
                if not first and self.rng.random() < self.preempt:
                    break
                first = False
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
                    self.bars[op[1]].arrive(op[2] if len(op) > 2 else None)
                elif kind == "check":
                    b, k = op[1], op[2]
                    assert self.bars[b].completed > k, (
                        f"{name}: uses data of phase {k} of {b}, which has completed "
                        f"{self.bars[b].completed}")
                elif kind in ("write", "read"):
                    if self.versions is None:
                        self.versions = {}
                    res, v = op[1], op[2]
                    last, seen = self.versions.get(res, (-1, True))
                    if kind == "write":
                        # versions may skip (a unit that leaves the buffer
                        # unused); the one written before must have been read
                        assert v > last and seen, (
                            f"{name}: writes version {v} of {res} while version {last} "
                            f"{'was' if seen else 'was not yet'} read")
                        self.versions[res] = (v, False)
                    else:
                        assert v == last and not seen, (
                            f"{name}: reads version {v} of {res}, which holds {last}")
                        self.versions[res] = (v, True)
                elif kind == "commit":
                    # ("commit", barrier[, issuer[, phase tag]])
                    issuer = op[2] if len(op) > 2 and op[2] is not None else name
                    tag = op[3] if len(op) > 3 else None
                    t = max(self.now + self.rng.randint(1, 40), self.last_ready.get(issuer, 0))
                    self.last_ready[issuer] = t
                    self.seq += 1
                    self.pending.append((t, self.seq, op[1], tag))


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


def dq_roles(sim, units, KS=3, VS=2, drop=()):
    """tk_attn_bwd_dq_kernel: two 128-column buffers, step j in buffer j mod
    2 (S_j, then dP_j over it once the warps hold S_j in registers, then bf16
    dS_j over dP_j), separate K and V rings.  Buffer contents are versioned:
    S_{j+2} may overwrite buffer b only after the dQ product has read dS_j,
    and dP_j only after the warps have read S_j."""
    for b in ("fix_full", "fix_empty", "s_full", "dp_full", "acc_full"):
        sim.bar(b)
    sim.bar("s_read", 1), sim.bar("ds_full", 1), sim.bar("acc_empty", 1)
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
        # In-order execution: a product's writes and reads take effect in
        # issue order, so the buffer versions are advanced at issue.
        it = 0
        for uc, n in enumerate(units):
            yield ("wait", "fix_full", uc)
            yield ("wait", f"k_full{it % KS}", it // KS)
            yield ("write", f"buf{it & 1}", 3 * it)        # S_it
            yield ("commit", "s_full", None, it)
            for j in range(n):
                if "s_read" not in drop:
                    yield ("wait", "s_read", it)
                yield ("wait", f"v_full{it % VS}", it // VS)
                yield ("write", f"buf{it & 1}", 3 * it + 1)    # dP_it over S_it
                yield ("commit", "dp_full", None, it)
                yield ("commit", f"v_empty{it % VS}", None, it // VS)
                if j + 1 == n:
                    yield ("commit", "fix_empty", None, uc)
                if j + 1 < n:
                    yield ("wait", f"k_full{(it + 1) % KS}", (it + 1) // KS)
                    yield ("write", f"buf{(it + 1) & 1}", 3 * (it + 1))   # S_{it+1}
                    yield ("commit", "s_full", None, it + 1)
                if j == 0 and uc > 0:
                    yield ("wait", "acc_empty", uc - 1)
                yield ("wait", "ds_full", it)
                yield ("read", f"buf{it & 1}", 3 * it + 2)     # dS_it, by dQ += dS K
                yield ("commit", f"k_empty{it % KS}", None, it // KS)
                it += 1
            yield ("commit", "acc_full", None, uc)

    def warps():
        it = 0
        for uc, n in enumerate(units):
            for _ in range(n):
                yield ("wait", "s_full", it)
                yield ("read", f"buf{it & 1}", 3 * it)
                yield ("arrive", "s_read", it)
                yield ("wait", "dp_full", it)
                yield ("read", f"buf{it & 1}", 3 * it + 1)
                yield ("write", f"buf{it & 1}", 3 * it + 2)    # dS over dP
                yield ("arrive", "ds_full", it)
                it += 1
            yield ("wait", "acc_full", uc)
            yield ("arrive", "acc_empty", uc)

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


def fwd_roles(sim, units, split_p, S=None, QB=None, single_fin=False, drop=(), half=False,
              idle0=False, half_shared_stages=False):
    """tk_attn_fwd_kernel (one CTA).  units = list of (n0, n1): the K/V steps
    of Q tile 0 and Q tile 1 of each unit (n1 = n0 + 1 for a causal diagonal
    block, n0 = n1 otherwise).  half: a launch of at most 128 queries (P split
    from S at either head dim), where tile 1 holds no query row in any unit:
    its softmax warps and MMA thread keep the barriers of their own tile
    (S, P, P V done, the final row statistics, O) but read no S, V or
    statistics, and neither wait for K/V or Q tiles nor release them; the
    stage and Q-buffer barriers take tile 0's commits alone, and no
    exponential turns are taken.  half_shared_stages replays the first
    version, where tile 1's thread still committed every stage release (a
    second arrival that can run a whole phase ahead).  idle0: tile 0's warps
    split into a working role and a role for the warps whose rows all lie
    past the last query, which keep the protocol with no waits for V and no
    final statistics; tile 0's 4-warp barriers then take one arrival from
    each.  split_p: head dim 64 (P in its own tensor
    memory columns, one MMA issuer per tile, exponential turns); otherwise
    head dim 128 (P over S, one issuer for both tiles).  single_fin replays
    the earlier one-buffer fin_full, and `drop` leaves out the softmax's
    wait for the converted V tile ("v_ready") or, with P over S, the MMA
    thread's wait for the K tile ("k_wait"), for the negative tests.

    The four softmax warps of a tile, and the four converter warps, act as one
    role each: their 4-arrival barriers are modelled with one arrival."""
    S = S or (8 if split_p else 4)
    QB = QB or (2 if split_p else 1)
    nissue = 2 if split_p and (not half or half_shared_stages) else 1
    if idle0:
        for name in ("s_free0", "p_full0", "fin_full0_0", "fin_full1_0"):
            sim.bar(name, 2)
    for t in range(2):
        for b in range(QB):
            sim.bar(f"q_full{b}_{t}")
        for name in ("s_full", "p_full", "o_full", "o_free", "s_free", "pv_done", "exp_turn"):
            sim.bar(f"{name}{t}")
        for par in range(2):
            sim.bar(f"fin_full{par}_{t}")
        sim.bar(f"mma_done{t}")
    for b in range(QB):
        sim.bar(f"q_empty{b}", nissue)
    for s_ in range(S):
        sim.bar(f"kv_full{s_}"), sim.bar(f"kv_empty{s_}", nissue), sim.bar(f"v_ready{s_}")
    sim.bar("conv_bar")
    sim.bars["exp_turn0"].completed = 1  # tile 0 takes the first turn (set at start-up)
    units = [tuple(u) + (half,) for u in units]

    def fin(uc, t):
        # double-buffered by unit parity; the earlier version had one buffer
        return (f"fin_full0_{t}", uc) if single_fin else (f"fin_full{uc & 1}_{t}", uc >> 1)

    def producer():
        kv_idx = 0
        for uc, (n0, n1, _) in enumerate(units):
            qb = uc % QB
            if uc >= QB:
                yield ("wait", f"q_empty{qb}", uc // QB - 1)
            yield ("commit", f"q_full{qb}_0", f"tma_q{qb}")
            yield ("commit", f"q_full{qb}_1", f"tma_q{qb}")
            for _ in range(n1):
                for _kv in range(2):
                    s_, fill = kv_idx % S, kv_idx // S
                    if fill > 0:
                        yield ("wait", f"kv_empty{s_}", fill - 1)
                    yield ("commit", f"kv_full{s_}", f"tma{s_}")  # loads land in any order
                    kv_idx += 1
        # load_exit: the last fill of every stage and the last load of each Q buffer
        for s_ in range(min(S, kv_idx)):
            last = kv_idx - 1 - ((kv_idx - 1 - s_) % S)
            yield ("wait", f"kv_full{s_}", last // S)
        nq = len(units)
        for b in range(min(QB, nq)):
            last = nq - 1 - ((nq - 1 - b) % QB)
            yield ("wait", f"q_full{b}_0", last // QB)
            yield ("wait", f"q_full{b}_1", last // QB)

    def softmax(t, idle_warps=False):
        steps = turns = kvb = 0
        s_waits = 0
        for uc, (n0, n1, idle1) in enumerate(units):
            n_t = n1 if t else n0
            idle = (t == 1 and idle1) or idle_warps
            for j in range(n_t):
                yield ("wait", f"s_full{t}", s_waits)
                s_waits += 1
                if split_p:
                    yield ("arrive", f"s_free{t}", s_waits - 1)
                take_turn = split_p and not idle1 and (t == 0 or j < n0)
                if take_turn:
                    yield ("wait", f"exp_turn{t}", turns)
                    turns += 1
                    yield ("arrive", f"exp_turn{t ^ 1}")
                if split_p:
                    if steps > 0:
                        yield ("wait", f"pv_done{t}", steps - 1)
                    steps += 1
                vidx = kvb + 2 * j + 1
                if "v_ready" not in drop and not idle:
                    yield ("wait", f"v_ready{vidx % S}", vidx // S)
                if j == n_t - 1 and not idle:
                    yield ("write", f"fin{uc & 1 if not single_fin else 0}_{t}",
                           uc >> 1 if not single_fin else uc)
                yield ("arrive", f"p_full{t}", s_waits - 1)
                if j == n_t - 1:
                    yield ("arrive", *fin(uc, t))
            kvb += 2 * n1

    def converter():
        kvb = conv = 0
        pend = None
        for uc in range(len(units) + 1):
            have = uc < len(units)
            n1 = units[uc][1] if have else 0
            for j in range(n1 + 1):
                if pend is not None and (j == 1 or not have):
                    for t in range(2):
                        bar, k = fin(pend, t)
                        yield ("wait", bar, k)
                        yield ("wait", f"o_full{t}", pend)
                        if not (t == 1 and units[pend][2]):
                            yield ("read", f"fin{pend & 1 if not single_fin else 0}_{t}",
                                   pend >> 1 if not single_fin else pend)
                        yield ("arrive", f"o_free{t}")
                    pend = None
                if j == n1:
                    break
                vidx = kvb + 2 * j + 1
                st = vidx % S
                yield ("wait", f"kv_full{st}", vidx // S)
                yield ("arrive", "conv_bar")  # the four warps agree on the tile's range
                yield ("wait", "conv_bar", conv)
                conv += 1
                yield ("arrive", f"v_ready{st}")
            if not have:
                break
            pend = uc
            kvb += 2 * n1

    def mma_split(t):
        p_cnt = s_cnt = kvb = 0
        for uc, (n0, n1, idle1) in enumerate(units):
            n_t = n1 if t else n0
            idle = t == 1 and idle1
            qb = uc % QB
            for j in range(n1 + 1):
                kidx = kvb + 2 * j
                vidx = kidx - 1
                ks, vs = kidx % S, vidx % S
                do_s, do_pv = j < n_t, 1 <= j <= n_t
                stages = not idle or half_shared_stages  # waits for and releases K/V, Q
                if do_s:
                    if stages:
                        yield ("wait", f"kv_full{ks}", kidx // S)
                    if j == 0 and stages:
                        yield ("wait", f"q_full{qb}_{t}", uc // QB)
                    if s_cnt > 0:
                        yield ("wait", f"s_free{t}", s_cnt - 1)
                    s_cnt += 1
                    yield ("commit", f"s_full{t}")
                if do_pv:
                    if j == 1 and uc > 0:
                        yield ("wait", f"o_free{t}", uc - 1)
                    yield ("wait", f"p_full{t}", p_cnt)
                    p_cnt += 1
                    if not idle:
                        yield ("check", f"v_ready{vs}", vidx // S)  # V_{j-1} converted
                    yield ("commit", f"pv_done{t}")
                    if j == n_t:
                        yield ("commit", f"o_full{t}")
                if j < n1 and stages:
                    yield ("commit", f"kv_empty{ks}", None, kidx // S)
                if j >= 1 and stages:
                    yield ("commit", f"kv_empty{vs}", None, vidx // S)
                if j == n1 - 1 and stages:
                    yield ("commit", f"q_empty{qb}", None, uc // QB)
            kvb += 2 * n1
        yield ("commit", f"mma_done{t}")
        yield ("wait", f"mma_done{t}", 0)

    def mma_shared():
        p_cnt = [0, 0]
        kvb = 0
        for uc, (n0, n1, idle1) in enumerate(units):
            for j in range(n1 + 1):
                kidx = kvb + 2 * j
                vidx = kidx - 1
                ks, vs = kidx % S, vidx % S
                k_ready = False
                for t in range(2):
                    n_t = n1 if t else n0
                    idle = t == 1 and idle1
                    do_pv, do_s = 1 <= j <= n_t, j < n_t
                    if do_pv:
                        if j == 1 and uc > 0:
                            yield ("wait", f"o_free{t}", uc - 1)
                        yield ("wait", f"p_full{t}", p_cnt[t])
                        p_cnt[t] += 1
                    if do_s:
                        if j == 0:
                            yield ("wait", f"q_full0_{t}", uc)
                        if not k_ready and "k_wait" not in drop:
                            yield ("wait", f"kv_full{ks}", kidx // S)
                        k_ready = True
                    if do_pv and not idle:
                        yield ("check", f"v_ready{vs}", vidx // S)  # V_{j-1} converted
                    if do_s:
                        if not idle:
                            yield ("check", f"kv_full{ks}", kidx // S)  # K_j landed
                        yield ("commit", f"s_full{t}")
                    if do_pv and j == n_t:
                        yield ("commit", f"o_full{t}")
                if j < n1:
                    yield ("commit", f"kv_empty{ks}", None, kidx // S)
                if j >= 1:
                    yield ("commit", f"kv_empty{vs}", None, vidx // S)
                if j == n1 - 1:
                    yield ("commit", "q_empty0", None, uc)
            kvb += 2 * n1
        yield ("commit", "mma_done0")
        yield ("wait", "mma_done0", 0)

    roles = {"producer": producer(), "softmax0": softmax(0), "softmax1": softmax(1),
             "converter": converter()}
    if idle0:
        roles["softmax0_idle"] = softmax(0, idle_warps=True)
    if split_p:
        roles["mma0"], roles["mma1"] = mma_split(0), mma_split(1)
    else:
        roles["mma"] = mma_shared()
    return roles


def based_linear_roles(sim, units, drop=()):
    """tk_based_linear_kernel (one CTA): units = chunk counts of its slices.
    Per chunk the MMA thread issues S_qk; the state update (before a slice's
    last chunk, once phi(K) is written and the copy warps hold the previous
    state); A V_ext once A is written and the previous y read; phi(Q) S_ext
    (past a slice's first chunk) once phi(Q) and the state copy are in.  The
    copy warps load the updated state, release it, and store the copy once
    the phi(Q) S_ext products issued before are done.  Versioned buffers:
    the two feature panels, the state copy in shared memory and the state in
    tensor memory."""
    for b in ("s_full", "p_full", "y_full0", "y_full1", "y_free0", "y_free1", "phik_full",
              "phik_empty", "phiq_full", "phiq_empty", "st_full", "st_read", "sx_full",
              "sext_free"):
        sim.bar(b)
    for st in range(2):
        sim.bar(f"in_full{st}"), sim.bar(f"in_empty{st}")

    def producer():
        it = 0
        for nc in units:
            for _ in range(nc):
                if it >= 2:
                    yield ("wait", f"in_empty{it & 1}", (it >> 1) - 1)
                yield ("commit", f"in_full{it & 1}", "tma")
                it += 1

    def mma():
        it = cv = ups = upw = dn = 0
        for nc in units:
            for c in range(nc):
                yield ("wait", f"in_full{it & 1}", it >> 1)
                yield ("commit", "s_full", None, it)
                yield ("wait", "phik_full", it)
                if c + 1 < nc:
                    if ups > upw:
                        yield ("wait", "st_read", upw)
                        upw += 1
                    yield ("read", "phik", it)
                    yield ("write", "state", ups)      # S^T (+)= V_ext^T phi(K)
                    yield ("commit", "st_full", None, ups)
                    ups += 1
                yield ("commit", "phik_empty", None, it)
                if it >= 2:  # the y of the chunk two back, the Y buffer's previous use
                    yield ("wait", f"y_free{it & 1}", (it >> 1) - 1)
                yield ("wait", "p_full", it)
                yield ("write", f"ybuf{it & 1}", it >> 1)
                yield ("wait", "phiq_full", it)
                if c > 0:
                    yield ("wait", "sx_full", cv)
                    yield ("read", "phiq", it)
                    yield ("read", "sext", cv)
                    cv += 1
                    yield ("commit", "sext_free", None, dn)
                    dn += 1
                yield ("commit", f"y_full{it & 1}", None, it >> 1)
                yield ("commit", "phiq_empty", None, it)
                yield ("commit", f"in_empty{it & 1}", None, it >> 1)
                it += 1

    def twarps():  # A of a chunk, then the y of the chunk before it
        def epilogue(e):
            yield ("wait", f"y_full{e & 1}", e >> 1)
            yield ("read", f"ybuf{e & 1}", e >> 1)
            yield ("arrive", f"y_free{e & 1}", e >> 1)
        it = 0
        for nc in units:
            for _ in range(nc):
                yield ("wait", "s_full", it)
                yield ("arrive", "p_full", it)
                if it > 0:
                    yield from epilogue(it - 1)
                it += 1
        if it > 0:
            yield from epilogue(it - 1)

    def features(kind):  # phi(K) and phi(Q) are built by warps of their own
        it = 0
        for nc in units:
            for c in range(nc):
                if it > 0:
                    yield ("wait", f"phi{kind}_empty", it - 1)
                if (c + 1 < nc) if kind == "k" else (c > 0):
                    yield ("write", f"phi{kind}", it)
                yield ("arrive", f"phi{kind}_full", it)
                it += 1

    def converter():
        cv = dseen = 0
        for nc in units:
            for c in range(nc - 1):
                yield ("wait", "st_full", cv)
                yield ("read", "state", cv)
                yield ("arrive", "st_read", cv)
                d = dseen + c
                if d > 0 and "sext_free" not in drop:
                    yield ("wait", "sext_free", d - 1)
                yield ("write", "sext", cv)
                yield ("arrive", "sx_full", cv)
                cv += 1
            dseen += nc - 1

    return {"producer": producer(), "mma": mma(), "twarps": twarps(),
            "features_k": features("k"), "features_q": features("q"), "converter": converter()}


FWD_UNITS = [
    [(1, 1)], [(1, 2)], [(2, 2)], [(4, 4)],
    [(1, 2), (1, 2), (1, 2)],              # single-step causal units, back to back
    [(1, 1), (1, 1), (1, 1), (1, 1)],
    [(3, 4), (1, 2), (5, 6), (2, 3)],       # causal, mixed lengths
    [(6, 6), (2, 2), (9, 9)],
    [(1, 2), (7, 8), (1, 2), (1, 2), (3, 4)],
]


@pytest.mark.parametrize("units", FWD_UNITS,
                         ids=lambda u: "-".join(f"{a}.{b}" for a, b in u))
@pytest.mark.parametrize("split_p", [True, False], ids=["d64_split_p", "d128_shared_sp"])
def test_forward_protocol(split_p, units):
    for seed in range(80):
        sim = Sim(seed)
        sim.run(fwd_roles(sim, units, split_p))


HALF_UNITS = [[(1, 1)] * 7, [(3, 3)] * 5, [(8, 8)] * 3, [(2, 2), (1, 1), (5, 5), (1, 1)]]


@pytest.mark.parametrize("units", HALF_UNITS, ids=["1x7", "3x5", "8x3", "mixed"])
@pytest.mark.parametrize("idle0", [False, True], ids=["tile0_full", "tile0_part"])
def test_forward_protocol_at_most_128_queries(units, idle0):
    """Launches of at most 128 queries: P split from S at either head dim
    (head dim 128: four stages, one Q buffer; 64: eight and two), tile 1 idle
    in every unit, tile 0's warps past the last query idle or not."""
    for seed in range(150):
        for S, QB in ((4, 1), (8, 2)):
            sim = Sim(seed)
            sim.run(fwd_roles(sim, units, True, S=S, QB=QB, half=True, idle0=idle0))


def test_forward_idle_tile_stage_releases_run_ahead():
    """The fault the single-issuer stage release fixed: when tile 1's MMA
    thread, which issues nothing, still gave every K/V stage one of its two
    releases, it could run a whole ring ahead and complete a stage's release
    for a fill that tile 0's P V was still reading."""
    failures = 0
    for seed in range(300):
        sim = Sim(seed)
        try:
            sim.run(fwd_roles(sim, [(8, 8)] * 3, True, S=4, QB=1, half=True, idle0=True,
                              half_shared_stages=True))
        except AssertionError as e:
            assert "lands in phase" in str(e) or "completed" in str(e), str(e)
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("split_p", [True, False], ids=["d64_split_p", "d128_shared_sp"])
def test_forward_single_fin_buffer_runs_ahead(split_p):
    """The race the double-buffered fin_full fixed: with one buffer per tile,
    a unit whose tile 0 takes a single step can publish its final row max and
    sum before the epilogue of the previous unit has read them."""
    failures = 0
    for seed in range(300):
        sim = Sim(seed)
        try:
            sim.run(fwd_roles(sim, [(1, 2)] * 5, split_p, single_fin=True))
        except AssertionError:
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("tiles,k_blocks", [(1, 1), (1, 7), (2, 3), (3, 1), (5, 4), (4, 13)])
def test_gemm_pair_protocol(tiles, k_blocks):
    for seed in range(60):
        sim = Sim(seed)
        sim.run(gemm_pair_roles(sim, tiles, k_blocks))


UNIT_LISTS = [[1], [2], [3], [4], [1, 1, 1], [5, 1, 2, 7], [3, 3], [1, 4, 1, 9, 2]]


@pytest.mark.parametrize("units", UNIT_LISTS, ids=lambda u: "-".join(map(str, u)))
@pytest.mark.parametrize("kernel", ["based", "based_linear", "dq", "dkdv"])
def test_protocol_completes_without_run_ahead(kernel, units):
    build = {"based": based_roles, "based_linear": based_linear_roles, "dq": dq_roles,
             "dkdv": dkdv_roles}[kernel]
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


@pytest.mark.parametrize("split_p,drop", [(True, "v_ready"), (False, "v_ready"),
                                          (False, "k_wait")])
def test_forward_model_sees_a_missing_wait(split_p, drop):
    """The data checks are live: without the softmax's wait for the converted
    V tile (or, with P over S, the MMA thread's wait for the K tile), the MMA
    thread issues a product whose operand has not landed in some
    interleavings."""
    failures = 0
    for seed in range(300):
        sim = Sim(seed)
        try:
            sim.run(fwd_roles(sim, [(3, 4), (2, 3), (4, 4)], split_p, drop=(drop,)))
        except AssertionError as e:
            assert "uses data" in str(e) or "completed" in str(e), str(e)
            failures += 1
    assert failures > 0


@pytest.mark.parametrize("kernel,drop", [("dq", "s_read"), ("based_linear", "sext_free")])
def test_buffer_models_see_a_missing_wait(kernel, drop):
    """The buffer versions are live: without the dQ warps' "S read" signal
    the dP product can overwrite S before the warps load it, and without
    the release of the old state copy the linear Based copy warps can
    overwrite it while phi(Q) S_ext still reads it."""
    build = {"dq": dq_roles, "based_linear": based_linear_roles}[kernel]
    failures = 0
    for seed in range(300):
        sim = Sim(seed)
        try:
            sim.run(build(sim, [5, 3, 4], drop=(drop,)))
        except AssertionError as e:
            assert "version" in str(e) or "completed" in str(e) or "phase" in str(e), str(e)
            failures += 1
    assert failures > 0
