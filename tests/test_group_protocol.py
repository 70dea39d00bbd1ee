"""Host-side model of the grouped prefill kernel's synchronisation protocol.

`gda_prefill_group_kernel` (csrc/gda_prefill_group.cu) coordinates one TMA producer, a
logit-MMA issuer, a value-MMA issuer and the compute warps through mbarriers whose waits
name a phase by its parity only.  This test replays that protocol as a discrete-event
model with random completion delays and random interleavings, for one, two and three
signal heads per item and ragged item lengths, and checks on every schedule that

- nothing deadlocks;
- every wait names a phase at most one ahead of the barrier's completed phases (a
  parity wait cannot tell phase k from phase k + 2);
- no asynchronous write (TMA into a ring slot, a logit MMA into a TMEM slot, a value MMA
  into an accumulator) overlaps another access to the same storage, and no P tile,
  row-exchange word or staged output row is written while a value MMA or an output TMA
  store reads its buffer.

The model mirrors the kernel's loops: slot assignment of the statistics sweep, the one
K / V ring consumed in order by two issuers that skip each other's entries, the P
buffers [buffer][half], the per-row exchange in the row's own bytes of P buffer 0, and
the per-item barriers (q_full / q_empty, o_final / o_free), and both epilogues: per-row
output stores (items longer than 28 key tiles) and the staged one, whose output rows go
through the P buffers to TMA stores issued by one thread of each row quarter.  Compute
warps are modelled as units of two row quarters x four key quarters.
"""
import random

import pytest

NR = 6                      # ring slots
QUARTERS, KQ = 2, 4         # compute units: row quarters x key quarters


class Bar:
    def __init__(self, name, count):
        self.name, self.count = name, count
        self.pending = 0
        self.tx = 0
        self.completed = 0

    def _maybe_complete(self):
        if self.pending == self.count and self.tx == 0:
            self.pending = 0
            self.completed += 1

    def arrive(self, n=1):
        self.pending += n
        assert self.pending <= self.count, f"{self.name}: {self.pending} arrivals of {self.count}"
        self._maybe_complete()


def compatible(k1, k2):
    """May two accesses to the same storage overlap in time?  Kinds: "r" (read), "w"
    (exclusive write), "pw" (compute warps writing their own chunks of P rows or staged
    output rows), "ex" (the row exchange's words), "ar" (an output TMA store reading staged
    rows) and ("mma", issuer, "r" | "w") for an MMA between its issue and its completion:
    one issuer's MMAs run in order, two issuers' MMAs are unordered."""
    if isinstance(k1, tuple) and isinstance(k2, tuple):
        return k1[1] == k2[1] or (k1[2] == "r" and k2[2] == "r")
    if isinstance(k1, tuple) or isinstance(k2, tuple):
        m, o = (k1, k2) if isinstance(k1, tuple) else (k2, k1)
        return m[2] == "r" and o in ("r", "ar")
    if "ar" in (k1, k2):
        return k1 in ("r", "ar") and k2 in ("r", "ar")
    return k1 == k2 and k1 in ("r", "pw", "ex")


class Storage:
    """Active accesses per storage unit (a TMEM slot, a ring slot, a Q tile, a quarter's
    rows of one P buffer half)."""

    def __init__(self):
        self.active = {}                    # key -> list of (kind, owner)

    def begin(self, key, kind, owner):
        acc = self.active.setdefault(key, [])
        for k2, o2 in acc:
            assert compatible(kind, k2), f"conflict on {key}: {kind} by {owner} while {k2} by {o2}"
        acc.append((kind, owner))

    def end(self, key, kind, owner):
        self.active[key].remove((kind, owner))


def simulate(S, items, seed, staged=False, skip_p_empty_wait=False, exchange_over_all_rows=False,
             skip_logit_o_free=False, skip_store_wait=False):
    """Runs one random schedule (`staged`: the epilogue that stages the output in the P
    buffers for TMA stores).  The other keyword switches plant protocol errors (for the
    checker's own tests): compute warps that do not wait for p_empty, a row exchange
    spread over every row of the P buffer (each quarter's words in all quarters' rows),
    a logit issuer that writes the accumulator columns in the statistics sweep without
    waiting for the previous item's epilogue, a store leader that does not wait for its
    TMA stores to read a buffer before it is written again."""
    M, NB = S + 1, 4 - S
    LAG = NB + 1
    rng = random.Random(seed)
    now = [0]
    events = []                              # (time, seq, fn)
    seq = [0]
    bars = {}
    mem = Storage()

    def bar(name, count):
        bars[name] = Bar(name, count)

    nunits = QUARTERS * KQ
    slow_quarter = rng.randrange(QUARTERS)
    slow_factor = rng.choice([1, 2, 6])
    bar("q_full", 1)
    bar("q_empty", 1)
    for s in range(NR):
        bar(f"r_full{s}", 1)
        bar(f"r_empty{s}", 1)
    for s in range(4):
        bar(f"s_full{s}", 1)
        bar(f"s_free{s}", nunits)
    for b in range(2):
        for h in range(2):
            bar(f"p_full{b}{h}", nunits // 2)
            bar(f"p_empty{b}{h}", 1)
    bar("o_final", 1)
    bar("o_free", nunits)
    bar("mma_idle", 2)

    def later(dt, fn):
        seq[0] += 1
        events.append((now[0] + dt, seq[0], fn))

    def slot_a(a):
        k = a % 4
        return S + k if k < 4 - S else k - (4 - S)

    def is_signal(v):
        return v % M != 0

    # --- asynchronous engines -------------------------------------------------
    pipe_free = [0]                          # the tensor pipe runs MMAs in issue order
    last_done = {"qk": 0, "pv": 0}           # per issuer: completion of its latest MMA

    def arrive_expect(barname, copies):
        """arrive.expect_tx: the phase also waits for `copies` transfers (one call)"""
        b = bars[barname]
        b.tx += copies
        b.arrive(1)

    def tma(barname, key):
        b = bars[barname]
        mem.begin(key, "w", "tma")

        def done():
            mem.end(key, "w", "tma")
            b.tx -= 1
            b._maybe_complete()
        later(rng.randint(1, 60), done)

    def mma(issuer, accesses, dur):
        """accesses: list of (key, kind) held from issue until the MMA completes."""
        accesses = [(key, ("mma", issuer, kind)) for key, kind in accesses]
        for key, kind in accesses:
            mem.begin(key, kind, issuer)
        start = max(now[0], pipe_free[0])
        end = start + dur
        pipe_free[0] = end
        last_done[issuer] = end

        def done():
            for key, kind in accesses:
                mem.end(key, kind, issuer)
        seq[0] += 1
        events.append((end, seq[0], done))

    def commit(issuer, barname):
        t = max(last_done[issuer], now[0]) + 1
        seq[0] += 1
        events.append((t, seq[0], lambda: bars[barname].arrive(1)))

    def W(name, phase):
        return ("wait", name, phase)

    # --- producer ---------------------------------------------------------------
    def producer():
        ct = 0
        for rr, nkv in enumerate(items):
            if rr > 0:
                yield W("q_empty", rr - 1)
            arrive_expect("q_full", M)
            for m in range(M):
                tma("q_full", ("Q", m))

            def load():
                nonlocal ct
                st = ct % NR
                if ct >= NR:
                    yield W(f"r_empty{st}", ct // NR - 1)
                arrive_expect(f"r_full{st}", 1)
                tma(f"r_full{st}", ("R", st))
                ct += 1
            for _ in range(nkv * M):                        # phase A: K tiles
                yield from load()
            nb = nkv * M
            for i in range(nb):                             # phase B: K(i), then V(i - LAG) halves
                yield from load()
                if i >= LAG and is_signal(i - LAG):
                    yield from load()
                    yield from load()
            for v in range(max(0, nb - LAG), nb):
                if is_signal(v):
                    yield from load()
                    yield from load()

    # --- logit-MMA issuer --------------------------------------------------------
    def qk_issuer():
        cnt = [0] * 4
        ct = 0
        nitem = 0
        for rr, nkv in enumerate(items):
            yield W("q_full", rr)
            o_ready = False

            def qk(m, slot):
                nonlocal ct, o_ready
                k = cnt[slot]
                cnt[slot] += 1
                if slot < S and not o_ready:
                    o_ready = True
                    if nitem > 0 and not skip_logit_o_free:
                        yield W("o_free", nitem - 1)
                st = ct % NR
                yield W(f"r_full{st}", ct // NR)
                if k >= 1:
                    yield W(f"s_free{slot}", k - 1)
                mma("qk", [(("T", slot), "w"), (("Q", m), "r"), (("R", st), "r")], rng.randint(4, 20))
                commit("qk", f"s_full{slot}")
                commit("qk", f"r_empty{st}")
                ct += 1
            na = nkv * M
            for a in range(na):
                yield from qk(a % M, slot_a(a))
            nb = nkv * M
            for i in range(nb):
                yield from qk(i % M, S + i % NB)
                if i == nb - 1:
                    commit("qk", "q_empty")
                if i >= LAG and is_signal(i - LAG):
                    ct += 2
            for v in range(max(0, nb - LAG), nb):
                if is_signal(v):
                    ct += 2
            nitem += 1
        commit("qk", "mma_idle")
        yield W("mma_idle", 0)

    # --- value-MMA issuer --------------------------------------------------------
    def pv_issuer():
        ct = 0
        pk = 0
        nitem = 0
        for rr, nkv in enumerate(items):
            o_ready = False

            def pv(v):
                nonlocal ct, pk, o_ready
                h = v % M - 1
                pb = pk & 1
                if not o_ready:
                    o_ready = True
                    if nitem > 0:
                        yield W("o_free", nitem - 1)
                for half in range(2):
                    yield W(f"p_full{pb}{half}", pk >> 1)
                    st = ct % NR
                    yield W(f"r_full{st}", ct // NR)
                    mma("pv", [(("T", h), "w"), (("P", pb, half), "r"), (("R", st), "r")], rng.randint(8, 30))
                    commit("pv", f"p_empty{pb}{half}")
                    commit("pv", f"r_empty{st}")
                    ct += 1
                pk += 1
            ct += nkv * M                                       # the phase-A K tiles
            nb = nkv * M
            for i in range(nb):
                ct += 1                                         # K tile of logit use i
                if i >= LAG and is_signal(i - LAG):
                    yield from pv(i - LAG)
            for v in range(max(0, nb - LAG), nb):
                if is_signal(v):
                    yield from pv(v)
            commit("pv", "o_final")
            nitem += 1
        commit("pv", "mma_idle")
        yield W("mma_idle", 0)

    # --- compute units -------------------------------------------------------------
    def compute(quarter, kq):
        me = f"c{quarter}{kq}"
        half = kq * 2 // KQ
        cnt = [0] * 4
        pk = 0
        leader = kq == 0
        groups = []                          # the leader's store groups: [done flag]
        tag = "X" if half == 0 else "Y"

        def store(pb):
            """one bulk group: TMA stores of both halves of the quarter's rows of buffer pb"""
            keys = [("X", pb, quarter), ("Y", pb, quarter)]
            for key in keys:
                mem.begin(key, "ar", f"st{quarter}")
            g = [False]
            groups.append(g)

            def done():
                for key in keys:
                    mem.end(key, "ar", f"st{quarter}")
                g[0] = True
            later(rng.randint(1, 80), done)

        def wait_read(n):
            """cp.async.bulk.wait_group.read n: every group but the n most recent has read"""
            if skip_store_wait:
                return
            yield ("cond", lambda: all(g[0] for g in groups[:len(groups) - n]))

        def acquire(slot):
            k = cnt[slot]
            cnt[slot] += 1
            yield W(f"s_full{slot}", k)
            mem.begin(("T", slot), "r", me)

        def release(slot):
            mem.end(("T", slot), "r", me)
            bars[f"s_free{slot}"].arrive(1)

        def math():
            # one row quarter's warps run slower (their sub-partition also hosts an issuer)
            yield ("sleep", rng.randint(0, 40) * (slow_factor if quarter == slow_quarter else 1))

        for rr, nkv in enumerate(items):
            # phase A: the slot is released after the tile's sum (and a possible re-read)
            for j in range(nkv):
                for m in range(M):
                    slot = slot_a(j * M + m)
                    yield from acquire(slot)
                    yield from math()
                    release(slot)
            # row exchange in this quarter's rows of P buffer 0, half 0 (staged: once the
            # previous item's output stores have read the P buffers)
            if staged and rr > 0:
                if leader:
                    yield from wait_read(0)
                yield ("bar", quarter)
            xq = range(QUARTERS) if exchange_over_all_rows else [quarter]
            for q in xq:
                mem.begin(("X", 0, q), "ex", me)
            yield from math()
            yield ("bar", quarter)
            yield from math()
            for q in xq:
                mem.end(("X", 0, q), "ex", me)
            yield ("bar", quarter)
            # phase B: the slot is released right after the load
            for j in range(nkv):
                slot = S + (j * M) % NB
                yield from acquire(slot)
                release(slot)
                yield from math()
                for h in range(S):
                    slot = S + (j * M + 1 + h) % NB
                    yield from acquire(slot)
                    release(slot)
                    pb = pk & 1
                    if pk >= 2 and not skip_p_empty_wait:
                        yield W(f"p_empty{pb}{half}", (pk >> 1) - 1)
                    key = ("X" if half == 0 else "Y", pb, quarter)
                    mem.begin(key, "pw", me)                   # P formation and stores
                    yield from math()
                    mem.end(key, "pw", me)
                    bars[f"p_full{pb}{half}"].arrive(1)
                    pk += 1
            # epilogue: accumulators, sums of squares in P buffer 0 half 1 rows of the quarter
            yield W("o_final", rr)
            for h in range(S):
                mem.begin(("T", h), "r", me)
            for q in xq:
                mem.begin(("Y", 0, q), "ex", me)
            yield from math()
            yield ("bar", quarter)
            yield from math()
            for q in xq:
                mem.end(("Y", 0, q), "ex", me)
            if staged:
                # heads 0 and 2 staged in P buffer 1, head 1 in buffer 0 (this unit's half of
                # the quarter's rows); the leader stores them after the quarter's barrier
                yield ("bar", quarter)
                for h in range(min(S, 2)):
                    key = (tag, 1 - h % 2, quarter)
                    mem.begin(key, "pw", me)
                    yield from math()
                    mem.end(key, "pw", me)
                yield ("bar", quarter)
                if leader:
                    for h in range(min(S, 2)):
                        store(1 - h % 2)
            for h in range(S):
                mem.end(("T", h), "r", me)
            bars["o_free"].arrive(1)
            if staged and S > 2:
                if leader:
                    yield from wait_read(1)
                yield ("bar", quarter)
                key = (tag, 1, quarter)
                mem.begin(key, "pw", me)
                yield from math()
                mem.end(key, "pw", me)
                yield ("bar", quarter)
                if leader:
                    store(1)
            yield ("bar", quarter)
        if staged and leader:
            yield from wait_read(0)

    # The P-buffer rows a quarter's units write (and its exchange words) conflict with a value
    # MMA that reads the whole buffer: map the MMA's read of ("P", pb, half) onto every quarter.
    orig_begin, orig_end = mem.begin, mem.end

    def expand(key):
        if key[0] == "P":
            tag = "X" if key[2] == 0 else "Y"
            return [(tag, key[1], q) for q in range(QUARTERS)]
        return [key]

    mem.begin = lambda key, kind, owner: [orig_begin(k, kind, owner) for k in expand(key)]
    mem.end = lambda key, kind, owner: [orig_end(k, kind, owner) for k in expand(key)]

    roles = {"producer": producer(), "qk": qk_issuer(), "pv": pv_issuer()}
    for q in range(QUARTERS):
        for k in range(KQ):
            roles[f"c{q}{k}"] = compute(q, k)
    blocked = {name: None for name in roles}
    done = set()
    bar_gen = {q: 0 for q in range(QUARTERS)}
    bar_arrived = {q: set() for q in range(QUARTERS)}
    bar_mine = {}
    steps = 0
    while len(done) < len(roles):
        steps += 1
        assert steps < 3_000_000, "model did not finish"
        runnable = []
        for name in roles:
            if name in done:
                continue
            op = blocked[name]
            if op is None:
                runnable.append(name)
            elif op[0] == "wait":
                b = bars[op[1]]
                assert b.completed <= op[2] + 1, (
                    f"{name} waits for phase {op[2]} of {op[1]}, which has completed {b.completed}")
                if b.completed >= op[2] + 1:
                    runnable.append(name)
            elif op[0] == "sleep":
                if now[0] >= op[1]:
                    runnable.append(name)
            elif op[0] == "bar":
                if bar_gen[op[1]] > bar_mine[name]:
                    runnable.append(name)
            elif op[0] == "cond":
                if op[1]():
                    runnable.append(name)
        if not runnable or (events and rng.random() < 0.3):
            if not events:
                wake = [blocked[n][1] for n in roles if n not in done and blocked[n] and blocked[n][0] == "sleep"]
                if not wake:
                    raise AssertionError("deadlock: " + str({n: blocked[n] for n in roles if n not in done}))
                now[0] = max(now[0], min(wake))
                continue
            events.sort()
            t, _, fn = events.pop(0)
            now[0] = max(now[0], t)
            fn()
            continue
        name = rng.choice(runnable)
        blocked[name] = None
        try:
            op = next(roles[name])
        except StopIteration:
            done.add(name)
            continue
        if op[0] == "sleep":
            op = ("sleep", now[0] + op[1])
        elif op[0] == "bar":
            q = op[1]
            bar_mine[name] = bar_gen[q]
            bar_arrived[q].add(name)
            if len(bar_arrived[q]) == KQ:
                bar_arrived[q].clear()
                bar_gen[q] += 1
        blocked[name] = op
        now[0] += 1
    return steps


@pytest.mark.parametrize("staged", [False, True], ids=["row_stores", "staged_stores"])
@pytest.mark.parametrize("S", [1, 2, 3])
def test_group_protocol_random_schedules(S, staged):
    rng = random.Random(100 + S)
    for seed in range(40):
        items = [rng.randint(1, 7) for _ in range(rng.randint(1, 4))]
        simulate(S, items, seed=1000 * S + seed, staged=staged)


@pytest.mark.parametrize("mutation", ["skip_p_empty_wait", "exchange_over_all_rows", "skip_logit_o_free",
                                      "skip_store_wait"])
def test_group_protocol_checker_catches_planted_errors(mutation):
    """The checker itself: each planted protocol error must fail on some schedule
    (the exchange spread over all rows is the layout that let a fast row quarter's P
    writes overwrite a slow quarter's statistics)."""
    caught = 0
    for seed in range(90):
        S = 1 + seed % 3
        try:
            simulate(S, [1, 2, 1, 3, 1], seed, staged=mutation == "skip_store_wait", **{mutation: True})
        except AssertionError:
            caught += 1
    assert caught > 0
