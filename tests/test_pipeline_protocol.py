"""The forward kernel's mbarrier protocol, modelled on the CPU for each of
its three step orders:

* D = 64: one MMA-issuing warp per Q tile, a ring of four whole K/V stages,
  two Q buffers, P apart from S (S_{j+1} issued once the softmax has loaded
  S_j);
* D = 128, two Q tiles: one MMA warp interleaving both tiles
  (S0_j, P.V1_{j-1}, S1_j, P.V0_j), two whole stages, one Q buffer, P written
  over S;
* D = 128, heads of one Q tile: the D = 64 order with P in the idle tile's S
  columns, and each stage's K and V landing and released on barriers of their
  own, the producer loading K one step ahead of V.

Each role of a CTA -- the TMA producer, the MMA issuer(s), the softmax
warpgroup of each Q tile and the epilogue -- is a coroutine that follows the
kernel's own sequence of waits, arrivals and commits
(exact_attention_10_gb300/csrc/fa_fwd_kernel.cuh: load_role, MmaIssuer::tile,
tile_interleaved, mma_role, softmax_role, epilogue_role).  Barriers keep
phase counts exactly as mbarriers do: a parity wait on phase k returns once
k has completed, and a waiter that finds its barrier two phases past k would
mistake the parity (a lost phase), which the model reports.  TMA copies and
tcgen05 commits arrive as soon as they are issued; the hardware may delay
them, which only removes interleavings, never adds a dependency.  The model
checks liveness and phase accounting, not the data hazards that the issue
order of the tensor core's operations guards.

A CTA holds a sequence of parts, each a run of n key steps of one CTA tile
of which Q tile w computes the first n_w (a causal or band tile's shorter
tile may have none).  Random interleavings over many part sequences must all
finish.  Two pins: the producer order the one-tile kernel first had, which
held a part's last V until after the next part's Q load although the MMA
warp frees the single Q buffer only after that V is read, must deadlock once
a CTA holds two parts; and a softmax that skips the wait for its part's last
P.V must be reported as a lost phase.

The balanced variant's merge path (the epilogue's job queue to the merge warp
and the merge warp's ring of copy buffers) is modelled the same way at the
end of this file.
"""
from __future__ import annotations

import random
from dataclasses import dataclass

import pytest


@dataclass(frozen=True)
class Order:
    stages: int      # K/V ring depth
    q_bufs: int      # Q buffers
    mma_warps: int   # MMA-issuing warps (one per Q tile, or one for both)
    sep: bool        # P apart from S
    split_kv: bool   # K and V of a stage on separate barriers
    tiles: int       # Q tiles with work


ORDERS = {
    "d64": Order(stages=4, q_bufs=2, mma_warps=2, sep=True, split_kv=False, tiles=2),
    "d128": Order(stages=2, q_bufs=1, mma_warps=1, sep=False, split_kv=False, tiles=2),
    "d128_one_tile": Order(stages=2, q_bufs=1, mma_warps=1, sep=True, split_kv=True, tiles=1),
}


class Barrier:
    def __init__(self, name: str, count: int = 1):
        self.name, self.count, self.phase, self.pending = name, count, 0, 0

    def arrive(self):
        self.pending += 1
        if self.pending == self.count:
            self.pending = 0
            self.phase += 1


class Aliased(Exception):
    pass


def wait(bar: Barrier, k: int):
    """Parity wait for phase k of `bar` (k < 0: the phase before the first,
    complete from the start)."""
    return ("wait", bar, k)


class CTA:
    def __init__(self, o: Order):
        b, m = Barrier, o.mma_warps
        self.full = [b(f"full{s}") for s in range(o.stages)]              # stage (or K) landed
        self.empty = [b(f"empty{s}", m) for s in range(o.stages)]         # stage (or K) read by every MMA warp
        self.v_full = [b(f"v_full{s}") for s in range(o.stages)]          # split: V landed
        self.v_empty = [b(f"v_empty{s}", m) for s in range(o.stages)]     # split: V read
        self.q_full = [b(f"q_full{q}") for q in range(o.q_bufs)]
        self.q_empty = [b(f"q_empty{q}", m) for q in range(o.q_bufs)]
        # per Q tile (a warpgroup's 128 arrivals count as one here)
        self.s_full = [b(f"s_full{w}") for w in range(2)]
        self.s_free = [b(f"s_free{w}") for w in range(2)]
        self.p_full = [b(f"p_full{w}") for w in range(2)]
        self.o_done = [b(f"o_done{w}") for w in range(2)]
        self.st_ready = [b(f"st_ready{w}") for w in range(2)]
        self.st_free = [b(f"st_free{w}") for w in range(2)]
        self.o_free = [b(f"o_free{w}") for w in range(2)]


def loader(c: CTA, o: Order, parts, flush_before_q: bool = True):
    step = it = nv = 0

    def load_v():
        nonlocal nv
        st, use = nv % o.stages, nv // o.stages
        yield wait(c.v_empty[st], use - 1)
        c.v_full[st].arrive()
        nv += 1

    for n, _, _ in parts:
        if o.split_kv and flush_before_q and nv < step:   # the previous part's last V
            yield from load_v()
        qb, quse = it % o.q_bufs, it // o.q_bufs
        yield wait(c.q_empty[qb], quse - 1)
        c.q_full[qb].arrive()
        it += 1
        for _ in range(n):
            st, use = step % o.stages, step // o.stages
            yield wait(c.empty[st], use - 1)
            c.full[st].arrive()              # K (and V, unless split) of this step
            if o.split_kv and nv < step:
                yield from load_v()          # V of the previous step
            step += 1
    if o.split_kv and nv < step:
        yield from load_v()                  # the last step's V


class Issuer:
    """MMA issue state of one Q tile (MmaIssuer)."""

    def __init__(self, c: CTA, o: Order, w: int):
        self.c, self.o, self.w = c, o, w
        self.n_s = self.n_pv = self.n_t = 0

    def issue_s(self):
        if self.o.sep and self.n_s > 0:
            yield wait(self.c.s_free[self.w], self.n_s - 1)
        self.c.s_full[self.w].arrive()       # commit after S
        self.n_s += 1

    def issue_pv(self, accumulate: bool):
        if not accumulate:                   # the part's first P.V overwrites O: the epilogue has read it
            if self.n_t > 0:
                yield wait(self.c.o_free[self.w], self.n_t - 1)
            self.n_t += 1
        yield wait(self.c.p_full[self.w], self.n_pv)
        self.c.o_done[self.w].arrive()
        self.n_pv += 1


def tile_sep(m: Issuer, step0: int, n: int, nw: int):
    """MmaIssuer::tile, the separate-P order."""
    c, o = m.c, m.o
    yield wait(c.full[step0 % o.stages], step0 // o.stages)
    if nw > 0:
        yield from m.issue_s()
    if o.split_kv:
        c.empty[step0 % o.stages].arrive()
    for j in range(n):
        if j + 1 < n:
            g = step0 + j + 1
            yield wait(c.full[g % o.stages], g // o.stages)
            if j + 1 < nw:
                yield from m.issue_s()
            if o.split_kv:
                c.empty[g % o.stages].arrive()
        g = step0 + j
        if o.split_kv:
            yield wait(c.v_full[g % o.stages], g // o.stages)
        if j < nw:
            yield from m.issue_pv(j > 0)
        (c.v_empty if o.split_kv else c.empty)[g % o.stages].arrive()


def tile_interleaved(m0: Issuer, m1: Issuer, step0: int, n: int, n0: int, n1: int):
    c, o = m0.c, m0.o
    prev = None
    for j in range(n):
        g = step0 + j
        yield wait(c.full[g % o.stages], g // o.stages)
        if j < n0:
            yield from m0.issue_s()
        if j >= 1:
            if j - 1 < n1:
                yield from m1.issue_pv(j - 1 > 0)
            c.empty[prev].arrive()           # K_{j-1} and V_{j-1} read
        if j < n1:
            yield from m1.issue_s()
        if j < n0:
            yield from m0.issue_pv(j > 0)
        prev = g % o.stages
    if n - 1 < n1:
        yield from m1.issue_pv(n - 1 > 0)
    c.empty[prev].arrive()


def mma(c: CTA, o: Order, parts, w: int):
    """mma_role of warp w (w = 0 issues both tiles when one warp serves both)."""
    m, m1 = Issuer(c, o, w), Issuer(c, o, 1)
    step = it = 0
    for n, n0, n1 in parts:
        qb = it % o.q_bufs
        yield wait(c.q_full[qb], it // o.q_bufs)
        if o.sep:
            yield from tile_sep(m, step, n, n1 if w else n0)
        else:
            yield from tile_interleaved(m, m1, step, n, n0, n1)
        step += n
        c.q_empty[qb].arrive()
        it += 1


def softmax(c: CTA, o: Order, parts, w: int, last_pv_wait: bool = True):
    s_phase = o_phase = n_st = 0
    for part in parts:
        np_ = part[1 + w]
        if np_ == 0:
            continue
        for jr in range(np_):
            yield wait(c.s_full[w], s_phase)
            s_phase += 1
            if o.sep:
                c.s_free[w].arrive()
            if o.sep and jr > 0:
                yield wait(c.o_done[w], o_phase)
                o_phase += 1
            c.p_full[w].arrive()
        if o.sep and last_pv_wait:
            yield wait(c.o_done[w], o_phase)  # the part's last P.V
            o_phase += 1
        if n_st > 0:
            yield wait(c.st_free[w], n_st - 1)
        n_st += 1
        c.st_ready[w].arrive()


def epilogue(c: CTA, o: Order, parts):
    taken, pv = [0, 0], [0, 0]
    for part in parts:
        for w in range(o.tiles):
            np_ = part[1 + w]
            if np_ == 0:
                continue
            yield wait(c.st_ready[w], taken[w])
            taken[w] += 1
            c.st_free[w].arrive()
            pv[w] += np_
            yield wait(c.o_done[w], pv[w] - 1)
            c.o_free[w].arrive()


def run(order: str, parts, seed: int, flush_before_q: bool = True, last_pv_wait: bool = True) -> str:
    """'done', 'deadlock' or 'aliased' for one random interleaving."""
    o = ORDERS[order]
    c = CTA(o)
    roles = [loader(c, o, parts, flush_before_q)]
    roles += [mma(c, o, parts, w) for w in range(o.mma_warps)]
    roles += [softmax(c, o, parts, w, last_pv_wait) for w in range(o.tiles)]
    roles.append(epilogue(c, o, parts))
    blocked = [None] * len(roles)
    live = set(range(len(roles)))
    rng = random.Random(seed)

    def ready(i):
        w = blocked[i]
        if w is None:
            return True
        _, bar, k = w
        if bar.phase > k + 1:
            raise Aliased(f"{bar.name}: phase {bar.phase} while waiting for {k}")
        return bar.phase >= k + 1

    try:
        while live:
            runnable = [i for i in live if ready(i)]
            if not runnable:
                return "deadlock"
            i = rng.choice(runnable)
            try:
                blocked[i] = next(roles[i])
            except StopIteration:
                live.discard(i)
                blocked[i] = None
    except Aliased:
        return "aliased"
    return "done"


def one_tile_parts(lengths):
    return [(n, n, 0) for n in lengths]


def random_parts(rng: random.Random, tiles: int):
    """A CTA's parts: 1-4 runs of 1-7 steps; with two tiles, one of them
    (either) may stop early, down to no steps at all."""
    parts = []
    for _ in range(rng.randint(1, 4)):
        n = rng.randint(1, 7)
        if tiles == 1:
            parts.append((n, n, 0))
        elif rng.random() < 0.5:
            parts.append((n, rng.randint(0, n), n))   # causal-like: tile 0 shorter
        else:
            parts.append((n, n, rng.randint(0, n)))   # band-like: tile 1 shorter
    return parts


ONE_TILE_SETS = [(1,), (2,), (5,), (1, 1), (1, 4), (3, 2), (4, 1, 3), (1, 1, 1, 1), (7, 1), (2, 6, 1, 3)]


@pytest.mark.parametrize("lengths", ONE_TILE_SETS)
def test_one_tile_order_always_completes(lengths):
    for seed in range(300):
        assert run("d128_one_tile", one_tile_parts(lengths), seed) == "done", (lengths, seed)


@pytest.mark.parametrize("order", ["d64", "d128", "d128_one_tile"])
def test_every_order_completes_on_random_part_sequences(order):
    rng = random.Random(sum(map(ord, order)))
    for _ in range(150):
        parts = random_parts(rng, ORDERS[order].tiles)
        for seed in range(20):
            assert run(order, parts, seed) == "done", (order, parts, seed)


@pytest.mark.parametrize("lengths", [(1, 1), (3, 2), (4, 1, 3)])
def test_holding_the_last_v_past_the_next_q_load_deadlocks(lengths):
    """The first pin: without the flush before the next part's Q load the
    model finds the deadlock the kernel hit (a bounded wait expired), in every
    interleaving of a CTA with two or more parts."""
    parts = one_tile_parts(lengths)
    assert all(run("d128_one_tile", parts, seed, flush_before_q=False) == "deadlock" for seed in range(50))


def test_single_part_needs_no_flush():
    """One part per CTA never reaches the hand-over, so the old order passed
    there, as it did on the GPU for every test with one part per CTA."""
    for seed in range(100):
        assert run("d128_one_tile", one_tile_parts((5,)), seed, flush_before_q=False) == "done"


@pytest.mark.parametrize("order", ["d64", "d128_one_tile"])
def test_a_lost_phase_is_reported(order):
    """The second pin: a softmax that skips the wait for its part's last P.V
    lets its count of o_done phases fall behind, so a later parity wait can
    see a phase two past the one it means; the model must flag it."""
    parts = [(3, 3, 3), (2, 2, 2), (4, 4, 4)] if ORDERS[order].tiles == 2 else one_tile_parts((3, 2, 4))
    outcomes = {run(order, parts, seed, last_pv_wait=False) for seed in range(200)}
    assert "aliased" in outcomes, outcomes


def test_model_matches_the_kernel_constants(kernel_constants):
    """The orders above use the kernel's own ring depths, Q buffers and issue
    structure: D = 64 and the two-tile D = 128 order as compiled, the
    one-tile order as the D = 128 kernel runs it (separate P, K and V split)."""
    k64, k128 = kernel_constants["fwd64"], kernel_constants["fwd128"]
    assert kernel_constants["q_tiles"] == 2
    d64, d128, one = ORDERS["d64"], ORDERS["d128"], ORDERS["d128_one_tile"]
    assert (d64.stages, d64.q_bufs, d64.mma_warps, d64.sep, d64.split_kv) == \
        (k64["stages"], k64["q_bufs"], k64["mma_warps"], bool(k64["sep"]), bool(k64["split_kv"]))
    assert (d128.stages, d128.q_bufs, d128.mma_warps, d128.sep) == \
        (k128["stages"], k128["q_bufs"], k128["mma_warps"], bool(k128["sep"]))
    assert (one.stages, one.q_bufs, one.mma_warps, one.split_kv) == \
        (k128["stages"], k128["q_bufs"], k128["mma_warps"], bool(k128["split_kv"]))


# ---------------------------------------------------------------- merge queue
# The balanced variant's merge path (epilogue_role's post, merge_role): the
# epilogue hands merge jobs to the merge warp through kJobSlots = 2 slots
# (job_full / job_empty); the merge warp brings each job's (m, l) in with one
# bulk copy (ml_full) and streams its chunks of partial O through
# kMergeBufs = 4 buffers (merge_full), issuing the next chunk into a buffer as
# soon as it has read it and numbering chunks across jobs, so a buffer's
# phase is its chunk count so far; a job with no parts tells it to stop.
JOB_SLOTS, MERGE_BUFS = 2, 4


def merge_run(jobs, seed: int, carry_count: bool = True) -> str:
    job_full = [Barrier(f"job_full{j}") for j in range(JOB_SLOTS)]
    job_empty = [Barrier(f"job_empty{j}") for j in range(JOB_SLOTS)]
    merge_full = [Barrier(f"merge_full{i}") for i in range(MERGE_BUFS)]
    ml_full = Barrier("ml_full")
    posted = []

    def epilogue_posts():
        for n, nchunks in enumerate(list(jobs) + [0]):   # the last job (no parts) stops the merge warp
            j = n % JOB_SLOTS
            yield wait(job_empty[j], n // JOB_SLOTS - 1)
            posted.append(nchunks)
            job_full[j].arrive()

    def merge_warp():
        n_jobs = streamed = ml_uses = 0
        while True:
            j = n_jobs % JOB_SLOTS
            yield wait(job_full[j], n_jobs // JOB_SLOTS)
            nchunks = posted[n_jobs]
            if nchunks == 0:
                return
            first = streamed if carry_count else 0
            issued = 0
            ml_full.arrive()                          # the (m, l) copy lands
            while issued < MERGE_BUFS and issued < nchunks:
                merge_full[(first + issued) % MERGE_BUFS].arrive()
                issued += 1
            yield wait(ml_full, ml_uses)
            ml_uses += 1
            for k in range(nchunks):
                g = first + k
                yield wait(merge_full[g % MERGE_BUFS], g // MERGE_BUFS)
                if issued < nchunks:                  # the next chunk into the buffer just read
                    merge_full[(first + issued) % MERGE_BUFS].arrive()
                    issued += 1
            streamed = first + issued
            job_empty[j].arrive()
            n_jobs += 1

    roles = [epilogue_posts(), merge_warp()]
    blocked = [None, None]
    live = {0, 1}
    rng = random.Random(seed)
    try:
        while live:
            runnable = []
            for i in live:
                w = blocked[i]
                if w is not None:
                    _, bar, k = w
                    if bar.phase > k + 1:
                        raise Aliased(bar.name)
                    if bar.phase < k + 1:
                        continue
                runnable.append(i)
            if not runnable:
                return "deadlock"
            i = rng.choice(runnable)
            try:
                blocked[i] = next(roles[i])
            except StopIteration:
                live.discard(i)
                blocked[i] = None
    except Aliased:
        return "aliased"
    return "done"


def test_merge_queue_completes():
    rng = random.Random(7)
    for _ in range(200):
        jobs = [rng.randint(1, 19) for _ in range(rng.randint(1, 6))]   # chunks per job: parts x row blocks
        for seed in range(10):
            assert merge_run(jobs, seed) == "done", (jobs, seed)


def test_merge_buffers_need_the_count_carried_across_jobs():
    """The pin: restarting the chunk count at each job would wait on a
    buffer's phase from an earlier job, which the model flags."""
    outcomes = {merge_run([3, 5, 2], seed, carry_count=False) for seed in range(50)}
    assert "aliased" in outcomes, outcomes
