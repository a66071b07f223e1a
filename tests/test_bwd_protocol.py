"""The backward kernel's mbarrier protocol, modelled on the CPU for its four
passes (exact_attention_10_gb300/csrc/fa_bwd_kernel.cuh: bwd_load, bwd_mma,
bwd_compute, bwd_mma_pipe, bwd_compute_pipe):

* D = 64, dQ and dK/dV passes: pipelined (S_{g+1} and dP_{g+1} issued once the
  compute warps have loaded S_g and dP_g), three stages of both streamed tiles;
* D = 128, dQ pass: pipelined, K and V in separate rings of three and two
  slots, V's slot freed once dP is computed;
* D = 128, dK/dV pass: P^T and dS^T overwrite S and dP, two stages; per step
  the MMA warp issues dV_g, S_{g+1}, dK_g, dP_{g+1} (each overwrite after the
  read it displaces, in issue order), S and dP completing separate barriers
  (sd_full, dp_full) so that the compute warps start on S_{g+1} while dK_g and
  dP_{g+1} still run;
* D = 64, fused pass (bwd_mma_dq, bwd_dq_out): the pipelined dK/dV pass plus a
  second MMA warp that issues each step's dQ product once P / dS are written
  and the read-out warps have loaded the previous product, and the read-out
  warps; pd_free (the P^T / dS^T buffers) and res_empty (the resident K and
  V) count both MMA warps.

The producer, the MMA warp and the two compute warpgroups (column halves) are
coroutines following the kernel's waits, arrivals and commits; barriers keep
exact phase counts, and a waiter that finds its barrier two phases past the
one it means (a lost phase: its parity would read as not yet complete) is
reported.  Copies and commits arrive when issued (in the fused pass's model,
copies land at a random later time, in any order).  Random interleavings over
CTAs holding one or several resident tiles of varying length must finish.

The models of the fused pass and of the D = 128 dK/dV pass also track what
each buffer holds (the resident K and V, the stages, S / P^T and dP / dS^T
per column half, the accumulators; a buffer holds its tile only once its
copy has landed) and report a read of the wrong tile or step, or an
overwrite before the last read, as a race.

The pin: in the pipelined dQ pass nothing holds the compute warps back from
finishing step g + 1 before the MMA warp waits for step g, so one p_full
barrier can run two phases ahead of its waiter; the kernel alternates two
barriers there, and the model must flag the single-barrier form.  In the
fused pass, a pd_free that counted only the first MMA warp would let the
compute warps overwrite dS^T before the dQ product has read it, and a
res_empty that counted only the first MMA warp would let the next tile's K
overwrite the resident tile that the last dQ product still reads; the model
flags both races; and in the D = 128 dK/dV pass, dP_{g+1} issued ahead of
dK_g would overwrite dS^T_g before dK_g reads it.
"""
from __future__ import annotations

import random
from dataclasses import dataclass

import pytest


@dataclass(frozen=True)
class Pass:
    pipeline: bool
    kv: bool            # dK/dV pass (else dQ)
    split: bool         # K and V in separate rings (D = 128 dQ pass)
    ring0: int          # stages, or slots of ring 0
    ring1: int          # slots of ring 1 (split)
    fused: bool = False  # the dK/dV pass with the dQ products (D = 64 default)


PASSES = {
    "d64_dq": Pass(pipeline=True, kv=False, split=False, ring0=3, ring1=3),
    "d64_kv": Pass(pipeline=True, kv=True, split=False, ring0=3, ring1=3),
    "d64_fused": Pass(pipeline=True, kv=True, split=False, ring0=3, ring1=3, fused=True),
    "d128_dq": Pass(pipeline=True, kv=False, split=True, ring0=3, ring1=2),
    "d128_kv": Pass(pipeline=False, kv=True, split=False, ring0=2, ring1=2),
}
COMPUTE = 2   # compute warpgroups, each arriving once per barrier phase


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


class Race(Exception):
    pass


def wait(bar: Barrier, k: int):
    return ("wait", bar, k)


class CTA:
    def __init__(self, q: Pass, alternate_p_full: bool, dq_counted: bool = True, res_dq_counted: bool = True):
        b = Barrier
        self.full = [b(f"full{s}") for s in range(q.ring0)]
        self.empty = [b(f"empty{s}") for s in range(q.ring0)]
        self.full1 = [b(f"full1_{s}") for s in range(q.ring1)]
        self.empty1 = [b(f"empty1_{s}") for s in range(q.ring1)]
        self.res_full, self.res_empty, self.sd_full = b("res_full"), b("res_empty"), b("sd_full")
        self.p_full, self.p_full_odd = b("p_full", COMPUTE), b("p_full_odd", COMPUTE)
        self.acc_full, self.acc_free = b("acc_full"), b("acc_free", COMPUTE)
        self.sd_free, self.pd_free = b("sd_free", COMPUTE), b("pd_free")
        self.alternate = alternate_p_full
        if q.fused:   # both MMA warps read the P^T / dS^T buffers and the resident tiles
            self.pd_free = b("pd_free", 2 if dq_counted else 1)
            self.res_empty = b("res_empty", 2 if res_dq_counted else 1)
            self.dq_full, self.dq_free = b("dq_full"), b("dq_free")
        self.dq_done = 0   # fused: dQ products issued
        # fused: what the buffers hold -- the resident K and V (tile), stages
        # (step); products issued (dV / dK), S and dP loaded and accumulators
        # read out (tiles), per compute warpgroup
        self.res, self.stage = None, [None] * q.ring0
        self.dp_full = Barrier("dp_full")   # D = 128 dK/dV pass: dP of a step ready (S's: sd_full)
        self.s_reg, self.dp_reg = [None] * COMPUTE, [None] * COMPUTE   # (what, step) per column half
        self.prod_done, self.sd_loaded, self.acc_read = 0, [0] * COMPUTE, [0] * COMPUTE
        self.inflight = []   # fused: copies issued, not landed: (barrier, buffer setter, value)

    def p_full_dq(self, g: int):
        """The barrier and phase that carry step g's P / dS in the pipelined dQ pass."""
        if self.alternate:
            return (self.p_full_odd if g & 1 else self.p_full), g >> 1
        return self.p_full, g


def loader(c: CTA, q: Pass, tiles):
    step = t = 0
    for n in tiles:
        if t > 0:
            yield wait(c.res_empty, t - 1)
        c.res_full.arrive()
        t += 1
        for _ in range(n):
            k0 = step % q.ring0
            yield wait(c.empty[k0], step // q.ring0 - 1)
            if q.split:
                k1 = step % q.ring1
                yield wait(c.empty1[k1], step // q.ring1 - 1)
                c.full1[k1].arrive()
            c.full[k0].arrive()
            step += 1


def mma_pipe(c: CTA, q: Pass, tiles):
    g = done = 0

    def issue_sd(gs):
        if gs > 0:
            yield wait(c.sd_free, gs - 1)
        yield wait(c.full[gs % q.ring0], gs // q.ring0)
        if q.split:
            yield wait(c.full1[gs % q.ring1], gs // q.ring1)
        c.sd_full.arrive()
        if q.split:
            c.empty1[gs % q.ring1].arrive()   # V's slot is free once dP is computed

    for n in tiles:
        yield wait(c.res_full, done)
        yield from issue_sd(g)
        for j in range(n):
            if j + 1 < n:
                yield from issue_sd(g + 1)
            if j == 0 and done > 0:
                yield wait(c.acc_free, done - 1)
            if q.kv:
                yield wait(c.p_full, g)
            else:
                yield wait(*c.p_full_dq(g))
            if q.kv:
                c.pd_free.arrive()
            c.empty[g % q.ring0].arrive()
            if j == n - 1:
                c.acc_full.arrive()
                c.res_empty.arrive()
            g += 1
        done += 1


def compute_pipe(c: CTA, q: Pass, tiles, pd_wait: bool = True):
    g = done = 0
    for n in tiles:
        for _ in range(n):
            yield wait(c.sd_full, g)
            c.sd_free.arrive()
            if q.kv and pd_wait and g > 0:
                yield wait(c.pd_free, g - 1)
            if q.kv:
                c.p_full.arrive()
            else:
                c.p_full_dq(g)[0].arrive()
            g += 1
        yield wait(c.acc_full, done)
        c.acc_free.arrive()
        done += 1


def check(ok: bool, what: str):
    if not ok:
        raise Race(what)


def copy(c: CTA, bar: Barrier, setter, value):
    """Issue a copy: its buffer holds nothing usable until it lands (and arrives on `bar`)."""
    setter(("loading", value))
    c.inflight.append((bar, setter, value))


def loader_fused(c: CTA, q: Pass, tiles):
    step = 0

    def set_res(v):
        c.res = v

    def set_stage(i):
        return lambda v: c.stage.__setitem__(i, v)

    for t, n in enumerate(tiles):
        if t > 0:
            yield wait(c.res_empty, t - 1)
        copy(c, c.res_full, set_res, t)
        for _ in range(n):
            yield wait(c.empty[step % q.ring0], step // q.ring0 - 1)
            copy(c, c.full[step % q.ring0], set_stage(step % q.ring0), step)
            step += 1


def mma_fused(c: CTA, q: Pass, tiles):
    g = 0

    def issue_sd(gs, t):
        if gs > 0:
            yield wait(c.sd_free, gs - 1)
        yield wait(c.full[gs % q.ring0], gs // q.ring0)
        check(c.res == t and c.stage[gs % q.ring0] == gs, f"S and dP of step {gs}: K, V or stage not its own")
        check(min(c.sd_loaded) >= gs, f"S of step {gs} over S of step {gs - 1} before it was loaded")
        c.sd_full.arrive()

    for t, n in enumerate(tiles):
        yield wait(c.res_full, t)
        yield from issue_sd(g, t)
        for j in range(n):
            if j + 1 < n:
                yield from issue_sd(g + 1, t)
            if j == 0 and t > 0:
                yield wait(c.acc_free, t - 1)
            yield wait(c.p_full, g)
            check(c.stage[g % q.ring0] == g, f"products of step {g}: stage not its own")
            check(j > 0 or min(c.acc_read) == t, f"tile {t}'s first products before tile {t - 1}'s accumulators were read")
            c.prod_done += 1
            c.pd_free.arrive()
            c.empty[g % q.ring0].arrive()
            if j == n - 1:
                c.acc_full.arrive()
                c.res_empty.arrive()
            g += 1


def compute_fused(c: CTA, q: Pass, tiles, h: int):
    g = 0
    for t, n in enumerate(tiles):
        for _ in range(n):
            yield wait(c.sd_full, g)
            c.sd_loaded[h] = g + 1
            c.sd_free.arrive()
            if g > 0:
                yield wait(c.pd_free, g - 1)
            check(c.dq_done >= g and c.prod_done >= g, f"P^T / dS^T of step {g} written before step {g - 1}'s products")
            c.p_full.arrive()
            g += 1
        yield wait(c.acc_full, t)
        check(c.prod_done == g, f"tile {t}'s accumulators read before its last products")
        c.acc_read[h] = t + 1
        c.acc_free.arrive()


def dq_mma_fused(c: CTA, q: Pass, tiles):
    g = 0
    for t, n in enumerate(tiles):
        yield wait(c.res_full, t)
        for j in range(n):
            yield wait(c.p_full, g)
            if g > 0:
                yield wait(c.dq_free, g - 1)
            check(c.res == t, f"dQ of step {g}: K not tile {t}'s")
            c.dq_done += 1
            c.dq_full.arrive()
            c.pd_free.arrive()
            if j == n - 1:
                c.res_empty.arrive()
            g += 1


def dq_out_fused(c: CTA, tiles):
    g = 0
    for n in tiles:
        for _ in range(n):
            yield wait(c.dq_full, g)
            c.dq_free.arrive()
            g += 1


def mma_serial(c: CTA, q: Pass, tiles, dp_before_dk: bool = False):
    g = 0

    def issue_s(gs, t):
        check(c.res == t and c.stage[gs % q.ring0] == gs, f"S of step {gs}: K or stage not its own")
        for h in range(COMPUTE):   # the previous S was loaded (and P^T written over it and read by dV)
            check(c.s_reg[h] in (None, ("pt", gs - 1)), f"S of step {gs} over {c.s_reg[h]}")
            c.s_reg[h] = ("s", gs)
        c.sd_full.arrive()

    def issue_dp(gs, t):
        check(c.res == t and c.stage[gs % q.ring0] == gs, f"dP of step {gs}: V or stage not its own")
        for h in range(COMPUTE):   # dS^T of the previous step was read by dK
            check(c.dp_reg[h] in (None, ("read", gs - 1)), f"dP of step {gs} over {c.dp_reg[h]}")
            c.dp_reg[h] = ("dp", gs)
        c.dp_full.arrive()

    for t, n in enumerate(tiles):
        yield wait(c.res_full, t)
        yield wait(c.full[g % q.ring0], g // q.ring0)
        issue_s(g, t)
        yield None   # (the tensor pipe takes time: others may run between two issues)
        issue_dp(g, t)
        for j in range(n):
            if j == 0 and t > 0:
                yield wait(c.acc_free, t - 1)
            yield wait(c.p_full, g)
            check(c.stage[g % q.ring0] == g, f"products of step {g}: stage not its own")
            check(j > 0 or min(c.acc_read) == t, f"tile {t}'s first products before tile {t - 1}'s accumulators were read")
            for h in range(COMPUTE):   # dV_g reads P^T_g
                check(c.s_reg[h] == ("pt", g), f"dV of step {g} reads {c.s_reg[h]}")
            if j + 1 < n:
                yield wait(c.full[(g + 1) % q.ring0], (g + 1) // q.ring0)
                issue_s(g + 1, t)
                yield None
                if dp_before_dk:
                    issue_dp(g + 1, t)
            for h in range(COMPUTE):   # dK_g reads dS^T_g
                check(c.dp_reg[h] == ("dst", g), f"dK of step {g} reads {c.dp_reg[h]}")
                c.dp_reg[h] = ("read", g)
            c.prod_done += 1
            c.empty[g % q.ring0].arrive()
            if j == n - 1:
                c.acc_full.arrive()
                c.res_empty.arrive()
            if j + 1 < n and not dp_before_dk:
                issue_dp(g + 1, t)
            g += 1


def compute_serial(c: CTA, q: Pass, tiles, h: int):
    g = 0
    for t, n in enumerate(tiles):
        for _ in range(n):
            yield wait(c.sd_full, g)
            check(c.s_reg[h] == ("s", g), f"step {g} loads {c.s_reg[h]} for S")
            c.s_reg[h] = ("pt", g)     # S loaded, P^T written over it
            yield wait(c.dp_full, g)
            check(c.dp_reg[h] == ("dp", g), f"step {g} loads {c.dp_reg[h]} for dP")
            c.dp_reg[h] = ("dst", g)   # dP loaded, dS^T written over it
            c.p_full.arrive()
            g += 1
        yield wait(c.acc_full, t)
        check(c.prod_done == g, f"tile {t}'s accumulators read before its last products")
        c.acc_read[h] = t + 1
        c.acc_free.arrive()


def run(name: str, tiles, seed: int, alternate_p_full: bool = True, pd_wait: bool = True,
        dq_counted: bool = True, res_dq_counted: bool = True, dp_before_dk: bool = False) -> str:
    q = PASSES[name]
    c = CTA(q, alternate_p_full, dq_counted, res_dq_counted)
    if q.fused:
        roles = [loader_fused(c, q, tiles), mma_fused(c, q, tiles), dq_mma_fused(c, q, tiles), dq_out_fused(c, tiles)]
        roles += [compute_fused(c, q, tiles, h) for h in range(COMPUTE)]
    elif q.pipeline:
        roles = [loader(c, q, tiles), mma_pipe(c, q, tiles)] + [compute_pipe(c, q, tiles, pd_wait) for _ in range(COMPUTE)]
    else:
        roles = [loader_fused(c, q, tiles), mma_serial(c, q, tiles, dp_before_dk)]
        roles += [compute_serial(c, q, tiles, h) for h in range(COMPUTE)]
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
            if c.inflight:   # the copy engine: land one copy in flight
                runnable.append(-1)
            if not runnable:
                return "deadlock"
            i = rng.choice(runnable)
            if i < 0:
                bar, setter, value = c.inflight.pop(rng.randrange(len(c.inflight)))
                setter(value)
                bar.arrive()
                continue
            try:
                blocked[i] = next(roles[i])
            except StopIteration:
                live.discard(i)
                blocked[i] = None
    except Aliased:
        return "aliased"
    except Race:
        return "race"
    return "done"


@pytest.mark.parametrize("name", sorted(PASSES))
def test_every_pass_completes_on_random_tile_sequences(name):
    rng = random.Random(sum(map(ord, name)))
    for _ in range(150):
        tiles = [rng.randint(1, 6) for _ in range(rng.randint(1, 4))]
        for seed in range(20):
            assert run(name, tiles, seed) == "done", (name, tiles, seed)


@pytest.mark.parametrize("name", ["d64_dq", "d128_dq"])
def test_single_p_full_barrier_in_the_pipelined_dq_pass_is_flagged(name):
    """The pin: with one p_full barrier the compute warps can complete two of
    its phases before the MMA warp waits for the first."""
    outcomes = {run(name, [5, 3], seed, alternate_p_full=False) for seed in range(200)}
    assert "aliased" in outcomes, outcomes


def test_pipelined_kv_pass_needs_the_pd_free_wait():
    """In the pipelined dK/dV pass the single P^T / dS^T buffers are what hold
    the compute warps to one step ahead; without their wait on pd_free the
    same lost phase appears."""
    outcomes = {run("d64_kv", [5, 3], seed, pd_wait=False) for seed in range(200)}
    assert "aliased" in outcomes, outcomes


def test_fused_pass_needs_pd_free_to_count_the_dq_warp():
    """The fused pass's pin: with pd_free completed by the first MMA warp
    alone, the compute warps can overwrite dS^T before the dQ product of the
    previous step was issued."""
    outcomes = {run("d64_fused", [5, 3], seed, dq_counted=False) for seed in range(300)}
    assert "race" in outcomes, outcomes


def test_fused_pass_needs_res_empty_to_count_the_dq_warp():
    """With res_empty completed by the first MMA warp's last products alone,
    the producer can load the next tile's K over this tile's while the dQ
    product of its last step still has to read it."""
    outcomes = {run("d64_fused", [3, 4, 3, 2], seed, res_dq_counted=False) for seed in range(400)}
    assert "race" in outcomes, outcomes


def test_d128_kv_pass_needs_dk_before_the_next_dp():
    """dS^T_g sits in dP's columns: the next step's dP may only follow dK_g."""
    outcomes = {run("d128_kv", [4, 3], seed, dp_before_dk=True) for seed in range(100)}
    assert "race" in outcomes, outcomes


def test_model_matches_the_kernel_constants(kernel_constants):
    """The passes above use the kernel's own pipelining choice, ring layout
    and slot counts."""
    for name, q in PASSES.items():
        k = kernel_constants[name]
        assert (q.pipeline, q.split, q.ring0) == (bool(k["pipeline"]), bool(k["split"]), k["ring0"]), name
        if q.split:
            assert q.ring1 == k["ring1"], name
