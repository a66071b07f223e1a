// Exhaustive check of the work decomposition in fa_schedule.h on the CPU:
// every (tile, step) unit is assigned to exactly one part; part slots are
// distinct and in range; a CTA's partial parts come before its whole tiles;
// and for each tile and Q tile the parts the merge expects (sched_part_slots)
// are exactly the parts that hold work.
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <string>
#include <vector>

#include "fa_schedule.h"

using namespace fa;

static int check_schedule(const Schedule &s, bool planned, int wl, int wr);

// A schedule of G CTAs, balanced or not, for the band (wl, wr) as given
// (kSchedUnbounded: no bound); the planner supplies its mask fields.
// split = 2: the tail split (non-causal), every CTA first taking
// floor(T / G) whole tiles, the rest spread over the first gt CTAs (all G
// when gt <= 0).
static int check(int N, int Nkv, int BH, int causal, int G, int split, int wl, int wr, int gt = 0)
{
    if (G > kSchedMaxGrid)
        return 0;
    Schedule s = sched_plan(N, Nkv, BH, causal != 0, G, 1, wl, wr);
    s.G = G;
    s.split = split ? 1 : 0;
    if (split == 2) {
        if (causal || s.T <= G)
            return 0;
        s.W = s.T / G;
        if (s.T == s.W * G)
            return 0;
    }
    s.U = sched_total_units(s);
    if (s.U > kSchedMaxUnits)
        return 0;
    sched_fill_ranges(s, gt);
    return check_schedule(s, false, wl, wr);
}

// The planner's schedule for `sms` SMs: valid, and a balanced one cuts no
// tile into more parts than the merge handles.
static int check_plan(int N, int Nkv, int BH, int causal, int sms, int wl, int wr)
{
    for (int mode : {0, 2}) {   // as planned (auto), and the balanced schedule forced
        const Schedule s = sched_plan(N, Nkv, BH, causal != 0, sms, mode, wl, wr);
        const int rr_grid = s.T < sms ? s.T : sms;
        if (s.G < 1 || (!s.split && s.G != (rr_grid < kSchedMaxGrid ? rr_grid : kSchedMaxGrid))) {
            std::printf("bad grid %d (mode %d)\n", s.G, mode);
            return 1;
        }
        if (check_schedule(s, true, wl, wr)) {
            std::printf("(mode %d)\n", mode);
            return 1;
        }
    }
    return 0;
}

// Every key a row of a Q tile sees lies in that Q tile's steps, which are a
// prefix of its CTA tile's steps, and each row's [sched_row_lo, sched_row_hi)
// is exactly its visible keys (brute force over the rows' bands as given,
// before the planner drops bounds that cannot bind).
static int check_key_ranges(const Schedule &s, int wl, int wr)
{
    for (int ct = 0; ct < s.C; ++ct) {
        const int ks = sched_kv_start(s, ct), n = sched_steps_ct(s, ct);
        for (int w = 0; w < 2; ++w) {
            const int r0 = ct * 256 + w * 128;
            const int nw = sched_kv_tiles(s, ct, w);
            if (r0 >= s.N) {
                if (nw != 0) { std::printf("padding Q tile has steps\n"); return 1; }
                continue;
            }
            if (nw < 1 || nw > n) { std::printf("ct %d w %d: %d steps of %d\n", ct, w, nw, n); return 1; }
            if (s.wl >= kSchedUnbounded && sched_kv_tiles_t<false>(s, ct, w) != nw) {   // the no-left-bound form
                std::printf("ct %d w %d: %d steps by the step-end form, %d in general\n", ct, w,
                            sched_kv_tiles_t<false>(s, ct, w), nw);
                return 1;
            }
            for (int r = r0; r < r0 + 128 && r < s.N; ++r) {
                long long lo = 0, hi = s.Nkv - 1;
                if (s.causal) {
                    if (wl < kSchedUnbounded) lo = (long long)r + s.off - wl;
                    if (wr < kSchedUnbounded) hi = (long long)r + s.off + wr;
                    if (lo < 0) lo = 0;
                    if (hi > s.Nkv - 1) hi = s.Nkv - 1;
                    const int rl = sched_row_lo(s, r), rh = sched_row_hi(s, r);
                    const bool same = (hi < lo) ? (rl == rh) : (rl == lo && rh == hi + 1);
                    if (!same) {
                        std::printf("row %d: keys [%lld, %lld], row bounds [%d, %d)\n", r, lo, hi, rl, rh);
                        return 1;
                    }
                }
                if (hi < lo)
                    continue;   // this row sees no key
                if (lo / 128 < ks || hi / 128 >= ks + nw) {
                    std::printf("ct %d w %d row %d keys [%lld, %lld] outside steps [%d, %d)\n", ct, w, r, lo, hi, ks,
                                ks + nw);
                    return 1;
                }
            }
        }
    }
    return 0;
}

// Without a left bound the kernel walks whole tiles with the step-end forms
// (PartIter::next_t<false, false>, sched_decode_t<false, false>): the same
// parts and tiles as the general forms.
static int check_no_band_forms(const Schedule &s)
{
    if (s.split || s.wl < kSchedUnbounded)
        return 0;
    for (int c = 0; c < s.G; ++c) {
        PartIter a, b;
        a.init_t<false>(s, c);
        b.init_t<false>(s, c);
        Part pa, pb;
        for (;;) {
            const bool ma = a.next_t<false, true>(s, pa), mb = b.next_t<false, false>(s, pb);
            if (ma != mb || (ma && (pa.tile != pb.tile || pa.kb != pb.kb || pa.ke != pb.ke))) {
                std::printf("c=%d: step-end walk differs at tile %d\n", c, pa.tile);
                return 1;
            }
            if (!ma)
                break;
            int bh1, ct1, bh2, ct2;
            sched_decode_t<false, true>(s, pa.tile, bh1, ct1);
            sched_decode_t<false, false>(s, pa.tile, bh2, ct2);
            if (bh1 != bh2 || ct1 != ct2) {
                std::printf("tile %d decodes differently\n", pa.tile);
                return 1;
            }
        }
    }
    return 0;
}

static int check_schedule(const Schedule &s, bool planned, int wl, int wr)
{
    const int G = s.G, split = s.split;
    if (check_key_ranges(s, wl, wr) || check_no_band_forms(s))
        return 1;
    std::vector<std::vector<int>> cover(s.T);
    for (int t = 0; t < s.T; ++t)
        cover[t].assign(sched_steps(s, t), 0);
    std::map<std::pair<int, int>, std::set<int>> slots_with_work;   // (tile, w) -> slots
    std::set<int> used_slots;
    long long units = 0;
    const int tail0 = s.W * G;   // tail split: tiles before tail0 are whole tiles, W per CTA
    if (s.W > 0 && (!split || s.causal)) {
        std::printf("whole tiles before the units outside a non-causal balanced schedule\n");
        return 1;
    }
    for (int c = 0; c < G; ++c) {
        PartIter it;
        it.init(s, c);
        Part p;
        int nparts = 0;
        while (it.next(s, p)) {
            ++nparts;
            if (p.tile < 0 || p.tile >= s.T || p.kb < 0 || p.ke > (int)cover[p.tile].size() || p.kb >= p.ke) {
                std::printf("bad part c=%d tile=%d kb=%d ke=%d\n", c, p.tile, p.kb, p.ke);
                return 1;
            }
            if (split && p.tile < tail0) {   // a whole tile of the tail split: CTA c's own, kept whole
                if (p.tile / s.W != c || p.kb != 0 || p.ke != (int)cover[p.tile].size() || p.slot != -1) {
                    std::printf("c=%d: whole part of tile %d wrong (kb %d ke %d slot %d)\n", c, p.tile, p.kb, p.ke, p.slot);
                    return 1;
                }
                for (int j = p.kb; j < p.ke; ++j)
                    ++cover[p.tile][j];
                units += p.ke - p.kb;
                continue;
            }
            if (split && p.ts != (int)sched_prefix(s, p.tile)) {
                std::printf("part of tile %d carries first unit %d, expected %lld\n", p.tile, p.ts, sched_prefix(s, p.tile));
                return 1;
            }
            if (split) {   // the neighbour walk from this CTA finds the same CTAs as the searches
                int pt, n, clo, chi, lo2, hi2;
                sched_tile_ctas(s, p.tile, pt, n, clo, chi);
                sched_tile_ctas_near(s, p.ts, n, c, lo2, hi2);
                if (lo2 != clo || hi2 != chi) {
                    std::printf("tile %d: CTAs %d..%d by search, %d..%d by walk from %d\n", p.tile, clo, chi, lo2, hi2, c);
                    return 1;
                }
            }
            for (int j = p.kb; j < p.ke; ++j)
                ++cover[p.tile][j];
            units += p.ke - p.kb;
            const bool whole = p.kb == 0 && p.ke == (int)cover[p.tile].size();
            if (split && nparts > 2 && !whole) {   // partial parts come first
                std::printf("partial part %d of c=%d comes late\n", nparts, c);
                return 1;
            }
            if (split) {
                if (p.slot < 2 * c || p.slot > 2 * c + 1) {
                    std::printf("slot %d out of range for c=%d\n", p.slot, c);
                    return 1;
                }
                int bh, ct;
                sched_decode(s, p.tile, bh, ct);
                for (int w = 0; w < 2; ++w) {
                    const int nw = sched_kv_tiles(s, ct, w);
                    const bool work = p.kb < nw;
                    const bool direct = p.kb == 0 && p.ke >= nw;
                    if (work && !direct) {
                        if (!used_slots.insert(p.slot * 2 + w).second) {
                            std::printf("slot %d reused (tile %d w %d)\n", p.slot, p.tile, w);
                            return 1;
                        }
                    }
                    if (work)
                        slots_with_work[{p.tile, w}].insert(p.slot);
                }
            } else if (!whole || p.slot != -1) {
                std::printf("round-robin part not whole\n");
                return 1;
            }
        }
        (void)nparts;
    }
    for (int t = 0; t < s.T; ++t)
        for (size_t j = 0; j < cover[t].size(); ++j)
            if (cover[t][j] != 1) {
                std::printf("unit (%d,%zu) covered %d times\n", t, j, cover[t][j]);
                return 1;
            }
    const long long whole_units = split ? (long long)tail0 * s.nkv : 0;   // (non-causal: nkv units per tile)
    if (units != s.U + whole_units) {
        std::printf("units %lld != U %lld + %lld\n", units, s.U, whole_units);
        return 1;
    }
    if (split) {
        for (int t = tail0; t < s.T; ++t) {
            int bh, ct;
            sched_decode(s, t, bh, ct);
            for (int w = 0; w < 2; ++w) {
                const int nw = sched_kv_tiles(s, ct, w);
                int sl[4096];
                const int n = sched_part_slots(s, t, nw, sl, 4096);
                std::set<int> got(sl, sl + (n < 4096 ? n : 4096));
                const auto &want = slots_with_work[{t, w}];
                if (nw == 0 ? n != 0 : (got != want || (int)want.size() != n)) {
                    std::printf("merge slots mismatch tile %d w %d: expected %zu got %d\n", t, w, want.size(), n);
                    return 1;
                }
                if (planned && n > sched_max_parts(s)) {
                    std::printf("tile %d w %d cut into %d parts\n", t, w, n);
                    return 1;
                }
            }
        }
    }
    return 0;
}

// sched_plan_limited with a workspace limit of `limit` bytes: an automatic
// balanced plan that needs more falls back to whole tiles (no workspace);
// one that fits, a whole-tile plan and an explicit balanced request are kept
// as sched_plan makes them.  *fell_back counts the fallbacks seen.
static int check_limited(int N, int Nkv, int BH, int causal, int sms, int wl, int wr, int D,
                         unsigned long long limit, int *fell_back)
{
    const Schedule a = sched_plan(N, Nkv, BH, causal != 0, sms, 0, wl, wr);
    const Schedule l = sched_plan_limited(N, Nkv, BH, causal != 0, sms, 0, wl, wr, D, limit);
    const bool over = a.split && sched_workspace_bytes(a, D) > limit;
    if (over) {
        ++*fell_back;
        const Schedule w = sched_plan(N, Nkv, BH, causal != 0, sms, 1, wl, wr);
        if (l.split || sched_workspace_bytes(l, D) != 0 || l.G != w.G || l.T != w.T || l.U != w.U)
            return 1;
    } else if (l.split != a.split || l.G != a.G || l.T != a.T || l.U != a.U) {
        return 1;
    }
    for (int mode = 1; mode <= 2; ++mode) {   // explicit requests are never changed
        const Schedule e = sched_plan(N, Nkv, BH, causal != 0, sms, mode, wl, wr);
        const Schedule el = sched_plan_limited(N, Nkv, BH, causal != 0, sms, mode, wl, wr, D, limit);
        if (e.split != el.split || e.G != el.G || e.U != el.U)
            return 1;
    }
    return check_schedule(l, true, wl, wr);
}

int main(int argc, char **argv)
{
    // "tail" then "N Nkv BH G gt" cases: tail splits of non-causal heads
    if (argc > 1 && std::string(argv[1]) == "tail") {
        int failures = 0, cases = 0;
        for (int i = 2; i + 5 <= argc; i += 5) {
            const int N = std::atoi(argv[i]), Nkv = std::atoi(argv[i + 1]), BH = std::atoi(argv[i + 2]);
            const int G = std::atoi(argv[i + 3]), gt = std::atoi(argv[i + 4]);
            ++cases;
            if (check(N, Nkv, BH, 0, G, 2, kSchedUnbounded, kSchedUnbounded, gt)) {
                std::printf("FAILED tail N=%d Nkv=%d BH=%d G=%d gt=%d\n", N, Nkv, BH, G, gt);
                ++failures;
            }
        }
        std::printf("%d cases, %d failures\n", cases, failures);
        return failures ? 1 : 0;
    }
    // "limit L" then "N Nkv BH causal sms wl wr D" cases: the no-allocation planner
    if (argc > 2 && std::string(argv[1]) == "limit") {
        const unsigned long long limit = std::strtoull(argv[2], nullptr, 10);
        int failures = 0, cases = 0, fell_back = 0;
        for (int i = 3; i + 8 <= argc; i += 8) {
            int v[8];
            for (int k = 0; k < 8; ++k)
                v[k] = std::atoi(argv[i + k]);
            const int wl = v[5] < 0 ? kSchedUnbounded : v[5], wr = v[6] < 0 ? kSchedUnbounded : v[6];
            ++cases;
            if (check_limited(v[0], v[1], v[2], v[3], v[4], wl, wr, v[7], limit, &fell_back)) {
                std::printf("FAILED limit N=%d Nkv=%d BH=%d causal=%d sms=%d D=%d\n", v[0], v[1], v[2], v[3], v[4], v[7]);
                ++failures;
            }
        }
        std::printf("%d cases, %d failures, %d fallbacks\n", cases, failures, fell_back);
        return failures ? 1 : 0;
    }
    // "N Nkv BH causal G split wl wr" cases, repeated; or "plan" then "N Nkv BH causal sms wl wr" cases
    // (wl, wr < 0: unbounded)
    int failures = 0, cases = 0;
    const bool plan = argc > 1 && std::string(argv[1]) == "plan";
    const int width = plan ? 7 : 8;
    for (int i = plan ? 2 : 1; i + width <= argc; i += width) {
        const int N = std::atoi(argv[i]), Nkv = std::atoi(argv[i + 1]), BH = std::atoi(argv[i + 2]);
        const int causal = std::atoi(argv[i + 3]), G = std::atoi(argv[i + 4]), split = plan ? 0 : std::atoi(argv[i + 5]);
        int wl = std::atoi(argv[i + width - 2]), wr = std::atoi(argv[i + width - 1]);
        wl = wl < 0 ? kSchedUnbounded : wl;
        wr = wr < 0 ? kSchedUnbounded : wr;
        ++cases;
        if (plan ? check_plan(N, Nkv, BH, causal, G, wl, wr) : check(N, Nkv, BH, causal, G, split, wl, wr)) {
            std::printf("FAILED N=%d Nkv=%d BH=%d causal=%d G/sms=%d split=%d plan=%d wl=%d wr=%d\n", N, Nkv, BH, causal, G,
                        split, (int)plan, wl, wr);
            ++failures;
        }
    }
    std::printf("%d cases, %d failures\n", cases, failures);
    return failures ? 1 : 0;
}
