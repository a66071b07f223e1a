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

static int check_schedule(const Schedule &s, bool planned);

static int check(int N, int Nkv, int BH, int causal, int G, int split)
{
    Schedule s{};
    s.N = N;
    s.Nkv = Nkv;
    s.off = causal ? Nkv - N : 0;
    s.BH = BH;
    s.C = (N + 255) / 256;
    s.T = BH * s.C;
    s.nkv = (Nkv + 127) / 128;
    s.causal = causal;
    s.G = G;
    s.split = split;
    s.U = sched_total_units(s);
    if (G > kSchedMaxGrid || s.U > kSchedMaxUnits)
        return 0;
    sched_fill_ranges(s);
    return check_schedule(s, false);
}

// The planner's schedule for `sms` SMs: valid, and a balanced one cuts no
// tile into more parts than the merge handles.
static int check_plan(int N, int Nkv, int BH, int causal, int sms)
{
    const Schedule s = sched_plan(N, Nkv, BH, causal != 0, sms);
    if (s.G < 1 || (!s.split && s.G != (s.T < sms ? s.T : sms))) {
        std::printf("bad grid %d\n", s.G);
        return 1;
    }
    return check_schedule(s, true);
}

static int check_schedule(const Schedule &s, bool planned)
{
    const int G = s.G, split = s.split;
    std::vector<std::vector<int>> cover(s.T);
    for (int t = 0; t < s.T; ++t)
        cover[t].assign(sched_steps(s, t), 0);
    std::map<std::pair<int, int>, std::set<int>> slots_with_work;   // (tile, w) -> slots
    std::set<int> used_slots;
    long long units = 0;
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
    if (units != s.U) {
        std::printf("units %lld != U %lld\n", units, s.U);
        return 1;
    }
    if (split) {
        for (int t = 0; t < s.T; ++t) {
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
                if (planned && n > kSchedMaxParts) {
                    std::printf("tile %d w %d cut into %d parts\n", t, w, n);
                    return 1;
                }
            }
        }
    }
    return 0;
}

int main(int argc, char **argv)
{
    // "N Nkv BH causal G split" cases, repeated; or "plan" then "N Nkv BH causal sms" cases
    int failures = 0, cases = 0;
    const bool plan = argc > 1 && std::string(argv[1]) == "plan";
    const int width = plan ? 5 : 6;
    for (int i = plan ? 2 : 1; i + width <= argc; i += width) {
        const int N = std::atoi(argv[i]), Nkv = std::atoi(argv[i + 1]), BH = std::atoi(argv[i + 2]);
        const int causal = std::atoi(argv[i + 3]), G = std::atoi(argv[i + 4]), split = plan ? 0 : std::atoi(argv[i + 5]);
        ++cases;
        if (plan ? check_plan(N, Nkv, BH, causal, G) : check(N, Nkv, BH, causal, G, split)) {
            std::printf("FAILED N=%d Nkv=%d BH=%d causal=%d G/sms=%d split=%d plan=%d\n", N, Nkv, BH, causal, G, split,
                        (int)plan);
            ++failures;
        }
    }
    std::printf("%d cases, %d failures\n", cases, failures);
    return failures ? 1 : 0;
}
