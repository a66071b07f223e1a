// fa_schedule.h -- work decomposition of the attention forward over the
// persistent CTAs (host and device code; builds with nvcc and plain g++).
//
// A CTA tile is 256 query rows of one head (two 128-row Q tiles); a unit is
// one K/V step (128 keys) of one CTA tile.  Causal tiles stop at the diagonal
// ("A09 - Advanced Triton & FlashAttention", causal masking: the loop bound),
// so their step counts differ.  Non-causal tiles are ordered head-major.  For
// the round-robin schedule causal tiles come in groups of one tile row (ct)
// over all heads, the heads interleaved, the groups longest first ("How to
// profile and optimise kernels", causal launch order).  For the balanced one
// tile rows are paired longest with shortest (C - 1 with 0, C - 2 with 1, ...)
// and each pair's tiles alternate long, short per head, so that every range
// of units holds a similar mix of long and short tiles; the middle row of an
// odd C comes last.
//
// Two schedules:
//  * round-robin (serpentine): round r hands tiles rG .. rG + G - 1 to the
//    CTAs, CTA c taking the c-th in even rounds and the (G - 1 - c)-th in odd
//    rounds, so the CTAs that took the longest tiles of one round take the
//    shortest of the next (for the longest-first causal order this is as
//    balanced as a greedy longest-first assignment, and 20 % shorter than
//    plain round-robin at N = 4096)
//  * balanced: CTA c runs units [floor(U c / G), floor(U (c+1) / G)) of the
//    ordered unit sequence, U = total units.  A tile cut by a range boundary
//    is computed in parts; each part writes a partial result (O normalised by
//    its own row sums, with its row max m and sum l) to a workspace slot, and
//    the last part to finish merges them.  A CTA holds at most two partial
//    parts (the first and the last of its range), in slots 2c and 2c + 1.
//    The mixed causal order spreads the fixed cost of each part evenly too.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

constexpr int kSchedBM = 128;        // rows per Q tile
constexpr int kSchedBN = 128;        // keys per step
constexpr int kSchedCtaRows = 256;   // rows per CTA tile
constexpr int kSchedMaxGrid = 160;   // CTAs of a balanced-schedule launch, at most
constexpr long long kSchedMaxUnits = 0x3fffffffLL;   // units of a balanced schedule, at most (32-bit unit indices)
constexpr int kSchedMaxParts = 8;                    // parts of one tile in a balanced schedule, at most

struct Schedule {
    int N;          // query rows per head
    int Nkv;        // keys per head
    int off;        // causal alignment: query i sees keys j <= i + off (off = Nkv - N, bottom-right)
    int BH;         // batch * heads
    int C;          // CTA tiles per head: ceil(N / 256)
    int T;          // CTA tiles: BH * C
    int nkv;        // K/V steps of a full row: ceil(Nkv / 128)
    int causal;     // 0 or 1
    int G;          // CTAs in the grid
    int split;      // 1: balanced schedule with partial tiles
    long long U;    // total units (the balanced schedule requires U <= kSchedMaxUnits)
    int range[kSchedMaxGrid + 1];   // balanced: range[c] = floor(U c / G), filled by sched_fill_ranges
};

// Causal steps of rows up to `last`: up to the step holding key last + off.
// Rows that see no key at all (last + off < 0) still take one step, fully
// masked, so that their O = 0 and LSE = -inf get written.
FA_HD int sched_causal_steps(const Schedule &s, int last)
{
    const int vis = last + s.off;
    if (vis < 0)
        return 1;
    const int n = vis / kSchedBN + 1;
    return n < s.nkv ? n : s.nkv;
}

// K/V steps visited by Q tile w (0 or 1) of CTA tile ct; 0 if it holds no valid row.
FA_HD int sched_kv_tiles(const Schedule &s, int ct, int w)
{
    const int r0 = ct * kSchedCtaRows + w * kSchedBM;
    if (r0 >= s.N)
        return 0;
    if (!s.causal)
        return s.nkv;
    const int last = (r0 + kSchedBM - 1 < s.N - 1) ? r0 + kSchedBM - 1 : s.N - 1;
    return sched_causal_steps(s, last);
}

// Steps of CTA tile ct: those of its last valid Q tile.
FA_HD int sched_steps_ct(const Schedule &s, int ct)
{
    if (!s.causal)
        return s.nkv;
    const int last = (ct * kSchedCtaRows + kSchedCtaRows - 1 < s.N - 1) ? ct * kSchedCtaRows + kSchedCtaRows - 1 : s.N - 1;
    return sched_causal_steps(s, last);
}

FA_HD void sched_decode(const Schedule &s, int t, int &bh, int &ct)
{
    if (s.causal && s.split) {   // pairs of tile rows, long and short alternating per head
        const int q = t / (2 * s.BH);
        if (q < s.C / 2) {
            const int i = t - q * 2 * s.BH;
            bh = i / 2;
            ct = (i & 1) ? q : s.C - 1 - q;
        } else {                  // the middle row of an odd C
            bh = t - q * 2 * s.BH;
            ct = s.C / 2;
        }
    } else if (s.causal) {        // one tile row per group, longest first, heads interleaved
        ct = s.C - 1 - t / s.BH;
        bh = t % s.BH;
    } else {          // head-major: neighbouring CTAs share a head's K/V in L2
        bh = t / s.C;
        ct = t % s.C;
    }
}

// The round-robin order alone (the kernel's whole-tile variant).
FA_HD void sched_decode_rr(const Schedule &s, int t, int &bh, int &ct)
{
    if (s.causal) {
        ct = s.C - 1 - t / s.BH;
        bh = t % s.BH;
    } else {
        bh = t / s.C;
        ct = t % s.C;
    }
}

FA_HD int sched_steps_rr(const Schedule &s, int t)
{
    if (!s.causal)
        return s.nkv;
    return sched_steps_ct(s, s.C - 1 - t / s.BH);
}

template <bool SPLIT>
FA_HD void sched_decode_t(const Schedule &s, int t, int &bh, int &ct)
{
    if (SPLIT)
        sched_decode(s, t, bh, ct);
    else
        sched_decode_rr(s, t, bh, ct);
}

FA_HD int sched_steps(const Schedule &s, int t)
{
    int bh, ct;
    sched_decode(s, t, bh, ct);
    return sched_steps_ct(s, ct);
}

// Units of all tiles before tile t.
FA_HD long long sched_prefix(const Schedule &s, int t)
{
    if (!s.causal)
        return (long long)t * s.nkv;
    if (s.split) {
        const int q = t / (2 * s.BH);
        long long acc = 0;
        for (int r = 0; r < q; ++r)
            acc += (long long)s.BH * (sched_steps_ct(s, s.C - 1 - r) + sched_steps_ct(s, r));
        const int i = t - q * 2 * s.BH;
        if (q < s.C / 2) {
            const int lg = sched_steps_ct(s, s.C - 1 - q), sh = sched_steps_ct(s, q);
            return acc + (long long)(i / 2) * (lg + sh) + ((i & 1) ? lg : 0);
        }
        return acc + (long long)i * sched_steps_ct(s, s.C / 2);
    }
    const int g = t / s.BH;   // tiles come in groups of BH with equal step counts
    long long acc = 0;
    for (int q = 0; q < g; ++q)
        acc += (long long)s.BH * sched_steps_ct(s, s.C - 1 - q);
    return acc + (long long)(t - g * s.BH) * sched_steps_ct(s, s.C - 1 - g);
}

FA_HD long long sched_total_units(const Schedule &s)
{
    return sched_prefix(s, s.T - 1) + sched_steps(s, s.T - 1);
}

// Fill the table of CTA range starts (host side; keeps 64-bit divisions out of
// the kernel).  Requires G <= kSchedMaxGrid and U <= kSchedMaxUnits.
inline void sched_fill_ranges(Schedule &s)
{
    for (int c = 0; c <= s.G; ++c)
        s.range[c] = (int)(((unsigned long long)s.U * (unsigned long long)c) / (unsigned long long)s.G);
}

// CTA whose range holds unit u (balanced schedule): the last c with
// range[c] <= u, which is a CTA with a non-empty range.
FA_HD int sched_cta_of_unit(const Schedule &s, int u)
{
    int lo = 0, hi = s.G - 1;   // range[0] = 0 <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (s.range[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Tile containing unit u (balanced schedule), with its first unit.
FA_HD int sched_tile_of_unit(const Schedule &s, int u, int &tstart)
{
    if (!s.causal) {
        const int t = u / s.nkv;
        tstart = t * s.nkv;
        return t;
    }
    // (balanced schedules only) pairs of tile rows, then the middle row of an odd C
    int acc = 0;
    for (int q = 0; q < s.C / 2; ++q) {
        const int lg = sched_steps_ct(s, s.C - 1 - q), sh = sched_steps_ct(s, q);
        const int gu = s.BH * (lg + sh);
        if (u < acc + gu) {
            const int rel = u - acc, pair = rel / (lg + sh), rem = rel - pair * (lg + sh);
            const bool second = rem >= lg;
            tstart = acc + pair * (lg + sh) + (second ? lg : 0);
            return q * 2 * s.BH + 2 * pair + (second ? 1 : 0);
        }
        acc += gu;
    }
    const int st = sched_steps_ct(s, s.C / 2);
    const int i = (u - acc) / st;
    tstart = acc + i * st;
    return (s.C / 2) * 2 * s.BH + i;
}

// A CTA's share of one tile: steps [kb, ke); slot >= 0 names its partial-result
// slot (balanced schedule), -1 for the round-robin schedule.
struct Part {
    int tile;
    int kb;
    int ke;
    int slot;
    int ts;     // balanced: the tile's first unit in the ordered sequence (0 for round-robin)
};

// The parts of CTA c.  Every role of the CTA walks the same sequence.  In the
// balanced schedule a CTA's range holds at most two partial parts, the first
// and the last; the last is taken first, then the rest in order, so that both
// partial parts (and the merges of their tiles, by whichever CTA finishes a
// tile last) come early and overlap the whole tiles that follow instead of
// waiting at the end of the launch.  The schedule is passed to each call
// rather than held, so that on the device it is read straight from kernel
// parameter space.
struct PartIter {
    int c;
    int u, ue, tstart;   // balanced: next unit, end of the in-order units, first unit of tile t; round-robin: u = round
    int t, tsteps;
    int lt, lke, lts;    // balanced: the range's last part, tile lt (first unit lts) steps [0, lke), still to come (lt >= 0)

    // The kernel knows its schedule at compile time (SPLIT = s.split) and
    // takes only that path; init / next decide at run time (host code).
    template <bool SPLIT>
    FA_HD void init_t(const Schedule &s, int c_)
    {
        c = c_;
        lt = -1;
        lke = 0;
        lts = 0;
        if (SPLIT) {
            u = s.range[c];
            ue = s.range[c + 1];
            if (u < ue) {
                int ls;
                const int tl = sched_tile_of_unit(s, ue - 1, ls);
                if (ls > u) {   // the range ends in a later tile than it starts in
                    lt = tl;
                    lke = ue - ls;
                    lts = ls;
                    ue = ls;
                }
                t = sched_tile_of_unit(s, u, tstart);
            } else {
                t = s.T;
            }
            tsteps = (t < s.T) ? sched_steps(s, t) : 0;
        } else {
            t = c;
            u = ue = tstart = 0;
            tsteps = 0;
        }
    }

    template <bool SPLIT>
    FA_HD bool next_t(const Schedule &s, Part &p)
    {
        if (SPLIT) {
            if (lt >= 0) {
                p.tile = lt;
                p.kb = 0;
                p.ke = lke;
                p.slot = 2 * c + 1;
                p.ts = lts;
                lt = -1;
                return true;
            }
            if (u >= ue)
                return false;
            p.tile = t;
            p.kb = u - tstart;
            p.ke = (ue - tstart < tsteps) ? ue - tstart : tsteps;
            p.slot = 2 * c + ((u == s.range[c]) ? 0 : 1);
            p.ts = tstart;
            u = tstart + p.ke;
            if (p.ke == tsteps) {
                tstart += tsteps;
                ++t;
                tsteps = (t < s.T) ? sched_steps(s, t) : 0;
            }
            return true;
        }
        if (t >= s.T)
            return false;
        p.tile = t;
        p.kb = 0;
        p.ke = sched_steps_rr(s, t);
        p.slot = -1;
        p.ts = 0;
        ++u;
        t = u * s.G + ((u & 1) ? s.G - 1 - c : c);
        return true;
    }

    FA_HD void init(const Schedule &s, int c_)
    {
        if (s.split)
            init_t<true>(s, c_);
        else
            init_t<false>(s, c_);
    }

    FA_HD bool next(const Schedule &s, Part &p)
    {
        return s.split ? next_t<true>(s, p) : next_t<false>(s, p);
    }
};

// The CTAs that may hold parts of tile t (first unit pt, n units): clo .. chi.
FA_HD void sched_tile_ctas(const Schedule &s, int t, int &pt, int &n, int &clo, int &chi)
{
    pt = (int)sched_prefix(s, t);
    n = sched_steps(s, t);
    clo = sched_cta_of_unit(s, pt);
    chi = sched_cta_of_unit(s, pt + n - 1);
}

// The CTAs that hold parts of the tile with first unit pt and n units, found
// by walking out from c0, a CTA known to hold one of them: clo .. chi.
FA_HD void sched_tile_ctas_near(const Schedule &s, int pt, int n, int c0, int &clo, int &chi)
{
    clo = c0;
    while (clo > 0 && s.range[clo] > pt)
        --clo;
    chi = c0;
    while (chi + 1 < s.G && s.range[chi + 1] < pt + n)
        ++chi;
}

// Whether CTA c holds a part of tile t (first unit pt, n units) in which a Q
// tile visiting nw steps has work; if so, writes the part's slot.
FA_HD bool sched_part_slot(const Schedule &s, int pt, int n, int nw, int c, int &slot)
{
    const int st = s.range[c], en = s.range[c + 1];
    const int kb = (st > pt) ? st - pt : 0;
    const int ke = (en - pt < n) ? en - pt : n;
    slot = 2 * c + ((pt > st) ? 1 : 0);
    return ke > kb && kb < nw;   // CTAs with empty ranges hold no part
}

// Parts of tile t in which Q tile w (visiting nw steps) has work, for the
// merge: returns their count and writes up to `max_slots` of their slots.
FA_HD int sched_part_slots(const Schedule &s, int t, int nw, int *slots, int max_slots)
{
    int pt, n, clo, chi;
    sched_tile_ctas(s, t, pt, n, clo, chi);
    int count = 0;
    for (int c = clo; c <= chi; ++c) {
        int slot;
        if (sched_part_slot(s, pt, n, nw, c, slot)) {
            if (slots && count < max_slots)
                slots[count] = slot;
            ++count;
        }
    }
    return count;
}

// Work decomposition for one call on `sms` SMs (host side).  The balanced
// schedule is taken when the round-robin schedule of whole tiles would leave
// the machine idle in its last wave for more than ~4% of the run and for at
// least kSchedMinGain steps (a split tile costs its parts a partial write and
// one of them a merge); its grid is kept small enough that no tile is cut
// into more than kSchedMaxParts parts.  Parts have fixed costs (a partial
// write, a merge, a pipeline start), so with many tiles the balanced schedule
// is taken only where every CTA's range spans at least two tiles, and not
// for causal attention, whose short tiles lose to those costs (measured).
// With few long tiles -- decoding a few queries against many keys -- whole
// tiles would leave most SMs idle, and the balanced schedule (split-KV) is
// taken whenever it at least halves the makespan.
constexpr int kSchedMinGain = 4;

// mode: 0 = as above, 1 = round-robin, 2 = balanced wherever it can be built.
// N query rows against Nkv keys per head.
inline Schedule sched_plan(int N, int Nkv, int BH, bool causal, int sms, int mode = 0)
{
    Schedule s{};
    s.N = N;
    s.Nkv = Nkv;
    s.off = causal ? Nkv - N : 0;
    s.BH = BH;
    s.C = (N + kSchedCtaRows - 1) / kSchedCtaRows;
    s.T = BH * s.C;
    s.nkv = (Nkv + kSchedBN - 1) / kSchedBN;
    s.causal = causal ? 1 : 0;
    s.split = 0;
    s.G = s.T < sms ? s.T : sms;
    if (s.G > kSchedMaxGrid)   // (a larger part than this library targets runs on kSchedMaxGrid CTAs)
        s.G = kSchedMaxGrid;
    s.U = sched_total_units(s);
    // round-robin (serpentine) makespan: the largest CTA load
    long long rr = 0;
    {
        long long load[kSchedMaxGrid] = {};
        for (int t = 0; t < s.T; ++t) {
            const int r = t / s.G, k = t - r * s.G;
            load[(r & 1) ? s.G - 1 - k : k] += sched_steps(s, t);
        }
        for (int c = 0; c < s.G; ++c)
            rr = load[c] > rr ? load[c] : rr;
    }
    if (s.U > kSchedMaxUnits || mode == 1)
        return s;
    const int max_steps = sched_steps_ct(s, s.C - 1);   // the last tile row is the longest
    long long G = (s.U < sms) ? s.U : sms;
    if (G > kSchedMaxGrid)
        G = kSchedMaxGrid;
    // Ranges of at least `need` units cut a tile of max_steps steps into at
    // most (max_steps - 1) / need + 2 <= kSchedMaxParts parts.
    const long long need = (max_steps - 1 + kSchedMaxParts - 3) / (kSchedMaxParts - 2);
    if (need > 0 && s.U / G < need)
        G = s.U / need;
    if (G < 1)
        return s;
    const long long balanced = (s.U + G - 1) / G;
    const bool many_tiles = !causal && balanced >= 2LL * max_steps && rr * 100 > balanced * 104 &&
                            rr - balanced >= kSchedMinGain;
    const bool few_long_tiles = 2LL * s.T <= sms && max_steps >= 32 && rr >= 2 * balanced;
    const bool pays = many_tiles || few_long_tiles;
    if (mode == 2 || pays) {
        s.split = 1;
        s.G = (int)G;
        s.U = sched_total_units(s);   // the same total in the balanced order
        sched_fill_ranges(s);
    }
    return s;
}

}  // namespace fa
