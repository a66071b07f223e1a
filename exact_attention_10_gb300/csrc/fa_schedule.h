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
//  * tail split (a balanced schedule with W > 0, non-causal only): CTA c
//    first runs whole tiles cW .. cW + W - 1, W = floor(T / G); only the
//    T - WG tiles of the last, partial wave are laid out as units (from 0)
//    and split into ranges as above, over the first Gt CTAs.  A CTA's tail
//    part comes first, so that the merges overlap its whole tiles; and only
//    the last wave's tiles are cut, about half as many parts and merges as
//    when every range is cut (each CTA then has one tail part, not two).
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
constexpr int kSchedMaxParts = 32;      // parts of one tile in a balanced schedule: at most 32 for heads of
constexpr int kSchedMaxPartsTall = 8;    // <= 32 query rows, 16 for <= 64, 8 for taller heads (the merge
constexpr int kSchedShortRows = 64;      // warp stages (m, l) of 8 parts x 128 rows, 16 x 64 or 32 x 32)
constexpr int kSchedUnbounded = 0x3fffffff;          // a band bound that never binds

struct Schedule {
    int N;          // query rows per head
    int Nkv;        // keys per head
    int off;        // masked ("causal"): query i sits at key position i + off (off = Nkv - N, bottom-right)
    int wl, wr;     // masked: query i sees keys [i + off - wl, i + off + wr] (kSchedUnbounded: no bound);
                    // a bound that cannot bind is stored as kSchedUnbounded (sched_band_normalize)
    int ka, ra;     // masked: the first key of row r lies in step ((r + ra) >> 7) + ka (floor division of r + off - wl)
    int kb, rb;     // masked: the last key of row r lies in step ((r + rb) >> 7) + kb (floor division of r + off + wr)
    int BH;         // batch * heads
    int C;          // CTA tiles per head: ceil(N / 256)
    int T;          // CTA tiles: BH * C
    int nkv;        // K/V steps of a full row: ceil(Nkv / 128)
    int causal;     // 0 or 1
    int rev;        // masked: 1 if the first tile row is longer than the last (a band bounded on the left only)
    int G;          // CTAs in the grid
    int split;      // 1: balanced schedule with partial tiles
    int W;          // balanced: whole tiles per CTA before its units (tail split; 0: every tile is in units)
    long long U;    // units laid out in ranges (balanced; the tail's alone when W > 0; at most kSchedMaxUnits)
    int range[kSchedMaxGrid + 1];   // balanced: range[c] = floor(U c / G), filled by sched_fill_ranges
};

// Band bounds that cannot bind become kSchedUnbounded: with off = Nkv - N,
// query rows sit at positions off .. Nkv - 1, so wl >= Nkv clips nothing on
// the left and wr >= N - 1 nothing on the right.  After this, r + off - wl
// and the step offsets below stay within 32-bit range for any valid sizes.
FA_HD void sched_band_normalize(int N, int Nkv, int &wl, int &wr)
{
    if (wl < 0 || wl >= Nkv || wl >= kSchedUnbounded)
        wl = kSchedUnbounded;
    if (wr < 0 || wr >= N - 1 || wr >= kSchedUnbounded)
        wr = kSchedUnbounded;
}

// Masked attention (a band, of which causal is one case): rows first .. last
// see keys [first + off - wl, last + off + wr]; the K/V steps holding them are
// [ks, ke).  Rows whose bands hold no key still take one step, fully masked,
// so that their O = 0 and LSE = -inf get written.  (32-bit arithmetic on the
// offsets that sched_plan precomputes: floor((r + x) / 128) = ((r + rx) >> 7) + kx
// with x = 128 kx + rx, 0 <= rx < 128.)
FA_HD void sched_band_steps(const Schedule &s, int first, int last, int &ks, int &ke)
{
    int a = (int)(((uint32_t)first + (uint32_t)s.ra) >> 7) + s.ka;
    int b = (int)(((uint32_t)last + (uint32_t)s.rb) >> 7) + s.kb + 1;
    a = a < 0 ? 0 : (a > s.nkv - 1 ? s.nkv - 1 : a);
    b = b > s.nkv ? s.nkv : b;
    ks = a;
    ke = b <= a ? a + 1 : b;
}

// Keys of query row r (0 <= r < N) under the band, clipped to [0, Nkv):
// [sched_row_lo, sched_row_hi), empty when they are equal.
FA_HD int sched_row_lo(const Schedule &s, int r)
{
    const int lo = r + s.off - s.wl;   // (normalised wl < Nkv: no overflow)
    return (s.wl >= kSchedUnbounded || lo < 0) ? 0 : lo;
}

FA_HD int sched_row_hi(const Schedule &s, int r)
{
    const int pos = r + s.off;   // <= Nkv - 1
    if (s.wr >= kSchedUnbounded || s.wr >= s.Nkv - pos - 1)
        return s.Nkv;
    const int hi = pos + s.wr + 1;
    return hi < 0 ? 0 : hi;
}

// First K/V step of CTA tile ct (its rows' earliest visible key); 0 unmasked.
FA_HD int sched_kv_start(const Schedule &s, int ct)
{
    if (!s.causal)
        return 0;
    const int first = ct * kSchedCtaRows;
    const int last = (first + kSchedCtaRows - 1 < s.N - 1) ? first + kSchedCtaRows - 1 : s.N - 1;
    int ks, ke;
    sched_band_steps(s, first, last, ks, ke);
    return ks;
}

// K/V steps visited by Q tile w (0 or 1) of CTA tile ct, counted from the
// tile's first step sched_kv_start(ct) (a Q tile's steps are a prefix of its
// CTA tile's: a later Q tile may take a first step that is fully masked for
// it); 0 if it holds no valid row.
FA_HD int sched_kv_tiles(const Schedule &s, int ct, int w)
{
    const int r0 = ct * kSchedCtaRows + w * kSchedBM;
    if (r0 >= s.N)
        return 0;
    if (!s.causal)
        return s.nkv;
    const int last = (r0 + kSchedBM - 1 < s.N - 1) ? r0 + kSchedBM - 1 : s.N - 1;
    int ks, ke;
    sched_band_steps(s, r0, last, ks, ke);
    return ke - sched_kv_start(s, ct);
}

// Masks without a left bound start every row's steps at 0: the steps of rows
// up to `last` end at this step (the end half of sched_band_steps alone).
FA_HD int sched_step_end(const Schedule &s, int last)
{
    const int b = (int)(((uint32_t)last + (uint32_t)s.rb) >> 7) + s.kb + 1;
    return b < 1 ? 1 : (b > s.nkv ? s.nkv : b);
}

// sched_kv_tiles in the kernel: BAND (a left bound) takes the general form,
// other masks the step end alone.
template <bool BAND>
FA_HD int sched_kv_tiles_t(const Schedule &s, int ct, int w)
{
    if (BAND)
        return sched_kv_tiles(s, ct, w);
    const int r0 = ct * kSchedCtaRows + w * kSchedBM;
    if (r0 >= s.N)
        return 0;
    if (!s.causal)
        return s.nkv;
    return sched_step_end(s, (r0 + kSchedBM - 1 < s.N - 1) ? r0 + kSchedBM - 1 : s.N - 1);
}

// Steps of CTA tile ct: from its first step to its last valid row's last.
FA_HD int sched_steps_ct(const Schedule &s, int ct)
{
    if (!s.causal)
        return s.nkv;
    const int first = ct * kSchedCtaRows;
    const int last = (first + kSchedCtaRows - 1 < s.N - 1) ? first + kSchedCtaRows - 1 : s.N - 1;
    int ks, ke;
    sched_band_steps(s, first, last, ks, ke);
    return ke - ks;
}

// Parts a tile of this schedule may be cut into: decoding-sized heads take
// more (32 for at most 32 query rows, 16 for at most 64), so a few long heads
// spread over more SMs; taller heads 8.  The merge warp's (m, l) staging is
// the same size in every case (sched_ml_rows rows per part).
FA_HD int sched_max_parts(const Schedule &s)
{
    return s.N <= kSchedShortRows / 2 ? kSchedMaxParts : (s.N <= kSchedShortRows ? kSchedMaxParts / 2 : kSchedMaxPartsTall);
}

// Rows of (m, l) the merge stages per part for a merge of `nparts` parts.
FA_HD constexpr int sched_ml_rows(int nparts)
{
    return nparts > kSchedMaxParts / 2 ? kSchedShortRows / 2 : (nparts > kSchedMaxPartsTall ? kSchedShortRows : 128);
}

// Tile rows by length: the q-th longest and the q-th shortest (step counts
// are monotone in the row for causal masks and one-sided bands, and equal but
// for the clipped ends for two-sided ones).
FA_HD int sched_long_row(const Schedule &s, int q)
{
    return s.rev ? q : s.C - 1 - q;
}

FA_HD int sched_short_row(const Schedule &s, int q)
{
    return s.rev ? s.C - 1 - q : q;
}

FA_HD void sched_decode(const Schedule &s, int t, int &bh, int &ct)
{
    if (s.causal && s.split) {   // pairs of tile rows, long and short alternating per head
        const int q = t / (2 * s.BH);
        if (q < s.C / 2) {
            const int i = t - q * 2 * s.BH;
            bh = i / 2;
            ct = (i & 1) ? sched_short_row(s, q) : sched_long_row(s, q);
        } else {                  // the middle row of an odd C
            bh = t - q * 2 * s.BH;
            ct = s.C / 2;
        }
    } else if (s.causal) {        // one tile row per group, longest first, heads interleaved
        ct = sched_long_row(s, t / s.BH);
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
        ct = sched_long_row(s, t / s.BH);
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
    return sched_steps_ct(s, sched_long_row(s, t / s.BH));
}

// The kernel's forms: BAND = false (no left bound) knows that rows are
// longest last (rev = 0) and that steps start at 0.
template <bool SPLIT, bool BAND = true>
FA_HD void sched_decode_t(const Schedule &s, int t, int &bh, int &ct)
{
    if (SPLIT) {
        sched_decode(s, t, bh, ct);
    } else if (BAND) {
        sched_decode_rr(s, t, bh, ct);
    } else if (s.causal) {
        ct = s.C - 1 - t / s.BH;
        bh = t % s.BH;
    } else {
        bh = t / s.C;
        ct = t % s.C;
    }
}

template <bool BAND>
FA_HD int sched_steps_rr_t(const Schedule &s, int t)
{
    if (BAND)
        return sched_steps_rr(s, t);
    if (!s.causal)
        return s.nkv;
    const int first = (s.C - 1 - t / s.BH) * kSchedCtaRows;
    return sched_step_end(s, (first + kSchedCtaRows - 1 < s.N - 1) ? first + kSchedCtaRows - 1 : s.N - 1);
}

FA_HD int sched_steps(const Schedule &s, int t)
{
    int bh, ct;
    sched_decode(s, t, bh, ct);
    return sched_steps_ct(s, ct);
}

// Units of all tiles before tile t (tail split: the tail's tiles before t,
// for t >= WG).
FA_HD long long sched_prefix(const Schedule &s, int t)
{
    if (!s.causal)
        return (long long)(t - s.W * s.G) * s.nkv;
    if (s.split) {
        const int q = t / (2 * s.BH);
        long long acc = 0;
        for (int r = 0; r < q; ++r)
            acc += (long long)s.BH * (sched_steps_ct(s, sched_long_row(s, r)) + sched_steps_ct(s, sched_short_row(s, r)));
        const int i = t - q * 2 * s.BH;
        if (q < s.C / 2) {
            const int lg = sched_steps_ct(s, sched_long_row(s, q)), sh = sched_steps_ct(s, sched_short_row(s, q));
            return acc + (long long)(i / 2) * (lg + sh) + ((i & 1) ? lg : 0);
        }
        return acc + (long long)i * sched_steps_ct(s, s.C / 2);
    }
    const int g = t / s.BH;   // tiles come in groups of BH with equal step counts
    long long acc = 0;
    for (int q = 0; q < g; ++q)
        acc += (long long)s.BH * sched_steps_ct(s, sched_long_row(s, q));
    return acc + (long long)(t - g * s.BH) * sched_steps_ct(s, sched_long_row(s, g));
}

FA_HD long long sched_total_units(const Schedule &s)
{
    return sched_prefix(s, s.T - 1) + sched_steps(s, s.T - 1);
}

// Fill the table of CTA range starts (host side; keeps 64-bit divisions out of
// the kernel): the units split evenly over the first gt CTAs (all G when gt
// is 0); the others' ranges are empty.  Requires G <= kSchedMaxGrid and
// U <= kSchedMaxUnits.
inline void sched_fill_ranges(Schedule &s, int gt = 0)
{
    if (gt <= 0 || gt > s.G)
        gt = s.G;
    for (int c = 0; c <= s.G; ++c)
        s.range[c] = (int)(((unsigned long long)s.U * (unsigned long long)(c < gt ? c : gt)) / (unsigned long long)gt);
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
    if (!s.causal) {   // (tail split: the tail's tiles follow the WG whole ones)
        const int t = u / s.nkv;
        tstart = t * s.nkv;
        return t + s.W * s.G;
    }
    // (balanced schedules only) pairs of tile rows, then the middle row of an odd C
    int acc = 0;
    for (int q = 0; q < s.C / 2; ++q) {
        const int lg = sched_steps_ct(s, sched_long_row(s, q)), sh = sched_steps_ct(s, sched_short_row(s, q));
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
    int wt, we;          // balanced: the whole tiles wt .. we - 1 still to come after the range (tail split)

    // The kernel knows its schedule at compile time (SPLIT = s.split) and
    // takes only that path; init / next decide at run time (host code).
    template <bool SPLIT>
    FA_HD void init_t(const Schedule &s, int c_)
    {
        c = c_;
        lt = -1;
        lke = 0;
        lts = 0;
        wt = we = 0;
        if (SPLIT) {
            wt = c * s.W;
            we = wt + s.W;
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

    template <bool SPLIT, bool BAND = true>
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
            if (u >= ue) {
                if (wt >= we)
                    return false;
                p.tile = wt;   // a whole tile of a tail split
                p.kb = 0;
                p.ke = sched_steps(s, wt);
                p.slot = -1;
                p.ts = 0;
                ++wt;
                return true;
            }
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
        p.ke = sched_steps_rr_t<BAND>(s, t);
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

// Work decomposition for one call on `sms` SMs (host side).  Without a mask
// and with more tiles than SMs, the tail split is taken when the round-robin
// schedule of whole tiles would leave the machine idle in its last wave for
// more than ~4% of the run and for at least kSchedMinGain steps (a split tile
// costs its parts a partial write and one of them a merge), and only where
// those fixed costs are amortised: every CTA runs at least two whole tiles,
// or the tiles are at least kSchedTailSteps long.  (Measured: B4 H16 N2048,
// B2 H16 N4096 and B1 H8 N8192 at D = 64 gain 2, 1.4 and 10 %; B2 H8 N3000,
// one whole tile of 24 steps per CTA, loses 10-15 %.)  The tail is spread
// over few enough CTAs that no tile is cut into more than sched_max_parts
// parts.  Causal attention keeps whole tiles: its short tiles lose to the
// parts' fixed costs (measured).
// With few long tiles -- decoding a few queries against many keys -- whole
// tiles would leave most SMs idle, and the balanced schedule (split-KV) is
// taken whenever it at least halves the makespan; for heads of at most 64
// query rows, whose merges are cheap, whenever it saves more than 10 %.
constexpr int kSchedMinGain = 4;
constexpr int kSchedTailSteps = 64;

// mode: 0 = as above, 1 = round-robin, 2 = balanced wherever it can be built.
// N query rows against Nkv keys per head; `causal` here means masked by the
// band [i + off - wl, i + off + wr] (causal proper: wl unbounded, wr = 0).
inline Schedule sched_plan(int N, int Nkv, int BH, bool causal, int sms, int mode = 0, int wl = kSchedUnbounded,
                           int wr = 0)
{
    Schedule s{};
    s.N = N;
    s.Nkv = Nkv;
    s.off = causal ? Nkv - N : 0;
    if (!causal) {
        wl = kSchedUnbounded;
        wr = kSchedUnbounded;
    }
    sched_band_normalize(N, Nkv, wl, wr);
    s.wl = wl;
    s.wr = wr;
    {
        const long long lo_off = (long long)s.off - wl, hi_off = (long long)s.off + wr;
        const long long ka = (lo_off >= 0) ? lo_off / kSchedBN : -((-lo_off + kSchedBN - 1) / kSchedBN);
        const long long kb = (hi_off >= 0) ? hi_off / kSchedBN : -((-hi_off + kSchedBN - 1) / kSchedBN);
        s.ka = (wl >= kSchedUnbounded) ? -(1 << 29) : (int)ka;
        s.ra = (wl >= kSchedUnbounded) ? 0 : (int)(lo_off - ka * kSchedBN);
        s.kb = (wr >= kSchedUnbounded) ? (1 << 29) : (int)kb;
        s.rb = (wr >= kSchedUnbounded) ? 0 : (int)(hi_off - kb * kSchedBN);
    }
    s.BH = BH;
    s.C = (N + kSchedCtaRows - 1) / kSchedCtaRows;
    s.T = BH * s.C;
    s.nkv = (Nkv + kSchedBN - 1) / kSchedBN;
    s.causal = causal ? 1 : 0;
    s.rev = 0;
    s.split = 0;
    // the longest tile row: an end row for causal masks and one-sided bands,
    // any unclipped row for two-sided ones -- found by looking at every row
    int max_steps = 0;
    if (causal) {
        s.rev = sched_steps_ct(s, 0) > sched_steps_ct(s, s.C - 1) ? 1 : 0;
        for (int ct = 0; ct < s.C; ++ct) {
            const int n = sched_steps_ct(s, ct);
            max_steps = n > max_steps ? n : max_steps;
        }
    } else {
        max_steps = s.nkv;
    }
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
    long long G = (s.U < sms) ? s.U : sms;
    if (G > kSchedMaxGrid)
        G = kSchedMaxGrid;
    // Ranges of at least `need` units cut a tile of max_steps steps into at
    // most (max_steps - 1) / need + 2 <= sched_max_parts parts.
    const int mp = sched_max_parts(s);
    const long long need = (max_steps - 1 + mp - 3) / (mp - 2);
    if (need > 0 && s.U / G < need)
        G = s.U / need;
    if (G < 1)
        return s;
    const long long balanced = (s.U + G - 1) / G;
    if (mode == 0 && !causal && s.T > s.G) {   // the tail split, or whole tiles
        const int W = s.T / s.G, L = s.T - W * s.G;
        if (L == 0 || (W < 2 && s.nkv < kSchedTailSteps))
            return s;
        const long long ut = (long long)L * s.nkv;
        long long gt = s.G;
        if (need > 0 && ut / gt < need)
            gt = ut / need;
        if (gt < 1)
            return s;
        const long long tail = (long long)W * s.nkv + (ut + gt - 1) / gt;
        if (!(rr * 100 > tail * 104 && rr - tail >= kSchedMinGain))
            return s;
        s.split = 1;
        s.W = W;
        s.U = ut;
        sched_fill_ranges(s, (int)gt);
        return s;
    }
    const bool few_long_tiles = 2LL * s.T <= sms && max_steps >= 32 && rr >= 2 * balanced;
    // decoding-sized heads (at most 64 query rows) merge cheaply: balance
    // whenever it shortens the makespan by more than 10 %
    const bool short_heads = N <= kSchedShortRows && rr * 100 > balanced * 110;
    const bool pays = few_long_tiles || short_heads;
    if (mode == 2 || pays) {
        s.split = 1;
        s.G = (int)G;
        s.U = sched_total_units(s);   // the same total in the balanced order
        sched_fill_ranges(s);
    }
    return s;
}

// Workspace bytes of a balanced schedule at head size D: a partial O
// ([256 rows][D] fp32) and (m, l) per row for two slots per CTA, then two
// int counters per CTA tile (one per Q tile).  Whole tiles need none.
inline unsigned long long sched_workspace_bytes(const Schedule &s, int D)
{
    if (!s.split)
        return 0ull;
    const unsigned long long slots = 2ull * (unsigned long long)s.G;
    return slots * 256ull * (unsigned long long)D * 4ull + slots * 256ull * 8ull + 2ull * (unsigned long long)s.T * 4ull;
}

// The plan of a call that may not allocate (a fixed workspace of `limit`
// bytes): the planner's choice for `mode`, except that an automatic choice
// of the balanced schedule whose workspace exceeds the limit falls back to
// whole tiles, which need none.  An explicit request is kept as it is (the
// caller reports the limit).
inline Schedule sched_plan_limited(int N, int Nkv, int BH, bool causal, int sms, int mode, int wl, int wr, int D,
                                   unsigned long long limit)
{
    Schedule s = sched_plan(N, Nkv, BH, causal, sms, mode, wl, wr);
    if (mode == 0 && s.split && sched_workspace_bytes(s, D) > limit)
        s = sched_plan(N, Nkv, BH, causal, sms, 1, wl, wr);
    return s;
}

}  // namespace fa
