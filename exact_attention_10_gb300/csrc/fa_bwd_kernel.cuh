// fa_bwd_kernel.cuh -- FlashAttention-2 backward for GB300 (sm_103a).
//
// What it computes, for an upstream gradient dO and the forward's O and LSE
// (per batch*head slice; P recomputed from the saved LSE, never stored):
//   P[i,j]  = exp(s q_i.k_j - LSE_i)    (0 where the causal mask hides j > i)
//   delta_i = sum_d dO[i,d] O[i,d]
//   dS[i,j] = P[i,j] (dO_i.v_j - delta_i)
//   dV_j = sum_i P[i,j] dO_i,   dK_j = s sum_i dS[i,j] q_i,   dQ_i = s sum_j dS[i,j] k_j
// ("FlashAttention 2 from PyTorch to Triton", What I am building: the
// backward recovers P as exp(S - L) from the saved L; its limitations list:
// a precomputed D = rowsum(dO o O), dK and dV built per key tile by iterating
// over query tiles, dQ accumulated by atomics or in a second pass.)
//
// Three kernels, in stream order:
//   fa_bwd_prep   per query row: delta = rowsum(dO o O) and lg = LSE * log2(e),
//                 stored negated (as the passes add them), laid out [B*H][N
//                 rounded up to 128], with lg = +inf on the padding rows (and
//                 rows that see no key) so their P is 0;
//   fa_bwd_sm103<..., KV = true>   dK, dV: a CTA holds one 128-key tile of K
//                 and V and streams the query tiles (Q, dO, lg, delta) past it;
//   fa_bwd_sm103<..., KV = false>  dQ: a CTA holds one 128-row tile of Q and
//                 dO and streams the key tiles (K, V) past it -- the second
//                 pass, which keeps dQ deterministic and out of atomics.
// Both main passes recompute S and dP; that costs two extra tile products
// per (query tile, key tile) pair over a single pass with atomic dQ.
//
// At D = 64 the default is that single pass instead (FQ, "fused"): the dK/dV
// pass also computes each step's dQ product dS K (dS^T goes to shared memory
// so that it can serve as the MMA's A operand for both dK and dQ), and four
// more warps read the product out of TMEM and add it into an fp32 dQ
// accumulator [B*H][Npad][D] in global memory with tensor reductions (fp32
// adds in L2); fa_bwd_prep zeroes the accumulator first and
// fa_bwd_dq_convert scales and rounds it into dQ last.  The order of the adds
// varies between calls, so dQ may differ in its last bits from call to call.
//
// Per (resident tile, streamed tile) step, with M = 128 lanes of TMEM on the
// resident tile's rows:
//   KV:  S^T = K Q^T,  dP^T = V dO^T  (tcgen05, both operands K-major in smem)
//        compute warps: P^T = exp2(S^T * s log2 e - lg), dS^T = P^T (dP^T - delta)
//        dV += P^T dO,  dK += dS^T Q  (P^T, dS^T from TMEM; dO, Q MN-major)
//   dQ:  S = Q K^T,  dP = dO V^T;  P = exp2(S * s log2 e - lg), dS = P (dP - delta)
//        dQ += dS K  (dS from TMEM, K MN-major)
// The scale s is applied to dK and dQ when they are written out.
//
// Warp roles (384 threads): warpgroups 0 and 1 compute (warpgroup h takes
// columns [64h, 64h + 64) of S and dP for all 128 lanes) and write the
// accumulators out at the end of a tile; warp 8 is the TMA producer; warp 9
// issues the MMAs and owns TMEM.  The fused pass has 512: warp 10 issues the
// dQ products and warps 12-15 read them out (warp 11 idles).
//
// Tensor memory (512 columns): S or S^T [0,128), dP or dP^T [128,256), then
// the accumulators: dV [256, 256+D) and dK [256+D, 256+2D) (KV) or dQ
// [256, 256+D).  The dK/dV pass at D = 128 has no columns left: P and dS are
// written as 16-bit pairs over the scores they came from (warpgroup h's 64
// columns become 32 columns at 64h within the same region, so neither
// warpgroup overwrites scores the other still has to read), and MMAs from one
// thread run in issue order, so the next step's S follows the dV product
// that reads P^T and its dP the dK product that reads dS^T (bwd_mma).
// Pipelined passes keep P^T and dS^T (or dS) in buffers of
// their own after the accumulators (kColP, kColDS), and the fused pass puts
// its dQ product where dS^T would be (kColDQ), dS^T going to shared memory.
//
// Every mbarrier wait is bounded as in the forward kernel; on expiry the
// kernel records the site in the status word, leaves its loops, waits (with a
// time bound) for its copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "fa_fwd_kernel.cuh"

namespace fa {
namespace bwd {

constexpr int kThreads = 384;
constexpr int kComputeThreads = 256;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTile = 128;   // rows of a resident or streamed tile (keys or queries)
// Registers per thread after setmaxnreg: 2 x 128 x 200 + 128 x 96 = 63488, within
// the 384 x 168 = 64512 the block is launched with.
constexpr uint32_t kRegsCompute = 200;
constexpr uint32_t kRegsProducer = 96;
// The fused pass (dK, dV and dQ in one pass, D = 64): 512 threads.  Warp 10
// issues the dQ products, warps 12-15 read them out of TMEM and add them into
// an fp32 dQ accumulator in global memory.  2 x 128 x 192 + 2 x 128 x 64 =
// 65536 registers, the 512 x 128 the block is launched with.
constexpr int kThreadsFused = 512;
constexpr int kMmaWarpDq = 10;
constexpr int kDqWarp0 = 12;
constexpr uint32_t kRegsComputeFused = 192;
constexpr uint32_t kRegsOtherFused = 64;

// Wait sites (status word), after the forward's.
enum : uint32_t {
    kSiteBwdResEmpty = 32, kSiteBwdSlotEmpty, kSiteBwdResFull, kSiteBwdSlotFull, kSiteBwdPFull, kSiteBwdAccFree,
    kSiteBwdSdFull, kSiteBwdAccFull, kSiteBwdDrain, kSiteBwdTail, kSiteBwdSdFree, kSiteBwdPdFree, kSiteBwdDqFull,
    kSiteBwdDqFree
};

struct Params {
    void *dA;          // KV: dK ([B*H, Nkv, D]); dQ pass: dQ ([B*H, N, D]); the input type
    void *dB;          // KV: dV; dQ pass: unused
    const float *lg;   // -LSE * log2(e) per query row, [B*H][Npad]; -inf on padding rows and rows without keys
    const float *dl;   // -delta = -rowsum(dO o O) per query row, [B*H][Npad]
    int N;             // query rows per head
    int Nkv;           // keys per head
    int Npad;          // N rounded up to a multiple of 128
    int BH;
    int nqt;           // 128-row query tiles per head (Npad / 128)
    int nkt;           // 128-key tiles per head
    int T;             // work tiles of the pass: BH * nkt (KV) or BH * nqt (dQ pass)
    int off;           // masked: query i sits at key position i + off (off = Nkv - N, bottom-right)
    int wl, wr;        // masked: query i sees keys [i + off - wl, i + off + wr] (kSchedUnbounded: no bound)
    int square_causal; // masked, N = Nkv, (unbounded, 0): tile rows go longest first
    float qk2;         // scale * log2(e)
    float scale;
};

// FQ: the fused pass (KV, D = 64 only): dQ products beside dK and dV.
template <int D, bool KV, bool FQ = false>
struct BCfg {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static_assert(!FQ || (KV && D == 64), "the fused pass is the dK/dV pass at D = 64");
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;     // [128 rows, 64 columns] of 16-bit
    static constexpr int kTileBytes = kTile * D * 2;
    static constexpr int kVecBytes = KV ? 2 * kTile * 4 : 0;   // lg and delta of the streamed query tile
    static constexpr int kStages = (D == 64) ? 3 : 2;
    static constexpr int kStageBytes = 2 * kTileBytes + kVecBytes;   // a multiple of 1024
    static constexpr int kResOff = 0;                                 // the resident pair of tiles
    static constexpr int kStageOff = 2 * kTileBytes;
    // The dQ pass at D = 128 streams K and V through separate rings, 3 slots
    // of K and 2 of V, instead of 2 stages of both: V is done with once dP is
    // computed, K only after the step's dQ product, and the third K slot lets
    // the next steps' tiles load while it runs.  (Both rings: 224 KB with the
    // resident Q and dO.)
    static constexpr bool kSplitRing = !KV && D == 128;
    static constexpr int kRing0 = kSplitRing ? 3 : kStages;   // slots of streamed tile 0 (KV: Q; dQ pass: K)
    static constexpr int kRing1 = kSplitRing ? 2 : kStages;   // slots of streamed tile 1 (KV: dO; dQ pass: V)
    static constexpr int kRing1Off = kStageOff + kRing0 * kTileBytes;   // split rings: tile 1's ring
    // The fused pass: dS^T as an MMA operand, 16-bit [128 keys][128 queries]
    // in two 64-column boxes (K-major for dK += dS^T Q, MN-major as dS for
    // dQ = dS K); then the fp32 dQ product of a step, [128 queries][64] in two
    // 32-column boxes, staged for the reduction into the accumulator.
    static constexpr int kDsOff = kStageOff + kStages * kStageBytes;
    static constexpr int kDqOff = kDsOff + (FQ ? kTile * kTile * 2 : 0);
    static constexpr int kDqBoxBytes = kTile * 128;   // [128 rows, 32 fp32 columns]
    static constexpr int kBarOff = kSplitRing ? kRing1Off + kRing1 * kTileBytes : kDqOff + (FQ ? kTile * D * 4 : 0);
    // full/empty per slot (unified stages, or ring 0 then ring 1), then res_full, res_empty,
    // sd_full, p_full, acc_full, acc_free, drain, sd_free, pd_free, p_full_odd (dQ pass) or dp_full
    // (the dK/dV pass at D = 128); fused: dq_full, dq_free
    static constexpr int kRingBars = kSplitRing ? 2 * (kRing0 + kRing1) : 2 * kStages;
    static constexpr int kNumBars = kRingBars + 10 + (FQ ? 2 : 0);
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;           // TMEM address, abort flag
    static constexpr int kSmem = kMiscOff + 16 + 1024;                // + slack to align the base to 1024
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(kStageBytes % 1024 == 0, "stages keep the tiles' 1024-byte swizzle alignment");
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
    // Pipelined passes: dQ pass: two 64-column dS buffers after dQ (dS of step g
    // in buffer g % 2); KV pass (D = 64): one P^T and one dS^T buffer after dV, dK.
    static constexpr uint32_t kColDS = KV ? 256 + 2 * D + 64 : 256 + D;
    static constexpr uint32_t kColP = 256 + 2 * D;
    static constexpr uint32_t kColDQ = 256 + 2 * D + 64;   // fused: the step's dQ product, where dS^T sits otherwise
    static_assert((KV && D == 128) || (KV ? kColDS + 64 : kColDS + 128) <= kTmemCols, "pipelined buffers fit TMEM");
    // Shared-memory address of streamed tile 0 / 1 of global step g.
    __device__ static uint32_t slot0(uint32_t sStage, int g)
    {
        return kSplitRing ? sStage + (uint32_t)((g % kRing0) * kTileBytes) : sStage + (uint32_t)((g % kStages) * kStageBytes);
    }
    __device__ static uint32_t slot1(uint32_t sStage, int g)
    {
        return kSplitRing ? sStage + (uint32_t)(kRing1Off - kStageOff + (g % kRing1) * kTileBytes)
                          : slot0(sStage, g) + (uint32_t)kTileBytes;
    }
};

template <int D, bool KV, bool FQ = false>
struct BBars {
    uint32_t base;
    using C = BCfg<D, KV, FQ>;
    __device__ uint32_t full(int s) const { return base + 8u * s; }                    // slot s of ring 0 / stage s
    __device__ uint32_t empty(int s) const { return base + 8u * (C::kRing0 + s); }
    __device__ uint32_t full1(int s) const { return C::kSplitRing ? base + 8u * (2 * C::kRing0 + s) : full(s); }
    __device__ uint32_t empty1(int s) const
    {
        return C::kSplitRing ? base + 8u * (2 * C::kRing0 + C::kRing1 + s) : empty(s);
    }
    __device__ uint32_t at(int k) const { return base + 8u * (C::kRingBars + k); }
    __device__ uint32_t res_full() const { return at(0); }    // TMA -> MMA: resident tiles landed
    __device__ uint32_t res_empty() const { return at(1); }   // MMA -> TMA: the tile's last MMAs done
    __device__ uint32_t sd_full() const { return at(2); }     // MMA -> compute: S and dP of a step ready
    __device__ uint32_t p_full() const { return at(3); }      // compute -> MMA: P / dS written
    __device__ uint32_t acc_full() const { return at(4); }    // MMA -> compute: a tile's accumulators final
    __device__ uint32_t acc_free() const { return at(5); }    // compute -> MMA: accumulators read out
    __device__ uint32_t drain() const { return at(6); }
    __device__ uint32_t sd_free() const { return at(7); }     // compute -> MMA: S and dP loaded (pipelined)
    __device__ uint32_t pd_free() const { return at(8); }     // MMA -> compute: P / dS buffers read (pipelined KV)
    // p_full of step g in the pipelined dQ pass, which alternates two barriers:
    // there the compute warps may finish step g + 1 before the MMA warp has
    // waited for step g (nothing else holds them back), and one barrier two
    // phases ahead of its waiter would read as not yet complete.
    __device__ uint32_t p_full_dq(int g) const { return (g & 1) ? at(9) : at(3); }
    // The serialized dK/dV pass (D = 128) uses the same slot for dP's
    // completion (MMA -> compute; S's is sd_full).
    __device__ uint32_t dp_full() const { return at(9); }
    __device__ uint32_t dq_full() const { return at(10); }    // fused: dQ MMA -> read-out warps: the step's dQ product done
    __device__ uint32_t dq_free() const { return at(11); }    // fused: read-out warps -> dQ MMA: dQ product loaded
};

// Streamed tiles of resident tile rt under a band mask, [s0, s0 + n): the
// dK/dV pass's key tile sees the query tiles whose rows' bands reach one of
// its keys, the dQ pass's query tile the key tiles its rows' bands reach.
// An empty range still takes one (fully masked) step, so the tile's
// gradients are written as zeros.
template <bool KV>
__device__ __forceinline__ void bwd_band_range(const Params &p, int rt, int &s0, int &n)
{
    const long long big = 1ll << 40;
    const long long wl = p.wl >= kSchedUnbounded ? big : p.wl, wr = p.wr >= kSchedUnbounded ? big : p.wr;
    const int ns = KV ? p.nqt : p.nkt, lim = KV ? p.N : p.Nkv;
    long long lo, hi;
    if (KV) {   // keys k0 .. k1; queries i with i + off - wl <= k1 and i + off + wr >= k0
        const long long k0 = (long long)rt * kTile, k1 = min((long long)rt * kTile + kTile - 1, (long long)p.Nkv - 1);
        lo = k0 - p.off - wr;
        hi = k1 - p.off + wl;
    } else {    // rows r0 .. r1 see keys r0 + off - wl .. r1 + off + wr
        const long long r0 = (long long)rt * kTile, r1 = min((long long)rt * kTile + kTile - 1, (long long)p.N - 1);
        lo = r0 + p.off - wl;
        hi = r1 + p.off + wr;
    }
    lo = lo < 0 ? 0 : lo;
    hi = hi > lim - 1 ? lim - 1 : hi;
    if (lo > hi) {   // no row of the tile pair can see the other
        s0 = (int)min(lo / kTile, (long long)ns - 1);
        n = 1;
    } else {
        s0 = (int)(lo / kTile);
        n = (int)(hi / kTile) + 1 - s0;
    }
}

// Work tile t -> (head, resident tile index), and the streamed tiles it
// visits, [s0, s0 + n).  Square causal: the dK/dV pass's key tile kt sees
// query tiles kt .. nqt-1, the dQ pass's query tile qt sees key tiles 0 .. qt;
// tiles go longest first, heads interleaved.  Otherwise head-major, with the
// band's range when masked.
template <bool KV>
__device__ __forceinline__ void bwd_decode(const Params &p, bool causal, int t, int &bh, int &rt, int &s0, int &n)
{
    if (causal && p.square_causal) {
        const int g = t / p.BH;
        bh = t - g * p.BH;
        rt = KV ? g : p.nqt - 1 - g;
        s0 = KV ? rt : 0;
        n = KV ? p.nqt - rt : rt + 1;
        return;
    }
    const int nres = KV ? p.nkt : p.nqt;
    bh = t / nres;
    rt = t - bh * nres;
    if (causal) {
        bwd_band_range<KV>(p, rt, s0, n);
    } else {
        s0 = 0;
        n = KV ? p.nqt : p.nkt;
    }
}

// The band mask of one step, in terms of d = key - query: with (kt, qt) the
// step's key and query tiles, d = 128 (kt - qt) + x where x = lane - column
// (KV) or column - lane (dQ pass), and key j is visible from query i iff
// e_lo <= x <= e_hi.  `whole` when every x in [-127, 127] is visible.
struct StepMask {
    int e_lo, e_hi;
    bool whole;
};

// This thread's test for the step's mask, one unsigned compare per score:
// column `col` is visible iff (uint)(a + sgn * col) < width, folding the band
// (e_lo <= x <= e_hi with x = key - query = sgn * (col - row) ... ) and, in
// the dQ pass, the keys past Nkv (col < limit) into `a` and `width`.
struct LaneMask {
    int a;
    uint32_t width;
};

template <bool KV>
__device__ __forceinline__ LaneMask bwd_lane_mask(const StepMask &m, int row, int limit)
{
    // KV: x = row - col, visible iff e_lo <= row - col <= e_hi, i.e. col in
    //     [row - e_hi, row - e_lo]; dQ pass: x = col - row, col in
    //     [row + e_lo, row + e_hi] and col < limit.
    int lo = KV ? row - m.e_hi : row + m.e_lo;
    int hi = KV ? row - m.e_lo : row + m.e_hi;
    if (!KV && hi > limit - 1)
        hi = limit - 1;
    if (lo < 0)
        lo = 0;
    return LaneMask{-lo, hi >= lo ? (uint32_t)(hi - lo + 1) : 0u};
}

__device__ __forceinline__ StepMask bwd_step_mask(const Params &p, bool causal, int kt, int qt)
{
    StepMask m{-1024, 1024, true};
    if (!causal)
        return m;
    const long long base = (long long)kTile * (kt - qt);
    if (p.wl < kSchedUnbounded)
        m.e_lo = (int)max(-1024ll, min(1024ll, (long long)p.off - p.wl - base));
    if (p.wr < kSchedUnbounded)
        m.e_hi = (int)max(-1024ll, min(1024ll, (long long)p.off + p.wr - base));
    m.whole = m.e_lo <= -(kTile - 1) && m.e_hi >= kTile - 1;
    return m;
}

// Work tiles of CTA c on a grid of G: serpentine rounds (c-th tile of even
// rounds, (G-1-c)-th of odd rounds), as in the forward's whole-tile schedule.
__device__ __forceinline__ int bwd_tile(int r, int c, int G)
{
    return r * G + ((r & 1) ? G - 1 - c : c);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// TMEM column of the 16-bit A operand's k-block kk (16 rows of the streamed
// tile): warpgroup kk / 4 wrote it, 8 columns per block within its 64.
__device__ __forceinline__ uint32_t a_col(int kk)
{
    return (uint32_t)(64 * (kk / 4) + 8 * (kk % 4));
}

// PTX of the fused pass (bulk tensor reductions, 16-byte shared stores) and
// of the backward's programmatic dependent launch.
namespace fq {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 2-D tiled tensor reduction shared -> global: adds the box at `src` to the
// tensor at (c0, c1) element by element (fp32 add for an fp32 map), as one
// bulk async-group operation; c0 * 4 bytes must be a multiple of 16.
__device__ __forceinline__ void tma_reduce_add_2d(const void *tmap, uint32_t src, int c0, int c1)
{
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}

// Programmatic dependent launch: let the next kernel on the stream start
// launching (its blocks still wait for this grid with grid_wait before they
// read what it wrote); and wait until the previous kernel on the stream has
// completed and its writes are visible (a no-op when this launch did not
// allow programmatic serialization).
__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void grid_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Close this thread's bulk async-group operations issued so far into a group.
__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group of this thread has finished reading
// its shared-memory source (the source may then be overwritten).
__device__ __forceinline__ void bulk_wait_group_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace fq

// Waits for the given phases of up to three barriers (`use` false: skipped),
// all of them by every lane.  A check on a barrier takes ~150 cycles even when
// the phase completed long before; the three are issued back to back so that
// their latencies overlap, and the bounded waits (warp-collective, so entered
// on warp-uniform votes) follow for the ones not yet complete.
__device__ __forceinline__ bool warp_wait_all(uint32_t b0, uint32_t p0, bool u0, uint32_t b1, uint32_t p1, bool u1,
                                              uint32_t b2, uint32_t p2, bool u2, Ctl c, uint32_t site)
{
    const bool d0 = !u0 || ptx::mbar_try_wait(b0, p0);
    const bool d1 = !u1 || ptx::mbar_try_wait(b1, p1);
    const bool d2 = !u2 || ptx::mbar_try_wait(b2, p2);
    const bool a0 = __all_sync(0xffffffffu, d0), a1 = __all_sync(0xffffffffu, d1), a2 = __all_sync(0xffffffffu, d2);
    return (a0 || warp_wait(b0, p0, c, site)) && (a1 || warp_wait(b1, p1, c, site)) && (a2 || warp_wait(b2, p2, c, site));
}

// ------------------------------------------------------------------ producer

template <int D, bool KV, bool FQ>
__device__ void bwd_load(const CUtensorMap *tmR0, const CUtensorMap *tmR1, const CUtensorMap *tmS0,
                         const CUtensorMap *tmS1, const Params &p, bool causal, uint32_t sRes, uint32_t sStage,
                         BBars<D, KV, FQ> b, Ctl c)
{
    using C = BCfg<D, KV, FQ>;
    int step = 0, tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<KV>(p, causal, t, bh, rt, s0, n);
        if (tiles > 0 && !warp_wait(b.res_empty(), (uint32_t)(tiles - 1) & 1u, c, kSiteBwdResEmpty))
            break;
        if (ptx::elect_one()) {
            ptx::mbar_arrive_expect_tx(b.res_full(), 2 * C::kTileBytes);
            for (int x = 0; x < C::kBoxes; ++x) {
                ptx::tma_load_3d(sRes + x * C::kBoxBytes, tmR0, b.res_full(), x * 64, rt * kTile, bh);
                ptx::tma_load_3d(sRes + C::kTileBytes + x * C::kBoxBytes, tmR1, b.res_full(), x * 64, rt * kTile, bh);
            }
        }
        __syncwarp();
        ++tiles;
        for (int j = 0; j < n; ++j, ++step) {
            const int row = (s0 + j) * kTile;
            if (C::kSplitRing) {   // K into ring 0, V into ring 1, each on its own barriers
                const int k0 = step % C::kRing0, k1 = step % C::kRing1;
                if (!warp_wait(b.empty(k0), ((uint32_t)(step / C::kRing0) & 1u) ^ 1u, c, kSiteBwdSlotEmpty) ||
                    !warp_wait(b.empty1(k1), ((uint32_t)(step / C::kRing1) & 1u) ^ 1u, c, kSiteBwdSlotEmpty)) {
                    ok = false;
                    break;
                }
                if (ptx::elect_one()) {
                    const uint32_t d0 = C::slot0(sStage, step), d1 = C::slot1(sStage, step);
                    ptx::mbar_arrive_expect_tx(b.full(k0), C::kTileBytes);
                    ptx::mbar_arrive_expect_tx(b.full1(k1), C::kTileBytes);
                    for (int x = 0; x < C::kBoxes; ++x) {
                        ptx::tma_load_3d(d0 + x * C::kBoxBytes, tmS0, b.full(k0), x * 64, row, bh);
                        ptx::tma_load_3d(d1 + x * C::kBoxBytes, tmS1, b.full1(k1), x * 64, row, bh);
                    }
                }
                __syncwarp();
                continue;
            }
            const int st = step % C::kStages;
            const uint32_t use = (uint32_t)(step / C::kStages);
            if (!warp_wait(b.empty(st), (use & 1u) ^ 1u, c, kSiteBwdSlotEmpty)) {
                ok = false;
                break;
            }
            if (ptx::elect_one()) {
                const uint32_t dst = sStage + st * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(b.full(st), C::kStageBytes);
                for (int x = 0; x < C::kBoxes; ++x) {
                    ptx::tma_load_3d(dst + x * C::kBoxBytes, tmS0, b.full(st), x * 64, row, bh);
                    ptx::tma_load_3d(dst + C::kTileBytes + x * C::kBoxBytes, tmS1, b.full(st), x * 64, row, bh);
                }
                if (KV) {   // the query tile's lg and delta: 512 bytes each, 16-byte aligned (Npad % 128 == 0)
                    const size_t off = (size_t)bh * p.Npad + row;
                    ptx::bulk_load(dst + 2 * C::kTileBytes, p.lg + off, kTile * 4, b.full(st));
                    ptx::bulk_load(dst + 2 * C::kTileBytes + kTile * 4, p.dl + off, kTile * 4, b.full(st));
                }
            }
            __syncwarp();
        }
    }
    // Tail: every copy issued has landed (time-bounded), so no asynchronous
    // write targets this CTA's shared memory after exit.
    for (int s = 0; s < C::kRing0 && s < step; ++s) {
        const int last = step - 1 - ((step - 1 - s) % C::kRing0);
        wait_landed(b.full(s), (uint32_t)(last / C::kRing0) & 1u, c, kSiteBwdTail);
    }
    for (int s = 0; C::kSplitRing && s < C::kRing1 && s < step; ++s) {
        const int last = step - 1 - ((step - 1 - s) % C::kRing1);
        wait_landed(b.full1(s), (uint32_t)(last / C::kRing1) & 1u, c, kSiteBwdTail);
    }
    if (tiles > 0)
        wait_landed(b.res_full(), (uint32_t)(tiles - 1) & 1u, c, kSiteBwdTail);
}

// ------------------------------------------------------------------ MMA issuer

// The serialized pass (the dK/dV pass at D = 128, where TMEM holds S, dP, dV
// and dK and nothing else): P^T and dS^T are written over S and dP (16-bit
// pairs, see the header), so a step's S and dP can only be computed once the
// previous step's products have read them.  Per step g the MMA warp issues
// dV_g (reads P^T_g), S_{g+1} (overwrites it), dK_g (reads dS^T_g) and
// dP_{g+1} (overwrites it): MMAs from one thread run in issue order, so each
// overwrite follows the read it displaces.  S and dP complete separate
// barriers (sd_full, dp_full), so the compute warps start on S_{g+1} while
// dK_g and dP_{g+1} still run.
template <int D, bool BF16, bool KV>
__device__ void bwd_mma(const Params &p, bool causal, uint32_t sRes, uint32_t sStage, uint32_t tmem,
                        BBars<D, KV> b, Ctl c)
{
    static_assert(KV, "the serialized pass is the dK/dV pass");
    using C = BCfg<D, KV>;
    constexpr uint32_t kIdescSS = instr_desc_f16(BF16, kTile, kTile, false);   // both operands K-major
    constexpr uint32_t kIdescTS = instr_desc_f16(BF16, kTile, D, true);        // B MN-major
    const uint32_t r0_lo = desc_lo(sRes, 16), r1_lo = desc_lo(sRes + C::kTileBytes, 16);
    const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP;
    const uint32_t tAcc0 = tmem + C::kColAcc0, tAcc1 = tmem + C::kColAcc1;
    int g = 0, tiles = 0;
    bool ok = true;

    auto stage_ready = [&](int gs) -> bool {
        if (!warp_wait(b.full(gs % C::kStages), (uint32_t)(gs / C::kStages) & 1u, c, kSiteBwdSlotFull))
            return false;
        ptx::tc_fence_after_sync();
        return true;
    };
    // S^T = K Q^T (or dP^T = V dO^T) of step gs into `col`, then `bar`: K-major
    // operands advance 32 bytes per k-step inside a 128-byte swizzle row and
    // one box (16 KB) per 64 columns.
    auto issue_sd = [&](int gs, uint32_t r_lo, uint32_t s_off, uint32_t col, uint32_t bar) {
        const uint32_t s_lo = desc_lo(sStage + (uint32_t)((gs % C::kStages) * C::kStageBytes) + s_off, 16);
        if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk / 4) * (C::kBoxBytes >> 4) + (kk % 4) * 2);
                ptx::mma_ss(col, desc_from_lo(r_lo + off), desc_from_lo(s_lo + off), kIdescSS, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(bar);
        }
        __syncwarp();
    };

    for (int r = 0; ok; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<KV>(p, causal, t, bh, rt, s0, n);
        if (!warp_wait(b.res_full(), (uint32_t)tiles & 1u, c, kSiteBwdResFull))
            break;
        ptx::tc_fence_after_sync();
        if (!stage_ready(g))
            break;
        issue_sd(g, r0_lo, 0u, tS, b.sd_full());
        issue_sd(g, r1_lo, (uint32_t)C::kTileBytes, tDP, b.dp_full());
        for (int j = 0; j < n; ++j, ++g) {
            if (j == 0 && tiles > 0 &&   // the accumulators are overwritten: the previous tile's were read
                !warp_wait(b.acc_free(), (uint32_t)(tiles - 1) & 1u, c, kSiteBwdAccFree)) {
                ok = false;
                break;
            }
            if (!warp_wait(b.p_full(), (uint32_t)g & 1u, c, kSiteBwdPFull)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            // dV += P^T dO, dK += dS^T Q: the 16-bit A operand from TMEM, 8 columns
            // per 16 rows of the streamed tile; the B operand the streamed tile
            // read MN-major (16 rows = 2 KB per k-step, leading byte offset = the
            // box stride).
            const int st = g % C::kStages;
            const uint32_t sa = sStage + (uint32_t)(st * C::kStageBytes);
            const uint32_t m0_lo = desc_lo(sa + C::kTileBytes, C::kBoxBytes);   // dO
            const uint32_t m1_lo = desc_lo(sa, C::kBoxBytes);                   // Q
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    ptx::mma_ts(tAcc0, tS + a_col(kk), desc_from_lo(m0_lo + kk * (2048 >> 4)), kIdescTS,
                                (j > 0 || kk > 0) ? 1u : 0u);
            }
            __syncwarp();
            if (j + 1 < n) {   // S_{g+1} over P^T_g, behind dV_g
                if (!stage_ready(g + 1)) {
                    ok = false;
                    break;
                }
                issue_sd(g + 1, r0_lo, 0u, tS, b.sd_full());
            }
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    ptx::mma_ts(tAcc1, tDP + a_col(kk), desc_from_lo(m1_lo + kk * (2048 >> 4)), kIdescTS,
                                (j > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(b.empty(st));
                if (j == n - 1) {
                    ptx::mma_commit(b.acc_full());
                    ptx::mma_commit(b.res_empty());
                }
            }
            __syncwarp();
            if (j + 1 < n)   // dP_{g+1} over dS^T_g, behind dK_g
                issue_sd(g + 1, r1_lo, (uint32_t)C::kTileBytes, tDP, b.dp_full());
        }
        ++tiles;
    }
    // Drain: every MMA this warp issued has completed before TMEM is freed.
    if (ptx::elect_one())
        ptx::mma_commit(b.drain());
    __syncwarp();
    wait_landed(b.drain(), 0u, c, kSiteBwdDrain);
}

// ------------------------------------------------------------------ compute

// Write 32 fp32 columns of one accumulator row (times `mul`) as 16-bit values
// to global memory at `dst` (64 bytes, 16-byte aligned).
template <bool BF16>
__device__ __forceinline__ void store_row32(void *dst, const uint32_t (&v)[32], float mul)
{
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float a = __uint_as_float(v[2 * i]) * mul, bb = __uint_as_float(v[2 * i + 1]) * mul;
        pk[i] = BF16 ? ptx::pack_bf16x2(a, bb) : ptx::pack_f16x2(a, bb);
    }
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        ptx::st_global_v4(d4 + q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// The serialized pass's compute warps: per step, S (sd_full): P^T = exp2(S^T
// s log2 e - lg) over this warpgroup's 64 columns of S; then dP (dp_full):
// dS^T = P^T (dP^T - delta) over its 64 columns of dP.  Each is written as
// 32 columns of 16-bit pairs at the start of the columns it came from, once
// this thread has loaded them.
template <int D, bool BF16, bool CAUSAL, bool KV>
__device__ void bwd_compute(const Params &p, uint32_t tmem, uint32_t sStage, BBars<D, KV> b, Ctl c)
{
    static_assert(KV, "the serialized pass is the dK/dV pass");
    using C = BCfg<D, KV>;
    const int h = threadIdx.x / 128;                // column half of S and dP
    const int warp = threadIdx.x / 32;
    const int lane_row = (warp % 4) * 32 + threadIdx.x % 32;   // TMEM lane = row of the resident tile
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + C::kColS + lane_off + 64 * h, tDP = tmem + C::kColDP + lane_off + 64 * h;
    const uint64_t qk2 = ptx::f2_pack(p.qk2, p.qk2);
    int step = 0, tiles = 0;
    for (int r = 0;; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<KV>(p, CAUSAL, t, bh, rt, s0, n);
        for (int j = 0; j < n; ++j, ++step) {
            const int st = step % C::kStages;
            const int si = s0 + j;   // streamed (query) tile index
            if (!warp_wait(b.sd_full(), (uint32_t)step & 1u, c, kSiteBwdSdFull))
                return;
            ptx::tc_fence_after_sync();
            const uint32_t vec = sStage + st * C::kStageBytes + 2 * C::kTileBytes;   // lg[128], delta[128]
            // Masks: the band's edges (the causal diagonal); padding queries
            // and queries without keys have lg = +inf (stored as -lg = -inf),
            // so their P is already 0.
            const StepMask sm = bwd_step_mask(p, CAUSAL, rt, si);
            const bool masked = !sm.whole;   // warp-uniform
            uint32_t pv[64];   // S, then P (fp32)
            ptx::tmem_ld64(tS, pv);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
                const float4 lg4 = ptx::ld_shared_v4f32(vec + (uint32_t)(64 * h + i) * 4);   // -lg of four queries
                float x[4];
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(pv[i]), __uint_as_float(pv[i + 1])), qk2,
                                           ptx::f2_pack(lg4.x, lg4.y)),
                               x[0], x[1]);
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(pv[i + 2]), __uint_as_float(pv[i + 3])), qk2,
                                           ptx::f2_pack(lg4.z, lg4.w)),
                               x[2], x[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pv[i + e] = __float_as_uint(ptx::ex2(x[e]));
            }
            if (masked) {   // lane = key, column = query
                const LaneMask lm = bwd_lane_mask<KV>(sm, lane_row, kTile);
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    pv[i] = ((uint32_t)(lm.a + 64 * h + i) < lm.width) ? pv[i] : 0u;
            }
            {   // P^T over the first 32 of this warpgroup's S columns
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = BF16 ? ptx::pack_bf16x2(__uint_as_float(pv[2 * i]), __uint_as_float(pv[2 * i + 1]))
                                 : ptx::pack_f16x2(__uint_as_float(pv[2 * i]), __uint_as_float(pv[2 * i + 1]));
                ptx::tmem_st32(tS, pk);
            }
            if (!warp_wait(b.dp_full(), (uint32_t)step & 1u, c, kSiteBwdSdFull))
                return;
            ptx::tc_fence_after_sync();
            // dS^T over the first 32 of this warpgroup's dP columns, in two
            // halves of 32 dP columns each (all of this thread's dP columns are
            // loaded before any is overwritten).
            uint32_t dv[2][32];
            ptx::tmem_ld32(tDP, dv[0]);
            ptx::tmem_ld32(tDP + 32, dv[1]);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
                uint32_t dk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int q = 32 * ch + i;   // this warpgroup's column
                    const float4 d4 = ptx::ld_shared_v4f32(vec + kTile * 4 + (uint32_t)(64 * h + q) * 4);   // -delta
                    float ds[4];
                    ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(pv[q]), __uint_as_float(pv[q + 1])),
                                               ptx::f2_add(ptx::f2_pack(__uint_as_float(dv[ch][i]), __uint_as_float(dv[ch][i + 1])),
                                                           ptx::f2_pack(d4.x, d4.y))),
                                   ds[0], ds[1]);
                    ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(pv[q + 2]), __uint_as_float(pv[q + 3])),
                                               ptx::f2_add(ptx::f2_pack(__uint_as_float(dv[ch][i + 2]), __uint_as_float(dv[ch][i + 3])),
                                                           ptx::f2_pack(d4.z, d4.w))),
                                   ds[2], ds[3]);
                    dk[i / 2] = BF16 ? ptx::pack_bf16x2(ds[0], ds[1]) : ptx::pack_f16x2(ds[0], ds[1]);
                    dk[i / 2 + 1] = BF16 ? ptx::pack_bf16x2(ds[2], ds[3]) : ptx::pack_f16x2(ds[2], ds[3]);
                }
                tmem_st16(tDP + 16 * ch, dk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.p_full());
        }
        // The tile's accumulators, written out once: KV: warpgroup 0 writes dV,
        // warpgroup 1 dK (times the scale); dQ pass: warpgroup h writes
        // columns [h D/2, (h+1) D/2) of dQ (times the scale).
        if (!warp_wait(b.acc_full(), (uint32_t)tiles & 1u, c, kSiteBwdAccFull))
            return;
        ptx::tc_fence_after_sync();
        const int grow = rt * kTile + lane_row;   // row within the head
        if (KV) {
            const uint32_t tA = tmem + (h ? C::kColAcc1 : C::kColAcc0) + lane_off;
            char *dst = static_cast<char *>(h ? p.dA : p.dB) + ((size_t)bh * p.Nkv + grow) * D * 2;
            const float mul = h ? p.scale : 1.f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t v[32];
                ptx::tmem_ld32(tA + 32 * cc, v);
                ptx::tmem_wait_ld();
                if (grow < p.Nkv)
                    store_row32<BF16>(dst + cc * 64, v, mul);
            }
        } else {
            const uint32_t tA = tmem + C::kColAcc0 + lane_off;
            char *dst = static_cast<char *>(p.dA) + ((size_t)bh * p.N + grow) * D * 2;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int col = h * (D / 2) + 32 * cc;
                uint32_t v[32];
                ptx::tmem_ld32(tA + col, v);
                ptx::tmem_wait_ld();
                if (grow < p.N)
                    store_row32<BF16>(dst + col * 2, v, p.scale);
            }
        }
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(b.acc_free());
        ++tiles;
    }
}

// ------------------------------------------------------------------ dQ pass, pipelined

// Pipelined: D = 64, and the dQ pass at D = 128 (K and V in rings of their
// own).  The pipelined order wants S_{g+2} right after the products of step
// g, and stage g + 2 can only be loaded once they have released stage g; with
// the two stages of both tiles that fit beside the resident tiles at D = 128
// that load was exposed on every step (measured on the dQ pass: 892 -> 840
// TFLOP/s at N = 16384).  The dK/dV pass at D = 128 has no TMEM left for
// separate P^T / dS^T buffers and keeps them over S and dP (bwd_mma,
// bwd_compute).
template <int D, bool KV>
constexpr bool kPipeline = (D == 64) || (!KV && D == 128);

// The dQ pass overlaps the compute warps with the tensor core: as soon as the
// compute warps have loaded S_g and dP_g into registers (sd_free), the next
// step's S_{g+1} and dP_{g+1} are issued into the same columns, and dQ += dS_g K_g
// follows once dS_g is written (p_full).  dS alternates between two TMEM
// buffers; the compute warps write buffer g % 2 only after waiting for
// sd_full of step g, whose commit follows the MMA that read the buffer at
// step g - 2, so no extra barrier guards it.  Tensor-pipe order per step:
// S_{g+1}, dP_{g+1}, dQ_g.
//
// The fused pass (FQ) takes dS^T from shared memory for dK += dS^T Q (warp
// 10 reads the same tile as dS for the dQ products, bwd_mma_dq), and its
// pd_free, res_empty and drain barriers also count warp 10's commits.
template <int D, bool BF16, bool KV, bool FQ>
__device__ void bwd_mma_pipe(const Params &p, bool causal, uint32_t sRes, uint32_t sStage, uint32_t sDs, uint32_t tmem,
                             BBars<D, KV, FQ> b, Ctl c)
{
    using C = BCfg<D, KV, FQ>;
    constexpr uint32_t kIdescSS = instr_desc_f16(BF16, kTile, kTile, false);
    constexpr uint32_t kIdescTS = instr_desc_f16(BF16, kTile, D, true);
    const uint32_t r0_lo = desc_lo(sRes, 16), r1_lo = desc_lo(sRes + C::kTileBytes, 16);
    const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP;
    const uint32_t tAcc0 = tmem + C::kColAcc0, tAcc1 = tmem + C::kColAcc1;
    int g = 0, tiles = 0;   // global step, tiles started
    bool ok = true;

    // S_g = R0 S0_g^T and dP_g = R1 S1_g^T into their columns (the previous
    // step's S and dP must have been loaded by the compute warps).
    auto issue_sd = [&](int gs) -> bool {
        if (C::kSplitRing) {   // the dQ pass at D = 128 (measured 1.4-4 % faster; neutral in the fused pass)
            if (!warp_wait_all(b.sd_free(), (uint32_t)(gs - 1) & 1u, gs > 0, b.full(gs % C::kRing0),
                               (uint32_t)(gs / C::kRing0) & 1u, true, b.full1(gs % C::kRing1),
                               (uint32_t)(gs / C::kRing1) & 1u, true, c, kSiteBwdSlotFull))
                return false;
        } else {
            if (gs > 0 && !warp_wait(b.sd_free(), (uint32_t)(gs - 1) & 1u, c, kSiteBwdSdFree))
                return false;
            if (!warp_wait(b.full(gs % C::kRing0), (uint32_t)(gs / C::kRing0) & 1u, c, kSiteBwdSlotFull))
                return false;
        }
        ptx::tc_fence_after_sync();
        const uint32_t s0_lo = desc_lo(C::slot0(sStage, gs), 16), s1_lo = desc_lo(C::slot1(sStage, gs), 16);
        if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk / 4) * (C::kBoxBytes >> 4) + (kk % 4) * 2);
                ptx::mma_ss(tS, desc_from_lo(r0_lo + off), desc_from_lo(s0_lo + off), kIdescSS, kk > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk / 4) * (C::kBoxBytes >> 4) + (kk % 4) * 2);
                ptx::mma_ss(tDP, desc_from_lo(r1_lo + off), desc_from_lo(s1_lo + off), kIdescSS, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(b.sd_full());
            if (C::kSplitRing)
                ptx::mma_commit(b.empty1(gs % C::kRing1));   // V's slot is free once dP is computed
        }
        __syncwarp();
        return true;
    };

    for (int r = 0; ok; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<KV>(p, causal, t, bh, rt, s0, n);
        if (!warp_wait(b.res_full(), (uint32_t)tiles & 1u, c, kSiteBwdResFull))
            break;
        ptx::tc_fence_after_sync();
        if (!issue_sd(g))
            break;
        for (int j = 0; j < n; ++j, ++g) {
            if (j + 1 < n && !issue_sd(g + 1)) {
                ok = false;
                break;
            }
            if (j == 0 && tiles > 0 &&   // the accumulators are overwritten: the previous tile's were read out
                !warp_wait(b.acc_free(), (uint32_t)(tiles - 1) & 1u, c, kSiteBwdAccFree)) {
                ok = false;
                break;
            }
            const bool pok = KV ? warp_wait(b.p_full(), (uint32_t)g & 1u, c, kSiteBwdPFull)
                                : warp_wait(b.p_full_dq(g), (uint32_t)(g >> 1) & 1u, c, kSiteBwdPFull);
            if (!pok) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            const int st = g % C::kRing0;
            // KV:  dV += P^T_g dO_g, dK += dS^T_g Q_g;  dQ pass: dQ += dS_g K_g.
            // The A operand comes from a TMEM buffer (8 columns per 16 rows of the
            // streamed tile), the B operand is the streamed tile read MN-major
            // (16 rows = 2 KB per k-step).
            const uint32_t m0_lo = desc_lo(KV ? C::slot1(sStage, g) : C::slot0(sStage, g), C::kBoxBytes);   // KV: dO; dQ: K
            const uint32_t m1_lo = desc_lo(C::slot0(sStage, g), C::kBoxBytes);                               // KV: Q
            const uint32_t tA0 = tmem + (KV ? C::kColP : C::kColDS + 64u * (uint32_t)(g & 1));
            const uint32_t tA1 = tmem + C::kColDS;
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    ptx::mma_ts(tAcc0, tA0 + 8 * kk, desc_from_lo(m0_lo + kk * (2048 >> 4)), kIdescTS,
                                (j > 0 || kk > 0) ? 1u : 0u);
                if (KV && FQ) {   // dS^T K-major in shared memory: 32 bytes per k-step, a box per 64 queries
                    const uint32_t ds_lo = desc_lo(sDs, 16);
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        ptx::mma_ss(tAcc1, desc_from_lo(ds_lo + (uint32_t)((kk / 4) * (C::kBoxBytes >> 4) + (kk % 4) * 2)),
                                    desc_from_lo(m1_lo + kk * (2048 >> 4)), kIdescTS, (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(b.pd_free());
                } else if (KV) {
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk)
                        ptx::mma_ts(tAcc1, tA1 + 8 * kk, desc_from_lo(m1_lo + kk * (2048 >> 4)), kIdescTS,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(b.pd_free());
                }
                ptx::mma_commit(b.empty(st));
                if (j == n - 1) {
                    ptx::mma_commit(b.acc_full());
                    ptx::mma_commit(b.res_empty());
                }
            }
            __syncwarp();
        }
        ++tiles;
    }
    if (ptx::elect_one())
        ptx::mma_commit(b.drain());
    __syncwarp();
    wait_landed(b.drain(), 0u, c, kSiteBwdDrain);
}

// FQ: dS^T goes to the shared-memory tile at sDs instead of TMEM.
template <int D, bool BF16, bool CAUSAL, bool KV, bool FQ>
__device__ void bwd_compute_pipe(const Params &p, uint32_t tmem, uint32_t sStage, uint32_t sDs, BBars<D, KV, FQ> b,
                                 Ctl c)
{
    using C = BCfg<D, KV, FQ>;
    const int h = threadIdx.x / 128;                            // column half of S and dP
    const int warp = threadIdx.x / 32;
    const int row = (warp % 4) * 32 + threadIdx.x % 32;         // TMEM lane = row of the resident tile
    const uint32_t lane_off = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t tS = tmem + C::kColS + lane_off + 64 * h, tDP = tmem + C::kColDP + lane_off + 64 * h;
    const uint64_t qk2 = ptx::f2_pack(p.qk2, p.qk2);
    int g = 0, tiles = 0;
    for (int r = 0;; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<KV>(p, CAUSAL, t, bh, rt, s0, n);
        uint64_t nlg = 0, ndl = 0;   // dQ pass: this thread's query row's -lg and -delta
        if (!KV) {
            const size_t off = (size_t)bh * p.Npad + (size_t)rt * kTile + row;
            nlg = ptx::f2_pack(p.lg[off], p.lg[off]);
            ndl = ptx::f2_pack(p.dl[off], p.dl[off]);
        }
        for (int j = 0; j < n; ++j, ++g) {
            const int si = s0 + j;   // streamed tile
            if (!warp_wait(b.sd_full(), (uint32_t)g & 1u, c, kSiteBwdSdFull))
                return;
            ptx::tc_fence_after_sync();
            uint32_t sv[64], dv[64];
            ptx::tmem_ld64(tS, sv);   // this warpgroup's 64 columns of S and dP, then release both
            ptx::tmem_ld64(tDP, dv);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.sd_free());
            // KV: lane = key, column = query (lg and delta per column, from the
            // stage); dQ pass: lane = query, column = key.  Masks: the band's
            // edges (the causal diagonal), and in the dQ pass keys past Nkv
            // (padding queries and queries without keys have lg = +inf, stored as -inf).
            const uint32_t vec = sStage + (g % C::kStages) * C::kStageBytes + 2 * C::kTileBytes;
            const int limit = KV ? kTile : p.Nkv - si * kTile;   // dQ pass: columns >= limit past Nkv
            const StepMask sm = bwd_step_mask(p, CAUSAL, KV ? rt : si, KV ? si : rt);
            const bool masked = !sm.whole || limit < 64 * h + 64;
            const LaneMask lm = bwd_lane_mask<KV>(sm, row, limit);
            // Scaled scores x = S * s log2(e) - lg in place; masked steps then set
            // hidden scores to -inf (exp2 gives 0) in a separate pass, so the
            // main loop carries no mask code.
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
                uint64_t nl01 = nlg, nl23 = nlg;   // -lg, as pairs (KV: four queries' in one load)
                if (KV) {
                    const float4 l4 = ptx::ld_shared_v4f32(vec + (uint32_t)(64 * h + i) * 4);
                    nl01 = ptx::f2_pack(l4.x, l4.y);
                    nl23 = ptx::f2_pack(l4.z, l4.w);
                }
                float x0, x1, x2, x3;
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), qk2, nl01),
                               x0, x1);
                ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])), qk2, nl23),
                               x2, x3);
                sv[i] = __float_as_uint(x0);
                sv[i + 1] = __float_as_uint(x1);
                sv[i + 2] = __float_as_uint(x2);
                sv[i + 3] = __float_as_uint(x3);
            }
            if (masked) {
                const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll
                for (int i = 0; i < 64; ++i)
                    sv[i] = ((uint32_t)(lm.a + 64 * h + i) < lm.width) ? sv[i] : ninf;
            }
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
                uint64_t nd[2] = {ndl, ndl};   // -delta, as pairs (KV: four queries' in one load)
                if (KV) {
                    const float4 d4 = ptx::ld_shared_v4f32(vec + kTile * 4 + (uint32_t)(64 * h + i) * 4);
                    nd[0] = ptx::f2_pack(d4.x, d4.y);
                    nd[1] = ptx::f2_pack(d4.z, d4.w);
                }
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float p0 = ptx::ex2(__uint_as_float(sv[i + e])), p1 = ptx::ex2(__uint_as_float(sv[i + e + 1]));
                    float d0, d1;
                    ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(p0, p1),
                                               ptx::f2_add(ptx::f2_pack(__uint_as_float(dv[i + e]), __uint_as_float(dv[i + e + 1])),
                                                           nd[e / 2])),
                                   d0, d1);
                    sv[i + e] = __float_as_uint(p0);   // P, kept for KV's P^T
                    sv[i + e + 1] = __float_as_uint(p1);
                    dv[i + e] = __float_as_uint(d0);   // dS
                    dv[i + e + 1] = __float_as_uint(d1);
                }
            }
            uint32_t pk[32], dk[32];   // P and dS as 16-bit pairs, both packed before the wait below
#pragma unroll
            for (int i = 0; i < 32; ++i)
                dk[i] = BF16 ? ptx::pack_bf16x2(__uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1]))
                             : ptx::pack_f16x2(__uint_as_float(dv[2 * i]), __uint_as_float(dv[2 * i + 1]));
            if (KV) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    pk[i] = BF16 ? ptx::pack_bf16x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]))
                                 : ptx::pack_f16x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]));
                // the single P^T / dS^T buffers: the previous step's products must have read them
                if (g > 0 && !warp_wait(b.pd_free(), (uint32_t)(g - 1) & 1u, c, kSiteBwdPdFree))
                    return;
                ptx::tc_fence_after_sync();
                ptx::tmem_st32(tmem + C::kColP + lane_off + 32 * h, pk);
            }
            if (FQ) {   // key row `row`, queries [64h, 64h + 64): one 128-byte swizzled row of box h
                const uint32_t rb = sDs + (uint32_t)(h * C::kBoxBytes + row * 128);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    fq::st_shared_v4(rb + (uint32_t)((ch ^ (row & 7)) << 4), dk[4 * ch], dk[4 * ch + 1], dk[4 * ch + 2],
                                      dk[4 * ch + 3]);
                ptx::fence_proxy_async_smem();   // visible to the tensor core's reads
            } else {
                ptx::tmem_st32(tmem + C::kColDS + (KV ? 0u : 64u * (uint32_t)(g & 1)) + lane_off + 32 * h, dk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(KV ? b.p_full() : b.p_full_dq(g));
        }
        // The tile's accumulators (see bwd_compute).
        if (!warp_wait(b.acc_full(), (uint32_t)tiles & 1u, c, kSiteBwdAccFull))
            return;
        ptx::tc_fence_after_sync();
        const int grow = rt * kTile + row;
        if (KV) {
            const uint32_t tA = tmem + (h ? C::kColAcc1 : C::kColAcc0) + lane_off;
            char *dst = static_cast<char *>(h ? p.dA : p.dB) + ((size_t)bh * p.Nkv + grow) * D * 2;
            const float mul = h ? p.scale : 1.f;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t v[32];
                ptx::tmem_ld32(tA + 32 * cc, v);
                ptx::tmem_wait_ld();
                if (grow < p.Nkv)
                    store_row32<BF16>(dst + cc * 64, v, mul);
            }
        } else {
            char *dst = static_cast<char *>(p.dA) + ((size_t)bh * p.N + grow) * D * 2;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int col = h * (D / 2) + 32 * cc;
                uint32_t v[32];
                ptx::tmem_ld32(tmem + C::kColAcc0 + lane_off + col, v);
                ptx::tmem_wait_ld();
                if (grow < p.N)
                    store_row32<BF16>(dst + col * 2, v, p.scale);
            }
        }
        ptx::tc_fence_before_sync();
        ptx::mbar_arrive(b.acc_free());
        ++tiles;
    }
}

// ------------------------------------------------------------------ fused pass: dQ

// The fused pass's dQ products (warp 10): per step g, once the compute warps
// have written dS^T_g (p_full) and the read-out warps have loaded the
// previous product (dq_free), dQ_g = dS_g K into the dQ columns -- A is the
// dS^T tile read MN-major (dS: M = 128 queries, contiguous, a box per 64; K =
// 128 keys, 16 rows = 2 KB per k-step), B the resident K tile read MN-major
// as in dV += P^T dO.  Its commits: dq_full (the product is final), pd_free
// (the dS^T tile was read; that barrier also counts warp 9's commit of dV and
// dK), res_empty after a tile's last step (K was read), and drain.
template <int D, bool BF16, bool CAUSAL>
__device__ void bwd_mma_dq(const Params &p, uint32_t sRes, uint32_t sDs, uint32_t tmem, BBars<D, true, true> b, Ctl c)
{
    using C = BCfg<D, true, true>;
    // instr_desc_f16 with bit 15 (A MN-major) set as well: A and B MN-major
    constexpr uint32_t kIdesc = instr_desc_f16(BF16, kTile, D, true) | (1u << 15);
    const uint32_t a_lo = desc_lo(sDs, C::kBoxBytes), k_lo = desc_lo(sRes, C::kBoxBytes);
    const uint32_t tDQ = tmem + C::kColDQ;
    int g = 0, tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<true>(p, CAUSAL, t, bh, rt, s0, n);
        if (!warp_wait(b.res_full(), (uint32_t)tiles & 1u, c, kSiteBwdResFull))
            break;
        for (int j = 0; j < n; ++j, ++g) {
            if (!warp_wait(b.p_full(), (uint32_t)g & 1u, c, kSiteBwdPFull) ||
                (g > 0 && !warp_wait(b.dq_free(), (uint32_t)(g - 1) & 1u, c, kSiteBwdDqFree))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk)
                    ptx::mma_ss(tDQ, desc_from_lo(a_lo + kk * (2048 >> 4)), desc_from_lo(k_lo + kk * (2048 >> 4)), kIdesc,
                                kk > 0 ? 1u : 0u);
                ptx::mma_commit(b.dq_full());
                ptx::mma_commit(b.pd_free());
                if (j == n - 1)
                    ptx::mma_commit(b.res_empty());
            }
            __syncwarp();
        }
        ++tiles;
    }
    if (ptx::elect_one())
        ptx::mma_commit(b.drain());
    __syncwarp();
    wait_landed(b.drain(), 0u, c, kSiteBwdDrain);
}

// Read-out warps (12-15) sync among themselves (named barrier 3) and agree
// (named barrier 4, true iff `ok` held in every thread).
__device__ __forceinline__ void dq_sync()
{
    asm volatile("bar.sync 3, 128;" ::: "memory");
}

__device__ __forceinline__ bool dq_all(bool ok)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 4, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

// The fused pass's read-out (warps 12-15, a thread per query row of the
// streamed tile): per step, the dQ product's row from TMEM into the fp32
// staging tile (two 32-column boxes, 128-byte swizzle), released to the next
// product (dq_free), then one thread adds the tile into the accumulator rows
// of the step's query tile with two tensor reductions (fp32 add in L2).  The
// staging is rewritten only after the previous reductions have read it.
template <int D, bool CAUSAL>
__device__ void bwd_dq_out(const CUtensorMap *tmDQ, const Params &p, uint32_t tmem, uint32_t sDq,
                           BBars<D, true, true> b, Ctl c)
{
    using C = BCfg<D, true, true>;
    static_assert(D == 64, "two 32-column boxes");
    const int warp = threadIdx.x / 32;
    const int q = (warp % 4) * 32 + threadIdx.x % 32;   // TMEM lane = query row of the streamed tile
    const uint32_t tq = tmem + C::kColDQ + ((uint32_t)((warp % 4) * 32) << 16);
    const bool leader = threadIdx.x == kDqWarp0 * 32;
    bool pending = false;   // leader: reductions issued whose reads of the staging may still run
    int g = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int t = bwd_tile(r, blockIdx.x, gridDim.x);
        if (t >= p.T)
            break;
        int bh, rt, s0, n;
        bwd_decode<true>(p, CAUSAL, t, bh, rt, s0, n);
        for (int j = 0; j < n; ++j, ++g) {
            if (!dq_all(wait_bounded(b.dq_full(), (uint32_t)g & 1u, c, kSiteBwdDqFull))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after_sync();
            // Two round trips to TMEM of 32 columns each (box 0, then box 1);
            // the product is released as soon as the second has landed.
            uint32_t v[2][16];
            ptx::tmem_ld16(tq, v[0]);
            ptx::tmem_ld16(tq + 16, v[1]);
            if (leader && pending)
                fq::bulk_wait_group_read0();
            dq_sync();   // the staging is free
            auto stage_box = [&](int box) {   // this row's 32 columns of box `box`: 8 swizzled 16-byte chunks
                const uint32_t rowb = sDq + (uint32_t)(box * C::kDqBoxBytes + q * 128);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    fq::st_shared_v4(rowb + (uint32_t)((ch ^ (q & 7)) << 4), v[ch / 4][4 * (ch % 4)],
                                      v[ch / 4][4 * (ch % 4) + 1], v[ch / 4][4 * (ch % 4) + 2], v[ch / 4][4 * (ch % 4) + 3]);
            };
            ptx::tmem_wait_ld();
            stage_box(0);
            ptx::tmem_ld16(tq + 32, v[0]);
            ptx::tmem_ld16(tq + 48, v[1]);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.dq_free());
            stage_box(1);
            ptx::fence_proxy_async_smem();   // the staging, visible to the reductions
            dq_sync();
            if (leader) {
                const int y = bh * p.Npad + (s0 + j) * kTile;
                fq::tma_reduce_add_2d(tmDQ, sDq, 0, y);
                fq::tma_reduce_add_2d(tmDQ, sDq + C::kDqBoxBytes, 32, y);
                fq::bulk_commit_group();
                pending = true;
            }
        }
    }
    if (leader && pending)
        fq::bulk_wait_group0();   // the reductions are done with the staging (and complete) before exit
}

// ------------------------------------------------------------------ kernels

// KV = true:  tmR0 = K, tmR1 = V (resident), tmS0 = Q, tmS1 = dO (streamed)
// KV = false: tmR0 = Q, tmR1 = dO (resident), tmS0 = K, tmS1 = V (streamed)
// FQ (fused, KV at D = 64): tmDQ = the fp32 dQ accumulator [B*H*Npad, D] (32 x 128 boxes); otherwise unused.
template <int D, bool BF16, bool CAUSAL, bool KV, bool FQ = false>
__global__ void __launch_bounds__(FQ ? kThreadsFused : kThreads, 1)
    fa_bwd_sm103(const __grid_constant__ CUtensorMap tmR0, const __grid_constant__ CUtensorMap tmR1,
                 const __grid_constant__ CUtensorMap tmS0, const __grid_constant__ CUtensorMap tmS1,
                 const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ Params p)
{
    using C = BCfg<D, KV, FQ>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128-byte swizzle atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sRes = base + C::kResOff;
    const uint32_t sStage = base + C::kStageOff;
    const uint32_t sDs = base + C::kDsOff, sDq = base + C::kDqOff;
    BBars<D, KV, FQ> b{base + C::kBarOff};
    uint32_t *misc = reinterpret_cast<uint32_t *>(base_ptr + C::kMiscOff);
    Ctl c{reinterpret_cast<volatile int *>(misc + 1)};
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kRing0; ++s) {
            ptx::mbar_init(b.full(s), 1);
            ptx::mbar_init(b.empty(s), 1);
        }
        for (int s = 0; C::kSplitRing && s < C::kRing1; ++s) {
            ptx::mbar_init(b.full1(s), 1);
            ptx::mbar_init(b.empty1(s), 1);
        }
        // the fused pass's two MMA warps both commit res_empty, drain and pd_free
        ptx::mbar_init(b.res_full(), 1);
        ptx::mbar_init(b.res_empty(), FQ ? 2 : 1);
        ptx::mbar_init(b.sd_full(), 1);
        ptx::mbar_init(b.p_full(), kComputeThreads);
        ptx::mbar_init(b.acc_full(), 1);
        ptx::mbar_init(b.acc_free(), kComputeThreads);
        ptx::mbar_init(b.drain(), FQ ? 2 : 1);
        ptx::mbar_init(b.sd_free(), kComputeThreads);
        ptx::mbar_init(b.pd_free(), FQ ? 2 : 1);
        ptx::mbar_init(b.p_full_dq(1), KV ? 1 : kComputeThreads);   // KV: dp_full, committed by the MMA warp
        if (FQ) {
            ptx::mbar_init(b.dq_full(), 1);
            ptx::mbar_init(b.dq_free(), 128);
        }
        *c.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(misc), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        ptx::prefetch_tensormap(&tmR0);
        ptx::prefetch_tensormap(&tmR1);
        ptx::prefetch_tensormap(&tmS0);
        ptx::prefetch_tensormap(&tmS1);
        if (FQ)
            ptx::prefetch_tensormap(&tmDQ);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc);
    // Launched right behind the previous kernel of the backward (programmatic
    // dependent launch): the set-up above overlaps its end.
    fq::grid_launch_dependents();   // the next kernel may start launching
    fq::grid_wait();                // the previous kernel's results (-lg, -delta, the zeroed accumulator) are written

    if (threadIdx.x < kComputeThreads) {
        ptx::regs_increase<FQ ? kRegsComputeFused : kRegsCompute>();
        if constexpr (kPipeline<D, KV>)
            bwd_compute_pipe<D, BF16, CAUSAL, KV, FQ>(p, tmem, sStage, sDs, b, c);
        else
            bwd_compute<D, BF16, CAUSAL, KV>(p, tmem, sStage, b, c);
    } else if (FQ && warp >= kDqWarp0) {
        ptx::regs_decrease<kRegsOtherFused>();
        if constexpr (FQ)
            bwd_dq_out<D, CAUSAL>(&tmDQ, p, tmem, sDq, b, c);
    } else {
        ptx::regs_decrease<FQ ? kRegsOtherFused : kRegsProducer>();
        if (warp == kLoadWarp)
            bwd_load<D, KV, FQ>(&tmR0, &tmR1, &tmS0, &tmS1, p, CAUSAL, sRes, sStage, b, c);
        else if (warp == kMmaWarp)
        {
            if constexpr (kPipeline<D, KV>)
                bwd_mma_pipe<D, BF16, KV, FQ>(p, CAUSAL, sRes, sStage, sDs, tmem, b, c);
            else
                bwd_mma<D, BF16, KV>(p, CAUSAL, sRes, sStage, tmem, b, c);
        }
        else if (FQ && warp == kMmaWarpDq)
        {
            if constexpr (FQ)
                bwd_mma_dq<D, BF16, CAUSAL>(p, sRes, sDs, tmem, b, c);
        }
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// -delta = -rowsum(dO o O) and -lg = -LSE * log2(e) per query row (negated,
// as the passes add them), padded to whole 128-row tiles: D / 8 threads per
// row, 16 bytes each.  dqa (the fused
// pass's fp32 dQ accumulator, [rows][D], or null): zeroed, 8 values a thread.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
    fa_bwd_prep(const uint16_t *O, const uint16_t *dO, const float *LSE, float *lg, float *dl, float *dqa, int N,
                int Npad, long long rows)
{
    fq::grid_launch_dependents();   // the fused pass may start launching behind this kernel
    constexpr int kTpr = D / 8;   // threads per row: 8 or 16, a divisor of 32
    const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = g / kTpr;
    const int part = (int)(g % kTpr);
    if (row >= rows)   // whole row groups leave together (kTpr divides the warp)
        return;
    const long long bh = row / Npad;
    const int i = (int)(row - bh * Npad);
    if (dqa) {
        float4 *z = reinterpret_cast<float4 *>(dqa + row * D + 8 * part);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.f;
    if (i < N) {
        const size_t e = ((size_t)bh * N + i) * D + 8 * part;
        const uint4 o4 = *reinterpret_cast<const uint4 *>(O + e);
        const uint4 d4 = *reinterpret_cast<const uint4 *>(dO + e);
        const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float o0, o1, d0, d1;
            if (BF16) {
                o0 = __uint_as_float(ow[k] << 16);
                o1 = __uint_as_float(ow[k] & 0xffff0000u);
                d0 = __uint_as_float(dw[k] << 16);
                d1 = __uint_as_float(dw[k] & 0xffff0000u);
            } else {
                o0 = __half2float(__ushort_as_half((unsigned short)(ow[k] & 0xffffu)));
                o1 = __half2float(__ushort_as_half((unsigned short)(ow[k] >> 16)));
                d0 = __half2float(__ushort_as_half((unsigned short)(dw[k] & 0xffffu)));
                d1 = __half2float(__ushort_as_half((unsigned short)(dw[k] >> 16)));
            }
            acc = fmaf(o0, d0, acc);
            acc = fmaf(o1, d1, acc);
        }
    }
    const int lane = threadIdx.x % 32;
    const uint32_t group = ((1u << kTpr) - 1u) << (lane & ~(kTpr - 1));
#pragma unroll
    for (int m = kTpr / 2; m > 0; m /= 2)
        acc += __shfl_xor_sync(group, acc, m);
    if (part == 0) {   // negated, as the passes add them
        float l = -INFINITY;
        if (i < N) {
            const float lse = LSE[(size_t)bh * N + i];
            l = (lse == -INFINITY) ? -INFINITY : -(lse * 1.4426950408889634f);   // a row without keys: P = 0
        }
        lg[row] = l;
        dl[row] = (i < N) ? -acc : 0.f;
    }
}

// The fused pass's dQ: dQ = scale * the fp32 accumulator, in the input type,
// for the N real rows of each head (8 values a thread).
template <bool BF16>
__global__ void __launch_bounds__(256)
    fa_bwd_dq_convert(const float *dqa, uint16_t *dQ, int N, int Npad, int D, long long elems, float scale)
{
    fq::grid_wait();   // launched right behind the fused pass: its accumulator is complete
    const long long e = ((long long)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (e >= elems)
        return;
    const long long row = e / D;   // of [B*H*N]; D is a multiple of 8
    const int col = (int)(e - row * D);
    const long long bh = row / N;
    const long long src = (bh * Npad + (row - bh * N)) * D + col;
    const float4 a = *reinterpret_cast<const float4 *>(dqa + src);
    const float4 b = *reinterpret_cast<const float4 *>(dqa + src + 4);
    uint4 o;
    o.x = BF16 ? ptx::pack_bf16x2(a.x * scale, a.y * scale) : ptx::pack_f16x2(a.x * scale, a.y * scale);
    o.y = BF16 ? ptx::pack_bf16x2(a.z * scale, a.w * scale) : ptx::pack_f16x2(a.z * scale, a.w * scale);
    o.z = BF16 ? ptx::pack_bf16x2(b.x * scale, b.y * scale) : ptx::pack_f16x2(b.x * scale, b.y * scale);
    o.w = BF16 ? ptx::pack_bf16x2(b.z * scale, b.w * scale) : ptx::pack_f16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4 *>(dQ + e) = o;
}

}  // namespace bwd
}  // namespace fa
