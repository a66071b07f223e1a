// fa_fwd_kernel.cuh -- FlashAttention-2 forward for GB300 (sm_103a).
//
// What it computes (for each batch*head slice and query row i):
//   O[i,:] = sum_j softmax_j(scale * q_i . k_j) v_j,  LSE[i] = log sum_j exp(scale * q_i . k_j)
// over all keys, or keys j <= i when CAUSAL, by the FlashAttention-2 forward
// recurrence: K/V tiles stream past an on-chip Q tile; per row a running max m
// and sum l rescale an fp32 accumulator by exp(m_old - m_new), and the
// accumulator is divided by l once at the end.  The N x N scores never leave
// the chip.  ("FlashAttention 2 from PyTorch to Triton", What I am building;
// "A09 - Advanced Triton & FlashAttention", 3. Deep Dive: the rescaling update.)
//
// Work decomposition.  A CTA tile is 256 query rows of one head, split into
// two 128-row Q tiles that share every K/V tile.  Persistent CTAs (one per SM)
// walk the CTA tiles; causal launches take the longest tiles first, heads
// interleaved ("How to profile and optimise kernels", causal launch order).
//
// Warp roles (512 threads, four warpgroups):
//   warpgroup 0  softmax of Q tile 0: S -> P, running max m and sum l (a row per thread),
//                and the (rare) O rescale
//   warpgroup 1  the same for Q tile 1
//   warpgroup 2  epilogue for both Q tiles: O = acc / l and LSE, written once per tile
//   warpgroup 3  warp 12: TMA producer (Q tiles, then K_j and V_j into a stage ring)
//                warps 13, 14: tcgen05 MMA issuers for Q tiles 0 and 1 at D = 64;
//                warp 13 alone issues for both at D = 128 (warp 13 owns TMEM)
//                warp 15: merge warp of the balanced variants
// Registers are rebalanced with setmaxnreg: the softmax warpgroups hold a
// 128-score row per thread, the other two need little.  The producer warps
// run as whole warps with one elected lane issuing, so their control state is
// warp-uniform.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [256+D,256+2D)
//   D = 64:  P0 [384,448) and P1 [448,512) hold P (two 16-bit values per
//            column), so S_{j+1} may be computed while softmax still works on
//            S_j: the softmax releases S_w as soon as it has loaded it.
//   D = 128: no room for separate P: P_w overwrites columns [0,64) of S_w,
//            and S_w of step j+1 is issued after the MMA that reads P_w(j)
//            (tcgen05 MMAs from one thread execute in issue order).  When
//            every head has at most 128 query rows (decoding), Q tile 1 is
//            idle: P_0 goes to S1's columns and the steps run in the D = 64
//            order, with each stage's K and V released separately.
// P feeds the P.V MMA as its TMEM A operand.
//
// MMA issue order per K/V step j, per Q tile w:
//   D = 64:  S_w(j+1) as soon as the softmax has loaded S_w(j), then O_w += P_w(j) V_j;
//            each tile has its own issuing warp, so the two streams interleave
//            on the tensor core by themselves
//   D = 128: one warp issues S0(j), O1 += P1(j-1) V_{j-1}, S1(j), O0 += P0(j) V_j,
//            each P.V once P_w has overwritten S_w; heads of one Q tile run
//            the D = 64 order instead
// so each softmax warpgroup's work overlaps the other tile's MMAs.
//
// Softmax follows the exp2 form ("How to profile and optimise kernels", exp2):
// qk_scale = scale*log2(e) is folded once, the row max is taken on raw scores
// and then scaled (valid because scale > 0), m is kept in log2 units, and
// LSE = (m + log2 l) * ln 2.  P is rounded to the input type for the P.V MMA;
// l is summed from the fp32 P (the P cast section of the same page).
// l and O are rescaled by exp2(m_old - m_new) only for rows whose max moved
// (alpha = 1 otherwise, "A09 - Advanced Triton & FlashAttention", 3. Deep
// Dive: the rescaling update); a warp whose 32 rows all kept their max skips
// the O rescale.  As more keys are seen a new maximum becomes ever rarer, so
// the softmax warps do the rescale themselves before releasing P instead of
// handing it to other warps every step.
// Masking happens only on the diagonal tile (causal) and the ragged last key
// tile; tiles above the diagonal are never loaded ("A09 - Advanced Triton &
// FlashAttention", causal masking: skipping beats masking).  Masked scores
// are -inf, and a row whose visible maximum is still -inf uses a shift of 0 so
// that no -inf - (-inf) NaN can arise ("Triton: FlashAttention-2 Forward
// Pass", masks and sentinels).
//
// Every mbarrier wait is bounded (about one second of global time).  On
// expiry the kernel records the failing wait in a device status word, all
// roles leave their loops, in-flight copies and MMAs are drained with bounded
// waits, TMEM is freed and the kernel returns.
#pragma once

#include <cuda.h>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "fa_schedule.h"
#include "sm103_ptx.cuh"

namespace fa {

// Device status word: 0 = fine; otherwise 1 | (site << 8) of the first wait
// that expired.  Each translation unit that includes this header has its own
// (device code is not linked across units); fa_sync_status() reads and clears
// every unit's word (take_status_word_on).
static __device__ unsigned int g_status_word;

// fa_sync_status's read of this unit's status word: one thread takes the
// word and clears it in a single atomic exchange, so a timeout that a kernel
// on another stream records meanwhile is kept for the next read, never lost.
static __device__ unsigned int g_status_taken;
static __global__ void take_status_kernel()
{
    g_status_taken = atomicExch(&g_status_word, 0u);
}

// Host: read and clear this unit's status word (current device) on stream
// `s` into *word; false if a launch or copy failed.
static inline bool take_status_word_on(cudaStream_t s, unsigned int *word)
{
    *word = 0;
    take_status_kernel<<<1, 1, 0, s>>>();
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyFromSymbolAsync(word, g_status_taken, sizeof *word, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        *word = 0;
        return false;
    }
    return true;
}

constexpr int kBM = 128;        // query rows per Q tile (one TMEM lane each)
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kQTiles = 2;      // Q tiles per CTA tile
constexpr int kCtaRows = kBM * kQTiles;
constexpr int kThreads = 512;
// Masks, a template parameter of the kernel: none; keys up to a bound after
// the query (causal, or any band unbounded on the left: K/V steps start at 0
// and one compare per score masks); a band with a left bound (K/V steps start
// where the tile's band does, two-sided masking).  Separate variants keep the
// causal hot loop free of the band's extra compares.
constexpr int kMaskNone = 0;
constexpr int kMaskCausal = 1;
constexpr int kMaskBand = 2;
constexpr int kEpilogueWarpgroup = 2;
constexpr int kLoadWarp = 12;
constexpr int kMmaWarp = 13;          // MMA issuer(s): warp 13 (and 14 at D = 64)
constexpr int kMergeWarp = 15;        // merges split tiles (balanced schedule)
constexpr uint32_t kRegsSoftmax = 184;   // 2 x 128 x 184 + 128 x 64 + 128 x 80 = 65536 (launch: 512 x 128)
constexpr uint32_t kRegsEpilogue = 64;
constexpr uint32_t kRegsProducer = 80;
constexpr int kPerTileBars = 7;
constexpr int kMergeBufs = 4;            // merge staging buffers in flight
constexpr int kMergeOBytes = 4096;       // partial O bytes per staging buffer
constexpr int kMaxMergeParts = kSchedMaxParts;   // parts of one split tile, at most (the planner keeps to it)
// (m, l) staging of a merge: parts x rows x 8 bytes -- 8 parts of 128 rows,
// 16 of 64 or 32 of 32 (sched_ml_rows; the planner allows more than 8 parts
// only for heads that short).
constexpr int kMlBytes = kSchedMaxPartsTall * kBM * 8;
static_assert(kSchedMaxParts * sched_ml_rows(kSchedMaxParts) * 8 <= kMlBytes &&
                  (kSchedMaxParts / 2) * sched_ml_rows(kSchedMaxParts / 2) * 8 <= kMlBytes,
              "merge staging holds the short-head parts");
constexpr int kJobSlots = 2;             // merge jobs queued from the epilogue to the merge warp

// A merge job, posted by the epilogue in shared memory: the Q tile's rows
// [orow0, orow0 + nrows) of the [B*H*N] output rows, the workspace counter to
// reset, and each part's partial O and (m, l) (row 0 of the Q tile in its
// slot).  nparts = 0 tells the merge warp to stop.
struct MergeJob {
    long long orow0;
    int nrows;
    int nparts;
    int counter;
    int pad;
    unsigned long long o_addr[kMaxMergeParts];
    unsigned long long ml_addr[kMaxMergeParts];
};
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kLn2 = 0.69314718055994530942f;
// Guarded lazy rescale (softmax_role): a new row max may leave the reference
// max in place when it exceeds it by at most kLazyMax (log2 units) and the
// row's sum is at least kLazyWeight times the new maximum's probability.
constexpr float kLazyMax = 8.f;
constexpr float kLazyWeight = 16.f;

// Wait sites recorded in the status word.
enum : uint32_t {
    kSiteLoadQEmpty = 1, kSiteLoadSlotEmpty, kSiteMmaQFull, kSiteMmaSlotFull, kSiteMmaPFull, kSiteMmaOFree,
    kSiteMmaSFree, kSiteSoftSFull, kSiteSoftODone, kSiteSoftStFree, kSiteEpiStReady, kSiteEpiODone, kSiteDrain,
    kSiteTail, kSiteMerge, kSiteMergeTail, kSiteMergeJob, kSiteEpiJobFree
};

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static constexpr bool kSeparateP = (D == 64);
    // One MMA-issuing warp per Q tile at D = 64, where the many small MMAs of a
    // step would outrun one issuer; one warp for both tiles at D = 128, where
    // its interleaved order keeps the two softmax warpgroups out of phase.
    static constexpr int kMmaWarps = (D == 64) ? 2 : 1;
    static constexpr int kBoxes = D / 64;              // 128-byte-wide TMA boxes per tile row
    static constexpr int kBoxBytes = kBM * 128;        // one [128 rows, 64 cols] 16-bit box
    static constexpr int kTileBytes = kBM * D * 2;     // one [128, D] 16-bit tile
    static constexpr int kStages = (D == 64) ? 4 : 2;  // K/V ring depth; a stage holds K_j and V_j
    static constexpr int kStageBytes = 2 * kTileBytes;
    // At D = 128 (two stages), in the separate-P order of heads of one Q
    // tile, a stage's K and V land and are released on barriers of their
    // own: K once the step's S MMA read it, V once its P.V did, and the
    // producer loads K one step ahead of V.  (The two-tile interleaved order
    // keeps whole stages: two tiles' work per step already hides the loads.)
    static constexpr bool kSplitKV = (D == 128);
    static constexpr int kQBufs = (D == 64) ? 2 : 1;   // Q buffers: the next CTA tile's Q loads early
    static constexpr int kQBufBytes = kQTiles * kTileBytes;
    static constexpr int kQOff = 0;
    static constexpr int kStageOff = kQBufs * kQBufBytes;
    static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
    // full[kStages], empty[kStages], q_full[kQBufs], q_empty[kQBufs], then per
    // Q tile: s_full, s_free, p_full, o_done, st_ready, st_free, o_free; then drain
    static constexpr int kNumBars = 2 * kStages + 2 * kQBufs + kPerTileBars * kQTiles + 1 + kMergeBufs + 1 + 2 * kJobSlots;
    static constexpr int kHandOff = kBarOff + kNumBars * 8;            // float2 [2 tiles][128]
    static constexpr int kMiscOff = kHandOff + kQTiles * kBM * 8;
    // Merge staging: kMergeBufs buffers, each the partial O of kMergeRows rows
    // of one part; the parts' (m, l) of the Q tile, float2 [parts][128 or 64
    // rows] (turned into merge weights in place); the job queue, kJobSlots MergeJobs.
    static constexpr int kMergeRows = kMergeOBytes / (D * 4);
    static constexpr int kMergeOff = (kMiscOff + 16 + 127) & ~127;
    static constexpr int kMlOff = kMergeOff + kMergeBufs * kMergeOBytes;
    static constexpr int kJobOff = kMlOff + kMlBytes;
    // The split ring's V barriers, v_full[kStages] and v_empty[kStages], come
    // after everything else (the merge area, which whole-tile launches do not
    // have): moving the other barriers by their 32 bytes measured 4.6 %
    // slower on long causal calls at D = 128.
    static constexpr int kVBarBytes = kSplitKV ? 16 * kStages : 0;
    __host__ __device__ static constexpr int vbar_off(bool split)
    {
        return split ? ((kJobOff + kJobSlots * (int)sizeof(MergeJob) + 7) & ~7) : kMiscOff + 16;
    }
    // Shared memory of a launch (+ slack to align the base to 1024).
    static constexpr int kSmemSplit = vbar_off(true) + kVBarBytes + 1024;
    static constexpr int kSmemWhole = vbar_off(false) + kVBarBytes + 1024;
    __host__ __device__ static constexpr int smem_bytes(bool split) { return split ? kSmemSplit : kSmemWhole; }
    static_assert(kSmemSplit <= 232448 && kSmemWhole <= kSmemSplit, "shared memory per CTA");
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t col_s(int w) { return w ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t col_o(int w) { return w ? 256u + D : 256u; }
    __host__ __device__ static constexpr uint32_t col_p(int w) { return kSeparateP ? (w ? 448u : 384u) : col_s(w); }
    // At D = 128 a launch whose heads have at most 128 query rows (decoding)
    // leaves Q tile 1 idle, so P_0 takes tile 1's S columns and the steps run
    // in the separate-P order of D = 64.
    __host__ __device__ static constexpr uint32_t col_p_one_tile() { return col_s(1); }
};

struct FwdParams {
    void *O;
    float *LSE;
    int N;               // query rows per head
    int Nkv;             // keys per head
    int off;             // causal: query i sees keys j <= i + off (Nkv - N, bottom-right alignment)
    float qk_scale;      // scale * log2(e)
    Schedule sch;        // work decomposition (fa_schedule.h)
    float *part_o;       // balanced schedule: partial O, [2 * grid slots][256 rows][D] fp32
    float2 *part_ml;     // balanced schedule: partial (m, l) per row, [2 * grid slots][256]
    int *counters;       // balanced schedule: finished parts per (tile, Q tile), zero between launches
};

// Separate-P order (S_{j+1} issued while the softmax of step j runs): always
// at D = 64; at D = 128 when no CTA tile has a second Q tile.
template <int D>
__device__ __forceinline__ bool separate_p(const FwdParams &p)
{
    return Cfg<D>::kSeparateP || p.N <= kBM;
}

// K and V of a stage on separate barriers (D = 128, separate-P order).
template <int D>
__device__ __forceinline__ bool split_kv(const FwdParams &p)
{
    return Cfg<D>::kSplitKV && p.N <= kBM;
}

// Shared-memory matrix descriptor (tcgen05), 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), `lbo` = leading byte offset.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t instr_desc_f16(bool bf16, int M, int N, bool b_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Q-tile step count within a part: Q tile w of the part's tile visits steps
// [0, nw); the part covers [kb, ke); its share is [kb, min(ke, nw)).
__device__ __forceinline__ int part_steps(const Part &pt, int nw)
{
    const int e = (pt.ke < nw) ? pt.ke : nw;
    return (e > pt.kb) ? e - pt.kb : 0;
}

struct Ctl {
    volatile int *abort_flag;
};

static __device__ __noinline__ void record_timeout(Ctl c, uint32_t site)
{
    *c.abort_flag = 1;
    atomicCAS(&g_status_word, 0u, 1u | (site << 8));
}

// Bounded wait by one thread; false if it gave up (timeout or abort).  Each
// poll is a try_wait, which suspends the thread for a hardware-chosen time
// until the phase completes.  (An explicit suspend-time hint of 20 us or 1 us
// measured 1 % slower on the D = 64 workloads than leaving it to the
// hardware.)  kSuspendNs is the hint for waits bounded by time alone.
constexpr uint32_t kSuspendNs = 20000;

// INLINE: record a timeout without a call, for waits that hold many live
// registers (a call there makes the caller save them around it, as spills).
template <bool INLINE = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Ctl c, uint32_t site)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((spin & 7u) == 0) {
            if (*c.abort_flag)
                return false;
            if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
                if (INLINE) {
                    *c.abort_flag = 1;
                    atomicCAS(&g_status_word, 0u, 1u | (site << 8));
                } else {
                    record_timeout(c, site);
                }
                return false;
            }
        }
    }
}

// Bounded wait by a whole warp; the outcome is warp-uniform.
template <bool INLINE = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl c, uint32_t site)
{
    const bool ok = wait_bounded<INLINE>(bar, parity, c, site);
    return __all_sync(0xffffffffu, ok);
}

template <int D>
struct Bars {
    uint32_t base;
    uint32_t vbase;   // the split ring's V barriers
    // TMA -> MMA: stage s landed (K_j alone when K and V are split)
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    // MMA -> TMA: stage s read (K_j alone when split)
    __device__ uint32_t empty(int s) const { return base + 8u * (Cfg<D>::kStages + s); }
    __device__ uint32_t v_full(int s) const { return vbase + 8u * s; }                          // split: V_j landed
    __device__ uint32_t v_empty(int s) const { return vbase + 8u * (Cfg<D>::kStages + s); }     // split: V_j read
    __device__ uint32_t q_full(int qb) const { return base + 8u * (2 * Cfg<D>::kStages + qb); }
    __device__ uint32_t q_empty(int qb) const { return base + 8u * (2 * Cfg<D>::kStages + Cfg<D>::kQBufs + qb); }
    __device__ uint32_t per_tile(int w, int k) const
    {
        return base + 8u * (2 * Cfg<D>::kStages + 2 * Cfg<D>::kQBufs + kPerTileBars * w + k);
    }
    __device__ uint32_t s_full(int w) const { return per_tile(w, 0); }     // MMA -> softmax: S_w ready
    __device__ uint32_t s_free(int w) const { return per_tile(w, 1); }     // softmax -> MMA: S_w loaded (separate-P order)
    __device__ uint32_t p_full(int w) const { return per_tile(w, 2); }     // softmax -> MMA: P_w written, O_w rescaled
    __device__ uint32_t o_done(int w) const { return per_tile(w, 3); }     // MMA -> softmax, epilogue: P.V done
    __device__ uint32_t st_ready(int w) const { return per_tile(w, 4); }   // softmax -> epilogue: final (m, l) written
    __device__ uint32_t st_free(int w) const { return per_tile(w, 5); }    // epilogue -> softmax: (m, l) read
    __device__ uint32_t o_free(int w) const { return per_tile(w, 6); }     // epilogue -> MMA: O_w read out
    __device__ uint32_t drain() const { return per_tile(kQTiles, 0); }
    __device__ uint32_t merge_full(int i) const { return per_tile(kQTiles, 1 + i); }   // bulk copy -> merge warp: buffer i landed
    __device__ uint32_t ml_full() const { return per_tile(kQTiles, 1 + kMergeBufs); }    // bulk copy -> merge warp: (m, l) landed
    __device__ uint32_t job_full(int j) const { return per_tile(kQTiles, 2 + kMergeBufs + j); }               // epilogue -> merge warp
    __device__ uint32_t job_empty(int j) const { return per_tile(kQTiles, 2 + kMergeBufs + kJobSlots + j); }  // merge warp -> epilogue
};

// ------------------------------------------------------------------ producer

// TMA producer, run by a whole warp; one elected lane issues the copies.
// Per CTA tile: both Q tiles into the Q buffer, then for each step j the
// pair K_j, V_j into the next stage of the ring.  With K and V split, the
// copies go K_0, K_1, V_0, K_2, V_1, ... (V_j after K_{j+1} within a part),
// each half waiting only for its own half of the stage.
// SKV: K and V of a stage on separate barriers (split_kv): heads of at most
// 128 query rows, whose every K/V tile is read by one CTA only, so the copies
// carry an L2 evict-first hint (the partial results, the merge's code and
// the next launch's data stay; measured 116.8 -> 108.5 us on 4 queries x
// 32768 keys x 32 heads with L2 flushed).
template <int D, int MASK, bool SPLIT, bool SKV>
__device__ void load_role(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                          const FwdParams &p, uint32_t sQ, uint32_t sStage, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    int step = 0;   // K/V stages filled so far (K halves when split)
    int it = 0;     // parts started by this CTA (one Q load each)
    int nv = 0;     // split: V halves filled so far; V of step nv is pending while nv < step
    int pv_bh = 0, pv_row = 0;   // ... its head and first key
    bool ok = true;
    const uint64_t kv_policy = ptx::l2_policy_evict_first();   // split K/V (decoding): each K/V tile is read once
    auto load_v = [&]() -> bool {
        const int st = nv % C::kStages;
        const uint32_t use = (uint32_t)(nv / C::kStages);
        if (!warp_wait(b.v_empty(st), (use & 1u) ^ 1u, c, kSiteLoadSlotEmpty))
            return false;
        if (ptx::elect_one()) {
            const uint32_t dst = sStage + st * C::kStageBytes + C::kTileBytes;
            ptx::mbar_arrive_expect_tx(b.v_full(st), C::kTileBytes);
            for (int x = 0; x < C::kBoxes; ++x)
                ptx::tma_load_3d_hint(dst + x * C::kBoxBytes, tmV, b.v_full(st), x * 64, pv_row, pv_bh, kv_policy);
        }
        __syncwarp();
        ++nv;
        return true;
    };
    PartIter parts;
    parts.init_t<SPLIT>(p.sch, blockIdx.x);
    Part pt;
    while (ok && parts.next_t<SPLIT, MASK == kMaskBand>(p.sch, pt)) {
        int bh, ct;
        sched_decode_t<SPLIT, MASK == kMaskBand>(p.sch, pt.tile, bh, ct);
        // The previous part's last V before the Q buffer is waited for: the
        // MMA warp frees that buffer only after the part's last P.V.
        if (SKV && nv < step && !load_v()) { ok = false; break; }
        const int qb = it % C::kQBufs;
        const uint32_t quse = (uint32_t)(it / C::kQBufs);
        if (!warp_wait(b.q_empty(qb), (quse & 1u) ^ 1u, c, kSiteLoadQEmpty)) { ok = false; break; }
        if (ptx::elect_one()) {
            const uint32_t dst = sQ + qb * C::kQBufBytes;
            ptx::mbar_arrive_expect_tx(b.q_full(qb), kQTiles * C::kTileBytes);
            for (int w = 0; w < kQTiles; ++w)
                for (int x = 0; x < C::kBoxes; ++x)
                    ptx::tma_load_3d(dst + w * C::kTileBytes + x * C::kBoxBytes, tmQ, b.q_full(qb), x * 64,
                                     ct * kCtaRows + w * kBM, bh);
        }
        __syncwarp();
        ++it;
        const int ks = (MASK == kMaskBand) ? sched_kv_start(p.sch, ct) : 0;   // the tile's first key step
        for (int j = pt.kb; j < pt.ke; ++j, ++step) {
            const int st = step % C::kStages;
            const uint32_t use = (uint32_t)(step / C::kStages);
            if (!warp_wait(b.empty(st), (use & 1u) ^ 1u, c, kSiteLoadSlotEmpty)) { ok = false; break; }
            if (ptx::elect_one()) {
                const uint32_t dst = sStage + st * C::kStageBytes;
                ptx::mbar_arrive_expect_tx(b.full(st), SKV ? C::kTileBytes : C::kStageBytes);
                for (int x = 0; x < C::kBoxes; ++x) {
                    if (SKV)
                        ptx::tma_load_3d_hint(dst + x * C::kBoxBytes, tmK, b.full(st), x * 64, (ks + j) * kBN, bh, kv_policy);
                    else
                        ptx::tma_load_3d(dst + x * C::kBoxBytes, tmK, b.full(st), x * 64, (ks + j) * kBN, bh);
                }
                if (!SKV)
                    for (int x = 0; x < C::kBoxes; ++x)
                        ptx::tma_load_3d(dst + C::kTileBytes + x * C::kBoxBytes, tmV, b.full(st), x * 64,
                                         (ks + j) * kBN, bh);
            }
            __syncwarp();
            if (SKV) {   // V of the previous step, then this step's V becomes the pending one
                if (nv < step && !load_v()) { ++step; ok = false; break; }
                pv_bh = bh;
                pv_row = (ks + j) * kBN;
            }
        }
    }
    if (SKV && ok && nv < step)   // the last step's V
        load_v();
    // Tail: every copy issued has landed and (unless aborting) every stage and
    // the Q buffer have been released by the MMA warp, so no asynchronous
    // write or arrive targets this CTA's shared memory after exit.
    for (int s = 0; s < C::kStages && s < step; ++s) {
        const int last = step - 1 - ((step - 1 - s) % C::kStages);   // last step that used stage s
        const uint32_t use = (uint32_t)(last / C::kStages);
        warp_wait(b.full(s), use & 1u, c, kSiteTail);
        if (!*c.abort_flag)
            warp_wait(b.empty(s), use & 1u, c, kSiteTail);
    }
    for (int s = 0; SKV && s < C::kStages && s < nv; ++s) {
        const int last = nv - 1 - ((nv - 1 - s) % C::kStages);
        const uint32_t use = (uint32_t)(last / C::kStages);
        warp_wait(b.v_full(s), use & 1u, c, kSiteTail);
        if (!*c.abort_flag)
            warp_wait(b.v_empty(s), use & 1u, c, kSiteTail);
    }
    for (int qb = 0; qb < C::kQBufs && qb < it; ++qb) {
        const int last = it - 1 - ((it - 1 - qb) % C::kQBufs);   // last CTA tile that used Q buffer qb
        const uint32_t use = (uint32_t)(last / C::kQBufs);
        warp_wait(b.q_full(qb), use & 1u, c, kSiteTail);
        if (!*c.abort_flag)
            warp_wait(b.q_empty(qb), use & 1u, c, kSiteTail);
    }
}

// ------------------------------------------------------------------ MMA issuer

// Upper word of every shared-memory descriptor used here: stride byte offset
// 1024 (8 rows of 128 bytes), descriptor version 1, 128-byte swizzle.
constexpr uint32_t kDescHi = (1024u >> 4) | (1u << 14) | (2u << 29);

__device__ __forceinline__ uint64_t desc_from_lo(uint32_t lo)
{
    return ((uint64_t)kDescHi << 32) | lo;
}

// Lower descriptor word: start address and leading byte offset (both >> 4).
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo)
{
    return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}

// The MMA-issuing warps, one per Q tile.  A single thread issues a tcgen05.mma
// only every ~60-80 cycles whatever its shape, so one issuer cannot keep the
// tensor core busy with the small per-step MMAs of attention (N = 64 P.V at
// D = 64); two issuers on different schedulers reach the full rate.  Each
// warp runs its control flow and waits as a whole warp, so loop state and
// descriptors stay warp-uniform; one elected lane (the same lane every time,
// as tcgen05.commit tracks the MMAs of the lane that issued them) issues the
// tcgen05.mma and tcgen05.commit instructions.  Tile-level ping-pong between
// the two softmax warpgroups falls out of the two independent MMA streams.
template <int D, bool BF16, bool SEP>
struct MmaIssuer {
    using C = Cfg<D>;
    static constexpr uint32_t kIdescQK = instr_desc_f16(BF16, kBM, kBN, false);   // S = Q K^T, both K-major
    static constexpr uint32_t kIdescPV = instr_desc_f16(BF16, kBM, D, true);      // O += P V, V is MN-major
    int w;               // Q tile served by this warp
    uint32_t q_lo;       // descriptor lower word of Q tile w in Q buffer 0
    uint32_t k_lo;       // descriptor lower word of K in stage 0, K-major (leading byte offset unused)
    uint32_t v_lo;       // same for V in stage 0 (MN-major: leading byte offset = box stride)
    uint32_t tS, tO, tP; // TMEM columns of S_w, O_w, P_w
    Bars<D> b;
    Ctl c;
    uint32_t n_s, n_pv, n_t;   // S and P.V MMAs issued, CTA tiles whose first P.V was issued
    uint32_t q_cur;            // descriptor lower word of Q tile w in the current Q buffer

    __device__ bool stage_wait(int step, int &st) const
    {
        st = step % C::kStages;
        if (!warp_wait(b.full(st), (uint32_t)(step / C::kStages) & 1u, c, kSiteMmaSlotFull))
            return false;
        ptx::tc_fence_after_sync();
        return true;
    }

    // Split K and V: wait for V of `step` (K is what stage_wait waits for).
    __device__ bool v_wait(int step) const
    {
        const int st = step % C::kStages;
        if (!warp_wait(b.v_full(st), (uint32_t)(step / C::kStages) & 1u, c, kSiteMmaSlotFull))
            return false;
        ptx::tc_fence_after_sync();
        return true;
    }

    // Release a stage (its K half when split) once this warp's MMAs reading
    // it have completed (the empty barrier expects one such arrival from
    // each MMA warp).
    __device__ void release(int st) const
    {
        if (ptx::elect_one())
            ptx::mma_commit(b.empty(st));
        __syncwarp();
    }

    // Split K and V: release the V half of a stage.
    __device__ void release_v(int st) const
    {
        if (ptx::elect_one())
            ptx::mma_commit(b.v_empty(st));
        __syncwarp();
    }

    // S_w = Q_w K^T over D/16 k-steps: K-major operands advance 32 bytes per
    // step inside a 128-byte swizzle row and 16 KB per 64-column box.
    __device__ bool issue_s(int st)
    {
        if (SEP && n_s > 0) {   // the softmax has loaded the previous S_w
            if (!warp_wait(b.s_free(w), (n_s - 1) & 1u, c, kSiteMmaSFree))
                return false;
            ptx::tc_fence_after_sync();
        }
        const uint32_t ka = k_lo + (uint32_t)(st * (C::kStageBytes >> 4));
        if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)((kk / 4) * (C::kBoxBytes >> 4) + (kk % 4) * 2);
                ptx::mma_ss(tS, desc_from_lo(q_cur + off), desc_from_lo(ka + off), kIdescQK, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(b.s_full(w));
        }
        __syncwarp();
        ++n_s;
        return true;
    }

    // O_w (+)= P_w V over 128/16 k-steps: P from TMEM (8 columns per step),
    // V MN-major: 16 key rows = 2 KB per step.
    __device__ bool issue_pv(int st, bool accumulate)
    {
        if (!accumulate) {   // first P.V of a CTA tile overwrites O_w: the epilogue must have read it
            if (n_t > 0 && !warp_wait(b.o_free(w), (n_t - 1) & 1u, c, kSiteMmaOFree))
                return false;
            ++n_t;
        }
        if (!warp_wait(b.p_full(w), n_pv & 1u, c, kSiteMmaPFull))
            return false;
        ptx::tc_fence_after_sync();
        const uint32_t va = v_lo + (uint32_t)(st * (C::kStageBytes >> 4));
        if (ptx::elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
                ptx::mma_ts(tO, tP + kk * 8, desc_from_lo(va + kk * (2048 >> 4)), kIdescPV,
                            (accumulate || kk > 0) ? 1u : 0u);
            ptx::mma_commit(b.o_done(w));
        }
        __syncwarp();
        ++n_pv;
        return true;
    }

    // One CTA tile in the separate-P order: S_w of step j+1 as soon as the
    // softmax has loaded S_w(j), then P.V of step j.  Steps 0..n-1 of the K/V
    // stream, of which Q tile w uses the first nw; every stage is waited for
    // and released by this warp, used or not.  (At D = 128 this order runs
    // only for heads of one Q tile, whose stages are split into K and V.)
    __device__ bool tile(int step0, int n, int nw)
    {
        int st;
        if (!stage_wait(step0, st))
            return false;
        if (nw > 0 && !issue_s(st))
            return false;
        if (C::kSplitKV)
            release(st);   // K_0 read
        for (int j = 0; j < n; ++j) {
            int st_next = st;
            if (j + 1 < n) {
                if (!stage_wait(step0 + j + 1, st_next))
                    return false;
                if (j + 1 < nw && !issue_s(st_next))
                    return false;
                if (C::kSplitKV)
                    release(st_next);   // K_{j+1} read
            }
            if (C::kSplitKV && !v_wait(step0 + j))
                return false;
            if (j < nw && !issue_pv(st, j > 0))
                return false;
            if (C::kSplitKV)
                release_v(st);   // V_j read
            else
                release(st);
            st = st_next;
        }
        return true;
    }
};

// One warp for both Q tiles (D = 128): per step S0_j, P.V1_{j-1}, S1_j, P.V0_j,
// so each softmax warpgroup works while the tensor core runs the other
// tile's MMAs, and P_w(j) overwrites S_w(j) in TMEM before S_w(j+1) is issued.
template <int D, bool BF16>
__device__ bool tile_interleaved(MmaIssuer<D, BF16, false> &m0, MmaIssuer<D, BF16, false> &m1, int step0, int n, int n0,
                                 int n1)
{
    int st, prev = -1;
    for (int j = 0; j < n; ++j) {
        if (!m0.stage_wait(step0 + j, st))
            return false;
        if (j < n0 && !m0.issue_s(st))
            return false;
        if (j >= 1) {
            if (j - 1 < n1 && !m1.issue_pv(prev, j - 1 > 0))
                return false;
            m0.release(prev);   // K_{j-1} and V_{j-1} both read
        }
        if (j < n1 && !m1.issue_s(st))
            return false;
        if (j < n0 && !m0.issue_pv(st, j > 0))
            return false;
        prev = st;
    }
    if (n - 1 < n1 && !m1.issue_pv(prev, n - 1 > 0))
        return false;
    m0.release(prev);
    return true;
}

// SEP: separate-P order (always at D = 64; at D = 128 for heads of one Q
// tile, P_0 in tile 1's S columns), else the two-tile interleaved order.
template <int D, bool BF16, int MASK, bool SPLIT, bool SEP>
__device__ void mma_role(int w, const FwdParams &p, uint32_t sQ, uint32_t sStage, uint32_t tmem, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    auto make = [&](int q) {
        return MmaIssuer<D, BF16, SEP>{q,
                                  desc_lo(sQ + q * C::kTileBytes, 16),
                                  desc_lo(sStage, 16),
                                  desc_lo(sStage + C::kTileBytes, C::kBoxBytes),
                                  tmem + C::col_s(q),
                                  tmem + C::col_o(q),
                                  tmem + C::col_p(q),
                                  b,
                                  c,
                                  0u, 0u, 0u, 0u};
    };
    MmaIssuer<D, BF16, SEP> m = make(w);            // this warp's tile (D = 64) or tile 0 (D = 128)
    MmaIssuer<D, BF16, SEP> m1 = make(1);           // tile 1 when one warp serves both
    if (!C::kSeparateP && SEP)                      // D = 128, heads of one Q tile
        m.tP = tmem + C::col_p_one_tile();
    int step = 0, it = 0;
    PartIter parts;
    parts.init_t<SPLIT>(p.sch, blockIdx.x);
    Part pt;
    while (parts.next_t<SPLIT, MASK == kMaskBand>(p.sch, pt)) {
        int bh, ct;
        sched_decode_t<SPLIT, MASK == kMaskBand>(p.sch, pt.tile, bh, ct);
        const int n0 = part_steps(pt, sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, 0)), n1 = part_steps(pt, sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, 1));
        const int n = pt.ke - pt.kb;
        const int qb = it % C::kQBufs;
        if (!warp_wait(b.q_full(qb), (uint32_t)(it / C::kQBufs) & 1u, c, kSiteMmaQFull))
            break;
        ptx::tc_fence_after_sync();
        m.q_cur = m.q_lo + (uint32_t)(qb * (C::kQBufBytes >> 4));
        m1.q_cur = m1.q_lo + (uint32_t)(qb * (C::kQBufBytes >> 4));
        bool ok;
        if constexpr (SEP)
            ok = m.tile(step, n, w ? n1 : n0);
        else
            ok = tile_interleaved(m, m1, step, n, n0, n1);
        if (!ok)
            break;
        step += n;
        if (ptx::elect_one())   // Q buffer free once this warp's S MMAs of the part completed
            ptx::mma_commit(b.q_empty(qb));
        __syncwarp();
        ++it;
    }
    // Drain: all MMAs this warp issued have completed before TMEM is freed.
    if (ptx::elect_one())
        ptx::mma_commit(b.drain());
    __syncwarp();
    warp_wait(b.drain(), 0u, c, kSiteDrain);
}

// ------------------------------------------------------------------ softmax

// Hide keys i >= hi (0 <= i < 128, hi per thread) of this thread's row of S
// in TMEM, by writing -inf there, before the row is read: the 32-column
// chunks that every row of the warp hides are overwritten whole, and the
// chunks that the warp's rows split are read, masked row by row and written
// back.  Warp-collective (tS is the warp's lane quarter of S).  Out of line
// and rolled, so the softmax loop carries one call instead of a compare and
// select per score; it runs on masked steps only (the causal diagonal, the
// ragged last key tile), and the scores read afterwards are the ones the
// per-score mask would have produced.
static __device__ __noinline__ void mask_s_tail(uint32_t tS, int hi)
{
    hi = hi < 0 ? 0 : (hi > kBN ? kBN : hi);
    const int lo_w = __reduce_min_sync(0xffffffffu, hi), hi_w = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll 1
    for (int c0 = 0; c0 < kBN; c0 += 32) {
        uint32_t x[32];
        if (c0 >= hi_w) {   // hidden in every row of the warp
#pragma unroll
            for (int i = 0; i < 32; ++i)
                x[i] = ninf;
            ptx::tmem_st32(tS + (uint32_t)c0, x);
        } else if (c0 + 32 > lo_w) {   // the warp's rows split this chunk
            ptx::tmem_ld32(tS + (uint32_t)c0, x);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
                x[i] = (c0 + i < hi) ? x[i] : ninf;
            ptx::tmem_st32(tS + (uint32_t)c0, x);
        }
    }
    ptx::tmem_wait_st();
}

// SEP as in mma_role.  At D = 128 its waits record a timeout inline: they
// hold S, P or O rescale registers, which a call made the balanced variant
// spill (1.3 % slower); at D = 64 the inline form measured 1.4 % slower.
template <int D, bool BF16, int MASK, bool SPLIT, bool SEP>
__device__ void softmax_role(const FwdParams &p, uint32_t tmem, Bars<D> b, Ctl c, float2 *handoff)
{
    using C = Cfg<D>;
    constexpr bool CAUSAL = MASK != kMaskNone;
    const int w = threadIdx.x / 128;              // Q tile of this warpgroup
    const int t = threadIdx.x % 128;              // row within the Q tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(t & ~31) << 16;
    const uint32_t tS = tmem + C::col_s(w) + lane_off;
    constexpr bool sep = SEP;                        // P_w apart from S_w: S_w is released once loaded
    const uint32_t tP = tmem + ((SEP && !C::kSeparateP) ? C::col_p_one_tile() : C::col_p(w)) + lane_off;   // (w = 0)
    const uint32_t tO = tmem + C::col_o(w) + lane_off;
    const uint64_t qk2 = ptx::f2_pack(p.qk_scale, p.qk_scale);
    uint32_t s_phase = 0, o_phase = 0, n_st = 0;

    PartIter parts;
    parts.init_t<SPLIT>(p.sch, blockIdx.x);
    Part pt;
    while (parts.next_t<SPLIT, MASK == kMaskBand>(p.sch, pt)) {
        int bh, ct;
        sched_decode_t<SPLIT, MASK == kMaskBand>(p.sch, pt.tile, bh, ct);
        const int nw = sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, w);    // steps of this Q tile in the whole tile
        const int np = part_steps(pt, nw);              // ... of which this part holds steps kb .. kb + np - 1
        if (np == 0)
            continue;
        const int row = ct * kCtaRows + w * kBM + t;                // query index (may be >= N: padding)
        // Masked attention sees a band of keys: this row [row_lo, row_hi); a
        // step needs masking where some row's band edge or the key count ends
        // inside it: past the Q tile's first row's upper edge, before its last
        // row's lower edge (kMaskBand only), or past Nkv.
        const int ks = (MASK == kMaskBand) ? sched_kv_start(p.sch, ct) : 0;   // the tile's first key step
        int row_lo = 0, row_hi = p.Nkv, edge_lo = 0, edge_hi = p.Nkv;
        if (CAUSAL) {
            const int first = ct * kCtaRows + w * kBM, r = min(row, p.N - 1);
            row_hi = sched_row_hi(p.sch, r);
            edge_hi = sched_row_hi(p.sch, first);
            if (MASK == kMaskBand) {
                row_lo = sched_row_lo(p.sch, r);
                edge_lo = sched_row_lo(p.sch, min(first + kBM - 1, p.N - 1));
            }
        }
        float m = -INFINITY, l = 0.f;                               // running max (log2 units), row sum

        // One step of the recurrence; false if a wait gave up.  At D = 64 a
        // masked step without a left band bound has the keys its rows hide
        // set to -inf in TMEM before S is read (mask_s_tail, out of line), so
        // the loop body holds no per-score mask code: the size of the loop
        // body sets how often its instructions are fetched anew (measured:
        // B2 H16 N4096 3-5 % and N16384 3-8 % faster, results bit for bit
        // the same).  At D = 128, where a step carries twice the tensor work,
        // the call measured 1.5 % slower than the per-score code, which it
        // keeps.
        auto step = [&](int jr, int kb0, bool masked) -> bool {
            if (!warp_wait<D == 128>(b.s_full(w), s_phase & 1u, c, kSiteSoftSFull))
                return false;
            ++s_phase;
            ptx::tc_fence_after_sync();
            constexpr bool TMEM_MASK = (D == 64 && MASK != kMaskBand);
            if (TMEM_MASK && masked)
                mask_s_tail(tS, row_hi - kb0);   // keys kb0 + i with i < row_hi - kb0 are visible

            uint32_t r[2][64];
            ptx::tmem_ld64(tS, r[0]);   // the whole row of S_w in two instructions
            ptx::tmem_ld64(tS + 64, r[1]);
            ptx::tmem_wait_ld();
            if (sep) {   // S_w may now be overwritten by the next step's MMA
                ptx::tc_fence_before_sync();
                ptx::mbar_arrive(b.s_free(w));
            }

            float s[128];
#pragma unroll
            for (int i = 0; i < 128; ++i)
                s[i] = __uint_as_float(r[i / 64][i % 64]);

            if (!TMEM_MASK && masked) {
                if (MASK == kMaskBand) {
                    // key kb0 + i is visible iff row_lo <= kb0 + i < row_hi (one unsigned compare)
                    const int lo = row_lo - kb0;
                    const uint32_t width = (uint32_t)(row_hi - row_lo);
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        s[i] = ((uint32_t)(i - lo) < width) ? s[i] : -INFINITY;
                } else {
                    const int hi = row_hi - kb0;   // keys kb0 + i with i < hi are visible
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        s[i] = (i < hi) ? s[i] : -INFINITY;
                }
            }

            float mx[8];   // eight partial maxima: s[0..15] pairwise, then s[16..127] two at a time
#pragma unroll
            for (int k = 0; k < 8; ++k)
                mx[k] = fmaxf(s[2 * k], s[2 * k + 1]);
#pragma unroll
            for (int i = 16; i < 128; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mx[k] = ptx::fmax3(mx[k], s[i + 2 * k], s[i + 2 * k + 1]);
            const float tile_max = ptx::fmax3(ptx::fmax3(mx[0], mx[1], mx[2]), ptx::fmax3(mx[3], mx[4], mx[5]),
                                              fmaxf(mx[6], mx[7])) * p.qk_scale;
            // The reference max m moves only when this tile holds a larger
            // score (always on the first visible tile, where m = -inf);
            // otherwise alpha = 1 and nothing is rescaled.  Any reference
            // gives the same exact result (the recurrence divides by l
            // relative to the same m), so a larger score may also leave m
            // where it is (a guarded lazy rescale):
            //  * the new score exceeds m by at most kLazyMax (log2 units),
            //    so every probability stays at most 2^kLazyMax, and
            //  * the row's sum so far is at least kLazyWeight times that
            //    score's probability, so no single key carries more than
            //    1/kLazyWeight of the row's weight.
            // The second condition guards the precision: the largest
            // probability is then no longer exactly 1, so its 16-bit
            // rounding (relative 2^-8 in bf16) reaches the output, but
            // weighted by at most 1/kLazyWeight.  Rows dominated by one key
            // (large logits) never meet it and rescale exactly.  Most steps
            // of long rows meet both, and a warp none of whose rows moved
            // skips the rescale of O.
            const bool up = tile_max > m;
            const float dlt = tile_max - m;   // (+inf on the first visible tile)
            const bool lazy = up && dlt <= kLazyMax && l >= kLazyWeight * ptx::ex2(dlt);
            const bool move = up && !lazy;
            const float m_new = move ? tile_max : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;   // no visible key yet: shift 0
            const float alpha = move ? ptx::ex2(m - m_use) : 1.f;     // 0 on the first tile (m = -inf)
            const uint64_t negm2 = ptx::f2_pack(-m_use, -m_use);

            // Exponentials into packed 16-bit pairs first (registers only), so
            // they overlap the previous step's P.V, which still reads P_w.
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const uint64_t x = ptx::f2_fma(ptx::f2_pack(s[2 * i], s[2 * i + 1]), qk2, negm2);
                float x0, x1;
                ptx::f2_unpack(x, x0, x1);
                const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                acc[i & 3] = ptx::f2_add(acc[i & 3], ptx::f2_pack(p0, p1));
                pk[i] = BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
            }
            if (sep && jr > 0) {   // P.V of the previous step done: P_w may be overwritten, O_w is final
                if (!warp_wait<D == 128>(b.o_done(w), o_phase & 1u, c, kSiteSoftODone))
                    return false;
                ++o_phase;
                ptx::tc_fence_after_sync();
            }   // (otherwise S_w(j) is issued after P.V_w(j-1), so s_full already implies it)
            ptx::tmem_st64(tP, pk);
            const uint64_t a2 = ptx::f2_add(ptx::f2_add(acc[0], acc[1]), ptx::f2_add(acc[2], acc[3]));
            float a_lo, a_hi;
            ptx::f2_unpack(a2, a_lo, a_hi);
            l = l * alpha + (a_lo + a_hi);
            m = m_new;

            // O_w *= alpha for the rows of this warp, skipped when no row's max
            // moved (ever less likely as more keys have been seen).
            if (jr > 0 && __any_sync(0xffffffffu, move)) {
                const uint64_t al2 = ptx::f2_pack(alpha, alpha);
                uint32_t o[D / 64][64];   // all of O_w's row, 64 columns per instruction, one wait
#pragma unroll
                for (int q = 0; q < D / 64; ++q)
                    ptx::tmem_ld64(tO + q * 64, o[q]);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < D / 64; ++q) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float lo, hi;
                        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[q][2 * i]), __uint_as_float(o[q][2 * i + 1])),
                                                   al2),
                                       lo, hi);
                        o[q][2 * i] = __float_as_uint(lo);
                        o[q][2 * i + 1] = __float_as_uint(hi);
                    }
                    ptx::tmem_st64(tO + q * 64, o[q]);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.p_full(w));
            return true;
        };

        for (int jr = 0; jr < np; ++jr) {
            const int kb0 = (ks + pt.kb + jr) * kBN;   // this step's first key
            // masked where some row's band edge or the key count ends inside the step
            const bool masked = (MASK == kMaskBand) ? (kb0 < edge_lo || kb0 + kBN > edge_hi)   // (edge_hi <= Nkv)
                                                    : ((CAUSAL && kb0 + kBN > edge_hi) || kb0 + kBN > p.Nkv);
            if (!step(jr, kb0, masked))
                return;
        }
        if (sep) {   // account for the last P.V of this tile
            if (!warp_wait<D == 128>(b.o_done(w), o_phase & 1u, c, kSiteSoftODone))
                return;
            ++o_phase;
        }
        // Final row statistics for the epilogue warps (slot reused only once read).
        if (n_st > 0 && !warp_wait<D == 128>(b.st_free(w), (n_st - 1) & 1u, c, kSiteSoftStFree))
            return;
        handoff[w * kBM + t] = make_float2(m, l);
        ++n_st;
        ptx::mbar_arrive(b.st_ready(w));
    }
}

// ------------------------------------------------------------------ epilogue

// Epilogue warps sync among themselves (named barrier 1, 128 threads).
__device__ __forceinline__ void epilogue_sync()
{
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Epilogue warps sync and agree (named barrier 2): true iff `ok` held in every
// thread.  Keeps the warpgroup's decisions to leave uniform, so that no warp
// is left waiting at a barrier that the others have left.
__device__ __forceinline__ bool epilogue_all(bool ok)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

// Wait bounded by time alone (not by the abort flag): for copies in flight
// that must land before the CTA may exit.
__device__ __forceinline__ void wait_landed(uint32_t bar, uint32_t parity, Ctl c, uint32_t site)
{
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
        if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
            record_timeout(c, site);
            return;
        }
    }
}

__device__ __forceinline__ float4 ld_cg_f4(const float *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ float2 ld_cg_f2(const float2 *p)
{
    float2 v;
    asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// Merge the partial results of one Q tile of a split tile: with per-part row
// max m_k and sum l_k (log2 units) and O_k normalised by l_k,
//   M = max_k m_k,  L = sum_k l_k 2^(m_k - M),  O = sum_k (l_k 2^(m_k - M) / L) O_k,
//   LSE = (M + log2 L) ln 2
// -- the same rescaling identity the recurrence uses between K/V tiles
// ("A09 - Advanced Triton & FlashAttention", 3. Deep Dive).  A row may see no
// key in some part (m_k = -inf, l_k = 0: its weight is 0), or in none at all
// (queries against fewer keys, causal): then M = -inf, O = 0 and LSE = -inf.
//
// One warp does all merges, off the path of the warps that read accumulators
// out of TMEM: it takes jobs from the epilogue's queue, brings each part's
// (m, l) into shared memory with one bulk copy, turns them into the weights
// l_k 2^(m_k - M) / L in place (a lane per row) and writes LSE, then streams
// the partial O through kMergeBufs buffers (a chunk: kMergeRows rows of one
// part, in the order row block, part), each lane adding weight x O for 4
// columns of 8 rows of a chunk, and writes O.  Every wait is bounded; on a
// failed wait the copies in flight are let land and the warp stops.
template <int D, bool BF16>
__device__ void merge_role(const FwdParams &p, uint32_t sbuf, uint32_t sml, const MergeJob *jobs, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    constexpr int R = C::kMergeRows;              // 16 or 8 rows per chunk
    constexpr int kTpr = D / 4;                   // lanes per row of a chunk
    constexpr int kPos = R * kTpr / 32;           // positions (4 columns of a row) per lane: 8
    constexpr int kRowStep = 32 / kTpr;           // rows between a lane's positions: 2 or 1
    const int lane = threadIdx.x % 32;
    const int row0 = lane / kTpr, col = (lane % kTpr) * 4;
    uint32_t n_jobs = 0, streamed = 0, ml_uses = 0;   // jobs taken; O chunks and (m, l) copies so far

    for (;;) {
        const int j = (int)(n_jobs % kJobSlots);
        if (!warp_wait(b.job_full(j), (n_jobs / kJobSlots) & 1u, c, kSiteMergeJob))
            return;
        const MergeJob &job = jobs[j];
        const int nparts = job.nparts, nrows = job.nrows;
        if (nparts == 0)
            return;   // stop
        const int nchunks = ((nrows + R - 1) / R) * nparts;
        const int ml_rows = sched_ml_rows(nparts);   // staged rows per part
        const uint32_t first = streamed;
        int i_rb = 0, i_pi = 0, issued = 0;   // next chunk to stream (lane 0)
        auto issue_next = [&]() {
            const uint32_t g = first + (uint32_t)issued, buf = g % kMergeBufs;
            const float *src = reinterpret_cast<const float *>(job.o_addr[i_pi]) + i_rb * R * D;
            ptx::mbar_arrive_expect_tx(b.merge_full((int)buf), kMergeOBytes);
            ptx::bulk_load(sbuf + buf * kMergeOBytes, src, kMergeOBytes, b.merge_full((int)buf));
            if (++i_pi == nparts) {
                i_pi = 0;
                ++i_rb;
            }
            ++issued;
        };
        if (nrows > ml_rows) {   // more parts than the staging holds for this many rows: the planner never does this
            if (lane == 0)
                record_timeout(c, kSiteMergeJob);
            __syncwarp();
            return;
        }
        if (lane == 0) {
            ptx::fence_proxy_async_global();   // the parts' partials, made visible by the counter's acquire
            ptx::mbar_arrive_expect_tx(b.ml_full(), (uint32_t)(nparts * ml_rows * 8));
            for (int k = 0; k < nparts; ++k)
                ptx::bulk_load(sml + k * ml_rows * 8, reinterpret_cast<const void *>(job.ml_addr[k]),
                               (uint32_t)(ml_rows * 8), b.ml_full());
            while (issued < kMergeBufs && issued < nchunks)
                issue_next();
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        bool ok = warp_wait(b.ml_full(), ml_uses & 1u, c, kSiteMerge);
        const bool ml_landed = ok;
        ++ml_uses;
        if (ok) {
            // weights in place of m; a lane per row
            for (int r = lane; r < ml_rows; r += 32) {
                float M = -INFINITY;
                for (int k = 0; k < nparts; ++k)
                    M = fmaxf(M, ptx::ld_shared_f32(sml + (k * ml_rows + r) * 8));
                const float Mu = (M == -INFINITY) ? 0.f : M;   // no key seen at all: every weight is 0
                float L = 0.f;
                for (int k = 0; k < nparts; ++k) {
                    const uint32_t a = sml + (k * ml_rows + r) * 8;
                    const float e = ptx::ld_shared_f32(a + 4) * ptx::ex2(ptx::ld_shared_f32(a) - Mu);
                    ptx::st_shared_f32(a, e);
                    L += e;
                }
                const float inv_L = (L > 0.f) ? 1.f / L : 0.f;
                for (int k = 0; k < nparts; ++k) {
                    const uint32_t a = sml + (k * ml_rows + r) * 8;
                    ptx::st_shared_f32(a, ptx::ld_shared_f32(a) * inv_L);
                }
                if (r < nrows)
                    p.LSE[job.orow0 + r] = (M + log2f(L)) * kLn2;
            }
            __syncwarp();
        }
        uint64_t acc[kPos][2];
        int k = 0, rb = 0, pi = 0;
        for (; ok && k < nchunks; ++k) {
            const uint32_t g = first + (uint32_t)k, buf = g % kMergeBufs;
            ok = warp_wait(b.merge_full((int)buf), (g / kMergeBufs) & 1u, c, kSiteMerge);
            if (!ok)
                break;
            if (pi == 0) {
#pragma unroll
                for (int q = 0; q < kPos; ++q)
                    acc[q][0] = acc[q][1] = 0ull;
            }
            const uint32_t so = sbuf + buf * kMergeOBytes + (uint32_t)(row0 * D + col) * 4;
            const uint32_t sw = sml + (uint32_t)(pi * ml_rows + rb * R + row0) * 8;
#pragma unroll
            for (int q = 0; q < kPos; ++q) {
                const float wt = ptx::ld_shared_f32(sw + q * kRowStep * 8);
                const float4 o = ptx::ld_shared_v4f32(so + q * kRowStep * D * 4);
                const uint64_t w2 = ptx::f2_pack(wt, wt);
                acc[q][0] = ptx::f2_fma(ptx::f2_pack(o.x, o.y), w2, acc[q][0]);
                acc[q][1] = ptx::f2_fma(ptx::f2_pack(o.z, o.w), w2, acc[q][1]);
            }
            __syncwarp();   // every lane is done with this buffer
            if (lane == 0 && issued < nchunks)
                issue_next();   // into the buffer just read
            issued = __shfl_sync(0xffffffffu, issued, 0);
            if (pi == nparts - 1) {
                const int r0 = rb * R + row0;
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.O) + ((size_t)(job.orow0 + r0) * D + col) * 2;
#pragma unroll
                for (int q = 0; q < kPos; ++q) {
                    if (r0 + q * kRowStep >= nrows)
                        continue;
                    float x0, x1, x2, x3;
                    ptx::f2_unpack(acc[q][0], x0, x1);
                    ptx::f2_unpack(acc[q][1], x2, x3);
                    const uint32_t lo = BF16 ? ptx::pack_bf16x2(x0, x1) : ptx::pack_f16x2(x0, x1);
                    const uint32_t hi = BF16 ? ptx::pack_bf16x2(x2, x3) : ptx::pack_f16x2(x2, x3);
                    *reinterpret_cast<uint2 *>(dst + (size_t)q * kRowStep * D * 2) = make_uint2(lo, hi);
                }
            }
            if (++pi == nparts) {
                pi = 0;
                ++rb;
            }
        }
        streamed = first + (uint32_t)issued;
        if (!ok) {   // let every copy in flight land before the CTA may exit
            if (lane == 0) {
                if (!ml_landed)
                    wait_landed(b.ml_full(), (ml_uses - 1) & 1u, c, kSiteMergeTail);
                for (int q = k; q < issued; ++q)
                    wait_landed(b.merge_full((int)((first + q) % kMergeBufs)), ((first + q) / kMergeBufs) & 1u, c,
                                kSiteMergeTail);
            }
            __syncwarp();
            return;
        }
        if (lane == 0) {
            p.counters[job.counter] = 0;   // ready for the next launch
            ptx::mbar_arrive(b.job_empty(j));
        }
        __syncwarp();
        ++n_jobs;
    }
}

// Per finished part: for each Q tile, read O_w out of TMEM, then release it
// to the next part's first P.V.  A part that holds all of its Q tile's steps
// writes O = acc / l in the input type and LSE = (m + log2 l) ln 2; a part of
// a split tile writes its partial result to its workspace slot, and the part
// that finishes last hands the merge of that Q tile to the merge warp.
template <int D, bool BF16, int MASK, bool SPLIT>
__device__ void epilogue_role(const FwdParams &p, uint32_t tmem, Bars<D> b, Ctl c, uint32_t s_handoff, uint32_t s_flag,
                              uint32_t s_jobs)
{
    using C = Cfg<D>;
    const int t = threadIdx.x % 128;              // row within a Q tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(t & ~31) << 16;
    // Phase bits: bit w = parity of the st_ready(w) completions taken, bit
    // 2 + w = parity of the P.V products of Q tile w done (o_done(w)).
    uint32_t ph = 0;
    uint32_t n_jobs = 0;                          // merge jobs posted

    // Post a job in the next queue slot: nparts = 0 stops the merge warp.
    // Thread k fills part k; false if the wait for a free slot gave up.
    auto post = [&](int nparts, long long orow0, int nrows, int counter, int tile_ts, int n, int nw, int w, int clo,
                    int chi) -> bool {
        const int j = (int)(n_jobs % kJobSlots);
        if (!epilogue_all(warp_wait(b.job_empty(j), ((n_jobs / kJobSlots) & 1u) ^ 1u, c, kSiteEpiJobFree)))
            return false;
        const uint32_t job = s_jobs + j * (uint32_t)sizeof(MergeJob);
        if (t == 0) {
            ptx::st_shared_u64(job + offsetof(MergeJob, orow0), (uint64_t)orow0);
            ptx::st_shared_u32(job + offsetof(MergeJob, nrows), (uint32_t)nrows);
            ptx::st_shared_u32(job + offsetof(MergeJob, nparts), (uint32_t)nparts);
            ptx::st_shared_u32(job + offsetof(MergeJob, counter), (uint32_t)counter);
        }
        int k = 0, slot;
        for (int cc = clo; cc <= chi && nparts > 0; ++cc)
            if (sched_part_slot(p.sch, tile_ts, n, nw, cc, slot)) {
                if (t == k && k < kMaxMergeParts) {
                    const size_t srow = (size_t)slot * kCtaRows + w * kBM;
                    ptx::st_shared_u64(job + offsetof(MergeJob, o_addr) + 8 * k, reinterpret_cast<uint64_t>(p.part_o + srow * D));
                    ptx::st_shared_u64(job + offsetof(MergeJob, ml_addr) + 8 * k, reinterpret_cast<uint64_t>(p.part_ml + srow));
                }
                ++k;
            }
        epilogue_sync();   // the job is complete before it is handed over
        if (t == 0)
            ptx::mbar_arrive(b.job_full(j));
        ++n_jobs;
        return true;
    };

    PartIter parts;
    parts.init_t<SPLIT>(p.sch, blockIdx.x);
    Part pt;
    while (parts.next_t<SPLIT, MASK == kMaskBand>(p.sch, pt)) {
        int bh, ct;
        sched_decode_t<SPLIT, MASK == kMaskBand>(p.sch, pt.tile, bh, ct);
        uint32_t published = 0;                   // bit w: Q tile w wrote a partial result
#pragma unroll
        for (int w = 0; w < kQTiles; ++w) {
            const int nw = sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, w);
            const int np = part_steps(pt, nw);
            if (np == 0)
                continue;
            // (the whole-tile variant has no warpgroup barrier to keep in step,
            // so each warp may leave on its own)
            bool ok = warp_wait(b.st_ready(w), (ph >> w) & 1u, c, kSiteEpiStReady);
            if (!(SPLIT ? epilogue_all(ok) : ok))
                return;
            ph ^= 1u << w;
            const float2 st = ptx::ld_shared_v2f32(s_handoff + (w * kBM + t) * 8);
            ptx::mbar_arrive(b.st_free(w));
            ph ^= ((uint32_t)np & 1u) << (2 + w);   // the part's last P.V completes phase (done so far - 1) of o_done(w)
            ok = warp_wait(b.o_done(w), ((ph >> (2 + w)) & 1u) ^ 1u, c, kSiteEpiODone);
            if (!(SPLIT ? epilogue_all(ok) : ok))
                return;
            ptx::tc_fence_after_sync();
            const bool whole = !SPLIT || (pt.kb == 0 && pt.ke >= nw);   // no other part holds steps of this Q tile
            const float inv_l = (st.y > 0.f) ? 1.f / st.y : 0.f;   // a row that saw no key: O = 0
            const uint64_t il2 = ptx::f2_pack(inv_l, inv_l);
            const int row = ct * kCtaRows + w * kBM + t;
            const bool valid = row < p.N;
            const uint32_t tO = tmem + C::col_o(w) + lane_off;
            if (whole) {
                uint8_t *orow =
                    reinterpret_cast<uint8_t *>(p.O) + ((size_t)bh * p.N + (size_t)(valid ? row : 0)) * D * 2;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + q * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {   // packed in place: o[i] = columns 2i, 2i + 1
                        float x, y;
                        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2),
                                       x, y);
                        o[i] = BF16 ? ptx::pack_bf16x2(x, y) : ptx::pack_f16x2(x, y);
                    }
                    if (valid) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            ptx::st_global_v4(orow + q * 64 + v * 16, o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                    }
                }
                if (valid)
                    p.LSE[(size_t)bh * p.N + row] = (st.x + log2f(st.y)) * kLn2;
            } else {   // a part of a split tile: the partial result of the valid rows (the merge reads no other)
                float *prow = p.part_o + ((size_t)pt.slot * kCtaRows + w * kBM + t) * D;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + q * 32, o);   // (warp-collective: every lane loads)
                    ptx::tmem_wait_ld();
                    if (!valid)
                        continue;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float x0, x1, x2, x3;
                        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1])), il2),
                                       x0, x1);
                        ptx::f2_unpack(ptx::f2_mul(ptx::f2_pack(__uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3])), il2),
                                       x2, x3);
                        ptx::st_global_v4(prow + q * 32 + 4 * u, __float_as_uint(x0), __float_as_uint(x1),
                                          __float_as_uint(x2), __float_as_uint(x3));
                    }
                }
                if (valid)
                    p.part_ml[(size_t)pt.slot * kCtaRows + w * kBM + t] = st;
                published |= 1u << w;
            }
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.o_free(w));
        }
        if (!SPLIT || published == 0)
            continue;
        // Split tile: make this part's partials visible, count it in, and
        // hand over the merge of each Q tile for which it is the last part to
        // finish.  The tile's parts are held by this CTA and its neighbours.
        const int n = sched_steps(p.sch, pt.tile);
        int clo, chi;
        sched_tile_ctas_near(p.sch, pt.ts, n, blockIdx.x, clo, chi);
        __threadfence();
        epilogue_sync();
        if (t == 0) {
            int last = 0;
            for (int w = 0; w < kQTiles; ++w) {
                if (!(published >> w & 1u))
                    continue;
                const int nw = sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, w);
                int expected = 0, slot;
                for (int cc = clo; cc <= chi; ++cc)
                    expected += sched_part_slot(p.sch, pt.ts, n, nw, cc, slot) ? 1 : 0;
                const int done = atomicAdd(&p.counters[2 * pt.tile + w], 1) + 1;
                if (done == expected)
                    last |= 1 << w;
            }
            if (last)
                __threadfence();   // acquire: the other parts' partials are visible to this CTA
            ptx::st_shared_u32(s_flag, (uint32_t)last);
        }
        epilogue_sync();
        const int last = (int)ptx::ld_shared_u32(s_flag);
        epilogue_sync();   // every thread has read the flag before it is reused
#pragma unroll 1
        for (int w = 0; w < kQTiles; ++w) {
            if (!(last >> w & 1))
                continue;
            const int nw = sched_kv_tiles_t<MASK == kMaskBand>(p.sch, ct, w);
            int nparts = 0, slot;
            for (int cc = clo; cc <= chi; ++cc)
                nparts += sched_part_slot(p.sch, pt.ts, n, nw, cc, slot) ? 1 : 0;
            const int r_base = ct * kCtaRows + w * kBM;
            if (!post(nparts < kMaxMergeParts ? nparts : kMaxMergeParts, (long long)bh * p.N + r_base,
                      (p.N - r_base < kBM) ? p.N - r_base : kBM, 2 * pt.tile + w, pt.ts, n, nw, w, clo, chi))
                return;
        }
    }
    if (SPLIT)
        post(0, 0, 0, 0, 0, 0, 0, 0, 0, -1);   // stop the merge warp
}

// ------------------------------------------------------------------ kernel

template <int D, bool BF16, int MASK, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p)
{
    using C = Cfg<D>;
    constexpr bool CAUSAL = MASK != kMaskNone;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;    // 128-byte swizzle atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kQOff;
    const uint32_t sStage = base + C::kStageOff;
    Bars<D> b{base + C::kBarOff, base + (uint32_t)C::vbar_off(SPLIT)};
    float2 *handoff = reinterpret_cast<float2 *>(base_ptr + C::kHandOff);
    uint32_t *misc = reinterpret_cast<uint32_t *>(base_ptr + C::kMiscOff);
    Ctl c{reinterpret_cast<volatile int *>(misc + 1)};

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int wg = warp / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(b.full(s), 1);
            ptx::mbar_init(b.empty(s), C::kMmaWarps);
            if (C::kSplitKV) {
                ptx::mbar_init(b.v_full(s), 1);
                ptx::mbar_init(b.v_empty(s), C::kMmaWarps);
            }
        }
        for (int qb = 0; qb < C::kQBufs; ++qb) {
            ptx::mbar_init(b.q_full(qb), 1);
            ptx::mbar_init(b.q_empty(qb), C::kMmaWarps);
        }
        for (int w = 0; w < kQTiles; ++w) {
            ptx::mbar_init(b.s_full(w), 1);
            ptx::mbar_init(b.s_free(w), kBM);
            ptx::mbar_init(b.p_full(w), kBM);
            ptx::mbar_init(b.o_done(w), 1);
            ptx::mbar_init(b.st_ready(w), kBM);
            ptx::mbar_init(b.st_free(w), kBM);
            ptx::mbar_init(b.o_free(w), kBM);
        }
        ptx::mbar_init(b.drain(), C::kMmaWarps);
        for (int i = 0; SPLIT && i < kMergeBufs; ++i)
            ptx::mbar_init(b.merge_full(i), 1);
        if (SPLIT)
            ptx::mbar_init(b.ml_full(), 1);
        for (int j = 0; SPLIT && j < kJobSlots; ++j) {
            ptx::mbar_init(b.job_full(j), 1);
            ptx::mbar_init(b.job_empty(j), 1);
        }
        *c.abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(misc), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmV);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(misc);

    if (wg < kEpilogueWarpgroup) {
        ptx::regs_increase<kRegsSoftmax>();
        if constexpr (C::kSeparateP)
            softmax_role<D, BF16, MASK, SPLIT, true>(p, tmem, b, c, handoff);
        else if (separate_p<D>(p))
            softmax_role<D, BF16, MASK, SPLIT, true>(p, tmem, b, c, handoff);
        else
            softmax_role<D, BF16, MASK, SPLIT, false>(p, tmem, b, c, handoff);
    } else if (wg == kEpilogueWarpgroup) {
        ptx::regs_decrease<kRegsEpilogue>();
        epilogue_role<D, BF16, MASK, SPLIT>(p, tmem, b, c, base + C::kHandOff, base + C::kMiscOff + 8, base + C::kJobOff);
    } else {
        ptx::regs_decrease<kRegsProducer>();
        if (warp == kLoadWarp) {
            if constexpr (!C::kSplitKV)
                load_role<D, MASK, SPLIT, false>(&tmQ, &tmK, &tmV, p, sQ, sStage, b, c);
            else if (split_kv<D>(p))
                load_role<D, MASK, SPLIT, true>(&tmQ, &tmK, &tmV, p, sQ, sStage, b, c);
            else
                load_role<D, MASK, SPLIT, false>(&tmQ, &tmK, &tmV, p, sQ, sStage, b, c);
        }
        else if (warp < kMmaWarp + C::kMmaWarps) {
            if constexpr (C::kSeparateP)
                mma_role<D, BF16, MASK, SPLIT, true>(warp - kMmaWarp, p, sQ, sStage, tmem, b, c);
            else if (separate_p<D>(p))
                mma_role<D, BF16, MASK, SPLIT, true>(warp - kMmaWarp, p, sQ, sStage, tmem, b, c);
            else
                mma_role<D, BF16, MASK, SPLIT, false>(warp - kMmaWarp, p, sQ, sStage, tmem, b, c);
        }
        else if (SPLIT && warp == kMergeWarp)
            merge_role<D, BF16>(p, base + C::kMergeOff, base + C::kMlOff,
                                reinterpret_cast<const MergeJob *>(base_ptr + C::kJobOff), b, c);
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace fa
