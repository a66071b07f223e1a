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
// Warp roles (320 threads):
//   warps 0-3  softmax/correction/epilogue for Q tile 0 (one thread per row)
//   warps 4-7  the same for Q tile 1
//   warp  8    TMA producer: Q tiles, then K_j, V_j into a ring of smem slots
//   warp  9    tcgen05 MMA issuer (one thread) and TMEM owner
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [256+D,256+2D)
//   P_w (16-bit, two per column) overwrites columns [0,64) of S_w once the
//   softmax warps have read S_w, and feeds the P.V MMA as its TMEM A operand.
//
// MMA issue order per K/V step j (w = Q tile):
//   S0_j = Q0 K_j^T,  O1 += P1_{j-1} V_{j-1},  S1_j = Q1 K_j^T,  O0 += P0_j V_j
// so each softmax warpgroup has two MMAs' worth of time to turn S into P.
// tcgen05 MMAs from one thread execute in issue order, so S_w of step j+1 may
// be issued right after the MMA that reads P_w of step j.
//
// Softmax follows the exp2 form ("How to profile and optimise kernels", exp2):
// qk_scale = scale*log2(e) is folded once, the row max is taken on raw scores
// and then scaled (valid because scale > 0), m is kept in log2 units, and
// LSE = (m + log2 l) * ln 2.  P is rounded to the input type for the P.V MMA;
// l is summed from the fp32 P (the P cast section of the same page).
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
#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {

// Device status word: 0 = fine; otherwise 1 | (site << 8) of the first wait
// that expired.  Read and cleared by fa_sync_status().
__device__ unsigned int g_status_word;

constexpr int kBM = 128;        // query rows per Q tile (one TMEM lane each)
constexpr int kBN = 128;        // keys per K/V tile
constexpr int kQTiles = 2;      // Q tiles per CTA tile
constexpr int kCtaRows = kBM * kQTiles;
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr float kLn2 = 0.69314718055994530942f;

// Wait sites recorded in the status word.
enum : uint32_t {
    kSiteLoadQEmpty = 1, kSiteLoadSlotEmpty, kSiteMmaQFull, kSiteMmaSlotFull, kSiteMmaPFull,
    kSiteSoftSFull, kSiteSoftODone, kSiteDrain, kSiteTail
};

template <int D>
struct Cfg {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    static constexpr int kBoxes = D / 64;              // 128-byte-wide TMA boxes per tile row
    static constexpr int kBoxBytes = kBM * 128;        // one [128 rows, 64 cols] 16-bit box
    static constexpr int kTileBytes = kBM * D * 2;     // one [128, D] 16-bit tile
    static constexpr int kSlots = (D == 64) ? 8 : 4;   // K/V ring depth (K and V tiles alternate)
    static constexpr int kQOff = 0;
    static constexpr int kSlotOff = kQTiles * kTileBytes;
    static constexpr int kBarOff = kSlotOff + kSlots * kTileBytes;
    // full[kSlots], empty[kSlots], q_full, q_empty, s_full[2], p_full[2], o_done[2], drain
    static constexpr int kNumBars = 2 * kSlots + 9;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;   // + slack to align the base to 1024
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

struct FwdParams {
    void *O;
    float *LSE;
    int N;
    int BH;
    int ctiles_per_bh;   // ceil(N / 256)
    int total_tiles;     // BH * ctiles_per_bh
    float qk_scale;      // scale * log2(e)
};

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

template <bool CAUSAL>
__device__ __forceinline__ void decode_tile(int t, const FwdParams &p, int &bh, int &ct)
{
    if (CAUSAL) {   // longest first, heads interleaved
        ct = p.ctiles_per_bh - 1 - t / p.BH;
        bh = t % p.BH;
    } else {        // head-major: neighbouring CTAs share a head's K/V in L2
        bh = t / p.ctiles_per_bh;
        ct = t % p.ctiles_per_bh;
    }
}

// K/V tiles visited by Q tile w of CTA tile ct; 0 if it holds no valid row.
template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles(int ct, int w, int N)
{
    const int r0 = ct * kCtaRows + w * kBM;
    if (r0 >= N)
        return 0;
    if (!CAUSAL)
        return (N + kBN - 1) / kBN;
    const int last = min(r0 + kBM - 1, N - 1);
    return last / kBN + 1;
}

struct Ctl {
    volatile int *abort_flag;
};

__device__ __noinline__ void record_timeout(Ctl c, uint32_t site)
{
    *c.abort_flag = 1;
    atomicCAS(&g_status_word, 0u, 1u | (site << 8));
}

// Bounded wait by one thread; false if it gave up (timeout or abort).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, Ctl c, uint32_t site)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((spin & 63u) == 0) {
            if (*c.abort_flag)
                return false;
            if (ptx::global_timer_ns() - t0 > kWaitLimitNs) {
                record_timeout(c, site);
                return false;
            }
        }
    }
}

// Bounded wait by a whole warp; the outcome is warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, Ctl c, uint32_t site)
{
    const bool ok = wait_bounded(bar, parity, c, site);
    return __all_sync(0xffffffffu, ok);
}

template <int D>
struct Bars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (Cfg<D>::kSlots + s); }
    __device__ uint32_t q_full() const { return base + 8u * (2 * Cfg<D>::kSlots); }
    __device__ uint32_t q_empty() const { return q_full() + 8u; }
    __device__ uint32_t s_full(int w) const { return q_full() + 16u + 8u * w; }
    __device__ uint32_t p_full(int w) const { return q_full() + 32u + 8u * w; }
    __device__ uint32_t o_done(int w) const { return q_full() + 48u + 8u * w; }
    __device__ uint32_t drain() const { return q_full() + 64u; }
};

// ------------------------------------------------------------------ producer

template <int D, bool CAUSAL>
__device__ void load_role(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                          const FwdParams &p, uint32_t sQ, uint32_t sSlot, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    int item = 0;   // K/V tiles issued so far (K_0, V_0, K_1, ...)
    int it = 0;     // CTA tiles started by this CTA
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
        int bh, ct;
        decode_tile<CAUSAL>(t, p, bh, ct);
        const int n = max(kv_tiles<CAUSAL>(ct, 0, p.N), kv_tiles<CAUSAL>(ct, 1, p.N));
        if (!wait_bounded(b.q_empty(), (it & 1) ^ 1, c, kSiteLoadQEmpty)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(b.q_full(), kQTiles * C::kTileBytes);
        for (int w = 0; w < kQTiles; ++w)
            for (int x = 0; x < C::kBoxes; ++x)
                ptx::tma_load_3d(sQ + w * C::kTileBytes + x * C::kBoxBytes, tmQ, b.q_full(), x * 64,
                                 ct * kCtaRows + w * kBM, bh);
        for (int j = 0; ok && j < n; ++j) {
            for (int kv = 0; kv < 2; ++kv) {
                const int slot = item % C::kSlots;
                const uint32_t use = (uint32_t)(item / C::kSlots);
                if (!wait_bounded(b.empty(slot), (use & 1u) ^ 1u, c, kSiteLoadSlotEmpty)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(b.full(slot), C::kTileBytes);
                const CUtensorMap *tm = kv ? tmV : tmK;
                for (int x = 0; x < C::kBoxes; ++x)
                    ptx::tma_load_3d(sSlot + slot * C::kTileBytes + x * C::kBoxBytes, tm, b.full(slot), x * 64,
                                     j * kBN, bh);
                ++item;
            }
        }
    }
    // Tail: every copy this thread issued has landed and (unless aborting)
    // every slot and the Q buffer have been released by the MMA warp, so no
    // asynchronous write or arrive targets this CTA's shared memory after exit.
    for (int s = 0; s < C::kSlots && s < item; ++s) {
        const int last = item - 1 - ((item - 1 - s) % C::kSlots);   // last item that used slot s
        const uint32_t use = (uint32_t)(last / C::kSlots);
        wait_bounded(b.full(s), use & 1u, c, kSiteTail);
        if (!*c.abort_flag)
            wait_bounded(b.empty(s), use & 1u, c, kSiteTail);
    }
    if (it > 0) {
        wait_bounded(b.q_full(), (uint32_t)((it - 1) & 1), c, kSiteTail);
        if (!*c.abort_flag)
            wait_bounded(b.q_empty(), (uint32_t)((it - 1) & 1), c, kSiteTail);
    }
}

// ------------------------------------------------------------------ MMA issuer

template <int D, bool BF16, bool CAUSAL>
__device__ void mma_role(const FwdParams &p, uint32_t sQ, uint32_t sSlot, uint32_t tmem, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    constexpr uint32_t kIdescQK = instr_desc_f16(BF16, kBM, kBN, false);   // S = Q K^T, both K-major
    constexpr uint32_t kIdescPV = instr_desc_f16(BF16, kBM, D, true);      // O += P V, V is MN-major
    const uint32_t tS[2] = {tmem + C::kColS0, tmem + C::kColS1};
    const uint32_t tO[2] = {tmem + C::kColO0, tmem + C::kColO1};
    uint32_t p_phase[2] = {0u, 0u};
    int item = 0, it = 0;
    bool ok = true;

    // S_w = Q_w K^T over D/16 k-steps; K-major operands advance 32 bytes per
    // step inside a 128-byte swizzle row, and 16 KB per 64-column box.
    auto issue_s = [&](int w, int kslot) {
        const uint32_t qa = sQ + w * C::kTileBytes;
        const uint32_t ka = sSlot + kslot * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::kBoxBytes + (kk % 4) * 32;
            ptx::mma_ss(tS[w], smem_desc_sw128(qa + off, 16), smem_desc_sw128(ka + off, 16), kIdescQK,
                        kk > 0 ? 1u : 0u);
        }
    };
    // O_w (+)= P_w V over 128/16 k-steps; P from TMEM (8 columns per step),
    // V MN-major: 16 key rows = 2 KB per step, 64-column boxes 16 KB apart.
    auto issue_pv = [&](int w, int vslot, bool accumulate) {
        const uint32_t va = sSlot + vslot * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
            ptx::mma_ts(tO[w], tS[w] + kk * 8, smem_desc_sw128(va + kk * 2048, C::kBoxBytes), kIdescPV,
                        (accumulate || kk > 0) ? 1u : 0u);
    };

    for (int t = blockIdx.x; ok && t < p.total_tiles; t += gridDim.x, ++it) {
        int bh, ct;
        decode_tile<CAUSAL>(t, p, bh, ct);
        const int n0 = kv_tiles<CAUSAL>(ct, 0, p.N), n1 = kv_tiles<CAUSAL>(ct, 1, p.N);
        const int n = max(n0, n1);
        if (!wait_bounded(b.q_full(), (uint32_t)(it & 1), c, kSiteMmaQFull)) { ok = false; break; }
        ptx::tc_fence_after_sync();
        int vprev = -1;
        for (int j = 0; j < n; ++j) {
            const int kslot = item % C::kSlots;
            if (!wait_bounded(b.full(kslot), (uint32_t)(item / C::kSlots) & 1u, c, kSiteMmaSlotFull)) { ok = false; break; }
            ptx::tc_fence_after_sync();
            ++item;
            if (j < n0) {
                issue_s(0, kslot);
                ptx::mma_commit(b.s_full(0));
            }
            if (j >= 1) {
                if (j - 1 < n1) {
                    if (!wait_bounded(b.p_full(1), p_phase[1] & 1u, c, kSiteMmaPFull)) { ok = false; break; }
                    ++p_phase[1];
                    ptx::tc_fence_after_sync();
                    issue_pv(1, vprev, j - 1 > 0);
                    ptx::mma_commit(b.o_done(1));
                }
                ptx::mma_commit(b.empty(vprev));   // V_{j-1} read by both P.V MMAs
            }
            if (j < n1) {
                issue_s(1, kslot);
                ptx::mma_commit(b.s_full(1));
            }
            ptx::mma_commit(b.empty(kslot));       // K_j read by both S MMAs
            const int vslot = item % C::kSlots;
            if (!wait_bounded(b.full(vslot), (uint32_t)(item / C::kSlots) & 1u, c, kSiteMmaSlotFull)) { ok = false; break; }
            ptx::tc_fence_after_sync();
            ++item;
            if (j < n0) {
                if (!wait_bounded(b.p_full(0), p_phase[0] & 1u, c, kSiteMmaPFull)) { ok = false; break; }
                ++p_phase[0];
                ptx::tc_fence_after_sync();
                issue_pv(0, vslot, j > 0);
                ptx::mma_commit(b.o_done(0));
            }
            vprev = vslot;
        }
        if (!ok)
            break;
        if (n - 1 < n1) {
            if (!wait_bounded(b.p_full(1), p_phase[1] & 1u, c, kSiteMmaPFull)) { ok = false; break; }
            ++p_phase[1];
            ptx::tc_fence_after_sync();
            issue_pv(1, vprev, n - 1 > 0);
            ptx::mma_commit(b.o_done(1));
        }
        ptx::mma_commit(b.empty(vprev));
        ptx::mma_commit(b.q_empty());
    }
    // Drain: all MMAs this thread issued have completed before TMEM is freed.
    ptx::mma_commit(b.drain());
    wait_bounded(b.drain(), 0u, c, kSiteDrain);
}

// ------------------------------------------------------------------ softmax

template <int D, bool BF16, bool CAUSAL>
__device__ void softmax_role(const FwdParams &p, uint32_t tmem, Bars<D> b, Ctl c)
{
    using C = Cfg<D>;
    const int w = threadIdx.x / 128;              // Q tile of this warpgroup
    const int wq = (threadIdx.x / 32) % 4;        // warp within the warpgroup: TMEM lanes 32*wq..
    const int lane = threadIdx.x % 32;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + (w ? C::kColS1 : C::kColS0) + lane_off;
    const uint32_t tO = tmem + (w ? C::kColO1 : C::kColO0) + lane_off;
    const float qk = p.qk_scale;
    uint32_t s_phase = 0, o_phase = 0;

    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        int bh, ct;
        decode_tile<CAUSAL>(t, p, bh, ct);
        const int nw = kv_tiles<CAUSAL>(ct, w, p.N);
        if (nw == 0)
            continue;
        const int row = ct * kCtaRows + w * kBM + wq * 32 + lane;   // query index (may be >= N: padding)
        const int row_limit = CAUSAL ? min(p.N, row + 1) : p.N;     // keys < row_limit are visible
        float m = -INFINITY, l = 0.f;

        for (int j = 0; j < nw; ++j) {
            if (!warp_wait(b.s_full(w), s_phase & 1u, c, kSiteSoftSFull))
                return;
            ++s_phase;
            ptx::tc_fence_after_sync();

            uint32_t r[4][32];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                ptx::tmem_ld32(tS + q * 32, r[q]);
            ptx::tmem_wait_ld();

            float s[128];
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    s[q * 32 + i] = __uint_as_float(r[q][i]);

            if ((CAUSAL && j == nw - 1) || (j + 1) * kBN > p.N) {
                const int lim = row_limit - j * kBN;
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    s[i] = (i < lim) ? s[i] : -INFINITY;
            }

            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mx[i] = s[i];
#pragma unroll
            for (int i = 8; i < 128; ++i)
                mx[i & 7] = fmaxf(mx[i & 7], s[i]);
            const float tile_max = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                         fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float m_new = fmaxf(m, tile_max * qk);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ptx::ex2(m - m_use);      // 0 on the first tile (m = -inf)
            const float neg_m = -m_use;

            float sum[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                sum[i] = 0.f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = ptx::ex2(fmaf(s[h * 64 + 2 * i], qk, neg_m));
                    const float p1 = ptx::ex2(fmaf(s[h * 64 + 2 * i + 1], qk, neg_m));
                    sum[i & 7] += p0 + p1;
                    pk[i] = BF16 ? ptx::pack_bf16x2(p0, p1) : ptx::pack_f16x2(p0, p1);
                }
                ptx::tmem_st32(tS + h * 32, pk);
            }
            const float rowsum = ((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]));
            l = l * alpha + rowsum;
            m = m_new;

            if (j > 0) {   // rescale O_w (after P.V of step j-1 completed)
                if (!warp_wait(b.o_done(w), o_phase & 1u, c, kSiteSoftODone))
                    return;
                ++o_phase;
                ptx::tc_fence_after_sync();
                if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + q * 32, o);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        ptx::tmem_st32(tO + q * 32, o);
                    }
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(b.p_full(w));
        }

        // Epilogue: O = acc / l in the input type, LSE = (m + log2 l) ln 2.
        if (!warp_wait(b.o_done(w), o_phase & 1u, c, kSiteSoftODone))
            return;
        ++o_phase;
        ptx::tc_fence_after_sync();
        const float inv_l = 1.f / l;
        const bool valid = row < p.N;
        uint8_t *orow = reinterpret_cast<uint8_t *>(p.O) + ((size_t)bh * p.N + (size_t)(valid ? row : 0)) * D * 2;
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + q * 32, o);
            ptx::tmem_wait_ld();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float a = __uint_as_float(o[2 * i]) * inv_l;
                const float z = __uint_as_float(o[2 * i + 1]) * inv_l;
                pk[i] = BF16 ? ptx::pack_bf16x2(a, z) : ptx::pack_f16x2(a, z);
            }
            if (valid) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    ptx::st_global_v4(orow + q * 64 + v * 16, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
        }
        if (valid)
            p.LSE[(size_t)bh * p.N + row] = (m + log2f(l)) * kLn2;
        ptx::tc_fence_before_sync();
    }
}

// ------------------------------------------------------------------ kernel

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const FwdParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;    // 128-byte swizzle atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kQOff;
    const uint32_t sSlot = base + C::kSlotOff;
    Bars<D> b{base + C::kBarOff};
    uint32_t *misc = reinterpret_cast<uint32_t *>(base_ptr + C::kMiscOff);
    Ctl c{reinterpret_cast<volatile int *>(misc + 1)};

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(b.full(s), 1);
            ptx::mbar_init(b.empty(s), 1);
        }
        ptx::mbar_init(b.q_full(), 1);
        ptx::mbar_init(b.q_empty(), 1);
        for (int w = 0; w < kQTiles; ++w) {
            ptx::mbar_init(b.s_full(w), 1);
            ptx::mbar_init(b.p_full(w), kBM);
            ptx::mbar_init(b.o_done(w), 1);
        }
        ptx::mbar_init(b.drain(), 1);
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

    if (warp < kLoadWarp) {
        softmax_role<D, BF16, CAUSAL>(p, tmem, b, c);
    } else if (warp == kLoadWarp) {
        if (lane == 0)
            load_role<D, CAUSAL>(&tmQ, &tmK, &tmV, p, sQ, sSlot, b, c);
        __syncwarp();
    } else {
        if (lane == 0)
            mma_role<D, BF16, CAUSAL>(p, sQ, sSlot, tmem, b, c);
        __syncwarp();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace fa
