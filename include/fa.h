/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 forward library.
 *
 * The operation is exact scaled-dot-product attention with an optional
 * causal mask and the per-row log-sum-exp:
 *
 *   O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] ) V[b,h,j,:]
 *   LSE[b,h,i] = log sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] )
 *
 * where j runs over all N keys, or over j <= i when causal.  It is computed
 * with the FlashAttention-2 forward recurrence: K/V tiles stream past an
 * on-chip Q tile, a running row max m and row sum l rescale an fp32 output
 * accumulator by exp(m_old - m_new), and the accumulator is divided by l once
 * at the end; the N x N score matrix is never written to memory.
 *
 * Sources (page title, section):
 *  - "FlashAttention 2 from PyTorch to Triton", What I am building: the
 *    recurrence, L = m + log(l) in natural-log units.
 *  - "A09 - Advanced Triton & FlashAttention", 3. Deep Dive: the rescaling
 *    update and its exactness; causal masking by block skipping.
 *  - "Building a Verifiable FlashAttention Forward from PyTorch to Triton",
 *    Scope: contiguous [B, H, N, D] self-attention, FP16/BF16, causal and
 *    non-causal, head dimension 64 or 128.
 *
 * Every call is asynchronous on the caller's stream and stream-ordered like a
 * kernel launch.  Nothing in this header throws.
 *
 * Device memory: calls that use the balanced schedule (below) need a
 * workspace for partial results -- per CTA two slots of [256, D] fp32 plus
 * (m, l) per row, and one int counter per (CTA tile, Q tile) -- about
 * 2 x 152 x 256 x (D + 2) x 4 bytes plus 8 bytes per 256 query rows per head.
 * It is allocated once per (device, stream) on the first such call, kept for
 * the life of the process, and reallocated larger (after synchronising that
 * stream) when a later call needs more; the counters are cleared with an
 * asynchronous memset when the buffer is new.  Calls on one stream share its
 * workspace in stream order; calls on different streams never share one.
 * Calls with the whole-tile schedule allocate nothing.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

/* The library is built with hidden symbol visibility; only these entry
 * points are exported. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st *fa_stream_t;

/* Element type of Q, K, V and O. */
typedef enum {
    FA_BF16 = 0,   /* bfloat16 */
    FA_FP16 = 1    /* IEEE binary16 */
} fa_dtype;

/*
 * Work decomposition over the persistent CTAs (one per SM).  A CTA tile is
 * 256 query rows of one head; a step is one 128-key tile of K and V.
 *  - FA_SCHEDULE_WHOLE_TILES: CTA c computes whole CTA tiles c, c + G, ...
 *  - FA_SCHEDULE_BALANCED: every CTA gets an equal share of all (tile, step)
 *    units; a tile cut by a share boundary is computed in parts whose partial
 *    results (O normalised per part, row max and sum) are merged by the last
 *    part to finish with the same rescaling rule the recurrence uses between
 *    key tiles ("A09 - Advanced Triton & FlashAttention", 3. Deep Dive).  This
 *    removes the idle SMs of a last partial wave of tiles.
 *  - FA_SCHEDULE_AUTO: the balanced schedule where it is expected to pay
 *    (non-causal calls whose shares span at least two tiles and whose last
 *    wave would leave SMs idle), whole tiles otherwise.
 * All three compute the same function; results agree to rounding.  The
 * pages describe one CTA per (Q tile, head) on a grid; these schedules are
 * this library's own.
 */
typedef enum {
    FA_SCHEDULE_AUTO = 0,
    FA_SCHEDULE_WHOLE_TILES = 1,
    FA_SCHEDULE_BALANCED = 2
} fa_schedule;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_VALUE = 1,      /* bad size, dtype, flag, scale, NULL, host pointer or overlapping output */
    FA_ERR_MISALIGNED = 2,         /* a pointer is not 16-byte aligned (the tensor-copy engine needs it) */
    FA_ERR_UNSUPPORTED_DEVICE = 3, /* no device, or the current device is not compute capability 10.3 */
    FA_ERR_CUDA = 4,               /* a CUDA runtime call or the launch failed */
    FA_ERR_DEVICE_TIMEOUT = 5,     /* a bounded in-kernel wait expired (reported by fa_sync_status) */
    FA_ERR_NO_ALLOC_LIMIT = 6      /* fa_fwd_noalloc: the call needs more than its static workspace */
} fa_status;

/*
 * fa_fwd -- attention forward for B*H independent heads.
 *
 * Q, K, V : device pointers to contiguous [B, H, N, D] tensors of `dtype`.
 *           They may alias one another (they are only read).
 * O       : device pointer to a contiguous [B, H, N, D] tensor of `dtype`;
 *           every element is written.  Must not overlap Q, K, V or LSE.
 * LSE     : device pointer to a contiguous [B, H, N] float32 tensor; row i
 *           receives log sum_j exp(scale * q_i . k_j) (natural log) over its
 *           visible keys.  Must not overlap Q, K, V or O.
 * B, H, N : batch, heads, sequence length (queries = keys = N); each >= 1 and
 *           B*H*N < 2^31.
 * D       : head dimension, 64 or 128.
 * causal  : 0 = every query sees all N keys; 1 = query i sees keys j <= i.
 *           Key tiles wholly above the diagonal are skipped, not masked.
 * scale   : softmax scale applied to q.k (usually 1/sqrt(D)); must be finite
 *           and > 0 (the kernel takes row maxima on unscaled scores).
 * stream  : CUDA stream the work is ordered on.
 *
 * All pointers belong to the caller and must stay valid until the work on
 * `stream` completes.  The device is the caller's current CUDA device.
 *
 * Returns FA_OK once the kernel is enqueued.  Argument errors are detected
 * before anything is enqueued and leave O and LSE untouched; FA_ERR_CUDA is
 * returned if a needed workspace cannot be allocated.  Errors raised inside
 * the kernel (a bounded wait that expired) are recorded in a per-device
 * status word and returned by fa_sync_status().
 *
 * fa_fwd uses FA_SCHEDULE_AUTO.
 */
FA_API fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                 int B, int H, int N, int D, int causal, float scale,
                 fa_dtype dtype, fa_stream_t stream);

/*
 * fa_fwd_ex -- fa_fwd with an explicit work decomposition `schedule` (see
 * fa_schedule); any other value returns FA_ERR_INVALID_VALUE.  A balanced
 * request the shape cannot take (more than 2^30 units of work) runs whole
 * tiles.
 */
FA_API fa_status fa_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE,
                    int B, int H, int N, int D, int causal, float scale,
                    fa_dtype dtype, fa_schedule schedule, fa_stream_t stream);

/*
 * fa_fwd_qkv -- fa_fwd_ex for Nq queries against Nkv keys per head: cross
 * attention, and decoding the last Nq positions of a longer sequence.
 *
 * Q, O : contiguous [B, H, Nq, D]; K, V : contiguous [B, H, Nkv, D];
 * LSE  : contiguous [B, H, Nq] float32.  Nq, Nkv >= 1, B*H*Nq < 2^31 and
 *        B*H*Nkv < 2^31; other arguments as for fa_fwd_ex.
 * causal: query i sees keys j <= i + (Nkv - Nq) -- aligned bottom-right, so
 *        the last query sees every key; with Nq = Nkv this is fa_fwd's mask.
 *        A query that sees no key (possible when Nq > Nkv) gets O = 0 and
 *        LSE = -inf.
 *
 * With few queries and many keys (decode) the balanced schedule splits each
 * head's keys over many CTAs and merges the partial results by their
 * log-sum-exp -- split-KV decoding; FA_SCHEDULE_AUTO picks it where it pays.
 * The pages fix only the square case; the bottom-right alignment is this
 * library's reading of the general one.
 */
FA_API fa_status fa_fwd_qkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                            int B, int H, int Nq, int Nkv, int D, int causal, float scale,
                            fa_dtype dtype, fa_schedule schedule, fa_stream_t stream);

/*
 * fa_fwd_band -- fa_fwd_qkv with a sliding-window (band) mask: with
 * i' = i + (Nkv - Nq), query i sees keys j in [i' - window_left,
 * i' + window_right]; a negative bound is unbounded on that side.  Causal is
 * (-1, 0), no mask (-1, -1), a causal window of W keys (W - 1, 0).  A query
 * whose band holds no key gets O = 0 and LSE = -inf.  Key tiles wholly
 * outside every row's band are skipped, not masked.  Other arguments as for
 * fa_fwd_qkv.
 */
FA_API fa_status fa_fwd_band(const void *Q, const void *K, const void *V, void *O, float *LSE,
                             int B, int H, int Nq, int Nkv, int D, int window_left, int window_right,
                             float scale, fa_dtype dtype, fa_schedule schedule, fa_stream_t stream);

/*
 * fa_fwd_noalloc -- fa_fwd_ex that allocates no memory, device or host, at
 * any call.  The pages describe nothing like it: the method itself needs no
 * scratch, and this entry point only concerns where this library's balanced
 * schedule keeps its partial results.
 *
 * Who needs it: callers that cannot let a library allocate device memory on
 * their behalf -- a serving loop whose latency budget has no room for the
 * implicit device-wide synchronisation cudaMalloc / cudaFree may perform, or
 * a framework that owns every byte of device memory through its own pool and
 * forbids allocations behind its back.  fa_fwd_ex would allocate its
 * per-stream workspace on the first balanced call; this entry point instead
 * uses a workspace compiled into the library: a static device array of
 * FA_NOALLOC_WORKSPACE_BYTES per device.
 *
 * Set-up: the first call on a device looks up that array's address
 * (cudaGetSymbolAddress, which may load the library's code onto the device)
 * and keeps it; make that first call before any stream capture.  Every call
 * clears the partial-result counters (which must start at zero) with an
 * asynchronous memset on `stream`.
 *
 * Limit: with FA_SCHEDULE_AUTO, where the automatic plan would split tiles
 * into more partial results than the array holds, the call runs whole tiles
 * instead, which need no workspace.  A call with FA_SCHEDULE_BALANCED whose
 * schedule needs more workspace than the array holds returns
 * FA_ERR_NO_ALLOC_LIMIT before anything is enqueued.  The partial-result
 * slots always fit; the counters take 8 bytes per 256 query rows per head,
 * so B*H*ceil(N/256) may reach
 * 966,656 -- e.g. B*H = 256 at N = 965,000.  Whole-tile calls need no
 * workspace and have no limit.
 *
 * Overlapping calls race: there is one workspace per device, so two calls
 * whose work can overlap (on different streams, without ordering between
 * them) must not both run the balanced schedule; calls on one stream are
 * ordered and safe.  Arguments, results and other errors are as for
 * fa_fwd_ex.
 */
#define FA_NOALLOC_WORKSPACE_BYTES (48u << 20)
FA_API fa_status fa_fwd_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE,
                                int B, int H, int N, int D, int causal, float scale,
                                fa_dtype dtype, fa_schedule schedule, fa_stream_t stream);

/*
 * fa_bwd -- attention backward: the gradients of fa_fwd's O with respect to
 * Q, K and V for an upstream gradient dO, from the forward's O and LSE.
 *
 * Q, K, V, O, dO : device pointers to contiguous [B, H, N, D] tensors of
 *                  `dtype` (O and LSE as fa_fwd wrote them for the same Q, K,
 *                  V, causal and scale).  Only read; they may alias one
 *                  another.
 * LSE            : device pointer to contiguous [B, H, N] float32.
 * dQ, dK, dV     : device pointers to contiguous [B, H, N, D] tensors of
 *                  `dtype`; every element is written.  None may overlap an
 *                  input or another output.
 * B, H, N, D, causal, scale, dtype, stream : as for fa_fwd; B*H*ceil(N/128)*128
 *                  must stay below 2^31.
 *
 * With P = exp(scale * Q K^T - LSE) (0 where causal hides key j > query i)
 * and delta = rowsum(dO o O):  dV = P^T dO,  dS = P o (dO V^T - delta),
 * dQ = scale * dS K,  dK = scale * dS^T Q.  P and dS are rounded to `dtype`
 * for the tensor-core products, which accumulate in fp32.  P is recomputed
 * from LSE ("FlashAttention 2 from PyTorch to Triton", What I am building);
 * dK and dV are accumulated per key tile over the query tiles.  dQ (the
 * page's list of limitations: "by atomics or a second pass"):
 *  - D = 64: in the same pass, each key tile's dQ products added into an
 *    fp32 accumulator in global memory by tensor reductions (fp32 adds in
 *    L2), then scaled and rounded to `dtype`.  The order of those adds varies
 *    from call to call, so dQ may differ in its last bits between calls;
 *    dK and dV do not.
 *  - D = 128, and any call through fa_bwd_ex with FA_BWD_DETERMINISTIC: in a
 *    second pass over the key tiles, without atomics; bit for bit the same
 *    on every call.
 *
 * Scratch: 8 bytes per query row (rounded up to 128 rows per head) for delta
 * and LSE * log2(e), plus 4 * D bytes per such row for the dQ accumulator on
 * the D = 64 single pass, allocated per (device, stream) on first use like
 * the balanced schedule's workspace.  Errors as for fa_fwd; FA_ERR_CUDA if
 * the scratch cannot be allocated.
 */
FA_API fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D, int causal,
                        float scale, fa_dtype dtype, fa_stream_t stream);

/*
 * fa_bwd_band -- fa_bwd for Nq queries against Nkv keys under the band mask
 * of fa_fwd_band (window_left, window_right; a negative bound is unbounded;
 * causal = (-1, 0), no mask = (-1, -1)), from that call's O and LSE.
 *
 * Q, O, dO, dQ : contiguous [B, H, Nq, D];  K, V, dK, dV : contiguous
 * [B, H, Nkv, D];  LSE : [B, H, Nq] float32.  A query that sees no key
 * (LSE = -inf) contributes nothing and gets dQ = 0; a key that no query sees
 * gets dK = dV = 0.  Each key tile visits only the query tiles whose bands
 * reach it, and each query tile only the key tiles its rows' bands reach.
 * Other arguments as for fa_bwd; B*H*Nkv must stay below 2^31 as well.
 */
FA_API fa_status fa_bwd_band(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                             const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nkv, int D,
                             int window_left, int window_right, float scale, fa_dtype dtype, fa_stream_t stream);

/* fa_bwd_ex flags. */
#define FA_BWD_DETERMINISTIC 1u /* dQ by the second pass at every D: the same bits on every call */

/*
 * fa_bwd_ex -- fa_bwd_band with `flags` (0 or FA_BWD_DETERMINISTIC; any other
 * bit: FA_ERR_INVALID_VALUE).  fa_bwd and fa_bwd_band are fa_bwd_ex with
 * flags = 0.
 */
FA_API fa_status fa_bwd_ex(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                           const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nkv, int D,
                           int window_left, int window_right, float scale, fa_dtype dtype, unsigned int flags,
                           fa_stream_t stream);

/*
 * fa_sync_status -- synchronise `stream`, then return and clear the device
 * status word of the current device: FA_OK, FA_ERR_DEVICE_TIMEOUT if a kernel
 * gave up on a wait since the last call, or FA_ERR_CUDA if the synchronise
 * itself failed.
 *
 * The word is read and cleared in one atomic exchange by a one-thread kernel
 * on `stream`, so a timeout recorded meanwhile is never lost.  There is one
 * word per device, shared by all streams: a timeout from a kernel on another
 * stream is reported by whichever call reads the word first, and a timeout
 * from a kernel on another stream that has not finished yet is reported only
 * by a later call.  To attribute a timeout to a stream, synchronise the
 * others first.
 *
 * Device resets: the library keeps, per device, a lazily created workspace,
 * the status word and the static workspace's address.  A call that follows
 * cudaDeviceReset() on that device in the same process is not supported.
 */
FA_API fa_status fa_sync_status(fa_stream_t stream);

/* Static, NUL-terminated description of a status code. */
FA_API const char *fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
