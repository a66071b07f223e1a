// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, TMA descriptor encoding, kernel selection and launch, and the
// device status word.
//
// The problem statement follows "Building a Verifiable FlashAttention Forward
// from PyTorch to Triton" (Scope: contiguous [B, H, N, D] self-attention,
// FP16/BF16, causal or not, D in {64, 128}) with the caller's softmax scale.
#include "fa.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa_bwd_launch.h"
#include "fa_launch.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, resolved through the runtime so the
// library has no link-time dependency on the driver library.
EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<EncodeTiledFn>(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

constexpr int kMaxDevices = fa_launch::kMaxDevices;

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_devices[kMaxDevices];

// Probe the current device once: compute capability 10.3 is required because
// the kernels are built for sm_103a only.
const DeviceInfo *device_info(int dev)
{
    if (dev < 0 || dev >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
            d.supported = (major == 10 && minor == 3);
            d.sms = sms;
        } else {
            cudaGetLastError();
        }
        d.probed = true;
    }
    return &d;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Device (or managed) memory of the current device.
bool is_device_pointer(const void *p, int dev)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeManaged)
        return true;
    return a.type == cudaMemoryTypeDevice && a.device == dev;
}

// Rank-3 map over [B*H, N, D] (innermost first): per-head row bounds, so a
// box that runs past N is zero-filled instead of reading the next head.
// Box = 64 columns (128 bytes, the 128-byte swizzle width) x 128 rows.
bool encode_map(CUtensorMap *m, const void *ptr, int BH, int N, int D, bool bf16)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)fa::kBM, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                           const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Rank-2 map over an fp32 [rows, D] array (the backward's dQ accumulator),
// 32 columns (128 bytes) x 128 rows per box, 128-byte swizzle: the fused
// backward pass adds its staged dQ products into it box by box.
bool encode_map_f32(CUtensorMap *m, float *ptr, long long rows, int D)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Per-(device, stream) workspace for split tiles: partial O and (m, l) for
// two slots per CTA, and one counter per (tile, Q tile) that must be zero
// when a launch starts (each launch leaves it zero).  Allocated on the first
// call that needs it on that stream and grown when a later call needs more;
// calls on different streams never share one, so they cannot race.
struct Workspace {
    int dev;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
    size_t counter_bytes;
};
constexpr int kMaxWorkspaces = 64;
Workspace g_ws[kMaxWorkspaces];
int g_ws_count = 0;

fa_status workspace_for(int dev, cudaStream_t stream, const fa::Schedule &sc, int D, fa::FwdParams *p)
{
    const size_t slots = (size_t)2 * sc.G;
    const size_t o_bytes = slots * fa::kCtaRows * D * sizeof(float);
    const size_t ml_bytes = slots * fa::kCtaRows * sizeof(float2);
    const size_t cnt_bytes = (size_t)2 * sc.T * sizeof(int);
    const size_t need = o_bytes + ml_bytes + cnt_bytes;
    std::lock_guard<std::mutex> lock(g_mu);
    Workspace *w = nullptr;
    for (int i = 0; i < g_ws_count; ++i)
        if (g_ws[i].dev == dev && g_ws[i].stream == stream)
            w = &g_ws[i];
    if (!w) {
        if (g_ws_count == kMaxWorkspaces)
            return FA_ERR_CUDA;
        w = &g_ws[g_ws_count++];
        *w = Workspace{dev, stream, nullptr, 0, 0};
    }
    if (w->bytes < need) {
        if (w->ptr) {
            // work already queued on this stream may still use the old buffer
            if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(w->ptr) != cudaSuccess) {
                cudaGetLastError();
                return FA_ERR_CUDA;
            }
            w->ptr = nullptr;
            w->bytes = 0;
        }
        if (cudaMalloc(&w->ptr, need) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_CUDA;
        }
        w->bytes = need;
        w->counter_bytes = 0;
    }
    // Counters sit at the end of the buffer and must be zero when a launch
    // starts.  Launches leave them zero, so they are cleared only when the
    // buffer is new or has grown (and after an expired in-kernel wait, by
    // fa_sync_status).
    const size_t cnt_off = w->bytes - cnt_bytes;
    if (w->counter_bytes != cnt_bytes) {
        if (cudaMemsetAsync(static_cast<char *>(w->ptr) + cnt_off, 0, cnt_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_CUDA;
        }
        w->counter_bytes = cnt_bytes;
    }
    p->part_o = static_cast<float *>(w->ptr);
    p->part_ml = reinterpret_cast<float2 *>(static_cast<char *>(w->ptr) + o_bytes);
    p->counters = reinterpret_cast<int *>(static_cast<char *>(w->ptr) + cnt_off);
    return FA_OK;
}

// Per-(device, stream) scratch of the backward: lg and delta per query row,
// [B*H][Npad] fp32 each.  Grown like the forward's workspace; calls on one
// stream reuse it in stream order.
struct BwdWorkspace {
    int dev;
    cudaStream_t stream;
    void *ptr;
    size_t bytes;
};
BwdWorkspace g_bws[kMaxWorkspaces];
int g_bws_count = 0;

void *bwd_workspace(int dev, cudaStream_t stream, size_t need)
{
    std::lock_guard<std::mutex> lock(g_mu);
    BwdWorkspace *w = nullptr;
    for (int i = 0; i < g_bws_count; ++i)
        if (g_bws[i].dev == dev && g_bws[i].stream == stream)
            w = &g_bws[i];
    if (!w) {
        if (g_bws_count == kMaxWorkspaces)
            return nullptr;
        w = &g_bws[g_bws_count++];
        *w = BwdWorkspace{dev, stream, nullptr, 0};
    }
    if (w->bytes < need) {
        if (w->ptr) {
            if (cudaStreamSynchronize(stream) != cudaSuccess || cudaFree(w->ptr) != cudaSuccess) {
                cudaGetLastError();
                return nullptr;
            }
            w->ptr = nullptr;
            w->bytes = 0;
        }
        if (cudaMalloc(&w->ptr, need) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        w->bytes = need;
    }
    return w->ptr;
}

}  // namespace

namespace fa_launch {

fa_status launch_whole(int D, bool bf16, bool causal, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev)
{
    return causal ? launch_mask<fa::kMaskCausal, false>(D, bf16, q, k, v, p, grid, s, dev)
                  : launch_mask<fa::kMaskNone, false>(D, bf16, q, k, v, p, grid, s, dev);
}

bool take_status_word_whole(cudaStream_t s, unsigned int *word)
{
    return fa::take_status_word_on(s, word);
}

}  // namespace fa_launch

namespace {

// Every entry point: N query rows against Nkv keys per head (Nkv = N but for
// fa_fwd_qkv / fa_fwd_band), masked by the band [i' - left, i' + right] with
// i' = i + Nkv - N (a negative bound: unbounded; causal = (-1, 0), no mask =
// (-1, -1)); no_alloc takes a balanced schedule's workspace from the
// library's static array.
fa_status fwd_impl(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N, int Nkv,
                   int D, int left, int right, float scale, fa_dtype dtype, fa_schedule schedule, fa_stream_t stream,
                   bool no_alloc)
{
    int wl = left, wr = right;   // bounds that cannot bind are dropped: a band of no bounds runs unmasked
    if (N >= 1 && Nkv >= 1)
        fa::sched_band_normalize(N, Nkv, wl, wr);
    const int causal = (wl < fa::kSchedUnbounded || wr < fa::kSchedUnbounded) ? 1 : 0;   // masked at all
    const bool band = wl < fa::kSchedUnbounded;   // bounded on the left: the kMaskBand kernels
    // Arguments first: nothing below touches the device until they are sound.
    if (dtype != FA_BF16 && dtype != FA_FP16)
        return FA_ERR_INVALID_VALUE;
    if (schedule != FA_SCHEDULE_AUTO && schedule != FA_SCHEDULE_WHOLE_TILES && schedule != FA_SCHEDULE_BALANCED)
        return FA_ERR_INVALID_VALUE;
    if (D != 64 && D != 128)
        return FA_ERR_INVALID_VALUE;
    if (B < 1 || H < 1 || N < 1 || Nkv < 1)
        return FA_ERR_INVALID_VALUE;
    if (!std::isfinite(scale) || !(scale > 0.f))
        return FA_ERR_INVALID_VALUE;
    const long long BH = (long long)B * H;
    if (BH * N >= (1ll << 31) || BH * Nkv >= (1ll << 31))
        return FA_ERR_INVALID_VALUE;
    if (!Q || !K || !V || !O || !LSE)
        return FA_ERR_INVALID_VALUE;
    const uintptr_t any = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                          reinterpret_cast<uintptr_t>(LSE);
    if (any & 15u)
        return FA_ERR_MISALIGNED;
    const size_t qbytes = (size_t)BH * N * D * 2, kbytes = (size_t)BH * Nkv * D * 2,
                 lbytes = (size_t)BH * N * sizeof(float);
    if (ranges_overlap(O, qbytes, Q, qbytes) || ranges_overlap(O, qbytes, K, kbytes) ||
        ranges_overlap(O, qbytes, V, kbytes) || ranges_overlap(LSE, lbytes, Q, qbytes) ||
        ranges_overlap(LSE, lbytes, K, kbytes) || ranges_overlap(LSE, lbytes, V, kbytes) ||
        ranges_overlap(LSE, lbytes, O, qbytes))
        return FA_ERR_INVALID_VALUE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_UNSUPPORTED_DEVICE;
    }
    const DeviceInfo *di = device_info(dev);
    if (!di || !di->supported)
        return FA_ERR_UNSUPPORTED_DEVICE;
    if (!is_device_pointer(Q, dev) || !is_device_pointer(K, dev) || !is_device_pointer(V, dev) ||
        !is_device_pointer(O, dev) || !is_device_pointer(LSE, dev))
        return FA_ERR_INVALID_VALUE;

    const bool bf16 = dtype == FA_BF16;
    alignas(64) CUtensorMap tq, tk, tv;
    if (!encode_map(&tq, Q, (int)BH, N, D, bf16) || !encode_map(&tk, K, (int)BH, Nkv, D, bf16) ||
        !encode_map(&tv, V, (int)BH, Nkv, D, bf16))
        return FA_ERR_CUDA;

    fa::FwdParams p{};
    p.O = O;
    p.LSE = LSE;
    p.N = N;
    p.Nkv = Nkv;
    p.off = causal ? Nkv - N : 0;
    p.qk_scale = scale * 1.4426950408889634f;   // scale * log2(e)
    // A call that may not allocate takes whole tiles where the automatic
    // plan would need more than its static workspace.
    p.sch = no_alloc ? fa::sched_plan_limited(N, Nkv, (int)BH, causal != 0, di->sms, (int)schedule, wl, wr, D,
                                              FA_NOALLOC_WORKSPACE_BYTES)
                     : fa::sched_plan(N, Nkv, (int)BH, causal != 0, di->sms, (int)schedule, wl, wr);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p.sch.split) {
        const fa_status ws =
            no_alloc ? fa_launch::noalloc_workspace(dev, s, p.sch, D, &p) : workspace_for(dev, s, p.sch, D, &p);
        if (ws != FA_OK)
            return ws;
    }
    if (p.sch.split)
        return band ? fa_launch::launch_band(D, bf16, true, tq, tk, tv, p, p.sch.G, s, dev)
                    : fa_launch::launch_split(D, bf16, causal != 0, tq, tk, tv, p, p.sch.G, s, dev);
    return band ? fa_launch::launch_band(D, bf16, false, tq, tk, tv, p, p.sch.G, s, dev)
                : fa_launch::launch_whole(D, bf16, causal != 0, tq, tk, tv, p, p.sch.G, s, dev);
}

}  // namespace

extern "C" fa_status fa_fwd_ex(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                               int N, int D, int causal, float scale, fa_dtype dtype, fa_schedule schedule,
                               fa_stream_t stream)
{
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_VALUE;
    return fwd_impl(Q, K, V, O, LSE, B, H, N, N, D, -1, causal ? 0 : -1, scale, dtype, schedule, stream, false);
}

extern "C" fa_status fa_fwd_qkv(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                int Nq, int Nkv, int D, int causal, float scale, fa_dtype dtype, fa_schedule schedule,
                                fa_stream_t stream)
{
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_VALUE;
    return fwd_impl(Q, K, V, O, LSE, B, H, Nq, Nkv, D, -1, causal ? 0 : -1, scale, dtype, schedule, stream, false);
}

extern "C" fa_status fa_fwd_band(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                 int Nq, int Nkv, int D, int window_left, int window_right, float scale, fa_dtype dtype,
                                 fa_schedule schedule, fa_stream_t stream)
{
    return fwd_impl(Q, K, V, O, LSE, B, H, Nq, Nkv, D, window_left, window_right, scale, dtype, schedule, stream,
                    false);
}

extern "C" fa_status fa_fwd_noalloc(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H,
                                    int N, int D, int causal, float scale, fa_dtype dtype, fa_schedule schedule,
                                    fa_stream_t stream)
{
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_VALUE;
    return fwd_impl(Q, K, V, O, LSE, B, H, N, N, D, -1, causal ? 0 : -1, scale, dtype, schedule, stream, true);
}

extern "C" fa_status fa_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int B, int H, int N,
                            int D, int causal, float scale, fa_dtype dtype, fa_stream_t stream)
{
    return fa_fwd_ex(Q, K, V, O, LSE, B, H, N, D, causal, scale, dtype, FA_SCHEDULE_AUTO, stream);
}

namespace {

// Every backward entry point: N query rows against Nkv keys per head, masked
// by the band [i' - left, i' + right], i' = i + Nkv - N (a negative bound:
// unbounded; causal = (-1, 0), no mask = (-1, -1)).
fa_status bwd_impl(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                   void *dQ, void *dK, void *dV, int B, int H, int N, int Nkv, int D, int left, int right, float scale,
                   fa_dtype dtype, unsigned int flags, fa_stream_t stream)
{
    if (flags & ~FA_BWD_DETERMINISTIC)
        return FA_ERR_INVALID_VALUE;
    int wl = left, wr = right;   // bounds that cannot bind are dropped: a band of no bounds runs unmasked
    if (N >= 1 && Nkv >= 1)
        fa::sched_band_normalize(N, Nkv, wl, wr);
    const bool masked = wl < fa::kSchedUnbounded || wr < fa::kSchedUnbounded;
    // Arguments first: nothing below touches the device until they are sound.
    if (dtype != FA_BF16 && dtype != FA_FP16)
        return FA_ERR_INVALID_VALUE;
    if (D != 64 && D != 128)
        return FA_ERR_INVALID_VALUE;
    if (B < 1 || H < 1 || N < 1 || Nkv < 1)
        return FA_ERR_INVALID_VALUE;
    if (!std::isfinite(scale) || !(scale > 0.f))
        return FA_ERR_INVALID_VALUE;
    const long long BH = (long long)B * H;
    const long long Npad = ((long long)N + 127) / 128 * 128;
    if (BH * Npad >= (1ll << 31) || BH * Nkv >= (1ll << 31))
        return FA_ERR_INVALID_VALUE;
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV)
        return FA_ERR_INVALID_VALUE;
    const uintptr_t any = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                          reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                          reinterpret_cast<uintptr_t>(dO) | reinterpret_cast<uintptr_t>(LSE) |
                          reinterpret_cast<uintptr_t>(dQ) | reinterpret_cast<uintptr_t>(dK) |
                          reinterpret_cast<uintptr_t>(dV);
    if (any & 15u)
        return FA_ERR_MISALIGNED;
    const size_t qbytes = (size_t)BH * N * D * 2, kbytes = (size_t)BH * Nkv * D * 2, lbytes = (size_t)BH * N * 4;
    const void *ins[6] = {Q, K, V, O, dO, LSE};
    const size_t in_bytes[6] = {qbytes, kbytes, kbytes, qbytes, qbytes, lbytes};
    void *outs[3] = {dQ, dK, dV};
    const size_t out_bytes[3] = {qbytes, kbytes, kbytes};
    for (int o = 0; o < 3; ++o) {   // outputs overlap no input and no other output
        for (int i = 0; i < 6; ++i)
            if (ranges_overlap(outs[o], out_bytes[o], ins[i], in_bytes[i]))
                return FA_ERR_INVALID_VALUE;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (ranges_overlap(outs[o], out_bytes[o], outs[o2], out_bytes[o2]))
                return FA_ERR_INVALID_VALUE;
    }

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_UNSUPPORTED_DEVICE;
    }
    const DeviceInfo *di = device_info(dev);
    if (!di || !di->supported)
        return FA_ERR_UNSUPPORTED_DEVICE;
    for (int i = 0; i < 6; ++i)
        if (!is_device_pointer(ins[i], dev))
            return FA_ERR_INVALID_VALUE;
    for (int o = 0; o < 3; ++o)
        if (!is_device_pointer(outs[o], dev))
            return FA_ERR_INVALID_VALUE;

    const bool bf16 = dtype == FA_BF16;
    fa_launch::BwdLaunch a{};
    if (!encode_map(&a.tq, Q, (int)BH, N, D, bf16) || !encode_map(&a.tk, K, (int)BH, Nkv, D, bf16) ||
        !encode_map(&a.tv, V, (int)BH, Nkv, D, bf16) || !encode_map(&a.tdo, dO, (int)BH, N, D, bf16))
        return FA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // D = 64 without FA_BWD_DETERMINISTIC: the fused pass, with an fp32 dQ
    // accumulator [B*H*Npad, D] after delta and lg (1024-byte aligned: Npad % 128 == 0)
    const bool fused = D == 64 && !(flags & FA_BWD_DETERMINISTIC);
    float *ws = static_cast<float *>(
        bwd_workspace(dev, s, (size_t)(2 + (fused ? D : 0)) * BH * Npad * sizeof(float)));
    if (!ws)
        return FA_ERR_CUDA;
    a.fused = fused;
    if (fused) {
        a.dqa = ws + 2 * BH * Npad;
        if (!encode_map_f32(&a.tdqa, a.dqa, BH * Npad, D))
            return FA_ERR_CUDA;
    }
    a.O = O;
    a.dO = dO;
    a.LSE = LSE;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.lg = ws;
    a.dl = ws + BH * Npad;
    a.BH = (int)BH;
    a.N = N;
    a.Nkv = Nkv;
    a.Npad = (int)Npad;
    a.D = D;
    a.sms = di->sms;
    a.bf16 = bf16;
    a.causal = masked;
    a.wl = wl;
    a.wr = wr;
    a.scale = scale;
    return fa_launch::launch_bwd(a, s, dev);
}

}  // namespace

extern "C" fa_status fa_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                            const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int N, int D, int causal,
                            float scale, fa_dtype dtype, fa_stream_t stream)
{
    if (causal != 0 && causal != 1)
        return FA_ERR_INVALID_VALUE;
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, N, D, -1, causal ? 0 : -1, scale, dtype, 0u, stream);
}

extern "C" fa_status fa_bwd_band(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                                 const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nkv, int D,
                                 int window_left, int window_right, float scale, fa_dtype dtype, fa_stream_t stream)
{
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nkv, D, window_left, window_right, scale, dtype, 0u,
                    stream);
}

extern "C" fa_status fa_bwd_ex(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                               const float *LSE, void *dQ, void *dK, void *dV, int B, int H, int Nq, int Nkv, int D,
                               int window_left, int window_right, float scale, fa_dtype dtype, unsigned int flags,
                               fa_stream_t stream)
{
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nkv, D, window_left, window_right, scale, dtype, flags,
                    stream);
}

extern "C" fa_status fa_sync_status(fa_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int w_whole = 0, w_split = 0, w_band = 0, w_bwd = 0;
    if (!fa_launch::take_status_word_whole(s, &w_whole) || !fa_launch::take_status_word_split(s, &w_split) ||
        !fa_launch::take_status_word_band(s, &w_band) || !fa_launch::take_status_word_bwd(s, &w_bwd))
        return FA_ERR_CUDA;
    if ((w_whole | w_split | w_band | w_bwd) != 0) {
        // an aborted launch may have left split-tile counters non-zero
        int dev = -1;
        cudaGetDevice(&dev);
        {
            std::lock_guard<std::mutex> lock(g_mu);
            for (int i = 0; i < g_ws_count; ++i)
                if (g_ws[i].dev == dev && g_ws[i].ptr)
                    g_ws[i].counter_bytes = 0;   // cleared again by the next call that uses it
        }
        return FA_ERR_DEVICE_TIMEOUT;
    }
    return FA_OK;
}

extern "C" const char *fa_status_string(fa_status s)
{
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_VALUE: return "invalid argument";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_UNSUPPORTED_DEVICE: return "no compute capability 10.3 device";
    case FA_ERR_CUDA: return "CUDA runtime or launch error";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside the kernel expired";
    case FA_ERR_NO_ALLOC_LIMIT: return "the call needs more than the no-allocation entry point's static workspace";
    }
    return "unknown status";
}
