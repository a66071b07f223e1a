// fa_bwd.cu -- the backward kernels (fa_bwd_kernel.cuh) and their launch:
// the per-row pre-pass, then the dQ pass and the dK/dV pass, or at D = 64 the
// fused pass and the dQ conversion, on one stream.
#include "fa_bwd_launch.h"

#include <mutex>
#include <utility>

#include "fa_bwd_kernel.cuh"

namespace fa_launch {

namespace {

constexpr int kMaxDev = 64;

// Launch `kern` on `stream` allowing programmatic dependent launch: it may
// start while the previous kernel on the stream finishes, and waits for that
// kernel's completion with griddepcontrol.wait before reading its results.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, bool BF16, bool CAUSAL, bool KV, bool FQ = false>
fa_status launch_pass(const CUtensorMap &r0, const CUtensorMap &r1, const CUtensorMap &s0, const CUtensorMap &s1,
                      const CUtensorMap &dq, const fa::bwd::Params &p, int grid, cudaStream_t stream, int dev)
{
    static std::mutex mu;
    static bool attr_set[kMaxDev] = {};
    auto kern = fa::bwd::fa_bwd_sm103<D, BF16, CAUSAL, KV, FQ>;
    constexpr int smem = fa::bwd::BCfg<D, KV, FQ>::kSmem;
    if (dev < 0 || dev >= kMaxDev)
        return FA_ERR_UNSUPPORTED_DEVICE;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
                cudaGetLastError();
                return FA_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
    }
    // right behind the previous kernel (programmatic dependent launch): see fa_bwd_sm103
    if (launch_dependent(kern, dim3(grid), dim3(FQ ? fa::bwd::kThreadsFused : fa::bwd::kThreads), smem, stream, r0, r1,
                         s0, s1, dq, p) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

template <int D, bool BF16, bool CAUSAL>
fa_status launch_all(const BwdLaunch &a, cudaStream_t s, int dev)
{
    const long long rows = (long long)a.BH * a.Npad;
    const long long threads = rows * (D / 8);
    const bool fused = (D == 64) && a.fused;
    fa::bwd::fa_bwd_prep<D, BF16><<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(
        static_cast<const uint16_t *>(a.O), static_cast<const uint16_t *>(a.dO), a.LSE, a.lg, a.dl,
        fused ? a.dqa : nullptr, a.N, a.Npad, rows);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    fa::bwd::Params p{};
    p.lg = a.lg;
    p.dl = a.dl;
    p.N = a.N;
    p.Nkv = a.Nkv;
    p.Npad = a.Npad;
    p.BH = a.BH;
    p.nqt = a.Npad / fa::bwd::kTile;
    p.nkt = (a.Nkv + fa::bwd::kTile - 1) / fa::bwd::kTile;
    p.off = a.Nkv - a.N;
    p.wl = a.wl;
    p.wr = a.wr;
    p.square_causal = (a.N == a.Nkv && a.wl >= fa::kSchedUnbounded && a.wr == 0) ? 1 : 0;
    p.qk2 = a.scale * 1.4426950408889634f;
    p.scale = a.scale;
    int grid;
    if constexpr (D == 64) {
        if (fused) {   // dK, dV and the dQ accumulator in one pass, then dQ from the accumulator
            p.T = a.BH * p.nkt;
            grid = p.T < a.sms ? p.T : a.sms;
            p.dA = a.dK;
            p.dB = a.dV;
            const fa_status st = launch_pass<D, BF16, CAUSAL, true, true>(a.tk, a.tv, a.tq, a.tdo, a.tdqa, p, grid, s, dev);
            if (st != FA_OK)
                return st;
            const long long elems = (long long)a.BH * a.N * D;
            if (launch_dependent(fa::bwd::fa_bwd_dq_convert<BF16>, dim3((unsigned)((elems / 8 + 255) / 256)), dim3(256),
                                 0, s, (const float *)a.dqa, static_cast<uint16_t *>(a.dQ), a.N, a.Npad, D, elems,
                                 a.scale) != cudaSuccess) {
                cudaGetLastError();
                return FA_ERR_CUDA;
            }
            return FA_OK;
        }
    }
    p.T = a.BH * p.nqt;
    grid = p.T < a.sms ? p.T : a.sms;
    p.dA = a.dQ;
    p.dB = nullptr;
    fa_status st = launch_pass<D, BF16, CAUSAL, false>(a.tq, a.tdo, a.tk, a.tv, a.tq, p, grid, s, dev);
    if (st != FA_OK)
        return st;
    p.T = a.BH * p.nkt;
    grid = p.T < a.sms ? p.T : a.sms;
    p.dA = a.dK;
    p.dB = a.dV;
    return launch_pass<D, BF16, CAUSAL, true>(a.tk, a.tv, a.tq, a.tdo, a.tq, p, grid, s, dev);
}

}  // namespace

fa_status launch_bwd(const BwdLaunch &a, cudaStream_t s, int dev)
{
    if (a.D == 64) {
        if (a.bf16)
            return a.causal ? launch_all<64, true, true>(a, s, dev) : launch_all<64, true, false>(a, s, dev);
        return a.causal ? launch_all<64, false, true>(a, s, dev) : launch_all<64, false, false>(a, s, dev);
    }
    if (a.bf16)
        return a.causal ? launch_all<128, true, true>(a, s, dev) : launch_all<128, true, false>(a, s, dev);
    return a.causal ? launch_all<128, false, true>(a, s, dev) : launch_all<128, false, false>(a, s, dev);
}

bool take_status_word_bwd(cudaStream_t s, unsigned int *word)
{
    return fa::take_status_word_on(s, word);
}

}  // namespace fa_launch
