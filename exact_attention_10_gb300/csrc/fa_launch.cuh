// fa_launch.cuh -- kernel selection and launch, shared by the three
// translation units that instantiate the kernels: fa_api.cu (whole-tile
// variants without a mask or with the causal one, and the C ABI), fa_split.cu
// (the same for the balanced schedule) and fa_band.cu (left-bounded band
// masks, both schedules).  Three units keep each nvcc run to eight kernels and
// let the build compile them in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace fa_launch {

constexpr int kMaxDevices = 64;

// Internal linkage: each translation unit launches its own kernels, and the
// once-per-device flags must stay private to this library (a template's
// static locals would otherwise be one object per process, shared with any
// other copy of the library loaded beside it).
namespace {

// Launch one variant on `grid` CTAs.  The dynamic shared-memory limit is
// raised once per device and variant.
template <int D, bool BF16, int MASK, bool SPLIT>
fa_status launch_variant(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const fa::FwdParams &p,
                         int grid, cudaStream_t stream, int dev)
{
    static std::mutex mu;
    static bool attr_set[kMaxDevices] = {};
    auto kern = fa::fa_fwd_sm103<D, BF16, MASK, SPLIT>;
    constexpr int smem = fa::Cfg<D>::smem_bytes(SPLIT);
    if (dev < 0 || dev >= kMaxDevices)
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
    kern<<<grid, fa::kThreads, smem, stream>>>(q, k, v, p);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    return FA_OK;
}

// The variants of one mask (kMaskNone, kMaskCausal or kMaskBand) and schedule.
template <int MASK, bool SPLIT>
fa_status launch_mask(int D, bool bf16, const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                      const fa::FwdParams &p, int grid, cudaStream_t s, int dev)
{
    if (D == 64)
        return bf16 ? launch_variant<64, true, MASK, SPLIT>(q, k, v, p, grid, s, dev)
                    : launch_variant<64, false, MASK, SPLIT>(q, k, v, p, grid, s, dev);
    return bf16 ? launch_variant<128, true, MASK, SPLIT>(q, k, v, p, grid, s, dev)
                : launch_variant<128, false, MASK, SPLIT>(q, k, v, p, grid, s, dev);
}

}  // namespace

// Defined in fa_api.cu, fa_split.cu and fa_band.cu respectively; `causal`
// selects kMaskCausal over kMaskNone, `split` the balanced schedule.
fa_status launch_whole(int D, bool bf16, bool causal, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev);
fa_status launch_split(int D, bool bf16, bool causal, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev);
fa_status launch_band(int D, bool bf16, bool split, const CUtensorMap &q, const CUtensorMap &k,
                      const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev);
bool take_status_word_whole(cudaStream_t s, unsigned int *word);
bool take_status_word_split(cudaStream_t s, unsigned int *word);
bool take_status_word_band(cudaStream_t s, unsigned int *word);

// The static workspace of fa_fwd_noalloc (fa_split.cu): points p's partial
// buffers into it for schedule `sc` and head size D, and clears the counters
// on `stream`.  FA_ERR_NO_ALLOC_LIMIT if the schedule needs more.
fa_status noalloc_workspace(int dev, cudaStream_t stream, const fa::Schedule &sc, int D, fa::FwdParams *p);

// Bytes of workspace a balanced schedule needs: partial O and (m, l) for two
// slots per CTA, then one counter per (tile, Q tile).
inline size_t workspace_bytes(const fa::Schedule &sc, int D, size_t *o_bytes, size_t *ml_bytes, size_t *cnt_bytes)
{
    const size_t slots = (size_t)2 * sc.G;
    *o_bytes = slots * fa::kCtaRows * D * sizeof(float);
    *ml_bytes = slots * fa::kCtaRows * sizeof(float2);
    *cnt_bytes = (size_t)2 * sc.T * sizeof(int);
    return *o_bytes + *ml_bytes + *cnt_bytes;   // (= fa::sched_workspace_bytes of a balanced schedule)
}

}  // namespace fa_launch
