// fa_split.cu -- the balanced-schedule kernel variants (tiles cut into parts,
// merged by the merge warp); see fa_launch.cuh.
#include "fa_launch.cuh"

#include <cstring>

namespace fa_launch {

fa_status launch_split(int D, bool bf16, bool causal, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev)
{
    return causal ? launch_mask<fa::kMaskCausal, true>(D, bf16, q, k, v, p, grid, s, dev)
                  : launch_mask<fa::kMaskNone, true>(D, bf16, q, k, v, p, grid, s, dev);
}

bool take_status_word_split(cudaStream_t s, unsigned int *word)
{
    return fa::take_status_word_on(s, word);
}

namespace {

// The workspace of fa_fwd_noalloc: one per device, zero at load, never
// allocated or freed by a call.
static __device__ __align__(256) unsigned char g_noalloc_ws[FA_NOALLOC_WORKSPACE_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

fa_status noalloc_workspace(int dev, cudaStream_t stream, const fa::Schedule &sc, int D, fa::FwdParams *p)
{
    size_t o_bytes, ml_bytes, cnt_bytes;
    const size_t need = workspace_bytes(sc, D, &o_bytes, &ml_bytes, &cnt_bytes);
    if (need > FA_NOALLOC_WORKSPACE_BYTES)
        return FA_ERR_NO_ALLOC_LIMIT;
    if (dev < 0 || dev >= kMaxDevices)
        return FA_ERR_UNSUPPORTED_DEVICE;
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {   // once per device
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_ws) != cudaSuccess || !addr) {
                cudaGetLastError();
                return FA_ERR_CUDA;
            }
            g_noalloc_ptr[dev] = addr;
        }
        base = g_noalloc_ptr[dev];
    }
    char *ws = static_cast<char *>(base);
    p->part_o = reinterpret_cast<float *>(ws);
    p->part_ml = reinterpret_cast<float2 *>(ws + o_bytes);
    p->counters = reinterpret_cast<int *>(ws + o_bytes + ml_bytes);
    if (cudaMemsetAsync(p->counters, 0, cnt_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    return FA_OK;
}

}  // namespace fa_launch
