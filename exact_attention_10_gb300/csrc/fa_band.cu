// fa_band.cu -- the kernel variants for band (sliding-window) masks with a
// left bound, whole-tile and balanced schedules; see fa_launch.cuh.
#include "fa_launch.cuh"

namespace fa_launch {

fa_status launch_band(int D, bool bf16, bool split, const CUtensorMap &q, const CUtensorMap &k,
                      const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev)
{
    return split ? launch_mask<fa::kMaskBand, true>(D, bf16, q, k, v, p, grid, s, dev)
                 : launch_mask<fa::kMaskBand, false>(D, bf16, q, k, v, p, grid, s, dev);
}

bool take_status_word_band(cudaStream_t s, unsigned int *word)
{
    return fa::take_status_word_on(s, word);
}

}  // namespace fa_launch
