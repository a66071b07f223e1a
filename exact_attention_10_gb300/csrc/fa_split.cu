// fa_split.cu -- the balanced-schedule kernel variants (tiles cut into parts,
// merged by the merge warp); see fa_launch.cuh.
#include "fa_launch.cuh"

namespace fa_launch {

fa_status launch_split(int D, bool bf16, bool causal, const CUtensorMap &q, const CUtensorMap &k,
                       const CUtensorMap &v, const fa::FwdParams &p, int grid, cudaStream_t s, int dev)
{
    return launch_any<true>(D, bf16, causal, q, k, v, p, grid, s, dev);
}

bool take_status_word_split(unsigned int *word)
{
    return take_status_word_here(word);
}

}  // namespace fa_launch
