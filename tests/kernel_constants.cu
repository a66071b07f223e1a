// Prints, as one JSON object, the pipeline constants of the forward and
// backward kernels that the CPU models of their mbarrier protocols assume
// (tests/test_pipeline_protocol.py, tests/test_bwd_protocol.py), so that a
// change to the kernels' ring depths or issue structure shows up there.
#include <cstdio>

#include "fa_bwd_kernel.cuh"

template <int D>
void fwd(const char *name, bool last)
{
    using C = fa::Cfg<D>;
    std::printf("\"%s\": {\"stages\": %d, \"q_bufs\": %d, \"mma_warps\": %d, \"sep\": %d, \"split_kv\": %d}%s", name,
                C::kStages, C::kQBufs, C::kMmaWarps, (int)C::kSeparateP, (int)C::kSplitKV, last ? "" : ", ");
}

template <int D, bool KV, bool FQ = false>
void bwd(const char *name, bool last)
{
    using C = fa::bwd::BCfg<D, KV, FQ>;
    std::printf("\"%s\": {\"pipeline\": %d, \"split\": %d, \"ring0\": %d, \"ring1\": %d}%s", name,
                (int)fa::bwd::kPipeline<D, KV>, (int)C::kSplitRing, C::kRing0, C::kRing1, last ? "" : ", ");
}

int main()
{
    std::printf("{\"q_tiles\": %d, ", fa::kQTiles);
    fwd<64>("fwd64", false);
    fwd<128>("fwd128", false);
    bwd<64, false>("d64_dq", false);
    bwd<64, true>("d64_kv", false);
    bwd<64, true, true>("d64_fused", false);
    bwd<128, false>("d128_dq", false);
    bwd<128, true>("d128_kv", true);
    std::printf("}\n");
    return 0;
}
