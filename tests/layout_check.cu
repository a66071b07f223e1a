// Shared-memory layout of the forward and backward kernels, checked on the
// host: for each head size and variant, every region (Q tiles, the K/V ring,
// mbarriers, the hand-off and misc words, the merge staging and job queue,
// the split ring's V barriers) lies inside the launch's shared memory, keeps
// the alignment its users need (1024 bytes for the 128-byte-swizzled TMA and
// MMA tiles, 128 for bulk-copy staging, 8 for mbarriers), and overlaps no
// other region.  Prints one line per layout and "ok" when all pass.
#include <cstdio>
#include <string>
#include <vector>

#include "fa_bwd_kernel.cuh"

namespace {

struct Region {
    const char *name;
    long off;
    long bytes;
    long align;
};

int failures = 0;

void check(const std::string &label, std::vector<Region> regions, long smem)
{
    // the launch adds up to 1023 bytes of slack to align its base to 1024
    const long usable = smem - 1024;
    long end = 0;
    for (size_t i = 0; i < regions.size(); ++i) {
        const Region &r = regions[i];
        if (r.bytes <= 0)
            continue;
        if (r.off % r.align != 0) {
            std::printf("FAIL %s: %s at %ld not %ld-byte aligned\n", label.c_str(), r.name, r.off, r.align);
            ++failures;
        }
        if (r.off < end) {
            std::printf("FAIL %s: %s at %ld overlaps the region before it (ends at %ld)\n", label.c_str(), r.name, r.off,
                        end);
            ++failures;
        }
        end = r.off + r.bytes;
    }
    if (end > usable) {
        std::printf("FAIL %s: regions end at %ld, past %ld usable bytes\n", label.c_str(), end, usable);
        ++failures;
    }
    if (smem > 232448) {
        std::printf("FAIL %s: %ld bytes of shared memory, above the 232448 a CTA may have\n", label.c_str(), smem);
        ++failures;
    }
    std::printf("%-26s %7ld bytes, regions end at %7ld:", label.c_str(), smem, end);
    for (const Region &r : regions)
        if (r.bytes > 0)
            std::printf(" %s@%ld", r.name, r.off);
    std::printf("\n");
}

template <int D>
void forward(bool split)
{
    using C = fa::Cfg<D>;
    if (C::kTileBytes % 1024 != 0 || C::kBoxBytes % 1024 != 0) {
        std::printf("FAIL forward D=%d: tiles or boxes not whole 1024-byte swizzle atoms\n", D);
        ++failures;
    }
    std::vector<Region> r = {
        {"Q", C::kQOff, (long)C::kQBufs * C::kQBufBytes, 1024},
        {"K/V ring", C::kStageOff, (long)C::kStages * C::kStageBytes, 1024},
        {"barriers", C::kBarOff, (long)C::kNumBars * 8, 8},
        {"handoff", C::kHandOff, (long)fa::kQTiles * fa::kBM * 8, 8},
        {"misc", C::kMiscOff, 16, 8},
    };
    if (split) {
        r.push_back({"merge staging", C::kMergeOff, (long)fa::kMergeBufs * fa::kMergeOBytes, 128});
        r.push_back({"(m,l) staging", C::kMlOff, (long)fa::kMlBytes, 16});
        r.push_back({"jobs", C::kJobOff, (long)fa::kJobSlots * (long)sizeof(fa::MergeJob), 8});
    }
    r.push_back({"V barriers", C::vbar_off(split), (long)C::kVBarBytes, 8});
    check("forward D=" + std::to_string(D) + (split ? " balanced" : " whole"), r, C::smem_bytes(split));
}

template <int D, bool KV, bool FQ = false>
void backward()
{
    using C = fa::bwd::BCfg<D, KV, FQ>;
    std::vector<Region> r = {{"resident tiles", C::kResOff, 2L * C::kTileBytes, 1024}};
    if (C::kSplitRing) {
        r.push_back({"ring 0", C::kStageOff, (long)C::kRing0 * C::kTileBytes, 1024});
        r.push_back({"ring 1", C::kRing1Off, (long)C::kRing1 * C::kTileBytes, 1024});
    } else {
        r.push_back({"stages", C::kStageOff, (long)C::kStages * C::kStageBytes, 1024});
    }
    if (FQ) {
        r.push_back({"dS^T tile", C::kDsOff, (long)fa::bwd::kTile * fa::bwd::kTile * 2, 1024});
        r.push_back({"dQ staging", C::kDqOff, 2L * C::kDqBoxBytes, 1024});
    }
    r.push_back({"barriers", C::kBarOff, (long)C::kNumBars * 8, 8});
    r.push_back({"misc", C::kMiscOff, 16, 8});
    check("backward D=" + std::to_string(D) + (FQ ? " fused" : (KV ? " dK/dV" : " dQ")), r, C::kSmem);
}

}  // namespace

int main()
{
    forward<64>(false);
    forward<64>(true);
    forward<128>(false);
    forward<128>(true);
    backward<64, false>();
    backward<64, true>();
    backward<64, true, true>();
    backward<128, false>();
    backward<128, true>();
    if (failures == 0)
        std::printf("ok\n");
    return failures == 0 ? 0 : 1;
}
