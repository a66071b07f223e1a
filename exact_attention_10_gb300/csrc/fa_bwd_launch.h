// fa_bwd_launch.h -- interface between the C ABI (fa_api.cu) and the backward
// kernels' translation unit (fa_bwd.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa_launch {

struct BwdLaunch {
    CUtensorMap tq, tk, tv, tdo;   // rank-3 maps over [B*H, rows, D], 64 x 128 boxes, 128-byte swizzle
    const void *O, *dO;            // [B*H, N, D], the input type
    const float *LSE;              // [B*H, N]
    void *dQ, *dK, *dV;            // dQ [B*H, N, D], dK and dV [B*H, Nkv, D], the input type
    float *lg, *dl;                // workspace: [B*H][Npad] each
    float *dqa;                    // fused: workspace, the fp32 dQ accumulator [B*H][Npad][D]
    CUtensorMap tdqa;              // fused: rank-2 map over dqa [B*H*Npad, D], 32 x 128 boxes, 128-byte swizzle
    bool fused;                    // D = 64: one pass for dK, dV and dQ (dQ through dqa)
    int BH, N, Nkv, Npad, D, sms;   // N query rows, Nkv keys per head
    bool bf16, causal;               // causal: masked by the band below
    int wl, wr;                      // band: query i sees keys [i + Nkv - N - wl, i + Nkv - N + wr] (kSchedUnbounded: none)
    float scale;
};

// Enqueue the pre-pass, then the dQ pass and the dK/dV pass, or (fused) the
// one pass and the conversion of the dQ accumulator, on `s`.
fa_status launch_bwd(const BwdLaunch &a, cudaStream_t s, int dev);
bool take_status_word_bwd(cudaStream_t s, unsigned int *word);

}  // namespace fa_launch
