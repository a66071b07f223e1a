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
    int BH, N, Nkv, Npad, D, sms;   // N query rows, Nkv keys per head
    bool bf16, causal;               // causal: masked by the band below
    int wl, wr;                      // band: query i sees keys [i + Nkv - N - wl, i + Nkv - N + wr] (kSchedUnbounded: none)
    float scale;
};

// Enqueue the pre-pass, the dQ pass and the dK/dV pass on `s`.
fa_status launch_bwd(const BwdLaunch &a, cudaStream_t s, int dev);
bool take_status_word_bwd(cudaStream_t s, unsigned int *word);

}  // namespace fa_launch
