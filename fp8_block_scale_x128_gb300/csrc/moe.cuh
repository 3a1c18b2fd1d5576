// Launcher of the small-M FP8 block-scale MoE layer (moe.cu).  Argument checks
// are done by the C ABI before it runs.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fp8bs.h"

namespace fp8bs {

constexpr size_t kMoeWsHeader = 256;  // the device error word, then the partial sums

struct MoeArgs {
    const uint16_t* x;
    const int32_t* ids;
    const float* tw;
    const uint8_t* w13;
    const float* s13;
    const uint8_t* w2;
    const float* s2;
    uint16_t* y;
    uint8_t* workspace;
    int M, S, H, I, E;
    int sm_count;
};

size_t moe_workspace_bytes(int64_t M, int64_t S, int64_t H, int64_t I);
cudaError_t launch_moe(const MoeArgs& a, cudaStream_t stream);

}  // namespace fp8bs
