// Launcher of the fused RMSNorm + 1x128 quant producer (rmsnorm_quant.cu).
// Argument checks are done by the C ABI before it runs.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace fp8bs {

cudaError_t launch_rmsnorm_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma,
                                 float eps, int kind, uint8_t* xq, void* xs, uint16_t* y, int64_t ldy,
                                 cudaStream_t stream);

}  // namespace fp8bs
