// Weight prepack: [N, K] e4m3fn codes + [N/128, K/128] block scales -> the
// tile-major GB300 layout the fused GEMM streams with one bulk copy per tile.
//
// The page "[AMD] Small-M FP8 block-scale GEMM with fused activation quant for
// gfx950 (Qwen3.5)", "Modifications", streams a (16,16)-preshuffled weight whose
// order suits the gfx950 MFMA.  Here each 128 x 128 tile is stored as the exact
// shared-memory image of a K-major, 128-byte-swizzled tcgen05 operand: row r,
// 16-byte chunk j lands at (r/8)*1024 + (r%8)*128 + ((j ^ (r%8)) * 16).  A
// 16 KB bulk copy then puts a ready MMA operand in shared memory, and the
// tiles of one n-tile row are contiguous, so a CTA's run of units is one
// contiguous stretch of HBM.
#include "internal.cuh"

namespace fp8bs {
namespace {

__global__ void __launch_bounds__(128)
    prepack_kernel(const uint8_t* __restrict__ wq, int64_t ldw, const void* __restrict__ ws,
                   int64_t N, int64_t K, int kind, uint8_t* __restrict__ packed) {
    const int kb = blockIdx.x, nt = blockIdx.y;
    const int KB = gridDim.x;
    const int r = threadIdx.x;
    const uint4* src = reinterpret_cast<const uint4*>(wq + (static_cast<int64_t>(nt) * kTile + r) * ldw +
                                                      static_cast<int64_t>(kb) * kTile);
    uint8_t* tile = packed + kHeaderBytes + (static_cast<size_t>(nt) * KB + kb) * kTileBytes;
    uint8_t* row = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint4 v = src[j];
        *reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) * 16)) = v;
    }
    if (r == 0) {
        const size_t idx = static_cast<size_t>(nt) * KB + kb;
        uint8_t* scales = packed + packed_scales_offset(N, K);
        if (kind == FP8BS_SCALE_UE8M0)
            scales[idx] = static_cast<const uint8_t*>(ws)[idx];
        else
            reinterpret_cast<float*>(scales)[idx] = static_cast<const float*>(ws)[idx];
        if (nt == 0 && kb == 0) {
            PackedHeader h;
            h.magic = kPackedMagic;
            h.version = kPackedVersion;
            h.n = N;
            h.k = K;
            h.scale_kind = kind;
            h.tile_bytes = kTileBytes;
            *reinterpret_cast<PackedHeader*>(packed) = h;
        }
    }
}

}  // namespace

cudaError_t launch_prepack(const uint8_t* wq, int64_t ldw, const void* ws, int64_t N, int64_t K,
                           int kind, void* packed, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>(K / kTile), static_cast<unsigned>(N / kTile));
    prepack_kernel<<<grid, 128, 0, stream>>>(wq, ldw, ws, N, K, kind, static_cast<uint8_t*>(packed));
    return cudaGetLastError();
}

}  // namespace fp8bs
