// Standalone quantisers.
//
// quant_1x128_kernel: bf16 activations -> e4m3fn codes + one scale per 1x128
// group ("[AMD] Small-M FP8 block-scale GEMM with fused activation quant for
// gfx950 (Qwen3.5)", "Modifications": row amax per 1x128 group via lane
// shuffles; the first of the two launches the fused kernel replaces).  Half a
// warp per group, 8 values (one 16-byte load) per lane; memory-bound, no
// tensor-core work.
//
// quant_weight_kernel: fp32 weights -> e4m3fn codes + one scale per 128x128
// block (the producer of the [N/128, K/128] weight_scale_inv of the same page;
// power-of-two scales per "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for
// dense 128x128 fp8 linears (6/8)", "Motivation").
#include "internal.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int kQuantWarps = 8;

// Two groups per warp: half-warp h of warp w takes group 2w + h; lane l of the
// half holds k = 8l .. 8l+7 (one 16-byte load).
template <int KIND>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quant_1x128_kernel(const uint16_t* __restrict__ x, int M, int K, int64_t ldx,
                       uint8_t* __restrict__ xq, void* __restrict__ xs, int pdl) {
    __shared__ float2 tab[kScaleTab];
    fill_scale_table(tab, threadIdx.x, kQuantWarps * 32);
    // programmatic dependent launch: let the next kernel (the GEMM on these
    // codes) start its prologue now; wait for the kernel before (the producer
    // of x) before the first read of x
    if (pdl) {
        ptx::griddep_launch_dependents();
        ptx::griddep_wait();
    }
    __syncthreads();
    const int l16 = threadIdx.x & 15;
    const int KB = K / kTile;
    const int64_t groups = static_cast<int64_t>(M) * KB;
    const int64_t half0 = static_cast<int64_t>(blockIdx.x) * (kQuantWarps * 2) + (threadIdx.x >> 4);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (kQuantWarps * 2);
    // every lane runs the same trip count so the shuffles stay converged
    const int64_t trips = (groups + stride - 1) / stride;
    for (int64_t t = 0; t < trips; ++t) {
        const int64_t g = half0 + t * stride;
        const bool valid = g < groups;
        const int m = valid ? static_cast<int>(g / KB) : 0;
        const int kb = valid ? static_cast<int>(g % KB) : 0;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (valid) raw = *reinterpret_cast<const uint4*>(x + m * ldx + kb * kTile + 8 * l16);
        const SliceQuant qs = quant_slice<KIND>(raw, tab);
        const uint2 codes = make_uint2(qs.lo, qs.hi);
        const float sf = qs.scale;
        const uint32_t sb = qs.byte;
        if (valid) {
            *reinterpret_cast<uint2*>(xq + static_cast<int64_t>(m) * K + kb * kTile + 8 * l16) = codes;
            if (l16 == 0) {
                if (KIND == FP8BS_SCALE_UE8M0)
                    static_cast<uint8_t*>(xs)[g] = static_cast<uint8_t>(sb);
                else
                    static_cast<float*>(xs)[g] = sf;
            }
        }
    }
}

// One CTA per 128x128 block; thread t covers row t/2, columns (t%2)*64 .. +63.
template <int KIND>
__global__ void __launch_bounds__(256)
    quant_weight_kernel(const float* __restrict__ w, int K, int64_t ldw, uint8_t* __restrict__ wq,
                        void* __restrict__ ws) {
    __shared__ float red[8];
    const int kb = blockIdx.x, nb = blockIdx.y, KB = gridDim.x;
    const int t = threadIdx.x;
    const int r = t >> 1, c0 = (t & 1) * 64;
    const float* src = w + (static_cast<int64_t>(nb) * kTile + r) * ldw + kb * kTile + c0;
    float4 v[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = reinterpret_cast<const float4*>(src)[i];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if ((t & 31) == 0) red[t >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float s = __fdiv_rn(amax, 448.0f);
    float scale = s;
    uint32_t byte = 0;
    if (KIND == FP8BS_SCALE_UE8M0) {
        byte = e8m0_ceil_byte(s);
        scale = e8m0_to_float(byte);
    }
    uint8_t* dst = wq + (static_cast<int64_t>(nb) * kTile + r) * K + kb * kTile + c0;
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        uint32_t word[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 q = v[i + j];
            if (amax == 0.0f) {
                word[j] = ((__float_as_uint(q.x) >> 31) << 7) | ((__float_as_uint(q.y) >> 31) << 15) |
                          ((__float_as_uint(q.z) >> 31) << 23) | ((__float_as_uint(q.w) >> 31) << 31);
            } else {
                word[j] = e4m3x2(__fdiv_rn(q.x, scale), __fdiv_rn(q.y, scale)) |
                          (e4m3x2(__fdiv_rn(q.z, scale), __fdiv_rn(q.w, scale)) << 16);
            }
        }
        reinterpret_cast<uint4*>(dst)[i / 4] = make_uint4(word[0], word[1], word[2], word[3]);
    }
    if (t == 0) {
        if (KIND == FP8BS_SCALE_UE8M0)
            static_cast<uint8_t*>(ws)[nb * KB + kb] = static_cast<uint8_t>(byte);
        else
            static_cast<float*>(ws)[nb * KB + kb] = scale;
    }
}

// Four values per thread, grid-stride.
__global__ void __launch_bounds__(256)
    encode_e4m3_kernel(const float4* __restrict__ v, int64_t n4, uint32_t* __restrict__ codes) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 q = v[i];
        codes[i] = e4m3x2(q.x, q.y) | (e4m3x2(q.z, q.w) << 16);
    }
}

}  // namespace

cudaError_t launch_encode_e4m3(const float* v, int64_t n, uint8_t* codes, cudaStream_t stream) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) return cudaSuccess;
    encode_e4m3_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const float4*>(v), n4, reinterpret_cast<uint32_t*>(codes));
    return cudaGetLastError();
}

cudaError_t launch_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int kind,
                         uint8_t* xq, void* xs, cudaStream_t stream, bool pdl) {
    const int64_t groups = M * (K / kTile);
    int64_t blocks = (groups + 2 * kQuantWarps - 1) / (2 * kQuantWarps);
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kQuantWarps * 32);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int pdl_flag = pdl ? 1 : 0;
    if (kind == FP8BS_SCALE_UE8M0)
        return cudaLaunchKernelEx(&cfg, quant_1x128_kernel<FP8BS_SCALE_UE8M0>, x, static_cast<int>(M),
                                  static_cast<int>(K), ldx, xq, xs, pdl_flag);
    return cudaLaunchKernelEx(&cfg, quant_1x128_kernel<FP8BS_SCALE_F32>, x, static_cast<int>(M), static_cast<int>(K),
                              ldx, xq, xs, pdl_flag);
}

cudaError_t launch_quant_weight(const float* w, int64_t N, int64_t K, int64_t ldw, int kind,
                                uint8_t* wq, void* ws, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>(K / kTile), static_cast<unsigned>(N / kTile));
    if (kind == FP8BS_SCALE_UE8M0)
        quant_weight_kernel<FP8BS_SCALE_UE8M0><<<grid, 256, 0, stream>>>(w, static_cast<int>(K), ldw, wq, ws);
    else
        quant_weight_kernel<FP8BS_SCALE_F32><<<grid, 256, 0, stream>>>(w, static_cast<int>(K), ldw, wq, ws);
    return cudaGetLastError();
}

}  // namespace fp8bs
