// Fused RMSNorm + 1x128 quant producer.
//
// "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense 128x128 fp8
// linears (6/8)", "Modifications": the input_norm / q_norm producers emit the
// ue8m0 1x128 activation scales themselves, so quantising the GEMM's input
// adds no launch.  Here the producer writes e4m3fn codes and fp32 or e8m0
// scales that fp8bs_gemm_prequant consumes directly, and (optionally) the bf16
// normalised row.
//
// Per row m:  r = 1 / sqrt(sum_k x[m,k]^2 / K + eps)      (fp32)
//             y[m,k] = bf16_rn((x[m,k] * r) * gamma[k])  (fp32 products)
//             xq, xs = the 1x128 quant of those bf16 values (the same rules,
//                      bit for bit, as fp8bs_quant).
//
// One CTA of 256 threads per row.  Half-warp h (16 of them) owns the groups
// h, h + 16, ...; lane l of the half holds k = 8l .. 8l+7 of each group (one
// 16-byte load), so the whole row stays in registers between the reduction
// and the quant.  The sum of squares is reduced in a fixed order (each
// thread's chunks in order, a butterfly within the warp, then the 8 warp sums
// in warp order), so every run gives the same bytes.  Memory-bound: x and
// gamma are read once, codes, scales and y written once.
#include "internal.cuh"
#include "producer.cuh"

namespace fp8bs {
namespace {

constexpr int kRnThreads = 256;
constexpr int kRnHalves = kRnThreads / 16;

// Two fp32 values -> two bf16 (nearest even), lo in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// Packed fp32 pairs (low word = first value): mul.rn.f32x2 is two independent
// IEEE multiplications, so a pair gives the same values as two scalar ones.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// J: groups per half-warp (the smallest of 1, 2, 4, 8 with 16 * J >= K / 128).
template <int KIND, int J>
__global__ void __launch_bounds__(kRnThreads)
    rmsnorm_quant_kernel(const uint16_t* __restrict__ x, int K, int64_t ldx, const uint16_t* __restrict__ gamma,
                         float eps, uint8_t* __restrict__ xq, void* __restrict__ xs, uint16_t* __restrict__ y,
                         int64_t ldy) {
    __shared__ float2 tab[kScaleTab];
    __shared__ float red[kRnThreads / 32];
    const int tid = threadIdx.x, h = tid >> 4, l16 = tid & 15;
    const int64_t m = blockIdx.x;
    const int KB = K / kTile;
    fill_scale_table(tab, tid, kRnThreads);

    // gamma is loaded with x (its latency hidden by the reduction) unless
    // that would not fit the registers (K > 8192)
    constexpr bool kEarlyGamma = J <= 4;
    uint4 raw[J], graw[kEarlyGamma ? J : 1];
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int g = h + kRnHalves * j;
        raw[j] = make_uint4(0, 0, 0, 0);
        if (g < KB) raw[j] = *reinterpret_cast<const uint4*>(x + m * ldx + g * kTile + 8 * l16);
        if constexpr (kEarlyGamma) {
            graw[j] = make_uint4(0, 0, 0, 0);
            if (g < KB) graw[j] = *reinterpret_cast<const uint4*>(gamma + g * kTile + 8 * l16);
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        float v[8];
        unpack_bf16x8(raw[j], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();  // also publishes the scale table
    float total = red[0];
#pragma unroll
    for (int w = 1; w < kRnThreads / 32; ++w) total += red[w];
    const float ms = __fdiv_rn(total, static_cast<float>(K)) + eps;
    // a zero row with eps 0 normalises to signed zeros, not NaN
    const float r = ms > 0.0f ? __frsqrt_rn(ms) : 0.0f;

    // normalise every group (the products in packed fp32 pairs: two IEEE
    // multiplications each, the same values as scalar ones), then quantise all
    // of them through the straight-line fast path so that the groups
    // interleave; a warp's rare groups are redone exactly, out of line
    uint4 nr[J];
    const uint64_t r2 = pack_f32x2(r, r);
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int g = h + kRnHalves * j;
        float v[8], gm[8];
        unpack_bf16x8(raw[j], v);
        if constexpr (kEarlyGamma) {
            unpack_bf16x8(graw[j], gm);
        } else {
            uint4 gr = make_uint4(0, 0, 0, 0);
            if (g < KB) gr = *reinterpret_cast<const uint4*>(gamma + g * kTile + 8 * l16);
            unpack_bf16x8(gr, gm);
        }
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint64_t p = mul_f32x2(mul_f32x2(pack_f32x2(v[2 * i], v[2 * i + 1]), r2),
                                         pack_f32x2(gm[2 * i], gm[2 * i + 1]));
            w[i] = pack_bf16x2(__uint_as_float(static_cast<uint32_t>(p)), __uint_as_float(static_cast<uint32_t>(p >> 32)));
        }
        nr[j] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    SliceQuant qs[J];
    bool rare[J];
#pragma unroll
    for (int j = 0; j < J; ++j) qs[j] = quant_slice_fast<KIND>(nr[j], tab, rare[j]);
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (__any_sync(0xFFFFFFFFu, rare[j])) {  // all 32 lanes take part
            const SliceQuant e = quant_slice_exact<KIND>(nr[j], tab);
            if (rare[j]) qs[j] = e;
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int g = h + kRnHalves * j;
        if (g < KB) {
            if (y) *reinterpret_cast<uint4*>(y + m * ldy + g * kTile + 8 * l16) = nr[j];
            *reinterpret_cast<uint2*>(xq + m * K + g * kTile + 8 * l16) = make_uint2(qs[j].lo, qs[j].hi);
            if (l16 == 0) {
                if (KIND == FP8BS_SCALE_UE8M0)
                    static_cast<uint8_t*>(xs)[m * KB + g] = static_cast<uint8_t>(qs[j].byte);
                else
                    static_cast<float*>(xs)[m * KB + g] = qs[j].scale;
            }
        }
    }
}

template <int KIND, int J>
cudaError_t launch_rn(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma, float eps,
                      uint8_t* xq, void* xs, uint16_t* y, int64_t ldy, cudaStream_t stream) {
    rmsnorm_quant_kernel<KIND, J><<<static_cast<unsigned>(M), kRnThreads, 0, stream>>>(
        x, static_cast<int>(K), ldx, gamma, eps, xq, xs, y, ldy);
    return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_rn_kind(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma,
                           float eps, uint8_t* xq, void* xs, uint16_t* y, int64_t ldy, cudaStream_t stream) {
    const int64_t halves = (K / kTile + kRnHalves - 1) / kRnHalves;
    if (halves <= 1) return launch_rn<KIND, 1>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
    if (halves <= 2) return launch_rn<KIND, 2>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
    if (halves <= 4) return launch_rn<KIND, 4>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
    return launch_rn<KIND, 8>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
}

}  // namespace

cudaError_t launch_rmsnorm_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma,
                                 float eps, int kind, uint8_t* xq, void* xs, uint16_t* y, int64_t ldy,
                                 cudaStream_t stream) {
    if (M < 1) return cudaSuccess;
    if (kind == FP8BS_SCALE_UE8M0)
        return launch_rn_kind<FP8BS_SCALE_UE8M0>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
    return launch_rn_kind<FP8BS_SCALE_F32>(x, M, K, ldx, gamma, eps, xq, xs, y, ldy, stream);
}

}  // namespace fp8bs
