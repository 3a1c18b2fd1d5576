// Shared definitions of the fp8bs CUDA library: packed-weight and workspace
// layouts, the device-side 1x128 quantiser, and the launchers the C ABI calls.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fp8bs.h"

namespace fp8bs {

constexpr int kTile = 128;                  // rows (n) and columns (k) of one weight tile
constexpr uint32_t kTileBytes = 128 * 128;  // e4m3 bytes of one tile
constexpr size_t kHeaderBytes = 256;        // packed-weight header
constexpr uint32_t kPackedMagic = 0x53423846u;  // "F8BS"
constexpr uint32_t kPackedVersion = 1;

// Header at the start of a packed weight.
struct PackedHeader {
    uint32_t magic;
    uint32_t version;
    int64_t n;
    int64_t k;
    int32_t scale_kind;
    uint32_t tile_bytes;
};

__host__ __device__ inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline size_t packed_scales_offset(int64_t N, int64_t K) {
    return kHeaderBytes + static_cast<size_t>(N / kTile) * static_cast<size_t>(K / kTile) * kTileBytes;
}

// Workspace: [0, 256) error word (+ pad); [256, 256 + 32 KB) one u32 arrival
// counter per (n-tile, 32-row quarter) -- a fixed region, so one workspace can
// serve weights of any shape; then the split-K partial tiles, one 128 x 32
// fp32 slot per (CTA, first/last n-tile of that CTA).
constexpr size_t kWsErrorBytes = 256;
constexpr size_t kWsCounterBytes = 32768;
constexpr int64_t kMaxFusedN = static_cast<int64_t>(kWsCounterBytes / (4 * sizeof(uint32_t))) * 128;
constexpr size_t kPartialSlotFloats = 128 * 32;

__host__ __device__ inline size_t ws_counters_offset() { return kWsErrorBytes; }
__host__ __device__ inline size_t ws_partials_offset() { return kWsErrorBytes + kWsCounterBytes; }

// Units of work per CTA the fused kernel keeps resident in shared memory.
constexpr int kMaxUnitsM16 = 12;
constexpr int kMaxUnitsM32 = 10;

// Grid of the fused kernel for T = (N/128) * (K/128) units on sm_count SMs:
// one CTA per SM when every CTA's share fits in shared memory, otherwise as
// many CTAs as needed.  Units are split evenly (stream-K over n-major order).
__host__ __device__ inline int fused_grid(int64_t T, int sm_count, int max_units) {
    int64_t g = T < sm_count ? T : sm_count;
    if (g < 1) g = 1;
    int64_t need = (T + max_units - 1) / max_units;
    if (need > g) g = need;
    return static_cast<int>(g);
}

// Device error word: 0, or the negated status of the first fault.
__device__ inline void record_error(uint32_t* err, int status) {
    if (err) atomicCAS(err, 0u, static_cast<uint32_t>(-status));
}

// ---------------------------------------------------------------------------
// Device-side quantiser pieces (bit-exact rules shared by every kernel)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

// Two fp32 values -> two e4m3fn codes, round to nearest even, saturating to
// +-448 (satfinite).  Returns lo's code in bits 0-7 and hi's in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The e8m0 byte of the smallest power of two >= s (s >= 0 finite), exponent
// clamped to [-127, 127]; s == 0 -> 0.
__device__ __forceinline__ uint32_t e8m0_ceil_byte(float s) {
    uint32_t b = __float_as_uint(s);
    uint32_t ef = b >> 23;
    uint32_t mant = b & 0x7FFFFFu;
    if (b == 0) return 0;
    if (ef == 0) return mant > (1u << 22) ? 1u : 0u;  // subnormal: 2^-126 or clamp to 2^-127
    uint32_t byte = ef + (mant != 0 ? 1u : 0u);
    return byte > 254u ? 254u : byte;
}

__device__ __forceinline__ float e8m0_to_float(uint32_t byte) {
    return byte == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(byte << 23);
}

// Quantise one 1x128 group held by 16 consecutive lanes, 8 consecutive values
// per lane (lane l of the half-warp holds k = 8l .. 8l+7).  Returns the 8 codes
// packed little-endian (value 8l in bits 0-7 of .x), and the scale in
// *scale_f32 (for ue8m0 also the byte in *scale_byte).  All 32 lanes of the
// warp must call it (the two half-warps hold two independent groups).
template <int KIND>
__device__ __forceinline__ uint2 quant_group_16lanes(const float (&v)[8], float* scale_f32,
                                                     uint32_t* scale_byte) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float s = __fdiv_rn(amax, 448.0f);
    float scale = s;
    if (KIND == FP8BS_SCALE_UE8M0) {
        const uint32_t byte = e8m0_ceil_byte(s);
        *scale_byte = byte;
        scale = e8m0_to_float(byte);
    }
    *scale_f32 = scale;
    uint2 c;
    if (amax == 0.0f) {
        // zero group: the signed zeros of x, no division
        c.x = c.y = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c.x |= (__float_as_uint(v[j]) >> 31) << (8 * j + 7);
            c.y |= (__float_as_uint(v[j + 4]) >> 31) << (8 * j + 7);
        }
        return c;
    }
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = __fdiv_rn(v[j], scale);
    c.x = e4m3x2(q[0], q[1]) | (e4m3x2(q[2], q[3]) << 16);
    c.y = e4m3x2(q[4], q[5]) | (e4m3x2(q[6], q[7]) << 16);
    return c;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float (&v)[8]) {
    v[0] = bf16_bits_to_float(raw.x & 0xFFFFu);
    v[1] = bf16_bits_to_float(raw.x >> 16);
    v[2] = bf16_bits_to_float(raw.y & 0xFFFFu);
    v[3] = bf16_bits_to_float(raw.y >> 16);
    v[4] = bf16_bits_to_float(raw.z & 0xFFFFu);
    v[5] = bf16_bits_to_float(raw.z >> 16);
    v[6] = bf16_bits_to_float(raw.w & 0xFFFFu);
    v[7] = bf16_bits_to_float(raw.w >> 16);
}

// ---------------------------------------------------------------------------
// Launchers (argument checks are done by the C ABI before these run)
// ---------------------------------------------------------------------------

cudaError_t launch_encode_e4m3(const float* v, int64_t n, uint8_t* codes, cudaStream_t stream);
cudaError_t launch_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int kind,
                         uint8_t* xq, void* xs, cudaStream_t stream);
cudaError_t launch_quant_weight(const float* w, int64_t N, int64_t K, int64_t ldw, int kind,
                                uint8_t* wq, void* ws, cudaStream_t stream);
cudaError_t launch_prepack(const uint8_t* wq, int64_t ldw, const void* ws, int64_t N, int64_t K,
                           int kind, void* packed, cudaStream_t stream);

struct FusedArgs {
    const uint16_t* x;
    int64_t ldx;
    const uint8_t* packed;
    int M, N, K;
    int kind;
    uint16_t* y;
    int64_t ldy;
    uint8_t* workspace;
    uint8_t* xq_out;
    void* xs_out;
    int sm_count;
    long long timeout_cycles;
};

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream);

// Largest grid the fused kernel uses for an N x K weight on sm_count SMs.
int fused_max_grid(int64_t N, int64_t K, int sm_count);

}  // namespace fp8bs
