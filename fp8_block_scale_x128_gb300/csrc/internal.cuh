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

// Workspace layout (bytes).  The CTAs of one fused launch exchange their
// split-K partials through it: each partial value travels as a 64-bit word,
// 32 data bits and the call's 32-bit epoch, so a reader sees either an older
// word or the new one and needs no flag.  Words left by earlier calls carry
// older epochs, so nothing is cleared between calls.  Every region sits at a
// place that depends on sm_count only, never on N or K, so a workspace serves
// calls of any shape without a word of one call ever being taken for one of
// another.
//   [0, 256)                  device error word
//   [256, +4 KB)              epoch words, one per possible CTA index
//   then sm_count x 2 x 64 KB split-K partial slots: per CTA index one for the
//                             first and one for the last n-tile of its range,
//                             each [64 columns][128 rows] of tagged words
//   then 64 x K + 64 x K/128 x 4  codes and scales of the routed two-launch
//                             path (33 to 64 tokens) when the caller does not
//                             ask for them
constexpr size_t kWsErrorBytes = 256;
constexpr int kMaxCtas = 1024;  // epoch words; bound on the grid
constexpr size_t kWsGenBytes = kMaxCtas * sizeof(uint32_t);
constexpr size_t kSlotWords = 64 * 128;
constexpr size_t kSlotBytes = kSlotWords * sizeof(uint64_t);
constexpr int kSlotsPerCta = 2;

__host__ __device__ constexpr size_t ws_gen_offset() { return kWsErrorBytes; }
__host__ __device__ constexpr size_t ws_partials_offset() { return kWsErrorBytes + kWsGenBytes; }
__host__ __device__ constexpr size_t ws_act_offset(int sm_count) {
    return ws_partials_offset() + static_cast<size_t>(sm_count) * kSlotsPerCta * kSlotBytes;
}
__host__ __device__ constexpr size_t ws_total_bytes(int sm_count, int64_t K) {
    return ws_act_offset(sm_count) + static_cast<size_t>(FP8BS_MAX_M) * static_cast<size_t>(K) +
           static_cast<size_t>(FP8BS_MAX_M) * static_cast<size_t>(K / kTile) * sizeof(float);
}

// Largest token count the fused kernel quantises itself (its 16- and
// 32-token tiles; measured faster than the quant kernel + GEMM pair at every
// token count up to 32); fp8bs_gemm_fused runs larger calls as the quant,
// then the GEMM on its codes.
constexpr int kFusedMaxM = 32;

// Units of work (128x128 weight tiles) one CTA of the fused kernel owns at most.
constexpr int kMaxUnitsM16 = 12;
constexpr int kMaxUnitsM32 = 10;
constexpr int kMaxUnitsM64 = 10;

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

// Codes of the IEEE quotients RN32(v / scale) for the 8 bf16 values in raw.
// Scale table.  A group maximum amax is a bf16 value m * 2^e with
// m = 1 + i/128 (7 mantissa bits), so its scale RN32(amax / 448) equals
// RN32(m / 448) * 2^e and the reciprocal RN32(1 / scale) equals
// RN32(1 / RN32(m / 448)) * 2^-e -- exactly, while both are normal numbers
// (biased exponent of amax >= 10).  tab[i] = {RN32(m / 448), RN32(1 / that)},
// built with IEEE division by every block before it quantises.
constexpr int kScaleTab = 128;

__device__ __forceinline__ void fill_scale_table(float2* tab, int t, int nthreads) {
    for (int i = t; i < kScaleTab; i += nthreads) {
        const float m = 1.0f + static_cast<float>(i) * (1.0f / 128.0f);  // exact
        const float sm = __fdiv_rn(m, 448.0f);
        tab[i] = make_float2(sm, __frcp_rn(sm));
    }
}

// Result of quantising one 16-byte slice (8 values) of a 1x128 group.
struct SliceQuant {
    uint32_t lo, hi;  // 8 codes, little-endian (the slice's first value in bits 0-7 of lo)
    float scale;      // the group scale (fp32; for ue8m0 the power of two)
    uint32_t byte;    // ue8m0: the e8m0 byte of the scale
};

// Quantise one 1x128 group held by 16 consecutive lanes, 8 consecutive bf16
// values per lane (lane l of the half-warp holds k = 8l .. 8l+7).  All 32
// lanes of the warp must call it (each half-warp holds its own group).
//
// The codes are those of RN32(x / scale), computed without a division:
// from the correctly rounded reciprocal r = RN32(1 / scale), q0 = RN32(x r),
// the remainder x - q0 scale (an fma, exact), and q = RN32(q0 + remainder r)
// (an fma) is the correctly rounded quotient -- the division step of P.
// Markstein, "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990, which needs the reciprocal
// correctly rounded and no intermediate to over- or underflow.  A group whose
// amax is below 2^-60 is first multiplied by 2^64 (exact: the values are bf16,
// far from the top of the range), its scale too, so no remainder that can
// decide a code is subnormal; x / scale is unchanged.  (Quotients below
// 2^-10 round to a zero code whatever their last bits.)  ue8m0 scales are
// powers of two, so there x * (1 / scale) is the quotient itself.
template <int KIND>
__device__ __forceinline__ SliceQuant quant_slice(uint4 raw, const float2* __restrict__ tab) {
    float v[8];
    unpack_bf16x8(raw, v);
    const float m0 = fmaxf(fabsf(v[0]), fabsf(v[1])), m1 = fmaxf(fabsf(v[2]), fabsf(v[3]));
    const float m2 = fmaxf(fabsf(v[4]), fabsf(v[5])), m3 = fmaxf(fabsf(v[6]), fabsf(v[7]));
    const uint32_t mine = __float_as_uint(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
    // half-warp maxima (non-negative floats order like their bit patterns)
    const bool low_half = (threadIdx.x & 31u) < 16u;
    const uint32_t g0 = __reduce_max_sync(0xFFFFFFFFu, low_half ? mine : 0u);
    const uint32_t g1 = __reduce_max_sync(0xFFFFFFFFu, low_half ? 0u : mine);
    const uint32_t amax_bits = low_half ? g0 : g1;
    const float amax = __uint_as_float(amax_bits);
    SliceQuant out;
    out.byte = 0;
    if (amax_bits == 0) {
        // zero group: scale 0 (ue8m0: byte 0) and the signed zeros of x
        out.scale = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(0u) : 0.0f;
        out.lo = ((raw.x >> 15) & 1u) << 7 | ((raw.x >> 31) & 1u) << 15 | ((raw.y >> 15) & 1u) << 23 |
                 ((raw.y >> 31) & 1u) << 31;
        out.hi = ((raw.z >> 15) & 1u) << 7 | ((raw.z >> 31) & 1u) << 15 | ((raw.w >> 15) & 1u) << 23 |
                 ((raw.w >> 31) & 1u) << 31;
        return out;
    }
    const uint32_t e_biased = amax_bits >> 23;
    float s, recip;
    const bool normal_scale = e_biased >= 10u;
    if (normal_scale) {
        const float2 t = tab[(amax_bits >> 16) & 0x7Fu];
        const int shift = (static_cast<int>(e_biased) - 127) * (1 << 23);
        s = __int_as_float(__float_as_int(t.x) + shift);
        recip = __int_as_float(__float_as_int(t.y) - shift);
    } else {  // amax < 2^-117: the scale is subnormal, its reciprocal set below
        s = __fdiv_rn(amax, 448.0f);
        recip = 0.0f;
    }
    float sx = s, rx = recip;  // the scale and reciprocal the quotients use
    if (KIND == FP8BS_SCALE_UE8M0) {
        out.byte = e8m0_ceil_byte(s);
        out.scale = e8m0_to_float(out.byte);
        rx = e8m0_to_float(254u - out.byte);  // 2^(127 - e): exact
    } else {
        out.scale = s;
        if (!(amax >= 0x1p-60f)) {  // tiny group: work on x 2^64 (uniform per half-warp)
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] *= 0x1p64f;  // exact; signs kept
            sx = s * 0x1p64f;                              // exact, normal
            rx = normal_scale ? recip * 0x1p-64f : __frcp_rn(sx);
        }
    }
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = v[j] * rx;
        // the correction gives +0 for x = -0 (0 + -0 rounds to +0): the
        // quotient keeps the sign of x, which copysign restores
        if (KIND == FP8BS_SCALE_F32) a[j] = copysignf(fmaf(fmaf(-a[j], sx, v[j]), rx, a[j]), v[j]);
    }
    out.lo = e4m3x2(a[0], a[1]) | (e4m3x2(a[2], a[3]) << 16);
    out.hi = e4m3x2(a[4], a[5]) | (e4m3x2(a[6], a[7]) << 16);
    return out;
}

// quant_slice kept out of line: the exact path for the rare groups of a caller
// that quantises through quant_slice_fast.  One copy of its code instead of
// one per group in the caller's unrolled rounds, which keeps the hot round
// code compact in the instruction cache.  All 32 lanes call it.
template <int KIND>
__device__ __noinline__ SliceQuant quant_slice_exact(uint4 raw, const float2* __restrict__ tab) {
    return quant_slice<KIND>(raw, tab);
}

// The common case of quant_slice without a branch, for callers that quantise
// several groups at once: exact (the same codes and scale as quant_slice) for
// a group whose amax is at least 2^-60, where the scale is normal, its
// reciprocal comes from the table and no rescaling is needed.  rare is set for
// every other group (zero, tiny, subnormal scale, or NaN amax): the caller
// takes that group's result from quant_slice instead.  Being straight-line
// code, the calls for independent groups interleave.  All 32 lanes call it.
template <int KIND>
__device__ __forceinline__ SliceQuant quant_slice_fast(uint4 raw, const float2* __restrict__ tab, bool& rare) {
    float v[8];
    unpack_bf16x8(raw, v);
    const float m0 = fmaxf(fabsf(v[0]), fabsf(v[1])), m1 = fmaxf(fabsf(v[2]), fabsf(v[3]));
    const float m2 = fmaxf(fabsf(v[4]), fabsf(v[5])), m3 = fmaxf(fabsf(v[6]), fabsf(v[7]));
    const uint32_t mine = __float_as_uint(fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)));
    const bool low_half = (threadIdx.x & 31u) < 16u;
    const uint32_t g0 = __reduce_max_sync(0xFFFFFFFFu, low_half ? mine : 0u);
    const uint32_t g1 = __reduce_max_sync(0xFFFFFFFFu, low_half ? 0u : mine);
    const uint32_t amax_bits = low_half ? g0 : g1;
    rare = !(__uint_as_float(amax_bits) >= 0x1p-60f);
    // scale and reciprocal from the table, shifted by the exponent of amax
    // (unsigned arithmetic: a rare group's values are discarded)
    const float2 t = tab[(amax_bits >> 16) & 0x7Fu];
    const uint32_t shift = ((amax_bits >> 23) - 127u) << 23;
    const float s = __uint_as_float(__float_as_uint(t.x) + shift);
    float rx = __uint_as_float(__float_as_uint(t.y) - shift);
    SliceQuant out;
    if (KIND == FP8BS_SCALE_UE8M0) {
        // the smallest power of two >= s, s normal: its e8m0 byte, clamped
        const uint32_t b = __float_as_uint(s);
        const uint32_t byte = min((b >> 23) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u), 254u);
        out.byte = byte;
        out.scale = __uint_as_float(byte << 23);
        rx = __uint_as_float(byte == 254u ? 0x00400000u : (254u - byte) << 23);  // 2^(127 - e): exact
    } else {
        out.byte = 0;
        out.scale = s;
    }
    float a[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        a[j] = v[j] * rx;
        if (KIND == FP8BS_SCALE_F32) a[j] = copysignf(fmaf(fmaf(-a[j], s, v[j]), rx, a[j]), v[j]);
    }
    out.lo = e4m3x2(a[0], a[1]) | (e4m3x2(a[2], a[3]) << 16);
    out.hi = e4m3x2(a[4], a[5]) | (e4m3x2(a[6], a[7]) << 16);
    return out;
}

// ---------------------------------------------------------------------------
// Launchers (argument checks are done by the C ABI before these run)
// ---------------------------------------------------------------------------

cudaError_t launch_encode_e4m3(const float* v, int64_t n, uint8_t* codes, cudaStream_t stream);
// pdl: launched with programmatic dependent launch (the kernel lets its
// dependent start at once and waits for its predecessor before reading x).
cudaError_t launch_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int kind,
                         uint8_t* xq, void* xs, cudaStream_t stream, bool pdl = false);
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
    int pdl;
    // the two-launch path: pre-quantised activations instead of x (x unused)
    const uint8_t* xq_in = nullptr;  // [M][ldxq] e4m3 codes
    int64_t ldxq = 0;
    const void* xs_in = nullptr;     // [M][K/128] fp32 or e8m0 scales
};

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream);

// Whether the fused GEMM supports an N x K weight on sm_count SMs: one CTA per
// SM at most, so the K blocks of one n-tile must fit the resident units of
// all SMs.
bool fused_shape_supported(int64_t N, int64_t K, int sm_count);

}  // namespace fp8bs
