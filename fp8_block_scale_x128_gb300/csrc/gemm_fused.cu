// Fused small-M W8A8 FP8 block-scale linear for sm_103a.
//
// What it computes ("[AMD] Small-M FP8 block-scale GEMM with fused activation
// quant for gfx950 (Qwen3.5)", "Modifications"):
//   xq, xs = 1x128-group quant of bf16 x (row amax, scale, e4m3fn codes)
//   Y[m,n] = bf16( sum_kb P[n,m,kb] * (xs[m,kb] * ws[n/128,kb]) ),
//   P[n,m,kb] = sum_{k in kb} wq[n,k] * xq[m,k]
// in one launch.  The page's gfx950 design (per-wave MFMA over a preshuffled
// weight, LDS reduction) is prior art; this is the GB300 form of the same idea.
//
// Work unit: one (n-tile of 128 weight rows, 128-wide K block) = one 16 KB fp8
// weight tile.  The T = N/128 * K/128 units, in n-major order, are split evenly
// over a grid of (normally) one CTA per SM ("stream-K"): CTA c owns units
// [c*T/G, (c+1)*T/G).  Every CTA:
//   1. issues a bulk async copy (TMA, evict-first) for EVERY weight tile it
//      owns at once -- the whole share (at most 10-12 tiles) fits in shared
//      memory, so the HBM stream starts in the first microsecond;
//   2. meanwhile quantises the activation columns of its units into the
//      shared-memory B operands (K-major, 128-byte swizzle), with bit-exact
//      scales and codes;
//   3. one thread issues, per unit, four tcgen05.mma kind::f8f6f4 (K = 32 each)
//      with the weight tile as the 128-row A operand and the tokens as
//      N = 16 or 32 ("swap-AB"), into a TMEM accumulator of its own;
//   4. four epilogue warps (one per 32 TMEM lanes) read each unit's fp32
//      128 x N block, multiply by xs[m,kb] * ws[nt,kb] in fp32 and accumulate
//      in registers (the per-K-block rescale of the page);
//   5. a run of units that covers a whole n-tile writes bf16 Y directly; a
//      partial n-tile is written as an fp32 partial to the workspace, and the
//      last CTA to arrive (per-tile counter) sums all partials of that tile in
//      CTA order -- a fixed order, so results are deterministic -- and writes
//      bf16 Y.  No CTA ever waits for another.
// Every mbarrier wait is bounded; on expiry the kernel records
// FP8BS_ERR_TIMEOUT in the workspace error word, drains its own copies and
// MMAs (again bounded), frees TMEM and returns.
#include "internal.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int kThreads = 256;  // 8 warps: producer, MMA, scales/header, -, 4 epilogue

template <int MPAD>
struct Cfg {
    static constexpr int kUnits = MPAD == 16 ? kMaxUnitsM16 : kMaxUnitsM32;
    static constexpr uint32_t kBBytes = MPAD * 128;  // activation operand of one unit
    static constexpr uint32_t kTmemCols = MPAD == 16 ? 256 : 512;
    static constexpr uint32_t kOffW = 0;
    static constexpr uint32_t kOffB = kOffW + kUnits * kTileBytes;
    static constexpr uint32_t kOffXs = kOffB + kUnits * kBBytes;
    static constexpr uint32_t kOffWs = kOffXs + kUnits * MPAD * 4;
    static constexpr uint32_t kOffBar = (kOffWs + kUnits * 4 + 7) / 8 * 8;
    static constexpr uint32_t kOffMisc = kOffBar + 2 * kUnits * 8;
    static constexpr uint32_t kSmem = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
    // 16-byte slices of x per thread: units * MPAD rows * 16 slices / threads
    static constexpr int kSlices = (kUnits * MPAD * 16 + kThreads - 1) / kThreads;
    static_assert(kUnits * MPAD <= static_cast<int>(kTmemCols), "TMEM columns");
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(kBBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
};

struct Params {
    const uint16_t* x;
    int64_t ldx;
    const uint8_t* packed;
    const uint8_t* tiles;
    const uint8_t* wscales;
    int M, N, K, KB, kind;
    int64_t T;
    uint16_t* y;
    int64_t ldy;
    uint32_t* err;
    uint32_t* counters;
    float* partials;
    uint8_t* xq_out;
    void* xs_out;
    long long timeout;
};

enum : int { kMiscTmem = 0, kMiscAbort = 1, kMiscHdrOk = 2, kMiscIssued = 3 };

__device__ __forceinline__ int64_t unit_begin(int64_t c, int64_t T, int64_t G) { return c * T / G; }

// The CTA whose unit range holds unit u (inverse of unit_begin).
__device__ __forceinline__ int64_t cta_of(int64_t u, int64_t T, int64_t G) {
    return ((u + 1) * G + T - 1) / T - 1;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// Bounded wait by a single thread.  Returns false when the deadline passes
// (recording FP8BS_ERR_TIMEOUT and raising the CTA's abort flag) or, with
// honour_abort, when another role has already raised it.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, long long timeout, volatile uint32_t* misc,
                           uint32_t* err, bool honour_abort) {
    const long long t0 = clock64();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (honour_abort && misc[kMiscAbort] != 0) return false;
        if (clock64() - t0 > timeout) {
            record_error(err, FP8BS_ERR_TIMEOUT);
            misc[kMiscAbort] = 1;
            return false;
        }
    }
}

template <int MPAD>
__device__ __forceinline__ void store_y(const Params& p, int n, const float (&v)[MPAD]) {
#pragma unroll
    for (int m = 0; m < MPAD; ++m)
        if (m < p.M) p.y[m * p.ldy + n] = f32_to_bf16_rn(v[m]);
}

// Output of one n-tile's accumulator by one epilogue warp (rows q*32 .. +31).
template <int MPAD>
__device__ void flush_tile(const Params& p, int64_t nt, const float (&acc)[MPAD], int64_t c, int64_t G,
                           int64_t u0, int64_t u1, int q, int lane) {
    const int r = q * 32 + lane;
    const int n = static_cast<int>(nt * kTile + r);
    const int64_t t0 = nt * p.KB, t1 = t0 + p.KB;
    if (u0 <= t0 && u1 >= t1) {  // this CTA owns the whole K range of the tile
        store_y<MPAD>(p, n, acc);
        return;
    }
    const int M4 = (p.M + 3) >> 2;
    const int slot = (nt == u0 / p.KB) ? 0 : 1;
    float4* part = reinterpret_cast<float4*>(p.partials + (c * 2 + slot) * kPartialSlotFloats + r * MPAD);
#pragma unroll
    for (int j = 0; j < MPAD / 4; ++j)
        if (j < M4) part[j] = make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
    __threadfence();
    __syncwarp();
    const int64_t first = cta_of(t0, p.T, G), last = cta_of(t1 - 1, p.T, G);
    uint32_t is_last = 0;
    if (lane == 0) {
        const uint32_t prev = atomicAdd(&p.counters[nt * 4 + q], 1u);
        is_last = prev == static_cast<uint32_t>(last - first) ? 1u : 0u;
    }
    is_last = __shfl_sync(0xFFFFFFFFu, is_last, 0);
    if (!is_last) return;
    __threadfence();
    float sum[MPAD];
#pragma unroll
    for (int m = 0; m < MPAD; ++m) sum[m] = 0.0f;
    for (int64_t cc = first; cc <= last; ++cc) {  // fixed order: deterministic
        const int s2 = (nt == unit_begin(cc, p.T, G) / p.KB) ? 0 : 1;
        const float4* pp =
            reinterpret_cast<const float4*>(p.partials + (cc * 2 + s2) * kPartialSlotFloats + r * MPAD);
#pragma unroll
        for (int j = 0; j < MPAD / 4; ++j) {
            if (j < M4) {
                const float4 v = __ldcg(pp + j);
                sum[4 * j] += v.x;
                sum[4 * j + 1] += v.y;
                sum[4 * j + 2] += v.z;
                sum[4 * j + 3] += v.w;
            }
        }
    }
    store_y<MPAD>(p, n, sum);
    if (lane == 0) p.counters[nt * 4 + q] = 0;  // ready for the next launch
}

template <int MPAD, int KIND>
__global__ void __launch_bounds__(kThreads, 1) fused_quant_gemm_kernel(const Params p) {
    using C = Cfg<MPAD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem + C::kOffW;
    uint8_t* sB = smem + C::kOffB;
    float* sXs = reinterpret_cast<float*>(smem + C::kOffXs);
    float* sWs = reinterpret_cast<float*>(smem + C::kOffWs);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* accf = full + C::kUnits;
    volatile uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t u0 = unit_begin(c, p.T, G), u1 = unit_begin(c + 1, p.T, G);
    const int cnt = static_cast<int>(u1 - u0);

    // ---- set-up: barriers, TMEM ------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < cnt; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&accf[i], 1);
        }
        misc[kMiscAbort] = 0;
        misc[kMiscHdrOk] = 0;
        misc[kMiscIssued] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(const_cast<uint32_t*>(&misc[kMiscTmem]), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[kMiscTmem];

    // ---- 1. weight stream: every tile of this CTA in flight at once ------------
    if (tid == 0) {
        const uint64_t pol = ptx::policy_evict_first();
        for (int i = 0; i < cnt; ++i) {
            ptx::mbar_arrive_expect_tx(&full[i], kTileBytes);
            ptx::bulk_g2s(sW + i * kTileBytes, p.tiles + (u0 + i) * kTileBytes, kTileBytes, &full[i], pol);
        }
    }
    // weight block scales of the units; packed-weight header check
    if (warp == 2) {
        if (lane < cnt) {
            const int64_t u = u0 + lane;
            sWs[lane] = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(p.wscales[u])
                                                  : reinterpret_cast<const float*>(p.wscales)[u];
        }
        if (lane == 0) {
            const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
            const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->n == p.N &&
                            h->k == p.K && h->scale_kind == p.kind && h->tile_bytes == kTileBytes;
            if (!ok) record_error(p.err, FP8BS_ERR_SCALE_KIND);
            misc[kMiscHdrOk] = ok ? 1u : 0u;
        }
    }

    // ---- 2. activation quant into the B operands ------------------------------
    {
        uint4 raw[C::kSlices];
#pragma unroll
        for (int j = 0; j < C::kSlices; ++j) {
            const int s = tid + kThreads * j;
            const int g = s >> 4, part = s & 15;
            const int i = g / MPAD, m = g % MPAD;
            raw[j] = make_uint4(0, 0, 0, 0);
            if (i < cnt && m < p.M) {
                const int kb = static_cast<int>((u0 + i) % p.KB);
                raw[j] = __ldg(reinterpret_cast<const uint4*>(p.x + m * p.ldx + kb * kTile + part * 8));
            }
        }
#pragma unroll
        for (int j = 0; j < C::kSlices; ++j) {
            const int s = tid + kThreads * j;
            const int g = s >> 4, part = s & 15;
            const int i = g / MPAD, m = g % MPAD;
            float v[8];
            unpack_bf16x8(raw[j], v);
            float sf;
            uint32_t sb = 0;
            const uint2 codes = quant_group_16lanes<KIND>(v, &sf, &sb);  // padded rows -> zeros
            if (i < cnt) {
                uint8_t* row = sB + i * C::kBBytes + (m >> 3) * 1024 + (m & 7) * 128;
                *reinterpret_cast<uint2*>(row + (((part >> 1) ^ (m & 7)) << 4) + ((part & 1) << 3)) = codes;
                if (part == 0) sXs[i * MPAD + m] = sf;
                const int64_t u = u0 + i;
                if (m < p.M && u < p.KB) {  // n-tile 0's unit for this kb publishes xq / xs
                    if (p.xq_out)
                        *reinterpret_cast<uint2*>(p.xq_out + static_cast<int64_t>(m) * p.K + u * kTile + part * 8) =
                            codes;
                    if (p.xs_out && part == 0) {
                        if (KIND == FP8BS_SCALE_UE8M0)
                            static_cast<uint8_t*>(p.xs_out)[m * p.KB + u] = static_cast<uint8_t>(sb);
                        else
                            static_cast<float*>(p.xs_out)[m * p.KB + u] = sf;
                    }
                }
            }
        }
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();

    if (warp == 1) {
        // ---- 3. MMA issue (one thread) -------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_f8f6f4_e4m3(128, MPAD);
            int issued = 0;
            for (int i = 0; i < cnt; ++i) {
                if (!wait_phase(&full[i], 0, p.timeout, misc, p.err, true)) break;
                ptx::tc_fence_after();
                const uint32_t a = ptx::smem_addr(sW + i * kTileBytes);
                const uint32_t b = ptx::smem_addr(sB + i * C::kBBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ptx::mma_f8f6f4(tmem + i * MPAD, ptx::smem_desc_sw128(a + 32 * k),
                                    ptx::smem_desc_sw128(b + 32 * k), idesc, k > 0 ? 1u : 0u);
                ptx::mma_commit(&accf[i]);
                issued = i + 1;
            }
            misc[kMiscIssued] = issued;
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---- 4./5. rescale-accumulate and output ---------------------------------
        const int q = warp & 3;
        const bool hdr_ok = misc[kMiscHdrOk] != 0;
        float acc[MPAD];
#pragma unroll
        for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
        int64_t cur = u0 / p.KB;
        bool ok = true;
        for (int i = 0; i < cnt; ++i) {
            const int64_t nt = (u0 + i) / p.KB;
            if (nt != cur) {
                if (hdr_ok) flush_tile<MPAD>(p, cur, acc, c, G, u0, u1, q, lane);
#pragma unroll
                for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
                cur = nt;
            }
            uint32_t done = 0;
            if (lane == 0) done = wait_phase(&accf[i], 0, p.timeout, misc, p.err, true) ? 1u : 0u;
            done = __shfl_sync(0xFFFFFFFFu, done, 0);
            if (!done) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(i * MPAD);
            uint32_t r0[16], r1[16];
            ptx::tmem_ld_32x32b_x16(taddr, r0);
            if constexpr (MPAD == 32) ptx::tmem_ld_32x32b_x16(taddr + 16, r1);
            ptx::tmem_wait_ld();
            const float sw = sWs[i];
#pragma unroll
            for (int m = 0; m < 16; ++m) acc[m] = fmaf(__uint_as_float(r0[m]), sXs[i * MPAD + m] * sw, acc[m]);
            if constexpr (MPAD == 32) {
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    acc[16 + m] = fmaf(__uint_as_float(r1[m]), sXs[i * MPAD + 16 + m] * sw, acc[16 + m]);
            }
        }
        if (ok && hdr_ok) flush_tile<MPAD>(p, cur, acc, c, G, u0, u1, q, lane);
    }

    // ---- teardown -------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (misc[kMiscAbort] != 0) {
        // drain this CTA's own copies and MMAs before its shared memory and
        // TMEM go away (bounded as well)
        if (tid == 0) {
            for (int i = 0; i < cnt; ++i) wait_phase(&full[i], 0, p.timeout, misc, p.err, false);
            const int issued = static_cast<int>(misc[kMiscIssued]);
            for (int i = 0; i < issued; ++i) wait_phase(&accf[i], 0, p.timeout, misc, p.err, false);
        }
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int MPAD, int KIND>
cudaError_t launch_impl(const Params& p, int sm_count, cudaStream_t stream) {
    using C = Cfg<MPAD>;
    auto kern = fused_quant_gemm_kernel<MPAD, KIND>;
    // Opt in to the large dynamic shared memory once per device (not a stream
    // operation, so it is harmless during graph capture too).
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = 1;
    }
    const int G = fused_grid(p.T, sm_count, C::kUnits);
    kern<<<G, kThreads, C::kSmem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream) {
    Params p;
    p.x = a.x;
    p.ldx = a.ldx;
    p.packed = a.packed;
    p.tiles = a.packed + kHeaderBytes;
    p.wscales = a.packed + packed_scales_offset(a.N, a.K);
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = a.K / kTile;
    p.kind = a.kind;
    p.T = static_cast<int64_t>(a.N / kTile) * (a.K / kTile);
    p.y = a.y;
    p.ldy = a.ldy;
    p.err = reinterpret_cast<uint32_t*>(a.workspace);
    p.counters = reinterpret_cast<uint32_t*>(a.workspace + ws_counters_offset());
    p.partials = reinterpret_cast<float*>(a.workspace + ws_partials_offset());
    p.xq_out = a.xq_out;
    p.xs_out = a.xs_out;
    p.timeout = a.timeout_cycles;
    const bool small = a.M <= 16;
    if (a.kind == FP8BS_SCALE_UE8M0)
        return small ? launch_impl<16, FP8BS_SCALE_UE8M0>(p, a.sm_count, stream)
                     : launch_impl<32, FP8BS_SCALE_UE8M0>(p, a.sm_count, stream);
    return small ? launch_impl<16, FP8BS_SCALE_F32>(p, a.sm_count, stream)
                 : launch_impl<32, FP8BS_SCALE_F32>(p, a.sm_count, stream);
}

// Largest grid any variant uses for this shape (sizes the workspace).
int fused_max_grid(int64_t N, int64_t K, int sm_count) {
    const int64_t T = (N / kTile) * (K / kTile);
    const int g16 = fused_grid(T, sm_count, kMaxUnitsM16);
    const int g32 = fused_grid(T, sm_count, kMaxUnitsM32);
    return g16 > g32 ? g16 : g32;
}

}  // namespace fp8bs
