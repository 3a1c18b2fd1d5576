// Fused small-M W8A8 FP8 block-scale linear for sm_103a.
//
// What it computes ("[AMD] Small-M FP8 block-scale GEMM with fused activation
// quant for gfx950 (Qwen3.5)", "Modifications"):
//   xq, xs = 1x128-group quant of bf16 x (row amax, scale, e4m3fn codes)
//   Y[m,n] = bf16( sum_kb P[n,m,kb] * (xs[m,kb] * ws[n/128,kb]) ),
//   P[n,m,kb] = sum_{k in kb} wq[n,k] * xq[m,k]
// in one launch.  The page's gfx950 design (per-wave MFMA over a preshuffled
// weight, each wave quantising its own activations, LDS reduction) is prior
// art; this is the GB300 form of the same computation.
//
// Work unit: one (n-tile of 128 weight rows, 128-wide K block) = one 16 KB fp8
// weight tile.  The T = N/128 * K/128 units, in n-major order, are split evenly
// over at most one CTA per SM ("stream-K"): CTA c owns units [c*T/G, (c+1)*T/G)
// -- at most 10-12, all resident in shared memory -- and all CTAs of the grid
// are resident at once.  Every CTA:
//   1. issues a bulk async copy (TMA, evict-first) for EVERY weight tile it
//      owns at once, so the HBM stream starts in the first microsecond;
//   2. gets the quantised activations of its units' K blocks into the
//      shared-memory B operands (K-major, 128-byte swizzle):
//        - up to 8 tokens it quantises them itself (M x units groups);
//        - above that every CTA quantises 1/G of all M x K/128 groups and
//          publishes them in the workspace as 64-bit (4 codes, epoch) words,
//          and each CTA copies the words of its units' K blocks -- the
//          quantisation is then done once per group instead of once per CTA;
//   3. two threads (warps 1 and 3) issue, per unit, four tcgen05.mma
//      kind::f8f6f4 (K = 32 each) with the weight tile as the 128-row A
//      operand and the tokens as N = 16 or 32 ("swap-AB"), each unit into a
//      TMEM accumulator of its own;
//   4. four epilogue warps (one per 32 TMEM lanes) read each unit's fp32
//      128 x N block, multiply by xs[m,kb] * ws[nt,kb] in fp32 and accumulate
//      in registers (the per-K-block rescale of the page);
//   5. an n-tile whose whole K range the CTA owns is written as bf16 Y.
//      Otherwise the CTA holding the tile's first unit reduces it: the other
//      contributors publish their fp32 partials as (value, epoch) words and
//      exit; the reducer sums its own and their partials in CTA order -- a
//      fixed order, so results are deterministic -- and writes bf16 Y.
// A call's epoch is one more than the workspace's epoch word for the CTA's
// index, and every CTA moves the words of its index class on to it when it
// ends, so all words stay equal and every word written by an earlier call
// carries an older epoch.
// With programmatic dependent launch the next call's CTAs start while this
// one finishes: everything before griddepcontrol.wait reads only the packed
// weight; x, y and the workspace are touched after it.
// Every wait is bounded; on expiry the kernel records FP8BS_ERR_TIMEOUT in the
// workspace error word, drains its own copies and MMAs (again bounded), frees
// TMEM and returns.
#include "internal.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// 8 warps.  Warp 0: weight copies (one thread), then quant.  Warps 1 and 3:
// MMA issue (even / odd units); warp 3 first builds the scale table.  Warp 2:
// unit info and header check, then quant.  Warps 4-7: quant, then the
// epilogue (one warp per 32 TMEM lanes).
constexpr int kThreads = 256;
constexpr int kQuantThreads = kThreads - 64;  // all warps but the two MMA warps
constexpr int kQuantHalfWarps = kQuantThreads / 16;
constexpr int kLocalMaxM = 8;  // up to this many tokens every CTA quantises its own groups

__device__ __forceinline__ bool is_mma_warp(int warp) { return warp == 1 || warp == 3; }
// index of a quantising thread: warps 0, 2, 4, 5, 6, 7 -> 0 .. kQuantThreads-1
__device__ __forceinline__ int quant_index(int tid) {
    const int warp = tid >> 5;
    return warp == 0 ? tid : warp == 2 ? tid - 32 : tid - 64;
}

template <int MPAD, bool DIST>
struct Cfg {
    static constexpr int kUnits = MPAD == 16 ? kMaxUnitsM16 : kMaxUnitsM32;
    static constexpr int kRows = DIST ? MPAD : kLocalMaxM;  // largest M of this variant
    static constexpr uint32_t kBBytes = MPAD * 128;  // activation operand of one unit
    static constexpr uint32_t kTmemCols = MPAD == 16 ? 256 : 512;
    static constexpr uint32_t kOffW = 0;
    static constexpr uint32_t kOffB = kOffW + kUnits * kTileBytes;
    static constexpr uint32_t kOffXs = kOffB + kUnits * kBBytes;
    static constexpr uint32_t kOffWs = kOffXs + kUnits * MPAD * 4;
    static constexpr uint32_t kOffKb = kOffWs + kUnits * 4;
    static constexpr uint32_t kOffTab = (kOffKb + kUnits * 4 + 15) / 16 * 16;
    static constexpr uint32_t kOffBar = kOffTab + kScaleTab * 8;
    static constexpr uint32_t kOffMisc = kOffBar + 3 * kUnits * 8 + 8;  // + the header barrier
    static constexpr uint32_t kSmem = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
    // 16-byte activation slices per quantising thread: units * rows * 16
    static constexpr int kSlices = (kUnits * kRows * 16 + kQuantThreads - 1) / kQuantThreads;
    // scale words per quantising thread (exchange variant): units * rows
    static constexpr int kScaleSlices = (kUnits * kRows + kQuantThreads - 1) / kQuantThreads;
    static_assert(kUnits * MPAD <= static_cast<int>(kTmemCols), "TMEM columns");
    static_assert(kSmem <= 232448, "shared memory per CTA");
    static_assert(kBBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
};

struct Params {
    const uint16_t* x;
    int64_t ldx;
    const uint8_t* packed;    // header
    const uint8_t* tiles;     // first tile of this launch's n-tiles
    const uint8_t* wscales;   // first block scale of this launch's n-tiles
    int M, N, K, KB, kind;    // N, K of the whole weight
    uint32_t T;               // units of this launch
    uint64_t mdiv;            // ceil(2^32 / M): index -> (quotient, remainder) by M
    uint16_t* y;              // column 0 of this launch's n-tiles
    int64_t ldy;
    uint32_t* err;
    uint32_t* gen;            // epoch words
    uint64_t* ll;             // split-K slots: [grid][128 rows][32 cols] (value, epoch)
    uint64_t* xsw;            // activation scales: [K/128][32 rows] (scale bits, epoch)
    uint64_t* xqw;            // activation codes: [K/128][32 rows][32] (4 codes, epoch)
    uint8_t* xq_out;
    void* xs_out;
    long long timeout;
    int pdl;
};

enum : int { kMiscTmem = 0, kMiscAbort = 1, kMiscHdrOk = 2, kMiscIssued = 3 };

__device__ __forceinline__ uint32_t unit_begin(uint32_t c, uint32_t T, uint32_t G) {
    return static_cast<uint32_t>(static_cast<uint64_t>(c) * T / G);
}

// The CTA whose unit range holds unit u (inverse of unit_begin).
__device__ __forceinline__ uint32_t cta_of(uint32_t u, uint32_t T, uint32_t G) {
    return static_cast<uint32_t>((static_cast<uint64_t>(u + 1) * G + T - 1) / T - 1);
}

__device__ __forceinline__ uint32_t div_m(uint32_t g, uint64_t mdiv) { return static_cast<uint32_t>((g * mdiv) >> 32); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ void st_pair(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

__device__ __forceinline__ void st_word(uint64_t* p, uint64_t a) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}

__device__ __forceinline__ void ld_pair(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
    uint64_t a;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}

__device__ __forceinline__ uint32_t ld_u32_gpu(const uint32_t* p) {
    uint32_t a;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(a) : "l"(p) : "memory");
    return a;
}

__device__ __forceinline__ uint64_t tag(uint32_t data, uint32_t epoch) {
    return static_cast<uint64_t>(data) | (static_cast<uint64_t>(epoch) << 32);
}

__device__ __forceinline__ bool tagged(uint64_t w, uint32_t epoch) { return static_cast<uint32_t>(w >> 32) == epoch; }

__device__ __forceinline__ bool timed_out(long long t0, long long timeout, volatile uint32_t* misc, uint32_t* err) {
    if (misc[kMiscAbort] != 0) return true;
    if (clock64() - t0 > timeout) {
        record_error(err, FP8BS_ERR_TIMEOUT);
        misc[kMiscAbort] = 1;
        return true;
    }
    return false;
}

// Bounded wait by a single thread.  Returns false when the deadline passes
// (recording FP8BS_ERR_TIMEOUT and raising the CTA's abort flag) or, with
// honour_abort, when another role has already raised it.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, long long timeout,
                                        volatile uint32_t* misc, uint32_t* err, bool honour_abort) {
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

struct WordPair {
    uint64_t a, b;
    bool ok;
};

// Re-reads a pair of exchange words (first read: a, b) until both carry the
// epoch (bounded; .ok false on expiry).  All by value: nothing goes through
// memory.
__device__ __noinline__ WordPair poll_pair(const uint64_t* p, uint64_t a, uint64_t b, uint32_t epoch,
                                           long long timeout, volatile uint32_t* misc, uint32_t* err) {
    const long long t0 = clock64();
    WordPair r{a, b, true};
    while (!(tagged(r.a, epoch) && tagged(r.b, epoch))) {
        if (timed_out(t0, timeout, misc, err)) {
            r.ok = false;
            return r;
        }
        ld_pair(p, r.a, r.b);
    }
    return r;
}

// The same for a single word.
__device__ __noinline__ WordPair poll_word(const uint64_t* p, uint64_t a, uint32_t epoch, long long timeout,
                                           volatile uint32_t* misc, uint32_t* err) {
    const long long t0 = clock64();
    WordPair r{a, 0, true};
    while (!tagged(r.a, epoch)) {
        if (timed_out(t0, timeout, misc, err)) {
            r.ok = false;
            return r;
        }
        r.a = ld_word(p);
    }
    return r;
}

template <int MPAD>
__device__ __forceinline__ void store_y(const Params& p, int n, const float (&v)[MPAD]) {
#pragma unroll
    for (int m = 0; m < MPAD; ++m)
        if (m < p.M) p.y[m * p.ldy + n] = f32_to_bf16_rn(v[m]);
}

// Output of one n-tile's accumulator by one epilogue warp (rows q*32 .. +31).
// role 0: this CTA owns the tile's whole K range -> bf16 Y.
// role 1: a later contributor -> publish the partial in this CTA's slot.
// role 2: the reducer -> wait for the other contributors' partials, sum in CTA
//         order, bf16 Y.
template <int MPAD>
__device__ __forceinline__ void flush_tile(const Params& p, uint32_t nt, const float (&acc)[MPAD], uint32_t c,
                                           uint32_t G, int role, int q, int lane, uint32_t epoch,
                                           volatile uint32_t* misc) {
    const int r = q * 32 + lane;
    const int n = static_cast<int>(nt) * kTile + r;
    const int pairs = (p.M + 1) >> 1;
    if (role == 0) {
        store_y<MPAD>(p, n, acc);
        return;
    }
    if (role == 1) {
        uint64_t* slot = p.ll + (static_cast<size_t>(c) * 128 + r) * 32;
#pragma unroll
        for (int j = 0; j < MPAD / 2; ++j)
            if (j < pairs)
                st_pair(slot + 2 * j, tag(__float_as_uint(acc[2 * j]), epoch),
                        tag(__float_as_uint(acc[2 * j + 1]), epoch));
        return;
    }
    float sum[MPAD];
#pragma unroll
    for (int m = 0; m < MPAD; ++m) sum[m] = acc[m];
    const uint32_t last = cta_of((nt + 1) * static_cast<uint32_t>(p.KB) - 1, p.T, G);
    for (uint32_t cc = c + 1; cc <= last; ++cc) {  // fixed order: deterministic
        const uint64_t* slot = p.ll + (static_cast<size_t>(cc) * 128 + r) * 32;
        uint64_t w[MPAD];
#pragma unroll
        for (int j = 0; j < MPAD / 2; ++j) {  // all words of this contributor in flight at once
            if (j < pairs) ld_pair(slot + 2 * j, w[2 * j], w[2 * j + 1]);
            else w[2 * j] = w[2 * j + 1] = tag(0, epoch);
        }
#pragma unroll
        for (int j = 0; j < MPAD / 2; ++j) {
            if (j < pairs && !(tagged(w[2 * j], epoch) && tagged(w[2 * j + 1], epoch))) {
                const WordPair rr = poll_pair(slot + 2 * j, w[2 * j], w[2 * j + 1], epoch, p.timeout, misc, p.err);
                if (!rr.ok) return;
                w[2 * j] = rr.a;
                w[2 * j + 1] = rr.b;
            }
        }
#pragma unroll
        for (int m = 0; m < MPAD; ++m) sum[m] += __uint_as_float(static_cast<uint32_t>(w[m]));
    }
    store_y<MPAD>(p, n, sum);
}

// Store one quantised slice (unit i, row m, 16-byte part l16) into the B
// operand, the group scale into sXs, then arrive on unit i's barrier.
template <int MPAD>
__device__ __forceinline__ void put_slice(uint8_t* sB, float* sXs, uint64_t* bready, int i, int m, int l16,
                                          uint32_t lo, uint32_t hi, float scale, bool with_scale) {
    uint8_t* row = sB + i * (MPAD * 128) + (m >> 3) * 1024 + (m & 7) * 128;
    *reinterpret_cast<uint2*>(row + (((l16 >> 1) ^ (m & 7)) << 4) + ((l16 & 1) << 3)) = make_uint2(lo, hi);
    if (with_scale) sXs[i * MPAD + m] = scale;
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(&bready[i]);
}

template <int KIND>
__device__ __forceinline__ void put_xq_out(const Params& p, uint32_t m, uint32_t kb, int l16, const SliceQuant& qs) {
    if (p.xq_out)
        *reinterpret_cast<uint2*>(p.xq_out + static_cast<int64_t>(m) * p.K + kb * kTile + l16 * 8) =
            make_uint2(qs.lo, qs.hi);
    if (p.xs_out && l16 == 0) {
        if (KIND == FP8BS_SCALE_UE8M0)
            static_cast<uint8_t*>(p.xs_out)[m * p.KB + kb] = static_cast<uint8_t>(qs.byte);
        else
            static_cast<float*>(p.xs_out)[m * p.KB + kb] = qs.scale;
    }
}

template <int MPAD, int KIND, bool DIST>
__global__ void __launch_bounds__(kThreads, 1) fused_quant_gemm_kernel(const Params p) {
    using C = Cfg<MPAD, DIST>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sW = smem + C::kOffW;
    uint8_t* sB = smem + C::kOffB;
    float* sXs = reinterpret_cast<float*>(smem + C::kOffXs);
    float* sWs = reinterpret_cast<float*>(smem + C::kOffWs);
    int* sKb = reinterpret_cast<int*>(smem + C::kOffKb);
    float2* sTab = reinterpret_cast<float2*>(smem + C::kOffTab);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* accf = full + C::kUnits;
    uint64_t* bready = accf + C::kUnits;
    uint64_t* hdr_bar = bready + C::kUnits;  // completes once misc[kMiscHdrOk] is written
    volatile uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t u0 = unit_begin(c, p.T, G), u1 = unit_begin(c + 1, p.T, G);
    const int cnt = static_cast<int>(u1 - u0);
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    const uint32_t nt0 = u0 / KB, kb0 = u0 - nt0 * KB;

    // ---- set-up: barriers, TMEM, scale table, per-unit K block and weight scale
    if (tid == 0) {
        // arrivals per unit: one per 16-byte code slice, plus one per scale word
        // when the activations come through the workspace
        const uint32_t arrivals = static_cast<uint32_t>(p.M) * (DIST ? 17 : 16);
        for (int i = 0; i < cnt; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&accf[i], 1);
            ptx::mbar_init(&bready[i], arrivals);
        }
        ptx::mbar_init(hdr_bar, 1);
        misc[kMiscAbort] = 0;
        misc[kMiscHdrOk] = 0;
        misc[kMiscIssued] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(const_cast<uint32_t*>(&misc[kMiscTmem]), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == 3) fill_scale_table(sTab, lane, 32);
    if (warp == 2 && lane < cnt) {
        uint32_t kb = kb0 + lane;
        while (kb >= KB) kb -= KB;
        sKb[lane] = static_cast<int>(kb);
        const uint32_t u = u0 + lane;
        sWs[lane] = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(p.wscales[u])
                                              : reinterpret_cast<const float*>(p.wscales)[u];
    }
    if (p.pdl) ptx::griddep_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[kMiscTmem];

    // ---- 1. weight stream: every tile of this CTA in flight at once ------------
    if (tid == 0) {
        const uint64_t pol = ptx::policy_evict_first();
        for (int i = 0; i < cnt; ++i) {
            ptx::mbar_arrive_expect_tx(&full[i], kTileBytes);
            ptx::bulk_g2s(sW + i * kTileBytes, p.tiles + static_cast<size_t>(u0 + i) * kTileBytes, kTileBytes,
                          &full[i], pol);
        }
    }
    if (warp == 2 && lane == 0) {  // packed-weight header check
        const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
        const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->n == p.N && h->k == p.K &&
                        h->scale_kind == p.kind && h->tile_bytes == kTileBytes;
        misc[kMiscHdrOk] = ok ? 1u : 0u;
        ptx::mbar_arrive(hdr_bar);  // release: the epilogue reads the flag after waiting here
    }
    // Everything below may read what the previous kernel on the stream wrote.
    if (p.pdl) ptx::griddep_wait();
    if (warp == 2 && lane == 0 && misc[kMiscHdrOk] == 0) record_error(p.err, FP8BS_ERR_SCALE_KIND);

    uint32_t epoch = 0;
    if (!is_mma_warp(warp)) {
        const int qt = quant_index(tid);
        const int qw = qt >> 5;
        const int l16 = qt & 15;
        if constexpr (!DIST) {
            // ---- 2. quantise this CTA's own units' groups ------------------------
            // slice s = (unit i, row m, part l16), s = qt + kQuantThreads * j;
            // all loads in flight first, then two slices at a time.
            const int slices = cnt * p.M * 16;
            uint4 raw[C::kSlices + 1];
#pragma unroll
            for (int j = 0; j < C::kSlices + 1; ++j) {
                const int sl = qt + kQuantThreads * j;
                raw[j] = make_uint4(0, 0, 0, 0);
                if (j < C::kSlices && sl < slices) {
                    const uint32_t g = static_cast<uint32_t>(sl) >> 4;
                    const int i = static_cast<int>(div_m(g, p.mdiv));
                    const int m = static_cast<int>(g) - i * p.M;
                    raw[j] = __ldg(reinterpret_cast<const uint4*>(p.x + m * p.ldx + sKb[i] * kTile + l16 * 8));
                }
            }
            epoch = ld_u32_gpu(p.gen + c) + 1;
#pragma unroll
            for (int j = 0; j < C::kSlices; j += 2) {
                if (kQuantThreads * j + qw * 32 < slices) {  // warp-uniform: the reductions need all lanes
                    const SliceQuant q0 = quant_slice<KIND>(raw[j], sTab);
                    const SliceQuant q1 = quant_slice<KIND>(raw[j + 1], sTab);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int sl = qt + kQuantThreads * (j + h);
                        const SliceQuant& qs = h == 0 ? q0 : q1;
                        if (j + h < C::kSlices && sl < slices) {
                            const uint32_t g = static_cast<uint32_t>(sl) >> 4;
                            const int i = static_cast<int>(div_m(g, p.mdiv));
                            const int m = static_cast<int>(g) - i * p.M;
                            if (u0 + i < KB) put_xq_out<KIND>(p, m, sKb[i], l16, qs);  // n-tile 0 publishes xq / xs
                            put_slice<MPAD>(sB, sXs, bready, i, m, l16, qs.lo, qs.hi, qs.scale, l16 == 0);
                        }
                    }
                }
            }
        } else {
            // ---- 2a. this CTA's share of all groups: quantise, publish ----------
            // group g = kb * M + m; half-warp h takes g0 + h, g0 + h + 12, ...
            const uint32_t NG = static_cast<uint32_t>(p.M) * KB;
            const uint32_t g0 = unit_begin(c, NG, G), g1 = unit_begin(c + 1, NG, G);
            const int hw = qt >> 4;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (g0 + hw < g1) {
                const uint32_t g = g0 + hw;
                const uint32_t kb = div_m(g, p.mdiv), m = g - kb * static_cast<uint32_t>(p.M);
                raw = *reinterpret_cast<const uint4*>(p.x + m * p.ldx + kb * kTile + l16 * 8);
            }
            epoch = ld_u32_gpu(p.gen + c) + 1;
            for (uint32_t base = g0; base + qw * 2 < g1; base += kQuantHalfWarps) {  // warp-uniform
                const uint32_t g = base + hw;
                const bool valid = g < g1;
                const uint32_t kb = div_m(g, p.mdiv), m = g - kb * static_cast<uint32_t>(p.M);
                if (base != g0 && valid) raw = *reinterpret_cast<const uint4*>(p.x + m * p.ldx + kb * kTile + l16 * 8);
                const SliceQuant qs = quant_slice<KIND>(valid ? raw : make_uint4(0, 0, 0, 0), sTab);
                if (valid) {
                    const size_t row = static_cast<size_t>(kb) * 32 + m;
                    st_pair(p.xqw + row * 32 + 2 * l16, tag(qs.lo, epoch), tag(qs.hi, epoch));
                    const uint32_t sbits = KIND == FP8BS_SCALE_UE8M0 ? qs.byte : __float_as_uint(qs.scale);
                    if (l16 == 0) st_word(p.xsw + row, tag(sbits, epoch));
                    put_xq_out<KIND>(p, m, kb, l16, qs);
                }
            }
            // ---- 2b. the codes and scales of this CTA's units into shared memory
            // code slice (unit i, row m, part l16); scale slice (unit i, row m):
            // all loads in flight first, then each is re-read until it carries
            // this call's epoch.
            const int slices = cnt * p.M * 16;
            const int sslices = cnt * p.M;
            uint64_t w[C::kSlices][2];
#pragma unroll
            for (int j = 0; j < C::kSlices; ++j) {
                const int sl = qt + kQuantThreads * j;
                w[j][0] = w[j][1] = 0;
                if (sl < slices) {
                    const uint32_t g = static_cast<uint32_t>(sl) >> 4;
                    const int i = static_cast<int>(div_m(g, p.mdiv));
                    const int m = static_cast<int>(g) - i * p.M;
                    ld_pair(p.xqw + (static_cast<size_t>(sKb[i]) * 32 + m) * 32 + 2 * l16, w[j][0], w[j][1]);
                }
            }
            uint64_t sw[C::kScaleSlices];
#pragma unroll
            for (int j = 0; j < C::kScaleSlices; ++j) {
                const int sl = qt + kQuantThreads * j;
                sw[j] = 0;
                if (sl < sslices) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(sl), p.mdiv));
                    const int m = sl - i * p.M;
                    sw[j] = ld_word(p.xsw + static_cast<size_t>(sKb[i]) * 32 + m);
                }
            }
#pragma unroll
            for (int j = 0; j < C::kSlices; ++j) {
                const int sl = qt + kQuantThreads * j;
                if (sl < slices) {
                    const uint32_t g = static_cast<uint32_t>(sl) >> 4;
                    const int i = static_cast<int>(div_m(g, p.mdiv));
                    const int m = static_cast<int>(g) - i * p.M;
                    bool ok = true;
                    if (!(tagged(w[j][0], epoch) && tagged(w[j][1], epoch))) {
                        const uint64_t* src = p.xqw + (static_cast<size_t>(sKb[i]) * 32 + m) * 32 + 2 * l16;
                        const WordPair r = poll_pair(src, w[j][0], w[j][1], epoch, p.timeout, misc, p.err);
                        ok = r.ok;
                        w[j][0] = r.a;
                        w[j][1] = r.b;
                    }
                    if (ok)
                        put_slice<MPAD>(sB, sXs, bready, i, m, l16, static_cast<uint32_t>(w[j][0]),
                                        static_cast<uint32_t>(w[j][1]), 0.0f, false);
                }
            }
#pragma unroll
            for (int j = 0; j < C::kScaleSlices; ++j) {
                const int sl = qt + kQuantThreads * j;
                if (sl < sslices) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(sl), p.mdiv));
                    const int m = sl - i * p.M;
                    bool ok = true;
                    if (!tagged(sw[j], epoch)) {
                        const uint64_t* src = p.xsw + static_cast<size_t>(sKb[i]) * 32 + m;
                        const WordPair r = poll_word(src, sw[j], epoch, p.timeout, misc, p.err);
                        ok = r.ok;
                        sw[j] = r.a;
                    }
                    if (ok) {
                        const uint32_t bits = static_cast<uint32_t>(sw[j]);
                        sXs[i * MPAD + m] = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(bits) : __uint_as_float(bits);
                        ptx::mbar_arrive(&bready[i]);
                    }
                }
            }
        }
    } else {
        epoch = ld_u32_gpu(p.gen + c) + 1;
    }

    if (is_mma_warp(warp)) {
        // ---- 3. MMA issue: lane 0 of warp 1 takes the even units, of warp 3 the odd
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_f8f6f4_e4m3(128, MPAD);
            for (int i = warp == 1 ? 0 : 1; i < cnt; i += 2) {
                if (!wait_phase(&bready[i], 0, p.timeout, misc, p.err, true)) break;
                if (!wait_phase(&full[i], 0, p.timeout, misc, p.err, true)) break;
                ptx::tc_fence_after();
                const uint32_t a = ptx::smem_addr(sW + i * kTileBytes);
                const uint32_t b = ptx::smem_addr(sB + i * C::kBBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ptx::mma_f8f6f4(tmem + i * MPAD, ptx::smem_desc_sw128(a + 32 * k),
                                    ptx::smem_desc_sw128(b + 32 * k), idesc, k > 0 ? 1u : 0u);
                ptx::mma_commit(&accf[i]);
                atomicOr(const_cast<uint32_t*>(&misc[kMiscIssued]), 1u << i);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---- 4./5. rescale-accumulate and output ---------------------------------
        const int q = warp & 3;
        uint32_t hdr = 0;
        if (lane == 0) hdr = wait_phase(hdr_bar, 0, p.timeout, misc, p.err, true) && misc[kMiscHdrOk] != 0;
        const bool hdr_ok = __shfl_sync(0xFFFFFFFFu, hdr, 0) != 0;
        float acc[MPAD];
#pragma unroll
        for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
        uint32_t cur = nt0, kb = kb0;
        for (int i = 0; i < cnt; ++i) {
            uint32_t done = 0;
            if (lane == 0)  // the MMA completion, and the operand barrier that published sXs[i]
                done = (wait_phase(&accf[i], 0, p.timeout, misc, p.err, true) &&
                        wait_phase(&bready[i], 0, p.timeout, misc, p.err, true)) ? 1u : 0u;
            done = __shfl_sync(0xFFFFFFFFu, done, 0);
            if (!done) break;
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
            if (++kb == KB || i == cnt - 1) {  // the tile ends here, or this CTA's range does
                // whole tile in this CTA -> 0; this CTA started inside the tile
                // -> 1 (publish); the tile goes on in later CTAs -> 2 (reduce)
                const bool starts_here = cur != nt0 || kb0 == 0;
                const bool ends_here = kb == KB;
                const int role = starts_here ? (ends_here ? 0 : 2) : 1;
                if (hdr_ok) flush_tile<MPAD>(p, cur, acc, c, G, role, q, lane, epoch, misc);
#pragma unroll
                for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
                ++cur;
                kb = 0;
            }
        }
    }

    // ---- teardown -------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (misc[kMiscAbort] != 0) {
        // drain this CTA's own copies and MMAs before its shared memory and
        // TMEM go away (bounded as well)
        if (tid == 0) {
            for (int i = 0; i < cnt; ++i) wait_phase(&full[i], 0, p.timeout, misc, p.err, false);
            const uint32_t issued = misc[kMiscIssued];
            for (int i = 0; i < cnt; ++i)
                if (issued & (1u << i)) wait_phase(&accf[i], 0, p.timeout, misc, p.err, false);
        }
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
    // every thread has read the old epoch: move this index class on to it
    if (warp == 2)
        for (uint32_t j = c + lane * G; j < static_cast<uint32_t>(kMaxCtas); j += 32 * G) p.gen[j] = epoch;
}

template <int MPAD, int KIND, bool DIST>
cudaError_t launch_impl(const Params& p, int grid, cudaStream_t stream) {
    using C = Cfg<MPAD, DIST>;
    auto kern = fused_quant_gemm_kernel<MPAD, KIND, DIST>;
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int MPAD, int KIND, bool DIST>
cudaError_t launch_chunks(Params p, const FusedArgs& a, cudaStream_t stream) {
    // At most one CTA per SM, each with at most kUnits resident units: weights
    // with more units than that go in several launches of whole n-tiles.
    const int KB = a.K / kTile, NT = a.N / kTile;
    const int cap_units = a.sm_count * Cfg<MPAD, DIST>::kUnits;
    const int chunk_nt = cap_units / KB;  // >= 1 (checked by the caller)
    const size_t scale_bytes = a.kind == FP8BS_SCALE_UE8M0 ? 1 : 4;
    for (int nt_base = 0; nt_base < NT; nt_base += chunk_nt) {
        const int nts = NT - nt_base < chunk_nt ? NT - nt_base : chunk_nt;
        p.T = static_cast<uint32_t>(nts * KB);
        p.tiles = a.packed + kHeaderBytes + static_cast<size_t>(nt_base) * KB * kTileBytes;
        p.wscales = a.packed + packed_scales_offset(a.N, a.K) + static_cast<size_t>(nt_base) * KB * scale_bytes;
        p.y = a.y + static_cast<size_t>(nt_base) * kTile;
        p.xq_out = nt_base == 0 ? a.xq_out : nullptr;
        p.xs_out = nt_base == 0 ? a.xs_out : nullptr;
        p.pdl = nt_base == 0 ? a.pdl : 1;  // later chunks follow our own launch, which never writes packed
        const int grid = static_cast<int>(p.T) < a.sm_count ? static_cast<int>(p.T) : a.sm_count;
        const cudaError_t e = launch_impl<MPAD, KIND, DIST>(p, grid, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int KIND>
cudaError_t launch_kind(const Params& p, const FusedArgs& a, cudaStream_t stream) {
    if (a.M <= kLocalMaxM) return launch_chunks<16, KIND, false>(p, a, stream);
    if (a.M <= 16) return launch_chunks<16, KIND, true>(p, a, stream);
    return launch_chunks<32, KIND, true>(p, a, stream);
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream) {
    Params p;
    p.x = a.x;
    p.ldx = a.ldx;
    p.packed = a.packed;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = a.K / kTile;
    p.kind = a.kind;
    p.mdiv = ((uint64_t(1) << 32) + static_cast<uint64_t>(a.M) - 1) / static_cast<uint64_t>(a.M);
    p.ldy = a.ldy;
    p.err = reinterpret_cast<uint32_t*>(a.workspace);
    p.gen = reinterpret_cast<uint32_t*>(a.workspace + ws_gen_offset());
    p.ll = reinterpret_cast<uint64_t*>(a.workspace + ws_partials_offset());
    p.xsw = reinterpret_cast<uint64_t*>(a.workspace + ws_xs_offset(a.sm_count));
    p.xqw = reinterpret_cast<uint64_t*>(a.workspace + ws_xq_offset(a.sm_count, a.K));
    p.timeout = a.timeout_cycles;
    p.pdl = a.pdl;
    if (a.kind == FP8BS_SCALE_UE8M0) return launch_kind<FP8BS_SCALE_UE8M0>(p, a, stream);
    return launch_kind<FP8BS_SCALE_F32>(p, a, stream);
}

bool fused_shape_supported(int64_t N, int64_t K, int sm_count) {
    if (N < kTile || K < kTile || N % kTile != 0 || K % kTile != 0) return false;
    if (sm_count < 1 || sm_count > kMaxCtas) return false;
    return K / kTile <= static_cast<int64_t>(sm_count) * kMaxUnitsM32;
}

}  // namespace fp8bs
