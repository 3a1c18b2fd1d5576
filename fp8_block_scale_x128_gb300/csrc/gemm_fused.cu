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
// over at most one CTA per SM ("stream-K"): CTA c owns units [c*T/G, (c+1)*T/G),
// at most 10-12.  A CTA needs about 110 KB of shared memory and 128 registers
// per thread, so two fit on an SM: with programmatic dependent launch the next
// call's CTAs stream their weights while this call's CTAs finish.
//   1. Weight ring: one thread keeps 4-5 tiles in flight with bulk async
//      copies (TMA, evict-first), refilling a slot as soon as the MMAs that
//      read it complete.  At entry, before the wait for the previous kernel
//      (they read only the packed weight), the first tiles go to the ring and
//      the rest of the CTA's tiles are prefetched into L2, so the whole weight
//      stream starts at once and the refills hit L2.
//   2. Activations into the shared-memory B operands (K-major, 128-byte
//      swizzle), for all of the CTA's units:
//        - up to 6 tokens every CTA quantises its own units' groups;
//        - above that each 1x128 group is quantised once, by one CTA, and
//          published in the workspace as 64-bit words that each carry 32 bits
//          of data (4 codes or the scale) and the call's epoch, with no fence
//          or flag; a CTA reads the words of its units' groups, re-reads the
//          ones that still carry an older epoch, and stores the codes into
//          its operands (a 64-bit access is single-copy atomic, so a word is
//          either old or wholly new);
//        - with caller-quantised input the codes and scales are copied with
//          cp.async.
//   3. Two threads (even and odd units) issue, per unit, four tcgen05.mma
//      kind::f8f6f4 (K = 32 each) with the weight tile as the 128-row A
//      operand and the tokens as N = 16 or 32 ("swap-AB"), into one of 4 TMEM
//      accumulator stages, and one commit that both frees the ring slot and
//      publishes the result.
//   4. Four epilogue warps (one per 32 TMEM lanes) read each accumulator,
//      free its stage, and accumulate P * (xs[m,kb] * ws[nt,kb]) in fp32
//      registers (the per-K-block rescale of the page).
//   5. An n-tile whose whole K range the CTA owns is written as bf16 Y.
//      Otherwise the tile's first CTA reduces it: each later contributor
//      writes its partial into its slot, either as tagged words (up to 12
//      tokens; no fence, no flag) or as fp32 followed by the slot's flags; the
//      reducer gathers the partials (polled words, or cp.async once the flags
//      are set) and sums them in CTA order -- a fixed order, so results are
//      deterministic -- and writes bf16 Y.
// A call's epoch is one more than the workspace's epoch word for the CTA's
// index; every CTA moves the words of its index class on to it when it ends,
// so all words stay equal and every word or flag of an earlier call is older.
// Every wait is bounded; on expiry the kernel records FP8BS_ERR_TIMEOUT in the
// workspace error word, drains its own copies and MMAs (again bounded), frees
// TMEM and returns.  The code of each role is kept small (rolled loops): the
// instruction footprint, not the arithmetic, bounds these short phases.
#include "internal.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// 8 warps.  Warp 0: weight ring (one thread).  Warps 1 and 3: MMA issue (one
// thread each, even and odd units: one thread cannot keep the tensor pipe
// fed); warp 1 also owns TMEM, warp 3 first builds the scale table.  Warp 2:
// unit info and header check, then quant.  Warps 4-7: quant, then the
// epilogue (one warp per 32 TMEM lanes).
constexpr int kThreads = 256;
constexpr int kQuantThreads = 160;  // warps 2 and 4-7
constexpr int kQuantHalfWarps = kQuantThreads / 16;
constexpr int kLocalMaxM = 6;  // up to this many tokens every CTA quantises its own groups
constexpr int kAccStages = 4;

// Where a CTA's activation codes come from.
enum : int {
    kSrcLocal = 0,     // every CTA quantises its own units' groups (few tokens)
    kSrcExchange = 1,  // each group quantised once, exchanged through the workspace
    kSrcInput = 2,     // codes and scales given by the caller (the two-launch path)
};

// MPAD 16 and 32: two CTAs per SM (the next call's CTAs start while this
// call's finish); MPAD 64: one CTA per SM with a deeper weight ring.
template <int MPAD, int SRC>
struct Cfg {
    static constexpr int kCtasPerSm = MPAD == 64 ? 1 : 2;
    static constexpr uint32_t kMaxSmem = MPAD == 64 ? 227 * 1024 : 112 * 1024;
    static constexpr int kUnits = MPAD == 16 ? kMaxUnitsM16 : (MPAD == 32 ? kMaxUnitsM32 : kMaxUnitsM64);
    static constexpr int kStages = MPAD == 16 ? 5 : (MPAD == 32 ? 4 : 8);
    static constexpr uint32_t kBBytes = MPAD * 128;  // activation operand of one unit
    static constexpr uint32_t kTmemCols = kAccStages * MPAD;
    static constexpr uint32_t kRingBytes = kStages * kTileBytes;
    static constexpr uint32_t kOffB = kRingBytes;
    static constexpr uint32_t kOffXs = kOffB + kUnits * kBBytes;
    static constexpr uint32_t kOffWs = kOffXs + kUnits * MPAD * 4;
    static constexpr uint32_t kOffKb = kOffWs + kUnits * 4;
    static constexpr uint32_t kOffTab = (kOffKb + kUnits * 4 + 15) / 16 * 16;
    static constexpr uint32_t kOffBar = kOffTab + kScaleTab * 8;
    // full[S], empty[S], acce[A], bready[U], hdr
    static constexpr uint32_t kNumBars = 2 * kStages + kAccStages + kUnits + 1;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmem = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
    // local quant: groups (unit, token) per half-warp
    static constexpr int kGroupsPerHw = (kUnits * kLocalMaxM + kQuantHalfWarps - 1) / kQuantHalfWarps;
    // exchange: groups (unit, token) per quantising thread
    static constexpr int kGroupsPerThread = (kUnits * MPAD + kQuantThreads - 1) / kQuantThreads;
    static_assert(kSmem <= kMaxSmem, "shared memory per CTA");
    static_assert(MPAD == 16 || MPAD == 32 || MPAD == 64, "token tile");
    static_assert(kBBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
    static_assert(kTmemCols >= 32 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
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
    uint32_t* pflag;          // partial flags [CTA][4 epilogue warps]
    uint64_t* slots;          // partial slots, 32 KB per CTA: [32 cols][128 rows] tagged or [64][128] fp32
    uint8_t* act;             // activation records [K/128][kKbRecBytes]
    uint8_t* xq_out;
    void* xs_out;
    const uint8_t* xq_in;     // kSrcInput: codes [M][ldxq], scales [M][K/128]
    int64_t ldxq;
    const void* xs_in;
    long long timeout;
    int pdl;
};

// kMiscCommitted + 0 / + 1: units committed by the even / odd MMA issuer
enum : int { kMiscTmem = 0, kMiscAbort = 1, kMiscHdrOk = 2, kMiscIssued = 3, kMiscCommitted = 4 };

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

// Activation words of K block kb: scales [32 rows], codes [32 rows][32 words].
__device__ __forceinline__ uint64_t* kb_scales(const Params& p, uint32_t kb) {
    return reinterpret_cast<uint64_t*>(p.act + kb * kKbRecBytes + kKbRecScales);
}
__device__ __forceinline__ uint64_t* kb_codes(const Params& p, uint32_t kb) {
    return reinterpret_cast<uint64_t*>(p.act + kb * kKbRecBytes + kKbRecCodes);
}

__device__ __forceinline__ uint64_t tag(uint32_t data, uint32_t epoch) {
    return static_cast<uint64_t>(data) | (static_cast<uint64_t>(epoch) << 32);
}
__device__ __forceinline__ bool tagged(uint64_t w, uint32_t epoch) { return static_cast<uint32_t>(w >> 32) == epoch; }

// Single-copy-atomic 64-bit exchange words (relaxed, GPU scope).
__device__ __forceinline__ void st_pair(uint64_t* p, uint64_t a, uint64_t b) {
    asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void ld_pair(const uint64_t* p, uint64_t& a, uint64_t& b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_word(uint64_t* p, uint64_t a) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(a) : "memory");
}
__device__ __forceinline__ uint64_t ld_word(const uint64_t* p) {
    uint64_t a;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(a) : "l"(p) : "memory");
    return a;
}

// Cold path of every bounded wait.
__device__ __noinline__ void raise_timeout(uint32_t* err, volatile uint32_t* misc) {
    record_error(err, FP8BS_ERR_TIMEOUT);
    misc[kMiscAbort] = 1;
}

// Bounded wait for an mbarrier phase by one thread: false on expiry (recorded)
// or once the CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Params& p, volatile uint32_t* misc) {
    if (ptx::mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (!ptx::mbar_test(bar, parity)) {
        if (misc[kMiscAbort] != 0) return false;
        if (clock64() - t0 > p.timeout) {
            raise_timeout(p.err, misc);
            return false;
        }
    }
    return true;
}

// Bookkeeping of a bounded poll begun at t0: true once the CTA has aborted,
// or (recorded) once the wait has run past the limit.
__device__ __forceinline__ bool gave_up(long long t0, const Params& p, volatile uint32_t* misc) {
    if (misc[kMiscAbort] != 0) return true;
    if (clock64() - t0 > p.timeout) {
        raise_timeout(p.err, misc);
        return true;
    }
    return false;
}

// Teardown drain: ignores the abort flag, still bounded.
__device__ __noinline__ void drain_bar(uint64_t* bar, uint32_t parity, long long timeout) {
    const long long t0 = clock64();
    while (!ptx::mbar_test(bar, parity) && clock64() - t0 <= timeout) {
    }
}

// Bounded wait until a flag carries the epoch (acquire), by one thread.
__device__ __forceinline__ bool wait_flag(const uint32_t* f, uint32_t epoch, const Params& p, volatile uint32_t* misc) {
    if (ptx::ld_acquire_u32(f) == epoch) return true;
    const long long t0 = clock64();
    while (ptx::ld_acquire_u32(f) != epoch) {
        if (misc[kMiscAbort] != 0) return false;
        if (clock64() - t0 > p.timeout) {
            raise_timeout(p.err, misc);
            return false;
        }
    }
    return true;
}

template <int MPAD>
__device__ __forceinline__ void store_y(const Params& p, int n, const float (&v)[MPAD]) {
#pragma unroll
    for (int m = 0; m < MPAD; ++m)
        if (m < p.M) p.y[m * p.ldy + n] = f32_to_bf16_rn(v[m]);
}

// Calls of up to this many tokens exchange split-K partials as tagged words;
// larger ones as fp32 with a flag per epilogue warp.  A tagged reader needs
// one round of loads per kTaggedRound words, a flagged one a single wait and
// one copy, plus the writer's fence.
constexpr int kTaggedMaxM = 12;
constexpr int kTaggedRound = 16;

// Word of the partial (contributor b + t / M, column t % M, row r).
__device__ __forceinline__ const uint64_t* partial_word(const Params& p, uint32_t b, int t, int r) {
    const int j = static_cast<int>(div_m(static_cast<uint32_t>(t), p.mdiv));
    const int m = t - j * p.M;
    return p.slots + static_cast<size_t>(b + j) * (32 * 128) + m * 128 + r;
}

__device__ __forceinline__ float* fp32_slot(const Params& p, uint32_t b) {
    return reinterpret_cast<float*>(p.slots + static_cast<size_t>(b) * (32 * 128));
}

// Output of one n-tile's accumulator by one epilogue warp (rows q*32 .. +31).
// role 0: this CTA owns the tile's whole K range -> bf16 Y.
// role 1: a later contributor -> write the partial of these rows into this
//         CTA's slot: tagged words (no fence, no flag) or fp32 and then this
//         warp's flag.
// role 2: the reducer -> gather the later contributors' partials of these
//         rows (batches that fit this warp's quarter of the idle weight ring),
//         sum in CTA order, bf16 Y.  Tagged words are read in rounds of loads
//         in flight, the stale ones re-read together until they carry the
//         epoch; fp32 partials are copied (cp.async) once their flags carry it.
// last: the CTA that holds the tile's last unit.  Returns false if a wait
// gave up.
template <int MPAD, int STAGE_FLOATS, bool TAGGED>
__device__ __forceinline__ bool flush_tile(const Params& p, uint32_t nt, float (&acc)[MPAD], uint32_t c, uint32_t last,
                                        int role, int q, int lane, uint32_t epoch, volatile uint32_t* misc,
                                        float* stage) {
    const int r = q * 32 + lane;
    const int n = static_cast<int>(nt) * kTile + r;
    if (role == 0) {
        store_y<MPAD>(p, n, acc);
        return true;
    }
    if (role == 1) {
        if constexpr (TAGGED) {
            uint64_t* slot = p.slots + static_cast<size_t>(c) * (32 * 128);
#pragma unroll
            for (int m = 0; m < MPAD; ++m)
                if (m < p.M) st_word(slot + m * 128 + r, tag(__float_as_uint(acc[m]), epoch));
        } else {
            float* slot = fp32_slot(p, c);
#pragma unroll
            for (int m = 0; m < MPAD; ++m)
                if (m < p.M) slot[m * 128 + r] = acc[m];
            __threadfence();
            __syncwarp();
            if (lane == 0) ptx::st_release_u32(p.pflag + c * 4 + q, epoch);
        }
        return true;
    }
    const int per = p.M * 32;               // floats per contributor (this warp's rows)
    const int batch = STAGE_FLOATS / per;   // contributors per batch (>= 4)
    float* st = stage + q * STAGE_FLOATS;   // this warp's quarter of the ring
#pragma unroll 1
    for (uint32_t b = c + 1; b <= last; b += batch) {
        const int nb = static_cast<int>(last + 1 - b) < batch ? static_cast<int>(last + 1 - b) : batch;
        bool ok = true;
        if constexpr (TAGGED) {
            const int nw = nb * p.M;        // this lane's words: t = j * M + m
#pragma unroll 1
            for (int base = 0; base < nw && ok; base += kTaggedRound) {
                uint64_t w[kTaggedRound];
#pragma unroll
                for (int k = 0; k < kTaggedRound; ++k)
                    w[k] = base + k < nw ? ld_word(partial_word(p, b, base + k, r)) : tag(0, epoch);
                const long long t0 = clock64();
                while (true) {
                    bool all = true;
#pragma unroll
                    for (int k = 0; k < kTaggedRound; ++k) all = all && tagged(w[k], epoch);
                    if (all) break;
                    if (gave_up(t0, p, misc)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int k = 0; k < kTaggedRound; ++k)
                        if (!tagged(w[k], epoch)) w[k] = ld_word(partial_word(p, b, base + k, r));
                }
#pragma unroll
                for (int k = 0; k < kTaggedRound; ++k)
                    if (base + k < nw) st[(base + k) * 32 + lane] = __uint_as_float(static_cast<uint32_t>(w[k]));
            }
            if (__any_sync(0xFFFFFFFFu, !ok)) return false;
        } else {
            if (lane < nb) ok = wait_flag(p.pflag + (b + lane) * 4 + q, epoch, p, misc);
            if (__any_sync(0xFFFFFFFFu, !ok)) return false;
            // 16-byte chunks: (contributor j, column m, rows 4k .. 4k+3 of this warp)
#pragma unroll 1
            for (int t = lane; t < nb * p.M * 8; t += 32) {
                const int jm = t >> 3, k = t & 7;
                const int j = jm / p.M;
                const int m = jm - j * p.M;
                ptx::cp_async16(st + jm * 32 + 4 * k, fp32_slot(p, b + j) + m * 128 + q * 32 + 4 * k);
            }
            ptx::cp_async_wait_all();
        }
        __syncwarp();
#pragma unroll 1
        for (int j = 0; j < nb; ++j) {
#pragma unroll
            for (int m = 0; m < MPAD; ++m)
                if (m < p.M) acc[m] += st[(j * p.M + m) * 32 + lane];
        }
        __syncwarp();
    }
    store_y<MPAD>(p, n, acc);
    return true;
}

// Store one quantised slice (unit i, row m, 16-byte part l16) into the B
// operand, the group scale into sXs, then arrive on unit i's barrier.
template <int MPAD>
__device__ __forceinline__ void put_slice(uint8_t* sB, float* sXs, uint64_t* bready, int i, int m, int l16,
                                          uint32_t lo, uint32_t hi, float scale) {
    uint8_t* row = sB + i * (MPAD * 128) + (m >> 3) * 1024 + (m & 7) * 128;
    *reinterpret_cast<uint2*>(row + (((l16 >> 1) ^ (m & 7)) << 4) + ((l16 & 1) << 3)) = make_uint2(lo, hi);
    if (l16 == 0) sXs[i * MPAD + m] = scale;
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

template <int MPAD, int KIND, int SRC, bool TAGGED>
__global__ void __launch_bounds__(kThreads, Cfg<MPAD, SRC>::kCtasPerSm)
    fused_quant_gemm_kernel(const __grid_constant__ Params p) {
    using C = Cfg<MPAD, SRC>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sRing = smem;
    uint8_t* sB = smem + C::kOffB;
    float* sXs = reinterpret_cast<float*>(smem + C::kOffXs);
    float* sWs = reinterpret_cast<float*>(smem + C::kOffWs);
    int* sKb = reinterpret_cast<int*>(smem + C::kOffKb);
    float2* sTab = reinterpret_cast<float2*>(smem + C::kOffTab);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + S;  // completes when the MMAs that read the slot are done
    uint64_t* acce = empty + S;
    uint64_t* bready = acce + kAccStages;
    uint64_t* hdr_bar = bready + C::kUnits;  // completes once misc[kMiscHdrOk] is written
    volatile uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t u0 = unit_begin(c, p.T, G), u1 = unit_begin(c + 1, p.T, G);
    const int cnt = static_cast<int>(u1 - u0);
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    const uint32_t nt0 = u0 / KB, kb0 = u0 - nt0 * KB;

    // ---- set-up; the first ring tiles go out at once ---------------------------
    if (tid == 0) {
        // arrivals per unit: one per 16-byte code slice (local quant), one per
        // 8-code chunk and one per scale (exchange), or one per copied group
        const uint32_t arrivals = static_cast<uint32_t>(p.M) * (SRC == kSrcLocal ? 16 : (SRC == kSrcExchange ? 17 : 1));
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < kAccStages; ++a) ptx::mbar_init(&acce[a], 4);
        for (int i = 0; i < cnt; ++i) ptx::mbar_init(&bready[i], arrivals);
        ptx::mbar_init(hdr_bar, 1);
        misc[kMiscAbort] = 0;
        misc[kMiscHdrOk] = 0;
        misc[kMiscCommitted] = 0;
        misc[kMiscCommitted + 1] = 0;
        ptx::fence_mbar_init();
        const uint64_t pol = ptx::policy_evict_first();
        const int pre = cnt < S ? cnt : S;
        for (int i = 0; i < pre; ++i) {
            ptx::mbar_arrive_expect_tx(&full[i], kTileBytes);
            ptx::bulk_g2s(sRing + i * kTileBytes, p.tiles + static_cast<size_t>(u0 + i) * kTileBytes, kTileBytes,
                          &full[i], pol);
        }
        misc[kMiscIssued] = static_cast<uint32_t>(pre);
        // the tiles that wait for a ring slot: start their HBM reads now, so
        // the refills find them in L2 (they are contiguous: n-major units)
        if (cnt > pre)
            ptx::bulk_prefetch_l2(p.tiles + static_cast<size_t>(u0 + pre) * kTileBytes,
                                  static_cast<uint32_t>(cnt - pre) * kTileBytes);
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

    if (warp == 2 && lane == 0) {  // packed-weight header check
        const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
        const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->n == p.N && h->k == p.K &&
                        h->scale_kind == p.kind && h->tile_bytes == kTileBytes;
        misc[kMiscHdrOk] = ok ? 1u : 0u;
        ptx::mbar_arrive(hdr_bar);  // release: the epilogue reads the flag after waiting here
    }
    // quantising threads: qt = 0 .. kQuantThreads-1 over warps 2, 4-7
    const int qt = warp == 2 ? tid - 64 : tid - 96;
    const int hw = qt >> 4;
    const int l16 = qt & 15;
    const int hw_first = hw & ~1;  // the warp's first half-warp
    // Everything below may read what the previous kernel on the stream wrote.
    if (p.pdl) ptx::griddep_wait();
    if (warp == 2 && lane == 0 && misc[kMiscHdrOk] == 0) record_error(p.err, FP8BS_ERR_SCALE_KIND);
    uint32_t epoch = 0;  // read by the quantising threads, after their x loads are in flight

    if (warp == 0) {
        // ---- 1. weight ring refills ------------------------------------------------
        if (lane == 0) {
            const uint64_t pol = ptx::policy_evict_first();
#pragma unroll 1
            for (int i = S; i < cnt; ++i) {
                const int s = i % S;
                if (!wait_bar(&empty[s], static_cast<uint32_t>((i / S - 1) & 1), p, misc)) break;
                ptx::mbar_arrive_expect_tx(&full[s], kTileBytes);
                ptx::bulk_g2s(sRing + s * kTileBytes, p.tiles + static_cast<size_t>(u0 + i) * kTileBytes, kTileBytes,
                              &full[s], pol);
                misc[kMiscIssued] = static_cast<uint32_t>(i + 1);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ---- 3. MMA issue: warp 1 the even units, warp 3 the odd ones -------------
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_f8f6f4_e4m3(128, MPAD);
            const int odd = warp == 3 ? 1 : 0;
#pragma unroll 1
            for (int i = odd; i < cnt; i += 2) {
                const int s = i % S, a = i % kAccStages;
                if (!wait_bar(&bready[i], 0, p, misc)) break;
                if (!wait_bar(&full[s], static_cast<uint32_t>((i / S) & 1), p, misc)) break;
                if (i >= kAccStages && !wait_bar(&acce[a], static_cast<uint32_t>((i / kAccStages - 1) & 1), p, misc))
                    break;
                ptx::tc_fence_after();
                const uint32_t wa = ptx::smem_addr(sRing + s * kTileBytes);
                const uint32_t xb = ptx::smem_addr(sB + i * C::kBBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ptx::mma_f8f6f4(tmem + a * MPAD, ptx::smem_desc_sw128(wa + 32 * k),
                                    ptx::smem_desc_sw128(xb + 32 * k), idesc, k > 0 ? 1u : 0u);
                ptx::mma_commit(&empty[s]);  // frees the slot and publishes the accumulator
                misc[kMiscCommitted + odd] = static_cast<uint32_t>(i + 1);
            }
        }
        __syncwarp();
    } else {
        if constexpr (SRC == kSrcLocal) {
            // ---- 2. quantise this CTA's own units' groups --------------------------
            // group g = i * M + m (unit i, token m); half-warp hw takes g = hw + 12 j.
            // All loads are in flight first; the rolled loop then quantises
            // raw[0] and shifts the rest down, so its body appears once.
            const int ngc = cnt * p.M;
            uint4 raw[C::kGroupsPerHw];
#pragma unroll
            for (int j = 0; j < C::kGroupsPerHw; ++j) {
                const int g = hw + kQuantHalfWarps * j;
                raw[j] = make_uint4(0, 0, 0, 0);
                if (g < ngc) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(g), p.mdiv));
                    const int m = g - i * p.M;
                    raw[j] = __ldg(reinterpret_cast<const uint4*>(p.x + m * p.ldx + sKb[i] * kTile + l16 * 8));
                }
            }
            epoch = ptx::ld_relaxed_u32(p.gen + c) + 1;
#pragma unroll 1
            for (int j = 0; hw_first + kQuantHalfWarps * j < ngc; ++j) {  // warp-uniform
                const int g = hw + kQuantHalfWarps * j;
                const SliceQuant qs = quant_slice<KIND>(raw[0], sTab);
                if (g < ngc) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(g), p.mdiv));
                    const int m = g - i * p.M;
                    if (u0 + i < KB) put_xq_out<KIND>(p, m, sKb[i], l16, qs);  // n-tile 0 publishes xq / xs
                    put_slice<MPAD>(sB, sXs, bready, i, m, l16, qs.lo, qs.hi, qs.scale);
                }
#pragma unroll
                for (int t = 0; t + 1 < C::kGroupsPerHw; ++t) raw[t] = raw[t + 1];
            }
        } else if constexpr (SRC == kSrcExchange) {
            // ---- 2a. this CTA's share of all groups: quantise, publish ------------
            // group g = kb * M + m; half-warp hw takes g0 + hw, g0 + hw + 12, ...
            const uint32_t NG = static_cast<uint32_t>(p.M) * KB;
            const uint32_t g0 = unit_begin(c, NG, G), g1 = unit_begin(c + 1, NG, G);
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (g0 + hw < g1) {
                const uint32_t g = g0 + hw;
                const uint32_t kb = div_m(g, p.mdiv), m = g - kb * static_cast<uint32_t>(p.M);
                raw = *reinterpret_cast<const uint4*>(p.x + m * p.ldx + kb * kTile + l16 * 8);
            }
            epoch = ptx::ld_relaxed_u32(p.gen + c) + 1;
#pragma unroll 1
            for (uint32_t base = g0; base + hw_first < g1; base += kQuantHalfWarps) {  // warp-uniform
                const uint32_t g = base + hw;
                const bool valid = g < g1;
                const uint32_t kb = div_m(g, p.mdiv), m = g - kb * static_cast<uint32_t>(p.M);
                if (base != g0) {
                    raw = make_uint4(0, 0, 0, 0);
                    if (valid) raw = *reinterpret_cast<const uint4*>(p.x + m * p.ldx + kb * kTile + l16 * 8);
                }
                const SliceQuant qs = quant_slice<KIND>(raw, sTab);
                if (valid) {  // no fence, no flag: each word carries the epoch
                    st_pair(kb_codes(p, kb) + m * 32 + 2 * l16, tag(qs.lo, epoch), tag(qs.hi, epoch));
                    if (l16 == 0)
                        st_word(kb_scales(p, kb) + m, tag(KIND == FP8BS_SCALE_UE8M0 ? qs.byte : __float_as_uint(qs.scale),
                                                          epoch));
                    put_xq_out<KIND>(p, m, kb, l16, qs);
                }
            }
            // ---- 2b. the groups of this CTA's units into shared memory -------------
            // chunk t = gi * 16 + l (group gi = i * M + m, 8 codes l): thread qt
            // takes t = qt + 160 j, in rounds of kRound loads in flight; the stale
            // ones are re-read together (one round trip per attempt, bounded)
            // until both words carry the epoch.  Then the scales, the same way.
            constexpr int kRound = 8;
            const int ngc = cnt * p.M;
            const int nch = ngc * 16;
            bool ok = true;
#pragma unroll 1
            for (int base = 0; base < nch && ok; base += kQuantThreads * kRound) {
                uint64_t w[kRound][2];
#pragma unroll
                for (int j = 0; j < kRound; ++j) {
                    const int t = base + qt + kQuantThreads * j;
                    w[j][0] = w[j][1] = tag(0, epoch);  // out of range: nothing to wait for
                    if (t < nch) {
                        const int gi = t >> 4, l = t & 15;
                        const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                        const int m = gi - i * p.M;
                        ld_pair(kb_codes(p, static_cast<uint32_t>(sKb[i])) + m * 32 + 2 * l, w[j][0], w[j][1]);
                    }
                }
                const long long t0 = clock64();
                while (true) {
                    bool all = true;
#pragma unroll
                    for (int j = 0; j < kRound; ++j) all = all && tagged(w[j][0], epoch) && tagged(w[j][1], epoch);
                    if (all) break;
                    if (gave_up(t0, p, misc)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < kRound; ++j) {
                        const int t = base + qt + kQuantThreads * j;
                        if (!(tagged(w[j][0], epoch) && tagged(w[j][1], epoch))) {
                            const int gi = t >> 4, l = t & 15;
                            const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                            const int m = gi - i * p.M;
                            ld_pair(kb_codes(p, static_cast<uint32_t>(sKb[i])) + m * 32 + 2 * l, w[j][0], w[j][1]);
                        }
                    }
                }
                if (!ok) break;
#pragma unroll
                for (int j = 0; j < kRound; ++j) {
                    const int t = base + qt + kQuantThreads * j;
                    if (t < nch) {
                        const int gi = t >> 4, l = t & 15;
                        const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                        const int m = gi - i * p.M;
                        uint8_t* row = sB + i * C::kBBytes + (m >> 3) * 1024 + (m & 7) * 128;
                        *reinterpret_cast<uint2*>(row + (((l >> 1) ^ (m & 7)) << 4) + ((l & 1) << 3)) =
                            make_uint2(static_cast<uint32_t>(w[j][0]), static_cast<uint32_t>(w[j][1]));
                    }
                }
                ptx::fence_proxy_async_smem();
#pragma unroll
                for (int j = 0; j < kRound; ++j) {
                    const int t = base + qt + kQuantThreads * j;
                    if (t < nch) ptx::mbar_arrive(&bready[static_cast<int>(div_m(static_cast<uint32_t>(t >> 4), p.mdiv))]);
                }
            }
            if (ok) {
                uint64_t sw[C::kGroupsPerThread];
#pragma unroll
                for (int j = 0; j < C::kGroupsPerThread; ++j) {
                    const int gi = qt + kQuantThreads * j;
                    sw[j] = tag(0, epoch);
                    if (gi < ngc) {
                        const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                        const int m = gi - i * p.M;
                        sw[j] = ld_word(kb_scales(p, static_cast<uint32_t>(sKb[i])) + m);
                    }
                }
                const long long t0 = clock64();
                while (true) {
                    bool all = true;
#pragma unroll
                    for (int j = 0; j < C::kGroupsPerThread; ++j) all = all && tagged(sw[j], epoch);
                    if (all) break;
                    if (gave_up(t0, p, misc)) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < C::kGroupsPerThread; ++j) {
                        const int gi = qt + kQuantThreads * j;
                        if (!tagged(sw[j], epoch)) {
                            const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                            const int m = gi - i * p.M;
                            sw[j] = ld_word(kb_scales(p, static_cast<uint32_t>(sKb[i])) + m);
                        }
                    }
                }
                if (ok) {
#pragma unroll
                    for (int j = 0; j < C::kGroupsPerThread; ++j) {
                        const int gi = qt + kQuantThreads * j;
                        if (gi < ngc) {
                            const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                            const int m = gi - i * p.M;
                            const uint32_t bits = static_cast<uint32_t>(sw[j]);
                            sXs[i * MPAD + m] = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(bits) : __uint_as_float(bits);
                            ptx::mbar_arrive(&bready[i]);
                        }
                    }
                }
            }
        } else {
            // ---- 2. the caller's codes and scales of this CTA's units --------------
            // group gi = i * M + m; thread qt takes gi = qt + 160 j: all copies in
            // flight, then one wait.
            const int ngc = cnt * p.M;
            uint32_t sbits[C::kGroupsPerThread];
#pragma unroll
            for (int j = 0; j < C::kGroupsPerThread; ++j) {
                const int gi = qt + kQuantThreads * j;
                sbits[j] = 0;
                if (gi < ngc) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                    const int m = gi - i * p.M;
                    const int kb = sKb[i];
                    const uint8_t* src = p.xq_in + m * p.ldxq + kb * kTile;
                    uint8_t* row = sB + i * C::kBBytes + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll 1
                    for (int ch = 0; ch < 8; ++ch) ptx::cp_async16(row + ((ch ^ (m & 7)) << 4), src + ch * 16);
                    sbits[j] = KIND == FP8BS_SCALE_UE8M0 ? static_cast<const uint8_t*>(p.xs_in)[m * p.KB + kb]
                                                         : static_cast<const uint32_t*>(p.xs_in)[m * p.KB + kb];
                }
            }
            epoch = ptx::ld_relaxed_u32(p.gen + c) + 1;
            ptx::cp_async_wait_all();
#pragma unroll
            for (int j = 0; j < C::kGroupsPerThread; ++j) {
                const int gi = qt + kQuantThreads * j;
                if (gi < ngc) {
                    const int i = static_cast<int>(div_m(static_cast<uint32_t>(gi), p.mdiv));
                    const int m = gi - i * p.M;
                    sXs[i * MPAD + m] = KIND == FP8BS_SCALE_UE8M0 ? e8m0_to_float(sbits[j]) : __uint_as_float(sbits[j]);
                    ptx::fence_proxy_async_smem();
                    ptx::mbar_arrive(&bready[i]);
                }
            }
        }

        if (warp >= 4) {
            // ---- 4./5. rescale-accumulate and output -------------------------------
            const int q = warp & 3;
            uint32_t hdr = 0;
            if (lane == 0) hdr = wait_bar(hdr_bar, 0, p, misc) && misc[kMiscHdrOk] != 0;
            const bool hdr_ok = __shfl_sync(0xFFFFFFFFu, hdr, 0) != 0;
            float acc[MPAD];
#pragma unroll
            for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
            uint32_t cur = nt0, kb = kb0;
            // the CTAs holding the last units of this CTA's first and last tiles
            // (only those two can be shared with other CTAs)
            const uint32_t ntl = nt0 + (kb0 + static_cast<uint32_t>(cnt) - 1) / static_cast<uint32_t>(KB);
            const uint32_t last0 = cta_of((nt0 + 1) * static_cast<uint32_t>(KB) - 1, p.T, G);
            const uint32_t lastl = cta_of((ntl + 1) * static_cast<uint32_t>(KB) - 1, p.T, G);
#pragma unroll 1
            for (int i = 0; i < cnt; ++i) {
                const int a = i % kAccStages;
                uint32_t done = 0;
                // the MMA completion (the slot's release: its phase cannot move on
                // before every epilogue warp has freed this unit's TMEM stage), and
                // the operand barrier that published sXs[i]
                if (lane == 0)
                    done = (wait_bar(&empty[i % S], static_cast<uint32_t>((i / S) & 1), p, misc) &&
                            wait_bar(&bready[i], 0, p, misc)) ? 1u : 0u;
                if (__shfl_sync(0xFFFFFFFFu, done, 0) == 0) break;
                ptx::tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * MPAD);
                uint32_t r[MPAD / 16][16];
#pragma unroll
                for (int h = 0; h < MPAD / 16; ++h) ptx::tmem_ld_32x32b_x16(taddr + 16 * h, r[h]);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&acce[a]);  // this warp is done with the stage
                const float sw = sWs[i];
#pragma unroll
                for (int h = 0; h < MPAD / 16; ++h) {
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        acc[16 * h + m] = fmaf(__uint_as_float(r[h][m]), sXs[i * MPAD + 16 * h + m] * sw, acc[16 * h + m]);
                }
                if (++kb == KB || i == cnt - 1) {  // the tile ends here, or this CTA's range does
                    // whole tile in this CTA -> 0; this CTA started inside the tile
                    // -> 1 (publish); the tile goes on in later CTAs -> 2 (reduce;
                    // always this CTA's last unit, so the weight ring is idle)
                    const bool starts_here = cur != nt0 || kb0 == 0;
                    const bool ends_here = kb == KB;
                    const int role = starts_here ? (ends_here ? 0 : 2) : 1;
                    if (hdr_ok && !flush_tile<MPAD, C::kRingBytes / 16, TAGGED>(p, cur, acc, c, cur == nt0 ? last0 : lastl,
                                                                                 role, q, lane, epoch, misc,
                                                                                 reinterpret_cast<float*>(sRing)))
                        break;
#pragma unroll
                    for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
                    ++cur;
                    kb = 0;
                }
            }
        }
    }

    // ---- teardown -------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (misc[kMiscAbort] != 0 && tid == 0) {
        // drain this CTA's own copies and MMAs before its shared memory and
        // TMEM go away (bounded as well)
        const int issued = static_cast<int>(misc[kMiscIssued]);
        for (int s = 0; s < S && s < issued; ++s) {
            const int uses = (issued - 1 - s) / S + 1;
            drain_bar(&full[s], static_cast<uint32_t>((uses - 1) & 1), p.timeout);
        }
        for (int odd = 0; odd < 2; ++odd) {
            const int committed = static_cast<int>(misc[kMiscCommitted + odd]);
            if (committed > 0) {  // the issuer's last commit covers all of its MMAs
                const int j = committed - 1;
                drain_bar(&empty[j % S], static_cast<uint32_t>((j / S) & 1), p.timeout);
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::kTmemCols);
    }
    // every thread has read the old epoch: move this index class on to it
    if (warp == 2)
        for (uint32_t j = c + lane * G; j < static_cast<uint32_t>(kMaxCtas); j += 32 * G) p.gen[j] = epoch;
}

template <int MPAD, int KIND, int SRC, bool TAGGED>
cudaError_t launch_impl(const Params& p, int grid, cudaStream_t stream) {
    using C = Cfg<MPAD, SRC>;
    auto kern = fused_quant_gemm_kernel<MPAD, KIND, SRC, TAGGED>;
    // Opt in to the dynamic shared memory once per device (not a stream
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

template <int MPAD, int KIND, int SRC, bool TAGGED>
cudaError_t launch_chunks(Params p, const FusedArgs& a, cudaStream_t stream) {
    // At most one CTA per SM with at most kUnits units each: weights with more
    // units than that go in several launches of whole n-tiles.
    const int KB = a.K / kTile, NT = a.N / kTile;
    const int cap_units = a.sm_count * Cfg<MPAD, SRC>::kUnits;
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
        const cudaError_t e = launch_impl<MPAD, KIND, SRC, TAGGED>(p, grid, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int KIND>
cudaError_t launch_kind(const Params& p, const FusedArgs& a, cudaStream_t stream) {
    if (a.xq_in) {
        if (a.M <= kTaggedMaxM) return launch_chunks<16, KIND, kSrcInput, true>(p, a, stream);
        if (a.M <= 16) return launch_chunks<16, KIND, kSrcInput, false>(p, a, stream);
        if (a.M <= 32) return launch_chunks<32, KIND, kSrcInput, false>(p, a, stream);
        return launch_chunks<64, KIND, kSrcInput, false>(p, a, stream);
    }
    if (a.M <= kLocalMaxM) return launch_chunks<16, KIND, kSrcLocal, true>(p, a, stream);
    if (a.M <= kTaggedMaxM) return launch_chunks<16, KIND, kSrcExchange, true>(p, a, stream);
    if (a.M <= 16) return launch_chunks<16, KIND, kSrcExchange, false>(p, a, stream);
    if (a.M <= 32) return launch_chunks<32, KIND, kSrcExchange, false>(p, a, stream);
    return launch_chunks<64, KIND, kSrcExchange, false>(p, a, stream);
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
    p.pflag = reinterpret_cast<uint32_t*>(a.workspace + ws_pflag_offset());
    p.slots = reinterpret_cast<uint64_t*>(a.workspace + ws_partials_offset());
    p.act = a.workspace + ws_act_offset(a.sm_count);
    p.xq_in = a.xq_in;
    p.ldxq = a.ldxq;
    p.xs_in = a.xs_in;
    p.timeout = a.timeout_cycles;
    p.pdl = a.pdl;
    if (a.kind == FP8BS_SCALE_UE8M0) return launch_kind<FP8BS_SCALE_UE8M0>(p, a, stream);
    return launch_kind<FP8BS_SCALE_F32>(p, a, stream);
}

bool fused_shape_supported(int64_t N, int64_t K, int sm_count) {
    if (N < kTile || K < kTile || N % kTile != 0 || K % kTile != 0) return false;
    if (sm_count < 1 || sm_count > kMaxCtas) return false;
    constexpr int64_t kMinUnits = kMaxUnitsM32 < kMaxUnitsM64 ? kMaxUnitsM32 : kMaxUnitsM64;
    return K / kTile <= static_cast<int64_t>(sm_count) * kMinUnits;
}

}  // namespace fp8bs
