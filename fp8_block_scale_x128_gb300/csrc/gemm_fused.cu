// Fused small-M W8A8 FP8 block-scale linear for sm_103a.
//
// What it computes ("[AMD] Small-M FP8 block-scale GEMM with fused activation
// quant for gfx950 (Qwen3.5)", "Modifications"):
//   xq, xs = 1x128-group quant of bf16 x (row amax, scale, e4m3fn codes)
//   Y[m,n] = bf16( sum_kb P[n,m,kb] * (xs[m,kb] * ws[n/128,kb]) ),
//   P[n,m,kb] = sum_{k in kb} wq[n,k] * xq[m,k]
// in one launch; with power-of-two (ue8m0) scales the scales are applied
// inside the MMA ("[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense
// 128x128 fp8 linears (6/8)", "Modifications").  The page's gfx950 design
// (per-wave MFMA over a preshuffled weight, each wave quantising its own
// activations, LDS reduction) is prior art; this is the GB300 form.
//
// Work unit: one (n-tile of 128 weight rows, 128-wide K block) = one 16 KB fp8
// weight tile.  The T = N/128 * K/128 units, in n-major order, are split
// evenly over at most one CTA per SM ("stream-K"): CTA c owns units
// [c*T/G, (c+1)*T/G), at most 10-12.  Two CTAs fit on an SM (up to 32
// tokens), so under programmatic dependent launch the next call's CTAs stream
// their weights while this call's CTAs finish.
//   1. Weight ring: one thread puts the CTA's first 4-8 tiles in flight with
//      bulk async copies (TMA, evict-first) and prefetches its other tiles
//      into L2, before the wait for the previous kernel; a slot is refilled
//      as soon as the MMAs that read it complete.
//   2. Every CTA quantises the 1x128 groups of the K blocks its units touch
//      (one "slot" per distinct K block, shared by units of equal K block),
//      straight into the shared-memory B operands (K-major, 128-byte
//      swizzle), K block by K block so the MMAs can start on the first.
//      With caller-quantised input the codes and scales are copied with
//      cp.async instead.
//   3. One warp issues the MMAs, the weight tile as the 128-row A operand
//      and the tokens as N = 16, 32 or 64 ("swap-AB"), K = 32 each.  In the
//      16-token kernel a watcher warp waits for each unit's operands and tile
//      and releases the issuer through a named barrier, so the issuer never
//      probes an mbarrier; the others probe in batches themselves:
//        fp32 scales: four tcgen05.mma kind::f8f6f4 per unit into its own
//        TMEM stage; four epilogue warps read each stage and accumulate
//        P * (xs * ws) in fp32 registers (the page's per-K-block rescale);
//        ue8m0 scales: kind::mxf8f6f4.block_scale MMAs whose per-32 scale
//        factors sit in TMEM -- each 128-group scale replicated over its four
//        32-blocks -- accumulating a tile's K range in one TMEM stage, read
//        once per tile.
//   4. Split-K: a tile whose K range the CTA owns whole goes straight to bf16
//      Y.  Otherwise the tile's contributors (consecutive CTAs) share the
//      reduction by columns: the last contributor -- the one that reaches the
//      tile first, at the start of its range -- publishes its whole partial;
//      every other contributor publishes the columns it does not own and
//      gathers the columns it owns from the others, summing them in CTA order
//      (a fixed order, so results are deterministic) before writing bf16 Y.
//      Partials travel as 64-bit words (fp32 bits | the call's epoch) with
//      plain relaxed stores and no fence or flag; a reader re-reads the words
//      that still carry an older epoch.
// A call's epoch is one more than the workspace's epoch word for the CTA's
// index (0 is skipped, so a never-written word never matches); every CTA moves
// the words of its index class on to it when it ends.  Every wait is bounded;
// on expiry the kernel records FP8BS_ERR_TIMEOUT in the workspace error word,
// drains its own copies and MMAs (again bounded), frees TMEM and returns.
#include <atomic>

#include "internal.cuh"
#include "ptx.cuh"
#include "trace.cuh"

namespace fp8bs {
namespace {

#ifdef FP8BS_TRACE
__device__ unsigned long long g_trace[kTraceCalls * kTraceCtas * kTracePoints * 2];
#endif

// 8 warps.  Warp 0: weight ring (one thread) and quant.  Warp 1: MMA issue
// (one elected thread) and TMEM.  Warp 2: unit info and header check, then
// quant.  Warp 3: scale table, then quant -- or, in the kernel that quantises
// up to 16 tokens itself, the issue watcher.  Warps 4-7: quant, then the
// epilogue (one warp per 32 TMEM lanes).
constexpr int kThreads = 256;
constexpr int kQuantDepth = 4;       // groups per half-warp with their x loads in flight
constexpr long long kSpinCycles = 4000;         // a wait probes without pause this long (~2 us) ...
constexpr unsigned kBackoffNs = 128;            // ... then sleeps this long between probes

// Where the activation codes come from.
enum : int {
    kSrcQuant = 0,  // every CTA quantises the groups its units need
    kSrcInput = 1,  // codes and scales given by the caller (the two-launch path)
};

template <int MPAD, int KIND>
struct Cfg {
    static constexpr int kCtasPerSm = MPAD == 64 ? 1 : 2;
    static constexpr uint32_t kMaxSmem = MPAD == 64 ? 227 * 1024 : 112 * 1024;
    static constexpr int kUnits = MPAD == 16 ? kMaxUnitsM16 : (MPAD == 32 ? kMaxUnitsM32 : kMaxUnitsM64);
    static constexpr int kStages = MPAD == 16 ? 5 : (MPAD == 32 ? 4 : 8);
    static constexpr uint32_t kBBytes = MPAD * 128;  // activation operand of one K block
    // TMEM accumulator stages: fp32 scales, one per unit -- as many as fit, so
    // the MMAs rarely wait for the epilogue; ue8m0, one per tile segment
    static constexpr int kAcc = KIND == FP8BS_SCALE_UE8M0 ? 4 : (MPAD == 16 ? 12 : 8);
    // then (ue8m0) the scale factors, every scale-factor address on a
    // 4-column boundary: 4 columns per unit for the weight (one per lane
    // quadrant) and 4 per K block for the tokens (MPAD/32 of them used)
    static constexpr uint32_t kSfaCol = kAcc * MPAD;
    static constexpr uint32_t kSfbCols = MPAD > 32 ? 2 : 1;
    static constexpr uint32_t kSfbCol = kSfaCol + 4 * kUnits;
    static constexpr uint32_t kTmemUsed = KIND == FP8BS_SCALE_UE8M0 ? kSfbCol + 4 * kUnits : kSfaCol;
    static constexpr uint32_t kTmemCols = kTmemUsed <= 128 ? 128 : (kTmemUsed <= 256 ? 256 : 512);
    static constexpr uint32_t kRingBytes = kStages * kTileBytes;
    static constexpr uint32_t kOffB = kRingBytes;
    static constexpr uint32_t kOffXs = kOffB + kUnits * kBBytes;  // [slot][MPAD] fp32 scale bits or e8m0 bytes
    static constexpr uint32_t kOffWs = kOffXs + kUnits * MPAD * 4;
    static constexpr uint32_t kOffTab = (kOffWs + kUnits * 4 + 15) / 16 * 16;
    static constexpr uint32_t kOffBar = kOffTab + kScaleTab * 8;
    // full[S], empty[S], acce[A], accfull[A], bready[U], hdr, sfready
    static constexpr uint32_t kNumBars = 2 * kStages + 2 * kAcc + kUnits + 2;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
#ifdef FP8BS_TRACE
    static constexpr uint32_t kOffTrace = kOffMisc + 64;  // timeline record (traced builds only)
    static constexpr uint32_t kSmem = kOffTrace + kTracePoints * 16 + 1024;
#else
    static constexpr uint32_t kSmem = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
#endif
    // the gather stage of one epilogue warp: its quarter of the (idle) ring
    static constexpr uint32_t kStageFloats = kRingBytes / 16;
    static_assert(kSmem <= kMaxSmem, "shared memory per CTA");
    static_assert(MPAD == 16 || MPAD == 32 || MPAD == 64, "token tile");
    static_assert(kBBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
    static_assert(kTmemUsed <= kTmemCols && kTmemCols * kCtasPerSm <= 512, "TMEM allocation");
    static_assert(kSfaCol % 4 == 0 && kSfbCol % 4 == 0, "scale-factor columns on 4-column boundaries");
    static_assert(kStageFloats >= MPAD * 32, "gather stage");
    static_assert(kUnits <= 15, "one named barrier (1..15) per unit");
    static_assert(KIND == FP8BS_SCALE_UE8M0 || kAcc >= 4, "four stages probed at once");
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
    uint64_t* slots;          // partial slots: [CTA][2][64 columns][128 rows] tagged words
    uint8_t* xq_out;
    void* xs_out;
    const uint8_t* xq_in;     // kSrcInput: codes [M][ldxq], scales [M][K/128]
    int64_t ldxq;
    const void* xs_in;
    long long timeout;
    int pdl;
};

enum : int {
    kMiscTmem = 0,
    kMiscAbort = 1,
    kMiscHdrOk = 2,
    kMiscIssued = 3,
    kMiscCommitted = 4,
    kMiscC0 = 5,      // + segment (2): the first contributor of the segment's n-tile
    kMiscC1 = 7,      // + segment (2): the last contributor
    kMiscWhich0 = 9,  // + segment (2): the first contributor's partial slot for that n-tile (0 or 1)
    kMiscMlo = 11,    // + segment (2): the first column this CTA owns of that n-tile's output
    kMiscMhi = 13,    // + segment (2): one past the last
};

__device__ __forceinline__ uint32_t unit_begin(uint32_t c, uint32_t T, uint32_t G) {
    return static_cast<uint32_t>(static_cast<uint64_t>(c) * T / G);
}

// The CTA whose unit range holds unit u (inverse of unit_begin).
__device__ __forceinline__ uint32_t cta_of(uint32_t u, uint32_t T, uint32_t G) {
    return static_cast<uint32_t>((static_cast<uint64_t>(u + 1) * G + T - 1) / T - 1);
}

__device__ __forceinline__ uint32_t div_m(uint32_t g, uint64_t mdiv) { return static_cast<uint32_t>((g * mdiv) >> 32); }

__device__ __forceinline__ uint64_t tag(uint32_t data, uint32_t epoch) {
    return static_cast<uint64_t>(data) | (static_cast<uint64_t>(epoch) << 32);
}
__device__ __forceinline__ bool tagged(uint64_t w, uint32_t epoch) { return static_cast<uint32_t>(w >> 32) == epoch; }

// Accesses to the partial words (single-copy-atomic 64-bit, relaxed, gpu
// scope) and to y (bf16, rounded to nearest even), done only
// where pred holds, with the predicate inside the instruction: a branch
// around an asm statement (which the compiler cannot predicate) costs a
// divergence-safe branch per word, and the unrolled gather loops were
// measured several times slower with them.  ld_word_if leaves w unchanged
// where pred is false.
__device__ __forceinline__ void st_word_if(uint64_t* p, uint64_t a, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q st.relaxed.gpu.global.b64 [%0], %1;\n\t}" ::"l"(p),
                 "l"(a), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void ld_word_if(uint64_t& w, const uint64_t* p, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t@q ld.relaxed.gpu.global.b64 %0, [%1];\n\t}"
                 : "+l"(w)
                 : "l"(p), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}
__device__ __forceinline__ void st_bf16_if(uint16_t* p, float v, bool pred) {
    asm volatile("{\n\t.reg .pred q;\n\t.reg .b16 h;\n\tsetp.ne.u32 q, %2, 0;\n\tcvt.rn.bf16.f32 h, %1;\n\t"
                 "@q st.global.b16 [%0], h;\n\t}" ::"l"(p),
                 "f"(v), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}

// Cold path of every bounded wait.
__device__ __noinline__ void raise_timeout(uint32_t* err, volatile uint32_t* misc) {
    record_error(err, FP8BS_ERR_TIMEOUT);
    misc[kMiscAbort] = 1;
}

// Bounded wait for an mbarrier phase by one thread: false on expiry (recorded)
// or once the CTA has aborted.  It probes without pause for kSpinCycles, then
// sleeps kBackoffNs between probes: a wait that long is a CTA waiting for its
// turn (the issuer and the epilogue of the next call's CTA wait through this
// call), and a spinning warp takes issue slots from the warps that work on
// the same SM (the activation quantisation was measured 2-3x slower with the
// waiters of the co-resident CTA spinning).
// The probe is inline; the loop after a first "not yet" is one out-of-line
// copy (shared by every wait site, which keeps the hot code compact).
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, long long timeout, uint32_t* err,
                                           volatile uint32_t* misc) {
    const long long t0 = clock64();
    while (!ptx::mbar_test(bar, parity)) {
        if (misc[kMiscAbort] != 0) return false;
        const long long dt = clock64() - t0;
        if (dt > timeout) {
            raise_timeout(err, misc);
            return false;
        }
        if (dt > kSpinCycles) __nanosleep(kBackoffNs);
    }
    return true;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Params& p, volatile uint32_t* misc) {
    if (ptx::mbar_test(bar, parity)) return true;
    return wait_bar_slow(bar, parity, p.timeout, p.err, misc);
}

// The same wait for a whole warp (lane 0 polls); false if it gave up.
__device__ __forceinline__ bool warp_wait_bar(uint64_t* bar, uint32_t parity, const Params& p, volatile uint32_t* misc,
                                              int lane) {
    uint32_t ok = 0;
    if (lane == 0) ok = wait_bar(bar, parity, p, misc) ? 1u : 0u;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Teardown drain: ignores the abort flag, still bounded.
__device__ __noinline__ void drain_bar(uint64_t* bar, uint32_t parity, long long timeout) {
    const long long t0 = clock64();
    while (!ptx::mbar_test(bar, parity) && clock64() - t0 <= timeout) {
    }
}

// Word offset (from p.slots) of CTA b's partial slot for an n-tile: slot 0
// if the tile holds b's first unit, else slot 1 (its last tile).  Of a
// tile's contributors c0..c1 only c0 can start before the tile, so which is
// 0 for every b > c0 and which0 (from the set-up) for c0.
__device__ __forceinline__ uint32_t slot_offset(uint32_t b, uint32_t c0, uint32_t which0) {
    return (b * kSlotsPerCta + (b == c0 ? which0 : 0u)) * static_cast<uint32_t>(kSlotWords);
}

// Output of one n-tile segment by one epilogue warp: its 32 rows r = q*32 +
// lane, acc = this CTA's partial sums of them.  c0..c1: the tile's
// contributors (consecutive CTAs), c this CTA.  Returns false if a wait gave up.
//   c0 == c1: the whole K range is here -> bf16 Y.
//   c == c1:  the last contributor (it reached the tile at the start of its
//             range) publishes every column and owns none.
//   else:     contributor s = c - c0, one of the S - 1 owners, owns columns
//             [s*M/(S-1), (s+1)*M/(S-1)): it publishes the others, then gathers
//             its own from the other contributors (rounds of loads in flight,
//             the stale words re-read until they carry the epoch) and sums
//             each column in CTA order, its own partial at its place.
// An owner's segment is always the last of its CTA's range, so the ring is
// idle and its quarter q serves as the stage for its own partials of the
// owned columns.
template <int MPAD>
__device__ __forceinline__ bool flush_segment(const Params& p, uint32_t nt, const float (&acc)[MPAD], uint32_t c,
                                              uint32_t c0, uint32_t c1, uint32_t which0, int m_lo, int m_hi, int q,
                                              int lane, uint32_t epoch, volatile uint32_t* misc, float* stage) {
    const int r = q * 32 + lane;
    uint16_t* yrow = p.y + static_cast<size_t>(nt) * kTile + r;
    if (c0 == c1) {
#pragma unroll
        for (int m = 0; m < MPAD; ++m) st_bf16_if(yrow + m * p.ldy, acc[m], m < p.M);
        return true;
    }
    const int owners = static_cast<int>(c1 - c0);
    const int s = static_cast<int>(c - c0);
    uint64_t* mine = p.slots + slot_offset(c, c0, which0) + r;
#pragma unroll
    for (int m = 0; m < MPAD; ++m)
        st_word_if(mine + m * kTile, tag(__float_as_uint(acc[m]), epoch), m < p.M && (m < m_lo || m >= m_hi));
    if (m_lo == m_hi) return true;
#ifdef FP8BS_TRACE
    if (q == 0 && lane == 0) {
        volatile unsigned long long* rec = reinterpret_cast<volatile unsigned long long*>(misc + 16);
        FP8BS_STAMP_CLK(rec, kTpGather);
    }
#endif
    const int width = m_hi - m_lo;
    float* own = stage;  // [width][32]: this CTA's partials of the owned columns
#pragma unroll
    for (int m = 0; m < MPAD; ++m)
        if (m >= m_lo && m < m_hi) own[(m - m_lo) * 32 + lane] = acc[m];
    __syncwarp();
    // word t = col * owners + j: column m_lo + col of the j-th other contributor,
    // b = c0 + j, or c0 + j + 1 from this CTA on.  Addresses come from
    // registers (no table in shared memory between the loads), and each
    // column is summed in a register as its words arrive, in CTA order, then
    // stored.
    const uint64_t* col0 = p.slots + static_cast<uint32_t>(m_lo * kTile + r);
    const int nw = owners * width;
#ifdef FP8BS_TRACE
    if (q == 0 && lane == 0) {
        volatile unsigned long long* rec = reinterpret_cast<volatile unsigned long long*>(misc + 16);
        FP8BS_STAMP_CLK(rec, kTpEpoch);  // the gather's set-up done, its loads about to go out
    }
#endif
    // rounds of 16 words per lane in flight.  With 16 tokens an owner often
    // has only a few words (3-4 at one token): a round then stops at the first
    // group of four past its last word (one uniform branch per group, kept
    // where measured to pay; with 32 or more tokens the words fill the round)
    constexpr int kRound = 16;
    constexpr bool kSkip = MPAD == 16;
    bool ok = true;
    int jr = 0, colr = 0;  // word `base` = column colr of the jr-th other contributor
    float run = 0.0f;      // the running sum of column colr
#pragma unroll 1
    for (int base = 0; base < nw && ok; base += kRound) {
        // word k of the round: its offset from col0 (recomputed for a re-read)
        const auto word_off = [&](int jj, int cc) {
            const uint32_t b = c0 + static_cast<uint32_t>(jj) + (static_cast<int>(c0) + jj >= static_cast<int>(c) ? 1u : 0u);
            return slot_offset(b, c0, which0) + static_cast<uint32_t>(cc * kTile);
        };
        // straight-line code throughout (selects and predicated accesses, no
        // branch per word)
        uint64_t w[kRound];
        uint32_t off[kRound];
        int j = jr, col = colr;
#pragma unroll
        for (int k = 0; k < kRound; ++k) w[k] = tag(0, epoch);
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            if (kSkip && k % 4 == 0 && base + k >= nw) break;
            off[k] = word_off(j, col);
            ld_word_if(w[k], col0 + off[k], base + k < nw);
            const bool wrap = j + 1 == owners;
            j = wrap ? 0 : j + 1;
            col = wrap ? col + 1 : col;
        }
        const long long t0 = clock64();
#ifdef FP8BS_TRACE
        bool first_check = true;
#endif
        while (true) {
            bool all = true;
#pragma unroll
            for (int k = 0; k < kRound; ++k) all = all && tagged(w[k], epoch);
#ifdef FP8BS_TRACE
            if (q == 0 && lane == 0) {
                volatile unsigned long long* rec = reinterpret_cast<volatile unsigned long long*>(misc + 16);
                if (first_check && base == 0) FP8BS_STAMP_CLK(rec, kTpGatherLoaded);  // first words back
                if (!all) {
                    rec[2 * kTpGatherPolls] = 1;
                    rec[2 * kTpGatherPolls + 1] = rec[2 * kTpGatherPolls + 1] + 1;
                }
            }
            first_check = false;
#endif
            if (all) break;
            if (misc[kMiscAbort] != 0) {
                ok = false;
                break;
            }
            if (clock64() - t0 > p.timeout) {
                raise_timeout(p.err, misc);
                ok = false;
                break;
            }
#pragma unroll
            for (int k = 0; k < kRound; ++k) {
                if (kSkip && k % 4 == 0 && base + k >= nw) break;
                ld_word_if(w[k], col0 + off[k], !tagged(w[k], epoch));
            }
        }
        if (!ok) break;
        // the sums in CTA order: the own partial enters just before the first
        // other contributor that follows this CTA (j == s); a column is
        // stored as soon as its last word is in
        j = jr;
        col = colr;
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            if (kSkip && k % 4 == 0 && base + k >= nw) break;
            const bool valid = base + k < nw, wrap = j + 1 == owners;
            const float ov = own[(col < width ? col : width - 1) * 32 + lane];
            run = valid && j == s ? run + ov : run;
            run = valid ? run + __uint_as_float(static_cast<uint32_t>(w[k])) : run;
            st_bf16_if(yrow + (m_lo + col) * p.ldy, run, valid && wrap);
            run = valid && wrap ? 0.0f : run;
            j = wrap ? 0 : j + 1;
            col = wrap ? col + 1 : col;
        }
        jr = j;  // the next round starts where this one ended
        colr = col;
    }
    if (__any_sync(0xFFFFFFFFu, !ok)) return false;
#ifdef FP8BS_TRACE
    if (q == 0 && lane == 0) {
        volatile unsigned long long* rec = reinterpret_cast<volatile unsigned long long*>(misc + 16);
        FP8BS_STAMP_CLK(rec, kTpGatherSummed);
    }
#endif
    return true;
}

// Store one quantised slice (K-block slot i, row m, 16-byte part l16) into the
// B operand and the group scale into sXs (the caller then fences and arrives
// on slot i's barrier), only where `on` holds: the stores carry the predicate,
// so a caller's unrolled groups stay straight-line.
template <int MPAD, int KIND>
__device__ __forceinline__ void put_slice(uint8_t* sB, uint32_t* sXs, int i, int m, int l16, const SliceQuant& qs,
                                          bool on) {
    uint8_t* row = sB + i * (MPAD * 128) + (m >> 3) * 1024 + (m & 7) * 128;
    ptx::st_shared_v2_if(row + (((l16 >> 1) ^ (m & 7)) << 4) + ((l16 & 1) << 3), qs.lo, qs.hi, on);
    ptx::st_shared_b32_if(sXs + i * MPAD + m, KIND == FP8BS_SCALE_UE8M0 ? qs.byte : __float_as_uint(qs.scale),
                          on && l16 == 0);
}

// The quantised activation of group (m, kb) to the caller's optional xq / xs
// outputs, where `on` holds.
template <int KIND>
__device__ __forceinline__ void put_xq_out(const Params& p, uint32_t m, uint32_t kb, int l16, const SliceQuant& qs,
                                           bool on) {
    ptx::st_global_v2_if(p.xq_out + static_cast<int64_t>(m) * p.K + kb * kTile + l16 * 8, qs.lo, qs.hi,
                         on && p.xq_out != nullptr);
    const bool s_on = on && p.xs_out != nullptr && l16 == 0;
    if (KIND == FP8BS_SCALE_UE8M0)
        ptx::st_global_b8_if(static_cast<uint8_t*>(p.xs_out) + m * p.KB + kb, qs.byte, s_on);
    else
        ptx::st_global_b32_if(static_cast<float*>(p.xs_out) + m * p.KB + kb, __float_as_uint(qs.scale), s_on);
}

template <int MPAD, int KIND, int SRC>
__global__ void __launch_bounds__(kThreads, Cfg<MPAD, KIND>::kCtasPerSm)
    fused_quant_gemm_kernel(const __grid_constant__ Params p) {
    using C = Cfg<MPAD, KIND>;
    constexpr int S = C::kStages;
    constexpr int NA = C::kAcc;
    constexpr bool kBlockScaled = KIND == FP8BS_SCALE_UE8M0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sRing = smem;
    uint8_t* sB = smem + C::kOffB;
    uint32_t* sXs = reinterpret_cast<uint32_t*>(smem + C::kOffXs);
    float* sWs = reinterpret_cast<float*>(smem + C::kOffWs);
    float2* sTab = reinterpret_cast<float2*>(smem + C::kOffTab);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* empty = full + S;  // completes when the MMAs that read the slot are done
    uint64_t* acce = empty + S;      // an accumulator stage has been read
    uint64_t* accfull = acce + NA;   // an accumulator stage holds its unit's (ue8m0: segment's) sum
    uint64_t* bready = accfull + NA;
    uint64_t* hdr_bar = bready + C::kUnits;  // completes once misc[kMiscHdrOk] is written
    uint64_t* sf_bar = hdr_bar + 1;          // ue8m0: the token scale factors are in TMEM
    volatile uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
#ifdef FP8BS_TRACE
    volatile unsigned long long* trec = reinterpret_cast<unsigned long long*>(smem + C::kOffTrace);
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * kTracePoints; ++i) trec[i] = 0;
        FP8BS_STAMP(trec, kTpEntry);
    }
#endif

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t G = gridDim.x, c = blockIdx.x;
    const uint32_t u0 = unit_begin(c, p.T, G), u1 = unit_begin(c + 1, p.T, G);
    const int cnt = static_cast<int>(u1 - u0);
    const uint32_t KB = static_cast<uint32_t>(p.KB);
    const uint32_t nt0 = u0 / KB, kb0 = u0 - nt0 * KB;
    // K-block slots: unit i uses slot i % KB (the range's distinct K blocks)
    const int nslots = cnt < p.KB ? cnt : p.KB;

    // ---- set-up; the first ring tiles go out at once ---------------------------
    if (tid == 0) {
        // arrivals per slot: one per 16-byte code slice (quant) or per copied group
        const uint32_t arrivals = static_cast<uint32_t>(p.M) * (SRC == kSrcQuant ? 16 : 1);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < NA; ++a) {
            ptx::mbar_init(&acce[a], 4);
            ptx::mbar_init(&accfull[a], 1);
        }
        for (int i = 0; i < nslots; ++i) ptx::mbar_init(&bready[i], arrivals);
        ptx::mbar_init(hdr_bar, 1);
        ptx::mbar_init(sf_bar, 4);
        misc[kMiscAbort] = 0;
        misc[kMiscHdrOk] = 0;
        misc[kMiscCommitted] = 0;
        ptx::fence_mbar_init();
        const uint64_t pol = ptx::policy_evict_first();
        const int pre = cnt < S ? cnt : S;
        for (int i = 0; i < pre; ++i) {
            ptx::mbar_arrive_expect_tx(&full[i], kTileBytes);
            ptx::bulk_g2s(sRing + i * kTileBytes, p.tiles + static_cast<size_t>(u0 + i) * kTileBytes, kTileBytes,
                          &full[i], pol);
        }
        misc[kMiscIssued] = static_cast<uint32_t>(pre);
        // the tiles beyond the ring into L2 (one bulk prefetch: they are
        // contiguous), so that their refills, issued in one burst by every
        // CTA as its first MMAs complete, come from L2 rather than DRAM
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
        const uint32_t u = u0 + static_cast<uint32_t>(lane);
        sWs[lane] = kBlockScaled ? __uint_as_float(p.wscales[u]) : reinterpret_cast<const float*>(p.wscales)[u];
    }
    if (p.pdl) ptx::griddep_launch_dependents();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[kMiscTmem];
    if (tid == 0) FP8BS_STAMP(trec, kTpSetup);

    if (warp == 2 && lane == 0) {  // packed-weight header check
        const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
        const bool ok = h->magic == kPackedMagic && h->version == kPackedVersion && h->n == p.N && h->k == p.K &&
                        h->scale_kind == p.kind && h->tile_bytes == kTileBytes;
        // the contributors of this CTA's (at most two) n-tiles: their 64-bit
        // divisions here, before the wait on the previous kernel
#pragma unroll 1
        for (uint32_t sg = 0; sg < 2; ++sg) {
            const uint32_t nt = nt0 + sg;
            const uint32_t a = cta_of(nt * KB, p.T, G);
            misc[kMiscC0 + sg] = a;
            misc[kMiscC1 + sg] = cta_of(nt * KB + KB - 1 < p.T ? nt * KB + KB - 1 : p.T - 1, p.T, G);
            misc[kMiscWhich0 + sg] = unit_begin(a, p.T, G) / KB == nt ? 0u : 1u;
            // owned columns: contributor s = c - c0 of the c1 - c0 owners (none for c1)
            const uint32_t b1 = misc[kMiscC1 + sg];
            const int owners = static_cast<int>(b1 - a), sc = static_cast<int>(c - a);
            const bool owner = c != b1 && owners > 0;
            misc[kMiscMlo + sg] = static_cast<uint32_t>(owner ? sc * p.M / owners : p.M);
            misc[kMiscMhi + sg] = static_cast<uint32_t>(owner ? (sc + 1) * p.M / owners : p.M);
        }
        misc[kMiscHdrOk] = ok ? 1u : 0u;
        ptx::mbar_arrive(hdr_bar);  // release: the epilogue reads the flag after waiting here
    }
    if (kBlockScaled && warp >= 4) {
        // weight scale factors: unit i's e8m0 byte in all four bytes of TMEM
        // column kSfaCol + 4i + q for the rows of quadrant q (row r reads lane
        // r, column base + r/32)
        const int q = warp & 3;
#pragma unroll 1
        for (int i = 0; i < cnt; ++i) {
            const uint32_t b = __float_as_uint(sWs[i]) & 0xFFu;
            ptx::tmem_st_32x32b_x1(tmem + (static_cast<uint32_t>(q * 32) << 16) + C::kSfaCol + 4 * i + q,
                                   b * 0x01010101u);
        }
        ptx::tmem_wait_st();
    }
    // the issue watcher (warp 3) where it was measured to pay: 16-token tiles
    // quantised here (with 32 the quant is the longer phase and needs warp 3)
    constexpr bool kWatch = MPAD == 16 && SRC == kSrcQuant;
    constexpr int kQuantHalfWarps = kWatch ? 12 : 14;  // warps 0, 2 (3) and 4-7
    constexpr int kQuantThreads = 16 * kQuantHalfWarps;
    const bool quant_warp = warp != 1 && !(kWatch && warp == 3);
    const int qt = warp == 0 ? tid : (kWatch && warp >= 4 ? tid - 64 : tid - 32);  // quantising threads
    const int hw = qt >> 4;
    const int l16 = qt & 15;
    const int hw_first = hw & ~1;  // the warp's first half-warp
    uint32_t epoch = 0;
    // ring refills (warp 0, lane 0): units S.. go into the slots their
    // predecessors free.  Between quantisation rounds the ring thread issues
    // those whose slots are already free, without waiting; after its share of
    // the quantisation it takes the rest in order, waiting for each slot.
    int refilled = S;
    const auto refill = [&](int i) {
        ptx::mbar_arrive_expect_tx(&full[i % S], kTileBytes);
        ptx::bulk_g2s(sRing + (i % S) * kTileBytes, p.tiles + static_cast<size_t>(u0 + i) * kTileBytes, kTileBytes,
                      &full[i % S], ptx::policy_evict_first());
        misc[kMiscIssued] = static_cast<uint32_t>(i + 1);
        if (i - S < 8) FP8BS_STAMP_CLK(trec, kTpRefill + i - S);
    };

    if (SRC == kSrcQuant && quant_warp) {
        // ---- 2. quantise the groups of this CTA's K-block slots -------------------
        // group g = slot * M + m (slot-major, so slot 0 is ready first); the
        // half-warp's t-th group is g = hw + H t (H = kQuantHalfWarps), in
        // rounds of kQuantDepth:
        // a round first issues the x loads of the next round, then quantises
        // its own groups, so one round of work covers the load latency.  (No
        // warm-up round on dummy values before the wait: measured slower, as
        // it competes with the quant of the CTA running on the same SM.)
        const int ng = nslots * p.M;
        {
            if (p.pdl) ptx::griddep_wait();
            if (tid == 64) FP8BS_STAMP(trec, kTpWait);
            epoch = ptx::ld_relaxed_u32(p.gen + c) + 1;
            if (epoch == 0) epoch = 1;
            // (loads, stores and arrivals below carry their group's condition
            // as a predicate: the round stays straight-line)
            uint4 raw[kQuantDepth], nxt[kQuantDepth];
#pragma unroll
            for (int k = 0; k < kQuantDepth; ++k) {
                const int g = hw + kQuantHalfWarps * k;
                raw[k] = make_uint4(0x3F8A3F81u + k, 0x3F933FA5u, 0xBF853F99u, 0x3FC13F87u);
                const uint32_t i = div_m(static_cast<uint32_t>(g), p.mdiv), m = g - i * p.M;
                const uint32_t kb = kb0 + i < KB ? kb0 + i : kb0 + i - KB;  // i < KB, kb0 < KB where used
                ptx::ld_global_v4_if(raw[k], p.x + m * p.ldx + kb * kTile + l16 * 8, g < ng);
            }
            if (tid == 64) FP8BS_STAMP_AFTER(trec, kTpXload, raw[0].x);
            uint32_t sink = 0;
#pragma unroll 1
            for (int t0 = 0; hw_first + kQuantHalfWarps * t0 < ng; t0 += kQuantDepth) {
                // the next round's loads first; then the round's kQuantDepth
                // groups: quantise all (independent chains the compiler can
                // interleave), store codes and scales, one proxy fence, the
                // arrivals
#pragma unroll
                for (int k = 0; k < kQuantDepth; ++k) {
                    const int g2 = hw + kQuantHalfWarps * (t0 + k + kQuantDepth);
                    nxt[k] = raw[k];
                    const uint32_t i2 = div_m(static_cast<uint32_t>(g2), p.mdiv), m2 = g2 - i2 * p.M;
                    const uint32_t kb2 = kb0 + i2 < KB ? kb0 + i2 : kb0 + i2 - KB;
                    ptx::ld_global_v4_if(nxt[k], p.x + m2 * p.ldx + kb2 * kTile + l16 * 8, g2 < ng);
                }
                // every slot of the round, valid or not (straight-line code, so
                // the groups interleave); a rare group is then redone exactly
                // (a round whose warp holds a single group computes only that one)
                SliceQuant qs[kQuantDepth];
                bool rare[kQuantDepth];
                if (hw_first + kQuantHalfWarps * (t0 + 1) >= ng) {  // warp-uniform
                    qs[0] = quant_slice_fast<KIND>(raw[0], sTab, rare[0]);
#pragma unroll
                    for (int k = 1; k < kQuantDepth; ++k) {
                        qs[k] = qs[0];
                        rare[k] = false;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < kQuantDepth; ++k) qs[k] = quant_slice_fast<KIND>(raw[k], sTab, rare[k]);
                }
#pragma unroll
                for (int k = 0; k < kQuantDepth; ++k) {
                    if (__any_sync(0xFFFFFFFFu, rare[k])) {
                        const SliceQuant r = quant_slice_exact<KIND>(raw[k], sTab);
                        if (rare[k]) qs[k] = r;
                    }
                    sink ^= qs[k].lo;
                }
                {
                    uint32_t slot_of[kQuantDepth];
#pragma unroll
                    for (int k = 0; k < kQuantDepth; ++k) {
                        const int g = hw + kQuantHalfWarps * (t0 + k);
                        const uint32_t i = div_m(static_cast<uint32_t>(g), p.mdiv), m = g - i * p.M;
                        slot_of[k] = i;
                        // n-tile 0 publishes xq / xs
                        put_xq_out<KIND>(p, m, u0 + i, l16, qs[k], g < ng && u0 + i < KB);
                        put_slice<MPAD, KIND>(sB, sXs, static_cast<int>(i), static_cast<int>(m), l16, qs[k], g < ng);
                    }
                    ptx::fence_proxy_async_smem();
#pragma unroll
                    for (int k = 0; k < kQuantDepth; ++k)
                        ptx::mbar_arrive_if(&bready[slot_of[k]], hw + kQuantHalfWarps * (t0 + k) < ng);
                }
#pragma unroll
                for (int k = 0; k < kQuantDepth; ++k) raw[k] = nxt[k];
                if (t0 == 0 && tid == 64) FP8BS_STAMP_CLK(trec, kTpQuantFirst);
                if (warp == 0) {
                    if (lane == 0)
                        while (refilled < cnt &&
                               ptx::mbar_test(&empty[refilled % S], static_cast<uint32_t>((refilled / S - 1) & 1)))
                            refill(refilled++);
                    __syncwarp();
                }
            }
            asm volatile("" ::"r"(sink));
        }
        if (tid == 64) FP8BS_STAMP_CLK(trec, kTpQuantDone);
    } else {
        if (p.pdl) ptx::griddep_wait();
        if (tid == 64) FP8BS_STAMP(trec, kTpWait);
        if (quant_warp) {
            epoch = ptx::ld_relaxed_u32(p.gen + c) + 1;
            if (epoch == 0) epoch = 1;
        }
    }
    if (warp == 2 && lane == 0 && misc[kMiscHdrOk] == 0) record_error(p.err, FP8BS_ERR_SCALE_KIND);

    if (SRC == kSrcInput && quant_warp) {
        // ---- 2'. the caller's codes and scales of this CTA's K-block slots -------
        // group g = slot * M + m; thread qt takes g = qt + 224 j: all copies in
        // flight, then one wait.
        const int ng = nslots * p.M;
#pragma unroll 1
        for (int g = qt; g < ng; g += kQuantThreads) {
            const uint32_t i = div_m(static_cast<uint32_t>(g), p.mdiv), m = g - i * p.M;
            const uint32_t kb = kb0 + i < KB ? kb0 + i : kb0 + i - KB;
            const uint8_t* src = p.xq_in + m * p.ldxq + kb * kTile;
            uint8_t* row = sB + i * C::kBBytes + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) ptx::cp_async16(row + ((ch ^ (m & 7)) << 4), src + ch * 16);
            sXs[i * MPAD + m] = kBlockScaled ? static_cast<const uint8_t*>(p.xs_in)[m * p.KB + kb]
                                             : static_cast<const uint32_t*>(p.xs_in)[m * p.KB + kb];
        }
        ptx::cp_async_wait_all();
        if (tid == 64) FP8BS_STAMP_CLK(trec, kTpXchgDone);
        ptx::fence_proxy_async_smem();
#pragma unroll 1
        for (int g = qt; g < ng; g += kQuantThreads) ptx::mbar_arrive(&bready[div_m(static_cast<uint32_t>(g), p.mdiv)]);
    }

    if (kBlockScaled && warp >= 4) {
        // token scale factors: slot i's e8m0 byte of token n in all four bytes
        // of lane n % 32 of every quadrant, column kSfbCol + 4i + n/32
        const int q = warp & 3;
        bool ok = true;
#pragma unroll 1
        for (int i = 0; i < nslots && ok; ++i) {
            ok = warp_wait_bar(&bready[i], 0, p, misc, lane);
#pragma unroll
            for (int h = 0; h < static_cast<int>(C::kSfbCols); ++h) {
                const int n = h * 32 + lane;
                const uint32_t b = n < p.M ? sXs[i * MPAD + n] & 0xFFu : 127u;
                ptx::tmem_st_32x32b_x1(tmem + (static_cast<uint32_t>(q * 32) << 16) + C::kSfbCol + 4 * i + h,
                                       b * 0x01010101u);
            }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sf_bar);
        if (tid == 128) FP8BS_STAMP_CLK(trec, kTpXchgDone);
    }

    if (warp == 0) {
        // ---- 1. weight ring refills ------------------------------------------------
        if (lane == 0) {
#pragma unroll 1
            for (int i = refilled; i < cnt; ++i) {
                if (!wait_bar(&empty[i % S], static_cast<uint32_t>((i / S - 1) & 1), p, misc)) break;
                refill(i);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- 3. MMA issue ----------------------------------------------------------
        // The whole warp runs this loop, with warp-uniform values, and one
        // elected lane issues each MMA and commit (measured to issue units
        // about twice as fast as the same loop run by lane 0 alone).  With
        // the watcher, unit i waits only on named barrier 1 + i, which warp 3
        // passes once the unit's operands, ring tile and accumulator stage
        // are ready: an mbarrier probe from this warp queues behind the
        // MMAs' shared-memory operand reads (~250 cycles each, measured), a
        // named barrier does not.  Without it the warp probes for itself, in
        // batches: the ring's first tiles once at the start, the K-block
        // operands four at a time, and waits on one barrier only when a batch
        // says not yet.  Nothing is stored to shared memory inside the loop
        // (a generic store waits behind those reads too); the count of
        // committed units is stored once, after it.
        bool ok = kWatch || !kBlockScaled || warp_wait_bar(sf_bar, 0, p, misc, lane);
        uint32_t known = 0;  // bit s: ring slot s holds its first tile; bit 16 + j: slot j's operand is ready
        if (!kWatch) {
            if (lane == 0)
                for (int s0 = 0; s0 < S && s0 < cnt; s0 += 4)
                    known |= ptx::mbar_test4(&full[s0], 0, &full[(s0 + 1) % S], 0, &full[(s0 + 2) % S], 0,
                                             &full[(s0 + 3) % S], 0) << s0;
            known = __shfl_sync(0xFFFFFFFFu, known, 0);
        }
        uint32_t seg = 0, kb = kb0;  // tile segment of unit i and its K block
        int islot = 0;               // unit i's K-block slot, i % KB
        int committed = 0;
#ifdef FP8BS_TRACE
        long long cyc[5] = {0, 0, 0, 0, 0}, t_prev = clock64();
#define FP8BS_ISS_LAP(j)                 \
    do {                                 \
        const long long t_ = clock64();  \
        cyc[j] += t_ - t_prev;           \
        t_prev = t_;                     \
    } while (0)
#else
#define FP8BS_ISS_LAP(j) ((void)0)
#endif
#pragma unroll 1
        for (int i = 0; i < cnt && ok; ++i) {
            FP8BS_ISS_LAP(4);
            const int s = i % S;
            const int slot = islot;  // i % KB, kept by increments (no division in this loop)
            const bool seg_start = i == 0 || kb == 0;
            const int a = static_cast<int>((kBlockScaled ? seg : static_cast<uint32_t>(i)) % NA);
            if constexpr (kWatch) {
                ptx::named_sync(1u + static_cast<uint32_t>(i), 64u);
                FP8BS_ISS_LAP(0);
            } else {
                const int use = static_cast<int>((kBlockScaled ? seg : static_cast<uint32_t>(i)) / NA);
                if (!kBlockScaled && !((known >> (16 + slot)) & 1u)) {
                    const int j = slot;  // probe this slot and the next three
                    uint32_t got = 0;
                    if (lane == 0)
                        got = ptx::mbar_test4(&bready[j], 0, &bready[j + 1 < nslots ? j + 1 : j], 0,
                                              &bready[j + 2 < nslots ? j + 2 : j], 0,
                                              &bready[j + 3 < nslots ? j + 3 : j], 0);
                    known |= __shfl_sync(0xFFFFFFFFu, got, 0) << (16 + j);
                    if (!((known >> (16 + slot)) & 1u)) {
                        if (!warp_wait_bar(&bready[slot], 0, p, misc, lane)) break;
                        known |= 1u << (16 + slot);
                    }
                }
                FP8BS_ISS_LAP(0);
                if (!(i < S && ((known >> i) & 1u)) &&
                    !warp_wait_bar(&full[s], static_cast<uint32_t>((i / S) & 1), p, misc, lane))
                    break;
                FP8BS_ISS_LAP(1);
                if ((seg_start || !kBlockScaled) && use > 0 &&
                    !warp_wait_bar(&acce[a], static_cast<uint32_t>((use - 1) & 1), p, misc, lane))
                    break;
                FP8BS_ISS_LAP(2);
            }
            ptx::tc_fence_after();
            const uint32_t wa = ptx::smem_addr(sRing + s * kTileBytes);
            const uint32_t xb = ptx::smem_addr(sB + slot * C::kBBytes);
            const uint32_t d = tmem + static_cast<uint32_t>(a * MPAD);
            if constexpr (kBlockScaled) {
                const uint32_t sfa = tmem + C::kSfaCol + 4 * i;
                const uint32_t sfb = tmem + C::kSfbCol + 4 * slot;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ptx::mma_mxf8f6f4_bs_warp(d, ptx::smem_desc_sw128(wa + 32 * k), ptx::smem_desc_sw128(xb + 32 * k),
                                              ptx::idesc_mxf8f6f4_e4m3_e8m0(128, MPAD, k, k), sfa, sfb,
                                              (k > 0 || !seg_start) ? 1u : 0u);
            } else {
                const uint32_t idesc = ptx::idesc_f8f6f4_e4m3(128, MPAD);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    ptx::mma_f8f6f4_warp(d, ptx::smem_desc_sw128(wa + 32 * k), ptx::smem_desc_sw128(xb + 32 * k), idesc,
                                         k > 0 ? 1u : 0u);
            }
            ptx::mma_commit_warp(&empty[s]);  // frees the ring slot
            committed = i + 1;
            if (++islot == p.KB) islot = 0;
            const bool seg_end = ++kb == KB || i == cnt - 1;
            // the stage's sum is complete: per unit (fp32), per segment (ue8m0).
            // Its own barrier, not the ring's: that one can run a phase ahead
            // before the epilogue looks; this one waits for the epilogue
            if (!kBlockScaled || seg_end) ptx::mma_commit_warp(&accfull[a]);
            FP8BS_ISS_LAP(3);
            if (seg_end) {
                kb = 0;
                ++seg;
            }
        }
        __syncwarp();
        if (lane == 0) misc[kMiscCommitted] = static_cast<uint32_t>(committed);
#ifdef FP8BS_TRACE
        if (lane == 0) {
            FP8BS_STAMP_CLK(trec, kTpMmaLast);
            for (int j = 0; j < 5; ++j) {
                trec[2 * (kTpIssCycles + j)] = 1;
                trec[2 * (kTpIssCycles + j) + 1] = static_cast<unsigned long long>(cyc[j]);
            }

        }
#endif
        __syncwarp();
    } else if (kWatch && warp == 3) {
        // ---- 3'. the issue watcher ---------------------------------------------------
        // Releases unit i to the issuer (named barrier 1 + i: each id serves
        // one unit, so no barrier is reused within a launch) once its K-block
        // operand (fp32 scales; ue8m0: the token scale factors in TMEM, which
        // follow every operand), its ring tile and its accumulator stage are
        // ready.  Operands and tiles are probed four at a time, ahead of the
        // unit; it waits on one barrier only when a probe says not yet.  A
        // probe of a tile four units on is sound: with a ring of at least four
        // slots, that slot's previous phase is one this warp already saw
        // complete.  After a failed wait it releases the remaining units
        // without waiting (their MMAs read stale operands; the call reports
        // the error), so the issuer never waits on a barrier nobody passes.
        bool ok = !kBlockScaled || warp_wait_bar(sf_bar, 0, p, misc, lane);
        uint32_t seg = 0, kb = kb0;
        int islot = 0;
        uint32_t op_known = 0, tile_known = 0;  // bit j: slot j's operand / unit j's tile is ready
        // the ring's first tiles were requested long before: probe them now,
        // while the operands are still being quantised
        if (lane == 0)
            for (int s0 = 0; s0 < S && s0 < cnt; s0 += 4)
                tile_known |= ptx::mbar_test4(&full[s0], 0, &full[s0 + 1 < S ? s0 + 1 : s0], 0,
                                              &full[s0 + 2 < S ? s0 + 2 : s0], 0, &full[s0 + 3 < S ? s0 + 3 : s0], 0)
                               << s0;
        tile_known = __shfl_sync(0xFFFFFFFFu, tile_known, 0) & ((1u << (S < cnt ? S : cnt)) - 1u);
#pragma unroll 1
        for (int i = 0; i < cnt; ++i) {
            const int s = i % S;
            const int slot = islot;
            const bool seg_start = i == 0 || kb == 0;
            const uint32_t su = kBlockScaled ? seg : static_cast<uint32_t>(i);
            const int a = static_cast<int>(su % NA), use = static_cast<int>(su / NA);
            if (ok && !kBlockScaled && !((op_known >> slot) & 1u)) {
                uint32_t got = 0;
                if (lane == 0) {
                    const int j1 = slot + 1 < nslots ? slot + 1 : slot, j2 = slot + 2 < nslots ? slot + 2 : slot;
                    const int j3 = slot + 3 < nslots ? slot + 3 : slot;
                    got = ptx::mbar_test4(&bready[slot], 0, &bready[j1], 0, &bready[j2], 0, &bready[j3], 0);
                }
                op_known |= __shfl_sync(0xFFFFFFFFu, got, 0) << slot;
                if (!((op_known >> slot) & 1u)) {
                    ok = warp_wait_bar(&bready[slot], 0, p, misc, lane);
                    op_known |= 1u << slot;
                }
            }
            if (ok && !((tile_known >> i) & 1u)) {
                uint32_t got = 0;
                if (lane == 0) {
                    const int i1 = i + 1 < cnt ? i + 1 : i, i2 = i + 2 < cnt ? i + 2 : i, i3 = i + 3 < cnt ? i + 3 : i;
                    got = ptx::mbar_test4(&full[s], static_cast<uint32_t>((i / S) & 1), &full[i1 % S],
                                          static_cast<uint32_t>((i1 / S) & 1), &full[i2 % S],
                                          static_cast<uint32_t>((i2 / S) & 1), &full[i3 % S],
                                          static_cast<uint32_t>((i3 / S) & 1));
                }
                tile_known |= __shfl_sync(0xFFFFFFFFu, got, 0) << i;
                if (!((tile_known >> i) & 1u)) {
                    ok = warp_wait_bar(&full[s], static_cast<uint32_t>((i / S) & 1), p, misc, lane);
                    tile_known |= 1u << i;
                }
            }
            if (ok && (seg_start || !kBlockScaled) && use > 0)
                ok = warp_wait_bar(&acce[a], static_cast<uint32_t>((use - 1) & 1), p, misc, lane);
            ptx::named_arrive(1u + static_cast<uint32_t>(i), 64u);
            if (++islot == p.KB) islot = 0;
            if (++kb == KB || i == cnt - 1) {
                kb = 0;
                ++seg;
            }
        }
    }

    if (warp >= 4) {
        // ---- 4./5. accumulate and output -------------------------------------------
        const int q = warp & 3;
        const bool hdr_ok = warp_wait_bar(hdr_bar, 0, p, misc, lane) && misc[kMiscHdrOk] != 0;
        float acc[MPAD];
        uint32_t seg = 0;
        int i = 0, seen = 0;  // seen: units whose MMAs are known to be complete
        int xslot = 0;        // unit i's K-block slot, i % KB (fp32 scales)
        bool ok = true;
#pragma unroll 1
        while (i < cnt && ok) {
            const uint32_t nt = nt0 + seg;
            const int seg_end = static_cast<int>((nt + 1) * KB - u0);
            const int ib = seg_end < cnt ? seg_end : cnt;
#pragma unroll
            for (int m = 0; m < MPAD; ++m) acc[m] = 0.0f;
            if constexpr (kBlockScaled) {
                // the segment's sum is in TMEM stage seg % NA once its last MMA is done
                const int a = static_cast<int>(seg % NA);
                ok = warp_wait_bar(&accfull[a], static_cast<uint32_t>((seg / NA) & 1), p, misc, lane);
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * MPAD);
#pragma unroll
                for (int h = 0; h < MPAD / 16; ++h) {
                    uint32_t rr[16];
                    ptx::tmem_ld_32x32b_x16(taddr + 16 * h, rr);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc[16 * h + m] = __uint_as_float(rr[m]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&acce[a]);
                i = ib;
            } else {
#pragma unroll 1
                for (; i < ib; ++i) {
                    const int a = i % NA;
                    if (i >= seen) {
                        // units complete in order.  16 tokens: one probe of
                        // units i..i+3 (their latencies overlap) tells how many
                        // are done; each of these stages' previous use is
                        // already seen complete (stages >= 8), so the parity
                        // tests are sound.  32 or 64: one probe of unit i+3
                        // covers four or none (measured the faster choice at
                        // each width).  If unit i is not done, wait for it.
                        uint32_t got = 0;
                        int n;
                        if constexpr (MPAD == 16) {
                            if (lane == 0) {
                                const int j1 = i + 1 < cnt ? i + 1 : i, j2 = i + 2 < cnt ? i + 2 : i;
                                const int j3 = i + 3 < cnt ? i + 3 : i;
                                got = ptx::mbar_test4(&accfull[a], static_cast<uint32_t>((i / NA) & 1), &accfull[j1 % NA],
                                                      static_cast<uint32_t>((j1 / NA) & 1), &accfull[j2 % NA],
                                                      static_cast<uint32_t>((j2 / NA) & 1), &accfull[j3 % NA],
                                                      static_cast<uint32_t>((j3 / NA) & 1));
                            }
                            n = __ffs(~__shfl_sync(0xFFFFFFFFu, got, 0)) - 1;  // leading units done
                        } else {
                            const int j = i + 3 < cnt ? i + 3 : cnt - 1;
                            if (lane == 0) got = ptx::mbar_test(&accfull[j % NA], static_cast<uint32_t>((j / NA) & 1)) ? 1u : 0u;
                            n = __shfl_sync(0xFFFFFFFFu, got, 0) != 0 ? j + 1 - i : 0;
                        }
                        if (n == 0) {
                            ok = warp_wait_bar(&accfull[a], static_cast<uint32_t>((i / NA) & 1), p, misc, lane);
                            if (!ok) break;
                            seen = i + 1;
                        } else {
                            seen = i + n < cnt ? i + n : cnt;
                        }
                    }
                    ptx::tc_fence_after();
                    if (i < 8 && tid == 128) FP8BS_STAMP_CLK(trec, kTpEpiSeen + i);
                    const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(a * MPAD);
                    const float sw = sWs[i];
                    const uint4* xs4 = reinterpret_cast<const uint4*>(sXs + xslot * MPAD);  // 64-byte aligned
                    if (++xslot == p.KB) xslot = 0;
#pragma unroll
                    for (int h = 0; h < MPAD / 16; ++h) {
                        uint32_t rr[16];
                        ptx::tmem_ld_32x32b_x16(taddr + 16 * h, rr);
                        uint32_t xs[16];
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            const uint4 t = xs4[4 * h + v];
                            xs[4 * v] = t.x;
                            xs[4 * v + 1] = t.y;
                            xs[4 * v + 2] = t.z;
                            xs[4 * v + 3] = t.w;
                        }
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            acc[16 * h + m] = fmaf(__uint_as_float(rr[m]), __uint_as_float(xs[m]) * sw, acc[16 * h + m]);
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    // the stage is released only if a later unit of this CTA takes it
                    if (lane == 0 && i + NA < cnt) ptx::mbar_arrive(&acce[a]);
                    if (i < 10 && tid == 128) FP8BS_STAMP_CLK(trec, kTpEpiUnit + i);
                }
                if (!ok) break;
            }
            if (ib == cnt && tid == 128) FP8BS_STAMP_CLK(trec, kTpEpiLast);
            // the tile's contributors (from the set-up); an owner's segment is
            // always the CTA's last
            const uint32_t c0 = misc[kMiscC0 + (seg & 1)], c1 = misc[kMiscC1 + (seg & 1)];
            if (hdr_ok)
                ok = flush_segment<MPAD>(p, nt, acc, c, c0, c1, misc[kMiscWhich0 + (seg & 1)],
                                         static_cast<int>(misc[kMiscMlo + (seg & 1)]),
                                         static_cast<int>(misc[kMiscMhi + (seg & 1)]), q, lane, epoch, misc,
                                         reinterpret_cast<float*>(sRing) + q * C::kStageFloats);
            if (tid == 128) FP8BS_STAMP_CLK(trec, c == c1 && c0 != c1 ? kTpPublish : kTpReduceEnd);
            ++seg;
        }
    }

    // ---- teardown -------------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) FP8BS_STAMP(trec, kTpTeardown);
    if (misc[kMiscAbort] != 0 && tid == 0) {
        // drain this CTA's own copies and MMAs before its shared memory and
        // TMEM go away (bounded as well)
        const int issued = static_cast<int>(misc[kMiscIssued]);
        for (int s = 0; s < S && s < issued; ++s) {
            const int uses = (issued - 1 - s) / S + 1;
            drain_bar(&full[s], static_cast<uint32_t>((uses - 1) & 1), p.timeout);
        }
        const int committed = static_cast<int>(misc[kMiscCommitted]);
        if (committed > 0) {  // the issuer's last commit covers all of its MMAs
            const int j = committed - 1;
            drain_bar(&empty[j % S], static_cast<uint32_t>((j / S) & 1), p.timeout);
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
#ifdef FP8BS_TRACE
    if (warp == 2) {
        if (lane == 0) FP8BS_STAMP(trec, kTpExit);
        __syncwarp();
        if (c < static_cast<uint32_t>(kTraceCtas))
            for (int v = lane; v < 2 * kTpCount; v += 32)
                g_trace[((epoch % kTraceCalls) * kTraceCtas + c) * (2 * kTracePoints) + v] = trec[v];
    }
#endif
}

template <int MPAD, int KIND, int SRC>
cudaError_t launch_impl(const Params& p, int grid, cudaStream_t stream) {
    using C = Cfg<MPAD, KIND>;
    auto kern = fused_quant_gemm_kernel<MPAD, KIND, SRC>;
    // Opt in to the dynamic shared memory once per device (not a stream
    // operation, so it is harmless during graph capture too).
    // The CTAs of a launch wait for one another: refuse a grid that the
    // device cannot hold at once (occupancy at this kernel's shared memory
    // and threads, times the device's multiprocessors), before launching.
    // Cached per device: resident CTAs per SM times SMs, once configured.
    static std::atomic<int> capacity[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int cap = dev >= 0 && dev < 64 ? capacity[dev].load(std::memory_order_relaxed) : 0;
    if (cap <= 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, C::kSmem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cap = per_sm * sms;
        if (dev >= 0 && dev < 64) capacity[dev].store(cap, std::memory_order_relaxed);
    }
    if (grid > cap) return cudaErrorCooperativeLaunchTooLarge;
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

template <int MPAD, int KIND, int SRC>
cudaError_t launch_chunks(Params p, const FusedArgs& a, cudaStream_t stream) {
    // At most one CTA per SM with at most kUnits units each: weights with more
    // units than that go in several launches of whole n-tiles.
    const int KB = a.K / kTile, NT = a.N / kTile;
    const int cap_units = a.sm_count * Cfg<MPAD, KIND>::kUnits;
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
        const cudaError_t e = launch_impl<MPAD, KIND, SRC>(p, grid, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int KIND>
cudaError_t launch_kind(const Params& p, const FusedArgs& a, cudaStream_t stream) {
    if (a.xq_in) {
        if (a.M <= 16) return launch_chunks<16, KIND, kSrcInput>(p, a, stream);
        if (a.M <= 32) return launch_chunks<32, KIND, kSrcInput>(p, a, stream);
        return launch_chunks<64, KIND, kSrcInput>(p, a, stream);
    }
    if (a.M <= 16) return launch_chunks<16, KIND, kSrcQuant>(p, a, stream);
    return launch_chunks<32, KIND, kSrcQuant>(p, a, stream);
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream) {
    if (!a.xq_in && a.M > kFusedMaxM) return cudaErrorInvalidValue;  // the API routes these through two launches
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
    p.slots = reinterpret_cast<uint64_t*>(a.workspace + ws_partials_offset());
    p.xq_in = a.xq_in;
    p.ldxq = a.ldxq;
    p.xs_in = a.xs_in;
    p.timeout = a.timeout_cycles;
    p.pdl = a.pdl;
    if (a.kind == FP8BS_SCALE_UE8M0) return launch_kind<FP8BS_SCALE_UE8M0>(p, a, stream);
    return launch_kind<FP8BS_SCALE_F32>(p, a, stream);
}

cudaError_t trace_copy(void* host_dst, size_t bytes) {
#ifdef FP8BS_TRACE
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return cudaMemcpyFromSymbol(host_dst, g_trace, bytes);
#else
    (void)host_dst;
    (void)bytes;
    return cudaErrorNotSupported;
#endif
}

bool fused_shape_supported(int64_t N, int64_t K, int sm_count) {
    if (N < kTile || K < kTile || N % kTile != 0 || K % kTile != 0) return false;
    if (sm_count < 1 || sm_count > kMaxCtas) return false;
    constexpr int64_t kMinUnits = kMaxUnitsM32 < kMaxUnitsM64 ? kMaxUnitsM32 : kMaxUnitsM64;
    return K / kTile <= static_cast<int64_t>(sm_count) * kMinUnits;
}

}  // namespace fp8bs
