// Optional per-phase timeline of the fused GEMM kernel.
//
// Compiled in only with -DFP8BS_TRACE (a separate build of the library, see
// native_build.build(trace=True)); the plain library records nothing and
// fp8bs_trace_read reports FP8BS_ERR_ARG there.  In a traced build every CTA of
// a call stamps its phase boundaries twice, with %globaltimer (ns, common to
// all SMs, for lining CTAs and calls up) and clock64 (SM cycles, for short
// intervals inside a CTA), into a shared-memory record; at the end of the call
// one warp copies the record to g_trace[call % kTraceCalls][cta], the call
// numbered by its workspace epoch.  Each stamp is taken by one thread at one
// place in the code, listed below.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace fp8bs {

constexpr int kTraceCalls = 256;
constexpr int kTraceCtas = 160;
constexpr int kTracePoints = 64;

enum TracePoint : int {
    kTpEntry = 0,       // thread 0, first instruction
    kTpSetup = 1,       // thread 0, after the set-up barrier (ring copies issued, TMEM allocated)
    kTpWait = 2,        // first quantising thread, the wait on the previous kernel returned
    kTpQuantFirst = 3,  // first quantising thread, its first group quantised (its x loads landed)
    kTpQuantDone = 4,   // first quantising thread, its share of the quant done (local) / published (exchange)
    kTpXchgDone = 5,    // first quantising thread, its exchanged codes and scales are in shared memory
    kTpMmaFirst = 6,    // (not stamped; kept free for ad-hoc stamps)
    kTpMmaLast = 7,     // the issuer of the last unit, its commit issued
    kTpEpiLast = 8,     // epilogue warp 0, the last unit accumulated
    kTpPublish = 9,     // epilogue warp 0, a partial published (later contributor of a shared tile)
    kTpReduceEnd = 10,  // epilogue warp 0, a shared tile gathered, summed and stored
    kTpTeardown = 11,   // thread 0, every role done
    kTpExit = 12,       // copying warp, record written (just before the CTA exits)
    kTpXload = 13,      // first quantising thread, its first x value landed
    kTpEpoch = 14,      // first quantising thread, the epoch word landed
    kTpGather = 15,     // epilogue warp 0, an owner's gather begins
    kTpMmaUnit = 16,    // + i (i < 10): (not stamped; kept free for ad-hoc stamps)
    kTpEpiUnit = 26,    // + i (i < 10): epilogue warp 0, unit i accumulated
    kTpRefill = 36,     // + j (j < 8): the ring thread, the refill of unit S + j issued
    kTpMmaIssued = 44,  // + i (i < 4): (not stamped; kept free for ad-hoc stamps)
    kTpEpiSeen = 48,    // + i (i < 8): epilogue warp 0, unit i's sum known complete (fp32 scales)
    kTpIssCycles = 56,  // + j (j < 5): the MMA issuer's cycles summed over its loop, in the clock field:
                        // waiting for operands (or the watcher's release), for ring tiles, for
                        // accumulator stages, issuing, the rest
    kTpGatherLoaded = 61,  // epilogue warp 0, an owner's first round of partial words back (tagged or not)
    kTpGatherPolls = 62,   // epilogue warp 0, an owner's re-polls summed over its rounds (count, clock field)
    kTpGatherSummed = 63,  // epilogue warp 0, an owner's columns summed and stored
    kTpCount = 64,
};

#ifdef FP8BS_TRACE
__device__ __forceinline__ unsigned long long trace_gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}
// rec: [kTracePoints][2] in shared memory (globaltimer, clock64)
// stamp taken once the 32-bit value v is available (a data dependence)
#define FP8BS_STAMP_AFTER(rec, pt, v)                                                \
    do {                                                                             \
        unsigned long long t_;                                                       \
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_) : "r"(v) : "memory");   \
        (rec)[2 * (pt)] = t_;                                                        \
        (rec)[2 * (pt) + 1] = static_cast<unsigned long long>(clock64());            \
    } while (0)
#define FP8BS_STAMP(rec, pt)                                                         \
    do {                                                                             \
        (rec)[2 * (pt)] = ::fp8bs::trace_gtimer();                                   \
        (rec)[2 * (pt) + 1] = static_cast<unsigned long long>(clock64());            \
    } while (0)
// clock64 only (reading %globaltimer takes hundreds of cycles, too slow for a
// stamp inside a per-unit loop); the globaltimer field is set to 1 (taken)
#define FP8BS_STAMP_CLK(rec, pt)                                                     \
    do {                                                                             \
        (rec)[2 * (pt)] = 1ull;                                                      \
        (rec)[2 * (pt) + 1] = static_cast<unsigned long long>(clock64());            \
    } while (0)
#else
#define FP8BS_STAMP(rec, pt) ((void)0)
#define FP8BS_STAMP_CLK(rec, pt) ((void)0)
#define FP8BS_STAMP_AFTER(rec, pt, v) ((void)0)
#endif

// Copy the timeline of the last kTraceCalls calls to host memory:
// [kTraceCalls][kTraceCtas][kTracePoints][2] uint64.  cudaErrorNotSupported
// in a library built without FP8BS_TRACE.
cudaError_t trace_copy(void* host_dst, size_t bytes);

}  // namespace fp8bs
