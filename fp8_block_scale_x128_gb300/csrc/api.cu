// C ABI of the fp8bs library (declared in include/fp8bs.h).
//
// Every entry point checks its arguments on the host first, in this order:
// null pointers and the scale kind (FP8BS_ERR_ARG), shapes (FP8BS_ERR_SHAPE),
// strides and alignment (FP8BS_ERR_ALIGN), buffer sizes (FP8BS_ERR_WORKSPACE).
// Nothing is enqueued when a check fails, and no check touches the GPU, so the
// checks run on machines without one.  The support rules follow "[AMD] Small-M
// FP8 block-scale GEMM with fused activation quant for gfx950 (Qwen3.5)",
// "Modifications" (bf16 input with 16-byte aligned rows, a contiguous
// [N/128, K/128] weight scale, M <= 32); a mismatching scale kind is refused
// rather than reinterpreted, as "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM
// for dense 128x128 fp8 linears (6/8)", "Modifications" requires.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.cuh"
#include "moe.cuh"
#include "producer.cuh"
#include "trace.cuh"

namespace {

using namespace fp8bs;

constexpr int64_t kMaxDim = int64_t(1) << 24;  // N, K bound (keeps every index in range)
constexpr long long kDefaultTimeoutCycles = 2000000000LL;  // ~1 s at 2 GHz

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool kind_ok(int kind) { return kind == FP8BS_SCALE_F32 || kind == FP8BS_SCALE_UE8M0; }

bool nk_ok(int64_t N, int64_t K) {
    return N >= kTile && K >= kTile && N % kTile == 0 && K % kTile == 0 && N <= kMaxDim && K <= kMaxDim;
}

int status_of(cudaError_t e) {
    if (e == cudaSuccess) return FP8BS_OK;
    // the launchers' refusal of a grid that cannot be resident at once
    return e == cudaErrorCooperativeLaunchTooLarge ? FP8BS_ERR_RESIDENCY : FP8BS_ERR_CUDA;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Diagnostic overrides (fp8bs_debug_config); 0: the defaults.
std::atomic<long long> g_timeout_override{0};
std::atomic<int> g_sm_override{0};

long long timeout_cycles() {
    const long long t = g_timeout_override.load(std::memory_order_relaxed);
    return t > 0 ? t : kDefaultTimeoutCycles;
}

// Multiprocessor count of the current device, cached per device (relaxed
// atomics: concurrent first calls from several host threads may both query).
int current_sm_count(int* out) {
    const int forced = g_sm_override.load(std::memory_order_relaxed);
    if (forced > 0) {
        *out = forced;
        return FP8BS_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8BS_ERR_CUDA;
    static std::atomic<int> cache[64];
    if (dev >= 0 && dev < 64) {
        const int n = cache[dev].load(std::memory_order_relaxed);
        if (n > 0) {
            *out = n;
            return FP8BS_OK;
        }
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return FP8BS_ERR_CUDA;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return FP8BS_OK;
}

size_t workspace_bytes_for(int64_t K, int sm_count) { return ws_total_bytes(sm_count, K); }

// Above kFusedMaxM tokens the fused call runs the quant and the GEMM on its
// codes as two launches: the single launch has no 64-token tile that
// quantises, and [P1] "Motivation" likewise keeps larger inputs on the
// library path.
constexpr int kTwoLaunchMinM = kFusedMaxM + 1;

// The fused call, routed: below kTwoLaunchMinM one launch; from it on the
// 1x128 quant, then the GEMM on those codes.  The codes and scales go to
// xq_out / xs_out when the caller asked for them, else to the workspace's
// activation records, which the GEMM on given codes does not use (room for
// 64 rows of codes and fp32 scales per K block).
cudaError_t launch_fused_routed(FusedArgs a, cudaStream_t stream) {
    if (a.M < kTwoLaunchMinM) return launch_fused(a, stream);
    uint8_t* act = a.workspace + ws_act_offset(a.sm_count);
    uint8_t* xq = a.xq_out ? a.xq_out : act;
    void* xs = a.xs_out ? a.xs_out : static_cast<void*>(act + static_cast<size_t>(FP8BS_MAX_M) * a.K);
    const cudaError_t e = launch_quant(a.x, a.M, a.K, a.ldx, a.kind, xq, xs, stream, a.pdl != 0);
    if (e != cudaSuccess) return e;
    a.xq_in = xq;
    a.ldxq = a.K;
    a.xs_in = xs;
    a.xq_out = nullptr;
    a.xs_out = nullptr;
    return launch_fused(a, stream);
}

// Scratch of fp8bs_gemm_fused_static: one fixed array per device, laid out like
// a caller's workspace for FP8BS_STATIC_MAX_SMS CTAs and K up to
// FP8BS_STATIC_MAX_K.
constexpr size_t kStaticScratchBytes = ws_total_bytes(FP8BS_STATIC_MAX_SMS, FP8BS_STATIC_MAX_K);
static_assert(kStaticScratchBytes == 22057216, "fp8bs.h states the scratch size");

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kStaticMaxDevices = 64;
std::mutex g_static_mu;
uint8_t* g_static_ptr[kStaticMaxDevices] = {};

// Address of the current device's scratch; the first call per device looks it
// up and zeroes it on `s` (the error word and the epoch words must start at
// zero), then waits for that, so a call from another thread or stream never
// sees a half-cleared scratch.  That set-up synchronises `s`, which would
// invalidate a stream capture: on a capturing stream it is refused
// (FP8BS_ERR_ARG) before the stream is touched.
int static_scratch(cudaStream_t s, uint8_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8BS_ERR_CUDA;
    if (dev < 0 || dev >= kStaticMaxDevices) return FP8BS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return FP8BS_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return FP8BS_ERR_ARG;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return FP8BS_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, kStaticScratchBytes, s) != cudaSuccess) return FP8BS_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return FP8BS_ERR_CUDA;
        g_static_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_static_ptr[dev];
    return FP8BS_OK;
}

}  // namespace

extern "C" {

const char* fp8bs_status_string(int status) {
    switch (status) {
        case FP8BS_OK: return "ok";
        case FP8BS_ERR_ARG: return "invalid argument (null pointer, scale kind or stride)";
        case FP8BS_ERR_SHAPE: return "unsupported shape (M, N or K)";
        case FP8BS_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
        case FP8BS_ERR_SCALE_KIND: return "packed weight has another scale kind or shape";
        case FP8BS_ERR_WORKSPACE: return "workspace or packed buffer too small or misaligned";
        case FP8BS_ERR_CUDA: return "CUDA runtime error";
        case FP8BS_ERR_TIMEOUT: return "device wait timed out";
        case FP8BS_ERR_DEVICE: return "device-side check failed";
        case FP8BS_ERR_RESIDENCY: return "the launch's CTAs cannot all be resident at once";
        default: return "unknown status";
    }
}

int fp8bs_version(void) { return (1 << 16) | 0; }

int fp8bs_encode_e4m3(const float* v, int64_t n, uint8_t* codes, void* stream) {
    if (n < 0 || n % 4 != 0) return FP8BS_ERR_SHAPE;
    if (n == 0) return FP8BS_OK;
    if (!v || !codes) return FP8BS_ERR_ARG;
    if (!aligned(v, 16) || !aligned(codes, 4)) return FP8BS_ERR_ALIGN;
    return status_of(launch_encode_e4m3(v, n, codes, as_stream(stream)));
}

int fp8bs_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int scale_kind, uint8_t* xq,
                void* xs, void* stream) {
    if (!kind_ok(scale_kind)) return FP8BS_ERR_ARG;
    if (M < 0 || K < kTile || K % kTile != 0 || K > kMaxDim || M > kMaxDim) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!x || !xq || !xs) return FP8BS_ERR_ARG;
    if (ldx < K) return FP8BS_ERR_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(xq, 8) ||
        (scale_kind == FP8BS_SCALE_F32 && !aligned(xs, 4)))
        return FP8BS_ERR_ALIGN;
    return status_of(launch_quant(x, M, K, ldx, scale_kind, xq, xs, as_stream(stream)));
}

int fp8bs_rmsnorm_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma, float eps,
                        int scale_kind, uint8_t* xq, void* xs, uint16_t* y, int64_t ldy, void* stream) {
    if (!kind_ok(scale_kind) || !(eps >= 0.0f) || !(eps <= 3.4e38f)) return FP8BS_ERR_ARG;
    if (M < 0 || K < kTile || K % kTile != 0 || K > FP8BS_RMSNORM_MAX_K || M > kMaxDim) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!x || !gamma || !xq || !xs) return FP8BS_ERR_ARG;
    if (ldx < K || (y && ldy < K)) return FP8BS_ERR_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(gamma, 16) || !aligned(xq, 8) ||
        (scale_kind == FP8BS_SCALE_F32 && !aligned(xs, 4)) || (y && (!aligned(y, 16) || ldy % 8 != 0)))
        return FP8BS_ERR_ALIGN;
    return status_of(launch_rmsnorm_quant(x, M, K, ldx, gamma, eps, scale_kind, xq, xs, y, ldy, as_stream(stream)));
}
size_t fp8bs_moe_workspace_bytes(int64_t M, int64_t S, int64_t H, int64_t I) {
    if (M < 0 || S < 1 || M * S > FP8BS_MOE_MAX_PAIRS || H < 512 || H % 512 != 0 || H > kMaxDim ||
        (I != 128 && I != 256 && I != FP8BS_MOE_MAX_I))
        return 0;
    return moe_workspace_bytes(M, S, H, I);
}
int fp8bs_moe_w8a16(const uint16_t* x, int64_t M, int64_t H, const int32_t* topk_ids, const float* topk_w,
                    int64_t S, const uint8_t* w13, const float* s13, const uint8_t* w2, const float* s2, int64_t E,
                    int64_t I, uint16_t* y, void* workspace, size_t workspace_bytes, void* stream) {
    if (M < 0 || S < 1 || M * S > FP8BS_MOE_MAX_PAIRS || E < 1 || E > FP8BS_MOE_MAX_EXPERTS || H < 512 ||
        H % 512 != 0 || H > kMaxDim || (I != 128 && I != 256 && I != FP8BS_MOE_MAX_I))
        return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!x || !topk_ids || !topk_w || !w13 || !s13 || !w2 || !s2 || !y || !workspace) return FP8BS_ERR_ARG;
    if (!aligned(x, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(w13, 16) || !aligned(s13, 4) ||
        !aligned(w2, 16) || !aligned(s2, 4) || !aligned(y, 8) || !aligned(workspace, 256))
        return FP8BS_ERR_ALIGN;
    if (workspace_bytes < moe_workspace_bytes(M, S, H, I)) return FP8BS_ERR_WORKSPACE;
    int sm = 0;
    const int rc = current_sm_count(&sm);
    if (rc != FP8BS_OK) return rc;
    MoeArgs a;
    a.x = x;
    a.ids = topk_ids;
    a.tw = topk_w;
    a.w13 = w13;
    a.s13 = s13;
    a.w2 = w2;
    a.s2 = s2;
    a.y = y;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.M = static_cast<int>(M);
    a.S = static_cast<int>(S);
    a.H = static_cast<int>(H);
    a.I = static_cast<int>(I);
    a.E = static_cast<int>(E);
    a.sm_count = sm;
    return status_of(launch_moe(a, as_stream(stream)));
}
int fp8bs_quant_weight(const float* w, int64_t N, int64_t K, int64_t ldw, int scale_kind, uint8_t* wq,
                       void* ws, void* stream) {
    if (!kind_ok(scale_kind)) return FP8BS_ERR_ARG;
    if (!nk_ok(N, K)) return FP8BS_ERR_SHAPE;
    if (!w || !wq || !ws) return FP8BS_ERR_ARG;
    if (ldw < K) return FP8BS_ERR_ARG;
    if (!aligned(w, 16) || ldw % 4 != 0 || !aligned(wq, 16) ||
        (scale_kind == FP8BS_SCALE_F32 && !aligned(ws, 4)))
        return FP8BS_ERR_ALIGN;
    return status_of(launch_quant_weight(w, N, K, ldw, scale_kind, wq, ws, as_stream(stream)));
}

size_t fp8bs_packed_weight_bytes(int64_t N, int64_t K, int scale_kind) {
    if (!kind_ok(scale_kind) || !nk_ok(N, K)) return 0;
    const size_t tiles = static_cast<size_t>(N / kTile) * static_cast<size_t>(K / kTile);
    const size_t scale_bytes = tiles * (scale_kind == FP8BS_SCALE_F32 ? 4 : 1);
    return round_up(packed_scales_offset(N, K) + scale_bytes, 256);
}

int fp8bs_prepack_weight(const uint8_t* wq, int64_t ldw, const void* ws, int64_t N, int64_t K,
                         int scale_kind, void* packed, size_t packed_bytes, void* stream) {
    if (!kind_ok(scale_kind)) return FP8BS_ERR_ARG;
    if (!nk_ok(N, K)) return FP8BS_ERR_SHAPE;
    if (!wq || !ws || !packed) return FP8BS_ERR_ARG;
    if (ldw < K) return FP8BS_ERR_ARG;
    if (!aligned(wq, 16) || ldw % 16 != 0 || !aligned(packed, 256) ||
        (scale_kind == FP8BS_SCALE_F32 && !aligned(ws, 4)))
        return FP8BS_ERR_ALIGN;
    if (packed_bytes < fp8bs_packed_weight_bytes(N, K, scale_kind)) return FP8BS_ERR_WORKSPACE;
    return status_of(launch_prepack(wq, ldw, ws, N, K, scale_kind, packed, as_stream(stream)));
}

size_t fp8bs_workspace_bytes(int64_t N, int64_t K, int sm_count) {
    if (!nk_ok(N, K)) return 0;
    if (sm_count <= 0 && current_sm_count(&sm_count) != FP8BS_OK) return 0;
    if (!fused_shape_supported(N, K, sm_count)) return 0;
    return workspace_bytes_for(K, sm_count);
}

int fp8bs_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace) return FP8BS_ERR_ARG;
    if (!aligned(workspace, 256)) return FP8BS_ERR_ALIGN;
    if (workspace_bytes < kWsErrorBytes) return FP8BS_ERR_WORKSPACE;
    return status_of(cudaMemsetAsync(workspace, 0, workspace_bytes, as_stream(stream)));
}

int fp8bs_gemm_fused(const uint16_t* x, int64_t M, int64_t ldx, const void* packed, size_t packed_bytes,
                     int64_t N, int64_t K, int scale_kind, uint16_t* y, int64_t ldy, void* workspace,
                     size_t workspace_bytes, uint8_t* xq_out, void* xs_out, unsigned flags, void* stream) {
    if (!kind_ok(scale_kind) || (flags & ~static_cast<unsigned>(FP8BS_FLAG_PDL)) != 0) return FP8BS_ERR_ARG;
    if (M < 0 || M > FP8BS_MAX_M || !nk_ok(N, K)) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!x || !packed || !y || !workspace) return FP8BS_ERR_ARG;
    if (ldx < K || ldy < N) return FP8BS_ERR_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(y, 16) || ldy % 8 != 0 || !aligned(packed, 256) ||
        !aligned(workspace, 256) || (xq_out && !aligned(xq_out, 16)) ||
        (xs_out && scale_kind == FP8BS_SCALE_F32 && !aligned(xs_out, 4)))
        return FP8BS_ERR_ALIGN;
    if (packed_bytes < fp8bs_packed_weight_bytes(N, K, scale_kind)) return FP8BS_ERR_WORKSPACE;
    int sm = 0;
    const int rc = current_sm_count(&sm);
    if (rc != FP8BS_OK) return rc;
    if (!fused_shape_supported(N, K, sm)) return FP8BS_ERR_SHAPE;
    if (workspace_bytes < workspace_bytes_for(K, sm)) return FP8BS_ERR_WORKSPACE;
    FusedArgs a;
    a.x = x;
    a.ldx = ldx;
    a.packed = static_cast<const uint8_t*>(packed);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.kind = scale_kind;
    a.y = y;
    a.ldy = ldy;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.xq_out = xq_out;
    a.xs_out = xs_out;
    a.sm_count = sm;
    a.timeout_cycles = timeout_cycles();
    a.pdl = (flags & FP8BS_FLAG_PDL) ? 1 : 0;
    return status_of(launch_fused_routed(a, as_stream(stream)));
}

int fp8bs_gemm_prequant(const uint8_t* xq, int64_t M, int64_t ldxq, const void* xs, const void* packed,
                        size_t packed_bytes, int64_t N, int64_t K, int scale_kind, uint16_t* y, int64_t ldy,
                        void* workspace, size_t workspace_bytes, unsigned flags, void* stream) {
    if (!kind_ok(scale_kind) || (flags & ~static_cast<unsigned>(FP8BS_FLAG_PDL)) != 0) return FP8BS_ERR_ARG;
    if (M < 0 || M > FP8BS_MAX_M || !nk_ok(N, K)) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!xq || !xs || !packed || !y || !workspace) return FP8BS_ERR_ARG;
    if (ldxq < K || ldy < N) return FP8BS_ERR_ARG;
    if (!aligned(xq, 16) || ldxq % 16 != 0 || !aligned(y, 16) || ldy % 8 != 0 || !aligned(packed, 256) ||
        !aligned(workspace, 256) || (scale_kind == FP8BS_SCALE_F32 && !aligned(xs, 4)))
        return FP8BS_ERR_ALIGN;
    if (packed_bytes < fp8bs_packed_weight_bytes(N, K, scale_kind)) return FP8BS_ERR_WORKSPACE;
    int sm = 0;
    const int rc = current_sm_count(&sm);
    if (rc != FP8BS_OK) return rc;
    if (!fused_shape_supported(N, K, sm)) return FP8BS_ERR_SHAPE;
    if (workspace_bytes < workspace_bytes_for(K, sm)) return FP8BS_ERR_WORKSPACE;
    FusedArgs a;
    a.x = nullptr;
    a.ldx = 0;
    a.packed = static_cast<const uint8_t*>(packed);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.kind = scale_kind;
    a.y = y;
    a.ldy = ldy;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.xq_out = nullptr;
    a.xs_out = nullptr;
    a.sm_count = sm;
    a.timeout_cycles = timeout_cycles();
    a.pdl = (flags & FP8BS_FLAG_PDL) ? 1 : 0;
    a.xq_in = xq;
    a.ldxq = ldxq;
    a.xs_in = xs;
    return status_of(launch_fused(a, as_stream(stream)));
}

int fp8bs_gemm_fused_static(const uint16_t* x, int64_t M, int64_t ldx, const void* packed,
                            size_t packed_bytes, int64_t N, int64_t K, int scale_kind, uint16_t* y,
                            int64_t ldy, uint8_t* xq_out, void* xs_out, uint32_t* status_out,
                            unsigned flags, void* stream) {
    if (!kind_ok(scale_kind) || (flags & ~static_cast<unsigned>(FP8BS_FLAG_PDL)) != 0) return FP8BS_ERR_ARG;
    if (M < 0 || M > FP8BS_MAX_M || !nk_ok(N, K)) return FP8BS_ERR_SHAPE;
    if (M == 0) return FP8BS_OK;
    if (!x || !packed || !y) return FP8BS_ERR_ARG;
    if (ldx < K || ldy < N) return FP8BS_ERR_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(y, 16) || ldy % 8 != 0 || !aligned(packed, 256) ||
        (xq_out && !aligned(xq_out, 16)) || (xs_out && scale_kind == FP8BS_SCALE_F32 && !aligned(xs_out, 4)) ||
        (status_out && !aligned(status_out, 4)))
        return FP8BS_ERR_ALIGN;
    if (packed_bytes < fp8bs_packed_weight_bytes(N, K, scale_kind)) return FP8BS_ERR_WORKSPACE;
    if (K > FP8BS_STATIC_MAX_K) return FP8BS_ERR_WORKSPACE;
    int sm = 0;
    int rc = current_sm_count(&sm);
    if (rc != FP8BS_OK) return rc;
    if (sm > FP8BS_STATIC_MAX_SMS) sm = FP8BS_STATIC_MAX_SMS;
    if (!fused_shape_supported(N, K, sm)) return FP8BS_ERR_SHAPE;
    if (workspace_bytes_for(K, sm) > kStaticScratchBytes) return FP8BS_ERR_WORKSPACE;
    uint8_t* scratch = nullptr;
    rc = static_scratch(as_stream(stream), &scratch);
    if (rc != FP8BS_OK) return rc;
    FusedArgs a;
    a.x = x;
    a.ldx = ldx;
    a.packed = static_cast<const uint8_t*>(packed);
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.kind = scale_kind;
    a.y = y;
    a.ldy = ldy;
    a.workspace = scratch;
    a.xq_out = xq_out;
    a.xs_out = xs_out;
    a.sm_count = sm;
    a.timeout_cycles = timeout_cycles();
    a.pdl = (flags & FP8BS_FLAG_PDL) ? 1 : 0;
    rc = status_of(launch_fused_routed(a, as_stream(stream)));
    if (rc != FP8BS_OK || !status_out) return rc;
    // this call's status, then a clean error word for the next call (both in
    // stream order; a memset allocates nothing)
    if (cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, as_stream(stream)) !=
        cudaSuccess)
        return FP8BS_ERR_CUDA;
    return status_of(cudaMemsetAsync(scratch, 0, sizeof(uint32_t), as_stream(stream)));
}

int fp8bs_debug_config(long long timeout_cycles, int sm_count_override) {
    g_timeout_override.store(timeout_cycles > 0 ? timeout_cycles : 0, std::memory_order_relaxed);
    g_sm_override.store(sm_count_override > 0 ? sm_count_override : 0, std::memory_order_relaxed);
    return FP8BS_OK;
}

int fp8bs_trace_read(void* host_dst, size_t bytes) {
    static_assert(FP8BS_TRACE_CALLS == kTraceCalls && FP8BS_TRACE_CTAS == kTraceCtas &&
                      FP8BS_TRACE_POINTS == kTracePoints,
                  "fp8bs.h states the trace layout");
    if (!host_dst) return FP8BS_ERR_ARG;
    const cudaError_t e = trace_copy(host_dst, bytes);
    if (e == cudaErrorNotSupported) return FP8BS_ERR_ARG;
    return status_of(e);
}

int fp8bs_check_error(void* workspace, void* stream) {
    if (!workspace) return FP8BS_ERR_ARG;
    if (!aligned(workspace, 256)) return FP8BS_ERR_ALIGN;
    cudaStream_t s = as_stream(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8BS_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8BS_ERR_CUDA;
    if (word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return FP8BS_ERR_CUDA;
        return -static_cast<int>(word);
    }
    return FP8BS_OK;
}

}  // extern "C"
