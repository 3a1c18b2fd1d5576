// Small-M FP8 block-scale MoE layer.
//
// "[AMD] gfx950 small-batch MoE: expert-count gate for the small sort and FP8
// block-scale small-M kernel", "Modifications": float8_e4m3fn w13 / w2 weights
// with contiguous [128 x 128] fp32 block scales, each block's scale applied to
// its partial sum; bf16 activations; no sort.  Per token m and slot s (expert
// e = ids[m, s], weight w[m, s]):
//   h = x[m] . w13[e]^T                  (gate rows 0..I-1, up rows I..2I-1)
//   a = bf16(silu(h_gate) * h_up)
//   y[m] = bf16(sum_s w[m, s] * (a . w2[e]^T))
//
// At decode sizes almost every routed expert sees one token, so the layer is a
// grouped matrix-vector product bound by the weight bytes: CUDA-core FMAs on
// weights decoded in registers, with every active expert's weights read once
// (the tokens routed to one expert share the read).  Three launches, no
// cross-CTA waits:
//   1. gate/up: items (active expert, 64-row tile of w13, 512-column split
//      of H); partial sums per split into the workspace;
//   2. down: items (active expert, 64-row tile of w2); the splits are summed
//      in split order, silu * up rounded to bf16, then a . w2^T per slot into
//      the workspace;
//   3. combine: the slots of each token summed in slot order, bf16 out.
// Launches 2 and 3 use programmatic dependent launch: each starts (routing
// scan, L2 prefetch of its weights) while the previous one runs, and reads
// the previous one's results only after griddepcontrol.wait.
//
// Every CTA finds the active experts itself: the routed (token, slot) pairs
// are scanned into a bitmap over the experts, whose set bits in ascending
// order are the active list.  No sort and no extra launch; items are dealt
// out to a persistent grid.
#include "internal.cuh"
#include "moe.cuh"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int kMoeThreads = 256;
constexpr int kSplitCols = 512;  // columns of H per gate/up item
constexpr int kRowsPerWarp = 8;  // weight rows a warp owns in an item
constexpr int kItemRows = kRowsPerWarp * (kMoeThreads / 32);  // 64: half a scale block
constexpr int kDownBatch = 16;   // down: pairs whose a vectors sit in shared memory at once
constexpr int kMaxPairs = FP8BS_MOE_MAX_PAIRS;
constexpr int kBitmapWords = FP8BS_MOE_MAX_EXPERTS / 32;

struct MoeParams {
    const uint16_t* x;   // [M, H] bf16
    const int32_t* ids;  // [M, S]
    const float* tw;     // [M, S]
    const uint8_t* w13;  // [E, 2I, H]
    const float* s13;    // [E, 2I/128, H/128]
    const uint8_t* w2;   // [E, H, I]
    const float* s2;     // [E, H/128, I/128]
    uint16_t* y;         // [M, H] bf16
    uint32_t* err;       // workspace error word
    float* p1;           // [M*S][H/512][2I] gate/up partial sums
    float* p2;           // [M*S][H] down projections
    int M, S, H, I, E;
    int pdl;
};

struct Route {
    uint32_t bitmap[kBitmapWords];
    int16_t ids[kMaxPairs];     // -1 for an id outside [0, E)
    int16_t active[kMaxPairs];  // active experts, ascending
    int16_t list[kMaxPairs];    // pairs of the current item's expert, ascending
    int n_active;
    int n_list;
};
static_assert(FP8BS_MOE_MAX_EXPERTS <= 32767 && kMaxPairs <= 32767, "16-bit routing tables");

// Copies ids (recording out-of-range ones), then the ascending active list.
__device__ void route_setup(const MoeParams& p, Route& rs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int MS = p.M * p.S;
    for (int q = tid; q < MS; q += kMoeThreads) {
        int e = p.ids[q];
        if (e < 0 || e >= p.E) {
            record_error(p.err, FP8BS_ERR_DEVICE);
            e = -1;
        }
        rs.ids[q] = static_cast<int16_t>(e);
    }
    for (int w = tid; w < kBitmapWords; w += kMoeThreads) rs.bitmap[w] = 0;
    __syncthreads();
    for (int q = tid; q < MS; q += kMoeThreads) {
        const int e = rs.ids[q];
        if (e >= 0) atomicOr(&rs.bitmap[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int kPer = kBitmapWords / 32;
        int mine = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) mine += __popc(rs.bitmap[lane * kPer + j]);
        int incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
        }
        int at = incl - mine;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            uint32_t word = rs.bitmap[lane * kPer + j];
            while (word) {
                const int b = __ffs(word) - 1;
                rs.active[at++] = static_cast<int16_t>((lane * kPer + j) * 32 + b);
                word &= word - 1;
            }
        }
        if (lane == 31) rs.n_active = incl;
    }
    __syncthreads();
}

// The pairs routed to expert e, ascending (warp 0), then a barrier.
__device__ void build_list(const MoeParams& p, Route& rs, int e) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (tid < 32) {
        const int MS = p.M * p.S;
        int n = 0;
        for (int base = 0; base < MS; base += 32) {
            const int q = base + lane;
            const bool hit = q < MS && rs.ids[q] == e;
            const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hit);
            if (hit) rs.list[n + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(q);
            n += __popc(bal);
        }
        if (lane == 0) rs.n_list = n;
    }
    __syncthreads();
}

// Weight decode with integer operations only (no conversion instruction): a
// code's 7 magnitude bits become bits 4-10 of a bf16 (exponent field = the
// e4m3 exponent, mantissa top = its 3 bits) and its sign bit 15, so a normal
// code 2^(e-7)(1 + m/8) lands on 2^(e-127)(1 + m/8) and a subnormal m 2^-9 on
// the bf16 subnormal m 2^-129: exactly 2^-120 times the code's value.  The
// other factor carries 2^64 (kXScale) and the partial sums 2^56 (kAccScale),
// so every product is a normal fp32 number and every scaling an exact power of
// two.  Products and sums use the mixed-precision FMA (bf16 inputs, fp32
// accumulate): each product is exact.
constexpr float kXScale = 0x1p64f;
constexpr float kAccScale = 0x1p56f;

// One weight word (4 codes) -> two bf16 pairs, each value exactly 2^-120
// times the code's value (the bf16 form of the decode above): even holds
// codes 0 and 2, odd codes 1 and 3.
__device__ __forceinline__ void decode4_bf16(uint32_t v, uint32_t& even, uint32_t& odd) {
    even = ((v << 4) & 0x07F007F0u) | ((v << 8) & 0x80008000u);
    odd = ((v >> 4) & 0x07F007F0u) | (v & 0x80008000u);
}

// acc + a.lo * b.lo + a.hi * b.hi: bf16 inputs, fp32 products (exact) and sums.
__device__ __forceinline__ float fma2_bf16(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Two bf16 words (values 0,1 and 2,3) scaled by 2^64, regrouped as the weight
// decode pairs them: even = (0, 2), odd = (1, 3).  Exact (a power-of-two
// scaling of bf16 values below 2^64).
__device__ __forceinline__ void scale_pair_bf16(uint32_t w01, uint32_t w23, uint32_t& even, uint32_t& odd) {
    uint32_t s01, s23;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(s01)
        : "f"(__uint_as_float(w01 & 0xFFFF0000u) * kXScale), "f"(__uint_as_float(w01 << 16) * kXScale));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(s23)
        : "f"(__uint_as_float(w23 & 0xFFFF0000u) * kXScale), "f"(__uint_as_float(w23 << 16) * kXScale));
    even = __byte_perm(s01, s23, 0x5410);
    odd = __byte_perm(s01, s23, 0x7632);
}

__device__ __forceinline__ float bf16_round(float v) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return __uint_as_float(static_cast<uint32_t>(r) << 16);
}

// ---- 1. gate / up -----------------------------------------------------------
// Item (active expert, 64-row tile rt of w13, split ks of H): warp w takes rows
// 8w .. 8w+7 of the tile; lane l holds columns 16l .. 16l+15 of the split,
// so lanes 8b .. 8b+7 cover 128-column block b: their sum times that block's
// scale, then the sum over the split's 4 blocks, in a fixed order.  The
// warp's 4 KB of weights go to shared memory with cp.async first, so their
// reads overlap the routing list and the x loads.
template <int NP>
__device__ __forceinline__ void gate_up_rows(const MoeParams& p, const Route& rs, const uint8_t* sW, int pb, int ks,
                                             int KS, int I2, int row0, float scale, int lane) {
    uint32_t xe[NP][4], xo[NP][4];  // this lane's 16 x values, scaled and paired as the decode pairs
#pragma unroll
    for (int t = 0; t < NP; ++t) {
        const int m = rs.list[pb + t] / p.S;
        const uint4* src =
            reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(m) * p.H + ks * kSplitCols + lane * 16);
        const uint4 lo = src[0], hi = src[1];
        scale_pair_bf16(lo.x, lo.y, xe[t][0], xo[t][0]);
        scale_pair_bf16(lo.z, lo.w, xe[t][1], xo[t][1]);
        scale_pair_bf16(hi.x, hi.y, xe[t][2], xo[t][2]);
        scale_pair_bf16(hi.z, hi.w, xe[t][3], xo[t][3]);
    }
    ptx::cp_async_wait_all();
    __syncwarp();
#pragma unroll 4
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const uint4 wv = *reinterpret_cast<const uint4*>(sW + r * kSplitCols + lane * 16);
        const uint32_t words[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t we[4], wo[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) decode4_bf16(words[q], we[q], wo[q]);
#pragma unroll
        for (int t = 0; t < NP; ++t) {
            float acc = 0.0f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fma2_bf16(xe[t][q], we[q], acc);
                acc = fma2_bf16(xo[t][q], wo[q], acc);
            }
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
            acc = acc * kAccScale * scale;
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 8);
            acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
            if (lane == 0)
                p.p1[(static_cast<size_t>(rs.list[pb + t]) * KS + ks) * I2 + row0 + r] = acc;
        }
    }
}

__global__ void __launch_bounds__(kMoeThreads) moe_gate_up_kernel(const __grid_constant__ MoeParams p) {
    __shared__ Route rs;
    extern __shared__ __align__(16) uint8_t sW1[];  // [8 warps][8 rows][512 B]
    route_setup(p, rs);
    if (p.pdl) ptx::griddep_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int I2 = 2 * p.I, RT = I2 / kItemRows, KS = p.H / kSplitCols, HB = p.H / kTile;
    const int items = rs.n_active * RT * KS;
    uint8_t* sW = sW1 + warp * kRowsPerWarp * kSplitCols;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int a = it / (RT * KS);
        const int rem = it - a * RT * KS;
        const int rt = rem / KS, ks = rem - rt * KS;
        const int e = rs.active[a];
        const int row0 = rt * kItemRows + warp * kRowsPerWarp;
        const uint8_t* W = p.w13 + (static_cast<size_t>(e) * I2 + row0) * p.H + ks * kSplitCols + lane * 16;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
            ptx::cp_async16(sW + r * kSplitCols + lane * 16, W + static_cast<size_t>(r) * p.H);
        build_list(p, rs, e);
        const int n_list = rs.n_list;
        const float scale = p.s13[(static_cast<size_t>(e) * (I2 / kTile) + row0 / kTile) * HB +
                                  ks * (kSplitCols / kTile) + (lane >> 3)];
        int pb = 0;
        for (; pb + 2 <= n_list; pb += 2) gate_up_rows<2>(p, rs, sW, pb, ks, KS, I2, row0, scale, lane);
        if (pb < n_list) gate_up_rows<1>(p, rs, sW, pb, ks, KS, I2, row0, scale, lane);
        ptx::cp_async_wait_all();  // an expert with no pairs left still drains its copies
        __syncthreads();  // the list and the warp's staging are rewritten by the next item
    }
}

// ---- 2. down ------------------------------------------------------------------
// Item (active expert, 64-row tile nt of w2).  The warp's 8 rows of weights go
// to shared memory with cp.async first; meanwhile a = bf16(silu(g) * u) of
// each pair of the expert goes to shared memory (g, u: the gate/up splits
// summed in split order).  Then the rows: I/16 lanes per row (16 columns
// each, 8 lanes per 128-column block), 32 / (I/16) rows per warp step.
__global__ void __launch_bounds__(kMoeThreads) moe_down_kernel(const __grid_constant__ MoeParams p) {
    __shared__ Route rs;
    extern __shared__ __align__(16) uint8_t smem2[];  // weights [8 warps][8 rows][I], then a [kDownBatch][I] bf16
    route_setup(p, rs);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int I = p.I, I2 = 2 * I, NT = p.H / kItemRows, KS = p.H / kSplitCols, IB = I / kTile;
    const int items = rs.n_active * NT;
    uint8_t* sW = smem2 + warp * kRowsPerWarp * I;
    uint16_t* sA = reinterpret_cast<uint16_t*>(smem2 + kItemRows * I);
    // the first item's weights do not depend on the previous launch
    if (tid == 0 && static_cast<int>(blockIdx.x) < items) {
        const int e = rs.active[blockIdx.x / NT], nt = blockIdx.x % NT;
        ptx::bulk_prefetch_l2(p.w2 + (static_cast<size_t>(e) * p.H + nt * kItemRows) * I,
                              static_cast<uint32_t>(kItemRows * I));
    }
    if (p.pdl) {
        ptx::griddep_wait();
        ptx::griddep_launch_dependents();
    }
    const int cpr = I / 16;        // lanes per row
    const int rpw = 32 / cpr;      // rows per warp step
    const int lr = lane / cpr, lc = lane % cpr;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int e = rs.active[it / NT], nt = it % NT;
        const int row_base = nt * kItemRows + warp * kRowsPerWarp;
        const uint8_t* W = p.w2 + (static_cast<size_t>(e) * p.H + row_base) * I;
        for (int r0 = 0; r0 < kRowsPerWarp; r0 += rpw)
            ptx::cp_async16(sW + (r0 + lr) * I + lc * 16, W + static_cast<size_t>(r0 + lr) * I + lc * 16);
        build_list(p, rs, e);
        const int n_list = rs.n_list;
        const float scale = p.s2[(static_cast<size_t>(e) * (p.H / kTile) + row_base / kTile) * IB + (lc >> 3)];
        for (int pb = 0; pb < n_list; pb += kDownBatch) {
            const int np = n_list - pb < kDownBatch ? n_list - pb : kDownBatch;
            for (int idx = tid; idx < np * I; idx += kMoeThreads) {
                const int t = idx / I, i = idx - t * I;
                const float* P = p.p1 + static_cast<size_t>(rs.list[pb + t]) * KS * I2;
                float g = 0.0f, u = 0.0f;
#pragma unroll 8
                for (int ks = 0; ks < KS; ++ks) {
                    g += P[ks * I2 + i];
                    u += P[ks * I2 + I + i];
                }
                // a * 2^64 as bf16 (exact), laid out as the weight decode pairs the
                // values: for lane chunk c (values 16c .. 16c+15), word q of the
                // even half holds values 4q and 4q+2, of the odd half 4q+1 and
                // 4q+3; the two 16-byte halves of chunk c sit at uint4 index
                // (h * cpr + c), so the lanes of a row read consecutive words
                const float v = bf16_round(g / (1.0f + expf(-g)) * u) * kXScale;
                uint16_t bits;
                asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(bits) : "f"(v));
                const int c = i >> 4, k = i & 15, q = k >> 2, h = k & 1, half = (k >> 1) & 1;
                sA[t * I + ((h * cpr + c) * 4 + q) * 2 + half] = bits;
            }
            ptx::cp_async_wait_all();
            __syncthreads();
            for (int r0 = 0; r0 < kRowsPerWarp; r0 += rpw) {
                const int row = row_base + r0 + lr;
                const uint4 wv = *reinterpret_cast<const uint4*>(sW + (r0 + lr) * I + lc * 16);
                uint32_t we[4], wo[4];
                decode4_bf16(wv.x, we[0], wo[0]);
                decode4_bf16(wv.y, we[1], wo[1]);
                decode4_bf16(wv.z, we[2], wo[2]);
                decode4_bf16(wv.w, we[3], wo[3]);
                for (int t = 0; t < np; ++t) {
                    const uint4* av = reinterpret_cast<const uint4*>(sA + t * I) + lc;
                    const uint4 ae = av[0], ao = av[cpr];
                    float acc = 0.0f;
                    acc = fma2_bf16(ae.x, we[0], acc);
                    acc = fma2_bf16(ao.x, wo[0], acc);
                    acc = fma2_bf16(ae.y, we[1], acc);
                    acc = fma2_bf16(ao.y, wo[1], acc);
                    acc = fma2_bf16(ae.z, we[2], acc);
                    acc = fma2_bf16(ao.z, wo[2], acc);
                    acc = fma2_bf16(ae.w, we[3], acc);
                    acc = fma2_bf16(ao.w, wo[3], acc);
                    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
                    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
                    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
                    acc = acc * kAccScale * scale;
                    for (int off = 8; off < cpr; off <<= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
                    if (lc == 0) p.p2[static_cast<size_t>(rs.list[pb + t]) * p.H + row] = acc;
                }
            }
            __syncthreads();  // sA is rewritten by the next batch
        }
        ptx::cp_async_wait_all();
        __syncthreads();  // the list and the staging are rewritten by the next item
    }
}

// ---- 3. combine -----------------------------------------------------------------
// Four outputs per thread: y[m, n..n+3] = bf16(sum over s, in slot order, of
// w[m, s] * p2[m*S + s, n..n+3]); pairs with an invalid id contribute nothing.
__global__ void __launch_bounds__(kMoeThreads) moe_combine_kernel(const __grid_constant__ MoeParams p) {
    if (p.pdl) ptx::griddep_wait();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * kMoeThreads + threadIdx.x;
    const int H4 = p.H / 4;
    if (idx >= static_cast<int64_t>(p.M) * H4) return;
    const int m = static_cast<int>(idx / H4), n = static_cast<int>(idx - static_cast<int64_t>(m) * H4) * 4;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int s = 0; s < p.S; ++s) {
        const int q = m * p.S + s;
        const int e = p.ids[q];
        if (e < 0 || e >= p.E) continue;
        const float w = p.tw[q];
        const float4 v = *reinterpret_cast<const float4*>(p.p2 + static_cast<size_t>(q) * p.H + n);
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    uint16_t b[4];
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b[0]) : "f"(acc.x));
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b[1]) : "f"(acc.y));
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b[2]) : "f"(acc.z));
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(b[3]) : "f"(acc.w));
    *reinterpret_cast<uint2*>(p.y + static_cast<size_t>(m) * p.H + n) =
        make_uint2(b[0] | (static_cast<uint32_t>(b[1]) << 16), b[2] | (static_cast<uint32_t>(b[3]) << 16));
}

cudaError_t launch_pdl(void (*kern)(MoeParams), const MoeParams& p, int grid, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kMoeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t moe_workspace_bytes(int64_t M, int64_t S, int64_t H, int64_t I) {
    const int64_t pairs = M * S;
    return kMoeWsHeader + static_cast<size_t>(pairs) * (H / kSplitCols) * (2 * I) * sizeof(float) +
           static_cast<size_t>(pairs) * H * sizeof(float);
}

cudaError_t launch_moe(const MoeArgs& a, cudaStream_t stream) {
    MoeParams p;
    p.x = a.x;
    p.ids = a.ids;
    p.tw = a.tw;
    p.w13 = a.w13;
    p.s13 = a.s13;
    p.w2 = a.w2;
    p.s2 = a.s2;
    p.y = a.y;
    p.err = reinterpret_cast<uint32_t*>(a.workspace);
    p.p1 = reinterpret_cast<float*>(a.workspace + kMoeWsHeader);
    p.p2 = p.p1 + static_cast<size_t>(a.M) * a.S * (a.H / kSplitCols) * (2 * a.I);
    p.M = a.M;
    p.S = a.S;
    p.H = a.H;
    p.I = a.I;
    p.E = a.E;
    p.pdl = 1;
    // persistent grids: every SM filled to its occupancy (queried once per
    // device and intermediate size)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static int occ1[64] = {0};
    static int occ2[64][3] = {{0}};
    const size_t smem1 = static_cast<size_t>(kItemRows) * kSplitCols;
    const size_t smem2 = static_cast<size_t>(kItemRows) * a.I + static_cast<size_t>(kDownBatch) * a.I * sizeof(uint16_t);
    const int ii = a.I == 128 ? 0 : (a.I == 256 ? 1 : 2);
    cudaError_t e;
    if (occ1[dev] == 0) {
        e = cudaFuncSetAttribute(moe_gate_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem1));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(moe_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kItemRows * FP8BS_MOE_MAX_I +
                                                  kDownBatch * FP8BS_MOE_MAX_I * sizeof(uint16_t)));
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_gate_up_kernel, kMoeThreads, smem1);
        if (e != cudaSuccess) return e;
        occ1[dev] = n > 0 ? n : 1;
    }
    if (occ2[dev][ii] == 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, moe_down_kernel, kMoeThreads, smem2);
        if (e != cudaSuccess) return e;
        occ2[dev][ii] = n > 0 ? n : 1;
    }
    moe_gate_up_kernel<<<a.sm_count * occ1[dev], kMoeThreads, smem1, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = launch_pdl(moe_down_kernel, p, a.sm_count * occ2[dev][ii], smem2, stream);
    if (e != cudaSuccess) return e;
    const int64_t threads = static_cast<int64_t>(a.M) * (a.H / 4);
    return launch_pdl(moe_combine_kernel, p, static_cast<int>((threads + kMoeThreads - 1) / kMoeThreads), 0, stream);
}

}  // namespace fp8bs
