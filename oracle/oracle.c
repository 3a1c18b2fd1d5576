/*
 * CPU oracle for the small-M W8A8 FP8 block-scale linear with 1x128 activation
 * quantisation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: it exists so that tests, the smoke check and the CPU-baseline leg of
 * the benchmark can compare the CUDA library against a plain, slow, obviously
 * correct restatement of what the method computes.  It shares no code, header,
 * table or constant generator with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "[AMD] Small-M FP8 block-scale GEMM with fused activation quant for
 *        gfx950 (Qwen3.5)", section "Modifications": bf16 activations are
 *        quantised to fp8 in 1x128 groups with a per-group scale from the row
 *        amax; the fp8 weight carries a [N/128, K/128] fp32 scale
 *        (weight_scale_inv); one MMA per 128-wide K block, then x_scale*w_scale
 *        applied in fp32; bf16 output.
 *   [P2] "[AMD] gfx950 small-batch MoE: expert-count gate for the small sort and
 *        FP8 block-scale small-M kernel", section "Modifications": names the fp8
 *        format float8_e4m3fn and the 128x128 fp32 block scale applied to each
 *        partial sum, for the w13 / w2 weights of its small-M MoE layer.
 *   [P4] "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense 128x128 fp8
 *        linears (6/8)", sections "Motivation" and "Modifications": power-of-two
 *        128x128 weight scales stored as one e8m0 byte per block, and ue8m0
 *        per-1x128 activation scales emitted by the fused input_norm / q_norm
 *        (RMSNorm) producers.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - e4m3fn is the OCP FP8 E4M3 format: bias 7, no infinities, NaN = S.1111.111,
 *     largest finite 448.  Encoding rounds to nearest, ties to even, and any
 *     finite magnitude >= 448 saturates to +-448 (never NaN).
 *   - fp32 scale = amax / 448 as one IEEE fp32 division; codes = enc(x / scale),
 *     again one IEEE fp32 division.
 *   - a group whose amax is 0 gets scale 0 (fp32) or the e8m0 byte 0 (2^-127);
 *     its codes are the signed zeros of x.
 *   - ue8m0 scale = the smallest power of two >= fp32(amax / 448), exponent
 *     clamped to [-127, 127], stored as the byte exponent + 127.
 *   - the fp64 result is rounded straight to bf16, nearest-even.
 *   - the RMSNorm producer normalises each whole row, x * gamma /
 *     sqrt(mean x^2 + eps), rounds that to bf16 and quantises the bf16 values.
 *   - the MoE layer: gate rows over up rows in w13, a = bf16(silu(gate) * up),
 *     y = bf16(sum over slots of weight * (a . w2^T)) (details at
 *     oracle_moe_w8a16).
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off -pthread (no fast-math: every
 * fp32 operation below must be the IEEE one).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_SCALE_F32 0
#define ORACLE_SCALE_UE8M0 1

/* ------------------------------------------------------------------------- */
/* bf16 and fp32 bit views                                                   */
/* ------------------------------------------------------------------------- */

static float bits_to_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_to_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 is the upper half of an fp32: widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* Round-half-to-even of a non-negative double to an integer-valued double,
 * written out so that it does not depend on the FPU rounding mode. */
static double round_half_even(double r) {
    double fl = floor(r);
    double frac = r - fl; /* exact: r and fl share the binade or fl is 0 */
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* fp64 -> bf16, round to nearest even, in one step (no fp32 detour).
 * bf16 has 8 significant bits, exponent range of fp32, subnormals below 2^-126
 * with quantum 2^-133, and overflows to infinity past the largest finite value. */
uint16_t oracle_f64_to_bf16(double v) {
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    int ex;
    frexp(a, &ex);     /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;    /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;
    double q = ldexp(1.0, E - 7);      /* spacing of bf16 values in this binade */
    double n = round_half_even(a / q); /* a / q is exact (power-of-two scale) */
    /* n in [0, 256]; n == 256 carries into the next binade, which the sum below
     * handles; for E == -126 and n < 128 the same sum gives the subnormal code. */
    long bits = ((long)(E + 127) << 7) + ((long)n - 128);
    if (bits >= 0x7F80) return (uint16_t)(sign | 0x7F80u);
    return (uint16_t)(sign | (uint16_t)bits);
}

/* ------------------------------------------------------------------------- */
/* e4m3fn codec [P2 "Modifications" names float8_e4m3fn]                     */
/* ------------------------------------------------------------------------- */

/* Value of one e4m3fn code: S EEEE MMM, bias 7.  Exponent field 0 is the
 * subnormal binade 2^-6 * M/8; code S.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Nearest e4m3fn code to a finite fp32 value, ties to the even code, magnitudes
 * at or beyond 448 saturate to +-448.  The sign of zero is kept. */
uint8_t oracle_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    if (isnan(v)) return (uint8_t)(sign | 0x7F); /* outside the contract */
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);
    int E = ex - 1;            /* a in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;        /* below 2^-6 the spacing stays 2^-9 */
    double q = ldexp(1.0, E - 3);      /* three mantissa bits */
    double n = round_half_even(a / q); /* in [0, 16] */
    /* Normal: code = ((E + 7) << 3) | (n - 8) with n in [8, 16); n == 16 carries
     * into the exponent.  For E == -6 the same expression gives the subnormal
     * code n when n < 8.  a < 448 keeps the result at or below 0x7E. */
    int code = ((E + 7) << 3) + ((int)n - 8);
    return (uint8_t)(sign | (uint8_t)code);
}

/* Encode every fp32 bit pattern in [first, first + count) (used to check a
 * hardware conversion exhaustively).  NaN inputs give 0x7F | sign. */
void oracle_e4m3_encode_bits(uint32_t first, uint64_t count, uint8_t* out) {
    for (uint64_t i = 0; i < count; ++i)
        out[i] = oracle_e4m3_encode(bits_to_f32((uint32_t)(first + i)));
}

/* ------------------------------------------------------------------------- */
/* e8m0 scale bytes [P4 "Modifications": one byte per 128x128 block]         */
/* ------------------------------------------------------------------------- */

/* An e8m0 byte b stands for 2^(b - 127); 255 is NaN. */
double oracle_e8m0_decode(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Smallest power of two >= s (s >= 0, finite), as an e8m0 byte, exponent clamped
 * to [-127, 127].  s == 0 gives byte 0. */
uint8_t oracle_e8m0_ceil(float s) {
    if (!(s > 0.0f)) return 0;
    int ex;
    double f = frexp((double)s, &ex); /* s = f * 2^ex, f in [0.5, 1) */
    int e = (f == 0.5) ? ex - 1 : ex; /* exact power of two stays put */
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* The fp32 value of an e8m0 byte (2^-127 is an fp32 subnormal, still exact). */
static float e8m0_to_f32(uint8_t b) { return (float)ldexp(1.0, (int)b - 127); }

/* ------------------------------------------------------------------------- */
/* One quantisation group: n values -> scale + codes                          */
/* ------------------------------------------------------------------------- */

/* Quantise one group given as fp32 values.  For the fp32 kind *scale_f32 gets
 * amax/448; for ue8m0 *scale_e8m0 gets the byte and *scale_f32 its value. */
static void quant_group(const float* v, int n, int stride, int kind, uint8_t* codes,
                        int code_stride, float* scale_f32, uint8_t* scale_e8m0) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[(long)i * stride]);
        if (a > amax) amax = a;
    }
    float s = amax / 448.0f; /* one IEEE fp32 division */
    float scale;
    if (kind == ORACLE_SCALE_UE8M0) {
        uint8_t b = oracle_e8m0_ceil(s);
        *scale_e8m0 = b;
        scale = e8m0_to_f32(b);
    } else {
        scale = s;
    }
    *scale_f32 = scale;
    for (int i = 0; i < n; ++i) {
        float x = v[(long)i * stride];
        uint8_t c;
        if (amax == 0.0f)
            c = signbit(x) ? 0x80 : 0x00; /* zero group: signed zeros, no division */
        else
            c = oracle_e4m3_encode(x / scale); /* one IEEE fp32 division */
        codes[(long)i * code_stride] = c;
    }
}

/* ------------------------------------------------------------------------- */
/* Activation quantisation, 1x128 groups [P1 "Modifications"; P4 ue8m0]       */
/* ------------------------------------------------------------------------- */

/* x: bf16 [M, K] with row stride ldx (elements).  xq: [M, K] codes, row stride K.
 * xs: [M, K/128] fp32 (kind 0) or e8m0 bytes (kind 1), row-major.
 * Returns 0, or -1 on a bad shape. */
int oracle_quant_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, int kind,
                       uint8_t* xq, void* xs) {
    if (M < 0 || K < 0 || K % 128 != 0 || ldx < K) return -1;
    int64_t KB = K / 128;
    float vals[128];
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            for (int i = 0; i < 128; ++i) vals[i] = oracle_bf16_to_f32(x[m * ldx + kb * 128 + i]);
            float sf;
            uint8_t se = 0;
            quant_group(vals, 128, 1, kind, xq + m * K + kb * 128, 1, &sf, &se);
            if (kind == ORACLE_SCALE_UE8M0)
                ((uint8_t*)xs)[m * KB + kb] = se;
            else
                ((float*)xs)[m * KB + kb] = sf;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Weight quantisation, 128x128 blocks (input generator)                      */
/* [P1 "Modifications": [N/128, K/128] fp32 weight_scale_inv;                 */
/*  P4 "Modifications": power-of-two block scales as e8m0]                    */
/* ------------------------------------------------------------------------- */

/* W: fp32 [N, K] row-major.  wq: [N, K] codes.  ws: [N/128, K/128] fp32 or e8m0.
 * Same rules as the activation groups, over 128x128 blocks. */
int oracle_quant_weight_128x128(const float* W, int64_t N, int64_t K, int kind, uint8_t* wq,
                                void* ws) {
    if (N < 0 || K < 0 || N % 128 != 0 || K % 128 != 0) return -1;
    int64_t NB = N / 128, KB = K / 128;
    float* blk = (float*)malloc(sizeof(float) * 128 * 128);
    uint8_t* cb = (uint8_t*)malloc(128 * 128);
    if (!blk || !cb) {
        free(blk);
        free(cb);
        return -2;
    }
    for (int64_t nb = 0; nb < NB; ++nb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c) blk[r * 128 + c] = W[(nb * 128 + r) * K + kb * 128 + c];
            float sf;
            uint8_t se = 0;
            quant_group(blk, 128 * 128, 1, kind, cb, 1, &sf, &se);
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c) wq[(nb * 128 + r) * K + kb * 128 + c] = cb[r * 128 + c];
            if (kind == ORACLE_SCALE_UE8M0)
                ((uint8_t*)ws)[nb * KB + kb] = se;
            else
                ((float*)ws)[nb * KB + kb] = sf;
        }
    }
    free(blk);
    free(cb);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Block-scale GEMM [P1 "Modifications": one MMA per 128-wide K block, then   */
/* x_scale * w_scale; P2 "Modifications": the block scale multiplies each     */
/* partial sum]                                                               */
/*                                                                           */
/*   Y[m,n] = bf16( sum_kb ( sum_{k in kb} xq[m,k] wq[n,k] ) xs[m,kb] ws[n/128,kb] ) */
/*                                                                           */
/* The inner sum is exact in fp64 (each product has at most 8 significant    */
/* bits and lies within [2^-18, 448^2]; 128 terms need fewer than 53 bits).   */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint8_t* xq;
    const void* xs;
    const uint8_t* wq;
    const void* ws;
    int64_t M, N, K;
    int kind;
    uint16_t* y;
    double* y64;
    int64_t n_begin, n_end;
    const double* table;
} gemm_job;

static double scale_value(const void* s, int64_t idx, int kind) {
    if (kind == ORACLE_SCALE_UE8M0) return oracle_e8m0_decode(((const uint8_t*)s)[idx]);
    return (double)((const float*)s)[idx];
}

static void* gemm_rows(void* arg) {
    gemm_job* j = (gemm_job*)arg;
    int64_t KB = j->K / 128;
    for (int64_t m = 0; m < j->M; ++m) {
        for (int64_t n = j->n_begin; n < j->n_end; ++n) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double p = 0.0;
                const uint8_t* a = j->xq + m * j->K + kb * 128;
                const uint8_t* b = j->wq + n * j->K + kb * 128;
                for (int i = 0; i < 128; ++i) p += j->table[a[i]] * j->table[b[i]];
                double sx = scale_value(j->xs, m * KB + kb, j->kind);
                double sw = scale_value(j->ws, (n / 128) * KB + kb, j->kind);
                acc += p * sx * sw;
            }
            if (j->y) j->y[m * j->N + n] = oracle_f64_to_bf16(acc);
            if (j->y64) j->y64[m * j->N + n] = acc;
        }
    }
    return NULL;
}

/* xq [M,K] codes, xs [M,K/128], wq [N,K] codes, ws [N/128,K/128] (fp32 or e8m0
 * per kind).  y: bf16 [M,N] (nullable); y64: fp64 [M,N] before rounding
 * (nullable).  nthreads > 1 splits the N rows over POSIX threads. */
int oracle_gemm(const uint8_t* xq, const void* xs, const uint8_t* wq, const void* ws, int64_t M,
                int64_t N, int64_t K, int kind, uint16_t* y, double* y64, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 128 != 0) return -1;
    double table[256];
    for (int c = 0; c < 256; ++c) table[c] = oracle_e4m3_decode((uint8_t)c);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    gemm_job jobs[256];
    pthread_t tids[256];
    int64_t chunk = (N + nthreads - 1) / nthreads;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        gemm_job jb = {xq, xs, wq, ws, M, N, K, kind, y, y64, t * chunk, (t + 1) * chunk, table};
        if (jb.n_end > N) jb.n_end = N;
        if (jb.n_begin >= jb.n_end) break;
        jobs[t] = jb;
        if (nthreads == 1) {
            gemm_rows(&jobs[t]);
        } else if (pthread_create(&tids[t], NULL, gemm_rows, &jobs[t]) != 0) {
            gemm_rows(&jobs[t]); /* no thread available: do it here */
            tids[t] = 0;
        }
        launched = t + 1;
    }
    if (nthreads > 1)
        for (int t = 0; t < launched; ++t)
            if (tids[t]) pthread_join(tids[t], NULL);
    return 0;
}

/* The whole linear: quantise x in 1x128 groups, then the block-scale GEMM.
 * xq/xs are scratch the caller provides ([M,K] bytes, [M,K/128] scales). */
int oracle_linear(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* wq,
                  const void* ws, int64_t N, int kind, uint8_t* xq, void* xs, uint16_t* y,
                  int nthreads) {
    int rc = oracle_quant_1x128(x, M, K, ldx, kind, xq, xs);
    if (rc) return rc;
    return oracle_gemm(xq, xs, wq, ws, M, N, K, kind, y, NULL, nthreads);
}

/* Bit helpers exposed for tests of the rounding rules. */
uint32_t oracle_f32_bits(float f) { return f32_to_bits(f); }

/* ------------------------------------------------------------------------- */
/* RMSNorm producer [P4 "Modifications": the fused input_norm / q_norm       */
/* producers emit the ue8m0 (or fp32) 1x128 scales of the normalised         */
/* activations, so the quant adds no launch]                                 */
/* ------------------------------------------------------------------------- */

/* Readings (the pages name the producer but print no formula):
 *   - RMSNorm over the whole row of K values:
 *       y[m,k] = x[m,k] * gamma[k] / sqrt(mean_k x[m,k]^2 + eps),
 *     x and gamma bf16, evaluated here in fp64;
 *   - the producer's output activation is that value rounded to bf16
 *     (nearest-even), and the 1x128 quant above takes those bf16 values, so the
 *     fused producer gives the bytes of "RMSNorm, then quant".
 * x: bf16 [M, K], row stride ldx.  gamma: bf16 [K].  y64: fp64 [M, K] (nullable),
 * y: bf16 [M, K] (nullable), both row stride K.  Returns 0, or -1 on a bad shape
 * or a negative eps. */
int oracle_rmsnorm(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const uint16_t* gamma,
                   double eps, double* y64, uint16_t* y) {
    if (M < 0 || K <= 0 || ldx < K || !(eps >= 0.0)) return -1;
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)oracle_bf16_to_f32(x[m * ldx + k]);
            ss += v * v;
        }
        double rms = sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)oracle_bf16_to_f32(x[m * ldx + k]);
            double g = (double)oracle_bf16_to_f32(gamma[k]);
            double r = rms > 0.0 ? v * g / rms : 0.0 * v * g; /* zero row, eps 0: signed zero */
            if (y64) y64[m * K + k] = r;
            if (y) y[m * K + k] = oracle_f64_to_bf16(r);
        }
    }
    return 0;
}

/* The producer: RMSNorm (above), rounded to bf16, then the 1x128 quant.
 * y: bf16 [M, K] scratch/output the caller provides; xq [M, K]; xs [M, K/128]. */
int oracle_rmsnorm_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                         const uint16_t* gamma, double eps, int kind, uint16_t* y, uint8_t* xq,
                         void* xs) {
    if (K % 128 != 0) return -1;
    int rc = oracle_rmsnorm(x, M, K, ldx, gamma, eps, NULL, y);
    if (rc) return rc;
    return oracle_quant_1x128(y, M, K, K, kind, xq, xs);
}

/* ------------------------------------------------------------------------- */
/* Small-M FP8 block-scale MoE [P2 "Modifications": float8_e4m3fn w13 / w2   */
/* with contiguous [128 x 128] fp32 block scales, each block's scale applied  */
/* to its partial sum; bf16 activations; routing given per token as S slots]  */
/* ------------------------------------------------------------------------- */

/* Readings (the page names the weights and the scale rule, not the layer):
 *   - w13[e] stacks the gate rows (0 .. I-1) over the up rows (I .. 2I-1),
 *     each [2I, H] row-major; w2[e] is [H, I]; scales s13 [E][2I/128][H/128]
 *     and s2 [E][H/128][I/128], fp32;
 *   - h = x . w13[e]^T with, per 128-wide K block, the block's partial sum
 *     times its scale (x in bf16, weights decoded exactly);
 *   - a = silu(h_gate) * h_up with silu(g) = g / (1 + exp(-g)), rounded to
 *     bf16: the intermediate activation the down projection reads;
 *   - o = a . w2[e]^T, the same block-scale rule;
 *   - y[m] = bf16(sum over the token's S slots of topk_w * o), with every slot
 *     summed (a token routed twice to one expert counts twice).
 * Everything else in fp64.  x: bf16 [M, H]; ids: int32 [M, S] in [0, E);
 * w: fp32 [M, S]; y: bf16 [M, H] (nullable); y64: fp64 [M, H] (nullable).
 * Returns 0, or -1 on a bad shape or an expert id out of range. */
int oracle_moe_w8a16(const uint16_t* x, int64_t M, int64_t H, const int32_t* ids,
                     const float* w, int64_t S, const uint8_t* w13, const float* s13,
                     const uint8_t* w2, const float* s2, int64_t E, int64_t I, uint16_t* y,
                     double* y64) {
    if (M < 0 || S < 1 || E < 1 || H <= 0 || I <= 0 || H % 128 != 0 || I % 128 != 0) return -1;
    for (int64_t p = 0; p < M * S; ++p)
        if (ids[p] < 0 || ids[p] >= E) return -1;
    double table[256];
    for (int c = 0; c < 256; ++c) table[c] = oracle_e4m3_decode((uint8_t)c);
    const int64_t HB = H / 128, IB = I / 128;
    double* h = (double*)malloc(sizeof(double) * (size_t)(2 * I));
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* acc = (double*)malloc(sizeof(double) * (size_t)H);
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    if (!h || !a || !acc || !xv) {
        free(h); free(a); free(acc); free(xv);
        return -1;
    }
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < H; ++k) xv[k] = (double)oracle_bf16_to_f32(x[m * H + k]);
        for (int64_t n = 0; n < H; ++n) acc[n] = 0.0;
        for (int64_t s = 0; s < S; ++s) {
            const int64_t e = ids[m * S + s];
            const uint8_t* W13 = w13 + e * (2 * I) * H;
            const float* S13 = s13 + e * (2 * I / 128) * HB;
            for (int64_t j = 0; j < 2 * I; ++j) {
                double hj = 0.0;
                for (int64_t kb = 0; kb < HB; ++kb) {
                    double part = 0.0;
                    for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) part += xv[k] * table[W13[j * H + k]];
                    hj += part * (double)S13[(j / 128) * HB + kb];
                }
                h[j] = hj;
            }
            for (int64_t i = 0; i < I; ++i) {
                const double g = h[i], u = h[I + i];
                const double act = g / (1.0 + exp(-g)) * u;
                a[i] = (double)oracle_bf16_to_f32(oracle_f64_to_bf16(act));
            }
            const uint8_t* W2 = w2 + e * H * I;
            const float* S2 = s2 + e * HB * IB;
            const double ws = (double)w[m * S + s];
            for (int64_t n = 0; n < H; ++n) {
                double o = 0.0;
                for (int64_t ib = 0; ib < IB; ++ib) {
                    double part = 0.0;
                    for (int64_t i = ib * 128; i < ib * 128 + 128; ++i) part += a[i] * table[W2[n * I + i]];
                    o += part * (double)S2[(n / 128) * IB + ib];
                }
                acc[n] += ws * o;
            }
        }
        for (int64_t n = 0; n < H; ++n) {
            if (y) y[m * H + n] = oracle_f64_to_bf16(acc[n]);
            if (y64) y64[m * H + n] = acc[n];
        }
    }
    free(h); free(a); free(acc); free(xv);
    return 0;
}
