/*
 * CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, single-threaded
 * restatement of what the method computes.  Only the test-suite, the smoke
 * check and the benchmark's CPU-baseline leg load it; the product library
 * never does.  It shares no source, header, table or constant with the CUDA
 * path.  Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off (see
 * oracle/build.py); floating point must stay IEEE (no -ffast-math).
 *
 * Sources (DeepSeek-V3 FP8 training excerpts; each page named by its address):
 *   [P2] xn--jj0bz6z98ct0a29q.com, board post 362465 -- increased-precision
 *        accumulation absorbs the dequantization of per-group scales.
 *   [P3] why-be.why-be.co.kr, board post 55081 -- Figure 7(b): tensor-core
 *        partial sums are copied to FP32 registers on CUDA cores at a fixed
 *        interval and accumulated there; fine groups adapt the scale to
 *        outliers.
 *   [P4] sunipension.com, board post 314414 -- Figure 7(a): activations are
 *        grouped and scaled per 1x128 tile (per token per 128 channels),
 *        weights per 128x128 block (128 input x 128 output channels); cached
 *        activations are converted from 1x128 tiles to 128x1 tiles for the
 *        backward pass; Figure 6: the Wgrad GEMM runs in FP8.
 *   [P1] why-be.why-be.co.kr, board post 65900 -- the scaling rule maps the
 *        largest magnitude of a group onto the largest FP8 value.
 *
 * Readings where the pages are silent or garbled (each also listed in the
 * design notes of the repository):
 *   R1 FP8 format is OCP E4M3 ("e4m3fn"): bias 7, no infinities, 0x7F/0xFF
 *      NaN, largest finite 448, smallest subnormal 2^-9.
 *   R2 scale s = amax / 448 as ONE IEEE fp32 division (round to nearest even),
 *      no flush to zero, not rounded to a power of two.
 *   R3 code = E4M3 round-to-nearest-even, saturating at +-448, of the fp32
 *      quotient x / s (ONE IEEE fp32 division).  The sign is kept, so a
 *      negative value whose quotient rounds to zero gives 0x80.
 *   R4 a group whose amax is 0 stores s = 0 and all codes 0x00.
 *   R5 the requantizer first dequantizes in fp32: xhat = decode(q) * s_in, one
 *      fp32 multiply, then quantizes 128x1 groups of xhat exactly as above.
 *   R6 the promotion interval equals the quantization group (128 along K), so
 *      the GEMM equals the FP64 product of the dequantized operands, summed in
 *      ascending k.
 *   R7 inputs are finite; NaN/Inf are outside the contract.
 *   R13 SwiGLU recompute: the SwiGLU output y = silu(g) * u = g * u / (1 + e^-g)
 *      of a cached bf16 gate g and up projection u, evaluated in FP64 (libm
 *      exp) and rounded once to bf16 (nearest, ties to even), is what the fused
 *      recompute-and-quantize step 1x128-quantizes.  Page: why-be.why-be.co.kr
 *      post 65900 (the inputs of the SwiGLU operator are cached and its output
 *      recomputed in the backward pass).
 *   R12 the power-of-two variant (the "_pow2" entry points): the scale is the
 *      smallest power of two s = 2^e with amax / s <= 448 (the exact
 *      2^ceil(log2(amax/448))), e clamped below at -127, the smallest scale an
 *      8-bit exponent (UE8M0) can hold; a zero group keeps s = 0.  The quotient
 *      x / s is then exact (a power-of-two division), and code = E4M3 RNE of it.
 *      Pages: why-be.why-be.co.kr post 55081 and sunipension.com post 314414
 *      give these scales as integral powers of 2 for the inputs of the Linear
 *      after attention and the gradients before the MoE down-projection.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define Q_GROUP 128
#define E4M3_MAX 448.0f

/* ---------------------------------------------------------------- E4M3 --- */

/* Value of a non-negative E4M3 code 0x00..0x7E (R1).  Exponent field e, mantissa
 * field m: e == 0 is subnormal, m/8 * 2^(1-7); otherwise (1 + m/8) * 2^(e-7). */
static double e4m3_magnitude(int code)
{
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    if (e == 0)
        return ldexp((double)m, -9);
    return ldexp(8.0 + (double)m, e - 10);
}

/* Decode any code to a double (exact); NaN for 0x7F and 0xFF. */
static const double *magnitudes(void);

double orc_e4m3_decode(uint8_t code)
{
    int mag = code & 0x7F;
    double v;
    if (mag == 0x7F)
        return NAN;
    v = magnitudes()[mag];
    return (code & 0x80) ? -v : v;
}

/* The 127 finite non-negative magnitudes, indexed by code 0x00..0x7E. */
static double mag_table[0x7F];
static int mag_table_ready = 0;

static const double *magnitudes(void)
{
    int c;
    if (!mag_table_ready) {
        for (c = 0; c < 0x7F; ++c)
            mag_table[c] = e4m3_magnitude(c);
        mag_table_ready = 1;
    }
    return mag_table;
}

/* Round an fp32 value to the nearest E4M3 code, ties to the even code (the code
 * whose mantissa LSB is 0), saturating to +-448 (R3).  Brute force: find the
 * bracketing pair of representable magnitudes by bisection over the 127 finite
 * codes (their values increase with the code), then compare with the midpoint
 * of the pair, which is exact in double. */
uint8_t orc_e4m3_encode(float y)
{
    const double *mag = magnitudes();
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    int lo = 0, hi = 0x7E, c;
    double mid;

    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    while (lo < hi) {           /* largest code with magnitude <= a */
        int t = (lo + hi + 1) / 2;
        if (mag[t] <= a)
            lo = t;
        else
            hi = t - 1;
    }
    if (mag[lo] == a)
        return (uint8_t)(sign | lo);
    mid = 0.5 * (mag[lo] + mag[lo + 1]);
    if (a < mid)
        c = lo;
    else if (a > mid)
        c = lo + 1;
    else
        c = (lo & 1) ? lo + 1 : lo;
    return (uint8_t)(sign | c);
}

/* ------------------------------------------------------------ helpers --- */

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Power-of-two scale of a group with largest magnitude amax > 0, reading
 * R12: the smallest 2^e (e >= -127) with amax <= 448 * 2^e.  Every comparison
 * is exact in double. */
static float pow2_scale(float amax)
{
    int e = -127;
    while (ldexp((double)E4M3_MAX, e) < (double)amax)
        ++e;
    return (float)ldexp(1.0, e);
}

/* Quantize one group of n fp32 values (amax -> scale -> codes), [P1], [P4]
 * Figure 7(a), readings R2-R4, or R12 when pow2 != 0.  Element i is read at
 * x[i*xs] and its code is written at q[i*qs]. */
static void quantize_group(const float *x, int64_t n, int64_t xs,
                           uint8_t *q, int64_t qs, float *s_out, int pow2)
{
    float amax = 0.0f, s;
    int64_t i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(x[i * xs]);
        if (a > amax)
            amax = a;
    }
    if (pow2)
        s = (amax == 0.0f) ? 0.0f : pow2_scale(amax);
    else
        s = amax / E4M3_MAX;
    *s_out = s;
    for (i = 0; i < n; ++i) {
        if (amax == 0.0f)
            q[i * qs] = 0x00;
        else if (pow2)   /* exact quotient; only values far below E4M3's range can round */
            q[i * qs] = orc_e4m3_encode((float)((double)x[i * xs] / (double)s));
        else
            q[i * qs] = orc_e4m3_encode(x[i * xs] / s);
    }
}

/* -------------------------------------------------------- quantizers --- */

/* 1x128 activation quantization, [P4] Figure 7(a): every row m is cut into
 * K/128 groups of 128 consecutive channels.
 *   x  bf16 bit patterns [M][K], row stride ldx (elements)
 *   q  codes [M][K], row stride ldq
 *   s  scales [M][K/128], row-major, dense
 * Returns 0, or -1 when K is not a multiple of 128. */
static int quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                           uint8_t *q, int64_t ldq, float *s, int pow2)
{
    float buf[Q_GROUP];
    int64_t m, kb, i, KB;
    if (K % Q_GROUP)
        return -1;
    KB = K / Q_GROUP;
    for (m = 0; m < M; ++m)
        for (kb = 0; kb < KB; ++kb) {
            for (i = 0; i < Q_GROUP; ++i)
                buf[i] = bf16_to_f32(x[m * ldx + kb * Q_GROUP + i]);
            quantize_group(buf, Q_GROUP, 1, q + m * ldq + kb * Q_GROUP, 1,
                           s + m * KB + kb, pow2);
        }
    return 0;
}

int orc_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t *q, int64_t ldq, float *s)
{
    return quant_act_1x128(x, M, K, ldx, q, ldq, s, 0);
}

/* The same with power-of-two scales (R12). */
int orc_quant_act_1x128_pow2(const uint16_t *x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t *q, int64_t ldq, float *s)
{
    return quant_act_1x128(x, M, K, ldx, q, ldq, s, 1);
}

/* 128x128 weight quantization, [P4] Figure 7(a): W[K][N] (K = input channels,
 * N = output channels) is cut into 128x128 blocks, one scale per block.
 *   w  bf16 bit patterns [K][N], row stride ldw
 *   q  codes [K][N] (same layout as w), row stride ldq
 *   s  scales [K/128][N/128], row-major, dense
 * Returns 0, or -1 when K or N is not a multiple of 128. */
static int quant_w_128x128(const uint16_t *w, int64_t K, int64_t N, int64_t ldw,
                           uint8_t *q, int64_t ldq, float *s, int pow2)
{
    float blk[Q_GROUP * Q_GROUP];
    uint8_t qb[Q_GROUP * Q_GROUP];
    int64_t kb, nb, i, j, KB, NB;
    if (K % Q_GROUP || N % Q_GROUP)
        return -1;
    KB = K / Q_GROUP;
    NB = N / Q_GROUP;
    for (kb = 0; kb < KB; ++kb)
        for (nb = 0; nb < NB; ++nb) {
            for (i = 0; i < Q_GROUP; ++i)
                for (j = 0; j < Q_GROUP; ++j)
                    blk[i * Q_GROUP + j] =
                        bf16_to_f32(w[(kb * Q_GROUP + i) * ldw + nb * Q_GROUP + j]);
            quantize_group(blk, Q_GROUP * Q_GROUP, 1, qb, 1, s + kb * NB + nb, pow2);
            for (i = 0; i < Q_GROUP; ++i)
                for (j = 0; j < Q_GROUP; ++j)
                    q[(kb * Q_GROUP + i) * ldq + nb * Q_GROUP + j] = qb[i * Q_GROUP + j];
        }
    return 0;
}

int orc_quant_w_128x128(const uint16_t *w, int64_t K, int64_t N, int64_t ldw,
                        uint8_t *q, int64_t ldq, float *s)
{
    return quant_w_128x128(w, K, N, ldw, q, ldq, s, 0);
}

/* The same with power-of-two scales (R12). */
int orc_quant_w_128x128_pow2(const uint16_t *w, int64_t K, int64_t N, int64_t ldw,
                             uint8_t *q, int64_t ldq, float *s)
{
    return quant_w_128x128(w, K, N, ldw, q, ldq, s, 1);
}

/* 1x128 -> 128x1 requantization for the backward pass, [P4] ("converted from a
 * 1x128 tile to a 128x1 tile"), reading R5.  Each value is dequantized in fp32
 * with its row-group scale, then every channel k is quantized in groups of 128
 * consecutive tokens, and the result is written transposed.
 *   q   codes [M][K], row stride ldq;  s  scales [M][K/128] row-major dense
 *   qT  codes [K][M], row stride ldqT; sT scales [K][M/128] row-major dense
 * Returns 0, or -1 when M or K is not a multiple of 128. */
static int requant_1x128_to_128x1(const uint8_t *q, const float *s, int64_t M, int64_t K,
                                  int64_t ldq, uint8_t *qT, int64_t ldqT, float *sT, int pow2)
{
    float col[Q_GROUP];
    int64_t k, mb, i, KB, MB;
    if (M % Q_GROUP || K % Q_GROUP)
        return -1;
    KB = K / Q_GROUP;
    MB = M / Q_GROUP;
    for (k = 0; k < K; ++k)
        for (mb = 0; mb < MB; ++mb) {
            for (i = 0; i < Q_GROUP; ++i) {
                int64_t m = mb * Q_GROUP + i;
                float dec = (float)orc_e4m3_decode(q[m * ldq + k]);
                col[i] = dec * s[m * KB + k / Q_GROUP];     /* one fp32 multiply */
            }
            quantize_group(col, Q_GROUP, 1, qT + k * ldqT + mb * Q_GROUP, 1,
                           sT + k * MB + mb, pow2);
        }
    return 0;
}

int orc_requant_1x128_to_128x1(const uint8_t *q, const float *s, int64_t M, int64_t K,
                               int64_t ldq, uint8_t *qT, int64_t ldqT, float *sT)
{
    return requant_1x128_to_128x1(q, s, M, K, ldq, qT, ldqT, sT, 0);
}

/* The same with power-of-two scales (R12) for the 128x1 groups; the input
 * scales are whatever the 1x128 codes were made with (powers of two in the
 * power-of-two pipeline, so the dequantizing multiply is exact there). */
int orc_requant_1x128_to_128x1_pow2(const uint8_t *q, const float *s, int64_t M, int64_t K,
                                    int64_t ldq, uint8_t *qT, int64_t ldqT, float *sT)
{
    return requant_1x128_to_128x1(q, s, M, K, ldq, qT, ldqT, sT, 1);
}

/* ------------------------------------------------------------- GEMMs --- */

/* Scale-granularity of operand B. */
#define ORC_SB_BLOCK128x128 0   /* sB[kb][n/128], dense [K/128][ceil(N/128)] */
#define ORC_SB_COL128x1     1   /* sB[kb][n],     dense [K/128][N]           */

static double sb_at(const float *sB, int sb_kind, int64_t kb, int64_t n, int64_t N)
{
    if (sb_kind == ORC_SB_COL128x1)
        return (double)sB[kb * N + n];
    return (double)sB[kb * ((N + Q_GROUP - 1) / Q_GROUP) + n / Q_GROUP];
}

/* One output element of the block-scaled GEMM, [P3] Figure 7(b), [P2],
 * reading R6: sum over ascending k of (decode(A[m][k]) * sA[m][k/128]) *
 * (decode(Bt[n][k]) * sB(k/128, n)), every product and sum in FP64.
 *   A   codes [M][K] row-major (lda);  sA [M][K/128] row-major dense
 *   Bt  codes of B stored K-major, Bt[n][k] = B[k][n] (ldb) */
static double gemm_element(const uint8_t *A, int64_t lda, const float *sA,
                           const uint8_t *Bt, int64_t ldb, const float *sB, int sb_kind,
                           int64_t m, int64_t n, int64_t N, int64_t K)
{
    int64_t k, KB = K / Q_GROUP;
    double acc = 0.0;
    for (k = 0; k < K; ++k) {
        double a = orc_e4m3_decode(A[m * lda + k]) * (double)sA[m * KB + k / Q_GROUP];
        double b = orc_e4m3_decode(Bt[n * ldb + k]) * sb_at(sB, sb_kind, k / Q_GROUP, n, N);
        acc += a * b;
    }
    return acc;
}

/* Full block-scaled GEMM: C[m][n] (double, [M][N] dense).  Returns -1 when K is
 * not a multiple of 128 or sb_kind is unknown. */
int orc_gemm_blockscaled(const uint8_t *A, int64_t lda, const float *sA,
                         const uint8_t *Bt, int64_t ldb, const float *sB, int sb_kind,
                         int64_t M, int64_t N, int64_t K, double *C)
{
    int64_t m, n;
    if (K % Q_GROUP || (sb_kind != ORC_SB_BLOCK128x128 && sb_kind != ORC_SB_COL128x1))
        return -1;
    for (m = 0; m < M; ++m)
        for (n = 0; n < N; ++n)
            C[m * N + n] = gemm_element(A, lda, sA, Bt, ldb, sB, sb_kind, m, n, N, K);
    return 0;
}

/* The same GEMM evaluated only at the `count` positions (ms[i], ns[i]). */
int orc_gemm_blockscaled_sample(const uint8_t *A, int64_t lda, const float *sA,
                                const uint8_t *Bt, int64_t ldb, const float *sB, int sb_kind,
                                int64_t M, int64_t N, int64_t K,
                                const int64_t *ms, const int64_t *ns, int64_t count, double *out)
{
    int64_t i;
    if (K % Q_GROUP || (sb_kind != ORC_SB_BLOCK128x128 && sb_kind != ORC_SB_COL128x1))
        return -1;
    for (i = 0; i < count; ++i) {
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N)
            return -2;
        out[i] = gemm_element(A, lda, sA, Bt, ldb, sB, sb_kind, ms[i], ns[i], N, K);
    }
    return 0;
}

/* Expert that owns row m, or -1 for a row outside every expert's range. */
static int expert_of_row(const int32_t *offsets, int G, int64_t m)
{
    int g;
    for (g = 0; g < G; ++g)
        if (m >= offsets[g] && m < offsets[g + 1])
            return g;
    return -1;
}

/* Grouped (MoE) block-scaled GEMM: expert g owns the rows [offsets[g],
 * offsets[g+1]) of A and multiplies them by its own weight B_g, [P2] (FP8
 * dispatch of MoE activations) with the GEMM of R6 per expert.
 *   A  codes [M_total][K] (lda);  sA [M_total][K/128] row-major dense
 *   B  codes [G][N][K] (each expert K-major, dense); sB [G][K/128][N/128] dense
 *   C  double [M_total][N]; rows outside every expert are left untouched. */
int orc_grouped_gemm_blockscaled(const uint8_t *A, int64_t lda, const float *sA,
                                 const uint8_t *B, const float *sB,
                                 const int32_t *offsets, int G,
                                 int64_t M_total, int64_t N, int64_t K, double *C)
{
    int64_t m, n, KB = K / Q_GROUP, NB = (N + Q_GROUP - 1) / Q_GROUP;
    int g;
    if (K % Q_GROUP || G <= 0)
        return -1;
    for (g = 0; g < G; ++g)
        if (offsets[g] > offsets[g + 1] || offsets[g] < 0 || offsets[g + 1] > M_total)
            return -2;
    for (m = 0; m < M_total; ++m) {
        g = expert_of_row(offsets, G, m);
        if (g < 0)
            continue;
        for (n = 0; n < N; ++n)
            C[m * N + n] = gemm_element(A, lda, sA, B + (int64_t)g * N * K, K,
                                        sB + (int64_t)g * KB * NB, ORC_SB_BLOCK128x128,
                                        m, n, N, K);
    }
    return 0;
}

/* The grouped GEMM evaluated only at (ms[i], ns[i]); a row outside every
 * expert yields NaN. */
int orc_grouped_gemm_blockscaled_sample(const uint8_t *A, int64_t lda, const float *sA,
                                        const uint8_t *B, const float *sB,
                                        const int32_t *offsets, int G,
                                        int64_t M_total, int64_t N, int64_t K,
                                        const int64_t *ms, const int64_t *ns, int64_t count,
                                        double *out)
{
    int64_t i, KB = K / Q_GROUP, NB = (N + Q_GROUP - 1) / Q_GROUP;
    if (K % Q_GROUP || G <= 0)
        return -1;
    for (i = 0; i < count; ++i) {
        int g;
        if (ms[i] < 0 || ms[i] >= M_total || ns[i] < 0 || ns[i] >= N)
            return -2;
        g = expert_of_row(offsets, G, ms[i]);
        out[i] = (g < 0) ? NAN
                         : gemm_element(A, lda, sA, B + (int64_t)g * N * K, K,
                                        sB + (int64_t)g * KB * NB, ORC_SB_BLOCK128x128,
                                        ms[i], ns[i], N, K);
    }
    return 0;
}

/* --------------------------------------------------------------- SwiGLU --- */

/* Round a finite double to the nearest bf16 value, ties to even; bf16 has 8
 * significant bits, subnormals down to 2^-133, and overflows to infinity
 * above its largest finite value (2 - 2^-7) * 2^127 by half an ulp or more.
 * Returns the bf16 bit pattern. */
static uint16_t bf16_round_double(double v)
{
    double a = fabs(v), q, r;
    int e;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    uint32_t u;
    float f;
    if (a == 0.0)
        return sign;
    frexp(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
    if (e - 1 < -126)
        e = -125;                   /* subnormal range: quantum 2^-133 */
    q = ldexp(1.0, e - 8);          /* 8 significant bits: ulp of a */
    r = nearbyint(a / q) * q;       /* exact scaling by a power of two; nearbyint rounds half to even */
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    f = (float)r;                   /* exact: r has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* One SwiGLU output, reading R13: bf16 of y = g * u * sigma(g), sigma(g) =
 * 1 / (1 + e^-g), rounded once to nearest, ties to even.  y is never exactly
 * a bf16 midpoint (for g != 0, sigma(g) is transcendental), so the rounding
 * direction is always defined; the value is computed in double, and when it
 * lies within 2^-45 (relative) of a midpoint m the side is decided again in
 * long double from quantities free of cancellation:
 *   g >= 0:  |y| = |gu| - |gu| t with t = 1 / (1 + e^g), so |y| > m exactly
 *            when |gu| - m (exact) > |gu| t;
 *   g <  0:  |y| = |gu| e^g / (1 + e^g), compared with m directly.
 * *ambiguous is set if even that cannot separate |y| from m. */
static uint16_t swiglu_bf16_one(uint16_t gb, uint16_t ub, int *ambiguous)
{
    double g = (double)bf16_to_f32(gb), u = (double)bf16_to_f32(ub);
    double gu = g * u;              /* exact: at most 16 significant bits */
    double a, q, lo, mid;
    int e, above;
    uint16_t sign, r;
    if (gu == 0.0)
        return bf16_round_double(gu);
    sign = signbit(gu) ? 0x8000 : 0x0000;
    a = fabs(gu) / (1.0 + exp(-g));
    frexp(a, &e);
    if (e - 1 < -126)
        e = -125;
    q = ldexp(1.0, e - 8);          /* bf16 quantum at a */
    lo = floor(a / q) * q;
    mid = lo + 0.5 * q;
    if (fabs(a - mid) > ldexp(a, -45))
        return bf16_round_double(sign ? -a : a);
    if (g >= 0.0) {
        long double d = (long double)fabs(gu) - (long double)mid;
        long double p = (long double)fabs(gu) / (1.0L + expl((long double)g));
        above = d > p;
        if (fabsl(d - p) <= ldexpl(p, -58) && p > 0.0L)
            *ambiguous = 1;
    } else {
        long double el = expl((long double)g);
        long double al = (long double)fabs(gu) * el / (1.0L + el);
        above = al > (long double)mid;
        if (fabsl(al - (long double)mid) <= ldexpl(al, -58))
            *ambiguous = 1;
    }
    r = bf16_round_double(above ? lo + q : lo);
    return (uint16_t)(sign | r);
}

/* SwiGLU output of cached bf16 inputs, reading R13: for m < M, f < F,
 * y[m][f] = bf16(g * u / (1 + exp(-g))) with g = gate[m*ldg + f] and
 * u = up[m*ldu + f], correctly rounded.  y is written as bf16 bit patterns at
 * y[m*ldy + f].  Returns the number of elements whose rounding direction could
 * not be decided (expected 0; see swiglu_bf16_one). */
int64_t orc_swiglu_bf16(const uint16_t *gate, int64_t ldg, const uint16_t *up, int64_t ldu,
                        int64_t M, int64_t F, uint16_t *y, int64_t ldy)
{
    int64_t m, f, undecided = 0;
    for (m = 0; m < M; ++m)
        for (f = 0; f < F; ++f) {
            int amb = 0;
            y[m * ldy + f] = swiglu_bf16_one(gate[m * ldg + f], up[m * ldu + f], &amb);
            undecided += amb;
        }
    return undecided;
}
