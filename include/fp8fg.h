/*
 * fp8fg.h -- C ABI of libfp8fg.so: fine-grained FP8 quantization and the
 * block-scaled FP8 GEMM on NVIDIA B300 (sm_103a).
 *
 * The method (DeepSeek-V3 FP8 training excerpts; pages named by address):
 *  - sunipension.com, board post 314414, Figure 7(a): activations are grouped
 *    and scaled per 1x128 tile (one token, 128 channels), weights per 128x128
 *    block (128 input x 128 output channels); cached activations are converted
 *    from 1x128 tiles to 128x1 tiles for the backward pass; Figure 6: the
 *    weight-gradient (Wgrad) GEMM runs in FP8.
 *  - why-be.why-be.co.kr, board post 55081, Figure 7(b): tensor-core partial
 *    sums are copied to FP32 registers on CUDA cores every K-interval and
 *    accumulated there in full FP32.
 *  - xn--jj0bz6z98ct0a29q.com, board post 362465: the per-group scales are
 *    applied during that FP32 promotion; MoE activations are dispatched in FP8.
 *  - why-be.why-be.co.kr, board post 65900: scaling maps the largest magnitude
 *    of a group onto the largest FP8 value.
 *
 * Numerics (identical on every entry point):
 *  - FP8 codes are OCP E4M3 ("e4m3fn", max 448) stored as uint8.
 *  - bf16 tensors are passed as their uint16 bit patterns.
 *  - For each group: amax = max |x| (fp32), s = amax / 448 (one IEEE fp32
 *    division, no flush to zero), code = E4M3 round-to-nearest-even, saturating,
 *    of the fp32 quotient x / s (one IEEE fp32 division); the sign of x is kept
 *    (a negative x that rounds to zero gives 0x80).  A group with amax == 0
 *    stores s = 0 and codes 0x00.  Inputs must be finite.
 *  - The GEMM promotion interval is the 128-wide K group: for every K-block kb
 *    the tensor-core partial sum of that block is multiplied by
 *    sA[m,kb] * sB[kb,n] and added to an FP32 accumulator; the output is
 *    rounded once to bf16 (nearest even).
 *
 * Conventions:
 *  - Every pointer is DEVICE memory owned by the caller; the library allocates
 *    nothing per call and keeps no pointer after the call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronises.  Calls on one stream run in order.
 *  - Argument checks run on the host before anything is launched; a non-OK
 *    status means nothing was launched.  FP8_ERR_CUDA reports a launch error.
 *  - Leading dimensions ("ld*") and strides are in ELEMENTS of the pointed-to
 *    type.  Device pointers must be 16-byte aligned, code/bf16 row strides must
 *    be multiples of 16 bytes.
 *  - Scale tensors have a logical shape and two explicit element strides, so
 *    the MN-major layout (stride 1 along the row/column index, which the GEMM
 *    reads fastest) and the row-major layout are both accepted.
 *  - Device-side waits are bounded.  A kernel that gives up sets a bit in a
 *    library-owned device status word and returns; read it with
 *    fp8_get_device_status().
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8_status {
    FP8_OK = 0,
    FP8_ERR_NULL = 1,            /* a required pointer is NULL */
    FP8_ERR_ALIGN = 2,           /* pointer not 16-byte aligned or stride not a multiple of 16 bytes */
    FP8_ERR_SHAPE = 3,           /* a size is negative, or not a multiple of 128 where required */
    FP8_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
    FP8_ERR_DEVICE_TIMEOUT = 5,  /* (device status) a bounded device wait gave up */
    FP8_ERR_ARG = 6,             /* an enum or stride argument is invalid */
    FP8_ERR_DEVICE = 7,          /* the current device is not sm_103 / lacks resources */
    FP8_ERR_DEVICE_GROUPS = 8,   /* (device status) group offsets were not valid */
    FP8_ERR_DEVICE_SCALES = 9,   /* (device status) a scale given to an _mx GEMM is not a power of two */
    FP8_ERR_DEVICE_BOUNDS = 10   /* (device status, bounds-checked debug build only) a device write fell
                                    outside its tensor or shared-memory tile and was skipped */
} fp8_status_t;

/* Layout of the codes written by fp8_quant_w_128x128. */
enum {
    FP8_KMAJOR_NK = 0,   /* q[n][k] (q + n*ldq + k): the K-major operand layout of the GEMMs */
    FP8_ROWMAJOR_KN = 1  /* q[k][n], same layout as the bf16 weight */
};

/* Granularity of the B-operand scales of fp8_gemm_blockscaled. */
enum {
    FP8_SB_BLOCK128x128 = 0, /* one scale per 128 (K) x 128 (N) block: logical sB[K/128][N/128] */
    FP8_SB_COL128x1 = 1      /* one scale per 128 (K) x 1 (N) column group: logical sB[K/128][N] */
};

/*
 * 1x128 activation quantization (Figure 7(a), activations).
 *   x     bf16 [M][K], row stride ldx (>= K)
 *   q     E4M3 codes [M][K], row stride ldq (>= K)
 *   s     fp32 scales, logical [M][K/128]; element (m, kb) at s[m*s_stride_m + kb*s_stride_kb].
 *         MN-major (the GEMM's preferred operand layout): s_stride_m = 1, s_stride_kb >= M.
 *         Row-major: s_stride_m = K/128, s_stride_kb = 1.
 * Requires K % 128 == 0; M may be any value >= 0 (M == 0 launches nothing).
 */
fp8_status_t fp8_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                 uint8_t* q, int64_t ldq,
                                 float* s, int64_t s_stride_m, int64_t s_stride_kb,
                                 void* stream);

/*
 * 128x128 weight quantization (Figure 7(a), weights).
 *   w        bf16 [K][N] (K input channels, N output channels), row stride ldw (>= N)
 *   q        E4M3 codes; q_layout FP8_KMAJOR_NK: q[n][k], row stride ldq (>= K);
 *            FP8_ROWMAJOR_KN: q[k][n], row stride ldq (>= N)
 *   s        fp32 scales, logical [K/128][N/128]; (kb, nb) at s[kb*s_stride_kb + nb*s_stride_nb]
 * Requires K % 128 == 0 and N % 128 == 0.
 */
fp8_status_t fp8_quant_w_128x128(const uint16_t* w, int64_t K, int64_t N, int64_t ldw,
                                 uint8_t* q, int64_t ldq, int q_layout,
                                 float* s, int64_t s_stride_kb, int64_t s_stride_nb,
                                 void* stream);

/*
 * 128x128 quantization of a batch of G weights in one launch (the experts of
 * an MoE layer; sunipension.com post 314414, Figure 7(a), applied per expert).
 * Weight g is w + g * w_batch_stride, its codes q + g * q_batch_stride and its
 * scales s + g * s_batch_stride; everything else is as in fp8_quant_w_128x128,
 * which is this call with G = 1.  For G > 1 the batch strides (elements) must
 * not make weights or code blocks overlap, and w_batch_stride * 2 and
 * q_batch_stride must be multiples of 16 bytes.
 */
fp8_status_t fp8_quant_w_128x128_batched(const uint16_t* w, int64_t G, int64_t K, int64_t N, int64_t ldw,
                                         int64_t w_batch_stride,
                                         uint8_t* q, int64_t ldq, int64_t q_batch_stride, int q_layout,
                                         float* s, int64_t s_stride_kb, int64_t s_stride_nb,
                                         int64_t s_batch_stride,
                                         void* stream);

/*
 * 1x128 -> 128x1 requantization for the backward pass (sunipension.com post
 * 314414: cached 1x128 activation tiles become 128x1 tiles).  Every value is
 * dequantized with one fp32 multiply, xhat = decode(q) * s, then every
 * channel k is quantized in groups of 128 consecutive rows (tokens) and the
 * result is written transposed.
 *   q    E4M3 codes [M][K], row stride ldq;  s  logical [M][K/128] at s[m*s_stride_m + kb*s_stride_kb]
 *   qT   E4M3 codes [K][M], row stride ldqT (>= M)
 *   sT   logical [K][M/128]; (k, mb) at sT[k*sT_stride_k + mb*sT_stride_mb]
 *        (for the Wgrad GEMM's operands, MN-major: sT_stride_k = 1, sT_stride_mb >= K)
 * Requires M % 128 == 0 and K % 128 == 0.
 */
fp8_status_t fp8_requant_1x128_to_128x1(const uint8_t* q, int64_t M, int64_t K, int64_t ldq,
                                        const float* s, int64_t s_stride_m, int64_t s_stride_kb,
                                        uint8_t* qT, int64_t ldqT,
                                        float* sT, int64_t sT_stride_k, int64_t sT_stride_mb,
                                        void* stream);

/*
 * SwiGLU recompute fused with 1x128 quantization (why-be.why-be.co.kr, board
 * post 65900: the inputs of the SwiGLU operator are cached and its output is
 * recomputed; sunipension.com post 314414, Figure 7(a): 1x128 activation
 * tiles).  For m < M, f < F:
 *   y[m][f] = bf16( silu(g) * u ),  silu(g) = g / (1 + e^-g),
 * with g = gate[m*ldg + f] and u = up[m*ldu + f] (bf16), evaluated in fp32 and
 * rounded once to bf16 (within one bf16 ulp of the correctly rounded value
 * while |g| <= 87); then y is 1x128-quantized exactly as fp8_quant_act_1x128
 * quantizes a bf16 tensor:
 *   q   E4M3 codes [M][F], row stride ldq (>= F, multiple of 16)
 *   s   fp32 scales, logical [M][F/128]; (m, fb) at s[m*s_stride_m + fb*s_stride_fb]
 *   y   optional bf16 [M][F] output of the rounded SwiGLU values (NULL: not written),
 *       row stride ldy
 * A fused gate/up projection output [M][2F] is passed as gate = base,
 * up = base + F, ldg = ldu = 2F.  Requires F % 128 == 0; M may be any value >= 0.
 */
fp8_status_t fp8_swiglu_quant_1x128(const uint16_t* gate, int64_t ldg, const uint16_t* up, int64_t ldu,
                                    int64_t M, int64_t F,
                                    uint8_t* q, int64_t ldq,
                                    float* s, int64_t s_stride_m, int64_t s_stride_fb,
                                    uint16_t* y, int64_t ldy,
                                    void* stream);

/*
 * Power-of-two scale variants of the three quantizers (why-be.why-be.co.kr,
 * board post 55081, and sunipension.com, board post 314414: the scaling
 * factors of the inputs of the Linear after attention, and of the gradients
 * before the MoE down-projection, are integral powers of 2).  Each group's
 * scale is the smallest power of two s = 2^e with amax / s <= 448, never below
 * 2^-127 (the smallest scale an 8-bit exponent can hold; fp32 bit pattern
 * 0x00400000); a zero group keeps s = 0 and codes 0x00.  The codes are the E4M3
 * round-to-nearest-even of x / s, which is exact (one multiply by 2^-e).  The
 * scales are written as fp32 values; these are the operands of
 * fp8_gemm_blockscaled_mx.  Arguments, layouts, requirements and status codes
 * are those of the call without the suffix.  The requantizer expects 1x128
 * inputs made with power-of-two scales (its dequantizing multiply is then
 * exact); it accepts any scales and applies the power-of-two rule to the
 * 128x1 groups.
 */
fp8_status_t fp8_quant_act_1x128_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                      uint8_t* q, int64_t ldq,
                                      float* s, int64_t s_stride_m, int64_t s_stride_kb,
                                      void* stream);
fp8_status_t fp8_quant_w_128x128_pow2(const uint16_t* w, int64_t K, int64_t N, int64_t ldw,
                                      uint8_t* q, int64_t ldq, int q_layout,
                                      float* s, int64_t s_stride_kb, int64_t s_stride_nb,
                                      void* stream);
fp8_status_t fp8_quant_w_128x128_batched_pow2(const uint16_t* w, int64_t G, int64_t K, int64_t N, int64_t ldw,
                                              int64_t w_batch_stride,
                                              uint8_t* q, int64_t ldq, int64_t q_batch_stride, int q_layout,
                                              float* s, int64_t s_stride_kb, int64_t s_stride_nb,
                                              int64_t s_batch_stride,
                                              void* stream);
fp8_status_t fp8_requant_1x128_to_128x1_pow2(const uint8_t* q, int64_t M, int64_t K, int64_t ldq,
                                             const float* s, int64_t s_stride_m, int64_t s_stride_kb,
                                             uint8_t* qT, int64_t ldqT,
                                             float* sT, int64_t sT_stride_k, int64_t sT_stride_mb,
                                             void* stream);

/*
 * Block-scaled FP8 GEMM with FP32 promotion every 128 K (Figure 7(b)):
 *   C[m][n] = bf16( sum_kb sA[m,kb] * sB(kb,n) * sum_{k in kb} A[m][k] * B[n][k] )
 * with the inner sums on tcgen05 tensor cores and the outer sum in FP32.
 *   A    E4M3 [M][K] (K contiguous), row stride lda
 *   sA   logical [M][K/128]; (m, kb) at sA[m*sa_stride_m + kb*sa_stride_kb]
 *   B    E4M3 [N][K] (K contiguous: the "K-major" / transposed weight), row stride ldb
 *   sB   sb_kind FP8_SB_BLOCK128x128 (forward, 128x128 weight blocks): logical
 *        [K/128][N/128], (kb, nb) at sB[kb*sb_stride_kb + nb*sb_stride_n];
 *        FP8_SB_COL128x1 (weight gradient, both operands 128x1-quantized along
 *        K): logical [K/128][N], (kb, n) at sB[kb*sb_stride_kb + n*sb_stride_n]
 *   C    bf16 [M][N], row stride ldc
 * Requires M % 128 == 0, N % 128 == 0, K % 128 == 0 (M, N or K == 0 launches nothing
 * when the output is empty; K == 0 with M*N > 0 is FP8_ERR_SHAPE).
 */
fp8_status_t fp8_gemm_blockscaled(const uint8_t* A, int64_t lda,
                                  const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                                  const uint8_t* B, int64_t ldb,
                                  const float* sB, int64_t sb_stride_kb, int64_t sb_stride_n,
                                  int sb_kind,
                                  uint16_t* C, int64_t ldc,
                                  int64_t M, int64_t N, int64_t K,
                                  void* stream);

/*
 * fp8_gemm_blockscaled with a quantizing epilogue: the GEMM's bf16 output
 * (rounded exactly as fp8_gemm_blockscaled rounds it) is 1x128-quantized in
 * the epilogue, as fp8_quant_act_1x128 would quantize it, so a GEMM whose
 * output feeds another FP8 GEMM writes codes and scales instead of bf16
 * (the pages cache and dispatch FP8 activations: xn--jj0bz6z98ct0a29q.com
 * post 362465; sunipension.com post 314414, Figure 7(a), 1x128 tiles).
 *   Cq   E4M3 codes [M][N], row stride ldcq (>= N, multiple of 16)
 *   sC   fp32 scales, logical [M][N/128]; (m, nb) at sC[m*sc_stride_m + nb*sc_stride_nb]
 * Every other argument, requirement and status is as in fp8_gemm_blockscaled.
 */
fp8_status_t fp8_gemm_blockscaled_q1x128(const uint8_t* A, int64_t lda,
                                         const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                                         const uint8_t* B, int64_t ldb,
                                         const float* sB, int64_t sb_stride_kb, int64_t sb_stride_n,
                                         int sb_kind,
                                         uint8_t* Cq, int64_t ldcq,
                                         float* sC, int64_t sc_stride_m, int64_t sc_stride_nb,
                                         int64_t M, int64_t N, int64_t K,
                                         void* stream);

/*
 * Grouped block-scaled FP8 GEMM for a variable-size MoE expert batch
 * (xn--jj0bz6z98ct0a29q.com post 362465: activations dispatched in FP8).
 * Expert g owns rows [off[g], off[g+1]) of A and C and multiplies them by B_g:
 *   C[m][n] = bf16( sum_kb sA[m,kb] * sB[g][kb][n/128] * sum_{k in kb} A[m][k] * B[g][n][k] )
 *   A               E4M3 [M_total][K], row stride lda;  sA as in fp8_gemm_blockscaled
 *   B               E4M3 [G][N][K], dense (expert stride N*K)
 *   sB              fp32 [G][K/128][N/128], dense
 *   d_group_offsets DEVICE int32 [G+1]; 0 <= off[0] <= ... <= off[G] <= M_total,
 *                   every entry a multiple of 128.  Read only on the device: the
 *                   host never synchronises.  Invalid offsets set
 *                   FP8_ERR_DEVICE_GROUPS in the device status and no tile is computed.
 *   C               bf16 [M_total][N], row stride ldc; rows outside every expert
 *                   are not written.
 * Requires M_total % 128 == 0, N % 128 == 0, K % 128 == 0, 1 <= G <= 1024.
 */
fp8_status_t fp8_grouped_gemm_blockscaled(const uint8_t* A, int64_t lda,
                                          const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                                          const uint8_t* B, const float* sB,
                                          const int32_t* d_group_offsets, int G,
                                          int64_t M_total, int64_t N, int64_t K,
                                          uint16_t* C, int64_t ldc,
                                          void* stream);

/*
 * Block-scaled FP8 GEMM with power-of-two scales applied by the tensor core
 * (why-be.why-be.co.kr post 55081 and sunipension.com post 314414: scaling
 * factors that are integral powers of 2).  Computes the same
 *   C[m][n] = bf16( sum_kb sA[m,kb] * sB(kb,n) * sum_{k in kb} A[m][k] * B[n][k] )
 * as fp8_gemm_blockscaled, with the same arguments, layouts, requirements and
 * status codes, but every scale must be a power of two in [2^-127, 2^127] or
 * zero (the fp32 output of the _pow2 quantizers): each 128-wide group's scale
 * becomes an 8-bit exponent (UE8M0) for its four 32-deep slices of K, and the
 * tensor core applies it inside the MMA (tcgen05.mma ... kind::mxf8f6f4
 * .block_scale), accumulating the whole K in FP32 tensor memory with no FP32
 * promotion on CUDA cores.  A scale that is not a power of two is used with
 * its exponent field alone and sets FP8_ERR_DEVICE_SCALES in the device status.
 */
fp8_status_t fp8_gemm_blockscaled_mx(const uint8_t* A, int64_t lda,
                                     const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                                     const uint8_t* B, int64_t ldb,
                                     const float* sB, int64_t sb_stride_kb, int64_t sb_stride_n,
                                     int sb_kind,
                                     uint16_t* C, int64_t ldc,
                                     int64_t M, int64_t N, int64_t K,
                                     void* stream);

/*
 * fp8_grouped_gemm_blockscaled with power-of-two scales applied by the tensor
 * core, as fp8_gemm_blockscaled_mx does; arguments, layouts, requirements and
 * status codes are those of fp8_grouped_gemm_blockscaled.
 */
fp8_status_t fp8_grouped_gemm_blockscaled_mx(const uint8_t* A, int64_t lda,
                                             const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                                             const uint8_t* B, const float* sB,
                                             const int32_t* d_group_offsets, int G,
                                             int64_t M_total, int64_t N, int64_t K,
                                             uint16_t* C, int64_t ldc,
                                             void* stream);

/*
 * Tensor-core accumulation probe (why-be.why-be.co.kr post 55081: the
 * previous generation's FP8 tensor cores keep about 14 bits when they
 * accumulate, hence the promotion every 128 K).  Computes
 *   D[m][n] = sum_{k < K} decode(A[m][k]) * decode(B[n][k])   (no scales)
 * for m < 128, n < 256 with tcgen05 FP8 MMAs accumulating the whole K in
 * tensor memory (no promotion), and writes D as fp32 [128][256] (row-major).
 *   A  E4M3 codes [128][K], dense (row stride K);  B  E4M3 codes [256][K], dense
 * Requires 128 <= K <= 2^24, K % 128 == 0.  One CTA; meant for measurements,
 * not speed.
 */
fp8_status_t fp8_mma_accumulation_probe(const uint8_t* A, const uint8_t* B, int64_t K, float* D, void* stream);

/*
 * Self-test of the library's bounded device waits (no counterpart on the
 * pages).  Launches one thread that waits on a shared-memory mbarrier which
 * nothing ever arrives on, with the same bounded wait the kernels use; after
 * timeout_ns (1 ns .. 1 s) it gives up, records FP8_ERR_DEVICE_TIMEOUT in the
 * device status word and returns, leaving the context usable.  Read the result
 * with fp8_get_device_status().  FP8_ERR_ARG for a timeout outside the range.
 */
fp8_status_t fp8_selftest_bounded_wait(uint64_t timeout_ns, void* stream);

/*
 * Self-test of the GEMM's failure path (no counterpart on the pages).  Runs
 * fp8_gemm_blockscaled (block scales) on dense operands -- A [M][K], sA
 * MN-major (sA[kb*M + m]), B [N][K], sB [K/128][N/128], C [M][N] -- with every
 * pipeline wait bounded by wait_ns (1 us .. 1 s) and the TMA producer
 * withholding every K-block after the first, so that a wait of the MMA issuer
 * runs out.  The kernel then records FP8_ERR_DEVICE_TIMEOUT, stops both CTAs
 * of every pair, lets the loads and MMAs it issued complete, frees its tensor
 * memory and returns; C is left undefined and the context stays usable.
 * Requires K >= 256 and the shapes of fp8_gemm_blockscaled.
 */
fp8_status_t fp8_selftest_gemm_timeout(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                       uint16_t* C, int64_t M, int64_t N, int64_t K, uint64_t wait_ns,
                                       void* stream);

/*
 * Device status word.  Waits for `stream`, copies the status word of the
 * current device into *out (FP8_OK or the first FP8_ERR_DEVICE_* recorded since
 * the last reset) and, if reset != 0, clears it.  Returns FP8_ERR_CUDA if the
 * copy fails.
 */
fp8_status_t fp8_get_device_status(void* stream, int32_t* out, int reset);

/* Static, human-readable name of a status code. */
const char* fp8_status_string(fp8_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fp8fg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */
