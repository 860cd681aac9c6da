// quant.cuh -- the three fine-grained FP8 quantizers (memory-bound kernels).
//
// Method (DeepSeek-V3 FP8 excerpt, sunipension.com post 314414, Figure 7(a)):
// activations are scaled per 1x128 tile, weights per 128x128 block, and the
// cached 1x128 activation tiles are converted to 128x1 tiles for the backward
// pass.  For each group: amax = max|x|, s = amax / 448, code = E4M3(x / s),
// with both divisions IEEE fp32 round-to-nearest-even (scaling rule of
// why-be.why-be.co.kr post 65900: largest magnitude onto the FP8 maximum).
//
// The quotient x / s must be the correctly rounded fp32 value, because E4M3
// rounds it a second time: with bf16 inputs the exact ratio lands on an E4M3
// rounding boundary for about 0.5% of the elements (exact ties, and values one
// fp32 ulp from a tie because s itself is rounded), so an approximate quotient
// is not enough.  Per group the kernels compute s = RN(amax / 448) and
// r = RN(1 / s) with IEEE division and reciprocal; per element they use
// Markstein's correction (P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): if r
// is within half an ulp of 1/s and q is within one ulp of x/s, the remainder
// e = x - q s is exact in one FMA and RN(q + e r) is RN(x/s).  q0 = RN(x r) can
// be up to 1.5 ulps away, so two correction steps are applied (the first one
// makes the value faithful, the second one exact):
//     q0 = x r;  q1 = q0 + (x - q0 s) r;  q = q1 + (x - q1 s) r
// as packed FP32x2 multiplies/FMAs on pairs of elements, followed by one
// E4M3x2 conversion (round to nearest even, saturating).  The sign bit of
// each input is OR-ed into its code, so -0 and negative values that round to
// zero keep the sign.  Groups with amax == 0 give zero codes; groups whose
// scale is below 2^-92 use IEEE division per element.
#pragma once

#include "ptx.cuh"

namespace fp8fg {

constexpr float kE4M3Max = 448.0f;
// Smallest scale for the reciprocal path: every element whose E4M3 code can
// be nonzero (x / s >= 2^-11) is then >= 2^-103, so the correction remainders
// (granularity about x 2^-46) stay in the normal fp32 range and are exact.
constexpr float kMinRecipScale = 0x1p-92f;

struct GroupScale {
    float s;    // amax / 448 (IEEE division)
    float r;    // RN(1 / s)
    int mode;   // 0: all-zero group, 1: reciprocal path, 2: IEEE division per element (tiny s)
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
    GroupScale g;
    g.s = __fdiv_rn(amax, kE4M3Max);
    g.r = __frcp_rn(g.s);
    g.mode = (amax == 0.0f) ? 0 : (g.s >= kMinRecipScale ? 1 : 2);
    return g;
}

// RN(x / s) for a pair of values by Markstein's two-step correction; r2 =
// (RN(1/s0), RN(1/s1)), ns2 = (-s0, -s1).
__device__ __forceinline__ float2 div2_markstein(float2 x, float2 r2, float2 ns2) {
    const float2 q0 = __fmul2_rn(x, r2);
    const float2 e0 = __ffma2_rn(q0, ns2, x);
    const float2 q1 = __ffma2_rn(e0, r2, q0);
    const float2 e1 = __ffma2_rn(q1, ns2, x);
    return __ffma2_rn(e1, r2, q1);
}

// Magnitude-only E4M3 codes of a pair (bits 7:0 from x.x, 15:8 from x.y); the
// sign bits are applied by the caller.
__device__ __forceinline__ uint32_t e4m3_pair(float2 q) { return cvt_e4m3x2(q.y, q.x); }

// Elementwise max of two pairs of 16-bit unsigned values.
__device__ __forceinline__ uint32_t umax16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Magnitude max of eight bf16 values as an |bf16|x2 word: with the sign bits
// cleared, the integer order of finite bf16 patterns is the order of values.
__device__ __forceinline__ uint32_t absmax_bf16x8(const uint4& v) {
    const uint32_t m = 0x7FFF7FFFu;
    return umax16x2(umax16x2(v.x & m, v.y & m), umax16x2(v.z & m, v.w & m));
}

// fp32 value of the larger half of an |bf16|x2 word.
__device__ __forceinline__ float hmax_bf16x2_to_f32(uint32_t w) {
    const uint32_t hi = w >> 16, lo = w & 0xFFFFu;
    return __uint_as_float((hi > lo ? hi : lo) << 16);
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// E4M3 code (sign included) of RN(x / s) by IEEE division; mode as in GroupScale.
__device__ __forceinline__ uint32_t quant_div(float x, float s, int mode) {
    if (mode == 0) return 0u;
    const uint32_t c = cvt_e4m3x2(0.0f, __fdiv_rn(fabsf(x), s)) & 0xFFu;
    return c | ((__float_as_uint(x) >> 24) & 0x80u);
}

// Eight codes of eight bf16 values (one 16-byte chunk) of one group.
__device__ __forceinline__ uint2 quant8_bf16(const uint4& v, const GroupScale& g) {
    if (g.mode == 1) {
        const float2 r2 = make_float2(g.r, g.r);
        const float2 ns2 = make_float2(-g.s, -g.s);
        const uint32_t c0 = e4m3_pair(div2_markstein(bf16x2_to_f32x2(v.x), r2, ns2));
        const uint32_t c1 = e4m3_pair(div2_markstein(bf16x2_to_f32x2(v.y), r2, ns2));
        const uint32_t c2 = e4m3_pair(div2_markstein(bf16x2_to_f32x2(v.z), r2, ns2));
        const uint32_t c3 = e4m3_pair(div2_markstein(bf16x2_to_f32x2(v.w), r2, ns2));
        // sign bits (bit 15 of each bf16) into bit 7 of each code byte
        const uint32_t sx = __byte_perm(v.x, v.y, 0x7531) & 0x80808080u;
        const uint32_t sy = __byte_perm(v.z, v.w, 0x7531) & 0x80808080u;
        return make_uint2(__byte_perm(c0, c1, 0x5410) | sx, __byte_perm(c2, c3, 0x5410) | sy);
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = bf16x2_to_f32x2(w[k]);
        const uint32_t c = quant_div(f.x, g.s, g.mode) | (quant_div(f.y, g.s, g.mode) << 8);
        o[k >> 1] |= c << (16 * (k & 1));
    }
    return make_uint2(o[0], o[1]);
}

// Transpose an 8x8 byte matrix held as rows (r[i].x = bytes 0-3, r[i].y =
// bytes 4-7 of row i) into columns (c[j] = bytes of column j, rows 0-7).
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& c0,
                                             uint32_t& c1, uint32_t& c2, uint32_t& c3) {
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140);  // a0.b0 a1.b0 a0.b1 a1.b1
    const uint32_t t1 = __byte_perm(a0, a1, 0x7362);  // a0.b2 a1.b2 a0.b3 a1.b3
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140);
    const uint32_t t3 = __byte_perm(a2, a3, 0x7362);
    c0 = __byte_perm(t0, t2, 0x5410);
    c1 = __byte_perm(t0, t2, 0x7632);
    c2 = __byte_perm(t1, t3, 0x5410);
    c3 = __byte_perm(t1, t3, 0x7632);
}

__device__ __forceinline__ void transpose8x8(const uint2 (&r)[8], uint2 (&c)[8]) {
    uint32_t lo[8], hi[8];
    transpose4x4(r[0].x, r[1].x, r[2].x, r[3].x, lo[0], lo[1], lo[2], lo[3]);  // rows 0-3, cols 0-3
    transpose4x4(r[4].x, r[5].x, r[6].x, r[7].x, hi[0], hi[1], hi[2], hi[3]);  // rows 4-7, cols 0-3
    transpose4x4(r[0].y, r[1].y, r[2].y, r[3].y, lo[4], lo[5], lo[6], lo[7]);  // rows 0-3, cols 4-7
    transpose4x4(r[4].y, r[5].y, r[6].y, r[7].y, hi[4], hi[5], hi[6], hi[7]);  // rows 4-7, cols 4-7
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = make_uint2(lo[j], hi[j]);
}

// ------------------------------------------------- 1x128 activations ----
//
// Four lanes own one group (128 bf16 = 16 chunks of 16 bytes; lane l%4 loads
// chunks l%4, l%4+4, l%4+8, l%4+12), so a warp covers 8 consecutive groups
// per slot and each lane quantizes 32 values with one scale computation.
// UNROLL slots per iteration keep 4*UNROLL 16-byte loads in flight per lane;
// grid-stride over slots in row-major group order.
template <int UNROLL>
__global__ void __launch_bounds__(256) k_quant_act_1x128(const uint16_t* __restrict__ x, int M, int KB,
                                                         int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ s, int64_t ssm, int64_t sskb) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 3;                  // chunk phase inside the group
    const int64_t n_groups = static_cast<int64_t>(M) * KB;
    const int64_t n_slots = (n_groups + 7) >> 3;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;

    // (m, kb) of this lane's group in the current slot; advance by 8*nw groups per slot
    const int64_t step = 8 * nw;
    const int step_m = static_cast<int>(step / KB);
    const int step_kb = static_cast<int>(step % KB);
    const int64_t g0 = 8 * wid + (lane >> 2);
    int m = static_cast<int>(g0 / KB);
    int kb = static_cast<int>(g0 % KB);

    for (int64_t p0 = wid; p0 < n_slots; p0 += nw * UNROLL) {
        uint4 v[UNROLL][4];
        int mu[UNROLL], kbu[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            mu[u] = m;
            kbu[u] = kb;
            const uint16_t* src = x + static_cast<int64_t>(m) * ldx + kb * 128 + sub * 8;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[u][i] = (m < M) ? ldg_nc_v4(src + 32 * i) : make_uint4(0u, 0u, 0u, 0u);
            m += step_m;
            kb += step_kb;
            if (kb >= KB) {
                kb -= KB;
                ++m;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const uint32_t h = umax16x2(umax16x2(absmax_bf16x8(v[u][0]), absmax_bf16x8(v[u][1])),
                                        umax16x2(absmax_bf16x8(v[u][2]), absmax_bf16x8(v[u][3])));
            float a = hmax_bf16x2_to_f32(h);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            if (mu[u] < M) {
                const GroupScale g = group_scale(a);
                uint8_t* dst = q + static_cast<int64_t>(mu[u]) * ldq + kbu[u] * 128 + sub * 8;
#pragma unroll
                for (int i = 0; i < 4; ++i) stg_v2(dst + 32 * i, quant8_bf16(v[u][i], g));
                if (sub == 0) s[static_cast<int64_t>(mu[u]) * ssm + static_cast<int64_t>(kbu[u]) * sskb] = g.s;
            }
        }
    }
}

// ------------------------------------------------------ 128x128 weights ----
//
// One CTA (256 threads) per 128x128 block per iteration.  Thread (warp w,
// lane l) holds rows 8*rb .. 8*rb+7 (rb = 2w + l/16) and columns 8*(l%16) ..
// +7 of the block: eight 16-byte loads, each row segment read by 16
// consecutive lanes; the next block's loads are issued before the current
// block is processed.  The block amax is reduced through shared memory; the
// K-major output layout is produced by an in-register 8x8 byte transpose.
__global__ void __launch_bounds__(256, 2) k_quant_w_128x128(const uint16_t* __restrict__ w, int KB, int NB,
                                                            int64_t ldw, uint8_t* __restrict__ q, int64_t ldq,
                                                            int kmajor, float* __restrict__ s, int64_t sskb,
                                                            int64_t ssnb) {
    __shared__ float red[2][8];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nc = lane & 15;
    const int rb = warp * 2 + (lane >> 4);
    const int n_blocks = KB * NB;
    int blk = blockIdx.x;
    if (blk >= n_blocks) return;
    uint4 v[8];
    auto load = [&](int b, uint4 (&dst)[8]) {
        const int kb_ = b / NB;
        const int nb_ = b - kb_ * NB;
        const uint16_t* src = w + (static_cast<int64_t>(kb_) * 128 + rb * 8) * ldw + nb_ * 128 + nc * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = ldg_nc_v4(src + i * ldw);
    };
    load(blk, v);
    int par = 0;
    for (; blk < n_blocks; blk += gridDim.x, par ^= 1) {
        const int kb = blk / NB;
        const int nb = blk - kb * NB;
        const int64_t row0 = static_cast<int64_t>(kb) * 128 + rb * 8;
        uint4 vn[8];
        const int nxt = blk + gridDim.x;
        if (nxt < n_blocks) load(nxt, vn);
        uint32_t h = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) h = umax16x2(h, absmax_bf16x8(v[i]));
        float a = hmax_bf16x2_to_f32(h);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (lane == 0) red[par][warp] = a;
        __syncthreads();
        a = red[par][0];
#pragma unroll
        for (int i = 1; i < 8; ++i) a = fmaxf(a, red[par][i]);
        const GroupScale g = group_scale(a);
        uint2 rows[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rows[i] = quant8_bf16(v[i], g);
        if (!kmajor) {
#pragma unroll
            for (int i = 0; i < 8; ++i) stg_v2(q + (row0 + i) * ldq + nb * 128 + nc * 8, rows[i]);
        } else {
            uint2 cols[8];
            transpose8x8(rows, cols);
            const int64_t n0 = static_cast<int64_t>(nb) * 128 + nc * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) stg_v2(q + (n0 + j) * ldq + row0, cols[j]);
        }
        if (threadIdx.x == 0) s[static_cast<int64_t>(kb) * sskb + static_cast<int64_t>(nb) * ssnb] = g.s;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = vn[i];
    }
}

// ------------------------------------------- 1x128 -> 128x1 requantizer ----

// Eight E4M3 codes (bytes of v, in order) -> eight fp32 values decode(q) * scale,
// one fp32 multiply each (E4M3 -> f16 -> f32 is exact).
__device__ __forceinline__ void dequant8(const uint2 v, float scale, float2 (&xr)[4]) {
    const uint32_t h[4] = {cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v.x & 0xFFFFu)),
                           cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v.x >> 16)),
                           cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v.y & 0xFFFFu)),
                           cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v.y >> 16))};
    const float2 sc = make_float2(scale, scale);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        xr[k] = __fmul2_rn(make_float2(f16_bits_to_f32(h[k] & 0xFFFFu), f16_bits_to_f32(h[k] >> 16)), sc);
}

// One CTA per 128 (rows) x 128 (channels) block per iteration.  Thread layout
// as in the weight quantizer, on bytes: eight 8-byte loads of codes and the
// eight row scales of its rows (the next block's are loaded before the
// current block is processed).  Pass 1 dequantizes (one fp32 multiply) and
// reduces the per-channel amax over the 128 rows (lane shuffle + shared
// memory); one thread per channel derives the channel's scale and reciprocal;
// pass 2 dequantizes again and quantizes; an 8x8 byte transpose and 8-byte
// stores write the transposed output.  The sign of every dequantized value is
// the sign bit of its input code, so the input bytes supply the sign bits.
__global__ void __launch_bounds__(256, 2) k_requant_1x128_to_128x1(const uint8_t* __restrict__ q, int MB, int KB,
                                                                   int64_t ldq, const float* __restrict__ s,
                                                                   int64_t ssm, int64_t sskb,
                                                                   uint8_t* __restrict__ qT, int64_t ldqT,
                                                                   float* __restrict__ sT, int64_t sTk,
                                                                   int64_t sTmb) {
    __shared__ __align__(16) float red[2][8][128];
    __shared__ __align__(16) float c_s[2][128];
    __shared__ __align__(16) float c_r[2][128];
    __shared__ __align__(16) int c_mode[2][128];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nc = lane & 15;
    const int rb = warp * 2 + (lane >> 4);
    const int n_blocks = MB * KB;
    int blk = blockIdx.x;
    if (blk >= n_blocks) return;
    uint2 v[8];
    float sr[8];
    auto load = [&](int b, uint2 (&dv)[8], float (&ds)[8]) {
        const int mb_ = b / KB;
        const int kb_ = b - mb_ * KB;
        const int64_t r0 = static_cast<int64_t>(mb_) * 128 + rb * 8;
        const int64_t c0 = static_cast<int64_t>(kb_) * 128 + nc * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) dv[i] = ldg_nc_v2(q + (r0 + i) * ldq + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i) ds[i] = __ldg(s + (r0 + i) * ssm + static_cast<int64_t>(kb_) * sskb);
    };
    load(blk, v, sr);
    int par = 0;
    for (; blk < n_blocks; blk += gridDim.x, par ^= 1) {
        const int mb = blk / KB;
        const int kb = blk - mb * KB;
        const int64_t row0 = static_cast<int64_t>(mb) * 128 + rb * 8;
        const int64_t col0 = static_cast<int64_t>(kb) * 128 + nc * 8;
        uint2 vn[8];
        float srn[8];
        const int nxt = blk + gridDim.x;
        if (nxt < n_blocks) load(nxt, vn, srn);

        // pass 1: per-channel amax of the dequantized values
        float ca[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) ca[j] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float2 xr[4];
            dequant8(v[i], sr[i], xr);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ca[2 * k] = fmaxf(ca[2 * k], fabsf(xr[k].x));
                ca[2 * k + 1] = fmaxf(ca[2 * k + 1], fabsf(xr[k].y));
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) ca[j] = fmaxf(ca[j], __shfl_xor_sync(0xffffffffu, ca[j], 16));
        if (lane < 16) {
            float4* dst = reinterpret_cast<float4*>(&red[par][warp][nc * 8]);
            dst[0] = make_float4(ca[0], ca[1], ca[2], ca[3]);
            dst[1] = make_float4(ca[4], ca[5], ca[6], ca[7]);
        }
        __syncthreads();
        if (threadIdx.x < 128) {                 // one scale computation per channel
            float a = red[par][0][threadIdx.x];
#pragma unroll
            for (int ww = 1; ww < 8; ++ww) a = fmaxf(a, red[par][ww][threadIdx.x]);
            const GroupScale g = group_scale(a);
            c_s[par][threadIdx.x] = g.s;
            c_r[par][threadIdx.x] = g.r;
            c_mode[par][threadIdx.x] = g.mode;
        }
        __syncthreads();

        // pass 2: dequantize again and quantize with the channel scales
        float cs[8], cr[8];
        int all_recip;
        {
            const float4* ps = reinterpret_cast<const float4*>(&c_s[par][nc * 8]);
            const float4* pr = reinterpret_cast<const float4*>(&c_r[par][nc * 8]);
            const int4* pm = reinterpret_cast<const int4*>(&c_mode[par][nc * 8]);
            const float4 s0 = ps[0], s1 = ps[1], r0 = pr[0], r1 = pr[1];
            cs[0] = s0.x; cs[1] = s0.y; cs[2] = s0.z; cs[3] = s0.w;
            cs[4] = s1.x; cs[5] = s1.y; cs[6] = s1.z; cs[7] = s1.w;
            cr[0] = r0.x; cr[1] = r0.y; cr[2] = r0.z; cr[3] = r0.w;
            cr[4] = r1.x; cr[5] = r1.y; cr[6] = r1.z; cr[7] = r1.w;
            const int4 m0 = pm[0], m1 = pm[1];
            // all eight channels take the reciprocal path iff the AND of their modes is 1
            all_recip = (m0.x & m0.y & m0.z & m0.w & m1.x & m1.y & m1.z & m1.w) == 1;
        }
        uint2 rows[8];
        if (all_recip) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 xr[4];
                dequant8(v[i], sr[i], xr);
                uint32_t c[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    c[k] = e4m3_pair(div2_markstein(xr[k], make_float2(cr[2 * k], cr[2 * k + 1]),
                                                    make_float2(-cs[2 * k], -cs[2 * k + 1])));
                rows[i] = make_uint2((__byte_perm(c[0], c[1], 0x5410)) | (v[i].x & 0x80808080u),
                                     (__byte_perm(c[2], c[3], 0x5410)) | (v[i].y & 0x80808080u));
            }
        } else {
            int cm[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cm[j] = c_mode[par][nc * 8 + j];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 xr[4];
                dequant8(v[i], sr[i], xr);
                uint32_t cw[2] = {0u, 0u};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t c = quant_div(xr[k].x, cs[2 * k], cm[2 * k]) |
                                       (quant_div(xr[k].y, cs[2 * k + 1], cm[2 * k + 1]) << 8);
                    cw[k >> 1] |= c << (16 * (k & 1));
                }
                rows[i] = make_uint2(cw[0], cw[1]);
            }
        }
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j) stg_v2(qT + (col0 + j) * ldqT + row0, cols[j]);
        if (rb == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) sT[(col0 + j) * sTk + static_cast<int64_t>(mb) * sTmb] = cs[j];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = vn[i];
            sr[i] = srn[i];
        }
    }
}

}  // namespace fp8fg
