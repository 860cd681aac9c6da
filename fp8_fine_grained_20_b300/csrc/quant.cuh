// quant.cuh -- the three fine-grained FP8 quantizers (memory-bound kernels).
//
// Method (DeepSeek-V3 FP8 excerpt, sunipension.com post 314414, Figure 7(a)):
// activations are scaled per 1x128 tile, weights per 128x128 block, and the
// cached 1x128 activation tiles are converted to 128x1 tiles for the backward
// pass.  For each group: amax = max|x|, s = amax / 448, code = E4M3(x / s),
// with both divisions IEEE fp32 round-to-nearest-even (scaling rule of
// why-be.why-be.co.kr post 65900: largest magnitude onto the FP8 maximum).
//
// Exact division without paying for it on every element: with r = RN(1/s),
// q0 = RN(|x| * r) lies within 5 fp32 ulps of RN(|x| / s) (relative error of
// r and of the product, each <= 2^-24, plus the final rounding; one binade
// boundary at most doubles the count).  E4M3 rounding is monotonic in the
// fp32 bit pattern of a non-negative value, so if the codes of the bit
// patterns q0 - 8 and q0 + 8 agree, that is the code of RN(|x| / s); only when
// an E4M3 rounding boundary lies inside that window (about 16 in 2^20 values)
// is the exact IEEE quotient computed.  Groups whose scale is an fp32
// subnormal (1/s would overflow) always take the exact quotient.
#pragma once

#include "ptx.cuh"

namespace fp8fg {

constexpr float kE4M3Max = 448.0f;
constexpr float kFltMinNormal = 1.17549435082228750797e-38f;

struct GroupScale {
    float s;    // amax / 448
    float r;    // RN(1 / s)
    int mode;   // 0: all-zero group, 1: fast path valid, 2: exact quotient only
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
    GroupScale g;
    g.s = __fdiv_rn(amax, kE4M3Max);
    g.r = __frcp_rn(g.s);
    g.mode = (amax == 0.0f) ? 0 : (g.s >= kFltMinNormal ? 1 : 2);
    return g;
}

// E4M3 code (sign included) of the fp32 quotient x / s.
__device__ __forceinline__ uint32_t quant_code(float x, const GroupScale& g) {
    const uint32_t sign = (__float_as_uint(x) >> 24) & 0x80u;
    const float ax = fabsf(x);
    uint32_t c;
    if (g.mode == 1) {
        const uint32_t b = __float_as_uint(__fmul_rn(ax, g.r));
        const uint32_t lo = max(b, 8u) - 8u;
        const uint32_t c2 = cvt_e4m3x2(__uint_as_float(b + 8u), __uint_as_float(lo));
        c = c2 & 0xFFu;
        if (c != (c2 >> 8)) c = cvt_e4m3x2(0.0f, __fdiv_rn(ax, g.s)) & 0xFFu;
    } else if (g.mode == 2) {
        c = cvt_e4m3x2(0.0f, __fdiv_rn(ax, g.s)) & 0xFFu;
    } else {
        return 0u;
    }
    return c | sign;
}

// Four codes packed little-endian into one word.
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, const GroupScale& g) {
    return quant_code(a, g) | (quant_code(b, g) << 8) | (quant_code(c, g) << 16) | (quant_code(d, g) << 24);
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float absmax8(const uint4& v) {
    float a = fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x)));
    a = fmaxf(a, fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))));
    a = fmaxf(a, fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))));
    a = fmaxf(a, fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w))));
    return a;
}

__device__ __forceinline__ uint2 quant8_bf16(const uint4& v, const GroupScale& g) {
    uint2 o;
    o.x = quant4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y), g);
    o.y = quant4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w), g);
    return o;
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
// A half-warp owns one group: 16 lanes x 16 bytes = 128 bf16.  Each warp
// processes UNROLL group pairs per iteration, all loads issued before any
// reduction, over a grid-stride loop in row-major group order.
template <int UNROLL>
__global__ void __launch_bounds__(256) k_quant_act_1x128(const uint16_t* __restrict__ x, int M, int KB,
                                                         int64_t ldx, uint8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ s, int64_t ssm, int64_t sskb) {
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4;
    const int hl = lane & 15;
    const int64_t n_groups = static_cast<int64_t>(M) * KB;
    const int64_t n_pairs = (n_groups + 1) >> 1;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;

    // (m, kb) of this lane's current group and the per-step advance by 2*nw groups
    const int64_t step = 2 * nw;
    const int step_m = static_cast<int>(step / KB);
    const int step_kb = static_cast<int>(step % KB);
    const int64_t g0 = 2 * wid + half;
    int m = static_cast<int>(g0 / KB);
    int kb = static_cast<int>(g0 % KB);

    for (int64_t p0 = wid; p0 < n_pairs; p0 += nw * UNROLL) {
        uint4 v[UNROLL];
        int mu[UNROLL], kbu[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            mu[u] = m;
            kbu[u] = kb;
            v[u] = (m < M) ? ldg_nc_v4(x + static_cast<int64_t>(m) * ldx + kb * 128 + hl * 8)
                           : make_uint4(0u, 0u, 0u, 0u);
            m += step_m;
            kb += step_kb;
            if (kb >= KB) {
                kb -= KB;
                ++m;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float a = absmax8(v[u]);
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            if (mu[u] < M) {
                const GroupScale g = group_scale(a);
                stg_v2(q + static_cast<int64_t>(mu[u]) * ldq + kbu[u] * 128 + hl * 8, quant8_bf16(v[u], g));
                if (hl == 0) s[static_cast<int64_t>(mu[u]) * ssm + static_cast<int64_t>(kbu[u]) * sskb] = g.s;
            }
        }
    }
}

// ------------------------------------------------------ 128x128 weights ----
//
// One CTA (256 threads) per 128x128 block per iteration.  Thread (warp w,
// lane l) holds rows 8*rb .. 8*rb+7 (rb = 2w + l/16) and columns 8*(l%16) ..
// +7 of the block: eight 16-byte loads, each row segment read by 16
// consecutive lanes.  The block amax is reduced through shared memory; the
// K-major output layout is produced by an in-register 8x8 byte transpose.
__global__ void __launch_bounds__(256) k_quant_w_128x128(const uint16_t* __restrict__ w, int KB, int NB,
                                                         int64_t ldw, uint8_t* __restrict__ q, int64_t ldq,
                                                         int kmajor, float* __restrict__ s, int64_t sskb,
                                                         int64_t ssnb) {
    __shared__ float red[2][8];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nc = lane & 15;
    const int rb = warp * 2 + (lane >> 4);
    int par = 0;
    for (int blk = blockIdx.x; blk < KB * NB; blk += gridDim.x, par ^= 1) {
        const int kb = blk / NB;
        const int nb = blk - kb * NB;
        const int64_t row0 = static_cast<int64_t>(kb) * 128 + rb * 8;
        const uint16_t* src = w + row0 * ldw + nb * 128 + nc * 8;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = ldg_nc_v4(src + i * ldw);
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, absmax8(v[i]));
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
    }
}

// ------------------------------------------- 1x128 -> 128x1 requantizer ----
//
// One CTA per 128 (rows) x 128 (channels) block per iteration.  Thread layout
// as in the weight quantizer, on bytes: eight 8-byte loads of codes, the eight
// row scales of its rows; dequantization in fp32 (exact E4M3 -> f16 -> f32
// conversion, then one fp32 multiply); per-channel amax over the 128 rows via
// a lane shuffle and shared memory; quantization; 8x8 byte transpose; 8-byte
// stores into the transposed output.
__global__ void __launch_bounds__(256) k_requant_1x128_to_128x1(const uint8_t* __restrict__ q, int MB, int KB,
                                                                int64_t ldq, const float* __restrict__ s,
                                                                int64_t ssm, int64_t sskb,
                                                                uint8_t* __restrict__ qT, int64_t ldqT,
                                                                float* __restrict__ sT, int64_t sTk,
                                                                int64_t sTmb) {
    __shared__ __align__(16) float red[2][8][128];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nc = lane & 15;
    const int rb = warp * 2 + (lane >> 4);
    int par = 0;
    for (int blk = blockIdx.x; blk < MB * KB; blk += gridDim.x, par ^= 1) {
        const int mb = blk / KB;
        const int kb = blk - mb * KB;
        const int64_t row0 = static_cast<int64_t>(mb) * 128 + rb * 8;
        const int64_t col0 = static_cast<int64_t>(kb) * 128 + nc * 8;
        uint2 v[8];
        float sr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = ldg_nc_v2(q + (row0 + i) * ldq + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) sr[i] = __ldg(s + (row0 + i) * ssm + static_cast<int64_t>(kb) * sskb);
        float xh[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t h01 = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].x & 0xFFFFu));
            const uint32_t h23 = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].x >> 16));
            const uint32_t h45 = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].y & 0xFFFFu));
            const uint32_t h67 = cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v[i].y >> 16));
            xh[i][0] = __fmul_rn(f16_bits_to_f32(h01 & 0xFFFFu), sr[i]);
            xh[i][1] = __fmul_rn(f16_bits_to_f32(h01 >> 16), sr[i]);
            xh[i][2] = __fmul_rn(f16_bits_to_f32(h23 & 0xFFFFu), sr[i]);
            xh[i][3] = __fmul_rn(f16_bits_to_f32(h23 >> 16), sr[i]);
            xh[i][4] = __fmul_rn(f16_bits_to_f32(h45 & 0xFFFFu), sr[i]);
            xh[i][5] = __fmul_rn(f16_bits_to_f32(h45 >> 16), sr[i]);
            xh[i][6] = __fmul_rn(f16_bits_to_f32(h67 & 0xFFFFu), sr[i]);
            xh[i][7] = __fmul_rn(f16_bits_to_f32(h67 >> 16), sr[i]);
        }
        float ca[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(xh[i][j]));
            ca[j] = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 16));
        }
        if (lane < 16) {
            float4* dst = reinterpret_cast<float4*>(&red[par][warp][nc * 8]);
            dst[0] = make_float4(ca[0], ca[1], ca[2], ca[3]);
            dst[1] = make_float4(ca[4], ca[5], ca[6], ca[7]);
        }
        __syncthreads();
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) {
            const float4* src = reinterpret_cast<const float4*>(&red[par][ww][nc * 8]);
            const float4 p0 = src[0], p1 = src[1];
            ca[0] = fmaxf(ca[0], p0.x);
            ca[1] = fmaxf(ca[1], p0.y);
            ca[2] = fmaxf(ca[2], p0.z);
            ca[3] = fmaxf(ca[3], p0.w);
            ca[4] = fmaxf(ca[4], p1.x);
            ca[5] = fmaxf(ca[5], p1.y);
            ca[6] = fmaxf(ca[6], p1.z);
            ca[7] = fmaxf(ca[7], p1.w);
        }
        GroupScale g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = group_scale(ca[j]);
        uint2 rows[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            rows[i].x = quant_code(xh[i][0], g[0]) | (quant_code(xh[i][1], g[1]) << 8) |
                        (quant_code(xh[i][2], g[2]) << 16) | (quant_code(xh[i][3], g[3]) << 24);
            rows[i].y = quant_code(xh[i][4], g[4]) | (quant_code(xh[i][5], g[5]) << 8) |
                        (quant_code(xh[i][6], g[6]) << 16) | (quant_code(xh[i][7], g[7]) << 24);
        }
        uint2 cols[8];
        transpose8x8(rows, cols);
#pragma unroll
        for (int j = 0; j < 8; ++j) stg_v2(qT + (col0 + j) * ldqT + row0, cols[j]);
        if (rb == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) sT[(col0 + j) * sTk + static_cast<int64_t>(mb) * sTmb] = g[j].s;
        }
    }
}

}  // namespace fp8fg
