// swiglu.cuh -- SwiGLU recompute fused with 1x128 FP8 quantization
// (memory-bound), for sm_103a.
//
// Method: the inputs of the SwiGLU operator are cached and its output is
// recomputed when it is needed again (why-be.why-be.co.kr post 65900); the
// recomputed output is the activation of the next FP8 GEMM, quantized per
// 1x128 tile (sunipension.com post 314414, Figure 7(a)).  One pass reads the
// cached bf16 gate g and up projection u and writes the E4M3 codes and fp32
// scales of y = silu(g) * u = g * u / (1 + e^-g), rounded to bf16 first (the
// value an unfused SwiGLU would store), so the output never goes through HBM
// in bf16; the bf16 y can optionally be written as well.
//
// Arithmetic per pair of elements, in fp32 (packed FP32x2 where it exists):
// e = 2^(-g log2 e) (MUFU ex2, flushing subnormal results), sigma = 1 / (1 + e)
// (MUFU rcp), y = (g sigma) u, rounded to bf16 (nearest even).  For g below
// about -88.7, e overflows to infinity and sigma is 0; for g above about 87, e
// flushes to 0 and sigma is 1.  While |g| <= 87 (sigma stays a normal fp32
// number) the result is within one bf16 ulp of the correctly rounded SwiGLU
// value.  The bf16 values are then
// quantized exactly as k_quant_act_1x128 quantizes its input (amax, the IEEE
// scale, exact quotients), so the codes equal the 1x128 quantization of the
// bf16 y bit for bit.
//
// Layout of the work: as k_quant_act_1x128 -- four lanes own one 1x128 group
// (each loads four 16-byte chunks of g and four of u), a warp covers eight
// groups per slot, UNROLL slots per iteration, grid-stride over slots.
#pragma once

#include "quant.cuh"

namespace fp8fg {

struct SwigluArgs {
    const uint16_t* g;
    int64_t ldg;
    const uint16_t* u;
    int64_t ldu;
    uint8_t* q;
    int64_t ldq;
    float* s;
    int64_t ssm, ssfb;
    uint16_t* y;     // optional bf16 output (nullptr: not written)
    int64_t ldy;
    int M, FB;
};

__device__ __forceinline__ float ex2_ftz(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// silu(g) * u of a bf16x2 gate word and a bf16x2 up word -> bf16x2.
__device__ __forceinline__ uint32_t swiglu2(uint32_t gw, uint32_t uw) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    const float2 g = bf16x2_to_f32x2(gw);
    const float2 u = bf16x2_to_f32x2(uw);
    const float2 a = __fmul2_rn(g, make_float2(kNegLog2e, kNegLog2e));
    const float2 d = __fadd2_rn(make_float2(ex2_ftz(a.x), ex2_ftz(a.y)), make_float2(1.0f, 1.0f));
    const float2 y = __fmul2_rn(__fmul2_rn(g, make_float2(rcp_ftz(d.x), rcp_ftz(d.y))), u);
    uint32_t w;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(y.y), "f"(y.x));
    return w;
}

// Eight bf16 gate and eight bf16 up values (one 16-byte chunk each) -> the
// eight bf16 SwiGLU outputs, packed as four bf16x2 words.
__device__ __forceinline__ uint4 swiglu8(const uint4& gv, const uint4& uv) {
    return make_uint4(swiglu2(gv.x, uv.x), swiglu2(gv.y, uv.y), swiglu2(gv.z, uv.z), swiglu2(gv.w, uv.w));
}

template <int UNROLL>
__global__ void __launch_bounds__(256) k_swiglu_quant_1x128(const SwigluArgs a) {
    const int lane = threadIdx.x & 31;
    const int sub = lane & 3;
    const int64_t n_groups = static_cast<int64_t>(a.M) * a.FB;
    const int64_t n_slots = (n_groups + 7) >> 3;
    const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t step = 8 * nw;
    const int step_m = static_cast<int>(step / a.FB);
    const int step_fb = static_cast<int>(step % a.FB);
    const int64_t g0 = 8 * wid + (lane >> 2);
    int m = static_cast<int>(g0 / a.FB);
    int fb = static_cast<int>(g0 % a.FB);

    for (int64_t p0 = wid; p0 < n_slots; p0 += nw * UNROLL) {
        uint4 vg[UNROLL][4], vu[UNROLL][4];
        int mu[UNROLL], fbu[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            mu[u] = m;
            fbu[u] = fb;
            const int64_t col = static_cast<int64_t>(fb) * 128 + sub * 8;
            const uint16_t* gs = a.g + static_cast<int64_t>(m) * a.ldg + col;
            const uint16_t* us = a.u + static_cast<int64_t>(m) * a.ldu + col;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                vg[u][i] = (m < a.M) ? ldg_nc_v4(gs + 32 * i) : make_uint4(0u, 0u, 0u, 0u);
                vu[u][i] = (m < a.M) ? ldg_nc_v4(us + 32 * i) : make_uint4(0u, 0u, 0u, 0u);
            }
            m += step_m;
            fb += step_fb;
            if (fb >= a.FB) {
                fb -= a.FB;
                ++m;
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            uint4 yv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) yv[i] = swiglu8(vg[u][i], vu[u][i]);
            const uint32_t h = umax16x2(umax16x2(absmax_bf16x8(yv[0]), absmax_bf16x8(yv[1])),
                                        umax16x2(absmax_bf16x8(yv[2]), absmax_bf16x8(yv[3])));
            float am = hmax_bf16x2_to_f32(h);
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
            if (mu[u] < a.M) {
                const GroupScale gsc = group_scale(am);
                const int64_t col = static_cast<int64_t>(fbu[u]) * 128 + sub * 8;
                uint8_t* dst = a.q + static_cast<int64_t>(mu[u]) * a.ldq + col;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (FP8_IN_BOUNDS(col + 32 * i + 8 <= static_cast<int64_t>(a.FB) * 128))
                        stg_v2(dst + 32 * i, quant8_bf16(yv[i], gsc));
                if (sub == 0 && FP8_IN_BOUNDS(mu[u] < a.M && fbu[u] < a.FB))
                    a.s[static_cast<int64_t>(mu[u]) * a.ssm + static_cast<int64_t>(fbu[u]) * a.ssfb] = gsc.s;
                if (a.y != nullptr) {
                    uint16_t* yd = a.y + static_cast<int64_t>(mu[u]) * a.ldy + col;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (FP8_IN_BOUNDS(col + 32 * i + 8 <= static_cast<int64_t>(a.FB) * 128)) stg_v4(yd + 32 * i, yv[i]);
                }
            }
        }
    }
}

}  // namespace fp8fg
