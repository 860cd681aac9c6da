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
// e = x - q s is exact in one FMA and RN(q + e r) is RN(x/s).  For an fp32
// dividend q0 = RN(x r) can be up to 1.5 ulps away, so two correction steps
// are applied (the first one makes the value faithful, the second one exact):
//     q0 = x r;  q1 = q0 + (x - q0 s) r;  q = q1 + (x - q1 s) r
// For a bf16 dividend one step is exact (div2_markstein_bf16 below says why).
// Both run as packed FP32x2 multiplies/FMAs on pairs of elements, followed by
// one E4M3x2 conversion (round to nearest even, saturating).  The sign bit of
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

// Power-of-two scale of a group: amax = m 2^E (m in [1, 2)) needs 448 2^e =
// 1.75 2^(e+8) >= amax, so e = E - 8 when m <= 1.75 and E - 7 otherwise;
// subnormal amax and anything below clamp to e = -127, whose scale 2^-127 is
// itself an fp32 subnormal (bit pattern 0x00400000).  r = 2^-e is exact.
__device__ __forceinline__ GroupScale group_scale_pow2(float amax) {
    GroupScale g;
    const uint32_t u = __float_as_uint(amax);
    const int eb = static_cast<int>(u >> 23);
    int e = eb - 135 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    if (eb == 0 || e < -127) e = -127;
    g.s = (e >= -126) ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23) : __uint_as_float(0x00400000u);
    g.r = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    g.mode = (amax == 0.0f) ? 0 : 1;
    if (amax == 0.0f) g.s = 0.0f;
    return g;
}

template <bool POW2>
__device__ __forceinline__ GroupScale group_scale_t(float amax) {
    return POW2 ? group_scale_pow2(amax) : group_scale(amax);
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

// RN(x / s) for a pair of bf16 dividends (8 significant bits): one correction
// step suffices, q0 = x r;  q = q0 + (x - q0 s) r.  With bf16 x and s = RN(amax
// / 448) for bf16 amax, the quotient depends only on the two significands and
// the exponent gap (every step scales exactly with a power of two while the
// scale is at least 2^-92), and the parity tests compare this quotient's
// codes with IEEE division over every bf16 significand pair and every gap at
// which a code can be nonzero, so the single step is exact for every input
// these quantizers accept.  fp32 dividends (the requantizer's) take the two
// steps above.
__device__ __forceinline__ float2 div2_markstein_bf16(float2 x, float2 r2, float2 ns2) {
    const float2 q0 = __fmul2_rn(x, r2);
    const float2 e0 = __ffma2_rn(q0, ns2, x);
    return __ffma2_rn(e0, r2, q0);
}

// RN(x / s) of a pair: Markstein's correction, or one multiply by r = 1/s
// when s is a power of two (then x r is the exact quotient, rounded once).
template <bool POW2>
__device__ __forceinline__ float2 div2_t(float2 x, float2 r2, float2 ns2) {
    if (POW2) return __fmul2_rn(x, r2);
    return div2_markstein(x, r2, ns2);
}

// RN(x / s) of a pair given NEGATED dividends nx = -x, nr2 = (-RN(1/s), ..)
// and s2 = (s, s): the same two correction steps as div2_markstein, written
// as e = q s + nx, q <- e (-r) + q.  Value for value this is div2_markstein;
// in addition the sign of a zero dividend survives (x = -0 gives -0, not +0),
// so no sign bits need to be restored after the E4M3 conversion.  With a
// power-of-two s the quotient is the single exact product nx (-r).
template <bool POW2>
__device__ __forceinline__ float2 div2_neg_t(float2 nx, float2 nr2, float2 s2) {
    float2 q = __fmul2_rn(nx, nr2);
    if constexpr (!POW2) {
#pragma unroll
        for (int i = 0; i < 2; ++i) q = __ffma2_rn(__ffma2_rn(q, s2, nx), nr2, q);
    }
    return q;
}

template <bool POW2>
__device__ __forceinline__ float2 div2_bf16_t(float2 x, float2 r2, float2 ns2) {
    if (POW2) return __fmul2_rn(x, r2);
    return div2_markstein_bf16(x, r2, ns2);
}

// Eight codes of eight bf16 values (one 16-byte chunk) of one group.
template <bool POW2 = false>
__device__ __forceinline__ uint2 quant8_bf16(const uint4& v, const GroupScale& g) {
    if (g.mode == 1) {
        const float2 r2 = make_float2(g.r, g.r);
        const float2 ns2 = make_float2(-g.s, -g.s);
        const uint32_t c0 = e4m3_pair(div2_bf16_t<POW2>(bf16x2_to_f32x2(v.x), r2, ns2));
        const uint32_t c1 = e4m3_pair(div2_bf16_t<POW2>(bf16x2_to_f32x2(v.y), r2, ns2));
        const uint32_t c2 = e4m3_pair(div2_bf16_t<POW2>(bf16x2_to_f32x2(v.z), r2, ns2));
        const uint32_t c3 = e4m3_pair(div2_bf16_t<POW2>(bf16x2_to_f32x2(v.w), r2, ns2));
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

// Transpose a 4x4 byte matrix held as rows a0..a3 (byte j of a_i = element
// (i, j)) into columns c0..c3 (byte i of c_j = element (i, j)).
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

// 8x8 byte matrix: rows r[i] (.x = bytes 0-3, .y = bytes 4-7 of row i) ->
// columns c[j] (.x = rows 0-3, .y = rows 4-7 of column j).
__device__ __forceinline__ void transpose8x8(const uint2 (&r)[8], uint2 (&c)[8]) {
    uint32_t lo[8], hi[8];
    transpose4x4(r[0].x, r[1].x, r[2].x, r[3].x, lo[0], lo[1], lo[2], lo[3]);
    transpose4x4(r[4].x, r[5].x, r[6].x, r[7].x, hi[0], hi[1], hi[2], hi[3]);
    transpose4x4(r[0].y, r[1].y, r[2].y, r[3].y, lo[4], lo[5], lo[6], lo[7]);
    transpose4x4(r[4].y, r[5].y, r[6].y, r[7].y, hi[4], hi[5], hi[6], hi[7]);
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = make_uint2(lo[j], hi[j]);
}

// Output staging for the transposed (128 rows x 128 bytes) tiles: row i
// starts at i*128 + 16*(i >> SHIFT), a shift that grows by one 16-byte bank
// group every 2^SHIFT rows, so the writers of one warp (same 16-byte column,
// rows 2^SHIFT apart) hit different bank groups, and rows never overlap.
template <int SHIFT>
__device__ __forceinline__ uint32_t stage_row(int i) {
    return static_cast<uint32_t>(i * 128 + 16 * (i >> SHIFT));
}
template <int SHIFT>
constexpr uint32_t stage_bytes() {
    return 127 * 128 + 16 * (127 >> SHIFT) + 128;
}

__device__ __forceinline__ void sts_v2(void* p, uint2 v) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(smem_addr(p)), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void sts_v4(void* p, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(p)), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ------------------------------------------------- 1x128 activations ----
//
// Four lanes own one group (128 bf16 = 16 chunks of 16 bytes; lane l%4 loads
// chunks l%4, l%4+4, l%4+8, l%4+12), so a warp covers 8 consecutive groups
// per slot and each lane quantizes 32 values with one scale computation.
// UNROLL slots per iteration keep 4*UNROLL 16-byte loads in flight per lane;
// grid-stride over slots in row-major group order.
template <int UNROLL, bool POW2 = false>
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
                const GroupScale g = group_scale_t<POW2>(a);
                uint8_t* dst = q + static_cast<int64_t>(mu[u]) * ldq + kbu[u] * 128 + sub * 8;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (FP8_IN_BOUNDS(kbu[u] * 128 + sub * 8 + 32 * i + 8 <= KB * 128))
                        stg_v2(dst + 32 * i, quant8_bf16<POW2>(v[u][i], g));
                if (sub == 0 && FP8_IN_BOUNDS(mu[u] < M && kbu[u] < KB))
                    s[static_cast<int64_t>(mu[u]) * ssm + static_cast<int64_t>(kbu[u]) * sskb] = g.s;
            }
        }
    }
}

// ------------------------------------------------------ 128x128 weights ----
//
// Persistent CTAs (two per SM), each owning every gridDim.x-th 128x128 block
// of a batch of weights (expert g, K-block kb, N-block nb).  TMA brings the
// 32 KB bf16 blocks into a WQ_STAGES-deep shared-memory ring, so that many
// blocks per CTA are in flight while one is processed.  A thread owns an 8x8
// sub-block (rows k = 8rb.., columns n = 8nc..): eight 16-byte shared loads
// (a warp reads two full 256-byte rows per load).  The block amax is reduced
// through shared memory; as soon as every thread holds its sub-block the
// stage is refilled.  Row-major output q[g][k][n]: 8-byte stores, 16 lanes per
// 128-byte output row.  K-major output q[g][n][k]: an in-register 8x8 byte
// transpose, then the 128 x 128-byte tile is staged in shared memory (rows
// skewed by a bank group every 8 rows, so a warp's writes do not conflict)
// and copied out with 16-byte stores, 8 lanes per 128-byte output row.
constexpr int WQ_STAGES = 3;
constexpr int WQ_THREADS = 256;
constexpr uint32_t WQ_TILE_BYTES = 128 * 128 * 2;
constexpr uint32_t WQ_STAGE_OUT = 16640;   // >= stage_bytes<3>(), multiple of 128
static_assert(WQ_STAGE_OUT >= stage_bytes<3>() && WQ_STAGE_OUT % 128 == 0, "weight staging tile");
constexpr size_t WQ_SMEM = 128 + WQ_STAGES * WQ_TILE_BYTES + WQ_STAGE_OUT + WQ_STAGES * 8 + 8 * 4;

struct QuantWArgs {
    uint8_t* q;
    int64_t ldq, q_gstride;   // row stride and expert stride of the codes (elements)
    float* s;
    int64_t sskb, ssnb, s_gstride;
    int G, KB, NB;
    int kmajor;
};

__device__ __forceinline__ uint4 lds_v4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_addr(p)));
    return v;
}

__device__ __forceinline__ uint32_t lds_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)));
    return v;
}

template <bool POW2 = false>
__global__ void __launch_bounds__(WQ_THREADS, 2) k_quant_w_128x128(const __grid_constant__ CUtensorMap tmW,
                                                                   const QuantWArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint8_t* tiles = base;
    uint8_t* out = base + WQ_STAGES * WQ_TILE_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(out + WQ_STAGE_OUT);
    float* red = reinterpret_cast<float*>(full + WQ_STAGES);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int rb = 2 * warp + (lane >> 4);    // rows 8 rb .. 8 rb + 7 of the block
    const int nc = lane & 15;                 // columns 8 nc .. 8 nc + 7
    const int per_g = a.KB * a.NB;
    const int total = a.G * per_g;

    auto issue = [&](int stage, int blk) {
        const int g = blk / per_g;
        const int r = blk - g * per_g;
        const int kb = r / a.NB;
        const int nb = r - kb * a.NB;
        mbar_arrive_expect_tx(&full[stage], WQ_TILE_BYTES);
        tma_load_3d(tiles + stage * WQ_TILE_BYTES, &tmW, &full[stage], nb * 128, kb * 128, g);
    };
    if (tid == 0) {
        for (int i = 0; i < WQ_STAGES; ++i) mbar_init(&full[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        for (int i = 0; i < WQ_STAGES; ++i) {
            const int blk = blockIdx.x + i * gridDim.x;
            if (blk < total) issue(i, blk);
        }
    }
    __syncthreads();

    bool ok = true;
    for (int i = 0;; ++i) {
        const int blk = blockIdx.x + i * gridDim.x;
        if (blk >= total) break;
        const int stage = i % WQ_STAGES;
        if (!__syncthreads_and(mbar_wait(&full[stage], (i / WQ_STAGES) & 1u, nullptr))) {
            if (tid == 0) record_status(kStatusTimeout);
            ok = false;
            break;
        }
        const int g = blk / per_g;
        const int r = blk - g * per_g;
        const int kb = r / a.NB;
        const int nb = r - kb * a.NB;
        const uint8_t* tile = tiles + stage * WQ_TILE_BYTES;   // bf16 [128 k][128 n], 256-byte rows

        uint4 v[8];
        uint32_t h = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = lds_v4(tile + (8 * rb + j) * 256 + nc * 16);
            h = umax16x2(h, absmax_bf16x8(v[j]));
        }
        float am = hmax_bf16x2_to_f32(h);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (lane == 0) red[warp] = am;
        __syncthreads();   // A: red[] complete; every thread holds its sub-block, the stage is free
        if (tid == 0) {
            const int nxt = blk + WQ_STAGES * gridDim.x;
            if (nxt < total) issue(stage, nxt);
        }
        am = red[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) am = fmaxf(am, red[k]);
        const GroupScale gs = group_scale_t<POW2>(am);
        if (tid == 0 && FP8_IN_BOUNDS(g < a.G && kb < a.KB && nb < a.NB))
            a.s[static_cast<int64_t>(g) * a.s_gstride + static_cast<int64_t>(kb) * a.sskb +
                static_cast<int64_t>(nb) * a.ssnb] = gs.s;

        uint2 rows[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) rows[j] = quant8_bf16<POW2>(v[j], gs);
        uint8_t* qg = a.q + static_cast<int64_t>(g) * a.q_gstride;
        if (!a.kmajor) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (FP8_IN_BOUNDS(kb * 128 + 8 * rb + j < a.KB * 128 && nb * 128 + 8 * nc + 8 <= a.NB * 128))
                    stg_v2(qg + static_cast<int64_t>(kb * 128 + 8 * rb + j) * a.ldq + nb * 128 + 8 * nc, rows[j]);
            __syncthreads();   // B: red[] may be rewritten by the next block
        } else {
            uint2 cols[8];
            transpose8x8(rows, cols);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (FP8_IN_BOUNDS(stage_row<3>(8 * nc + j) + 8 * rb + 8 <= WQ_STAGE_OUT))
                    sts_v2(out + stage_row<3>(8 * nc + j) + 8 * rb, cols[j]);
            __syncthreads();   // B: the staged tile is complete
            uint8_t* dst = qg + static_cast<int64_t>(nb * 128) * a.ldq + kb * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int id = tid + WQ_THREADS * u;    // 128 rows x 8 chunks of 16 bytes
                const int row = id >> 3, ch = id & 7;
                if (FP8_IN_BOUNDS(nb * 128 + row < a.NB * 128 && kb * 128 + 16 * ch + 16 <= a.KB * 128))
                    stg_v4(dst + static_cast<int64_t>(row) * a.ldq + 16 * ch, lds_v4(out + stage_row<3>(row) + 16 * ch));
            }
        }
    }
    // after an abort, let the loads still in flight land before the CTA may exit
    if (!ok && tid == 0) spin_ns(100000);
}

// ------------------------------------------- 1x128 -> 128x1 requantizer ----
//
// Persistent CTAs (RQ_CTAS_PER_SM per SM) of RQ_WARPS warps over 128 (tokens)
// x 128 (channels) blocks.  Warp 0 also feeds an RQ_STAGES-deep ring: TMA
// brings each 16 KB code block (128-byte swizzle) and cp.async the block's 128
// row scales (any strides, each stored twice so that one 16-byte shared load
// gives a row pair's scales as two FP32x2 operands), both completing on the
// stage's full barrier; when warp 0 starts block i it refills the stage of
// block i-1, once every warp has arrived on that stage's empty barrier.  Warp
// w owns channels 16w..16w+15 (one 16-byte column of the block), so no data
// crosses warps and the loop has no block-wide barrier.
//   Lane (g, c) = (lane / 4, lane % 4) owns channels 16w+4c..16w+4c+3 of the
// 16 rows 16j+2g+b (j < 8, b < 2): one 4-byte shared load per row.  The four
// codes of a row are negated (sign bits flipped, exact), widened to fp32 and
// multiplied by the row scale as two FP32x2 pairs (channels 4c, 4c+1 and
// 4c+2, 4c+3), which is -xhat.  Pass 1 takes each channel's amax over the
// lane's rows (three-operand |max|), then over the eight row groups by
// shuffles; lane (g, c) computes the scale of channel 4c + g % 4, and every
// lane receives its four channels' scales by shuffles.
//   Pass 2 decodes the same rows again (the same exact operations, so the same
// -xhat).  Holding all 64 values across the passes instead takes 120 registers
// against 60, i.e. two CTAs per SM instead of four; measured on B300 the two
// forms run equally fast on [8192, 7168] and this one 2% faster on [8192,
// 18432]: the time is set by the ALU and FMA pipes (the FP32x2 division chain
// holds the FMA pipe two cycles per instruction), not by latency or the extra
// decode.  Pass 2 then divides each pair by its two channels' scales (the
// division written on negated dividends keeps the sign of a zero value, so
// every code comes out of the E4M3 conversion with its sign already right) and
// converts the two rows 16j+2g, 16j+2g+1 of one channel into one 2-byte pair:
// adjacent bytes of a transposed output row.  The warp then releases the
// stage.  The pairs go to the warp's staging tile ([16 channels][128 tokens])
// whose 16-byte chunks are XOR-swizzled by channel / 4, so the four channel
// rows written by one store land in distinct banks, and the warp copies its 16
// output rows out with 16-byte stores, eight lanes per 128-byte row.
constexpr int RQ_STAGES = 2;
constexpr int RQ_CTAS_PER_SM = 4;
constexpr int RQ_WARPS = 8;                       // 16 channels each
constexpr int RQ_THREADS = 32 * RQ_WARPS;
constexpr uint32_t RQ_TILE_BYTES = 128 * 128;
constexpr uint32_t RQ_WSTAGE = 16 * 128;          // one warp's staged output rows
constexpr size_t RQ_SMEM = 1024 + RQ_STAGES * RQ_TILE_BYTES + RQ_WARPS * RQ_WSTAGE + RQ_STAGES * 256 * 4 +
                           2 * RQ_STAGES * 8;

struct RequantArgs {
    const float* s;
    int64_t ssm, sskb;
    uint8_t* qT;
    int64_t ldqT;
    float* sT;
    int64_t sTk, sTmb;
    int MB, KB;
};

// 2-byte shared store at a shared::cta address.
__device__ __forceinline__ void sts_u16_at(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(static_cast<uint16_t>(v)) : "memory");
}

// max(|a|, |b|, |c|) in one instruction (three-operand max with .abs).
__device__ __forceinline__ float fmax3_abs(float a, float b, float c) {
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Low and high fp16 halves of an f16x2 word as an fp32 pair.
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    return make_float2(f16_bits_to_f32(h & 0xFFFFu), f16_bits_to_f32(h >> 16));
}

// -xhat of one row's four codes (a 4-byte word) with row scale pair sb:
// channels (4c, 4c+1) in x01, (4c+2, 4c+3) in x23.
__device__ __forceinline__ void rq_decode4(uint32_t v, float2 sb, float2& x01, float2& x23) {
    v ^= 0x80808080u;
    x01 = __fmul2_rn(f16x2_to_f32x2(cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v & 0xFFFFu))), sb);
    x23 = __fmul2_rn(f16x2_to_f32x2(cvt_e4m3x2_to_f16x2(static_cast<uint16_t>(v >> 16))), sb);
}

template <bool POW2 = false>
__global__ void __launch_bounds__(RQ_THREADS, RQ_CTAS_PER_SM)
    k_requant_1x128_to_128x1(const __grid_constant__ CUtensorMap tmQ, const RequantArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* tiles = base;                                                  // [stage][128 m][128 k], swizzled
    uint8_t* stg = tiles + RQ_STAGES * RQ_TILE_BYTES;                       // [warp][16 k][128 m]
    float* sc = reinterpret_cast<float*>(stg + RQ_WARPS * RQ_WSTAGE);       // [stage][128 rows][2] row scales
    uint64_t* full = reinterpret_cast<uint64_t*>(sc + RQ_STAGES * 256);
    uint64_t* empty = full + RQ_STAGES;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total = a.MB * a.KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < RQ_STAGES; ++i) {
            mbar_init(&full[i], 33);   // expect-tx arrival + 32 cp.async arrivals
            mbar_init(&empty[i], RQ_WARPS);
        }
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
    }
    __syncthreads();

    // TMA of the codes (lane 0) and cp.async of the row scales (4 rows per
    // lane, each written twice) of block blk into a stage, both completing on
    // full[stage]: one expect-tx arrival + 32 cp.async arrivals.  Called by
    // warp 0 only.
    auto issue = [&](int stage, int blk) {
        const int mb = blk / a.KB;
        const int kb = blk - mb * a.KB;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[stage], RQ_TILE_BYTES);
            tma_load_2d(tiles + stage * RQ_TILE_BYTES, &tmQ, &full[stage], kb * 128, mb * 128);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = lane + 32 * j;
            const float* src = a.s + static_cast<int64_t>(mb * 128 + r) * a.ssm + static_cast<int64_t>(kb) * a.sskb;
            cp_async_4(sc + stage * 256 + 2 * r, src);
            cp_async_4(sc + stage * 256 + 2 * r + 1, src);
        }
        cp_async_arrive_noinc(&full[stage]);
    };
    if (warp == 0) {
        for (int i = 0; i < RQ_STAGES; ++i) {
            const int blk = blockIdx.x + i * gridDim.x;
            if (blk < total) issue(i, blk);
        }
    }

    const int w = warp;
    const int g = lane >> 2;
    const int c = lane & 3;
    // byte offset in a code tile of row 2g+b, channels 16w+4c..+3: the 16-byte
    // chunk w of row r sits at chunk w ^ (r % 8) (128-byte swizzle), and rows
    // 16j + 2g + b share that chunk for every j
    uint32_t roff[2];
#pragma unroll
    for (int b = 0; b < 2; ++b)
        roff[b] = static_cast<uint32_t>((2 * g + b) * 128 + ((w ^ ((2 * g + b) & 7)) << 4) + 4 * c);
    uint8_t* wst = stg + w * RQ_WSTAGE;
    // staging address of token pair 2g of channel row 4c (chunk 0): chunk j of
    // channel row r sits at chunk j ^ (r / 4); the row base is 2048-aligned, so
    // (ob ^ (j << 4)) + 128 ch addresses token pair 16j + 2g of channel 4c + ch
    const uint32_t ob = smem_addr(wst) + static_cast<uint32_t>(c * 512 + (c << 4) + 2 * g);
    // block blockIdx.x + i * gridDim.x is (mb, kb), advanced without a division
    const int step_mb = static_cast<int>(gridDim.x) / a.KB;
    const int step_kb = static_cast<int>(gridDim.x) - step_mb * a.KB;
    int mb = static_cast<int>(blockIdx.x) / a.KB;
    int kb = static_cast<int>(blockIdx.x) - mb * a.KB;
    bool ok = true;
    for (int i = 0;; ++i) {
        const int blk = blockIdx.x + i * gridDim.x;
        if (blk >= total) break;
        const int stage = i % RQ_STAGES;
        if (warp == 0 && i > 0) {
            // refill the stage of block i-1 with block i-1+RQ_STAGES
            const int64_t nxt = static_cast<int64_t>(blk) + static_cast<int64_t>(RQ_STAGES - 1) * gridDim.x;
            const int ps = (i - 1) % RQ_STAGES;
            if (nxt < total) {
                if (!__all_sync(0xffffffffu, mbar_wait(&empty[ps], ((i - 1) / RQ_STAGES) & 1u, nullptr))) {
                    ok = false;
                    break;
                }
                issue(ps, static_cast<int>(nxt));
            }
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (i / RQ_STAGES) & 1u, nullptr))) {
            ok = false;
            break;
        }
        const uint8_t* tile = tiles + stage * RQ_TILE_BYTES;
        const float* srow = sc + stage * 256;

        // pass 1: amax of -xhat over rows 16j+2g+b, channels 4c..4c+3
        float am[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // (s_r, s_r, s_r+1, s_r+1) for r = 16j + 2g
            const uint4 s4 = lds_v4(srow + 2 * (16 * j + 2 * g));
            float2 x[2][2];
#pragma unroll
            for (int b = 0; b < 2; ++b)
                rq_decode4(lds_u32(tile + roff[b] + 2048 * j),
                           b ? make_float2(__uint_as_float(s4.z), __uint_as_float(s4.w))
                             : make_float2(__uint_as_float(s4.x), __uint_as_float(s4.y)),
                           x[b][0], x[b][1]);
            am[0] = fmax3_abs(am[0], x[0][0].x, x[1][0].x);
            am[1] = fmax3_abs(am[1], x[0][0].y, x[1][0].y);
            am[2] = fmax3_abs(am[2], x[0][1].x, x[1][1].x);
            am[3] = fmax3_abs(am[3], x[0][1].y, x[1][1].y);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            am[k] = fmaxf(am[k], __shfl_xor_sync(0xffffffffu, am[k], 4));
            am[k] = fmaxf(am[k], __shfl_xor_sync(0xffffffffu, am[k], 8));
            am[k] = fmaxf(am[k], __shfl_xor_sync(0xffffffffu, am[k], 16));
        }
        // lane (g, c): channel 4c + g % 4
        const int gk = g & 3;
        const float amg = gk == 0 ? am[0] : gk == 1 ? am[1] : gk == 2 ? am[2] : am[3];
        const GroupScale gs = group_scale_t<POW2>(amg);
        if (g < 4 && FP8_IN_BOUNDS(kb * 128 + 16 * w + 4 * c + g < a.KB * 128 && mb < a.MB))
            a.sT[static_cast<int64_t>(kb * 128 + 16 * w + 4 * c + g) * a.sTk + static_cast<int64_t>(mb) * a.sTmb] =
                gs.s;
        float chs[4], chr[4];
        int chm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            chs[k] = __shfl_sync(0xffffffffu, gs.s, 4 * k + c);
            chr[k] = __shfl_sync(0xffffffffu, gs.r, 4 * k + c);
            chm[k] = __shfl_sync(0xffffffffu, gs.mode, 4 * k + c);
        }

        // pass 2: the codes of rows 16j+2g, +1 of channel 4c+ch are bytes 16j+2g, +1
        // of output row 4c+ch
        if (chm[0] == 1 && chm[1] == 1 && chm[2] == 1 && chm[3] == 1) {
            const float2 nr01 = make_float2(-chr[0], -chr[1]), s01 = make_float2(chs[0], chs[1]);
            const float2 nr23 = make_float2(-chr[2], -chr[3]), s23 = make_float2(chs[2], chs[3]);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 s4 = lds_v4(srow + 2 * (16 * j + 2 * g));
                float2 x[2][2];
#pragma unroll
                for (int b = 0; b < 2; ++b)
                    rq_decode4(lds_u32(tile + roff[b] + 2048 * j),
                               b ? make_float2(__uint_as_float(s4.z), __uint_as_float(s4.w))
                                 : make_float2(__uint_as_float(s4.x), __uint_as_float(s4.y)),
                               x[b][0], x[b][1]);
                const float2 q00 = div2_neg_t<POW2>(x[0][0], nr01, s01);
                const float2 q10 = div2_neg_t<POW2>(x[1][0], nr01, s01);
                const float2 q01 = div2_neg_t<POW2>(x[0][1], nr23, s23);
                const float2 q11 = div2_neg_t<POW2>(x[1][1], nr23, s23);
                const uint32_t at = ob ^ static_cast<uint32_t>(j << 4);
                if (FP8_IN_BOUNDS(at + 128 * 3 + 2 <= smem_addr(wst) + RQ_WSTAGE)) {
                    sts_u16_at(at, cvt_e4m3x2(q10.x, q00.x));
                    sts_u16_at(at + 128, cvt_e4m3x2(q10.y, q00.y));
                    sts_u16_at(at + 256, cvt_e4m3x2(q11.x, q01.x));
                    sts_u16_at(at + 384, cvt_e4m3x2(q11.y, q01.y));
                }
            }
        } else {
#pragma unroll 1
            for (int j = 0; j < 8; ++j) {
                const uint4 s4 = lds_v4(srow + 2 * (16 * j + 2 * g));
                float2 x[2][2];
#pragma unroll
                for (int b = 0; b < 2; ++b)
                    rq_decode4(lds_u32(tile + roff[b] + 2048 * j),
                               b ? make_float2(__uint_as_float(s4.z), __uint_as_float(s4.w))
                                 : make_float2(__uint_as_float(s4.x), __uint_as_float(s4.y)),
                               x[b][0], x[b][1]);
                const uint32_t at = ob ^ static_cast<uint32_t>(j << 4);
                const float v0[4] = {x[0][0].x, x[0][0].y, x[0][1].x, x[0][1].y};
                const float v1[4] = {x[1][0].x, x[1][0].y, x[1][1].x, x[1][1].y};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t code = quant_div(-v0[k], chs[k], chm[k]) | (quant_div(-v1[k], chs[k], chm[k]) << 8);
                    if (FP8_IN_BOUNDS(at + 128 * k + 2 <= smem_addr(wst) + RQ_WSTAGE)) sts_u16_at(at + 128 * k, code);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);   // this warp no longer reads the stage
        uint8_t* dst = a.qT + static_cast<int64_t>(kb * 128 + 16 * w) * a.ldqT + mb * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int id = lane + 32 * u;    // 16 rows x 8 chunks of 16 bytes
            const int row = id >> 3, ch = id & 7;
            if (FP8_IN_BOUNDS(kb * 128 + 16 * w + row < a.KB * 128 && mb * 128 + 16 * ch + 16 <= a.MB * 128))
                stg_v4(dst + static_cast<int64_t>(row) * a.ldqT + 16 * ch,
                       lds_v4(wst + row * 128 + ((ch ^ (row >> 2)) << 4)));
        }
        __syncwarp();
        mb += step_mb;
        kb += step_kb;
        if (kb >= a.KB) {
            kb -= a.KB;
            ++mb;
        }
    }
    if (warp == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    if (!ok && lane == 0) {
        record_status(kStatusTimeout);
        spin_ns(100000);   // let the loads still in flight land before the CTA may exit
    }
}

}  // namespace fp8fg
