// probe.cuh -- tensor-core accumulation probe (no promotion).
//
// The GEMM promotes tensor-core partial sums to FP32 every 128 K because the
// tensor cores of the previous generation keep fewer bits when they
// accumulate long sums (why-be.why-be.co.kr post 55081: about 14 bits on
// H800, and an error near 2% at K = 4096).  This kernel measures what the
// B300 tensor core keeps: one CTA computes D[128][256] = sum_k A[m][k] B[n][k]
// over E4M3 codes (no scales) with tcgen05.mma kind::f8f6f4, accumulating the
// whole K in TMEM, and writes D as FP32.  Single-CTA tcgen05 forms only;
// one shared-memory stage (the probe measures numerics, not speed).
#pragma once

#include "ptx.cuh"

namespace fp8fg {
namespace probe {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr uint32_t A_BYTES = BM * BK;
constexpr uint32_t B_BYTES = BN * BK;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
constexpr size_t SMEM = 1024 + A_BYTES + B_BYTES + 64;

// Launch: 1 CTA of 128 threads, SMEM bytes of dynamic shared memory.
__global__ void __launch_bounds__(128, 1) k_mma_accumulation_probe(const __grid_constant__ CUtensorMap tmA,
                                                                   const __grid_constant__ CUtensorMap tmB,
                                                                   int k_blocks, float* __restrict__ out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sm_a = base;
    uint8_t* sm_b = base + A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + A_BYTES + B_BYTES);
    uint64_t* mma_done = full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (threadIdx.x == 0) {
        for (int kb = 0; kb < k_blocks; ++kb) {
            const uint32_t ph = static_cast<uint32_t>(kb) & 1u;
            mbar_arrive_expect_tx(full, A_BYTES + B_BYTES);
            tma_load_2d(sm_a, &tmA, full, kb * BK, 0);
            tma_load_2d(sm_b, &tmB, full, kb * BK, 0);
            if (!mbar_wait(full, ph, nullptr)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint64_t ad = sdesc_kmajor_sw128(smem_addr(sm_a));
            const uint64_t bd = sdesc_kmajor_sw128(smem_addr(sm_b));
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
                umma_f8(tmem, ad + 2u * k, bd + 2u * k, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(mma_done);      // the stage is reused only after these MMAs complete
            if (!mbar_wait(mma_done, ph, nullptr)) {
                ok = false;
                break;
            }
        }
        if (!ok) {
            record_status(kStatusTimeout);
            spin_ns(100000);            // let a load or MMA still in flight finish
        }
    }
    __syncthreads();
    tc_fence_after_sync();
    // warp w reads TMEM lanes 32w .. 32w + 31 (rows), all 256 columns
    const int row = warp * 32 + lane;
    for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld_32cols(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c, r);
        tmem_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (FP8_IN_BOUNDS(row < BM && c + j < BN)) out[static_cast<int64_t>(row) * BN + c + j] = __uint_as_float(r[j]);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace probe
}  // namespace fp8fg
