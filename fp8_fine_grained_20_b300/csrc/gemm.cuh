// gemm.cuh -- block-scaled FP8 GEMM with FP32 promotion every 128 K, for
// sm_103a (tcgen05 + TMA + TMEM), in three flavours selected at compile time:
// forward (1x128 A scales x 128x128 B scales), weight gradient (1x128-along-K
// scales on both operands, i.e. a per-column B scale) and grouped (MoE
// experts, forward flavour per expert).
//
// Method (DeepSeek-V3 FP8 excerpts): tensor cores accumulate a K-interval with
// limited precision; at the end of the interval the partial sums are copied
// to FP32 registers on CUDA cores, multiplied by the two group scales and
// accumulated in full FP32 (why-be.why-be.co.kr post 55081, Figure 7(b);
// xn--jj0bz6z98ct0a29q.com post 362465).  The interval here is the 128-wide
// quantization group, so each promotion applies exactly one (sA, sB) pair.
//
// B300 design (not the H800 one, where two WGMMA warpgroups alternate
// between MMA and promotion):
//   * CTA pairs (clusters of 2 on neighbouring SMs), persistent: each pair
//     owns 256 x 256 output tiles in a grouped raster.  One tcgen05.mma with
//     cta_group::2 computes M = 256 (128 rows in each CTA) x N = 256, reading
//     A from each CTA's own shared memory and half of B's 256 rows from each
//     CTA, so every SM loads 32 KB per 128-deep K-block instead of 48 KB;
//   * warp 0 (both CTAs): TMA producer -- this CTA's A box (128 x 128 B) and B
//     half (128 x 128 B), 128-byte swizzle, 5-stage ring; the transaction
//     bytes of both CTAs are counted on the even CTA's "full" barrier; near
//     the end of each tile it asks L2 for the next tile's first K-blocks;
//   * warp 1 (even CTA): MMA issuer (the whole warp runs the loop, one elected
//     lane issues) -- per K-block, 4 x tcgen05.mma (K = 32)
//     into one of two 256-column TMEM partial buffers, then one commit to the
//     stage's "done" barrier in both CTAs, which both frees the smem stage for
//     the producers and publishes the partial to the promotion warps (the
//     issuing thread is the scarce resource: one commit per K-block, not two);
//   * warp 2 (both CTAs): scale loader -- cp.async of the K-block's 128 row
//     scales of this CTA and the tile's B scales into an 8-slot ring;
//   * warps 4-11 (both CTAs): promotion -- tcgen05.ld of this CTA's 128 x 256
//     partial (each warp: its 32 TMEM lanes = rows, one 128-column half, in
//     four 32-column loads, two in flight), release of the TMEM buffer to the
//     even CTA as soon as the last two loads land, acc += partial * sA * sB in
//     FP32 registers with packed FP32x2 FMAs; at tile end bf16 through
//     swizzled shared-memory staging tiles and TMA stores (or the 1x128
//     codes and scales of the quantizing epilogue).  With
//     per-column B scales (weight gradient) the loads use the 16x128b shape
//     instead, so that a thread holds one column in four of four rows and
//     reads 32 column scales per K-block rather than all 128 of its half.
//   The MMA of K-block kb+1 runs while K-block kb is promoted.
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quant.cuh"

namespace fp8fg {
namespace gemm {

constexpr int BM = 128;           // rows per CTA
constexpr int PM = 256;           // rows per CTA pair (MMA M)
constexpr int BN = 256;           // columns per tile (MMA N)
constexpr int BNH = BN / 2;       // B rows loaded by each CTA
constexpr int BK = 128;
constexpr int STAGES = 5;
constexpr int SSLOTS = 8;
constexpr int THREADS = 384;
constexpr int PROMO_WARPS = 8;
constexpr int GROUP_PM = 8;       // pair-rows sharing each n-block sweep of the raster
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t A_BYTES = BM * BK;
constexpr uint32_t B_BYTES = BNH * BK;
constexpr uint32_t STAGE_TX = 2 * (A_BYTES + B_BYTES);   // both CTAs' loads, counted in the even CTA
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_e4m3_f32(PM, BN);

constexpr int SB_BLOCK = 0;  // sB[kb][n/128]
constexpr int SB_COL = 1;    // sB[kb][n]

// bf16 epilogue staging: one 32-row x 64-column tile (4 KB, 128-byte TMA
// swizzle) per promotion warp
constexpr uint32_t C_STAGE_BYTES = 32 * 64 * 2;

constexpr size_t OFF_A = 0;
constexpr size_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr size_t OFF_C = OFF_B + STAGES * B_BYTES;
constexpr size_t OFF_SA = OFF_C + PROMO_WARPS * C_STAGE_BYTES;
constexpr size_t OFF_SB = OFF_SA + SSLOTS * BM * sizeof(float);
constexpr size_t OFF_BAR = OFF_SB + SSLOTS * BN * sizeof(float);
constexpr int N_BARS = 2 * STAGES + 2 + 2 * SSLOTS + 1;
constexpr size_t OFF_MISC = OFF_BAR + N_BARS * sizeof(uint64_t);
constexpr size_t OFF_GOFF = OFF_MISC + 16;
constexpr size_t SMEM_PLAIN = 1024 + OFF_GOFF;
// the grouped flavour's promotion warps park their tile's place here during
// the K-loop (16 bytes per warp)
constexpr size_t OFF_TSTASH = (OFF_GOFF + 2 * (MAX_GROUPS + 1) * sizeof(int) + 15) & ~size_t(15);
constexpr size_t SMEM_GROUPED = 1024 + OFF_TSTASH + PROMO_WARPS * 16;

struct Args {
    const float* sA;
    int64_t sa_sm, sa_skb;
    const float* sB;
    int64_t sb_skb, sb_sn;
    int64_t sb_group_stride;  // grouped: floats between experts' scale tables
    uint16_t* C;              // bf16 output (plain epilogue)
    int64_t ldc;
    int M, N, K;
    int m_blocks, n_blocks, k_blocks;  // n_blocks: 256-column tiles
    int sb_cols;              // number of valid sB columns: N/128 (block) or N (per column)
    const int32_t* offsets;   // grouped only (device)
    int G;
    uint64_t wait_ns;         // bound of every pipeline wait (kWaitTimeoutNs unless a test shortens it)
    int withhold;             // test only: the TMA producer stops after the first K-block of its first tile
};

// Outputs of the quantizing epilogue (a separate kernel parameter, so that
// the other kernels' parameter block and register allocation are unchanged).
struct QArgs {
    uint8_t* Cq;              // codes, row stride ldcq
    int64_t ldcq;
    float* sC;                // scales, logical [M][N/128] at sC[m*sc_m + nb*sc_nb]
    int64_t sc_m, sc_nb;
};

__device__ const float g_zero_scale = 0.0f;

// One pair tile: rows [row0, row0 + 256) of A and C (this CTA's half starts
// at row0 + 128 * rank), columns [nb * 256, nb * 256 + 256), expert g and the
// end of that expert's rows (rows at or beyond row_end are computed but not
// stored).
struct Tile {
    int row0, nb, g, row_end;
};

// Pair-tile index -> (pair-row, n-block): GROUP consecutive pair-rows share
// each n-block before moving on, so concurrently running pairs reuse A and B
// in L2.  The grouped power-of-two GEMM, whose A streams from DRAM, uses
// groups of 2 (each A row block is consumed by its n-blocks close together in
// time: measured 7% faster than 8 on the MoE workload); the others use 8.
// GROUP is a compile-time constant: a run-time group costs the promoting
// forward GEMM's epilogue enough registers to spill (measured 2.3x slower).
template <int GROUP>
__device__ __forceinline__ void raster(int t, int pair_rows, int n_blocks, int& pr, int& nb) {
    const int span = GROUP * n_blocks;
    const int grp = t / span;
    const int first = grp * GROUP;
    const int gm = min(GROUP, pair_rows - first);
    const int r = t - grp * span;
    pr = first + r % gm;
    nb = r / gm;
}

// Expert owning pair-row pr: the largest g with ppre[g] <= pr (ppre[g] = pair
// rows of experts 0..g-1; empty experts are skipped because their prefix
// equals the next one's).
__device__ __forceinline__ int expert_of_pair_row(int pr, const int* ppre, int G) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ppre[mid] <= pr) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <bool GROUPED, int GROUP = GROUP_PM>
__device__ __forceinline__ Tile tile_at(int t, const Args& p, int pair_rows, const int* goff, const int* ppre) {
    Tile x;
    int pr;
    raster<GROUP>(t, pair_rows, p.n_blocks, pr, x.nb);
    if (!GROUPED) {
        x.g = 0;
        x.row0 = pr * PM;
        x.row_end = p.M;
    } else {
        x.g = expert_of_pair_row(pr, ppre, p.G);
        x.row0 = goff[x.g] + (pr - ppre[x.g]) * PM;
        x.row_end = goff[x.g + 1];
    }
    return x;
}

// While the current tile's last K-blocks stream in, the producer asks L2 for
// the first PREFETCH_BLOCKS K-blocks of this CTA's boxes of its next tile, so
// the next tile does not start on DRAM latency (the shared-memory ring holds
// only the current tile's K-blocks at that point).
constexpr int PREFETCH_AHEAD = 16;   // K-blocks before the end of a tile
constexpr int PREFETCH_BLOCKS = 8;
template <bool GROUPED, int GROUP = GROUP_PM>
__device__ __noinline__ void prefetch_next_tile(int t, int num_tiles, const Args& p, int pair_rows, const int* goff,
                                                   const int* ppre, uint32_t rank, const CUtensorMap* tmA,
                                                   const CUtensorMap* tmB) {
    if (t >= num_tiles) return;
    const Tile tl = tile_at<GROUPED, GROUP>(t, p, pair_rows, goff, ppre);
    const int a_y = tl.row0 + static_cast<int>(rank) * BM;
    const int b_y = tl.g * p.N + tl.nb * BN + static_cast<int>(rank) * BNH;
    const int n = min(PREFETCH_BLOCKS, p.k_blocks);
    for (int kb = 0; kb < n; ++kb) {
        tma_prefetch_l2_2d(tmA, kb * BK, a_y);
        tma_prefetch_l2_2d(tmB, kb * BK, b_y);
    }
}


template <int SBK, int OFF>
__device__ __forceinline__ void promote32(float (&acc)[128], const uint32_t (&r)[32], float sc, float sa,
                                          const float* sbv) {
    if (SBK == SB_BLOCK) {
        const float2 sc2 = make_float2(sc, sc);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            float2 a = make_float2(acc[OFF + j], acc[OFF + j + 1]);
            a = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2, a);
            acc[OFF + j] = a.x;
            acc[OFF + j + 1] = a.y;
        }
    } else {
        const float2 sa2 = make_float2(sa, sa);
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 b = *reinterpret_cast<const float4*>(sbv + OFF + j);
            const float2 w0 = __fmul2_rn(sa2, make_float2(b.x, b.y));
            const float2 w1 = __fmul2_rn(sa2, make_float2(b.z, b.w));
            float2 a0 = make_float2(acc[OFF + j], acc[OFF + j + 1]);
            float2 a1 = make_float2(acc[OFF + j + 2], acc[OFF + j + 3]);
            a0 = __ffma2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), w0, a0);
            a1 = __ffma2_rn(make_float2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])), w1, a1);
            acc[OFF + j] = a0.x;
            acc[OFF + j + 1] = a0.y;
            acc[OFF + j + 2] = a1.x;
            acc[OFF + j + 3] = a1.y;
        }
    }
}

// Column-scale promotion of part of one 16x128b chunk (see
// tmem_ld_16x128b_x16): the thread's two rows (sa2 = their row scales) at its
// columns J0 .. J0+NJ-1 of the chunk (one column in four), sb[j - J0] their
// scales; acc[32 CH + 2j + e] is row e at column j.  Same arithmetic as
// promote32: acc += partial * (sA sB).
template <int CH, int J0, int NJ>
__device__ __forceinline__ void promote_col16(float (&acc)[128], const uint32_t (&r)[32], float2 sa2,
                                              const float (&sb)[NJ]) {
#pragma unroll
    for (int j = J0; j < J0 + NJ; ++j) {
        const float2 w = __fmul2_rn(sa2, make_float2(sb[j - J0], sb[j - J0]));
        float2 a = make_float2(acc[32 * CH + 2 * j], acc[32 * CH + 2 * j + 1]);
        a = __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), w, a);
        acc[32 * CH + 2 * j] = a.x;
        acc[32 * CH + 2 * j + 1] = a.y;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Records the timeout and stops both CTAs of the pair: the flag of this CTA
// and of its peer are set, so every bounded wait of the pair returns early.
__device__ __forceinline__ void signal_abort(volatile int* abort_flag, uint32_t peer) {
    *abort_flag = 1;
    st_shared_cluster_u32(mapa_shared(smem_addr(const_cast<int*>(abort_flag)), peer), 1u);
    record_status(kStatusTimeout);
}

// Launch: clusters of 2 CTAs along x, THREADS threads, SMEM_PLAIN or
// SMEM_GROUPED bytes of dynamic shared memory, one CTA per SM.  QOUT: the
// epilogue writes the bf16-rounded output 1x128-quantized (codes + scales)
// instead of bf16; each promotion thread holds exactly one 1x128 group (one
// row, 128 columns), so the group amax needs no communication.
template <int SBK, bool GROUPED, bool QOUT = false>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_blockscaled(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const Args p, const QArgs qo) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sm_a = base + OFF_A;
    uint8_t* sm_b = base + OFF_B;
    uint8_t* sm_c = base + OFF_C;
    float* sm_sa = reinterpret_cast<float*>(base + OFF_SA);
    float* sm_sb = reinterpret_cast<float*>(base + OFF_SB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + OFF_BAR);
    uint64_t* full = bars;               // even CTA: both CTAs' TMA bytes of a stage
    uint64_t* done = full + STAGES;      // both: the K-block held by a stage is multiplied
                                         // (stage free for TMA, partial ready for promotion)
    uint64_t* tempty = done + STAGES;    // even CTA: partial buffer read by both CTAs
    uint64_t* sfull = tempty + 2;
    uint64_t* sempty = sfull + SSLOTS;
    uint64_t* drain = sempty + SSLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + OFF_MISC + 4);
    int* groups_ok = reinterpret_cast<int*>(base + OFF_MISC + 8);
    int* goff = reinterpret_cast<int*>(base + OFF_GOFF);
    int* ppre = goff + (MAX_GROUPS + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&tempty[i], 2 * PROMO_WARPS);
        for (int i = 0; i < SSLOTS; ++i) {
            mbar_init(&sfull[i], 32);
            mbar_init(&sempty[i], PROMO_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *groups_ok = 1;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (!QOUT) tma_prefetch_desc(&tmC);
    }
    if (GROUPED) {
        for (int i = threadIdx.x; i <= p.G; i += THREADS) goff[i] = p.offsets[i];
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncthreads();
    if (GROUPED && threadIdx.x == 0) {
        // validate the offsets and build the prefix of pair-rows per expert
        bool ok = goff[0] >= 0 && goff[p.G] <= p.M && (goff[p.G] % BM) == 0;
        int acc = 0;
        for (int g = 0; g < p.G; ++g) {
            ok = ok && goff[g] <= goff[g + 1] && (goff[g] % BM) == 0;
            ppre[g] = acc;
            if (ok) acc += (goff[g + 1] - goff[g] + PM - 1) / PM;
        }
        ppre[p.G] = acc;
        if (!ok) {
            *groups_ok = 0;
            if (blockIdx.x == 0) record_status(kStatusBadGroups);
        }
    }
    tc_fence_before_sync();
    cluster_sync();     // barriers of both CTAs initialised, TMEM allocated, offsets checked
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int pair_rows = GROUPED ? ppre[p.G] : (p.m_blocks + 1) / 2;
    const int num_tiles = (*groups_ok) ? pair_rows * p.n_blocks : 0;
    const int pair = static_cast<int>(cluster_id_x());
    const int n_pairs = static_cast<int>(n_clusters_x());

    if (warp < 4) {
      regs_decrease<56>();
      if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true, withheld = false;
            for (int t = pair; ok && !withheld && t < num_tiles; t += n_pairs) {
                const Tile tl = tile_at<GROUPED>(t, p, pair_rows, goff, ppre);
                const int a_y = tl.row0 + static_cast<int>(rank) * BM;
                const int b_y = tl.g * p.N + tl.nb * BN + static_cast<int>(rank) * BNH;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&done[stage], phase ^ 1u, abort_flag, p.wait_ns)) {
                        signal_abort(abort_flag, peer);
                        ok = false;
                        break;
                    }
                    const uint32_t fbar = mapa_shared(smem_addr(&full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(&full[stage], STAGE_TX);
                    tma_load_2d_pair(sm_a + stage * A_BYTES, &tmA, fbar, kb * BK, a_y);
                    tma_load_2d_pair(sm_b + stage * B_BYTES, &tmB, fbar, kb * BK, b_y);
                    if (kb == max(0, p.k_blocks - PREFETCH_AHEAD))
                        prefetch_next_tile<GROUPED>(t + n_pairs, num_tiles, p, pair_rows, goff, ppre, rank, &tmA, &tmB);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (p.withhold) {   // test of the failure path: the next K-block never arrives
                        withheld = true;
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer ----
        // The whole warp runs the loop (warp-uniform descriptors); one elected
        // lane, the same throughout, issues the MMAs and their commits.
        if (leader) {
            uint32_t stage = 0, phase = 0, it = 0;
            bool ok = true;
            for (int t = pair; ok && t < num_tiles; t += n_pairs) {
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    const uint32_t buf = it & 1u;
                    const uint32_t tph = (it >> 1) & 1u;
                    const bool ready = mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, p.wait_ns) &&
                                       mbar_wait(&full[stage], phase, abort_flag, p.wait_ns);
                    if (!__all_sync(0xffffffffu, ready)) {
                        if (lane == 0) signal_abort(abort_flag, peer);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (elect_one_sync()) {
                        const uint32_t d = tmem + buf * BN;
                        const uint64_t ad = sdesc_kmajor_sw128(smem_addr(sm_a + stage * A_BYTES));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_addr(sm_b + stage * B_BYTES));
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k) {
                            // +32 bytes along K inside the 128-byte swizzle atom: +2 in the (>>4) address field
                            umma_f8_pair(d, ad + 2u * k, bd + 2u * k, IDESC, k > 0 ? 1u : 0u);
                        }
                        umma_commit_pair_mc(&done[stage], 0x3);
                    }
                    __syncwarp();
                    ++it;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every MMA this warp issued completes before TMEM is released
            if (elect_one_sync()) umma_commit_pair_mc(drain, 0x1);
            __syncwarp();
            mbar_wait(drain, 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        }
    } else if (warp == 2) {
        // ------------------------------------------------ scale loader ----
        // Scales contiguous along the rows (A) or columns (per-column B) in
        // global memory, the usual layout, are copied four per 16-byte
        // cp.async into the same shared-memory layout; other strides take one
        // copy per scale.  This warp shares its scheduler with two promotion
        // warps, so its instruction count is on their critical path.
        const bool vec_a = p.sa_sm == 1 && (p.sa_skb & 3) == 0 && (reinterpret_cast<uintptr_t>(p.sA) & 15u) == 0;
        const bool vec_b = SBK == SB_COL && p.sb_sn == 1 && (p.sb_skb & 3) == 0 && (p.sb_group_stride & 3) == 0 &&
                           (reinterpret_cast<uintptr_t>(p.sB) & 15u) == 0;
        uint32_t slot = 0, sph = 0;
        bool ok = true;
        for (int t = pair; ok && t < num_tiles; t += n_pairs) {
            const Tile tl = tile_at<GROUPED>(t, p, pair_rows, goff, ppre);
            const int r0 = tl.row0 + static_cast<int>(rank) * BM;
            const float* sb_base = p.sB + static_cast<int64_t>(tl.g) * p.sb_group_stride;
            for (int kb = 0; kb < p.k_blocks; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(&sempty[slot], sph ^ 1u, abort_flag, p.wait_ns))) {
                    if (lane == 0) signal_abort(abort_flag, peer);
                    ok = false;
                    break;
                }
                float* dsa = sm_sa + slot * BM;
                if (vec_a) {
                    const int row = r0 + 4 * lane;   // rows row .. row + 3: all in or all out (M % 128 == 0)
                    if (row < p.M) {
                        cp_async_16(dsa + 4 * lane, p.sA + row + static_cast<int64_t>(kb) * p.sa_skb);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) cp_async_4(dsa + 4 * lane + e, &g_zero_scale);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < BM / 32; ++i) {
                        const int r = lane + 32 * i;
                        const int row = r0 + r;
                        const float* src = (row < p.M) ? p.sA + static_cast<int64_t>(row) * p.sa_sm +
                                                             static_cast<int64_t>(kb) * p.sa_skb
                                                       : &g_zero_scale;
                        cp_async_4(dsa + r, src);
                    }
                }
                float* dsb = sm_sb + slot * BN;
                if (SBK == SB_COL && vec_b) {
                    // columns 4 lane .. + 3 of each 128-column half: all in or all out (N % 128 == 0)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 128 * h + 4 * lane;
                        const int c = tl.nb * BN + j;
                        if (c < p.sb_cols) {
                            cp_async_16(dsb + j, sb_base + static_cast<int64_t>(kb) * p.sb_skb + c);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) cp_async_4(dsb + j + e, &g_zero_scale);
                        }
                    }
                } else if (SBK == SB_BLOCK) {
                    if (lane < BN / 128) {
                        const int c = tl.nb * (BN / 128) + lane;
                        const float* src = (c < p.sb_cols) ? sb_base + static_cast<int64_t>(kb) * p.sb_skb +
                                                                 static_cast<int64_t>(c) * p.sb_sn
                                                           : &g_zero_scale;
                        cp_async_4(dsb + lane, src);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < BN / 32; ++i) {
                        const int j = lane + 32 * i;
                        const int c = tl.nb * BN + j;
                        const float* src = (c < p.sb_cols) ? sb_base + static_cast<int64_t>(kb) * p.sb_skb +
                                                                 static_cast<int64_t>(c) * p.sb_sn
                                                           : &g_zero_scale;
                        cp_async_4(dsb + j, src);
                    }
                }
                cp_async_arrive_noinc(&sfull[slot]);
                if (++slot == SSLOTS) {
                    slot = 0;
                    sph ^= 1u;
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
      }
    } else {
        // Registers of the promotion warps (setmaxnreg; the four other warps
        // drop to 56).  Measured on B300: the plain forward / data-gradient
        // flavour runs 7% faster with 184 than with 224 (the allocator then
        // spills 32 bytes instead of 92); the weight-gradient and quantizing
        // flavours are fastest with 224, the grouped one (with its tile's
        // place parked in shared memory, below) with 208.
        regs_increase<GROUPED ? 208 : (SBK == SB_BLOCK && !QOUT) ? 184 : 224>();
        // ------------------------------------- promotion and epilogue ----
        const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
        const int half = (warp - 4) >> 2;       // output columns half*128 .. +127
        const int row = quarter * 32 + lane;    // row of this CTA's 128-row half (32x32b loads)
        const int r4 = lane >> 2, q4 = lane & 3; // 16x128b loads: rows r4 (+8, +16, +24), columns q4 mod 4
        uint32_t it = 0;   // K-blocks promoted so far; every ring position derives from it
        bool ok = true;
        for (int t = pair; ok && t < num_tiles; t += n_pairs) {
            // the tile's place, found before the K-loop (the grouped search then runs
            // while few registers are live)
            Tile tl = tile_at<GROUPED>(t, p, pair_rows, goff, ppre);
            if constexpr (GROUPED) {
                // parked in shared memory until the epilogue: held in registers
                // across the K-loop it made the allocator spill inside the loop
                // (ncu: about three local stores per warp and K-block); parked,
                // the grouped GEMM runs 3-6% faster on B300
                if (lane == 0)
                    *reinterpret_cast<int4*>(base + OFF_TSTASH + 16 * (warp - 4)) =
                        make_int4(tl.row0, tl.row_end, tl.nb, tl.g);
                __syncwarp();
            }
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.0f;
            for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
                const uint32_t buf = it & 1u;
                const uint32_t slot = it % SSLOTS, sph = (it / SSLOTS) & 1u;
                const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
                const bool ready = mbar_wait(&sfull[slot], sph, abort_flag, p.wait_ns) &&
                                   mbar_wait(&done[stage], phase, abort_flag, p.wait_ns);
                if (!__all_sync(0xffffffffu, ready)) {  // warp-uniform: tcgen05.ld is .sync.aligned
                    if (lane == 0) signal_abort(abort_flag, peer);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN + half * 128;
                uint32_t r0[32], r1[32];
                if constexpr (SBK == SB_COL) {
                    // 16x128b chunks: ch = (lane half L = 16 (ch & 1), column half C = 64 (ch >> 1));
                    // a thread needs only the scales of its 32 columns (one column in four),
                    // each shared by both lane halves and loaded eight at a time
                    const float* sav = sm_sa + slot * BM + quarter * 32 + r4;
                    const float2 sa_lo = make_float2(sav[0], sav[8]);
                    const float2 sa_hi = make_float2(sav[16], sav[24]);
                    const float* sbw = sm_sb + slot * BN + half * 128 + q4;
                    float sbv[8];
                    tmem_ld_16x128b_x16(taddr, r0);
                    tmem_ld_16x128b_x16(taddr + (16u << 16), r1);
#pragma unroll
                    for (int j = 0; j < 8; ++j) sbv[j] = sbw[4 * j];
                    tmem_wait_ld2(r0, r1);
                    promote_col16<0, 0, 8>(acc, r0, sa_lo, sbv);
                    promote_col16<1, 0, 8>(acc, r1, sa_hi, sbv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) sbv[j] = sbw[32 + 4 * j];
                    promote_col16<0, 8, 8>(acc, r0, sa_lo, sbv);
                    tmem_ld_16x128b_x16(taddr + 64, r0);
                    promote_col16<1, 8, 8>(acc, r1, sa_hi, sbv);
                    tmem_ld_16x128b_x16(taddr + (16u << 16) + 64, r1);
                    tmem_wait_ld2(r0, r1);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(&tempty[buf]), 0));  // the even CTA's
#pragma unroll
                    for (int j = 0; j < 8; ++j) sbv[j] = sbw[64 + 4 * j];
                    promote_col16<2, 0, 8>(acc, r0, sa_lo, sbv);
                    promote_col16<3, 0, 8>(acc, r1, sa_hi, sbv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) sbv[j] = sbw[96 + 4 * j];
                    promote_col16<2, 8, 8>(acc, r0, sa_lo, sbv);
                    promote_col16<3, 8, 8>(acc, r1, sa_hi, sbv);
                } else {
                    const float sa = sm_sa[slot * BM + row];
                    const float* sbv = sm_sb + slot * BN + half * 128;
                    const float sc = __fmul_rn(sa, sm_sb[slot * BN + half]);
                    tmem_ld_32cols(taddr + 0, r0);
                    tmem_ld_32cols(taddr + 32, r1);
                    tmem_wait_ld2(r0, r1);
                    promote32<SBK, 0>(acc, r0, sc, sa, sbv);
                    tmem_ld_32cols(taddr + 64, r0);
                    promote32<SBK, 32>(acc, r1, sc, sa, sbv);
                    tmem_ld_32cols(taddr + 96, r1);
                    tmem_wait_ld2(r0, r1);
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(&tempty[buf]), 0));  // the even CTA's
                    promote32<SBK, 64>(acc, r0, sc, sa, sbv);
                    promote32<SBK, 96>(acc, r1, sc, sa, sbv);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[slot]);
            }
            if (!ok) break;
            if constexpr (GROUPED) {
                const volatile int* ts = reinterpret_cast<const volatile int*>(base + OFF_TSTASH + 16 * (warp - 4));
                tl.row0 = ts[0];
                tl.row_end = ts[1];
                tl.nb = ts[2];
                tl.g = ts[3];
            }
            const int grow = tl.row0 + static_cast<int>(rank) * BM + row;
            const int n0 = tl.nb * BN + half * 128;
            if constexpr (SBK == SB_COL) {
                // rows and groups are whole 128-row blocks: the test is uniform per CTA
                const int g0 = tl.row0 + static_cast<int>(rank) * BM + quarter * 32 + r4;
                if (!(tl.row0 + static_cast<int>(rank) * BM < tl.row_end && n0 < p.N)) continue;
                if constexpr (QOUT) {
#pragma unroll
                for (int rs = 0; rs < 4; ++rs) {          // rows g0 + 16 (rs >> 1) + 8 (rs & 1)
                    const int grw = g0 + 16 * (rs >> 1) + 8 * (rs & 1);
                    const int e = rs & 1, lh = rs >> 1;
                        // the row's 128 columns sit in the four lanes of this quad
                        uint32_t w[16];
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                w[8 * c + k] = pack_bf16x2(acc[32 * (2 * c + lh) + 2 * (2 * k) + e],
                                                           acc[32 * (2 * c + lh) + 2 * (2 * k + 1) + e]);
                        uint32_t h = 0u;
#pragma unroll
                        for (int k = 0; k < 16; ++k) h = umax16x2(h, w[k] & 0x7FFF7FFFu);
                        h = umax16x2(h, __shfl_xor_sync(0xffffffffu, h, 1));
                        h = umax16x2(h, __shfl_xor_sync(0xffffffffu, h, 2));
                        const GroupScale gs = group_scale(hmax_bf16x2_to_f32(h));
                        uint8_t* qrow = qo.Cq + static_cast<int64_t>(grw) * qo.ldcq + n0 + q4;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                // codes of columns 64c + 4j + q4, j = 8k .. 8k+7
                                const uint2 cd = quant8_bf16(
                                    make_uint4(w[8 * c + 4 * k], w[8 * c + 4 * k + 1], w[8 * c + 4 * k + 2],
                                               w[8 * c + 4 * k + 3]),
                                    gs);
#pragma unroll
                                for (int b = 0; b < 8; ++b)
                                    if (FP8_IN_BOUNDS(grw < p.M && n0 + q4 + 64 * c + 4 * (8 * k + b) < p.N))
                                        qrow[64 * c + 4 * (8 * k + b)] =
                                            static_cast<uint8_t>(((b < 4 ? cd.x : cd.y) >> (8 * (b & 3))) & 0xFFu);
                            }
                        if (q4 == 0 && FP8_IN_BOUNDS(grw < p.M && n0 < p.N))
                            qo.sC[static_cast<int64_t>(grw) * qo.sc_m + static_cast<int64_t>(n0 / 128) * qo.sc_nb] =
                                gs.s;
                }
                } else {
                    // 4x4 transposes of bf16 across the quad, two shuffles each: lane q then
                    // holds columns 4(4g + q) .. +3 of a row; the 8 bytes go into the warp's
                    // swizzled 32 x 64 staging tile (row r: 16-byte chunk j at j ^ (r % 8)),
                    // one TMA store per 64 columns
                    uint8_t* stg = sm_c + (warp - 4) * C_STAGE_BYTES;
                    const int wrow0 = tl.row0 + static_cast<int>(rank) * BM + quarter * 32;
                    const uint32_t sel_w0 = (q4 == 0) ? 0x5410u : (q4 == 1) ? 0x3254u : (q4 == 2) ? 0x7610u : 0x3276u;
                    const uint32_t sel_w1 = (q4 == 0) ? 0x7610u : (q4 == 1) ? 0x3276u : (q4 == 2) ? 0x5410u : 0x3254u;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        if (lane == 0) bulk_wait_read_all();   // the previous store has read the tile
                        __syncwarp();
#pragma unroll
                        for (int rs = 0; rs < 4; ++rs) {      // local rows 16 (rs >> 1) + 8 (rs & 1) + r4
                            const int e = rs & 1, lh = rs >> 1;
                            const int rl = 16 * lh + 8 * e + r4;
#pragma unroll
                            for (int g = 0; g < 4; ++g) {
                                const int o = 32 * (2 * c + lh) + 8 * g + e;   // acc[o + 2k]: column 4(4g+k) + q
                                const uint32_t p0 = pack_bf16x2(acc[o + 0], acc[o + 2]);
                                const uint32_t p1 = pack_bf16x2(acc[o + 4], acc[o + 6]);
                                const uint32_t x = (q4 & 2) ? p1 : p0;
                                const uint32_t y = __shfl_xor_sync(0xffffffffu, (q4 & 2) ? p0 : p1, 2);
                                const uint32_t rr =
                                    __shfl_xor_sync(0xffffffffu, __byte_perm(x, y, (q4 & 1) ? 0x5410u : 0x7632u), 1);
                                const uint32_t a = (q4 & 2) ? y : x;
                                const uint32_t b = (q4 & 2) ? x : y;
                                const uint32_t off = rl * 128 + (((2 * g + (q4 >> 1)) ^ r4) << 4) + (q4 & 1) * 8;
                                if (FP8_IN_BOUNDS(off + 8 <= C_STAGE_BYTES))
                                    sts_v2(stg + off, make_uint2(__byte_perm(a, rr, sel_w0), __byte_perm(b, rr, sel_w1)));
                            }
                        }
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0 && FP8_IN_BOUNDS(wrow0 + 32 <= p.M && n0 + 64 * c + 64 <= p.N)) {
                            tma_store_2d(&tmC, stg, n0 + 64 * c, wrow0);
                            bulk_commit_group();
                        }
                    }
                }
                continue;
            }
            if (!(grow < tl.row_end && n0 < p.N)) continue;
            if constexpr (QOUT) {
                // bf16 rounding of the output as the plain epilogue does, then the
                // 1x128 quantizer's arithmetic on those bf16 values
                uint32_t w[64];
#pragma unroll
                for (int j = 0; j < 64; ++j) w[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
                uint32_t h = 0u;
#pragma unroll
                for (int j = 0; j < 64; ++j) h = umax16x2(h, w[j] & 0x7FFF7FFFu);
                const GroupScale gs = group_scale(hmax_bf16x2_to_f32(h));
                uint8_t* qrow = qo.Cq + static_cast<int64_t>(grow) * qo.ldcq + n0;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint2 lo = quant8_bf16(make_uint4(w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3]), gs);
                    const uint2 hi =
                        quant8_bf16(make_uint4(w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]), gs);
                    if (FP8_IN_BOUNDS(grow < p.M && n0 + 16 * c + 16 <= p.N))
                        stg_v4(qrow + 16 * c, make_uint4(lo.x, lo.y, hi.x, hi.y));
                }
                if (FP8_IN_BOUNDS(grow < p.M && n0 < p.N))
                    qo.sC[static_cast<int64_t>(grow) * qo.sc_m + static_cast<int64_t>(n0 / 128) * qo.sc_nb] = gs.s;
            } else {
                // the warp's 32 rows x 128 columns in two 32 x 64 TMA stores: each lane
                // writes its row into the swizzled staging tile (16-byte chunk j of row r
                // at chunk j ^ (r % 8): conflict-free), then lane 0 issues the store
                uint8_t* stg = sm_c + (warp - 4) * C_STAGE_BYTES;
                const int wrow0 = tl.row0 + static_cast<int>(rank) * BM + quarter * 32;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (lane == 0) bulk_wait_read_all();   // the previous store has read the tile
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int o = 64 * h + 8 * j;
                        if (FP8_IN_BOUNDS(lane * 128 + ((j ^ (lane & 7)) << 4) + 16 <= static_cast<int>(C_STAGE_BYTES)))
                        sts_v4(stg + lane * 128 + ((j ^ (lane & 7)) << 4),
                               make_uint4(pack_bf16x2(acc[o + 0], acc[o + 1]), pack_bf16x2(acc[o + 2], acc[o + 3]),
                                          pack_bf16x2(acc[o + 4], acc[o + 5]), pack_bf16x2(acc[o + 6], acc[o + 7])));
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0 && FP8_IN_BOUNDS(wrow0 + 32 <= tl.row_end && n0 + 64 * h + 64 <= p.N)) {
                        tma_store_2d(&tmC, stg, n0 + 64 * h, wrow0);
                        bulk_commit_group();
                    }
                }
            }
        }
        // every store of this warp has completed before its staging tile is released
        if (!QOUT && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // Teardown.  After the first cluster barrier no thread of either CTA waits
    // or signals any more (the peer no longer touches this CTA's barriers or
    // TMEM), and an abort has set the flag of both CTAs; if one happened, the
    // producers' last TMA loads may still be landing, so both CTAs give them
    // 100 us before the memory they write is released.
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) spin_ns(100000);
        __syncthreads();
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace fp8fg
