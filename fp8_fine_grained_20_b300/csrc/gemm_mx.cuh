// gemm_mx.cuh -- block-scaled FP8 GEMM with power-of-two scales applied by the
// tensor core (tcgen05.mma ... kind::mxf8f6f4.block_scale, UE8M0 scales), for
// sm_103a.  Same operands and scale layouts as k_gemm_blockscaled, but every
// scale must be a power of two (the output of the *_pow2 quantizers).
//
// Method: the pages' scaling factors for some activations are integral powers
// of 2 (why-be.why-be.co.kr post 55081; sunipension.com post 314414).  With
// power-of-two scales the per-group scaling can be done inside the MMA: each
// 32-deep slice of K carries one 8-bit exponent scale per row of A and per
// column of B, so C = sum_kb sA[m,kb] sB(kb,n) sum_k A[m,k] B[n,k] is computed
// entirely by the tensor core, accumulating in FP32 tensor memory (which on
// this GPU keeps a 24-bit significand over any K), with no FP32 promotion on
// CUDA cores.  The 128-wide scale groups are replicated over their four
// 32-deep slices.
//
// Scale factors in tensor memory (measured on B300 with an in-bounds layout
// probe, and the layout the block-scaling section of the PTX ISA describes):
// for scale_vec::1X the A scale of row m is read from TMEM lane m, column
// base + m/32, byte sf_id; the B scale of column n from lane 32 (m/32) + n%32
// (the quadrant of the output row), column base + n/32, byte sf_id.
// tcgen05.cp .32x128b.warpx4 copies a 512-byte shared-memory atom -- 32
// chunks of 16 bytes, chunk i holding rows i, i+32, i+64, i+96 as four 32-bit
// words -- into four TMEM columns of every lane quadrant (lane L receives
// chunk L % 32), which is exactly that layout.  With a CTA pair, each CTA's
// TMEM receives its own shared memory's atom and holds the A scales of its own
// 128 rows and the B scales of all 256 columns.  A 32-bit word has four
// bytes and sf_id picks one, so one word carries the scales of four
// consecutive K-blocks: one set of copies serves four K-blocks.
//
// Warp roles (384 threads, clusters of 2 CTAs, persistent over 256 x 256 pair
// tiles in the grouped raster of gemm.cuh):
//   warp 0 (both CTAs): TMA producer, as in k_gemm_blockscaled, MX_STAGES-deep,
//     with the L2 prefetch of the next tile's first K-blocks;
//   warp 1 (even CTA): MMA issuer -- per group of four K-blocks, three
//     tcgen05.cp (A atom, two B atoms) into one of SF_SLOTS TMEM scale slots,
//     then per K-block four block-scaled MMAs (K = 32 each, sf_id = the
//     K-block's byte) into the single 256-column accumulator and one commit
//     that frees the smem stage; after the group's last K-block a commit that
//     frees the scale slot; after the tile's last K-block a commit that hands
//     the accumulator to the epilogue;
//   warp 3 (both CTAs): scale copier -- cp.async of the fp32 scales of this
//     CTA's A rows and of the tile's B columns, SF_RAW groups ahead;
//   warp 2 (both CTAs): scale converter -- UE8M0 bytes of those scales (the
//     fp32 exponent field; any non-power-of-two scale sets
//     FP8_ERR_DEVICE_SCALES) written as the atoms of a shared-memory slot,
//     published two groups per release arrive;
//   warps 4-11 (both CTAs): epilogue -- load the whole 128 x 256 FP32
//     accumulator of this CTA into registers (128 values per thread), release
//     it to the MMA issuer at once, then round to bf16 into swizzled staging
//     tiles and store them with TMA, overlapping the next tile's MMAs.
#pragma once

#include "gemm.cuh"

namespace fp8fg {
namespace gemm {

constexpr int MX_STAGES = 5;
constexpr int SF_SLOTS = 6;                 // groups of four K-blocks in flight (TMEM scale slots)
constexpr int KB_PER_SF = 4;                // K-blocks per scale word (bytes 0..3)
constexpr uint32_t SFA_BYTES = 512;         // one atom: 128 rows x 4 bytes
constexpr uint32_t SFB_BYTES = 1024;        // two atoms: 256 columns x 4 bytes
constexpr uint32_t SF_TMEM_COL0 = 256;      // the accumulator uses columns 0..255
constexpr uint32_t SF_TMEM_SLOT = 16;       // A at +0..3, B at +8..15
constexpr int kStatusBadScale = 9;

constexpr size_t MX_OFF_A = 0;
constexpr size_t MX_OFF_B = MX_OFF_A + MX_STAGES * A_BYTES;
constexpr size_t MX_OFF_C = MX_OFF_B + MX_STAGES * B_BYTES;   // per epilogue warp: a 32 x 64 bf16 staging tile
constexpr size_t MX_OFF_SFA = MX_OFF_C + PROMO_WARPS * C_STAGE_BYTES;
constexpr size_t MX_OFF_SFB = MX_OFF_SFA + SF_SLOTS * SFA_BYTES;
constexpr size_t MX_OFF_BAR = MX_OFF_SFB + SF_SLOTS * SFB_BYTES;
constexpr int MX_N_BARS = 2 * MX_STAGES + 2 * SF_SLOTS + 3 + 2 * 4;   // + rawfull / rawempty of the SF_RAW ring
constexpr size_t MX_OFF_MISC = MX_OFF_BAR + MX_N_BARS * sizeof(uint64_t);
constexpr size_t MX_OFF_GOFF = MX_OFF_MISC + 16;

// The fp32 scales are copied (cp.async, warp 3) into a ring of SF_RAW groups,
// so that several groups' global loads are in flight while the MMAs consume
// the current one; warp 2 converts each group to UE8M0 atoms.  A slot holds
// A as [K-block b][128 rows] and per-column B as [b][256 columns], so that
// scales contiguous in global memory (stride 1 along the rows or columns, the
// usual layout) are copied four at a time; per-block B scales are held as
// [value 4 h + b][lane] (h the column half, every lane its own copy).  The
// ring follows the expert offsets of the grouped kernel.
constexpr int SF_RAW = 4;
static_assert(MX_N_BARS == 2 * MX_STAGES + 2 * SF_SLOTS + 3 + 2 * SF_RAW, "barrier count");
constexpr uint32_t RAWA_BYTES = 16 * 32 * 4;
__host__ __device__ constexpr uint32_t mx_rawb_bytes(int sbk) { return (sbk == SB_BLOCK ? 8u : 32u) * 32u * 4u; }
__host__ __device__ constexpr size_t mx_off_rawa(bool grouped) {
    return (MX_OFF_GOFF + (grouped ? 2 * (MAX_GROUPS + 1) * sizeof(int) : 0) + 127) & ~size_t(127);
}
__host__ __device__ constexpr size_t mx_off_rawb(bool grouped) { return mx_off_rawa(grouped) + SF_RAW * RAWA_BYTES; }
// dynamic shared memory of a launch (1024 bytes of alignment slack included)
__host__ __device__ constexpr size_t mx_smem(int sbk, bool grouped) {
    return 1024 + mx_off_rawb(grouped) + SF_RAW * mx_rawb_bytes(sbk);
}
static_assert(SF_TMEM_COL0 + SF_SLOTS * SF_TMEM_SLOT <= TMEM_COLS, "tensor memory budget");
static_assert(mx_smem(SB_COL, false) <= 227 * 1024 && mx_smem(SB_BLOCK, true) <= 227 * 1024, "shared memory budget");

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4 with E4M3 A and B,
// both K-major, UE8M0 scales: B scale byte (bits 4-5), A and B formats E4M3 (0),
// N >> 3 at bits 17-22, scale type UE8M0 (bit 23), M >> 4 at bits 24-28, A
// scale byte (bits 29-30).
__host__ __device__ constexpr uint32_t idesc_mx_e4m3(int m, int n, uint32_t sf_id) {
    return (sf_id << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(m >> 4) << 24) | (sf_id << 29);
}

// Shared-memory descriptor of a tcgen05.cp source without swizzling: rows of
// 16 bytes, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(16u >> 4) << 16;
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;
}

__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem of both CTAs] (+)= (A * sA)[smem] * (B * sB)[smem]^T with the A and B
// scales read from tensor memory at sfa / sfb; issued by one thread of the
// even CTA.
__device__ __forceinline__ void umma_mx_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
        : "memory");
}

// UE8M0 byte of a power-of-two fp32 scale: its exponent field (2^-127, the
// fp32 subnormal 0x00400000, and 0 both give byte 0).  Anything else is not a
// valid scale for this kernel and is reported.
__device__ __forceinline__ uint32_t ue8m0_of(float s, bool& bad) {
    const uint32_t u = __float_as_uint(s);
    const uint32_t e = u >> 23;
    bad |= !(((u & 0x7FFFFFu) == 0u && e < 255u) || u == 0x00400000u);
    return e & 0xFFu;
}

// The UE8M0 bytes of four scales v[0], v[stride], v[2 stride], v[3 stride]
// (four K-blocks) as one word, byte b from v[b stride].  Instead of checking
// each value, mm collects the mantissa bits and hh the sign bits and the carry
// of adding one to the exponent (set for an exponent of 255): both stay zero
// for zero and normal powers of two, and the caller runs ue8m0_of on the
// values whenever either is not (which also admits 2^-127, 0x00400000).
__device__ __forceinline__ uint32_t ue8m0_word(const float* v, int stride, uint32_t& mm, uint32_t& hh) {
    uint32_t t[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t u = __float_as_uint(v[b * stride]);
        mm |= u & 0x7FFFFFu;
        hh |= u | (u + 0x800000u);
        t[b] = u << 1;   // exponent in the top byte
    }
    return __byte_perm(__byte_perm(t[0], t[1], 0x0073), __byte_perm(t[2], t[3], 0x0073), 0x5410);
}

// Arrive once on an mbarrier of this CTA or the peer with cluster-scope
// release, so that this thread's earlier shared-memory writes are visible to
// a tcgen05.cp the peer issues after its acquire.
__device__ __forceinline__ void mbar_arrive_cluster_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// The same with no ordering of this thread's earlier writes (see the
// publication protocol of the scale converter).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier of this CTA with CTA-scope release, or relaxed.
__device__ __forceinline__ void mbar_arrive_release_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_relaxed_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Launch: clusters of 2 CTAs along x, THREADS threads, mx_smem(SBK, GROUPED)
// bytes of dynamic shared memory, one CTA per SM.
template <int SBK, bool GROUPED, int MX_GROUP = GROUPED ? 2 : GROUP_PM>
__global__ void __launch_bounds__(THREADS, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const Args p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sm_a = base + MX_OFF_A;
    uint8_t* sm_b = base + MX_OFF_B;
    uint8_t* sm_c = base + MX_OFF_C;
    uint8_t* sm_sfa = base + MX_OFF_SFA;
    uint8_t* sm_sfb = base + MX_OFF_SFB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + MX_OFF_BAR);
    uint64_t* full = bars;                   // even CTA: TMA bytes of both CTAs
    uint64_t* done = full + MX_STAGES;       // both: the stage's MMAs completed (stage free)
    uint64_t* sfull = done + MX_STAGES;      // even CTA: both CTAs' scale atoms of a slot written
    uint64_t* sfdone = sfull + SF_SLOTS;     // both: the slot's copies and MMAs completed
    uint64_t* accfull = sfdone + SF_SLOTS;   // both: the tile's accumulator is complete
    uint64_t* accempty = accfull + 1;        // even CTA: both CTAs' epilogues hold the accumulator
    uint64_t* drain = accempty + 1;
    uint64_t* rawfull = drain + 1;           // this CTA: the copier's fp32 scales of a ring slot landed
    uint64_t* rawempty = rawfull + SF_RAW;   // this CTA: the converter has read a ring slot
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + MX_OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + MX_OFF_MISC + 4);
    int* groups_ok = reinterpret_cast<int*>(base + MX_OFF_MISC + 8);
    int* goff = reinterpret_cast<int*>(base + MX_OFF_GOFF);
    int* ppre = goff + (MAX_GROUPS + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < MX_STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&done[i], 1);
        }
        for (int i = 0; i < SF_SLOTS; ++i) {
            mbar_init(&sfull[i], 2);    // the converter warp of each CTA
            mbar_init(&sfdone[i], 1);
        }
        for (int i = 0; i < SF_RAW; ++i) {
            mbar_init(&rawfull[i], 32);   // one cp.async arrival per copier lane
            mbar_init(&rawempty[i], 1);
        }
        mbar_init(accfull, 1);
        mbar_init(accempty, 2 * PROMO_WARPS);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *groups_ok = 1;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
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
    cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int pair_rows = GROUPED ? ppre[p.G] : (p.m_blocks + 1) / 2;
    const int num_tiles = (*groups_ok) ? pair_rows * p.n_blocks : 0;
    const int pair = static_cast<int>(cluster_id_x());
    const int n_pairs = static_cast<int>(n_clusters_x());
    const int groups_per_tile = (p.k_blocks + KB_PER_SF - 1) / KB_PER_SF;

    // register split: 4 warps x 80 + 8 warps x 208 = 63,488 <= 384 x 168 launched
    if (warp < 4) {
      regs_decrease<80>();
      if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            bool ok = true;
            for (int t = pair; ok && t < num_tiles; t += n_pairs) {
                const Tile tl = tile_at<GROUPED, MX_GROUP>(t, p, pair_rows, goff, ppre);
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
                    if (kb == max(0, p.k_blocks - PREFETCH_AHEAD)) prefetch_next_tile<GROUPED, MX_GROUP>(
                        t + n_pairs, num_tiles, p, pair_rows, goff, ppre, rank, &tmA, &tmB);
                    if (++stage == MX_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer ----
        // The whole warp runs the loop, so every descriptor and address is
        // warp-uniform; one elected lane issues the tcgen05 instructions (the
        // same lane throughout, as a commit tracks only its own thread's MMAs).
        if (leader) {
            uint32_t stage = 0, phase = 0, grp = 0, tile_it = 0;
            bool ok = true;
            for (int t = pair; ok && t < num_tiles; t += n_pairs, ++tile_it) {
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    const uint32_t sslot = grp % SF_SLOTS, sph = (grp / SF_SLOTS) & 1u;
                    const uint32_t sfa_t = tmem + SF_TMEM_COL0 + sslot * SF_TMEM_SLOT;
                    const uint32_t sfb_t = sfa_t + 8;
                    const uint32_t j = static_cast<uint32_t>(kb % KB_PER_SF);
                    if (j == 0) {
                        // a new group: its scale atoms are in shared memory and the TMEM
                        // slot's previous group has finished its MMAs
                        const bool ready = mbar_spin<true>(&sfull[sslot], sph, abort_flag, p.wait_ns) &&
                                           mbar_spin(&sfdone[sslot], sph ^ 1u, abort_flag, p.wait_ns);
                        if (!__all_sync(0xffffffffu, ready)) {
                            if (lane == 0) signal_abort(abort_flag, peer);
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        if (elect_one_sync()) {
                            tc_cp_sf_pair(sfa_t, sdesc_sf_atom(smem_addr(sm_sfa + sslot * SFA_BYTES)));
                            tc_cp_sf_pair(sfb_t, sdesc_sf_atom(smem_addr(sm_sfb + sslot * SFB_BYTES)));
                            tc_cp_sf_pair(sfb_t + 4, sdesc_sf_atom(smem_addr(sm_sfb + sslot * SFB_BYTES + 512)));
                        }
                        __syncwarp();
                    }
                    const bool ready = (kb != 0 || mbar_spin(accempty, (tile_it & 1u) ^ 1u, abort_flag, p.wait_ns)) &&
                                       mbar_spin(&full[stage], phase, abort_flag, p.wait_ns);
                    if (!__all_sync(0xffffffffu, ready)) {
                        if (lane == 0) signal_abort(abort_flag, peer);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if (elect_one_sync()) {
                        const uint64_t ad = sdesc_kmajor_sw128(smem_addr(sm_a + stage * A_BYTES));
                        const uint64_t bd = sdesc_kmajor_sw128(smem_addr(sm_b + stage * B_BYTES));
                        const uint32_t idesc = idesc_mx_e4m3(PM, BN, j);
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_mx_pair(tmem, ad + 2u * k, bd + 2u * k, idesc, sfa_t, sfb_t,
                                         (kb > 0 || k > 0) ? 1u : 0u);
                        umma_commit_pair_mc(&done[stage], 0x3);
                        if (j == KB_PER_SF - 1 || kb == p.k_blocks - 1) umma_commit_pair_mc(&sfdone[sslot], 0x3);
                        if (kb == p.k_blocks - 1) umma_commit_pair_mc(accfull, 0x3);
                    }
                    __syncwarp();
                    if (j == KB_PER_SF - 1 || kb == p.k_blocks - 1) ++grp;
                    if (++stage == MX_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // every copy and MMA this warp issued completes before TMEM is released
            if (elect_one_sync()) umma_commit_pair_mc(drain, 0x1);
            __syncwarp();
            mbar_wait(drain, 0, nullptr, ok ? kWaitTimeoutNs : kDrainTimeoutNs);
        }
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------- scale copier and converter ----
        // Group q of this pair's scale sequence (tile by tile, four K-blocks per
        // group) goes through ring slot q % SF_RAW: warp 3 copies this CTA's A
        // scales (its 128 rows) and the tile's B scales (256 columns) with
        // cp.async, completing on rawfull; warp 2 converts them to the UE8M0
        // atoms of TMEM scale slot q % SF_SLOTS.  The converter has no copies
        // of its own in flight, so its proxy fence before publishing an atom
        // does not wait for the prefetches.
        const int ra_stride = static_cast<int>(RAWA_BYTES / sizeof(float));
        const int rb_stride = static_cast<int>(mx_rawb_bytes(SBK) / sizeof(float));
        float* raw_a = reinterpret_cast<float*>(base + mx_off_rawa(GROUPED));
        float* raw_b = reinterpret_cast<float*>(base + mx_off_rawb(GROUPED));
        const int total_groups = (num_tiles > pair) ? ((num_tiles - 1 - pair) / n_pairs + 1) * groups_per_tile : 0;
        if (warp == 3) {
            // four scales per 16-byte copy where they are contiguous and aligned
            const bool vec_a = p.sa_sm == 1 && (p.sa_skb & 3) == 0 && (reinterpret_cast<uintptr_t>(p.sA) & 15u) == 0;
            const bool vec_b = SBK == SB_COL && p.sb_sn == 1 && (p.sb_skb & 3) == 0 && (p.sb_group_stride & 3) == 0 &&
                               (reinterpret_cast<uintptr_t>(p.sB) & 15u) == 0;
            int it_t = pair, it_g = 0;
            for (int q = 0; q < total_groups; ++q) {
                const int slot = q % SF_RAW;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&rawempty[slot], ((q / SF_RAW) & 1) ^ 1, abort_flag, p.wait_ns))) {
                    if (lane == 0) signal_abort(abort_flag, peer);
                    break;
                }
                const Tile tl = tile_at<GROUPED, MX_GROUP>(it_t, p, pair_rows, goff, ppre);
                const int kb0 = it_g * KB_PER_SF;
                const int nk = min(KB_PER_SF, p.k_blocks - kb0);
                const int r0 = tl.row0 + static_cast<int>(rank) * BM;
                float* da = raw_a + slot * ra_stride;   // [b][128 rows]
                if (vec_a) {
                    const int row = r0 + 4 * lane;      // rows row .. row + 3 (all in or all out: M % 128 == 0)
#pragma unroll
                    for (int b = 0; b < KB_PER_SF; ++b) {
                        float* dst = da + 128 * b + 4 * lane;
                        if (row < p.M && b < nk) {
                            cp_async_16(dst, p.sA + row + static_cast<int64_t>(kb0 + b) * p.sa_skb);
                        } else {
#pragma unroll
                            for (int e = 0; e < 4; ++e) cp_async_4(dst + e, &g_zero_scale);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = r0 + lane + 32 * i;
#pragma unroll
                        for (int b = 0; b < KB_PER_SF; ++b) {
                            const float* src = (row < p.M && b < nk) ? p.sA + static_cast<int64_t>(row) * p.sa_sm +
                                                                           static_cast<int64_t>(kb0 + b) * p.sa_skb
                                                                     : &g_zero_scale;
                            cp_async_4(da + 128 * b + lane + 32 * i, src);
                        }
                    }
                }
                const float* sb_base = p.sB + static_cast<int64_t>(tl.g) * p.sb_group_stride;
                float* db = raw_b + slot * rb_stride;
                if constexpr (SBK == SB_BLOCK) {
                    // [value 4 h + b][lane]: every lane copies the two block scales
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = tl.nb * (BN / 128) + h;
#pragma unroll
                        for (int b = 0; b < KB_PER_SF; ++b) {
                            const float* src = (c < p.sb_cols && b < nk)
                                                   ? sb_base + static_cast<int64_t>(kb0 + b) * p.sb_skb +
                                                         static_cast<int64_t>(c) * p.sb_sn
                                                   : &g_zero_scale;
                            cp_async_4(db + 32 * (4 * h + b) + lane, src);
                        }
                    }
                } else if (vec_b) {
                    // [b][256 columns], four columns per copy (all in or all out: N % 128 == 0)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = tl.nb * BN + 128 * h + 4 * lane;
#pragma unroll
                        for (int b = 0; b < KB_PER_SF; ++b) {
                            float* dst = db + 256 * b + 128 * h + 4 * lane;
                            if (c < p.sb_cols && b < nk) {
                                cp_async_16(dst, sb_base + static_cast<int64_t>(kb0 + b) * p.sb_skb + c);
                            } else {
#pragma unroll
                                for (int e = 0; e < 4; ++e) cp_async_4(dst + e, &g_zero_scale);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int c = tl.nb * BN + 128 * h + lane + 32 * i;
#pragma unroll
                            for (int b = 0; b < KB_PER_SF; ++b) {
                                const float* src = (c < p.sb_cols && b < nk)
                                                       ? sb_base + static_cast<int64_t>(kb0 + b) * p.sb_skb +
                                                             static_cast<int64_t>(c) * p.sb_sn
                                                       : &g_zero_scale;
                                cp_async_4(db + 256 * b + 128 * h + lane + 32 * i, src);
                            }
                        }
                }
                cp_async_arrive_noinc(&rawfull[slot]);
                if (++it_g == groups_per_tile) {
                    it_g = 0;
                    it_t += n_pairs;
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else {
            // Groups are published two at a time: one release arrive (cluster
            // scope from the odd CTA, whose atoms the even CTA's tcgen05.cp
            // reads; CTA scope from the even CTA) orders the atoms of both, and
            // the second group's arrive is relaxed.  The MMA warp acquires the
            // first group's barrier before it waits on the second, so the second
            // group's atoms are visible to it as well.  A cluster-scope release
            // costs about 300 cycles on an idle B300 and over 1000 under this
            // kernel's memory traffic; one per group made the converter slower
            // than the MMAs.
            bool bad = false;
            const uint32_t sfull_even = mapa_shared(smem_addr(&sfull[0]), 0);
            bool ok = true;
            for (int q0 = 0; ok && q0 < total_groups; q0 += 2) {
                const int nq = min(2, total_groups - q0);
                uint32_t wa[2][4], wb[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (u >= nq) break;
                    const int q = q0 + u;
                    const int slot = q % SF_RAW;
                    if (!__all_sync(0xffffffffu, mbar_wait(&rawfull[slot], (q / SF_RAW) & 1, abort_flag, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    const float* va = raw_a + slot * ra_stride + lane;   // rows lane + 32 k of K-block b at 128 b + 32 k
                    const float* vb = raw_b + slot * rb_stride + lane;
                    uint32_t mm = 0, hh = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) wa[u][k] = ue8m0_word(va + 32 * k, 128, mm, hh);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (SBK == SB_BLOCK)   // word h = k of [value 4 h + b][lane]
                            wb[u][k] = (k < 2) ? ue8m0_word(vb + 128 * k, 32, mm, hh) : 0u;
                        else                   // columns 128 (k / 4) + lane + 32 (k % 4) of [b][256]
                            wb[u][k] = ue8m0_word(vb + 128 * (k >> 2) + 32 * (k & 3), 256, mm, hh);
                    }
                    if ((mm | (hh & 0x80000000u)) != 0u) {   // not all zero or normal powers of two: check each
#pragma unroll
                        for (int k = 0; k < 4; ++k)
#pragma unroll
                            for (int b = 0; b < KB_PER_SF; ++b) ue8m0_of(va[128 * b + 32 * k], bad);
#pragma unroll
                        for (int k = 0; k < (SBK == SB_BLOCK ? 2 : 8); ++k)
#pragma unroll
                            for (int b = 0; b < KB_PER_SF; ++b)
                                ue8m0_of(SBK == SB_BLOCK ? vb[32 * (4 * k + b)] : vb[256 * b + 128 * (k >> 2) + 32 * (k & 3)],
                                         bad);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&rawempty[slot]);   // the values are in registers
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (!ok || u >= nq) break;
                    const uint32_t q = static_cast<uint32_t>(q0 + u);
                    const uint32_t sslot = q % SF_SLOTS, sph = (q / SF_SLOTS) & 1u;
                    if (!__all_sync(0xffffffffu, mbar_wait(&sfdone[sslot], sph ^ 1u, abort_flag, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    if (FP8_IN_BOUNDS(sslot < SF_SLOTS)) {
                        sts_v4(sm_sfa + sslot * SFA_BYTES + 16 * lane, make_uint4(wa[u][0], wa[u][1], wa[u][2], wa[u][3]));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint4 w4 = (SBK == SB_BLOCK)
                                                 ? make_uint4(wb[u][h], wb[u][h], wb[u][h], wb[u][h])
                                                 : make_uint4(wb[u][4 * h], wb[u][4 * h + 1], wb[u][4 * h + 2], wb[u][4 * h + 3]);
                            sts_v4(sm_sfb + sslot * SFB_BYTES + 512 * h + 16 * lane, w4);
                        }
                    }
                }
                if (!ok) {
                    if (lane == 0) signal_abort(abort_flag, peer);
                    break;
                }
                fence_proxy_async_shared();   // the atoms are read by tcgen05.cp (async proxy)
                __syncwarp();
                if (lane == 0) {
                    const uint32_t s0 = static_cast<uint32_t>(q0) % SF_SLOTS;
                    if (rank == 0) {
                        mbar_arrive_release_cta(&sfull[s0]);
                        if (nq == 2) mbar_arrive_relaxed_cta(&sfull[(s0 + 1) % SF_SLOTS]);
                    } else {
                        mbar_arrive_cluster_release(sfull_even + s0 * sizeof(uint64_t));
                        if (nq == 2) mbar_arrive_cluster_relaxed(sfull_even + ((s0 + 1) % SF_SLOTS) * sizeof(uint64_t));
                    }
                }
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) record_status(kStatusBadScale);
        }
      }
    } else {
        regs_increase<208>();
        // ------------------------------------------------------ epilogue ----
        const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
        const int half = (warp - 4) >> 2;       // output columns half*128 .. +127
        uint32_t tile_it = 0;
        for (int t = pair; t < num_tiles; t += n_pairs, ++tile_it) {
            // the tile's place, found while no accumulator values are live
            const Tile tl = tile_at<GROUPED, MX_GROUP>(t, p, pair_rows, goff, ppre);
            const int n0 = tl.nb * BN + half * 128;
            if (!__all_sync(0xffffffffu, mbar_wait(accfull, tile_it & 1u, abort_flag, p.wait_ns))) {
                if (lane == 0) signal_abort(abort_flag, peer);
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld_32cols(taddr + 0, r0);
            tmem_ld_32cols(taddr + 32, r1);
            tmem_wait_ld2(r0, r1);
            tmem_ld_32cols(taddr + 64, r2);
            tmem_ld_32cols(taddr + 96, r3);
            tmem_wait_ld2(r2, r3);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_addr(accempty), 0));   // the even CTA's
            // the warp's 32 rows x 128 columns as bf16 in two 32 x 64 TMA stores: each
            // lane writes its row into the warp's 128-byte-swizzled staging tile
            // (16-byte chunk j of row r at chunk j ^ (r % 8)), then lane 0 issues the
            // store; plain per-thread global stores here filled the memory pipeline
            // that the MMA warp's barrier tests and copies also go through
            uint8_t* stg = sm_c + (warp - 4) * C_STAGE_BYTES;
            const int wrow0 = tl.row0 + static_cast<int>(rank) * BM + quarter * 32;
            const bool wstore = wrow0 + 32 <= tl.row_end;   // 128-row blocks: whole warps are in or out
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t(&ra)[32] = h ? r2 : r0;
                const uint32_t(&rb)[32] = h ? r3 : r1;
                if (lane == 0) bulk_wait_read_all();   // the previous store has read the tile
                __syncwarp();
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint32_t(&r)[32] = (jj < 4) ? ra : rb;
                    const int o = 8 * (jj & 3);
                    if (FP8_IN_BOUNDS(lane * 128 + ((jj ^ (lane & 7)) << 4) + 16 <= static_cast<int>(C_STAGE_BYTES)))
                        sts_v4(stg + lane * 128 + ((jj ^ (lane & 7)) << 4),
                               make_uint4(pack_bf16x2(__uint_as_float(r[o + 0]), __uint_as_float(r[o + 1])),
                                          pack_bf16x2(__uint_as_float(r[o + 2]), __uint_as_float(r[o + 3])),
                                          pack_bf16x2(__uint_as_float(r[o + 4]), __uint_as_float(r[o + 5])),
                                          pack_bf16x2(__uint_as_float(r[o + 6]), __uint_as_float(r[o + 7]))));
                }
                fence_proxy_async_shared();
                __syncwarp();
                // N is a multiple of 128: a 64-column box is in or out as a whole
                if (lane == 0 && wstore && n0 + 64 * h < p.N && FP8_IN_BOUNDS(n0 + 64 * h + 64 <= p.N)) {
                    tma_store_2d(&tmC, stg, n0 + 64 * h, wrow0);
                    bulk_commit_group();
                }
            }
        }
        // every store of this warp has completed before its staging tile is released
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    // Teardown.  After the first cluster barrier no thread of either CTA waits
    // or signals any more, and an abort has set the flag of both CTAs; if one
    // happened, the producers' last TMA loads may still be landing, so both
    // CTAs give them 100 us before the memory they write is released.
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
