// fp8fg.cu -- the C ABI of libfp8fg.so (declared in include/fp8fg.h):
// argument validation, tensor-map encoding and kernel launches on the
// caller's stream.  The library allocates no device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/fp8fg.h"
#include "gemm.cuh"
#include "gemm_mx.cuh"
#include "probe.cuh"
#include "quant.cuh"
#include "swiglu.cuh"

namespace {

using namespace fp8fg;

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int sm_count(int dev) {
    static int cache[kMaxDevices] = {0};
    if (dev < 0 || dev >= kMaxDevices) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

fp8_status_t launch_status() {
    return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// Resident CTAs per SM of a kernel (cached per device).
template <typename K>
int blocks_per_sm(K kernel, int threads, int dev, int* cache) {
    if (dev < 0 || dev >= kMaxDevices) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// -------------------------------------------------------- tensor maps ----

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major [rows][cols] uint8 matrix (row stride ld bytes) read in boxes of
// box_rows x 128 bytes with 128-byte swizzling; rows beyond `rows` read as 0.
bool make_kmajor_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 [rows][cols] output (row stride ld elements) written by 32-row x
// 64-column TMA stores from 128-byte-swizzled staging tiles.
bool make_c_store_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
    const cuuint32_t box[2] = {64u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tiled map without swizzling over a row-major tensor of `rank` dims (dims[0]
// innermost, strides in bytes for dims 1..rank-1), boxes of box[] elements.
bool make_plain_map(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, int rank, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Dynamic shared memory above 48 KB, once per kernel and device.
template <typename K>
bool allow_smem(K kernel, size_t bytes, int dev, int* done) {
    if (dev < 0 || dev >= kMaxDevices) return false;
    if (!done[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) !=
            cudaSuccess)
            return false;
        done[dev] = 1;
    }
    return true;
}

// Launch state of one CTA-pair GEMM kernel, per device: the shared-memory
// attribute is set once and the number of co-resident pairs is cached.
struct PairLaunch {
    int ready[kMaxDevices];
    int max_pairs[kMaxDevices];
};

// Configure a persistent CTA-pair launch of `kernel` (clusters of 2 along x):
// one pair per co-resident cluster slot, never more pairs than tiles.
template <typename KernelT>
fp8_status_t pair_config(KernelT kernel, size_t smem, PairLaunch& st, const gemm::Args& args, bool grouped,
                         cudaStream_t stream, cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) return FP8_ERR_CUDA;
    cfg = cudaLaunchConfig_t{};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(gemm::THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!st.ready[dev]) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return FP8_ERR_DEVICE;
        int n = 0;
        cfg.gridDim = dim3(2 * static_cast<unsigned>(sm_count(dev)), 1, 1);
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return FP8_ERR_DEVICE;
        }
        st.max_pairs[dev] = n;
        st.ready[dev] = 1;
    }
    // the grouped pair-row count is known only on the device: bound it by the
    // padded rows, each expert adding at most one half-empty pair-row
    int64_t pair_rows = (args.m_blocks + 1) / 2;
    if (grouped) pair_rows = std::min<int64_t>(args.m_blocks, (args.m_blocks + args.G + 1) / 2);
    const int64_t tiles = pair_rows * args.n_blocks;
    const int64_t pairs = std::max<int64_t>(1, std::min<int64_t>(tiles, st.max_pairs[dev]));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    return FP8_OK;
}

template <int SBK, bool GROUPED, bool QOUT = false>
fp8_status_t launch_gemm(const uint8_t* A, int64_t lda, int64_t a_rows, const uint8_t* B, int64_t ldb,
                         int64_t b_rows, const gemm::Args& args, cudaStream_t stream,
                         const gemm::QArgs& qargs = gemm::QArgs{}) {
    static PairLaunch st = {};
    auto kernel = gemm::k_gemm_blockscaled<SBK, GROUPED, QOUT>;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    const fp8_status_t rc =
        pair_config(kernel, GROUPED ? gemm::SMEM_GROUPED : gemm::SMEM_PLAIN, st, args, GROUPED, stream, cfg, attr);
    if (rc != FP8_OK) return rc;
    CUtensorMap tmA, tmB, tmC;
    if (!make_kmajor_map(&tmA, A, a_rows, args.K, lda, gemm::BM)) return FP8_ERR_CUDA;
    if (!make_kmajor_map(&tmB, B, b_rows, args.K, ldb, gemm::BNH)) return FP8_ERR_CUDA;
    memset(&tmC, 0, sizeof(tmC));
    if (!QOUT && !make_c_store_map(&tmC, args.C, args.M, args.N, args.ldc))
        return FP8_ERR_CUDA;
    if (cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, args, qargs) != cudaSuccess) {
        cudaGetLastError();
        return FP8_ERR_CUDA;
    }
    return launch_status();
}

template <int SBK, bool GROUPED>
fp8_status_t launch_gemm_mx(const uint8_t* A, int64_t lda, int64_t a_rows, const uint8_t* B, int64_t ldb,
                            int64_t b_rows, const gemm::Args& args, cudaStream_t stream) {
    static PairLaunch st = {};
    auto kernel = gemm::k_gemm_mx<SBK, GROUPED>;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    const fp8_status_t rc = pair_config(kernel, gemm::mx_smem(SBK, GROUPED), st, args,
                                        GROUPED, stream, cfg, attr);
    if (rc != FP8_OK) return rc;
    CUtensorMap tmA, tmB, tmC;
    if (!make_kmajor_map(&tmA, A, a_rows, args.K, lda, gemm::BM)) return FP8_ERR_CUDA;
    if (!make_kmajor_map(&tmB, B, b_rows, args.K, ldb, gemm::BNH)) return FP8_ERR_CUDA;
    if (!make_c_store_map(&tmC, args.C, args.M, args.N, args.ldc)) return FP8_ERR_CUDA;
    if (cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, args) != cudaSuccess) {
        cudaGetLastError();
        return FP8_ERR_CUDA;
    }
    return launch_status();
}

// Self-test of the bounded device wait: one thread waits on an mbarrier that
// nothing arrives on; when the bound expires it records the timeout status.
__global__ void k_selftest_bounded_wait(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0, nullptr, timeout_ns)) record_status(kStatusTimeout);
    }
}

}  // namespace

extern "C" {

int fp8fg_version(void) { return 100; }

const char* fp8_status_string(fp8_status_t s) {
    switch (s) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_NULL: return "FP8_ERR_NULL: a required pointer is NULL";
        case FP8_ERR_ALIGN: return "FP8_ERR_ALIGN: pointer not 16-byte aligned or stride not a multiple of 16 bytes";
        case FP8_ERR_SHAPE: return "FP8_ERR_SHAPE: size negative, too large, or not a multiple of 128 where required";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA: a CUDA call failed";
        case FP8_ERR_DEVICE_TIMEOUT: return "FP8_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
        case FP8_ERR_ARG: return "FP8_ERR_ARG: invalid enum or stride argument";
        case FP8_ERR_DEVICE: return "FP8_ERR_DEVICE: unsupported device or resource limit";
        case FP8_ERR_DEVICE_GROUPS: return "FP8_ERR_DEVICE_GROUPS: invalid group offsets seen on the device";
        case FP8_ERR_DEVICE_SCALES: return "FP8_ERR_DEVICE_SCALES: a scale given to an _mx GEMM is not a power of two";
        case FP8_ERR_DEVICE_BOUNDS: return "FP8_ERR_DEVICE_BOUNDS: a device write fell outside its tile (bounds-checked build)";
    }
    return "unknown fp8fg status";
}

fp8_status_t fp8_get_device_status(void* stream, int32_t* out, int reset) {
    if (!out) return FP8_ERR_NULL;
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return FP8_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, fp8fg::g_fp8_device_status, sizeof(int)) != cudaSuccess) return FP8_ERR_CUDA;
    *out = v;
    if (reset) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(fp8fg::g_fp8_device_status, &zero, sizeof(int)) != cudaSuccess) return FP8_ERR_CUDA;
    }
    return FP8_OK;
}

fp8_status_t fp8_selftest_bounded_wait(uint64_t timeout_ns, void* stream) {
    if (timeout_ns == 0 || timeout_ns > 1000000000ull) return FP8_ERR_ARG;
    k_selftest_bounded_wait<<<1, 32, 0, as_stream(stream)>>>(timeout_ns);
    return launch_status();
}

fp8_status_t fp8_mma_accumulation_probe(const uint8_t* A, const uint8_t* B, int64_t K, float* D, void* stream) {
    if (K <= 0 || K % 128 || K > (int64_t(1) << 24)) return FP8_ERR_SHAPE;
    if (!A || !B || !D) return FP8_ERR_NULL;
    if (!aligned16(A) || !aligned16(B) || (reinterpret_cast<uintptr_t>(D) & 3u)) return FP8_ERR_ALIGN;
    static int smem_ok[kMaxDevices] = {0};
    const int dev = current_device();
    if (!allow_smem(probe::k_mma_accumulation_probe, probe::SMEM, dev, smem_ok)) return FP8_ERR_DEVICE;
    CUtensorMap tmA, tmB;
    if (!make_kmajor_map(&tmA, A, probe::BM, K, K, probe::BM)) return FP8_ERR_CUDA;
    if (!make_kmajor_map(&tmB, B, probe::BN, K, K, probe::BN)) return FP8_ERR_CUDA;
    probe::k_mma_accumulation_probe<<<1, 128, probe::SMEM, as_stream(stream)>>>(tmA, tmB,
                                                                              static_cast<int>(K / 128), D);
    return launch_status();
}

}  // extern "C"

namespace {

template <bool POW2>
fp8_status_t quant_act_entry(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                             float* s, int64_t s_stride_m, int64_t s_stride_kb, void* stream) {
    if (M < 0 || K < 0 || K % 128) return FP8_ERR_SHAPE;
    if (M == 0 || K == 0) return FP8_OK;
    if (!x || !q || !s) return FP8_ERR_NULL;
    if (ldx < K || ldq < K || s_stride_m < 0 || s_stride_kb < 0) return FP8_ERR_ARG;
    if (!aligned16(x) || !aligned16(q) || (ldx * 2) % 16 || ldq % 16 || (reinterpret_cast<uintptr_t>(s) & 3u))
        return FP8_ERR_ALIGN;
    const int64_t KB = K / 128;
    if (M > INT32_MAX || M * KB > (int64_t(1) << 40)) return FP8_ERR_SHAPE;
    static int occ[kMaxDevices] = {0};
    const int dev = current_device();
    const int sms = sm_count(dev);
    if (sms <= 0) return FP8_ERR_CUDA;
    constexpr int UNROLL = 2;
    auto kernel = k_quant_act_1x128<UNROLL, POW2>;
    const int per_sm = blocks_per_sm(kernel, 256, dev, occ);
    const int64_t slots = ceil_div(M * KB, 8);           // a warp quantizes 8 groups per slot
    const int64_t want = ceil_div(slots, 8 * UNROLL);    // 8 warps per CTA, UNROLL slots each
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    kernel<<<grid, 256, 0, as_stream(stream)>>>(x, static_cast<int>(M), static_cast<int>(KB), ldx, q, ldq, s,
                                               s_stride_m, s_stride_kb);
    return launch_status();
}

template <bool POW2>
fp8_status_t quant_w_entry(const uint16_t* w, int64_t G, int64_t K, int64_t N, int64_t ldw, int64_t w_batch_stride,
                           uint8_t* q, int64_t ldq, int64_t q_batch_stride, int q_layout, float* s,
                           int64_t s_stride_kb, int64_t s_stride_nb, int64_t s_batch_stride, void* stream) {
    if (G < 0 || K < 0 || N < 0 || K % 128 || N % 128) return FP8_ERR_SHAPE;
    if (q_layout != FP8_KMAJOR_NK && q_layout != FP8_ROWMAJOR_KN) return FP8_ERR_ARG;
    if (G == 0 || K == 0 || N == 0) return FP8_OK;
    if (!w || !q || !s) return FP8_ERR_NULL;
    const bool kmajor = q_layout == FP8_KMAJOR_NK;
    const int64_t q_min_ld = kmajor ? K : N;
    if (ldw < N || ldq < q_min_ld || s_stride_kb < 0 || s_stride_nb < 0) return FP8_ERR_ARG;
    if (G > 1 && (w_batch_stride < K * ldw || q_batch_stride < (kmajor ? N : K) * ldq || s_batch_stride < 0))
        return FP8_ERR_ARG;
    if (!aligned16(w) || !aligned16(q) || (ldw * 2) % 16 || ldq % 16 || (reinterpret_cast<uintptr_t>(s) & 3u) ||
        (G > 1 && ((w_batch_stride * 2) % 16 || q_batch_stride % 16)))
        return FP8_ERR_ALIGN;
    const int64_t KB = K / 128, NB = N / 128;
    if (G * KB * NB > INT32_MAX || K > INT32_MAX || N > INT32_MAX) return FP8_ERR_SHAPE;
    static int smem_ok[kMaxDevices] = {0};
    const int dev = current_device();
    const int sms = sm_count(dev);
    if (sms <= 0) return FP8_ERR_CUDA;
    if (!allow_smem(k_quant_w_128x128<POW2>, WQ_SMEM, dev, smem_ok)) return FP8_ERR_DEVICE;
    CUtensorMap tm;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(G)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldw * 2),
                                   static_cast<cuuint64_t>((G > 1 ? w_batch_stride : K * ldw) * 2)};
    const cuuint32_t box[3] = {128u, 128u, 1u};
    if (!make_plain_map(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, 3, dims, strides, box)) return FP8_ERR_CUDA;
    QuantWArgs a{};
    a.q = q;
    a.ldq = ldq;
    a.q_gstride = q_batch_stride;
    a.s = s;
    a.sskb = s_stride_kb;
    a.ssnb = s_stride_nb;
    a.s_gstride = s_batch_stride;
    a.G = static_cast<int>(G);
    a.KB = static_cast<int>(KB);
    a.NB = static_cast<int>(NB);
    a.kmajor = kmajor ? 1 : 0;
    const int64_t blocks = G * KB * NB;
    const int64_t cap = 2 * static_cast<int64_t>(sms);
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    k_quant_w_128x128<POW2><<<grid, WQ_THREADS, WQ_SMEM, as_stream(stream)>>>(tm, a);
    return launch_status();
}

template <bool POW2>
fp8_status_t requant_entry(const uint8_t* q, int64_t M, int64_t K, int64_t ldq, const float* s, int64_t s_stride_m,
                           int64_t s_stride_kb, uint8_t* qT, int64_t ldqT, float* sT, int64_t sT_stride_k,
                           int64_t sT_stride_mb, void* stream) {
    if (M < 0 || K < 0 || M % 128 || K % 128) return FP8_ERR_SHAPE;
    if (M == 0 || K == 0) return FP8_OK;
    if (!q || !s || !qT || !sT) return FP8_ERR_NULL;
    if (ldq < K || ldqT < M || s_stride_m < 0 || s_stride_kb < 0 || sT_stride_k < 0 || sT_stride_mb < 0)
        return FP8_ERR_ARG;
    if (!aligned16(q) || !aligned16(qT) || ldq % 16 || ldqT % 16 || (reinterpret_cast<uintptr_t>(s) & 3u) ||
        (reinterpret_cast<uintptr_t>(sT) & 3u))
        return FP8_ERR_ALIGN;
    const int64_t MB = M / 128, KB = K / 128;
    if (MB * KB > INT32_MAX || M > INT32_MAX || K > INT32_MAX) return FP8_ERR_SHAPE;
    static int smem_ok[kMaxDevices] = {0};
    const int dev = current_device();
    const int sms = sm_count(dev);
    if (sms <= 0) return FP8_ERR_CUDA;
    if (!allow_smem(k_requant_1x128_to_128x1<POW2>, RQ_SMEM, dev, smem_ok)) return FP8_ERR_DEVICE;
    CUtensorMap tm;   // 128 x 128 code blocks, 128-byte swizzle
    if (!make_kmajor_map(&tm, q, M, K, ldq, 128)) return FP8_ERR_CUDA;
    RequantArgs a{};
    a.s = s;
    a.ssm = s_stride_m;
    a.sskb = s_stride_kb;
    a.qT = qT;
    a.ldqT = ldqT;
    a.sT = sT;
    a.sTk = sT_stride_k;
    a.sTmb = sT_stride_mb;
    a.MB = static_cast<int>(MB);
    a.KB = static_cast<int>(KB);
    const int64_t cap = RQ_CTAS_PER_SM * static_cast<int64_t>(sms);
    const int grid = static_cast<int>(MB * KB < cap ? MB * KB : cap);
    k_requant_1x128_to_128x1<POW2><<<grid, RQ_THREADS, RQ_SMEM, as_stream(stream)>>>(tm, a);
    return launch_status();
}

}  // namespace

extern "C" {

fp8_status_t fp8_quant_act_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                 float* s, int64_t s_stride_m, int64_t s_stride_kb, void* stream) {
    return quant_act_entry<false>(x, M, K, ldx, q, ldq, s, s_stride_m, s_stride_kb, stream);
}

fp8_status_t fp8_swiglu_quant_1x128(const uint16_t* gate, int64_t ldg, const uint16_t* up, int64_t ldu, int64_t M,
                                    int64_t F, uint8_t* q, int64_t ldq, float* s, int64_t s_stride_m,
                                    int64_t s_stride_fb, uint16_t* y, int64_t ldy, void* stream) {
    if (M < 0 || F < 0 || F % 128) return FP8_ERR_SHAPE;
    if (M == 0 || F == 0) return FP8_OK;
    if (!gate || !up || !q || !s) return FP8_ERR_NULL;
    if (ldg < F || ldu < F || ldq < F || s_stride_m < 0 || s_stride_fb < 0 || (y && ldy < F)) return FP8_ERR_ARG;
    if (!aligned16(gate) || !aligned16(up) || !aligned16(q) || (ldg * 2) % 16 || (ldu * 2) % 16 || ldq % 16 ||
        (reinterpret_cast<uintptr_t>(s) & 3u) || (y && (!aligned16(y) || (ldy * 2) % 16)))
        return FP8_ERR_ALIGN;
    const int64_t FB = F / 128;
    if (M > INT32_MAX || M * FB > (int64_t(1) << 40)) return FP8_ERR_SHAPE;
    static int occ[kMaxDevices] = {0};
    const int dev = current_device();
    const int sms = sm_count(dev);
    if (sms <= 0) return FP8_ERR_CUDA;
    constexpr int UNROLL = 2;
    auto kernel = k_swiglu_quant_1x128<UNROLL>;
    const int per_sm = blocks_per_sm(kernel, 256, dev, occ);
    const int64_t slots = ceil_div(M * FB, 8);
    const int64_t want = ceil_div(slots, 8 * UNROLL);
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    const int grid = static_cast<int>(want < cap ? want : cap);
    SwigluArgs a{};
    a.g = gate;
    a.ldg = ldg;
    a.u = up;
    a.ldu = ldu;
    a.q = q;
    a.ldq = ldq;
    a.s = s;
    a.ssm = s_stride_m;
    a.ssfb = s_stride_fb;
    a.y = y;
    a.ldy = ldy;
    a.M = static_cast<int>(M);
    a.FB = static_cast<int>(FB);
    kernel<<<grid, 256, 0, as_stream(stream)>>>(a);
    return launch_status();
}

fp8_status_t fp8_quant_act_1x128_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                      int64_t ldq, float* s, int64_t s_stride_m, int64_t s_stride_kb, void* stream) {
    return quant_act_entry<true>(x, M, K, ldx, q, ldq, s, s_stride_m, s_stride_kb, stream);
}

fp8_status_t fp8_quant_w_128x128_batched(const uint16_t* w, int64_t G, int64_t K, int64_t N, int64_t ldw,
                                         int64_t w_batch_stride, uint8_t* q, int64_t ldq, int64_t q_batch_stride,
                                         int q_layout, float* s, int64_t s_stride_kb, int64_t s_stride_nb,
                                         int64_t s_batch_stride, void* stream) {
    return quant_w_entry<false>(w, G, K, N, ldw, w_batch_stride, q, ldq, q_batch_stride, q_layout, s, s_stride_kb,
                                s_stride_nb, s_batch_stride, stream);
}

fp8_status_t fp8_quant_w_128x128_batched_pow2(const uint16_t* w, int64_t G, int64_t K, int64_t N, int64_t ldw,
                                              int64_t w_batch_stride, uint8_t* q, int64_t ldq,
                                              int64_t q_batch_stride, int q_layout, float* s, int64_t s_stride_kb,
                                              int64_t s_stride_nb, int64_t s_batch_stride, void* stream) {
    return quant_w_entry<true>(w, G, K, N, ldw, w_batch_stride, q, ldq, q_batch_stride, q_layout, s, s_stride_kb,
                               s_stride_nb, s_batch_stride, stream);
}

fp8_status_t fp8_quant_w_128x128(const uint16_t* w, int64_t K, int64_t N, int64_t ldw, uint8_t* q, int64_t ldq,
                                 int q_layout, float* s, int64_t s_stride_kb, int64_t s_stride_nb, void* stream) {
    return quant_w_entry<false>(w, 1, K, N, ldw, 0, q, ldq, 0, q_layout, s, s_stride_kb, s_stride_nb, 0, stream);
}

fp8_status_t fp8_quant_w_128x128_pow2(const uint16_t* w, int64_t K, int64_t N, int64_t ldw, uint8_t* q,
                                      int64_t ldq, int q_layout, float* s, int64_t s_stride_kb,
                                      int64_t s_stride_nb, void* stream) {
    return quant_w_entry<true>(w, 1, K, N, ldw, 0, q, ldq, 0, q_layout, s, s_stride_kb, s_stride_nb, 0, stream);
}

fp8_status_t fp8_requant_1x128_to_128x1(const uint8_t* q, int64_t M, int64_t K, int64_t ldq, const float* s,
                                        int64_t s_stride_m, int64_t s_stride_kb, uint8_t* qT, int64_t ldqT,
                                        float* sT, int64_t sT_stride_k, int64_t sT_stride_mb, void* stream) {
    return requant_entry<false>(q, M, K, ldq, s, s_stride_m, s_stride_kb, qT, ldqT, sT, sT_stride_k, sT_stride_mb,
                                stream);
}

fp8_status_t fp8_requant_1x128_to_128x1_pow2(const uint8_t* q, int64_t M, int64_t K, int64_t ldq, const float* s,
                                             int64_t s_stride_m, int64_t s_stride_kb, uint8_t* qT, int64_t ldqT,
                                             float* sT, int64_t sT_stride_k, int64_t sT_stride_mb, void* stream) {
    return requant_entry<true>(q, M, K, ldq, s, s_stride_m, s_stride_kb, qT, ldqT, sT, sT_stride_k, sT_stride_mb,
                               stream);
}

}  // extern "C"

namespace {

// Which kernel a GEMM entry point runs.
enum class GemmKind { kPromote, kPromoteQuantOut, kMx };

// Validation and launch shared by the bf16 epilogue, the quantizing epilogue
// and the power-of-two (hardware-scaled) kernel.  wait_ns / withhold: the
// pipeline-wait bound and the test-only withholding of TMA loads.
fp8_status_t gemm_entry(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                        const uint8_t* B, int64_t ldb, const float* sB, int64_t sb_stride_kb, int64_t sb_stride_n,
                        int sb_kind, uint16_t* C, int64_t ldc, uint8_t* Cq, int64_t ldcq, float* sC,
                        int64_t sc_stride_m, int64_t sc_stride_nb, int64_t M, int64_t N, int64_t K, GemmKind kind,
                        cudaStream_t stream, uint64_t wait_ns = kWaitTimeoutNs, int withhold = 0) {
    const bool qout = kind == GemmKind::kPromoteQuantOut;
    if (sb_kind != FP8_SB_BLOCK128x128 && sb_kind != FP8_SB_COL128x1) return FP8_ERR_ARG;
    if (M < 0 || N < 0 || K < 0 || M % 128 || N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8_OK;
    if (K == 0) return FP8_ERR_SHAPE;
    if (!A || !sA || !B || !sB || (qout ? (!Cq || !sC) : !C)) return FP8_ERR_NULL;
    if (lda < K || ldb < K || sa_stride_m < 0 || sa_stride_kb < 0 || sb_stride_kb < 0 || sb_stride_n < 0)
        return FP8_ERR_ARG;
    if (qout ? (ldcq < N || sc_stride_m < 0 || sc_stride_nb < 0) : ldc < N) return FP8_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || lda % 16 || ldb % 16 || (reinterpret_cast<uintptr_t>(sA) & 3u) ||
        (reinterpret_cast<uintptr_t>(sB) & 3u))
        return FP8_ERR_ALIGN;
    if (qout ? (!aligned16(Cq) || ldcq % 16 || (reinterpret_cast<uintptr_t>(sC) & 3u))
             : (!aligned16(C) || (ldc * 2) % 16))
        return FP8_ERR_ALIGN;
    if (M / 128 * ceil_div(N, gemm::BN) > INT32_MAX || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
        return FP8_ERR_SHAPE;
    gemm::Args a{};
    a.sA = sA;
    a.sa_sm = sa_stride_m;
    a.sa_skb = sa_stride_kb;
    a.sB = sB;
    a.sb_skb = sb_stride_kb;
    a.sb_sn = sb_stride_n;
    a.sb_group_stride = 0;
    a.C = C;
    a.ldc = ldc;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.m_blocks = static_cast<int>(M / gemm::BM);
    a.n_blocks = static_cast<int>(ceil_div(N, gemm::BN));
    a.k_blocks = static_cast<int>(K / gemm::BK);
    a.sb_cols = static_cast<int>(sb_kind == FP8_SB_COL128x1 ? N : N / 128);
    a.offsets = nullptr;
    a.G = 0;
    a.wait_ns = wait_ns;
    a.withhold = withhold;
    if (kind == GemmKind::kMx) {
        if (sb_kind == FP8_SB_COL128x1) return launch_gemm_mx<gemm::SB_COL, false>(A, lda, M, B, ldb, N, a, stream);
        return launch_gemm_mx<gemm::SB_BLOCK, false>(A, lda, M, B, ldb, N, a, stream);
    }
    if (qout) {
        const gemm::QArgs q{Cq, ldcq, sC, sc_stride_m, sc_stride_nb};
        if (sb_kind == FP8_SB_COL128x1)
            return launch_gemm<gemm::SB_COL, false, true>(A, lda, M, B, ldb, N, a, stream, q);
        return launch_gemm<gemm::SB_BLOCK, false, true>(A, lda, M, B, ldb, N, a, stream, q);
    }
    if (sb_kind == FP8_SB_COL128x1) return launch_gemm<gemm::SB_COL, false>(A, lda, M, B, ldb, N, a, stream);
    return launch_gemm<gemm::SB_BLOCK, false>(A, lda, M, B, ldb, N, a, stream);
}

}  // namespace

extern "C" {

fp8_status_t fp8_gemm_blockscaled(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m,
                                  int64_t sa_stride_kb, const uint8_t* B, int64_t ldb, const float* sB,
                                  int64_t sb_stride_kb, int64_t sb_stride_n, int sb_kind, uint16_t* C, int64_t ldc,
                                  int64_t M, int64_t N, int64_t K, void* stream) {
    return gemm_entry(A, lda, sA, sa_stride_m, sa_stride_kb, B, ldb, sB, sb_stride_kb, sb_stride_n, sb_kind, C, ldc,
                      nullptr, 0, nullptr, 0, 0, M, N, K, GemmKind::kPromote, as_stream(stream));
}

fp8_status_t fp8_selftest_gemm_timeout(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                                       uint16_t* C, int64_t M, int64_t N, int64_t K, uint64_t wait_ns,
                                       void* stream) {
    if (wait_ns < 1000ull || wait_ns > 1000000000ull) return FP8_ERR_ARG;
    if (K < 256) return FP8_ERR_SHAPE;
    return gemm_entry(A, K, sA, 1, M, B, K, sB, N / 128, 1, FP8_SB_BLOCK128x128, C, N, nullptr, 0, nullptr, 0, 0, M,
                      N, K, GemmKind::kPromote, as_stream(stream), wait_ns, 1);
}

fp8_status_t fp8_gemm_blockscaled_mx(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m,
                                     int64_t sa_stride_kb, const uint8_t* B, int64_t ldb, const float* sB,
                                     int64_t sb_stride_kb, int64_t sb_stride_n, int sb_kind, uint16_t* C, int64_t ldc,
                                     int64_t M, int64_t N, int64_t K, void* stream) {
    return gemm_entry(A, lda, sA, sa_stride_m, sa_stride_kb, B, ldb, sB, sb_stride_kb, sb_stride_n, sb_kind, C, ldc,
                      nullptr, 0, nullptr, 0, 0, M, N, K, GemmKind::kMx, as_stream(stream));
}

fp8_status_t fp8_gemm_blockscaled_q1x128(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m,
                                         int64_t sa_stride_kb, const uint8_t* B, int64_t ldb, const float* sB,
                                         int64_t sb_stride_kb, int64_t sb_stride_n, int sb_kind, uint8_t* Cq,
                                         int64_t ldcq, float* sC, int64_t sc_stride_m, int64_t sc_stride_nb,
                                         int64_t M, int64_t N, int64_t K, void* stream) {
    return gemm_entry(A, lda, sA, sa_stride_m, sa_stride_kb, B, ldb, sB, sb_stride_kb, sb_stride_n, sb_kind, nullptr,
                      0, Cq, ldcq, sC, sc_stride_m, sc_stride_nb, M, N, K, GemmKind::kPromoteQuantOut,
                      as_stream(stream));
}

}  // extern "C"

namespace {

fp8_status_t grouped_entry(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m, int64_t sa_stride_kb,
                           const uint8_t* B, const float* sB, const int32_t* d_group_offsets, int G, int64_t M_total,
                           int64_t N, int64_t K, uint16_t* C, int64_t ldc, bool mx, cudaStream_t stream) {
    if (G < 1 || G > gemm::MAX_GROUPS) return FP8_ERR_ARG;
    if (M_total < 0 || N < 0 || K < 0 || M_total % 128 || N % 128 || K % 128) return FP8_ERR_SHAPE;
    if (M_total == 0 || N == 0) return FP8_OK;
    if (K == 0) return FP8_ERR_SHAPE;
    if (!A || !sA || !B || !sB || !C || !d_group_offsets) return FP8_ERR_NULL;
    if (lda < K || ldc < N || sa_stride_m < 0 || sa_stride_kb < 0) return FP8_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || lda % 16 || (ldc * 2) % 16 ||
        (reinterpret_cast<uintptr_t>(sA) & 3u) || (reinterpret_cast<uintptr_t>(sB) & 3u) ||
        (reinterpret_cast<uintptr_t>(d_group_offsets) & 3u))
        return FP8_ERR_ALIGN;
    if (static_cast<int64_t>(G) * N > INT32_MAX || M_total > INT32_MAX || K > INT32_MAX ||
        M_total / 128 * ceil_div(N, gemm::BN) > INT32_MAX)
        return FP8_ERR_SHAPE;
    const int64_t KB = K / 128, NB = N / 128;
    gemm::Args a{};
    a.sA = sA;
    a.sa_sm = sa_stride_m;
    a.sa_skb = sa_stride_kb;
    a.sB = sB;
    a.sb_skb = NB;
    a.sb_sn = 1;
    a.sb_group_stride = KB * NB;
    a.C = C;
    a.ldc = ldc;
    a.M = static_cast<int>(M_total);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.m_blocks = static_cast<int>(M_total / gemm::BM);
    a.n_blocks = static_cast<int>(ceil_div(N, gemm::BN));
    a.k_blocks = static_cast<int>(KB);
    a.sb_cols = static_cast<int>(NB);
    a.offsets = d_group_offsets;
    a.G = G;
    a.wait_ns = kWaitTimeoutNs;
    a.withhold = 0;
    if (mx)
        return launch_gemm_mx<gemm::SB_BLOCK, true>(A, lda, M_total, B, K, static_cast<int64_t>(G) * N, a, stream);
    return launch_gemm<gemm::SB_BLOCK, true>(A, lda, M_total, B, K, static_cast<int64_t>(G) * N, a, stream);
}

}  // namespace

extern "C" {

fp8_status_t fp8_grouped_gemm_blockscaled(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m,
                                          int64_t sa_stride_kb, const uint8_t* B, const float* sB,
                                          const int32_t* d_group_offsets, int G, int64_t M_total, int64_t N,
                                          int64_t K, uint16_t* C, int64_t ldc, void* stream) {
    return grouped_entry(A, lda, sA, sa_stride_m, sa_stride_kb, B, sB, d_group_offsets, G, M_total, N, K, C, ldc,
                         false, as_stream(stream));
}

fp8_status_t fp8_grouped_gemm_blockscaled_mx(const uint8_t* A, int64_t lda, const float* sA, int64_t sa_stride_m,
                                             int64_t sa_stride_kb, const uint8_t* B, const float* sB,
                                             const int32_t* d_group_offsets, int G, int64_t M_total, int64_t N,
                                             int64_t K, uint16_t* C, int64_t ldc, void* stream) {
    return grouped_entry(A, lda, sA, sa_stride_m, sa_stride_kb, B, sB, d_group_offsets, G, M_total, N, K, C, ldc,
                         true, as_stream(stream));
}

}  // extern "C"
