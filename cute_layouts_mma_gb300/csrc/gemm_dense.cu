// BF16 and unscaled FP8 TN GEMM launchers (tcgen05 kind::f16 with BF16 operands,
// kind::f8f6f4 with E4M3 or E5M2 operands; fp32 accumulation, bf16 C and D).
#include <atomic>

#include "launch_kernel.cuh"

namespace tn {

// The same tiles as FP16: CTA pairs of 256 x 256 for M > 128, single CTAs of
// 128 x 256 otherwise.  A stage holds 128 bytes of K per row: 64 BF16 or 128 FP8
// elements.
using CfgBf16Pair = Config<KIND_BF16, 256, 6, 2, 64, 2, 2>;
using CfgBf16 = Config<KIND_BF16, 256, 4, 2, 64, 2, 1>;
using CfgE4m3Pair = Config<KIND_FP8_E4M3, 256, 6, 2, 64, 2, 2>;
using CfgE4m3 = Config<KIND_FP8_E4M3, 256, 4, 2, 64, 2, 1>;
using CfgE5m2Pair = Config<KIND_FP8_E5M2, 256, 6, 2, 64, 2, 2>;
using CfgE5m2 = Config<KIND_FP8_E5M2, 256, 4, 2, 64, 2, 1>;
// Skinny problems: 128-column tiles where they move fewer bytes per SM, 3 stages of two
// boxes of K (as FP16).
using CfgBf16N128 = Config<KIND_BF16, 128, 3, 2, 64, 2, 1, 4, 128, false, 0, 16, 2, 2>;
using CfgE4m3N128 = Config<KIND_FP8_E4M3, 128, 3, 2, 64, 2, 1, 4, 128, false, 0, 16, 2, 2>;
using CfgE5m2N128 = Config<KIND_FP8_E5M2, 128, 3, 2, 64, 2, 1, 4, 128, false, 0, 16, 2, 2>;
// Small problems (dispatch::use_small_tiles): 128 x 64 tiles on single CTAs, two boxes of K
// per stage (as FP16).
using CfgBf16N64 = Config<KIND_BF16, 64, 4, 2, 64, 1, 1, 4, 128, false, 0, 16, 2, 2>;
using CfgE4m3N64 = Config<KIND_FP8_E4M3, 64, 4, 2, 64, 1, 1, 4, 128, false, 0, 16, 2, 2>;
using CfgE5m2N64 = Config<KIND_FP8_E5M2, 64, 4, 2, 64, 1, 1, 4, 128, false, 0, 16, 2, 2>;

// Device-side record of an abandoned launch (a bounded wait ran out).
static __device__ unsigned int g_err_dense;

namespace {

std::atomic<uintptr_t> g_err_addr[kMaxDevices];

unsigned int* err_word(int dev) { return device_symbol(g_err_dense, g_err_addr, dev); }

template <class Cfg>
gemm_status_t run(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                  cudaStream_t stream, int sms, int dev, int split = 1) {
    constexpr bool k16 = operands_16bit(Cfg::KIND);
    const CUtensorMapDataType in_type = k16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t row_bytes = static_cast<uint64_t>(K) * (k16 ? 2 : 1);
    CUtensorMap ta, tb, td, tc;
    // A [M][K], 128-row boxes; B [N][K], BN/PAIR-row boxes; 128 bytes of K per box
    // (64 BF16 or 128 FP8 elements).  D, C: bf16 [M][N] in 32-row x EPI_COLS boxes.
    if (!encode_tma_2d(&ta, in_type, A, K, M, row_bytes, Cfg::kKBoxCoord, Cfg::BM, 128) ||
        !encode_tma_2d(&tb, in_type, B, K, N, row_bytes, Cfg::kKBoxCoord, Cfg::BN_CTA, 128) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
                       Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    if (C == nullptr)
        tc = td;
    else if (!encode_tma_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, N * 2, Cfg::EPI_COLS, 32,
                            Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (err == nullptr) return GEMM_ERR_CUDA;
    Params p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>((M + Cfg::BM_TILE - 1) / Cfg::BM_TILE);
    p.num_n_blocks = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int>((K + Cfg::kKCoordPerStage - 1) / Cfg::kKCoordPerStage);
    p.C = C;
    p.D = D;
    p.err = err;
    p.split = split;
    if (launch_config<Cfg>(ta, tb, ta, tb, td, tc, p, sms, dev, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

namespace {

// The instance and cluster split dispatch::dense_plan picks (K coordinates per stage:
// 64 BF16 or 128 FP8 elements).
template <class Pair, class Single, class SingleN128, class SmallN64>
gemm_status_t dispatch_dense(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                             cudaStream_t stream, int sms, int dev) {
    static_assert(Pair::BN == dispatch::kDensePair256.bn && Pair::PAIR == 2 && Single::BN == dispatch::kDenseSingle256.bn &&
                      SingleN128::BN == dispatch::kDenseSingle128.bn && SmallN64::BN == dispatch::kDenseSingle64.bn,
                  "dense tile shapes of the dispatch rules");
    int res256[dispatch::kMaxSplit + 1], res128[dispatch::kMaxSplit + 1];
    if (split_capacity<Single>(sms, dev, res256) != cudaSuccess ||
        split_capacity<SingleN128>(sms, dev, res128) != cudaSuccess)
        return GEMM_ERR_CUDA;
    const dispatch::DensePlan plan = dispatch::dense_plan(M, N, K, Single::kKCoordPerStage, sms, res256, res128);
    switch (plan.choice) {
        case dispatch::DENSE_PAIR_256: return run<Pair>(M, N, K, A, B, C, D, stream, sms, dev);
        case dispatch::DENSE_SINGLE_64: return run<SmallN64>(M, N, K, A, B, C, D, stream, sms, dev);
        case dispatch::DENSE_SINGLE_128: return run<SingleN128>(M, N, K, A, B, C, D, stream, sms, dev, plan.split);
        default: return run<Single>(M, N, K, A, B, C, D, stream, sms, dev, plan.split);
    }
}

}  // namespace

gemm_status_t launch_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                               void* D, cudaStream_t stream, int sms, int dev) {
    return dispatch_dense<CfgBf16Pair, CfgBf16, CfgBf16N128, CfgBf16N64>(M, N, K, A, B, C, D, stream, sms, dev);
}

gemm_status_t launch_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                              void* D, int fmt, cudaStream_t stream, int sms, int dev) {
    if (fmt == GEMM_FP8_E4M3)
        return dispatch_dense<CfgE4m3Pair, CfgE4m3, CfgE4m3N128, CfgE4m3N64>(M, N, K, A, B, C, D, stream, sms, dev);
    return dispatch_dense<CfgE5m2Pair, CfgE5m2, CfgE5m2N128, CfgE5m2N64>(M, N, K, A, B, C, D, stream, sms, dev);
}

unsigned int read_clear_error_dense() { return read_clear_word(g_err_dense); }

}  // namespace tn
