// FP16 TN GEMM launcher (tcgen05 kind::f16, fp32 or fp16 accumulation).
#include <atomic>

#include "launch_kernel.cuh"

namespace tn {

// CTA pairs (dispatch::use_pairs): 256 x 256 tiles, 6 stages of 64 K, two TMEM accumulators,
// epilogue staged in 32 x 64 chunks (128-byte rows), double-buffered.
using CfgF16Acc32Pair = Config<KIND_F16_ACC32, 256, 6, 2, 64, 2, 2>;
using CfgF16Acc16Pair = Config<KIND_F16_ACC16, 256, 6, 2, 64, 2, 2>;
// Single CTAs: 128 x 256 tiles, 4 stages.
using CfgF16Acc32 = Config<KIND_F16_ACC32, 256, 4, 2, 64, 2, 1>;
using CfgF16Acc16 = Config<KIND_F16_ACC16, 256, 4, 2, 64, 2, 1>;
// Skinny problems (fp32 accumulation): 128-column tiles where they move fewer bytes
// per SM than 128 x 256 ones (each instance with its own cluster split); 3 stages of
// two boxes of K (8 MMAs of N = 128 per barrier wait and commit).
using CfgF16N128 = Config<KIND_F16_ACC32, 128, 3, 2, 64, 2, 1, 4, 128, false, 0, 16, 2, 2>;
// Small problems (dispatch::use_small_tiles): 128 x 64 tiles on single CTAs, 4 stages of two
// 128-byte boxes of K per operand row (8 MMAs per barrier wait and commit: an N = 64 MMA is
// short, and with one box per stage the MMA thread's per-stage work bounded these launches),
// each epilogue warp staging its whole 32 x 64 slice.
using CfgF16N64 = Config<KIND_F16_ACC32, 64, 4, 2, 64, 1, 1, 4, 128, false, 0, 16, 2, 2>;
// Narrow K (fp32 accumulation): a whole K of at most 32 or 16 elements fits a 64- or
// 32-byte operand row, stored with the 64- or 32-byte swizzle; 2 or 1 MMAs per stage
// instead of 4 over zero-filled K.  These launches are bound by the C and D traffic,
// so the small stages leave room to stage a warp's whole 32 x 256 slice (C for the
// tile is fetched before its accumulator is ready).
using CfgF16K32Pair = Config<KIND_F16_ACC32, 256, 6, 2, 64, 4, 2, 4, 64>;
using CfgF16K32 = Config<KIND_F16_ACC32, 256, 6, 2, 64, 4, 1, 4, 64>;
using CfgF16K16Pair = Config<KIND_F16_ACC32, 256, 6, 2, 64, 4, 2, 4, 32>;
using CfgF16K16 = Config<KIND_F16_ACC32, 256, 6, 2, 64, 4, 1, 4, 32>;

// The instances behind dispatch::dense_choice.
static_assert(dispatch::kDensePair256.bn == CfgF16Acc32Pair::BN && dispatch::kDensePair256.pair == CfgF16Acc32Pair::PAIR &&
                  dispatch::kDenseSingle256.bn == CfgF16Acc32::BN && dispatch::kDenseSingle128.bn == CfgF16N128::BN &&
                  dispatch::kDenseSingle64.bn == CfgF16N64::BN && CfgF16Acc32::kStreamK && CfgF16N128::kStreamK,
              "dense tile shapes of the dispatch rules");

// Device-side record of an abandoned launch (a bounded wait ran out).
static __device__ unsigned int g_err_f16;

namespace {

std::atomic<uintptr_t> g_err_addr[kMaxDevices];

unsigned int* err_word(int dev) { return device_symbol(g_err_f16, g_err_addr, dev); }

// Tensor maps and kernel parameters of one FP16 launch.
template <class Cfg>
gemm_status_t prepare(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                      int dev, CUtensorMap& ta, CUtensorMap& tb, CUtensorMap& td, CUtensorMap& tc, Params& p) {
    p = Params{};
    // A: fp16 [M][K], 128-row boxes; B: fp16 [N][K], BN/PAIR-row boxes; kRowBytes
    // (128, or 64 / 32 for narrow K) of K per box, swizzled to match.  D: fp16 [M][N],
    // stored in 32-row x EPI_COLS boxes.
    constexpr int kKBox = Cfg::kKBoxCoord, kSw = Cfg::kRowBytes;
    if (!encode_tma_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, K * 2, kKBox, Cfg::BM, kSw) ||
        !encode_tma_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, K, N, K * 2, kKBox, Cfg::BN_CTA, kSw) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
                       Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    // C (if any): the same boxes as D, TMA-loaded into the epilogue staging buffers.
    if (C == nullptr)
        tc = td;
    else if (!encode_tma_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, C, N, M, N * 2, Cfg::EPI_COLS, 32, Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (err == nullptr) return GEMM_ERR_CUDA;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>((M + Cfg::BM_TILE - 1) / Cfg::BM_TILE);
    p.num_n_blocks = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int>((K + Cfg::kKCoordPerStage - 1) / Cfg::kKCoordPerStage);  // stages
    p.C = C;
    p.D = D;
    p.err = err;
    p.split = 1;
    return GEMM_OK;
}

template <class Cfg>
gemm_status_t run(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                  cudaStream_t stream, int sms, int dev, int split = 1) {
    CUtensorMap ta, tb, td, tc;
    Params p;
    const gemm_status_t st = prepare<Cfg>(M, N, K, A, B, C, D, dev, ta, tb, td, tc, p);
    if (st != GEMM_OK) return st;
    p.split = split;
    if (launch_config<Cfg>(ta, tb, ta, tb, td, tc, p, sms, dev, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

gemm_status_t launch_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                              void* D, int accum, cudaStream_t stream, int sms, int dev) {
    if (accum == GEMM_ACC_F32) {
        // narrow K: bound by the C and D traffic, pairs whenever M > 128
        if (K <= 16)
            return M > 128 ? run<CfgF16K16Pair>(M, N, K, A, B, C, D, stream, sms, dev)
                           : run<CfgF16K16>(M, N, K, A, B, C, D, stream, sms, dev);
        if (K <= 32)
            return M > 128 ? run<CfgF16K32Pair>(M, N, K, A, B, C, D, stream, sms, dev)
                           : run<CfgF16K32>(M, N, K, A, B, C, D, stream, sms, dev);
        int res256[dispatch::kMaxSplit + 1], res128[dispatch::kMaxSplit + 1];
        if (split_capacity<CfgF16Acc32>(sms, dev, res256) != cudaSuccess ||
            split_capacity<CfgF16N128>(sms, dev, res128) != cudaSuccess)
            return GEMM_ERR_CUDA;
        const dispatch::DensePlan plan = dispatch::dense_plan(M, N, K, 64, sms, res256, res128);
        switch (plan.choice) {
            case dispatch::DENSE_PAIR_256: return run<CfgF16Acc32Pair>(M, N, K, A, B, C, D, stream, sms, dev);
            case dispatch::DENSE_SINGLE_64: return run<CfgF16N64>(M, N, K, A, B, C, D, stream, sms, dev);
            case dispatch::DENSE_SINGLE_128:
                return run<CfgF16N128>(M, N, K, A, B, C, D, stream, sms, dev, plan.split);
            default: return run<CfgF16Acc32>(M, N, K, A, B, C, D, stream, sms, dev, plan.split);
        }
    }
    return dispatch::use_pairs(M, N, K, sms) ? run<CfgF16Acc16Pair>(M, N, K, A, B, C, D, stream, sms, dev)
                                          : run<CfgF16Acc16>(M, N, K, A, B, C, D, stream, sms, dev);
}

// ---------------------------------------------------------------- no-allocation variant
// Scratch of gemm_f16_noalloc, which keeps the stream-K schedule (units split the
// k-blocks of the last tiles and the finishing unit adds the others' fp32 partials
// from global memory): one fixed block per device, part of the loaded module, so the
// call never allocates.  20 MiB holds the partials (128 x 128 single-CTA tiles: 64 KB
// per SM) and flags of a device with up to 319 SMs (a 152-SM GB300 needs 9.5 MiB).
// Every call shares it: calls that overlap on the GPU would overwrite each other's
// partials and flags.
constexpr size_t kStaticScratchBytes = size_t(20) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

std::atomic<uintptr_t> g_static_scratch_addr[kMaxDevices];

// Device address of the fixed block on device `dev` (the current device), looked
// up once per device; null if the lookup fails.
void* static_scratch(int dev) {
    uintptr_t a = g_static_scratch_addr[dev].load(std::memory_order_acquire);
    if (a == 0) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress((void**)&ptr, g_static_scratch) != cudaSuccess) return nullptr;
        a = reinterpret_cast<uintptr_t>(ptr);
        g_static_scratch_addr[dev].store(a, std::memory_order_release);
    }
    return reinterpret_cast<void*>(a);
}

template <class Cfg>
gemm_status_t run_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                          cudaStream_t stream, int sms, int dev) {
    CUtensorMap ta, tb, td, tc;
    Params p;
    gemm_status_t st = prepare<Cfg>(M, N, K, A, B, C, D, dev, ta, tb, td, tc, p);
    if (st != GEMM_OK) return st;
    void* scratch = static_scratch(dev);
    if (scratch == nullptr) return GEMM_ERR_CUDA;
    st = launch_config_fixed_scratch<Cfg>(ta, tb, td, tc, p, sms, dev, stream, scratch, kStaticScratchBytes);
    if (st != GEMM_OK) return st;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

// Looks up the fixed block on device `dev` (the current device).  Under lazy module
// loading the lookup is what makes the driver load this module, and with it the
// block, on that device: the C ABI does it on its first accepted call on each device,
// so that the block is in place before the caller reserves the rest of the device's
// memory or starts a stream capture.
bool setup_fixed_scratch(int dev) { return static_scratch(dev) != nullptr; }

gemm_status_t launch_gemm_f16_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                                      void* D, cudaStream_t stream, int sms, int dev) {
    // Narrow K as gemm_f16 (one k-block: these instances never split, so they need no
    // scratch); otherwise the stream-K rule of dense_choice over the fixed block.
    if (K <= 16)
        return M > 128 ? run<CfgF16K16Pair>(M, N, K, A, B, C, D, stream, sms, dev)
                       : run<CfgF16K16>(M, N, K, A, B, C, D, stream, sms, dev);
    if (K <= 32)
        return M > 128 ? run<CfgF16K32Pair>(M, N, K, A, B, C, D, stream, sms, dev)
                       : run<CfgF16K32>(M, N, K, A, B, C, D, stream, sms, dev);
    switch (dispatch::dense_choice(M, N, K, 64, sms)) {
        case dispatch::DENSE_PAIR_256: return run_noalloc<CfgF16Acc32Pair>(M, N, K, A, B, C, D, stream, sms, dev);
        case dispatch::DENSE_SINGLE_64: return run_noalloc<CfgF16N64>(M, N, K, A, B, C, D, stream, sms, dev);
        case dispatch::DENSE_SINGLE_128: return run_noalloc<CfgF16N128>(M, N, K, A, B, C, D, stream, sms, dev);
        default: return run_noalloc<CfgF16Acc32>(M, N, K, A, B, C, D, stream, sms, dev);
    }
}

unsigned int read_clear_error_f16() { return read_clear_word(g_err_f16); }

}  // namespace tn
