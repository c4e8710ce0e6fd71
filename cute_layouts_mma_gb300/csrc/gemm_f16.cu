// FP16 TN GEMM launcher (tcgen05 kind::f16, fp32 or fp16 accumulation).
#include <atomic>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace tn {

// 128 x 256 tiles, 4 stages of 64 K, two TMEM accumulators, epilogue staged in
// 32 x 64 chunks (128-byte rows), double-buffered.
using CfgF16Acc32 = Config<KIND_F16_ACC32, 256, 4, 2, 64, 2>;
using CfgF16Acc16 = Config<KIND_F16_ACC16, 256, 4, 2, 64, 2>;

// Device-side record of an abandoned launch (a bounded wait ran out).
static __device__ unsigned int g_err_f16;

namespace {

std::atomic<uint32_t> g_attr_done[kMaxDevices];
std::atomic<uintptr_t> g_err_addr[kMaxDevices];

template <class Cfg>
cudaError_t ensure_attr(int dev, int bit) {
    if (g_attr_done[dev].load(std::memory_order_acquire) & (1u << bit)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(tn_gemm_kernel<Cfg>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_BYTES);
    if (e == cudaSuccess) g_attr_done[dev].fetch_or(1u << bit, std::memory_order_acq_rel);
    return e;
}

unsigned int* err_word(int dev) {
    uintptr_t a = g_err_addr[dev].load(std::memory_order_acquire);
    if (a == 0) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_err_f16) != cudaSuccess) return nullptr;
        a = reinterpret_cast<uintptr_t>(ptr);
        g_err_addr[dev].store(a, std::memory_order_release);
    }
    return reinterpret_cast<unsigned int*>(a);
}

template <class Cfg>
gemm_status_t run(int bit, int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                  void* D, cudaStream_t stream, int sms, int dev) {
    CUtensorMap ta, tb, td;
    // A: fp16 [M][K]; B: fp16 [N][K]; boxes of 64 elements (128 bytes) of K.
    // D: fp16 [M][N], stored in 32-row x EPI_COLS boxes from the epilogue staging.
    if (!encode_tma_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, A, K, M, K * 2, 64, Cfg::BM, 128) ||
        !encode_tma_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, K, N, K * 2, 64, Cfg::BN, 128) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
                       Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    if (ensure_attr<Cfg>(dev, bit) != cudaSuccess) return GEMM_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (err == nullptr) return GEMM_ERR_CUDA;
    Params p;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>((M + Cfg::BM - 1) / Cfg::BM);
    p.num_n_blocks = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int>((K + 63) / 64);
    p.C = C;
    p.D = D;
    p.err = err;
    const int tiles = p.num_m_blocks * p.num_n_blocks;
    const int grid = tiles < sms ? tiles : sms;
    tn_gemm_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, ta, tb, td, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

gemm_status_t launch_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                              void* D, int accum, cudaStream_t stream, int sms, int dev) {
    if (accum == GEMM_ACC_F32) return run<CfgF16Acc32>(0, M, N, K, A, B, C, D, stream, sms, dev);
    return run<CfgF16Acc16>(1, M, N, K, A, B, C, D, stream, sms, dev);
}

unsigned int read_clear_error_f16() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_f16, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_err_f16, &zero, sizeof(zero));
    return v;
}

}  // namespace tn
