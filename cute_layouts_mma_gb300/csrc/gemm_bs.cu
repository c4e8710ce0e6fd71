// Block-scaled TN GEMM launcher: NVFP4 (tcgen05 kind::mxf4nvf4, scale_vec::4X)
// and MXFP8 (kind::mxf8f6f4, scale_vec::1X), fp32 accumulation, bf16 output.
#include <atomic>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace tn {

// NVFP4: 128 x 256 tiles, one TMEM accumulator (the scale slots use the rest),
// epilogue staged in 32 x 32 chunks (64-byte rows), single-buffered.
using CfgNvfp4 = Config<KIND_NVFP4, 256, 4, 1, 32, 1>;
// MXFP8: 128 x 128 tiles, double-buffered accumulator.
using CfgMxfp8 = Config<KIND_MXFP8, 128, 6, 2, 32, 1>;

static __device__ unsigned int g_err_bs;

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
        if (cudaGetSymbolAddress(&ptr, g_err_bs) != cudaSuccess) return nullptr;
        a = reinterpret_cast<uintptr_t>(ptr);
        g_err_addr[dev].store(a, std::memory_order_release);
    }
    return reinterpret_cast<unsigned int*>(a);
}

template <class Cfg>
gemm_status_t run(int bit, int64_t M, int64_t N, int64_t K, const void* A, const void* SFA, const void* B,
                  const void* SFB, const void* C, void* D, cudaStream_t stream, int sms, int dev) {
    constexpr bool fp4 = Cfg::KIND == KIND_NVFP4;
    const int64_t row_bytes = fp4 ? K / 2 : K;    // data bytes per row
    const int64_t sf_cols = K / (fp4 ? 16 : 32);  // scale bytes per row
    CUtensorMap ta, tb, tsa, tsb, td;
    // Data boxes: 128 bytes of K (256 E2M1 / 128 E4M3 elements) x rows, 128B swizzle.
    // Scale boxes: 16 bytes (16 scale blocks) x rows, no swizzle.
    // D: bf16 [M][N], stored in 32-row x EPI_COLS boxes from the epilogue staging.
    if (!encode_tma_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, M, row_bytes, 128, Cfg::BM, 128) ||
        !encode_tma_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, N, row_bytes, 128, Cfg::BN, 128) ||
        !encode_tma_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFA, sf_cols, M, sf_cols, 16, Cfg::BM, 0) ||
        !encode_tma_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, sf_cols, N, sf_cols, 16, Cfg::BN, 0) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
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
    p.num_k_blocks = static_cast<int>(row_bytes / 128);
    p.C = C;
    p.D = D;
    p.err = err;
    const int tiles = p.num_m_blocks * p.num_n_blocks;
    const int grid = tiles < sms ? tiles : sms;
    tn_gemm_kernel<Cfg><<<grid, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(ta, tb, tsa, tsb, td, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

gemm_status_t launch_gemm_block_scaled(int64_t M, int64_t N, int64_t K, const void* A, const void* SFA,
                                       const void* B, const void* SFB, const void* C, void* D, int fmt,
                                       cudaStream_t stream, int sms, int dev) {
    if (fmt == GEMM_FMT_NVFP4) return run<CfgNvfp4>(0, M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev);
    return run<CfgMxfp8>(1, M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev);
}

unsigned int read_clear_error_block_scaled() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_bs, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_err_bs, &zero, sizeof(zero));
    return v;
}

}  // namespace tn
