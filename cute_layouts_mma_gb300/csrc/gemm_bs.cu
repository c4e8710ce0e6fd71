// Block-scaled TN GEMM launcher: NVFP4 (tcgen05 kind::mxf4nvf4, scale_vec::4X)
// and MXFP8 (kind::mxf8f6f4, scale_vec::1X), fp32 accumulation, bf16 output.
#include <atomic>

#include "launch_kernel.cuh"

namespace tn {

#ifndef TN_SCALE_COPY
// Scale movement (ScaleMode, gemm_kernel.cuh): NVFP4 one 16-byte scale slot per stage
// (in CTA pairs each CTA loads half of the tile's SFB and multicasts it to both);
// MXFP8 a ring of four 16-byte slots, each holding the scales of four k-blocks.  The
// scale writers place them in TMEM with tcgen05.st.
constexpr int kNvfp4Scales = SF_STAGE, kNvfp4SfSlots = 5;
constexpr int kMxfp8Scales = SF_RING, kMxfp8SfSlots = 4;
#else
// Test build only: every block-scaled instance moves its scales with the pages'
// tcgen05.cp.32x128b.warpx4 (repacked base tiles in shared memory, copied by the MMA
// thread).  On GB300 this measured 1.3-1.5x slower on single CTAs (the copies cost the
// tensor pipe) and 2.3-2.6x slower in CTA pairs (the peer's repacked tiles need a
// release.cluster arrival per stage) than tcgen05.st from the writer warps.
constexpr int kNvfp4Scales = SF_COPY, kNvfp4SfSlots = 5;
constexpr int kMxfp8Scales = SF_COPY, kMxfp8SfSlots = 5;
#endif

// NVFP4, CTA pairs (M > 128): 256 x 256 tiles, 5 stages, one TMEM accumulator
// (256 columns; the scale columns, 5 x 48, use the rest).  512 threads in four
// warpgroups: issuers and MMA, epilogue, scale writers, epilogue.  The first and third
// give registers to the epilogue warpgroups (setmaxnreg), so each of the 8 epilogue
// warps takes its whole 32 x 128 slice of the accumulator into registers with one TMEM
// round trip and releases it before rounding, staging (one 64-column buffer per warp; C
// TMA-loaded into it) and storing.
using CfgNvfp4Pair = Config<KIND_NVFP4, 256, 5, 1, 64, 1, 2, 8, 128, true, kNvfp4Scales, 16, kNvfp4SfSlots>;
// NVFP4, single CTAs (M <= 128): 128 x 128 tiles, 5 stages, two TMEM accumulators
// (2 x 128 + 5 x 32 scale columns), each epilogue warp staging its whole 32 x 128
// slice.  Measured 1.2-1.75x faster than 128 x 256 tiles with one accumulator on
// skinny problems: the next tile's MMAs no longer wait for the drain.
using CfgNvfp4 = Config<KIND_NVFP4, 128, 5, 2, 32, 4, 1, 4, 128, false, kNvfp4Scales, 16, kNvfp4SfSlots>;
// MXFP8: 128 x 128 tiles, 5 stages, double-buffered accumulator (one CTA per
// MMA: the skinny, HBM-bound shape is M = 128).  Each epilogue warp stages its whole
// 32 x 128 slice, so all of C for a tile is fetched before the accumulator is ready
// (a one-tile-per-CTA problem otherwise pays the C round trips after its mainloop).
using CfgMxfp8 = Config<KIND_MXFP8, 128, 5, 2, 32, 4, 1, 4, 128, false, kMxfp8Scales, 16, kMxfp8SfSlots>;
// MXFP8, CTA pairs (M > 128): the NVFP4 pair's layout (256 x 256 tiles, 5 stages,
// one accumulator, register drain).  A stage's scales take 12 TMEM columns (one copy
// set; each MMA's scale-factor ID picks its byte).
using CfgMxfp8Pair = Config<KIND_MXFP8, 256, 5, 1, 64, 1, 2, 8, 128, true, kMxfp8Scales, 16, kMxfp8SfSlots>;

static __device__ unsigned int g_err_bs;

namespace {

std::atomic<uintptr_t> g_err_addr[kMaxDevices];

unsigned int* err_word(int dev) { return device_symbol(g_err_bs, g_err_addr, dev); }

template <class Cfg>
gemm_status_t run(int64_t M, int64_t N, int64_t K, const void* A, const void* SFA, const void* B, const void* SFB,
                  const void* C, void* D, cudaStream_t stream, int sms, int dev) {
    constexpr bool fp4 = Cfg::KIND == KIND_NVFP4;
    const int64_t row_bytes = fp4 ? K / 2 : K;    // data bytes per row
    const int64_t sf_cols = K / (fp4 ? 16 : 32);  // scale bytes per row
    CUtensorMap ta, tb, tsa, tsb, td, tc;
    // Data boxes: 128 bytes of K (256 E2M1 / 128 E4M3 elements) x rows, 128B swizzle;
    // A boxes are this CTA's 128 rows, B boxes its BN/PAIR rows.  Scale boxes: SF_W bytes
    // (the scales of SF_KB k-blocks) x rows of the caller's row-major scale matrices, no
    // swizzle: this CTA's 128 SFA rows, all BN SFB rows of the tile.  D: bf16 [M][N], stored in
    // 32-row x EPI_COLS boxes from the staging.
    if (!encode_tma_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, M, row_bytes, 128, Cfg::BM, 128) ||
        !encode_tma_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, N, row_bytes, 128, Cfg::BN_CTA, 128) ||
        !encode_tma_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFA, sf_cols, M, sf_cols, Cfg::SF_W, Cfg::BM, 0) ||
        !encode_tma_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, sf_cols, N, sf_cols, Cfg::SF_W, Cfg::SFB_BOX_ROWS, 0) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
                       Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    // C (if any): the same boxes as D, TMA-loaded into the epilogue staging buffers.
    if (C == nullptr)
        tc = td;
    else if (!encode_tma_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, C, N, M, N * 2, Cfg::EPI_COLS, 32, Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    unsigned int* err = err_word(dev);
    if (err == nullptr) return GEMM_ERR_CUDA;
    Params p{};
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.num_m_blocks = static_cast<int>((M + Cfg::BM_TILE - 1) / Cfg::BM_TILE);
    p.num_n_blocks = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int>(row_bytes / 128);
    p.C = C;
    p.D = D;
    p.err = err;
    p.split = 1;
    if constexpr (Cfg::kSplit) {
        // skinny problems: each tile's k-blocks split inside a cluster
        int res[dispatch::kMaxSplit + 1];
        if (split_capacity<Cfg>(sms, dev, res) != cudaSuccess) return GEMM_ERR_CUDA;
        p.split = dispatch::choose_split(static_cast<long long>(p.num_m_blocks) * p.num_n_blocks, p.num_k_blocks,
                                         sms, res);
    }
    if (launch_config<Cfg>(ta, tb, tsa, tsb, td, tc, p, sms, dev, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

gemm_status_t launch_gemm_block_scaled(int64_t M, int64_t N, int64_t K, const void* A, const void* SFA,
                                       const void* B, const void* SFB, const void* C, void* D, int fmt,
                                       cudaStream_t stream, int sms, int dev) {
    const bool pair = dispatch::use_block_scaled_pair(M, N, sms);
    if (fmt == GEMM_FMT_NVFP4)
        return pair ? run<CfgNvfp4Pair>(M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev)
                    : run<CfgNvfp4>(M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev);
    return pair ? run<CfgMxfp8Pair>(M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev)
                : run<CfgMxfp8>(M, N, K, A, SFA, B, SFB, C, D, stream, sms, dev);
}

unsigned int read_clear_error_block_scaled() { return read_clear_word(g_err_bs); }

}  // namespace tn
