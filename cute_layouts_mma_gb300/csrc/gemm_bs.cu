// Block-scaled TN GEMM launcher: NVFP4 (tcgen05 kind::mxf4nvf4, scale_vec::4X)
// and MXFP8 (kind::mxf8f6f4, scale_vec::1X), fp32 accumulation, bf16 output.
#include <atomic>

#include "launch_kernel.cuh"

namespace tn {

// NVFP4, CTA pairs (M > 128): 256 x 256 tiles, 5 stages, one TMEM accumulator
// (256 columns; the scale slots, 5 x 48 columns, use the rest).  512 threads in
// four warpgroups: issuers and MMA, epilogue, scale writers, epilogue.  The first
// and third give registers to the epilogue warpgroups (setmaxnreg), so each of the
// 8 epilogue warps takes its whole 32 x 128 slice of the accumulator into
// registers with one TMEM round trip and releases it before rounding, staging
// (one 64-column buffer per warp; C TMA-loaded into it) and storing.
using CfgNvfp4Pair = Config<KIND_NVFP4, 256, 5, 1, 64, 1, 2, 8, 128, true>;
// NVFP4, single CTAs (M <= 128): 128 x 128 tiles, 5 stages, two TMEM accumulators
// (2 x 128 + 5 x 32 scale columns), each epilogue warp staging its whole 32 x 128
// slice.  Measured 1.2-1.75x faster than 128 x 256 tiles with one accumulator on
// skinny problems: the next tile's MMAs no longer wait for the drain, and stream-K
// cuts fewer pieces.
using CfgNvfp4 = Config<KIND_NVFP4, 128, 5, 2, 32, 4, 1>;
// MXFP8: 128 x 128 tiles, 5 stages, double-buffered accumulator (one CTA per
// MMA: the skinny, HBM-bound shape is M = 128).  Each epilogue warp stages its whole
// 32 x 128 slice, so all of C for a tile is fetched before the accumulator is ready
// (a one-tile-per-CTA problem otherwise pays the C round trips after its mainloop).
using CfgMxfp8 = Config<KIND_MXFP8, 128, 5, 2, 32, 4, 1>;
// MXFP8, CTA pairs (M > 128): the NVFP4 pair's layout (256 x 256 tiles, 5 stages,
// one accumulator, register drain, packed scales).  A stage's scales take 12 TMEM
// columns (one copy set; each MMA's scale-factor ID picks its byte).
using CfgMxfp8Pair = Config<KIND_MXFP8, 256, 5, 1, 64, 1, 2, 8, 128, true>;

static __device__ unsigned int g_err_bs;

namespace {

std::atomic<uintptr_t> g_err_addr[kMaxDevices];

unsigned int* err_word(int dev) { return device_symbol(g_err_bs, g_err_addr, dev); }

// One scale matrix to regroup: src [rows][cols16 * 16] bytes, row-major; dst
// [groups][cols16][group_rows][16] (group_rows a multiple of 32), rows at or past
// `rows` zero.
struct PackJob {
    const uint8_t* src;
    uint8_t* dst;
    int rows;
    int groups;
    int group_rows;
};

// Regroups SFA (128-row groups: one CTA's rows) and SFB (one group per tile's
// columns) into the packed blocks the stages load, one warp per block: lane l
// moves rows l, l+32, ... of the block, so each store instruction writes 512
// contiguous bytes.  A block holds exactly the bytes of the 16-byte-wide scale box
// of one stage, in the same row-major order.
__global__ void __launch_bounds__(256) pack_scales_kernel(PackJob a, PackJob b, int cols16) {
    griddep_wait();  // the scales may be written by the previous launch on the stream
    griddep_launch_dependents();
    const int w = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int blocks_a = a.groups * cols16;
    if (w >= blocks_a + b.groups * cols16) return;
    const PackJob& j = w < blocks_a ? a : b;
    const int blk = w < blocks_a ? w : w - blocks_a;
    const int g = blk / cols16, c = blk - g * cols16;
    const size_t pitch = static_cast<size_t>(cols16) * 16;
    uint4* out = reinterpret_cast<uint4*>(j.dst + static_cast<size_t>(blk) * j.group_rows * 16);
    for (int r = lane; r < j.group_rows; r += 32) {
        const long long row = static_cast<long long>(g) * j.group_rows + r;  // may pass INT_MAX near M = 2^31
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < j.rows) v = __ldg(reinterpret_cast<const uint4*>(j.src + static_cast<size_t>(row) * pitch + 16 * c));
        out[r] = v;
    }
}

// Enqueue the regrouping of SFA (ga groups of 128 rows) and SFB (gb groups of gb_rows)
// into `packed` on `stream`: SFA's blocks first, then SFB's.
cudaError_t launch_pack(const void* SFA, int64_t M, int ga, const void* SFB, int64_t N, int gb, int gb_rows,
                        int cols16, uint8_t* packed, cudaStream_t stream) {
    const PackJob a{static_cast<const uint8_t*>(SFA), packed, static_cast<int>(M), ga, 128};
    const PackJob b{static_cast<const uint8_t*>(SFB), packed + static_cast<size_t>(ga) * cols16 * 128 * 16,
                    static_cast<int>(N), gb, gb_rows};
    const long long warps = static_cast<long long>(ga + gb) * cols16;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>((warps + 7) / 8), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pack_scales_kernel, a, b, cols16);
}

template <class Cfg>
gemm_status_t run(int64_t M, int64_t N, int64_t K, const void* A, const void* SFA, const void* B, const void* SFB,
                  const void* C, void* D, cudaStream_t stream, int sms, int dev) {
    constexpr bool fp4 = Cfg::KIND == KIND_NVFP4;
    const int64_t row_bytes = fp4 ? K / 2 : K;    // data bytes per row
    const int64_t sf_cols = K / (fp4 ? 16 : 32);  // scale bytes per row
    CUtensorMap ta, tb, tsa, tsb, td, tc;
    // Data boxes: 128 bytes of K (256 E2M1 / 128 E4M3 elements) x rows, 128B swizzle;
    // A boxes are this CTA's 128 rows, B boxes its BN/PAIR rows.  Scale boxes (MXFP8):
    // 16 bytes (16 scale blocks) x rows, no swizzle: 128 SFA rows, all BN SFB rows of
    // the tile.  D: bf16 [M][N], stored in 32-row x EPI_COLS boxes from the staging.
    if (!encode_tma_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, M, row_bytes, 128, Cfg::BM, 128) ||
        !encode_tma_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, N, row_bytes, 128, Cfg::BN_CTA, 128) ||
        !encode_tma_2d(&td, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, N, M, N * 2, Cfg::EPI_COLS, 32,
                       Cfg::EPI_ROW_BYTES))
        return GEMM_ERR_CUDA;
    if constexpr (Cfg::kPackedScales) {
        tsa = ta;  // unused: the scales arrive as packed blocks
        tsb = ta;
    } else if (!encode_tma_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFA, sf_cols, M, sf_cols, 16, Cfg::BM, 0) ||
               !encode_tma_2d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT8, SFB, sf_cols, N, sf_cols, 16, Cfg::BN, 0)) {
        return GEMM_ERR_CUDA;
    }
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
    if constexpr (Cfg::kPackedScales) {
        // Packed scales for this call, taken from the device's stream-ordered pool and
        // returned on the same stream after the GEMM.  Row groups cover whole tiles.
        // SFA in groups of 128 rows (one CTA's rows), SFB in groups of BN rows (one tile).
        const int cols16 = static_cast<int>(sf_cols / 16);
        const int ga = p.num_m_blocks * (Cfg::BM_TILE / 128);
        const int gb = p.num_n_blocks;
        const size_t a_bytes = static_cast<size_t>(ga) * cols16 * 128 * 16;
        const size_t b_bytes = static_cast<size_t>(gb) * cols16 * Cfg::BN * 16;
        void* packed = nullptr;
        if (cudaMallocFromPoolAsync(&packed, a_bytes + b_bytes, scratch_pool(dev), stream) != cudaSuccess)
            return GEMM_ERR_CUDA;
        p.sfa_packed = static_cast<const uint8_t*>(packed);
        p.sfb_packed = static_cast<const uint8_t*>(packed) + a_bytes;
        p.sf_cols16 = cols16;
        cudaError_t e =
            launch_pack(SFA, M, ga, SFB, N, gb, Cfg::BN, cols16, static_cast<uint8_t*>(packed), stream);
        if (e == cudaSuccess) e = launch_config<Cfg>(ta, tb, tsa, tsb, td, tc, p, sms, dev, stream);
        const cudaError_t f = cudaFreeAsync(packed, stream);
        if (e != cudaSuccess || f != cudaSuccess) return GEMM_ERR_CUDA;
    } else if (launch_config<Cfg>(ta, tb, tsa, tsb, td, tc, p, sms, dev, stream) != cudaSuccess) {
        return GEMM_ERR_CUDA;
    }
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
