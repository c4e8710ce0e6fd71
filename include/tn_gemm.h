/*
 * tn_gemm.h -- C ABI of the GB300 (sm_103a) TN matrix multiply-accumulate library.
 *
 *   D = A x B + C,  A indexed (M,K), B indexed (N,K), both K-contiguous ("TN").
 *
 * Source of the operation:
 *   - "CuTe 中 A、B 如何加载到 MMA 寄存器", section 1: D = A x B + C with A
 *     indexed (M,K) and B indexed (N,K), K contiguous in both; C and D are M x N.
 *     The pages' FP16-in / FP16-accumulate atom (F16F16F16F16_TN) and the FP32-
 *     accumulate variant are the two accumulation modes of gemm_f16.
 *   - "数据布局及其记号", section on block-scaled MMA (TMEM scale factors):
 *     A_real[m,k] = A_low[m,k] * SFA[m, k // K_blk], likewise B with SFB[n, .],
 *     D = C + A_real x B_real; NVFP4 = E2M1 data + one E4M3 scale per 16
 *     K-elements, MXFP8 = E4M3 data + one E8M0 scale per 32 K-elements.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the
 *     library never frees or keeps caller memory.
 *   - No call allocates, frees or resizes device memory; none needs memory beyond the
 *     caller's operands.  Skinny problems, whose output tiles would leave more than
 *     half of the device's SMs idle, are split inside thread-block clusters: each
 *     tile goes to a cluster of up to 8 CTAs that share its k-blocks, and the cluster
 *     adds its fp32 partial sums in its own shared memory (distributed shared memory)
 *     before rounding.  Calls on different streams may therefore run concurrently.
 *     (gemm_f16_noalloc keeps a different, stream-K, schedule over a fixed block of
 *     the library's own device memory; see there.)
 *   - Matrices are dense and row-major with no padding: A rows are K elements
 *     long (NVFP4: K/2 bytes), B rows likewise, C and D rows are N elements.
 *     Scale-factor matrices are row-major u8 [rows][K / K_blk].
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and do not synchronise.  Arguments are checked on the host before
 *     anything is launched; a rejected call launches nothing.
 *   - D must not overlap A, B, SFA or SFB.  D may be exactly C (in place), or
 *     disjoint from it; a partial overlap is rejected.
 *   - All pointers must be 16-byte aligned.  Row pitches must be multiples of
 *     16 bytes (see each call).  M and N need not be multiples of any tile.
 *   - Device-side failures (a pipeline wait that exceeds its time limit) do not
 *     hang or fault the GPU: the kernel abandons its work, records the failure
 *     and returns; gemm_last_device_error() reports it.
 *   - Calls may be made from several host threads; the library's only state is
 *     per-device, set up on first use (kernel attributes, SM count).
 *   - The kernels' copies carry L2 eviction hints, which change no result: A is
 *     kept in L2 ahead of other lines (it is reused by every tile of its rows), C
 *     and D are read or written once and let go first, and so is B when the
 *     output has a single row of tiles.  A D that the next kernel reads at once
 *     may therefore come from DRAM rather than L2.
 *
 * Numerics: products are formed by the tensor cores
 * and summed in fp32 (GEMM_ACC_F32) or fp16 (GEMM_ACC_F16); C is added in fp32
 * and the result rounded once, to nearest even, to the output type.  When a tile
 * is split (inside a cluster, or by gemm_f16_noalloc's stream-K schedule) its fp32
 * sum is formed piecewise (contiguous k-ranges, added in fp32 in a fixed order), so
 * the order of the fp32 additions depends on M, N, K and the SM count; results are
 * deterministic for a given device and shape.
 */
#ifndef TN_GEMM_H
#define TN_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __DRIVER_TYPES_H__
typedef struct CUstream_st *cudaStream_t;
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1, /* a size, enum or pointer argument is out of range  */
    GEMM_ERR_UNSUPPORTED = 2, /* no GPU of compute capability 10.3 is current      */
    GEMM_ERR_ALIGNMENT = 3,   /* a pointer or a row pitch is not 16-byte aligned   */
    GEMM_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed                 */
    GEMM_ERR_TIMEOUT = 5      /* a kernel gave up on a pipeline wait (device side) */
} gemm_status_t;

enum { GEMM_ACC_F32 = 0, GEMM_ACC_F16 = 1 };   /* accum_dtype of gemm_f16        */
enum { GEMM_FMT_NVFP4 = 0, GEMM_FMT_MXFP8 = 1 }; /* fmt of gemm_block_scaled      */
enum { GEMM_FP8_E4M3 = 0, GEMM_FP8_E5M2 = 1 };   /* fmt of gemm_fp8               */

/*
 * FP16 TN GEMM:  D[m][n] = round_fp16( C[m][n] + sum_k A[m][k] * B[n][k] ).
 *
 *   M, N, K      sizes, each >= 1 and < 2^31.  K % 8 == 0 and N % 8 == 0 (16-byte
 *                row pitches for A, B, C, D).
 *   A            half[M][K], K contiguous.
 *   B            half[N][K], K contiguous.
 *   C            half[M][N] or NULL (NULL: C = 0, nothing is read).
 *   D            half[M][N], written; may equal C.
 *   accum_dtype  GEMM_ACC_F32: tensor-core sums in fp32.
 *                GEMM_ACC_F16: tensor-core sums in fp16 (the pages' F16F16F16F16
 *                atom); C is then added in fp32 before the final rounding.
 *   stream       cudaStream_t the kernel is launched on.
 * Returns GEMM_OK once the kernel is enqueued, else the first failed check.
 */
gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                       const void *C, void *D, int accum_dtype, cudaStream_t stream);

/*
 * BF16 TN GEMM:  D[m][n] = round_bf16( C[m][n] + sum_k A[m][k] * B[n][k] ).
 *
 * The same TN multiply-accumulate as gemm_f16 ("CuTe 中 A、B 如何加载到 MMA 寄存器",
 * section 1) with BF16 operands; products summed in fp32 by the tensor cores
 * (kind::f16 with BF16 inputs), C added in fp32, one RNE rounding to bf16.
 *
 *   M, N, K      each >= 1 and < 2^31; K % 8 == 0 and N % 8 == 0.
 *   A            bf16[M][K], K contiguous.   B  bf16[N][K], K contiguous.
 *   C            bf16[M][N] or NULL (zero).  D  bf16[M][N], written; may equal C.
 *   stream       cudaStream_t the kernel is launched on.
 * Returns GEMM_OK once the kernel is enqueued, else the first failed check.
 */
gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                        const void *C, void *D, cudaStream_t stream);

/*
 * FP8 TN GEMM without scale factors:
 *   D[m][n] = round_bf16( C[m][n] + sum_k decode(A[m][k]) * decode(B[n][k]) ).
 *
 * The TN multiply-accumulate of section 1 of the CuTe page with both operands
 * in the same FP8 format (kind::f8f6f4): GEMM_FP8_E4M3 (bias 7, max 448,
 * S.1111.111 NaN) or GEMM_FP8_E5M2 (bias 15, max 57344, IEEE Inf / NaN); the
 * same E4M3 data as the MXFP8 form of gemm_block_scaled with every scale 1.
 * Products summed in fp32, C added in fp32, one RNE rounding to bf16.
 *
 *   M, N, K      each >= 1 and < 2^31; K % 16 == 0 and N % 8 == 0.
 *   A            u8[M][K] FP8 codes, K contiguous.   B  u8[N][K], K contiguous.
 *   C            bf16[M][N] or NULL (zero).           D  bf16[M][N]; may equal C.
 *   fmt          GEMM_FP8_E4M3 or GEMM_FP8_E5M2 (A and B alike).
 * Returns GEMM_OK once the kernel is enqueued, else the first failed check.
 */
gemm_status_t gemm_fp8(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                       const void *C, void *D, int fmt, cudaStream_t stream);

/*
 * FP16 TN GEMM with fp32 accumulation on a fixed scratch block.
 *
 * The pages have no counterpart of this call: it exists for callers that must
 * not allocate device memory while they run.  Examples are a plugin inside a
 * host application that owns all device memory and hands out only the buffers
 * it chose, a serving loop that has reserved nearly all of HBM up front (so
 * any later allocation may fail), and code whose latency budget cannot absorb
 * an allocation.  gemm_f16 allocates nothing either; this call differs in its
 * schedule for skinny problems: stream-K, where every SM takes an equal share of
 * the k-blocks of the last tiles and the unit that finishes a tile adds the
 * others' fp32 partials from global memory.  Those partials live in a fixed
 * 20 MiB block that is part of the library's module and that every GPU which
 * loads the library holds until the process exits.  Stream-K uses every SM even
 * for a handful of tiles with very long K, where a cluster of 8 would leave most
 * of the device idle.
 *
 *   M, N, K, A, B, C, D, stream   as gemm_f16 (fp32 accumulation); the result
 *                agrees with gemm_f16's within the fp32 accumulation tolerance
 *                (the two may split a tile differently).  K <= 32 takes the same
 *                narrow-K instances as gemm_f16 (one k-block, never split).
 * Scratch limits:
 *   - The call never calls cudaMalloc, cudaFree or a pool allocator.  The block
 *     is loaded on a device by the first accepted call of any entry point of this
 *     library there (which also looks up its device address, once per device,
 *     with that device current): make one call on each device before reserving
 *     the rest of its memory and before any stream capture.
 *   - A stream-K launch (128 x 128 tiles on single CTAs) needs 64 KB of fp32
 *     partials per SM it runs on, plus flags: 9.5 MiB on a 152-SM GB300.  A
 *     launch whose need exceeds the 20 MiB block (a device of more than 319
 *     SMs) is refused with GEMM_ERR_INVALID_ARG and nothing is enqueued.
 *     Whole-tile launches use no scratch.
 *   - Every call on a device shares the block and it keeps the last call's
 *     contents: each call clears the flags it uses (an async memset on
 *     `stream`); partial sums are written before they are read.  Calls that
 *     overlap on the GPU (e.g. on two streams without ordering between them)
 *     race on the block and give wrong results; order them on one stream.
 * Returns as gemm_f16.
 */
gemm_status_t gemm_f16_noalloc(int64_t M, int64_t N, int64_t K, const void *A, const void *B,
                               const void *C, void *D, cudaStream_t stream);

/*
 * Block-scaled TN GEMM:
 *   D[m][n] = round_bf16( C[m][n] + sum_k (A[m][k] * SFA[m][k/K_blk])
 *                                         * (B[n][k] * SFB[n][k/K_blk]) ).
 *
 *   fmt == GEMM_FMT_NVFP4: K_blk = 16.  A is u8[M][K/2] holding two E2M1 codes
 *        per byte, element 2j in the low nibble and 2j+1 in the high nibble of
 *        byte j.  SFA is u8[M][K/16] of E4M3 scales; the sign bit must be 0
 *        (the tensor cores read the scale as unsigned E4M3).  K % 256 == 0.
 *   fmt == GEMM_FMT_MXFP8: K_blk = 32.  A is u8[M][K] of E4M3 codes.  SFA is
 *        u8[M][K/32] of E8M0 exponents (value 2^(e-127)).  K % 512 == 0.
 *   B, SFB       the same layouts with N rows.
 *   C            bf16[M][N] or NULL (NULL: C = 0, nothing is read).
 *   D            bf16[M][N], written; may equal C.  N % 8 == 0.
 * The K multiples make every scale-factor row a whole number of 16-byte
 * chunks.  Sums are fp32.  NaN scales or data give undefined (finite or NaN)
 * results in the affected outputs; no other effect.
 */
gemm_status_t gemm_block_scaled(int64_t M, int64_t N, int64_t K, const void *A,
                                const void *SFA, const void *B, const void *SFB,
                                const void *C, void *D, int fmt, cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *gemm_status_string(gemm_status_t status);

/*
 * Synchronises the current device, then returns GEMM_ERR_TIMEOUT if any kernel
 * of this library abandoned its work since the previous call (and clears that
 * record), GEMM_ERR_CUDA if the device reports an error, else GEMM_OK.
 */
gemm_status_t gemm_last_device_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TN_GEMM_H */
