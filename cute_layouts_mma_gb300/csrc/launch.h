// Host-side glue shared by the C-ABI (api.cu) and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tn_gemm.h"

namespace tn {

// Encode a 2-D tiled TMA map over a row-major matrix: `inner` elements per row
// (contiguous), `rows` rows `pitch` bytes apart, boxes of box_inner x box_rows.
// swizzle_bytes: 0 (none), 32, 64 or 128 -- the XOR swizzle of the box in shared
// memory (box rows of at most that many bytes).  Maps are cached per thread.
// Returns false if the driver rejects the map.
bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                   uint64_t rows, uint64_t pitch, uint32_t box_inner, uint32_t box_rows,
                   int swizzle_bytes);

// Launchers; arguments are already validated.  `sms` is the SM count of the
// current device, `dev` its ordinal.
gemm_status_t launch_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                              const void* C, void* D, int accum, cudaStream_t stream, int sms,
                              int dev);
gemm_status_t launch_gemm_block_scaled(int64_t M, int64_t N, int64_t K, const void* A,
                                       const void* SFA, const void* B, const void* SFB,
                                       const void* C, void* D, int fmt, cudaStream_t stream,
                                       int sms, int dev);

// FP16 with fp32 accumulation on the stream-K schedule, whose scratch is a fixed block
// inside the module (no allocation); arguments are already validated.
gemm_status_t launch_gemm_f16_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                                      const void* C, void* D, cudaStream_t stream, int sms, int dev);

// Loads the fixed block of launch_gemm_f16_noalloc on device `dev` (the current
// device); false if that fails.  Called once per device, on the first accepted call.
bool setup_fixed_scratch(int dev);

gemm_status_t launch_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                               const void* C, void* D, cudaStream_t stream, int sms, int dev);
gemm_status_t launch_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B,
                              const void* C, void* D, int fmt, cudaStream_t stream, int sms, int dev);

// Read and clear the device error word of each kernel family on the current
// device (synchronous).  Non-zero means a kernel abandoned its work.
unsigned int read_clear_error_f16();
unsigned int read_clear_error_block_scaled();
unsigned int read_clear_error_dense();

constexpr int kMaxDevices = 64;

}  // namespace tn
