// C ABI of the TN GEMM library: argument checks, TMA map encoding, dispatch.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.h"

namespace tn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

bool size_ok(int64_t x) { return x >= 1 && x < (int64_t(1) << 31); }

// Current device, its SM count, and whether it is a compute capability 10.3 part.
gemm_status_t device_info(int* dev, int* sms) {
    if (cudaGetDevice(dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    // First accepted call on this device: load the module block of gemm_f16_noalloc
    // now (lazy module loading would otherwise defer it to that call's first use).
    static std::atomic<bool> ready[kMaxDevices];
    if (!ready[*dev].load(std::memory_order_acquire)) {
        if (!setup_fixed_scratch(*dev)) return GEMM_ERR_CUDA;
        ready[*dev].store(true, std::memory_order_release);
    }
    return GEMM_OK;
}

// D may equal C or be disjoint from it.
bool c_d_ok(const void* C, const void* D, uint64_t bytes) {
    return C == nullptr || C == D || !overlaps(C, bytes, D, bytes);
}

}  // namespace

bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t pitch, uint32_t box_inner, uint32_t box_rows, int swizzle_bytes) {
    // Small per-thread cache: repeated calls on the same buffers skip the driver call.
    struct Entry {
        const void* base;
        uint64_t inner, rows, pitch;
        uint32_t box_inner, box_rows;
        int dtype, swz;
        CUtensorMap map;
    };
    constexpr int kEntries = 16;
    thread_local Entry cache[kEntries];
    thread_local int cache_used = 0, cache_next = 0;
    for (int i = 0; i < cache_used; ++i) {
        const Entry& e = cache[i];
        if (e.base == base && e.inner == inner && e.rows == rows && e.pitch == pitch && e.box_inner == box_inner &&
            e.box_rows == box_rows && e.dtype == static_cast<int>(dtype) && e.swz == swizzle_bytes) {
            *map = e.map;
            return true;
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (enc == nullptr) return false;
    std::memset(map, 0, sizeof(*map));
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUtensorMapSwizzle swz = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                   : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    Entry& e = cache[cache_next];
    e = Entry{base, inner, rows, pitch, box_inner, box_rows, static_cast<int>(dtype), swizzle_bytes, *map};
    cache_next = (cache_next + 1) % kEntries;
    if (cache_used < kEntries) ++cache_used;
    return true;
}

}  // namespace tn

extern "C" {

gemm_status_t gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                       int accum_dtype, cudaStream_t stream) {
    using namespace tn;
    if (!size_ok(M) || !size_ok(N) || !size_ok(K)) return GEMM_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr || D == nullptr) return GEMM_ERR_INVALID_ARG;
    if (accum_dtype != GEMM_ACC_F32 && accum_dtype != GEMM_ACC_F16) return GEMM_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (C != nullptr && !aligned16(C)))
        return GEMM_ERR_ALIGNMENT;
    const uint64_t abytes = uint64_t(M) * uint64_t(K) * 2, bbytes = uint64_t(N) * uint64_t(K) * 2;
    const uint64_t dbytes = uint64_t(M) * uint64_t(N) * 2;
    if (overlaps(D, dbytes, A, abytes) || overlaps(D, dbytes, B, bbytes) || !c_d_ok(C, D, dbytes))
        return GEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    gemm_status_t st = device_info(&dev, &sms);
    if (st != GEMM_OK) return st;
    return launch_gemm_f16(M, N, K, A, B, C, D, accum_dtype, stream, sms, dev);
}

gemm_status_t gemm_f16_noalloc(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                               void* D, cudaStream_t stream) {
    using namespace tn;
    if (!size_ok(M) || !size_ok(N) || !size_ok(K)) return GEMM_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr || D == nullptr) return GEMM_ERR_INVALID_ARG;
    if (K % 8 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (C != nullptr && !aligned16(C)))
        return GEMM_ERR_ALIGNMENT;
    const uint64_t abytes = uint64_t(M) * uint64_t(K) * 2, bbytes = uint64_t(N) * uint64_t(K) * 2;
    const uint64_t dbytes = uint64_t(M) * uint64_t(N) * 2;
    if (overlaps(D, dbytes, A, abytes) || overlaps(D, dbytes, B, bbytes) || !c_d_ok(C, D, dbytes))
        return GEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    gemm_status_t st = device_info(&dev, &sms);
    if (st != GEMM_OK) return st;
    return launch_gemm_f16_noalloc(M, N, K, A, B, C, D, stream, sms, dev);
}

// Checks shared by the BF16 and FP8 calls: elem_bytes per operand element, bf16 C / D.
static gemm_status_t check_dense(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C,
                                 void* D, int elem_bytes) {
    using namespace tn;
    if (!size_ok(M) || !size_ok(N) || !size_ok(K)) return GEMM_ERR_INVALID_ARG;
    if (A == nullptr || B == nullptr || D == nullptr) return GEMM_ERR_INVALID_ARG;
    if ((K * elem_bytes) % 16 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (C != nullptr && !aligned16(C)))
        return GEMM_ERR_ALIGNMENT;
    const uint64_t abytes = uint64_t(M) * uint64_t(K) * elem_bytes, bbytes = uint64_t(N) * uint64_t(K) * elem_bytes;
    const uint64_t dbytes = uint64_t(M) * uint64_t(N) * 2;
    if (overlaps(D, dbytes, A, abytes) || overlaps(D, dbytes, B, bbytes) || !c_d_ok(C, D, dbytes))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

gemm_status_t gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                        cudaStream_t stream) {
    using namespace tn;
    gemm_status_t st = check_dense(M, N, K, A, B, C, D, 2);
    if (st != GEMM_OK) return st;
    int dev = 0, sms = 0;
    st = device_info(&dev, &sms);
    if (st != GEMM_OK) return st;
    return launch_gemm_bf16(M, N, K, A, B, C, D, stream, sms, dev);
}

gemm_status_t gemm_fp8(int64_t M, int64_t N, int64_t K, const void* A, const void* B, const void* C, void* D,
                       int fmt, cudaStream_t stream) {
    using namespace tn;
    if (fmt != GEMM_FP8_E4M3 && fmt != GEMM_FP8_E5M2) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_dense(M, N, K, A, B, C, D, 1);
    if (st != GEMM_OK) return st;
    int dev = 0, sms = 0;
    st = device_info(&dev, &sms);
    if (st != GEMM_OK) return st;
    return launch_gemm_fp8(M, N, K, A, B, C, D, fmt, stream, sms, dev);
}

gemm_status_t gemm_block_scaled(int64_t M, int64_t N, int64_t K, const void* A, const void* SFA, const void* B,
                                const void* SFB, const void* C, void* D, int fmt, cudaStream_t stream) {
    using namespace tn;
    if (!size_ok(M) || !size_ok(N) || !size_ok(K)) return GEMM_ERR_INVALID_ARG;
    if (A == nullptr || SFA == nullptr || B == nullptr || SFB == nullptr || D == nullptr)
        return GEMM_ERR_INVALID_ARG;
    if (fmt != GEMM_FMT_NVFP4 && fmt != GEMM_FMT_MXFP8) return GEMM_ERR_INVALID_ARG;
    const int64_t kblk = fmt == GEMM_FMT_NVFP4 ? 16 : 32;
    if (K % kblk != 0) return GEMM_ERR_INVALID_ARG;  // K must be whole scale blocks
    // Every scale row (K / kblk bytes) must be whole 16-byte chunks.
    if ((K / kblk) % 16 != 0 || N % 8 != 0) return GEMM_ERR_ALIGNMENT;
    if (!aligned16(A) || !aligned16(SFA) || !aligned16(B) || !aligned16(SFB) || !aligned16(D) ||
        (C != nullptr && !aligned16(C)))
        return GEMM_ERR_ALIGNMENT;
    const uint64_t row = fmt == GEMM_FMT_NVFP4 ? uint64_t(K) / 2 : uint64_t(K);
    const uint64_t sfrow = uint64_t(K / kblk);
    const uint64_t dbytes = uint64_t(M) * uint64_t(N) * 2;
    if (overlaps(D, dbytes, A, uint64_t(M) * row) || overlaps(D, dbytes, B, uint64_t(N) * row) ||
        overlaps(D, dbytes, SFA, uint64_t(M) * sfrow) || overlaps(D, dbytes, SFB, uint64_t(N) * sfrow) ||
        !c_d_ok(C, D, dbytes))
        return GEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    gemm_status_t st = device_info(&dev, &sms);
    if (st != GEMM_OK) return st;
    return launch_gemm_block_scaled(M, N, K, A, SFA, B, SFB, C, D, fmt, stream, sms, dev);
}

const char* gemm_status_string(gemm_status_t status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: a size, enum or pointer argument is out of range";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: the current device is not compute capability 10.3";
        case GEMM_ERR_ALIGNMENT: return "GEMM_ERR_ALIGNMENT: a pointer or row pitch is not 16-byte aligned";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA runtime or driver call failed";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT: a kernel abandoned a pipeline wait past its time limit";
    }
    return "unknown gemm_status_t";
}

gemm_status_t gemm_last_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    const unsigned int a = tn::read_clear_error_f16();
    const unsigned int b = tn::read_clear_error_block_scaled();
    const unsigned int c = tn::read_clear_error_dense();
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    return (a | b | c) ? GEMM_ERR_TIMEOUT : GEMM_OK;
}

}  // extern "C"
