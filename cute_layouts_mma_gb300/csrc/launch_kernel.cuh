// Launch of one kernel configuration: persistent grid sized to the device, a
// (2,1,1) cluster for CTA-pair configurations.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include "dispatch.h"
#include "gemm_kernel.cuh"
#include "launch.h"

namespace tn {

// Scratch of a stream-K launch: fp32 partial sums and per-warp flags.
template <class Cfg>
constexpr size_t sk_partial_bytes(int units) {
    return static_cast<size_t>(units) * Cfg::PAIR * Cfg::BM * Cfg::BN * sizeof(float);
}
template <class Cfg>
constexpr size_t sk_flag_bytes(int units) {
    return (static_cast<size_t>(units) * Cfg::PAIR * Cfg::EPI_WARPS * sizeof(unsigned int) + 255) & ~size_t(255);
}

// Per-device stream-ordered pool the stream-K scratch is taken from (memory stays
// with the pool between calls; each call's block is returned on its stream).
cudaMemPool_t scratch_pool(int dev);

// Device address of a file-scope __device__ variable of the calling translation
// unit on device `dev` (the current device), looked up once per device and kept in
// `cache`; null if the lookup fails.
template <class T>
T* device_symbol(const T& symbol, std::atomic<uintptr_t> (&cache)[kMaxDevices], int dev) {
    uintptr_t a = cache[dev].load(std::memory_order_acquire);
    if (a == 0) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, symbol) != cudaSuccess) return nullptr;
        a = reinterpret_cast<uintptr_t>(ptr);
        cache[dev].store(a, std::memory_order_release);
    }
    return reinterpret_cast<T*>(a);
}

// Read a device error word of the current device and clear it if set (synchronous).
inline unsigned int read_clear_word(const unsigned int& word) {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, word, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(word, &zero, sizeof(zero));
    return v;
}

// Per-device, per-configuration launch state, set up on first use.
template <class Cfg>
struct LaunchState {
    static std::atomic<int> max_units[kMaxDevices];  // resident CTAs (PAIR=1) or clusters (PAIR=2)
};
template <class Cfg>
std::atomic<int> LaunchState<Cfg>::max_units[kMaxDevices];

using dispatch::Schedule;

// The schedule-relevant shape of an instance.
template <class Cfg>
constexpr dispatch::TileShape tile_shape() {
    return dispatch::TileShape{Cfg::BM_TILE, Cfg::BN, Cfg::PAIR, Cfg::kStreamK};
}

template <class Cfg>
Schedule choose_schedule(const Params& p, int max_units) {
    return dispatch::choose_schedule(static_cast<long long>(p.num_m_blocks) * p.num_n_blocks, p.num_k_blocks,
                                     max_units, Cfg::kStreamK);
}

template <class Cfg>
cudaError_t prepare_launch(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], int sms, int dev,
                           cudaStream_t stream, int* units_out) {
    auto kernel = tn_gemm_kernel<Cfg>;
    cfg = cudaLaunchConfig_t{};
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    if (Cfg::PAIR == 2) {
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = 2;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    int units = LaunchState<Cfg>::max_units[dev].load(std::memory_order_acquire);
    if (units == 0) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if constexpr (Cfg::kRegDrain) {
            // The warpgroups' register increases are met only by the decreases and the
            // launch's own allocation: the kernel must be launched with 128 registers
            // per thread (512 threads x 128 = the SM's 65536), or they would wait forever.
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            if (fa.numRegs != 128 || Cfg::THREADS * 128 != 65536) return cudaErrorInvalidConfiguration;
        }
        units = sms;
        if (Cfg::PAIR == 2) {
            cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
            if (e != cudaSuccess) return e;
            units = clusters > 0 ? clusters : sms / 2;
        }
        LaunchState<Cfg>::max_units[dev].store(units, std::memory_order_release);
    }
    *units_out = units;
    return cudaSuccess;
}

// Grid, stream-K fields of `p` and the programmatic-dependent-launch attribute for
// one launch: the kernel's set-up may overlap the previous launch on the stream;
// it waits (griddepcontrol.wait) before touching global memory.
template <class Cfg>
Schedule apply_schedule(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], Params& p, int units) {
    const Schedule sc = choose_schedule<Cfg>(p, units);
    cfg.gridDim = dim3(sc.units * Cfg::PAIR, 1, 1);
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
    p.sk_tiles = sc.sk_tiles;
    p.sk_total = static_cast<long long>(sc.sk_tiles) * p.num_k_blocks;
    p.ws = nullptr;
    p.flags = nullptr;
    return sc;
}

template <class Cfg>
cudaError_t launch_config(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const CUtensorMap& td, const CUtensorMap& tc, Params p,
                          int sms, int dev, cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    int units = 0;
    cudaError_t e = prepare_launch<Cfg>(cfg, attr, sms, dev, stream, &units);
    if (e != cudaSuccess) return e;
    const Schedule sc = apply_schedule<Cfg>(cfg, attr, p, units);
    if (sc.sk_tiles == 0) return cudaLaunchKernelEx(&cfg, tn_gemm_kernel<Cfg>, ta, tb, tsa, tsb, td, tc, p);
    // Stream-K scratch: taken from the device's stream-ordered pool for this call
    // and returned on the same stream after the kernel.
    const size_t pbytes = sk_partial_bytes<Cfg>(sc.units), fbytes = sk_flag_bytes<Cfg>(sc.units);
    void* scratch = nullptr;
    e = cudaMallocFromPoolAsync(&scratch, pbytes + fbytes, scratch_pool(dev), stream);
    if (e != cudaSuccess) return e;
    p.ws = static_cast<float*>(scratch);
    p.flags = reinterpret_cast<unsigned int*>(static_cast<char*>(scratch) + pbytes);
    e = cudaMemsetAsync(p.flags, 0, fbytes, stream);
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, tn_gemm_kernel<Cfg>, ta, tb, tsa, tsb, td, tc, p);
    const cudaError_t f = cudaFreeAsync(scratch, stream);
    return e != cudaSuccess ? e : f;
}

// Same launch, but the stream-K scratch is the caller's fixed block `scratch` of
// `capacity` bytes (256-byte aligned) instead of a pool allocation: nothing is
// allocated or freed.  A split launch whose partials and flags would not fit is
// refused with GEMM_ERR_INVALID_ARG before anything is enqueued.  The block's
// flags are cleared on `stream` before the kernel; its partials need no clearing
// (each is written before its flag is raised).
template <class Cfg>
gemm_status_t launch_config_fixed_scratch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                                          const CUtensorMap& tc, Params p, int sms, int dev, cudaStream_t stream,
                                          void* scratch, size_t capacity) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    int units = 0;
    if (prepare_launch<Cfg>(cfg, attr, sms, dev, stream, &units) != cudaSuccess) return GEMM_ERR_CUDA;
    const Schedule sc = apply_schedule<Cfg>(cfg, attr, p, units);
    if (sc.sk_tiles != 0) {
        const size_t pbytes = sk_partial_bytes<Cfg>(sc.units), fbytes = sk_flag_bytes<Cfg>(sc.units);
        if (scratch == nullptr || pbytes + fbytes > capacity) return GEMM_ERR_INVALID_ARG;
        p.ws = static_cast<float*>(scratch);
        p.flags = reinterpret_cast<unsigned int*>(static_cast<char*>(scratch) + pbytes);
        if (cudaMemsetAsync(p.flags, 0, fbytes, stream) != cudaSuccess) return GEMM_ERR_CUDA;
    }
    return cudaLaunchKernelEx(&cfg, tn_gemm_kernel<Cfg>, ta, tb, ta, tb, td, tc, p) == cudaSuccess ? GEMM_OK
                                                                                               : GEMM_ERR_CUDA;
}

}  // namespace tn
