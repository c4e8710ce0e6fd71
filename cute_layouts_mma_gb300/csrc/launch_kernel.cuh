// Launch of one kernel configuration: a persistent grid sized to the device (a
// (2,1,1) cluster per CTA pair for the pair configurations), or, for the cluster
// split, one (s,1,1) cluster per output tile.
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
    // co-resident clusters of s CTAs (s = 2 .. kMaxSplit) for the cluster split; 0 = not queried
    static std::atomic<int> resident[kMaxDevices][dispatch::kMaxSplit + 1];
};
template <class Cfg>
std::atomic<int> LaunchState<Cfg>::max_units[kMaxDevices];
template <class Cfg>
std::atomic<int> LaunchState<Cfg>::resident[kMaxDevices][dispatch::kMaxSplit + 1];

using dispatch::Schedule;
static_assert(dispatch::kMaxSplit == kMaxClusterSplit, "one largest cluster split");

// The schedule-relevant shape of an instance.
template <class Cfg>
constexpr dispatch::TileShape tile_shape() {
    return dispatch::TileShape{Cfg::BM_TILE, Cfg::BN, Cfg::PAIR, Cfg::kStreamK};
}

// The rule counts 128-byte k-blocks (kSub of them per stage); the schedule itself
// deals stages.
template <class Cfg>
Schedule choose_schedule(const Params& p, int max_units) {
    return dispatch::choose_schedule(static_cast<long long>(p.num_m_blocks) * p.num_n_blocks,
                                     p.num_k_blocks * Cfg::kSub, max_units, Cfg::kStreamK);
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

// Co-resident clusters of s CTAs of the instance on device `dev` (the current
// device), s = 1 .. kMaxSplit: res[1] = one CTA per SM, res[s] from the occupancy
// calculator for a (s,1,1) cluster launch; queried once per device.  A single-CTA
// instance only (the cluster split).
template <class Cfg>
cudaError_t split_capacity(int sms, int dev, int (&res)[dispatch::kMaxSplit + 1]) {
    static_assert(Cfg::PAIR == 1, "cluster split of single-CTA tiles");
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    int units = 0;
    cudaError_t e = prepare_launch<Cfg>(cfg, attr, sms, dev, nullptr, &units);
    if (e != cudaSuccess) return e;
    res[0] = 0;
    res[1] = units;
    for (int s = 2; s <= dispatch::kMaxSplit; ++s) {
        int n = LaunchState<Cfg>::resident[dev][s].load(std::memory_order_acquire);
        if (n == 0) {
            cudaLaunchAttribute a[1];
            a[0].id = cudaLaunchAttributeClusterDimension;
            a[0].val.clusterDim.x = static_cast<unsigned>(s);
            a[0].val.clusterDim.y = 1;
            a[0].val.clusterDim.z = 1;
            cfg.attrs = a;
            cfg.numAttrs = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(s * (sms / s)), 1, 1);
            e = cudaOccupancyMaxActiveClusters(&n, tn_gemm_kernel<Cfg>, &cfg);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();
                n = -1;  // this cluster size cannot be launched: never chosen
            }
            if (n == 0) n = -1;
            LaunchState<Cfg>::resident[dev][s].store(n, std::memory_order_release);
        }
        res[s] = n > 0 ? n : 0;
    }
    return cudaSuccess;
}

// m blocks per raster group for a launch of `units` concurrent tiles: the panels are
// this instance's tile-rows of A and tile-columns of B over the whole K (with their
// scales).
template <class Cfg>
int raster_for(const Params& p, int units) {
    const long long row = static_cast<long long>(p.num_k_blocks) * Cfg::kRowBytes * Cfg::kSub;
    const long long sf = Cfg::KIND == KIND_NVFP4 ? row / 8 : Cfg::KIND == KIND_MXFP8 ? row / 32 : 0;
    return dispatch::raster_group(p.num_m_blocks, p.num_n_blocks, units, Cfg::BM_TILE * (row + sf),
                                  static_cast<long long>(Cfg::BN) * (row + sf));
}

// Programmatic dependent launch: the kernel's set-up may overlap the previous
// launch on the stream; it waits (griddepcontrol.wait) before touching global memory.
inline void add_pdl(cudaLaunchConfig_t& cfg) {
    cfg.attrs[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    cfg.attrs[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
}

// One launch without scratch: whole tiles dealt round robin to persistent units
// (p.split == 1), or every tile given to its own cluster of p.split CTAs that split
// its k-blocks and add their partials through distributed shared memory.
template <class Cfg>
cudaError_t launch_config(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                          const CUtensorMap& td, const CUtensorMap& tc, Params p, int sms, int dev,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    int units = 0;
    cudaError_t e = prepare_launch<Cfg>(cfg, attr, sms, dev, stream, &units);
    if (e != cudaSuccess) return e;
    p.sk_tiles = 0;
    p.sk_total = 0;
    p.ws = nullptr;
    p.flags = nullptr;
    const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
    p.raster_group = raster_for<Cfg>(p, units);
    if (p.split > 1) {
        if (!Cfg::kSplit || p.split > dispatch::kMaxSplit || tiles * p.split > 0x7fffffffLL)
            return cudaErrorInvalidConfiguration;
        cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.split), 1, 1);
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = static_cast<unsigned>(p.split);
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    } else {
        p.split = 1;
        cfg.gridDim = dim3(static_cast<unsigned>((tiles < units ? tiles : units) * Cfg::PAIR), 1, 1);
    }
    add_pdl(cfg);
    return cudaLaunchKernelEx(&cfg, tn_gemm_kernel<Cfg>, ta, tb, tsa, tsb, td, tc, p);
}

// Same launch with the stream-K schedule, whose scratch is the caller's fixed block
// `scratch` of `capacity` bytes (256-byte aligned): nothing is allocated or freed.  A
// split launch whose partials and flags would not fit is refused with
// GEMM_ERR_INVALID_ARG before anything is enqueued.  The block's flags are cleared on
// `stream` before the kernel; its partials need no clearing (each is written before
// its flag is raised).
template <class Cfg>
gemm_status_t launch_config_fixed_scratch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                                          const CUtensorMap& tc, Params p, int sms, int dev, cudaStream_t stream,
                                          void* scratch, size_t capacity) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    int units = 0;
    if (prepare_launch<Cfg>(cfg, attr, sms, dev, stream, &units) != cudaSuccess) return GEMM_ERR_CUDA;
    const Schedule sc = choose_schedule<Cfg>(p, units);
    cfg.gridDim = dim3(sc.units * Cfg::PAIR, 1, 1);
    p.raster_group = raster_for<Cfg>(p, units);
    add_pdl(cfg);
    p.split = 1;
    p.sk_tiles = sc.sk_tiles;
    p.sk_total = static_cast<long long>(sc.sk_tiles) * p.num_k_blocks;
    p.ws = nullptr;
    p.flags = nullptr;
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
