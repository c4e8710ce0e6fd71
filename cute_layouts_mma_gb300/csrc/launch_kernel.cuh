// Launch of one kernel configuration: persistent grid sized to the device, a
// (2,1,1) cluster for CTA-pair configurations.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace tn {

// Stream-K is used when whole tiles would leave more than three quarters of the
// units idle, each unit's share is at least kStreamKMinShare k-blocks, and the
// accumulation is fp32.  Outside that range, measurement on GB300 favoured whole
// tiles: once a quarter of the SMs stream operands, skinny problems are bound by
// HBM rather than by SM count; dense FP16 runs at the power limit, where idle SMs
// raise the clock of the busy ones; and short shares leave each split tile in many
// pieces whose partials the finishing unit adds one after another.
constexpr double kStreamKMinIdle = 0.75;
constexpr long long kStreamKMinShare = 12;

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

// Schedule of one launch: units used and how many tiles (the last ones) are split.
struct Schedule {
    int units;
    int sk_tiles;
};

template <class Cfg>
Schedule choose_schedule(const Params& p, int max_units) {
    const long long tiles = static_cast<long long>(p.num_m_blocks) * p.num_n_blocks;
    Schedule sc{static_cast<int>(tiles < max_units ? tiles : max_units), 0};
    if (!Cfg::kStreamK) return sc;
    const long long rounds = (tiles + max_units - 1) / max_units;
    const double idle = 1.0 - static_cast<double>(tiles) / static_cast<double>(rounds * max_units);
    if (idle <= kStreamKMinIdle) return sc;
    const long long split = tiles % max_units;  // the tiles of the last, partly idle round
    if (split * p.num_k_blocks < kStreamKMinShare * max_units) return sc;
    return Schedule{max_units, static_cast<int>(split)};
}

// Launch configuration shared by every launch of Cfg: block, shared memory, stream,
// the (2,1,1) cluster of CTA pairs.  On first use per device it sets the kernel's
// shared-memory attribute and finds the units (resident CTAs, or clusters for
// PAIR = 2) the device keeps at once.
// Whether Cfg's own schedule would split tiles for this problem (units estimated
// as one per SM, or one per SM pair).  The launchers then switch to their
// 128-column instance: half as many pieces per split tile and half the partial
// bytes per piece, which measured 1.2-1.8x faster on such skinny problems.
template <class Cfg>
bool would_split(int64_t M, int64_t N, int64_t K, int k_per_block, int sms) {
    Params q{};
    q.num_m_blocks = static_cast<int>((M + Cfg::BM_TILE - 1) / Cfg::BM_TILE);
    q.num_n_blocks = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    q.num_k_blocks = static_cast<int>((K + k_per_block - 1) / k_per_block);
    return choose_schedule<Cfg>(q, Cfg::PAIR == 2 ? sms / 2 : sms).sk_tiles != 0;
}

// Dense kinds: CTA pairs (256 x 256 tiles) once their tiles fill every SM pair at least
// once; below that the single-CTA instances (128 x 256, or 128 x 128 with stream-K, or
// 128 x 64) spread the work over twice as many units.  Measured on GB300 (FP16, no C):
// 512 x 8192 x 2048 14.5 -> 13.7 us, 2048^2 x 1024 10.0 -> 9.1, 256 x 2048 x 8192
// 26.5 -> 22.7; 4096^2 x 1024 (256 pair tiles) stays on pairs (24.0 against 26.5).
inline bool use_pairs(int64_t M, int64_t N, int sms) {
    return M > 128 && ((M + 255) / 256) * ((N + 255) / 256) >= sms / 2;
}

// Small problems: whole tiles of `Big` (256 columns; CTA pairs for M > 128) would keep
// fewer than half of the units busy, K is short (at most 1024) and no stream-K split
// applies.  Such a launch is bound by each CTA's operand loads and its fixed latency,
// so the launchers switch to 128 x 64 tiles on single CTAs: many more CTAs, each
// loading a fraction of the bytes (FP16 256^3: 5.3 -> 3.7 us per call on GB300).
// Long K keeps the big tiles: an N = 64 MMA is too short for the single issuing
// thread to keep the tensor pipe busy.
template <class Big>
bool use_small_tiles(int64_t M, int64_t N, int64_t K, int k_per_block, int sms) {
    if (K > 1024) return false;
    const int64_t tiles = ((M + Big::BM_TILE - 1) / Big::BM_TILE) * ((N + Big::BN - 1) / Big::BN);
    const int units = Big::PAIR == 2 ? sms / 2 : sms;
    return 2 * tiles < units && !would_split<Big>(M, N, K, k_per_block, sms);
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
