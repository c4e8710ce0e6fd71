// Launch of one kernel configuration: persistent grid sized to the device, a
// (2,1,1) cluster for CTA-pair configurations.
#pragma once

#include <atomic>

#include "gemm_kernel.cuh"
#include "launch.h"

namespace tn {

// Per-device, per-configuration launch state, set up on first use.
template <class Cfg>
struct LaunchState {
    static std::atomic<int> max_units[kMaxDevices];  // resident CTAs (PAIR=1) or clusters (PAIR=2)
};
template <class Cfg>
std::atomic<int> LaunchState<Cfg>::max_units[kMaxDevices];

template <class Cfg>
cudaError_t launch_config(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                          const CUtensorMap& tsb, const CUtensorMap& td, const CUtensorMap& tc, const Params& p,
                          int sms, int dev, cudaStream_t stream) {
    auto kernel = tn_gemm_kernel<Cfg>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    if (Cfg::PAIR == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    int units = LaunchState<Cfg>::max_units[dev].load(std::memory_order_acquire);
    if (units == 0) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (Cfg::PAIR == 2) {
            cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
            if (e != cudaSuccess) return e;
            units = clusters > 0 ? clusters : sms / 2;
        } else {
            units = sms;
        }
        LaunchState<Cfg>::max_units[dev].store(units, std::memory_order_release);
    }
    const int tiles = p.num_m_blocks * p.num_n_blocks;
    const int used = tiles < units ? tiles : units;
    cfg.gridDim = dim3(used * Cfg::PAIR, 1, 1);
    return cudaLaunchKernelEx(&cfg, kernel, ta, tb, tsa, tsb, td, tc, p);
}

}  // namespace tn
