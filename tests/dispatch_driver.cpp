// Test driver for the launchers' instance choice (cute_layouts_mma_gb300/csrc/dispatch.h):
// for each problem on the command line prints
//   <dense choice of the fixed-scratch call> <whether that instance splits tiles with
//   stream-K> <block-scaled pair choice> <dense choice of gemm_f16 / gemm_bf16 /
//   gemm_fp8> <its cluster split> <cluster split of the block-scaled single-CTA
//   instance> <raster group of the 256 x 256 pair tiles>
// The co-resident cluster counts are a model of a device of 8 equal GPCs: a cluster of
// s single-CTA tiles (one CTA per SM) fits floor((sms / 8) / s) times in each.
//
//   dispatch_driver <sms> <M> <N> <K> <k_per_block> [<M> <N> <K> <k_per_block> ...]
#include <cstdio>
#include <cstdlib>

#include "dispatch.h"

using namespace tn::dispatch;

int main(int argc, char** argv) {
    if (argc < 6 || (argc - 2) % 4 != 0) {
        std::fprintf(stderr, "usage: %s sms (M N K k_per_block)...\n", argv[0]);
        return 2;
    }
    const int sms = std::atoi(argv[1]);
    int res[kMaxSplit + 1];
    res[0] = 0;
    for (int s = 1; s <= kMaxSplit; ++s) res[s] = 8 * ((sms / 8) / s);
    for (int i = 2; i + 3 < argc; i += 4) {
        const long long M = std::atoll(argv[i]), N = std::atoll(argv[i + 1]), K = std::atoll(argv[i + 2]);
        const int kpb = std::atoi(argv[i + 3]);
        const DenseChoice c = dense_choice(M, N, K, kpb, sms);
        const TileShape t = c == DENSE_PAIR_256     ? kDensePair256
                            : c == DENSE_SINGLE_64  ? kDenseSingle64
                            : c == DENSE_SINGLE_128 ? kDenseSingle128
                                                    : kDenseSingle256;
        const DensePlan plan = dense_plan(M, N, K, kpb, sms, res, res);
        const int bs_split = choose_split(tile_count(M, N, kDenseSingle128), static_cast<int>((K + kpb - 1) / kpb), sms, res);
        const long long row = ((K + kpb - 1) / kpb) * 128;
        const int group = raster_group((M + 255) / 256, (N + 255) / 256, sms / 2, 256 * row, 256 * row);
        std::printf("%d %d %d %d %d %d %d\n", static_cast<int>(c), would_split(M, N, K, kpb, sms, t) ? 1 : 0,
                    use_block_scaled_pair(M, N, sms) ? 1 : 0, static_cast<int>(plan.choice), plan.split, bs_split,
                    group);
    }
    return 0;
}
