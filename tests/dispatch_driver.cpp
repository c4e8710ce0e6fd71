// Test driver for the launchers' instance choice (cute_layouts_mma_gb300/csrc/dispatch.h):
// for each problem on the command line prints the dense choice, whether the chosen
// single-CTA instance splits tiles with stream-K, and the block-scaled pair choice.
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
    for (int i = 2; i + 3 < argc; i += 4) {
        const long long M = std::atoll(argv[i]), N = std::atoll(argv[i + 1]), K = std::atoll(argv[i + 2]);
        const int kpb = std::atoi(argv[i + 3]);
        const DenseChoice c = dense_choice(M, N, K, kpb, sms);
        const TileShape t = c == DENSE_PAIR_256     ? kDensePair256
                            : c == DENSE_SINGLE_64  ? kDenseSingle64
                            : c == DENSE_SINGLE_128 ? kDenseSingle128
                                                    : kDenseSingle256;
        std::printf("%d %d %d\n", static_cast<int>(c), would_split(M, N, K, kpb, sms, t) ? 1 : 0,
                    use_block_scaled_pair(M, N, sms) ? 1 : 0);
    }
    return 0;
}
