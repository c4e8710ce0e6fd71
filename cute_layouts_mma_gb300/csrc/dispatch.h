// Instance choice of the launchers: which tile shape and schedule a problem gets.
// Host-only and free of CUDA types, so that the CPU tests can hold the rules
// against the table of measured choices without a GPU.  The launchers
// (gemm_f16.cu, gemm_dense.cu, gemm_bs.cu, launch_kernel.cuh) call these with the
// constants of their kernel instances.
#pragma once

#include <cstdint>

namespace tn {
namespace dispatch {

// Stream-K is used when whole tiles would leave more than three quarters of the
// units idle, each unit's share is at least kStreamKMinShare k-blocks, and the
// accumulation is fp32.  Outside that range, measurement on GB300 favoured whole
// tiles: once a quarter of the SMs stream operands, skinny problems are bound by
// HBM rather than by SM count; dense FP16 runs at the power limit, where idle SMs
// raise the clock of the busy ones; and short shares leave each split tile in many
// pieces whose partials the finishing unit adds one after another.
constexpr double kStreamKMinIdle = 0.75;
constexpr long long kStreamKMinShare = 12;

// The shape of an instance's output tiles, as far as the schedule is concerned.
struct TileShape {
    int bm_tile;    // output rows per tile (128, or 256 for a CTA pair)
    int bn;         // output columns per tile
    int pair;       // CTAs per tile (1 or 2)
    bool stream_k;  // the instance can split tiles (fp32 partials)
};

// Schedule of one launch: units used and how many tiles (the last ones) are split.
struct Schedule {
    int units;
    int sk_tiles;
};

inline Schedule choose_schedule(long long tiles, int num_k_blocks, int max_units, bool stream_k) {
    Schedule sc{static_cast<int>(tiles < max_units ? tiles : max_units), 0};
    if (!stream_k || tiles <= 0) return sc;
    const long long rounds = (tiles + max_units - 1) / max_units;
    const double idle = 1.0 - static_cast<double>(tiles) / static_cast<double>(rounds * max_units);
    if (idle <= kStreamKMinIdle) return sc;
    const long long split = tiles % max_units;  // the tiles of the last, partly idle round
    if (split * num_k_blocks < kStreamKMinShare * max_units) return sc;
    return Schedule{max_units, static_cast<int>(split)};
}

inline long long tile_count(int64_t M, int64_t N, const TileShape& t) {
    return ((M + t.bm_tile - 1) / t.bm_tile) * ((N + t.bn - 1) / t.bn);
}

inline int units_of(const TileShape& t, int sms) { return t.pair == 2 ? sms / 2 : sms; }

// Whether an instance's own schedule would split tiles for this problem (units
// estimated as one per SM, or one per SM pair).
inline bool would_split(int64_t M, int64_t N, int64_t K, int k_per_block, int sms, const TileShape& t) {
    const int nkb = static_cast<int>((K + k_per_block - 1) / k_per_block);
    return choose_schedule(tile_count(M, N, t), nkb, units_of(t, sms), t.stream_k).sk_tiles != 0;
}

// Dense kinds: CTA pairs (256 x 256 tiles) once their tiles fill every SM pair at least
// once, or at least half of the SM pairs when K >= 2048; below that the single-CTA
// instances spread the work over twice as many units.  A single CTA loads 48 KB of
// operands per 128-byte k-block against 32 KB per CTA of a pair, so long-K problems
// favour pairs even with a few SM pairs idle.  Measured on GB300 (FP16, no C):
// 2048^2 x 4096 (64 pair tiles) 27.2 -> 24.4 us and 512 x 8192 x 2048 17.5 -> 15.7 us on
// pairs, but 2048^2 x 1024 9.4 -> 9.8 us, so short K keeps single CTAs; 4096^2 x 1024
// (256 pair tiles) runs on pairs.
inline bool use_pairs(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    return M > 128 && (pair_tiles >= sms / 2 || (K >= 2048 && 2 * pair_tiles >= sms / 2));
}

// Small problems: whole tiles of `big` would keep fewer than half of the units busy,
// K is short (at most 1024) and no stream-K split applies.  Such a launch is bound by
// each CTA's operand loads and its fixed latency, so the launchers switch to 128 x 64
// tiles on single CTAs: many more CTAs, each loading a fraction of the bytes (FP16
// 256^3: 5.3 -> 3.7 us per call on GB300).  Long K keeps the big tiles: an N = 64 MMA
// is too short for the single issuing thread to keep the tensor pipe busy.
inline bool use_small_tiles(int64_t M, int64_t N, int64_t K, int k_per_block, int sms, const TileShape& big) {
    if (K > 1024) return false;
    return 2 * tile_count(M, N, big) < units_of(big, sms) && !would_split(M, N, K, k_per_block, sms, big);
}

// Tile shapes of the dense instances (FP16 with fp32 accumulation, BF16, FP8), K > 32.
constexpr TileShape kDensePair256{256, 256, 2, true};
constexpr TileShape kDenseSingle256{128, 256, 1, true};
constexpr TileShape kDenseSingle128{128, 128, 1, true};
constexpr TileShape kDenseSingle64{128, 64, 1, true};

enum DenseChoice { DENSE_PAIR_256 = 0, DENSE_SINGLE_256 = 1, DENSE_SINGLE_128 = 2, DENSE_SINGLE_64 = 3 };

// CTA pairs when their tiles fill every SM pair; otherwise single CTAs: 128 x 64 tiles
// for small problems, the 128-column instance where the 256-column one would split.
// (The stream-K rule of the fixed-scratch call; dense_plan below is the rule of the
// calls that split tiles inside clusters.)
inline DenseChoice dense_choice(int64_t M, int64_t N, int64_t K, int k_per_block, int sms) {
    if (use_pairs(M, N, K, sms)) return DENSE_PAIR_256;
    if (use_small_tiles(M, N, K, k_per_block, sms, kDenseSingle256)) return DENSE_SINGLE_64;
    return would_split(M, N, K, k_per_block, sms, kDenseSingle256) ? DENSE_SINGLE_128 : DENSE_SINGLE_256;
}

// ------------------------------------------------------------------ cluster split
// A problem whose whole tiles fit one round of the device but leave more than half
// of its SMs idle gives each tile to a cluster of s single CTAs (s <= kMaxSplit, the
// portable cluster size): CTA r of the cluster sums k-blocks [r*nkb/s, (r+1)*nkb/s)
// of the tile, and the cluster adds its s fp32 partials through distributed shared
// memory.  The split is the largest s that keeps every CTA at least kSplitMinShare
// k-blocks, puts at most one CTA on each SM, and lets every tile's cluster be
// resident at once (resident[s]: co-resident clusters of s CTAs of the instance).
constexpr int kMaxSplit = 8;
constexpr int kSplitMinShare = 4;
constexpr double kSplitMinIdle = 0.5;

inline int choose_split(long long tiles, int nkb, int sms, const int* resident) {
    if (tiles <= 0 || tiles > sms) return 1;
    if (1.0 - static_cast<double>(tiles) / sms <= kSplitMinIdle) return 1;
    int best = 1;
    for (int s = 2; s <= kMaxSplit; ++s) {
        if (static_cast<long long>(nkb) < static_cast<long long>(s) * kSplitMinShare) break;
        if (tiles * s > sms) break;
        if (tiles <= resident[s]) best = s;
    }
    return best;
}

// Operand bytes one CTA of a single-CTA instance loads per k-block (128 bytes of K per
// operand row), and the fp32 partial tile a cluster split adds up.
inline long long kblock_bytes(int bn) { return 128LL * (128 + bn); }
inline long long partial_bytes(int bn) { return 128LL * bn * 4; }

// Estimated per-SM bytes of a single-CTA plan: the operand bytes of every round of
// whole tiles (or of one CTA's share of a split tile), plus, for a split, the partial
// tile written and read back through shared memory.  Single-CTA tiles are bound by
// the bytes each SM pulls from L2, so the plan with the fewest bytes per SM is taken.
inline long long plan_bytes(long long tiles, int nkb, int bn, int split, int sms) {
    if (split > 1) return ((nkb + split - 1) / split) * kblock_bytes(bn) + partial_bytes(bn);
    const long long rounds = (tiles + sms - 1) / sms;
    return rounds * nkb * kblock_bytes(bn);
}

struct DensePlan {
    DenseChoice choice;
    int split;  // cluster size of the split (1 = whole tiles)
};

// The dense instance and split for a problem: CTA pairs when their tiles fill every SM
// pair; 128 x 64 single-CTA tiles for small problems (K <= 1024 and the 128 x 256 tiles
// would keep fewer than half of the SMs busy: 1024^3 FP16 7.0 us against 12.6 us split
// in clusters); otherwise whichever of the
// 128 x 256 and 128 x 128 single-CTA instances, each with its own cluster split,
// moves the fewest bytes per SM, the 128 x 128 bytes weighted by 3/4 (below).  res256 / res128: resident
// clusters per cluster size of the two instances.
inline DensePlan dense_plan(int64_t M, int64_t N, int64_t K, int k_per_block, int sms, const int* res256,
                            const int* res128) {
    if (use_pairs(M, N, K, sms)) return DensePlan{DENSE_PAIR_256, 1};
    const int nkb = static_cast<int>((K + k_per_block - 1) / k_per_block);
    const long long t256 = tile_count(M, N, kDenseSingle256), t128 = tile_count(M, N, kDenseSingle128);
    const int s256 = choose_split(t256, nkb, sms, res256);
    const int s128 = choose_split(t128, nkb, sms, res128);
    if (K <= 1024 && 2 * t256 < sms) return DensePlan{DENSE_SINGLE_64, 1};
    const long long b256 = plan_bytes(t256, nkb, 256, s256, sms), b128 = plan_bytes(t128, nkb, 128, s128, sms);
    // The 128 x 128 instance's stages hold two boxes of K (8 MMAs per barrier wait and
    // commit), so it moves its bytes faster: it is taken up to 4/3 of the 128 x 256 bytes
    // (1024^2 x 4096 FP16 13.6 -> 12.6 us, 128 x 8192^2 28.7 -> 26.9 us).
    return 3 * b128 < 4 * b256 ? DensePlan{DENSE_SINGLE_128, s128} : DensePlan{DENSE_SINGLE_256, s256};
}

// ------------------------------------------------------------------ tile raster
// m blocks per raster group (tiles run down a group of m blocks, column by column): the
// largest group, up to kRasterMaxGroup, whose A panels, plus the B panels one wave of
// `units` tiles touches, fit in `budget` bytes of L2.  Then each A panel is read from
// memory about once and each B panel once per group.  a_panel / b_panel: bytes of one
// tile-row of A (and its scales) over the whole K, and of one tile-column of B.  The cap:
// a group of 32 (every m block of NVFP4 8192^3 at once) put 32 concurrent tiles on each
// B panel and ran 188 us against 185 us with 8 or 16 on GB300.
constexpr long long kRasterL2Budget = 64LL << 20;
constexpr int kRasterMaxGroup = 16;

inline int raster_group(long long num_m, long long num_n, long long units, long long a_panel, long long b_panel,
                        long long budget = kRasterL2Budget) {
    int best = 1;
    for (long long g = 1; g <= num_m && g <= kRasterMaxGroup; ++g) {
        const long long wave = units < g * num_n ? units : g * num_n;
        const long long cols = (wave + g - 1) / g + 1;
        if (g * a_panel + cols * b_panel <= budget) best = static_cast<int>(g);
    }
    return best;
}

// Block-scaled kinds: CTA pairs (256 x 256 tiles, whole tiles only) when M > 128 and the
// pair tiles fill at least half of the device's SM pairs; otherwise the single-CTA
// 128 x 128 instances, which also split skinny problems inside clusters.  Measured on
// GB300 (NVFP4 and MXFP8, K = 8192-16384): pairs faster from 40 tiles (1024 x 2560) up,
// single CTAs faster at 32 tiles (512 x 4096) and 16 tiles (256 x 4096).
inline bool use_block_scaled_pair(int64_t M, int64_t N, int sms) {
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    return M > 128 && 2 * pair_tiles >= sms / 2;
}

}  // namespace dispatch
}  // namespace tn
