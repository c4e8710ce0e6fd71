// Persistent, warp-specialised TN GEMM for sm_103a:  D = A x B^T + C  with A (M,K)
// and B (N,K) K-contiguous ("CuTe 中 A、B 如何加载到 MMA 寄存器", section 1), in
// FP16, BF16 or FP8, or in the block-scaled NVFP4 / MXFP8 forms ("数据布局及其记号",
// block-scaled MMA section).
//
// Work is dealt to persistent units (CTAs, or CTA pairs) as whole tiles, round
// robin; for skinny problems that would leave most SMs idle, each tile instead goes
// to a cluster of up to 8 CTAs that split its k-blocks and add their partial sums
// through distributed shared memory (the cluster split, see Params).  A launch
// overlaps the previous one on the stream (programmatic dependent launch): the
// set-up and each role's own bookkeeping run at once, and a thread waits for the
// previous grid (griddepcontrol.wait) only right before its first global-memory
// access -- the TMA issuers before their first load, the epilogue warps before
// theirs; the MMA issuer and the scale writers touch no global memory.
//
// Output tiles are (128 * PAIR) x BN.  With PAIR = 2 the two CTAs of a (2,1,1)
// cluster share a tile: CTA r loads A rows 128r .. 128r+127 and B rows
// (BN/2)r .. (BN/2)(r+1)-1 of the tile into its own shared memory, the leader
// (r = 0) issues one cta_group::2 MMA of 256 x BN per K step over both CTAs'
// operands, and each CTA's TMEM accumulates its own 128 rows x BN.  Per SM this
// halves the B bytes loaded from L2 and read by the tensor core.
//
// Warps of each CTA:
//   warps 0, 2   TMA issuers for A and B: per stage, load this CTA's A (warp 0) and
//                B (warp 2) boxes of kRowBytes of K (128, or 64 / 32 for narrow K;
//                kSub boxes one after the other along K) into swizzled shared memory
//                and arm the leader's `full` barrier with the bytes (PAIR = 2: the
//                peer's copies signal the leader's barrier directly).  A TMA
//                instruction occupies its issuing warp for a few hundred cycles
//                whatever the box size, so each operand stream has its own warp.
//   warp 3       (block-scaled only) issuer of the scale boxes: TMA boxes of the
//                caller's row-major SFA (this CTA's 128 rows) and SFB (the tile's BN
//                rows; in NVFP4 CTA pairs each CTA loads half and multicasts it to
//                both) into the scale slots.
//   warp 1       TMEM allocation; in the leader, the MMA issuer (one thread):
//                tcgen05.mma into a TMEM accumulator, 32 bytes of K per MMA;
//                tcgen05.commit frees the stage (`empty`, in both CTAs) and, at the
//                end of a tile, hands the accumulator to the epilogues
//                (`tmem_full`, in both CTAs).
//   warps 4-7    epilogue (and 12-15 in the register-drain layout): tcgen05.ld
//                of the accumulator (warp w reads TMEM lanes 32*(w%4) .. +31, i.e.
//                rows of the tile), adds any partial sums and C in fp32, rounds
//                once to fp16 / bf16, writes the 32-row chunk to a swizzled
//                shared-memory staging buffer and TMA-stores it (the store clips
//                rows / columns outside D); then releases the accumulator on the
//                leader's `tmem_empty`.  A stream-K piece that does not finish its
//                tile instead writes its fp32 sums to scratch and raises a flag.
//   warps 8-11   (block-scaled only) scale writers, one per TMEM lane quarter:
//                each turns the stage's row-major scale boxes into the 32-lane
//                base tiles the block-scaled MMA reads (local_lane = m % 32,
//                TCol = m // 32, byte = sfk) and writes them with tcgen05.st into
//                its own 32 lanes -- the four quarters together replicate the
//                tile to all four lane partitions -- then arrive on the leader's
//                `full` barrier of the stage, so that the MMA issuer waits on one
//                barrier per stage (a second wait per stage costs the single issuing
//                thread ~200 cycles of its 512-cycle stage).
// Register-drain layout (NVFP4 and MXFP8 CTA pairs): 512 threads, four warpgroups -- 0-3
// issuers and MMA, 4-7 epilogue, 8-11 scale writers, 12-15 epilogue.  setmaxnreg
// moves registers from the first and third to the epilogue warpgroups, so that an
// epilogue warp holds its whole 32 x 128 slice of the accumulator at once.
// Every wait is bounded: past the limit the kernel records a timeout in the
// device error word, makes the other warps give up, drains its in-flight copies
// and MMAs, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "ptx.cuh"

namespace tn {

enum Kind : int {
    KIND_F16_ACC32 = 0,  // FP16 operands, fp32 accumulation, fp16 C / D
    KIND_F16_ACC16 = 1,  // FP16 operands, fp16 accumulation, fp16 C / D
    KIND_NVFP4 = 2,      // block-scaled E2M1 (E4M3 scale per 16), bf16 C / D
    KIND_MXFP8 = 3,      // block-scaled E4M3 (E8M0 scale per 32), bf16 C / D
    KIND_BF16 = 4,       // BF16 operands, fp32 accumulation, bf16 C / D
    KIND_FP8_E4M3 = 5,   // unscaled E4M3 operands, fp32 accumulation, bf16 C / D
    KIND_FP8_E5M2 = 6    // unscaled E5M2 operands, fp32 accumulation, bf16 C / D
};

// C and D are fp16 for the FP16 kinds and bf16 for every other kind.
__host__ __device__ constexpr bool out_is_bf16(int kind) { return kind != KIND_F16_ACC32 && kind != KIND_F16_ACC16; }
// Two-byte operands (64 elements per 128-byte row slice) or one-byte ones (128).
__host__ __device__ constexpr bool operands_16bit(int kind) {
    return kind == KIND_F16_ACC32 || kind == KIND_F16_ACC16 || kind == KIND_BF16;
}
// MMAs without scale factors: kind::f16 (FP16, BF16) or kind::f8f6f4 (FP8).
__host__ __device__ constexpr bool is_dense(int kind) { return kind != KIND_NVFP4 && kind != KIND_MXFP8; }

// Largest cluster of the cluster split (the portable cluster size).
constexpr int kMaxClusterSplit = 8;

// Upper bound on any single pipeline wait; legitimate waits are microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Bound on the waits of the abandon path (in-flight copies / MMAs).
constexpr uint64_t kDrainLimitNs = 200000000ull;

struct Params {
    int M, N, K;
    int num_m_blocks, num_n_blocks, num_k_blocks;
    int raster_group;  // m blocks per raster group of the tile order (tile_coords)
    const void* C;  // [M][N] fp16 (FP16 kinds) or bf16 (block-scaled), or null
    void* D;        // [M][N], same type as C
    unsigned int* err;
    // Stream-K schedule (only with a caller-provided scratch block): the last
    // sk_tiles tiles (in tile order) are split across all units, each taking an
    // equal contiguous share of their (tile, k-block) sequence before its whole
    // tiles.  A tile cut between units is finished by the unit holding its k-block
    // 0 (that piece ends the unit's share); the later pieces, which begin the next
    // units' shares, leave fp32 partial sums in `ws` and raise their flag.  The
    // remaining tiles are dealt whole, round robin.
    int sk_tiles;          // 0: every tile whole
    long long sk_total;    // sk_tiles * num_k_blocks
    float* ws;             // partials: [unit][rank][epilogue warp][chunk][col/4][lane][4]
    unsigned int* flags;   // [unit][rank][epilogue warp]: 1 once that partial is written
    // Cluster split (1 = off): the `split` CTAs of a (split,1,1) cluster share one
    // tile, CTA r of the cluster summing k-blocks [r*nkb/split, (r+1)*nkb/split).
    // Each leaves its fp32 sums in its own shared memory; after a cluster barrier
    // the CTAs add the cluster's partials through distributed shared memory (each
    // CTA a share of the tile's 32-row chunks, the partials in rank order), add C,
    // round once and store.  No global scratch is involved.
    int split;
};

// How the block-scaled kinds move their scale factors (Config::SF_MODE).
//   SF_RING   a ring of SF_SLOTS scale slots of SF_W bytes per row (SF_KB k-blocks), freed
//             by the scale writers once read; the writers wait for the stage's MMAs
//             before storing into its TMEM scale columns.
//   SF_STAGE  one 16-byte slot per stage, refilled once the stage's MMAs are done; the
//             writers wait only for the slot.  In CTA pairs each CTA loads half of the
//             tile's SFB rows and multicasts them to both CTAs.
//   SF_COPY   as SF_STAGE, but the writers repack the slot in shared memory into base
//             tiles and the MMA thread copies them into TMEM with tcgen05.cp.
enum ScaleMode : int { SF_RING = 0, SF_STAGE = 1, SF_COPY = 2 };

enum SegKind : int { SEG_FULL = 0, SEG_PARTIAL = 1, SEG_OWNER = 2, SEG_SPLIT = 3 };

// The work of one unit as a sequence of segments: tile, k blocks [k0, k1), kind.
struct SegIter {
    long long pos, end;  // remaining stream-K share of the split tiles' (tile, k) sequence
    int tile;            // next whole tile (cluster split: the cluster's tile, -1 once taken)
};

__device__ __forceinline__ long long sk_share_begin(const Params& p, int unit, int units) {
    return p.sk_total * unit / units;
}

__device__ __forceinline__ void seg_begin(const Params& p, int unit, int units, SegIter& it) {
    if (p.split > 1) {
        // cluster split (one CTA per unit): CTA r of the cluster takes its k range
        const int r = unit % p.split;
        it.tile = unit / p.split;
        it.pos = static_cast<long long>(p.num_k_blocks) * r / p.split;
        it.end = static_cast<long long>(p.num_k_blocks) * (r + 1) / p.split;
        return;
    }
    it.pos = sk_share_begin(p, unit, units);
    it.end = sk_share_begin(p, unit + 1, units);
    it.tile = unit;
}

// SK = false compiles the whole-tile schedule alone; SPLIT adds the cluster split.
template <bool SK, bool SPLIT>
__device__ __forceinline__ bool seg_next(const Params& p, int units, SegIter& it, int& tile, int& k0, int& k1,
                                         int& kind) {
    if (SPLIT && p.split > 1) {
        if (it.tile < 0) return false;
        tile = it.tile;
        k0 = static_cast<int>(it.pos);
        k1 = static_cast<int>(it.end);
        kind = SEG_SPLIT;
        it.tile = -1;
        return true;
    }
    const int nkb = p.num_k_blocks;
    const int whole_tiles = p.num_m_blocks * p.num_n_blocks - (SK ? p.sk_tiles : 0);
    if (SK && it.pos < it.end) {
        const int t = static_cast<int>(it.pos / nkb);
        tile = whole_tiles + t;
        k0 = static_cast<int>(it.pos - static_cast<long long>(t) * nkb);
        const long long rem = it.end - it.pos;
        k1 = rem < static_cast<long long>(nkb - k0) ? k0 + static_cast<int>(rem) : nkb;
        kind = k0 == 0 ? (k1 == nkb ? SEG_FULL : SEG_OWNER) : SEG_PARTIAL;
        it.pos += k1 - k0;
        return true;
    }
    if (it.tile >= whole_tiles) return false;
    tile = it.tile;
    k0 = 0;
    k1 = nkb;
    kind = SEG_FULL;
    it.tile += units;
    return true;
}

template <int KIND_, int BN_, int STAGES_, int ACC_BUFS_, int EPI_COLS_, int EPI_BUFS_, int PAIR_,
          int EPI_WARPS_ = 4, int ROW_BYTES_ = 128, bool REG_DRAIN_ = false, int SF_MODE_ = 0, int SF_W_ = 16,
          int SF_SLOTS_ = 2, int KSUB_ = 1>
struct Config {
    static constexpr int KIND = KIND_;
    static constexpr int PAIR = PAIR_;  // CTAs per MMA (cta_group)
    static constexpr int BM = 128;      // output rows per CTA
    static constexpr int BM_TILE = BM * PAIR;
    static constexpr int BN = BN_;      // output columns per tile (MMA N)
    static constexpr int BN_CTA = BN / PAIR;  // B rows loaded per CTA
    static constexpr int STAGES = STAGES_;
    static constexpr int ACC_BUFS = ACC_BUFS_;
    // Epilogue staging: each epilogue warp stages 32 rows x EPI_COLS outputs
    // (64 or 128 bytes per row, 64B / 128B swizzle), EPI_BUFS buffers deep.
    static constexpr int EPI_COLS = EPI_COLS_;
    static constexpr int EPI_BUFS = EPI_BUFS_;
    // Stream-K needs fp32 accumulation (partials are fp32 sums); the 8-epilogue-warp
    // (register drain) configuration stays data-parallel.
    static constexpr bool kStreamK = KIND_ != KIND_F16_ACC16 && EPI_WARPS_ == 4;
    static constexpr int EPI_ROW_BYTES = EPI_COLS * 2;
    static constexpr int EPI_BUF_BYTES = 32 * EPI_ROW_BYTES;
    // 4 epilogue warps (warps 4-7), or 8 (also warps 12-15): two per TMEM lane
    // quarter, each draining half of the tile's columns.
    static constexpr int EPI_WARPS = EPI_WARPS_;
    static constexpr int EPI_SPLIT = EPI_WARPS / 4;      // column ranges per lane quarter
    static constexpr int BN_EPI = BN / EPI_SPLIT;         // columns drained by one epilogue warp
    static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "4 or 8 epilogue warps");
    static_assert(EPI_COLS == 32 || EPI_COLS == 64, "staging rows of 64 or 128 bytes");
    static_assert((BN / EPI_SPLIT) % EPI_COLS == 0, "whole staging chunks per epilogue warp");
    // Staging covers a warp's whole 32-row slice of the tile: the accumulator is
    // drained to shared memory and released before any store is issued.
    static constexpr bool kWholeTileStaging = EPI_COLS * EPI_BUFS == BN / EPI_SPLIT;
    // Register drain (block-scaled pairs, 8 epilogue warps, 512 threads = 4 warpgroups):
    // the issuers / MMA warpgroup and the scale writers give up registers
    // (setmaxnreg) so that each epilogue warp takes its whole 32 x 128 slice of the
    // accumulator into registers with one TMEM round trip and releases it at once;
    // rounding, staging (one 64-column buffer) and stores follow.
    static constexpr bool kRegDrain = REG_DRAIN_;
    static_assert(kRegDrain == (EPI_WARPS_ == 8), "8 epilogue warps exactly in the register-drain layout");
    static_assert(!kRegDrain || (EPI_BUFS_ == 1 && 2 * EPI_COLS_ * 2 == BN_),
                  "register drain: two 64-column chunks per warp, one staging buffer");
    // Registers per thread of each warpgroup under kRegDrain (launched with 128):
    // issuers and MMA, epilogue, scale writers, epilogue.  They add up to 4 x 128.
    static constexpr int kRegsIssue = 64, kRegsEpi = 184, kRegsWriter = 80;
    static_assert(kRegsIssue + kRegsWriter + 2 * kRegsEpi == 4 * 128, "register split adds up to the launch's");
    static_assert(PAIR == 1 || PAIR == 2, "one CTA or a CTA pair per MMA");
    static constexpr bool kBlockScaled = (KIND == KIND_NVFP4 || KIND == KIND_MXFP8);
    // warps 0-7 (A issuer, MMA, B issuer, scale loader, epilogue x4), 8-11 scale
    // writers; with kRegDrain warps 12-15 are the second epilogue set.
    static constexpr int THREADS = kRegDrain ? 512 : (kBlockScaled ? 384 : 256);
    // Bytes of K per operand row and stage: 128 (the 128-byte swizzle), or 64 / 32 for
    // problems whose whole K is narrower ("数据布局及其记号", swizzle section: the same
    // hierarchy with 8 x 64-byte and 8 x 32-byte atoms).  32 bytes of K per MMA.
    static constexpr int kRowBytes = ROW_BYTES_;
    static_assert(kRowBytes == 128 || kRowBytes == 64 || kRowBytes == 32, "128-, 64- or 32-byte operand rows");
    static_assert(kRowBytes == 128 || is_dense(KIND_), "block-scaled stages hold 128 bytes of K");
    // A stage holds kSub boxes of kRowBytes of K per operand row (dense kinds only):
    // kSub = 2 halves the MMA thread's barrier wait and commit per MMA, for tiles whose
    // MMAs are short (N = 64).
    static constexpr int kSub = KSUB_;
    static_assert(kSub == 1 || (kSub == 2 && is_dense(KIND_) && ROW_BYTES_ == 128), "two boxes per stage: dense kinds");
    static constexpr int kMmasPerSub = kRowBytes / 32;
    static constexpr int kMmasPerStage = kSub * kMmasPerSub;
    // Elements of K per 128-byte row slice, in TMA coordinates (NVFP4 maps are bytes).
    static constexpr int kKBoxCoord = operands_16bit(KIND) ? kRowBytes / 2 : kRowBytes;  // K of one box
    static constexpr int kKCoordPerStage = kSub * kKBoxCoord;

    static constexpr int A_SUB = BM * kRowBytes;      // one box of A
    static constexpr int B_SUB = BN_CTA * kRowBytes;  // one box of B
    static constexpr int A_BYTES = kSub * A_SUB;
    static constexpr int B_BYTES = kSub * B_SUB;
    static constexpr int SFB_TCOLS = kBlockScaled ? BN / 32 : 0;             // TMEM columns of a tile's SFB
    static_assert(!kBlockScaled || BN % 32 == 0, "block-scaled tiles of whole 32-row scale columns");
    // Scale ring (block-scaled): SF_SLOTS slots, each holding SF_W bytes of every scale
    // row this CTA needs (its 128 SFA rows, the tile's BN SFB rows), i.e. the scales of
    // SF_KB k-blocks (NVFP4: 16 bytes per k-block and row; MXFP8: 4).  One TMA box per
    // matrix fills a slot, so the strided scale rows are fetched SF_W bytes at a time.
    static constexpr int SF_W = kBlockScaled ? SF_W_ : 0;
    static constexpr int SF_SLOTS = kBlockScaled ? SF_SLOTS_ : 0;
    static constexpr int SF_KB = KIND == KIND_NVFP4 ? SF_W_ / 16 : SF_W_ / 4;
    static constexpr int SF_KB_BYTES = KIND == KIND_NVFP4 ? 16 : 4;  // scale bytes per row and k-block
    static_assert(!kBlockScaled || (SF_W_ % 16 == 0 && SF_W_ >= 16 && SF_SLOTS_ >= 1), "16-byte multiple scale boxes");
    // Scale copies (SF_COPY): the pages' tcgen05.cp.32x128b.warpx4 path.  The writers
    // repack the stage's slot in place into 32-lane x 16-byte base tiles (lane l = rows
    // l, l+32, l+64, l+96 of a 128-row group, one word each) and the MMA thread copies
    // the tiles into TMEM, replicated to the four lane partitions, before the stage's
    // MMAs.  Otherwise the writers place the same tiles with tcgen05.st.
    static constexpr int SF_MODE = SF_MODE_;
    static constexpr bool kScaleCp = kBlockScaled && SF_MODE_ == SF_COPY;
    static constexpr bool kStageSlots = kBlockScaled && SF_MODE_ != SF_RING;
    static_assert(!kStageSlots || (SF_W_ == 16 && SF_SLOTS_ == STAGES_), "one 16-byte scale slot per stage");
    // Stage slots in CTA pairs: each CTA loads half of the tile's SFB rows and multicasts
    // them into both CTAs' slots (a slot is free in both CTAs once the stage's MMAs, which
    // signal both CTAs, are done).
    static constexpr bool kSfbMulticast = kStageSlots && PAIR_ == 2;
    static constexpr int SFB_BOX_ROWS = kSfbMulticast ? BN_ / 2 : BN_;
    static constexpr int SFA_BYTES = BM * SF_W;  // per slot
    static constexpr int SFB_BYTES = BN * SF_W;
    static constexpr uint32_t TX_BYTES = PAIR * (A_BYTES + B_BYTES);             // both CTAs' operands

    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + SF_SLOTS * SFA_BYTES;
    static constexpr int OFF_EPI = OFF_SFB + SF_SLOTS * SFB_BYTES;  // 1024-byte aligned
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
    // barriers: full[S], empty[S], sf_full[R], sf_empty[R], tmem_full[ACC], tmem_empty[ACC], drain,
    // c_load[EPI_WARPS][EPI_BUFS]
    static constexpr int BAR_FULL = 0;
    static constexpr int BAR_EMPTY = STAGES;
    static constexpr int BAR_SFFULL = 2 * STAGES;                // [scale slot]: boxes landed
    static constexpr int BAR_SFEMPTY = BAR_SFFULL + SF_SLOTS;     // [scale slot]: writers done with it
    static constexpr int BAR_TFULL = BAR_SFEMPTY + SF_SLOTS;
    static constexpr int BAR_TEMPTY = BAR_TFULL + ACC_BUFS;
    static constexpr int BAR_DRAIN = BAR_TEMPTY + ACC_BUFS;
    static constexpr int BAR_CLOAD = BAR_DRAIN + 1;  // [epilogue warp][staging buffer]: C chunk landed
    static constexpr int NUM_BARS = BAR_CLOAD + EPI_WARPS * EPI_BUFS;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // TMEM base address, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack for 1024-byte alignment

    // TMEM (per CTA): ACC_BUFS accumulators of BN fp32 columns, then the scale slots.
    static constexpr int SF_COL0 = ACC_BUFS * BN;
    static constexpr int SF_COLS_PER_COPYSET = 4 + SFB_TCOLS;  // SFA tile (TCol = m // 32) + SFB (n // 32)
    static constexpr int SF_COLS_PER_STAGE =
        KIND == KIND_NVFP4 ? kMmasPerStage * SF_COLS_PER_COPYSET
                           : (KIND == KIND_MXFP8 ? SF_COLS_PER_COPYSET : 0);
    static constexpr int TMEM_USED = SF_COL0 + STAGES * SF_COLS_PER_STAGE;
    static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                     : TMEM_USED <= 64  ? 64
                                     : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256
                                                        : 512;
    static_assert(TMEM_USED <= 512, "TMEM holds 512 columns");
    static_assert(SMEM_BYTES <= 232448, "227 KB of dynamic shared memory per CTA");
    static_assert(BN % (16 * PAIR) == 0 && BN >= 16 && BN <= 256, "MMA N: multiple of 16 (32 for a pair), <= 256");
    static_assert(B_BYTES % 1024 == 0, "B stages stay 1024-byte aligned");
    static_assert(OFF_EPI % 1024 == 0, "staging buffers start on a swizzle-atom boundary");
    // Cluster split (Params::split > 1): single CTAs, 4 epilogue warps, fp32
    // accumulation, 128-byte operand rows.  After the mainloop the operand stages are
    // idle and hold the CTA's fp32 partial tile, [quarter][chunk][col/4][lane][4].
    // Each CTA receives, in its idle operand stages, one fp32 slot of 32 rows x EPI_COLS
    // per (owned chunk, source CTA): at most (4 * BN / EPI_COLS + kMaxClusterSplit - 1) slots.
    static constexpr bool kSplit = PAIR == 1 && EPI_WARPS_ == 4 && KIND_ != KIND_F16_ACC16 && ROW_BYTES_ == 128;
    static_assert(!kSplit || (4 * BN / EPI_COLS + kMaxClusterSplit - 1) * 32 * EPI_COLS * 4 <= STAGES * (A_BYTES + B_BYTES),
                  "the pushed partials fit the operand stages");
};

// Output tile -> (m block, n block).  Tiles run down groups of `group` m blocks
// (column by column within a group), so that the tiles in flight at one time share
// a few A panels and B panels in L2; the host picks the group so that one wave's
// panels fit in L2.  Odd groups sweep the columns backwards, so that a group starts
// on the B panels its predecessor read last, while they are still in L2.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int& mb, int& nb) {
    const int per_group = group * num_n;
    const int g = tile / per_group;
    const int first_m = g * group;
    const int gs = min(num_m - first_m, group);
    const int r = tile - g * per_group;
    mb = first_m + r % gs;
    nb = (g & 1) ? num_n - 1 - r / gs : r / gs;
}

// Bounded parity wait.  Returns false (and stops the other warps) after the
// time limit, or as soon as another warp has given up.  kCluster: acquire at
// cluster scope (the barrier receives arrivals from the peer CTA).
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* err) {
    auto poll = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (poll()) return true;
        if ((i & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, 1u);
                return false;
            }
        }
    }
}

// Bounded wait used only while abandoning work.
__device__ __forceinline__ void wait_bar_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainLimitNs) return;
    }
}

// Bounded pause used while abandoning work when completions cannot be observed.
__device__ __forceinline__ void pause_ns(uint64_t ns) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) {
    }
}

// Accumulator column -> fp32 value.  FP16 accumulation keeps one element per
// 32-bit TMEM column, in the low 16 bits.
template <int KIND>
__device__ __forceinline__ float acc_value(uint32_t r) {
    if constexpr (KIND == KIND_F16_ACC16) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(r & 0xFFFFu)));
    } else {
        return __uint_as_float(r);
    }
}

template <int KIND>
__device__ __forceinline__ void unpack8(uint4 v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (out_is_bf16(KIND)) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        } else {
            const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            const float2 x = __half22float2(h);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
}

template <int KIND>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (out_is_bf16(KIND)) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        } else {
            const __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Accumulator columns c .. c+COLS-1 of this warp's 32 TMEM lanes into r (issue only;
// the caller waits with tmem_ld_wait).
template <int COLS>
__device__ __forceinline__ void load_chunk(uint32_t tacc, int c, uint32_t* r) {
    tmem_ld_32x32b_x32(tacc + static_cast<uint32_t>(c), *reinterpret_cast<uint32_t(*)[32]>(r));
    if constexpr (COLS == 64)
        tmem_ld_32x32b_x32(tacc + static_cast<uint32_t>(c + 32), *reinterpret_cast<uint32_t(*)[32]>(r + 32));
}

// One thread's share of an epilogue chunk: output row `lane` of a 32-row x COLS
// chunk, 16-byte output vectors v0 .. v0+NV-1 (8 values each) from the accumulator
// words r[8v .. 8v+7].  With kCStaged the staging buffer already holds the matching
// C chunk (TMA-loaded with the D tensor map's swizzle; zero outside C); the thread
// adds its values in fp32, rounds once and writes the result back in place: 16-byte
// vector j of row l lives at vector j ^ f(l), the XOR swizzle the D tensor map uses.
template <int KIND, int COLS, int NV, bool kCStaged>
__device__ __forceinline__ void stage_vectors(const uint32_t* r, uint8_t* buf, int lane, int v0) {
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        uint4* slot = reinterpret_cast<uint4*>(buf + layout::swizzled_offset(COLS * 2, lane, 16 * (v0 + v)));
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = acc_value<KIND>(r[8 * v + i]);
        if constexpr (kCStaged) {
            float c[8];
            unpack8<KIND>(*slot, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] += c[i];
        }
        *slot = pack8<KIND>(f);
    }
}

// The whole row: columns 0 .. COLS-1 of the chunk from r[0 .. COLS-1].
template <int KIND, int COLS, bool kCStaged>
__device__ __forceinline__ void stage_chunk(const uint32_t* r, uint8_t* buf, int lane) {
    stage_vectors<KIND, COLS, COLS / 8, kCStaged>(r, buf, lane, 0);
}

// Scale-factor writer for one TMEM lane quarter.  The k-block's scales sit in a scale
// slot row-major: row r at raw + r * ROW holds the SF_KB_BYTES scale bytes of that row
// for this k-block (NVFP4: 16 = four per MMA; MXFP8: 4 = one per MMA).  Lane l of the
// warp (TMEM lane 32q + l) receives, for each copy set j, the base-tile row l: SFA
// scales of rows l, l+32, l+64, l+96 in columns 0..3 (TCol = m // 32, the four scales
// of the MMA in bytes 0..3, byte = sfk), then the SFB scales of rows l + 32c in columns
// 4 + c ("数据布局及其记号", block-scaled section).  NVFP4 has one copy set per MMA (word
// j of each row = that MMA's 4 scales); MXFP8 has one copy set per stage (each row's
// word = the stage's 4 scales, one per MMA, picked by the MMA's scale-factor ID).  Every
// quarter writes the same values: together the four warps replicate the tile to the
// four lane partitions.
template <int KIND, int SFB_TCOLS, int ROW>
__device__ __forceinline__ void write_scales(const uint8_t* raw_a, const uint8_t* raw_b, int lane, uint32_t taddr) {
    constexpr int SET = 4 + SFB_TCOLS;  // SFA columns (128 rows) + SFB columns (BN rows)
    if constexpr (KIND == KIND_NVFP4) {
        uint32_t R[SET][4];
#pragma unroll
        for (int c = 0; c < SET; ++c) {
            const uint8_t* src = (c < 4) ? raw_a + layout::sf_row(lane, c) * ROW : raw_b + layout::sf_row(lane, c - 4) * ROW;
            const uint4 x = *reinterpret_cast<const uint4*>(src);
            R[c][0] = x.x;
            R[c][1] = x.y;
            R[c][2] = x.z;
            R[c][3] = x.w;
        }
        uint32_t out[4 * SET];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < SET; ++c) out[j * SET + c] = R[c][j];
        static_assert((4 * SET) % 16 == 0, "whole 16-column stores");
#pragma unroll
        for (int i = 0; i < (4 * SET) / 16; ++i)
            tmem_st_32x32b_x16(taddr + 16 * i, *reinterpret_cast<const uint32_t(*)[16]>(&out[16 * i]));
    } else {
        uint32_t out[SET];
#pragma unroll
        for (int c = 0; c < SET; ++c) {
            const uint8_t* src = (c < 4) ? raw_a + layout::sf_row(lane, c) * ROW : raw_b + layout::sf_row(lane, c - 4) * ROW;
            out[c] = *reinterpret_cast<const uint32_t*>(src);
        }
        tmem_st_32x32b_x8(taddr, *reinterpret_cast<const uint32_t(*)[8]>(&out[0]));
        if constexpr (SET == 12) tmem_st_32x32b_x4(taddr + 8, *reinterpret_cast<const uint32_t(*)[4]>(&out[8]));
        static_assert(SET == 8 || SET == 12, "one SFA tile and one or two SFB tiles per stage");
    }
}

// Stream-K partial slot of one epilogue warp: 32 rows x BN_EPI fp32 sums laid out
// [chunk][col/4][lane][4], so that a warp's float4 accesses are 512 contiguous bytes.
template <class Cfg>
__device__ __forceinline__ float4* partial_slot(const Params& p, int unit, uint32_t rank, int e) {
    const size_t idx = (static_cast<size_t>(unit) * Cfg::PAIR + rank) * Cfg::EPI_WARPS + e;
    return reinterpret_cast<float4*>(p.ws) + idx * (32 * Cfg::BN_EPI / 4);
}

template <class Cfg>
__device__ __forceinline__ unsigned int* partial_flag(const Params& p, int unit, uint32_t rank, int e) {
    return p.flags + (static_cast<size_t>(unit) * Cfg::PAIR + rank) * Cfg::EPI_WARPS + e;
}

// Wait (lane 0 of the warp, bounded) until a peer unit has published its partial.
__device__ __forceinline__ bool wait_flag(const unsigned int* f, volatile int* abort_flag, unsigned int* err) {
    const uint64_t t0 = global_timer_ns();
    while (ld_acquire_gpu(f) != 1u) {
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(err, 1u);
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tn_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmC,
                   const Params p) {
    constexpr int KIND = Cfg::KIND;
    constexpr int PAIR = Cfg::PAIR;
    constexpr int BN = Cfg::BN;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int ACC_BUFS = Cfg::ACC_BUFS;
    constexpr bool kBS = Cfg::kBlockScaled;
    constexpr bool kPair = PAIR == 2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;  // 0 = leader
    const bool leader = rank == 0;
    const int cluster = static_cast<int>(blockIdx.x) / PAIR;
    const int num_clusters = static_cast<int>(gridDim.x) / PAIR;

    auto bar = [&](int i) -> uint32_t { return sbase + Cfg::OFF_BAR + 8 * i; };
    // the leader's copy of barrier i, as seen from this CTA
    auto leader_bar = [&](int i) -> uint32_t { return kPair ? mapa_shared(bar(i), 0u) : bar(i); };
    volatile uint32_t* tmem_base_slot = reinterpret_cast<volatile uint32_t*>(smem + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // the leader's A and B issuers, and (block-scaled) every scale-writer warp
            mbar_init(bar(Cfg::BAR_FULL + s), 2 + (kBS ? 4 * PAIR : 0));
            mbar_init(bar(Cfg::BAR_EMPTY + s), 1);
        }
        for (int r = 0; r < Cfg::SF_SLOTS; ++r) {
            mbar_init(bar(Cfg::BAR_SFFULL + r), 1);   // the scale loader (SFA and SFB boxes)
            mbar_init(bar(Cfg::BAR_SFEMPTY + r), 4);  // the four scale-writer warps
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            mbar_init(bar(Cfg::BAR_TFULL + b), 1);
            mbar_init(bar(Cfg::BAR_TEMPTY + b), Cfg::EPI_WARPS * PAIR);  // one arrival per epilogue warp
        }
        mbar_init(bar(Cfg::BAR_DRAIN), 1);
        for (int i = 0; i < Cfg::EPI_WARPS * Cfg::EPI_BUFS; ++i) mbar_init(bar(Cfg::BAR_CLOAD + i), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
        if (p.C != nullptr) tma_prefetch_desc(&tmC);
        if constexpr (kBS) {
            tma_prefetch_desc(&tmSFA);
            tma_prefetch_desc(&tmSFB);
        }
    }
    if (warp == 1) {
        if constexpr (kPair) {
            tmem_alloc_pair(sbase + Cfg::OFF_MISC, Cfg::TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(sbase + Cfg::OFF_MISC, Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before_sync();
    if constexpr (kPair)
        cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA signal
    else
        __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_base_slot;
    // The set-up above touched only this CTA's own shared memory, TMEM and parameters,
    // so it may overlap the end of the previous launch on the stream (launched with
    // programmatic stream serialization).  Global memory is touched only after the
    // previous grid has completed: each thread that reads or writes it waits for that
    // (griddep_wait) right before its first access, so that the roles' own set-up --
    // the first tile's coordinates, the code and parameters it fetches, ~1600 cycles
    // on a cold SM -- also overlaps the previous launch.  The next launch may start
    // its own set-up now.
    griddep_launch_dependents();

    // ------------------------------------------------------------------ TMA issuers
    // role 0: A, 1: B.  Each waits for its stage slot to be released by the MMAs that
    // last read it, arms the leader's `full` barrier with its bytes and issues one box.
    auto issue_loop = [&](const int role) {
        int s = 0;
        uint32_t ph = 0;
        uint32_t loads[STAGES];
#pragma unroll
        for (int i = 0; i < STAGES; ++i) loads[i] = 0;
        bool ok = true;
        SegIter it;
        seg_begin(p, cluster, num_clusters, it);
        int tile, k0, k1, kind;
        bool first_seg = true;
        bool dep_done = false;
        // L2 policy of the boxes: an A panel serves every tile of its m block, so it is
        // kept (evict_last); with a single row of tiles each B panel is read once, so it
        // goes first.  Otherwise B is left to the default policy.
        const bool hinted = role == 0 || p.num_m_blocks == 1;
        const uint64_t policy = role == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
        while (ok && seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind)) {
            int mb, nb;
            tile_coords(tile, p.num_m_blocks, p.num_n_blocks, p.raster_group, mb, nb);
            const int m0 = mb * Cfg::BM_TILE + static_cast<int>(rank) * Cfg::BM;  // this CTA's A rows
            const int n0 = nb * BN + static_cast<int>(rank) * Cfg::BN_CTA;        // this CTA's B rows
            for (int kb = k0; kb < k1; ++kb) {
                if (!wait_bar(bar(Cfg::BAR_EMPTY + s), ph ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
#ifdef TN_TIMEOUT_INJECT
                // Test build only: CTA 0's A issuer withholds its first stage, so the
                // MMA thread's bounded wait on that stage runs out.
                if (role == 0 && blockIdx.x == 0 && first_seg && kb == k0) {
                    ++loads[s];
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    continue;
                }
#endif
                if (!dep_done) {  // first global access of this thread
                    griddep_wait();
                    dep_done = true;
                }
                const int kx = kb * Cfg::kKCoordPerStage;
                const uint32_t dst =
                    role == 0 ? sbase + Cfg::OFF_A + s * Cfg::A_BYTES : sbase + Cfg::OFF_B + s * Cfg::B_BYTES;
                const CUtensorMap* map = role == 0 ? &tmA : &tmB;
                const int y = role == 0 ? m0 : n0;
                const uint32_t bytes = PAIR * (role == 0 ? Cfg::A_BYTES : Cfg::B_BYTES);
                const uint32_t sub_bytes = role == 0 ? Cfg::A_SUB : Cfg::B_SUB;
                if constexpr (kPair) {
                    if (leader) mbar_arrive_expect_tx(bar(Cfg::BAR_FULL + s), bytes);
                } else {
                    mbar_arrive_expect_tx(bar(Cfg::BAR_FULL + s), bytes);
                }
#pragma unroll
                for (int j = 0; j < Cfg::kSub; ++j) {
                    const uint32_t dj = dst + j * sub_bytes;
                    const int xj = kx + j * Cfg::kKBoxCoord;
                    if constexpr (kPair) {
                        if (hinted)
                            tma_load_2d_pair_hint(dj, map, leader_bar(Cfg::BAR_FULL + s), xj, y, policy);
                        else
                            tma_load_2d_pair(dj, map, leader_bar(Cfg::BAR_FULL + s), xj, y);
                    } else {
                        if (hinted)
                            tma_load_2d_hint(dj, map, bar(Cfg::BAR_FULL + s), xj, y, policy);
                        else
                            tma_load_2d(dj, map, bar(Cfg::BAR_FULL + s), xj, y);
                    }
                }
                ++loads[s];
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            first_seg = false;
        }
        (void)kind;
        (void)first_seg;
        if (ok && role == 0) {
            // Wait until the MMAs have released every stage, so that no
            // tcgen05.commit arrival is still in flight when the CTA exits.
            for (int i = 0; i < STAGES && ok; ++i) {
                ok = wait_bar(bar(Cfg::BAR_EMPTY + s), ph ^ 1u, abort_flag, p.err);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) {
            // Abandoning: let every issued TMA copy land before the CTA exits.
            for (int i = 0; i < STAGES; ++i) {
                if (loads[i] == 0) continue;
                if (!kPair || leader) wait_bar_drain(bar(Cfg::BAR_FULL + i), (loads[i] - 1u) & 1u);
            }
            // the peer's operand copies signal the leader's barriers: give them time
            if (kPair) pause_ns(kDrainLimitNs / 4);
        }
    };

    // ------------------------------------------------------------------ scale loader
    // (block-scaled only) Lane 0 of one warp.  A segment's k-blocks fall into groups of
    // SF_KB (the absolute k-block / SF_KB); for each group the segment touches, one
    // scale slot is filled with a TMA box of the caller's row-major SFA (SF_W bytes x
    // this CTA's 128 rows) and one of SFB (SF_W bytes x the tile's BN rows), unswizzled;
    // rows past M or N and bytes past the row end read as zero.  A slot is refilled
    // once the four scale writers have read it.
    auto scale_loop = [&]() {
        if constexpr (kBS) {
            constexpr int R = Cfg::SF_SLOTS;
            int r = 0;
            uint32_t ph = 0;
            uint32_t loads[R];
#pragma unroll
            for (int i = 0; i < R; ++i) loads[i] = 0;
            bool ok = true;
            SegIter it;
            seg_begin(p, cluster, num_clusters, it);
            int tile, k0, k1, kind;
            bool dep_done = false;
            while (ok && seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind)) {
                int mb, nb;
                tile_coords(tile, p.num_m_blocks, p.num_n_blocks, p.raster_group, mb, nb);
                const int m0 = mb * Cfg::BM_TILE + static_cast<int>(rank) * Cfg::BM;  // this CTA's SFA rows
                const int nb0 = nb * BN;                                              // the tile's SFB rows
                // stage slots: slot r = stage, refilled once the stage's MMAs are done, with
                // the 16-byte box of k-block kb (MXFP8: the box holding it); ring: one box
                // per group of SF_KB k-blocks the segment touches
                const int g_end = Cfg::kStageSlots ? k1 : (k1 + Cfg::SF_KB - 1) / Cfg::SF_KB;
                for (int g = Cfg::kStageSlots ? k0 : k0 / Cfg::SF_KB; g < g_end; ++g) {
                    const uint32_t free_bar = Cfg::kStageSlots ? bar(Cfg::BAR_EMPTY + r) : bar(Cfg::BAR_SFEMPTY + r);
                    if (!wait_bar(free_bar, ph ^ 1u, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    if (!dep_done) {  // first global access of this thread
                        griddep_wait();
                        dep_done = true;
                    }
                    const int x = Cfg::kStageSlots ? (KIND == KIND_NVFP4 ? g : (g >> 2)) * 16 : g * Cfg::SF_W;
                    const uint32_t sb = bar(Cfg::BAR_SFFULL + r);
                    mbar_arrive_expect_tx(sb, (Cfg::BM + BN) * Cfg::SF_W);  // all that lands in this CTA
                    tma_load_2d(sbase + Cfg::OFF_SFA + r * Cfg::SFA_BYTES, &tmSFA, sb, x, m0);
                    if constexpr (Cfg::kSfbMulticast) {
                        const int half = static_cast<int>(rank) * Cfg::SFB_BOX_ROWS;  // this CTA's half of SFB
                        tma_load_2d_multicast(sbase + Cfg::OFF_SFB + r * Cfg::SFB_BYTES + half * Cfg::SF_W, &tmSFB, sb, x,
                                              nb0 + half, 0x3);
                    } else {
                        tma_load_2d(sbase + Cfg::OFF_SFB + r * Cfg::SFB_BYTES, &tmSFB, sb, x, nb0);
                    }
                    ++loads[r];
                    if (++r == R) {
                        r = 0;
                        ph ^= 1u;
                    }
                }
            }
            (void)kind;
            if (!ok) {
                // Abandoning: let every issued scale box land before the CTA exits.
                for (int i = 0; i < R; ++i)
                    if (loads[i] != 0) wait_bar_drain(bar(Cfg::BAR_SFFULL + i), (loads[i] - 1u) & 1u);
            }
        }
    };

    // ------------------------------------------------------------------ roles
    auto mma_role = [&]() {
        if (lane == 0 && leader) {
            // ---------------------------------------------------------- MMA issuer
            // One thread issues every MMA; each tcgen05 instruction costs it tens of
            // cycles, so the loop keeps its own bookkeeping incremental (no divisions)
            // and the shared-memory descriptors precomputed.
            constexpr uint32_t kM = 128 * PAIR;
            // descriptor of stage 0; stage s adds s * (bytes / 16) to the start address
            const uint64_t adesc0 = layout::umma_smem_desc_kmajor(sbase + Cfg::OFF_A, Cfg::kRowBytes);
            const uint64_t bdesc0 = layout::umma_smem_desc_kmajor(sbase + Cfg::OFF_B, Cfg::kRowBytes);
            // scale tiles (copy mode): 32 rows x 16 bytes, row after row; +32 per 512-byte tile
            const uint64_t sfa_desc0 = layout::umma_smem_desc_noswizzle(sbase + Cfg::OFF_SFA, 128, 128);
            const uint64_t sfb_desc0 = layout::umma_smem_desc_noswizzle(sbase + Cfg::OFF_SFB, 128, 128);
            // copy mode: stage st's base tiles into its TMEM scale columns, replicated to the
            // four lane partitions (SFA to TCol 0-3 of each copy set, the 128-row group h of
            // SFB to TCol 4 + 4h)
            auto issue_scale_copies = [&](int st) {
                if constexpr (Cfg::kScaleCp) {
                    const uint32_t sf_t = tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + st * Cfg::SF_COLS_PER_STAGE);
                    const uint64_t da = sfa_desc0 + static_cast<uint64_t>((st * Cfg::SFA_BYTES) >> 4);
                    const uint64_t db = sfb_desc0 + static_cast<uint64_t>((st * Cfg::SFB_BYTES) >> 4);
                    constexpr int SETS = KIND == KIND_NVFP4 ? 4 : 1;
#pragma unroll
                    for (int j = 0; j < SETS; ++j) {
                        const uint32_t t = sf_t + j * Cfg::SF_COLS_PER_COPYSET;
                        if constexpr (kPair) {
                            tc_cp_32x128b_warpx4_pair(t, da + 32 * j);
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h) tc_cp_32x128b_warpx4_pair(t + 4 + 4 * h, db + 128 * h + 32 * j);
                        } else {
                            tc_cp_32x128b_warpx4(t, da + 32 * j);
#pragma unroll
                            for (int h = 0; h < BN / 128; ++h) tc_cp_32x128b_warpx4(t + 4 + 4 * h, db + 128 * h + 32 * j);
                        }
                    }
                }
            };
            bool cp_ahead = false;  // the current stage's scale copies were issued one stage early
            bool ok = true;
            int s = 0;
            uint32_t ph = 0;
            SegIter it;
            seg_begin(p, cluster, num_clusters, it);
            int tile, k0, k1, kind;
            for (int t_local = 0; ok && seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind); ++t_local) {
                const int buf = (ACC_BUFS == 1) ? 0 : (t_local & 1);
                const uint32_t use = static_cast<uint32_t>(ACC_BUFS == 1 ? t_local : (t_local >> 1));
                if (!wait_bar<kPair>(bar(Cfg::BAR_TEMPTY + buf), (use & 1u) ^ 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
                for (int kb = k0; kb < k1; ++kb) {
                    const bool acc_kb = kb != k0;  // the first k block of a segment starts from 0
                    // Operands landed and (block-scaled) scales written to TMEM.  The dense
                    // kinds' barrier completes through the arrivals of this CTA's issuers and
                    // the transaction bytes of both CTAs' copies, so a CTA-scope wait
                    // suffices (a cluster-scope acquire costs the issuing thread ~4% of the
                    // stage); the scale writers of the peer CTA arrive with cluster scope.
                    if (!wait_bar<kPair && kBS>(bar(Cfg::BAR_FULL + s), ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t adesc = adesc0 + static_cast<uint64_t>(s * (Cfg::A_BYTES >> 4));
                    const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(s * (Cfg::B_BYTES >> 4));
                    if constexpr (is_dense(KIND)) {
                        // MMAs of 32 bytes of K: 16 elements (kind::f16) or 32 (kind::f8f6f4)
                        constexpr uint32_t idesc =
                            idesc_dense(kM, BN, KIND != KIND_F16_ACC16,
                                        (KIND == KIND_BF16 || KIND == KIND_FP8_E5M2) ? 1u : 0u);
#pragma unroll
                        for (int j = 0; j < Cfg::kMmasPerStage; ++j) {
                            // box j / kMmasPerSub of the stage, 32-byte K step j % kMmasPerSub
                            constexpr int kPerSub = Cfg::kMmasPerSub;
                            const uint64_t da = adesc + static_cast<uint64_t>((j / kPerSub) * (Cfg::A_SUB >> 4) + 2 * (j % kPerSub));
                            const uint64_t db = bdesc + static_cast<uint64_t>((j / kPerSub) * (Cfg::B_SUB >> 4) + 2 * (j % kPerSub));
                            if constexpr (operands_16bit(KIND)) {
                                if constexpr (kPair)
                                    mma_f16_pair(d_tmem, da, db, idesc, acc_kb || j != 0);
                                else
                                    mma_f16(d_tmem, da, db, idesc, acc_kb || j != 0);
                            } else {
                                if constexpr (kPair)
                                    mma_f8f6f4_pair(d_tmem, da, db, idesc, acc_kb || j != 0);
                                else
                                    mma_f8f6f4(d_tmem, da, db, idesc, acc_kb || j != 0);
                            }
                        }
                    } else {
                        const uint32_t sf_tmem = tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + s * Cfg::SF_COLS_PER_STAGE);
                        if constexpr (Cfg::kScaleCp) {
                            if (!cp_ahead) issue_scale_copies(s);
                            cp_ahead = false;
                        }
                        if constexpr (KIND == KIND_NVFP4) {
                            constexpr uint32_t idesc = idesc_block_scaled(kM, BN, 1u, false, 0u);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t t = sf_tmem + j * Cfg::SF_COLS_PER_COPYSET;
                                if constexpr (kPair)
                                    mma_mxf4nvf4_4x_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, t, t + 4, acc_kb || j != 0);
                                else
                                    mma_mxf4nvf4_4x(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, t, t + 4, acc_kb || j != 0);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                constexpr uint32_t idesc0 = idesc_block_scaled(kM, BN, 0u, true, 0u);
                                const uint32_t idesc = idesc0 | (static_cast<uint32_t>(j) << 4) | (static_cast<uint32_t>(j) << 29);
                                if constexpr (kPair)
                                    mma_mxf8f6f4_1x_pair(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sf_tmem, sf_tmem + 4,
                                                         acc_kb || j != 0);
                                else
                                    mma_mxf8f6f4_1x(d_tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sf_tmem, sf_tmem + 4,
                                                    acc_kb || j != 0);
                            }
                        }
                    }
                    if constexpr (Cfg::kScaleCp) {
                        // the next stage's scale copies now, if its data is already there: they
                        // then land while this stage's MMAs run
                        const int sn = s + 1 == STAGES ? 0 : s + 1;
                        const uint32_t pn = s + 1 == STAGES ? ph ^ 1u : ph;
                        if (kPair ? mbar_test_wait_cluster(bar(Cfg::BAR_FULL + sn), pn)
                                  : mbar_try_wait(bar(Cfg::BAR_FULL + sn), pn)) {
                            tc_fence_after_sync();
                            issue_scale_copies(sn);
                            cp_ahead = true;
                        }
                    }
                    if constexpr (kPair)
                        tc_commit_pair(bar(Cfg::BAR_EMPTY + s), 0x3);
                    else
                        tc_commit(bar(Cfg::BAR_EMPTY + s));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }

                }
                (void)tile;
                (void)kind;
                if (!ok) break;
                if constexpr (kPair)
                    tc_commit_pair(bar(Cfg::BAR_TFULL + buf), 0x3);
                else
                    tc_commit(bar(Cfg::BAR_TFULL + buf));
            }
            if (!ok) {
                // Abandoning: wait for the MMAs already issued.
                if constexpr (kPair)
                    tc_commit_pair(bar(Cfg::BAR_DRAIN), 0x1);
                else
                    tc_commit(bar(Cfg::BAR_DRAIN));
                wait_bar_drain(bar(Cfg::BAR_DRAIN), 0u);
            }
        }
    };
    auto writer_role = [&]() {
        if constexpr (kBS) {
            // -------------------------------------------------------------- scale writers
            // Per k-block: the scales from the scale slot (waited for at the slot's first
            // k-block of the segment, released to the loader after its last), into the
            // stage's TMEM scale columns once the MMAs that last read those columns have
            // completed; then arrive on the stage's `full` barrier.
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            int s = 0, r = 0;
            uint32_t ph = 0, rph = 0;
            bool ok = true;
            SegIter it;
            seg_begin(p, cluster, num_clusters, it);
            int tile, k0, k1, kind;
            while (ok && Cfg::kScaleCp && seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind)) {
                // copy mode: warp q repacks 128-row group q of the stage's slot in place
                // (group 0: SFA, groups 1 ..: SFB rows 128(q-1) ..) into the base tiles
                // the MMA thread copies: NVFP4 one tile per MMA j (word j of each row),
                // MXFP8 one tile (the stage's word, kb % 4).
                constexpr int GROUPS = 1 + BN / 128;
                uint8_t* grp = q == 0 ? smem + Cfg::OFF_SFA : smem + Cfg::OFF_SFB + (q - 1) * 2048;
                for (int kb = k0; kb < k1; ++kb) {
                    ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_SFFULL + s), ph, abort_flag, p.err));
                    if (!ok) break;
                    if (q < GROUPS) {
                        uint8_t* g = grp + s * (q == 0 ? Cfg::SFA_BYTES : Cfg::SFB_BYTES);
                        uint4 x[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) x[i] = *reinterpret_cast<const uint4*>(g + (lane + 32 * i) * 16);
                        __syncwarp();
                        auto word = [](const uint4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; };
                        if constexpr (KIND == KIND_NVFP4) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                *reinterpret_cast<uint4*>(g + 512 * j + 16 * lane) =
                                    make_uint4(word(x[0], j), word(x[1], j), word(x[2], j), word(x[3], j));
                        } else {
                            const int j = kb & 3;
                            *reinterpret_cast<uint4*>(g + 16 * lane) =
                                make_uint4(word(x[0], j), word(x[1], j), word(x[2], j), word(x[3], j));
                        }
                        fence_proxy_async_smem();  // the tiles are read by tcgen05.cp (async proxy)
                    }
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kPair)
                            mbar_arrive_cluster(leader_bar(Cfg::BAR_FULL + s));  // release: shared-memory data
                        else
                            mbar_arrive(bar(Cfg::BAR_FULL + s));
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            while (ok && Cfg::SF_MODE == SF_STAGE &&
                   seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind)) {
                // stage slots: the slot's load was issued after the stage's previous MMAs
                // completed, so one wait covers both the data and the TMEM columns
                for (int kb = k0; kb < k1; ++kb) {
                    ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_SFFULL + s), ph, abort_flag, p.err));
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int off = KIND == KIND_NVFP4 ? 0 : (kb & 3) * Cfg::SF_KB_BYTES;
                    write_scales<KIND, Cfg::SFB_TCOLS, Cfg::SF_W>(
                        smem + Cfg::OFF_SFA + s * Cfg::SFA_BYTES + off, smem + Cfg::OFF_SFB + s * Cfg::SFB_BYTES + off,
                        lane, lane_base + static_cast<uint32_t>(Cfg::SF_COL0 + s * Cfg::SF_COLS_PER_STAGE));
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kPair)
                            mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_FULL + s));
                        else
                            mbar_arrive(bar(Cfg::BAR_FULL + s));
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            while (ok && Cfg::SF_MODE == SF_RING &&
                   seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind)) {
                for (int kb = k0; kb < k1; ++kb) {
                    const int in_slot = kb % Cfg::SF_KB;
                    if (kb == k0 || in_slot == 0) {
                        ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_SFFULL + r), rph, abort_flag, p.err));
                        if (!ok) break;
                    }
                    ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_EMPTY + s), ph ^ 1u, abort_flag, p.err));
                    if (!ok) break;
                    tc_fence_after_sync();
                    const int off = in_slot * Cfg::SF_KB_BYTES;
                    write_scales<KIND, Cfg::SFB_TCOLS, Cfg::SF_W>(
                        smem + Cfg::OFF_SFA + r * Cfg::SFA_BYTES + off, smem + Cfg::OFF_SFB + r * Cfg::SFB_BYTES + off,
                        lane, lane_base + static_cast<uint32_t>(Cfg::SF_COL0 + s * Cfg::SF_COLS_PER_STAGE));
                    if (kb == k1 - 1 || in_slot == Cfg::SF_KB - 1) {
                        __syncwarp();  // every lane has read the slot
                        if (lane == 0) mbar_arrive(bar(Cfg::BAR_SFEMPTY + r));
                        if (++r == Cfg::SF_SLOTS) {
                            r = 0;
                            rph ^= 1u;
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        // The scales are TMEM data whose writes tcgen05.wait::st has
                        // completed: the leader needs no release of generic memory.
                        if constexpr (kPair)
                            mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_FULL + s));
                        else
                            mbar_arrive(bar(Cfg::BAR_FULL + s));
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    };
    auto epilogue_role = [&]() {
        // -------------------------------------------------------------- epilogue
        griddep_wait();  // C loads and D stores below
        const uint64_t out_policy = l2_policy_evict_first();  // C and D are touched once
        constexpr int EC = Cfg::EPI_COLS;
        constexpr int EB = Cfg::EPI_BUFS;
        const int q = warp & 3;                       // TMEM lane quarter this warp may access
        const int e = warp < 8 ? warp - 4 : warp - 8;  // epilogue warp index (warps 12-15: 4-7)
        const int c_begin = (e >> 2) * Cfg::BN_EPI;    // this warp's columns of the tile
        const int c_end = c_begin + Cfg::BN_EPI;
        uint8_t* stg = smem + Cfg::OFF_EPI + e * (EB * Cfg::EPI_BUF_BYTES);
        const uint32_t stg_u32 = sbase + Cfg::OFF_EPI + e * (EB * Cfg::EPI_BUF_BYTES);
        const bool has_c = p.C != nullptr;
        uint32_t cph = 0;      // bit b: phase of this warp's C-load barrier for buffer b
        uint32_t cpending = 0;  // bit b: a C load into buffer b has not been waited for
        int eb = 0;
        int t_local = 0;
        // C chunk at column nc of rows m_warp.. into staging buffer b (lane 0); the
        // buffer must no longer be read by an earlier store.
        auto load_c = [&](int b, int nc, int m_warp) {
            const uint32_t cb = bar(Cfg::BAR_CLOAD + e * EB + b);
            mbar_arrive_expect_tx(cb, Cfg::EPI_BUF_BYTES);
            tma_load_2d_hint(stg_u32 + b * Cfg::EPI_BUF_BYTES, &tmC, cb, nc, m_warp, out_policy);
            cpending |= 1u << b;
        };
        bool ok = true;
        constexpr bool kSK = Cfg::kStreamK;
        SegIter it;
        seg_begin(p, cluster, num_clusters, it);
        int tile, k0, k1, kind;
        for (; ok && seg_next<Cfg::kStreamK, Cfg::kSplit>(p, num_clusters, it, tile, k0, k1, kind); ++t_local) {
            const int buf = (ACC_BUFS == 1) ? 0 : (t_local % ACC_BUFS);
            const uint32_t use = static_cast<uint32_t>(t_local / ACC_BUFS);
            int mb, nb;
            tile_coords(tile, p.num_m_blocks, p.num_n_blocks, p.raster_group, mb, nb);
            // first output row of this warp
            const int m_warp = mb * Cfg::BM_TILE + static_cast<int>(rank) * Cfg::BM + q * 32;
            const int n0 = nb * BN;
            const bool rows_in = m_warp < p.M;
            if constexpr (Cfg::kSplit) {
                if (kind == SEG_SPLIT) {
                    // Cluster split: the accumulator is pushed to the tile's owners after the
                    // roles (split_push), once every CTA of the cluster is past its mainloop.
                    ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_TFULL + buf), use & 1u, abort_flag, p.err));
                    if (!ok) break;
                    continue;
                }
            }
            if (kSK && kind == SEG_PARTIAL) {
                // A later piece of a tile another unit finishes: publish the fp32 sums.
                ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_TFULL + buf), use & 1u, abort_flag, p.err));
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t tacc =
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
                float4* slot = partial_slot<Cfg>(p, cluster, rank, e);
#pragma unroll 1
                for (int c = c_begin, b = 0; c < c_end; c += EC, ++b) {
                    uint32_t r[EC];
                    load_chunk<EC>(tacc, c, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < EC / 4; ++j)
                        __stcg(slot + (b * (EC / 4) + j) * 32 + lane,
                               make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                           __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
                }
                __threadfence();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_TEMPTY + buf));
                    else
                        mbar_arrive(bar(Cfg::BAR_TEMPTY + buf));
                    st_release_gpu(partial_flag<Cfg>(p, cluster, rank, e), 1u);
                }
                continue;
            }
            // Owner of a cut tile: the units after this one hold its later pieces.
            int first_peer = 0, last_peer = -1;
            if (kSK && kind == SEG_OWNER) {
                first_peer = cluster + 1;
                last_peer = first_peer;
                const int split_index = tile - (p.num_m_blocks * p.num_n_blocks - p.sk_tiles);
                const long long tile_end = static_cast<long long>(split_index + 1) * p.num_k_blocks;
                while (last_peer + 1 < num_clusters && sk_share_begin(p, last_peer + 1, num_clusters) < tile_end)
                    ++last_peer;
                bool got = true;
                if (lane == 0)
                    for (int u = first_peer; u <= last_peer && got; ++u)
                        got = wait_flag(partial_flag<Cfg>(p, u, rank, e), abort_flag, p.err);
                ok = __all_sync(0xffffffffu, __shfl_sync(0xffffffffu, got, 0));
                if (!ok) break;
                __syncwarp();  // orders the lanes' partial reads after lane 0's acquire
            }
            // fp32 sums of the later pieces of this chunk, added to the accumulator
            auto add_partials = [&](uint32_t* r, int b) {
                for (int u = first_peer; u <= last_peer; ++u) {
                    const float4* slot = partial_slot<Cfg>(p, u, rank, e);
#pragma unroll
                    for (int j = 0; j < EC / 4; ++j) {
                        const float4 v = __ldcg(slot + (b * (EC / 4) + j) * 32 + lane);
                        r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + v.x);
                        r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + v.y);
                        r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + v.z);
                        r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + v.w);
                    }
                }
            };
            // C does not depend on the accumulator: fetch it early
            if constexpr (Cfg::kWholeTileStaging) {
                if (rows_in && lane == 0) {
                    bulk_wait_group_read<0>();  // the previous tile's stores have read the buffers
                    if (has_c)
                        for (int c = c_begin, b = 0; c < c_end && n0 + c < p.N; c += EC, ++b) load_c(b, n0 + c, m_warp);
                }
                __syncwarp();
            } else if constexpr (Cfg::kRegDrain) {
                if (rows_in && lane == 0) {
                    bulk_wait_group_read<0>();  // the previous tile's stores have read the buffer
                    if (has_c && n0 + c_begin < p.N) load_c(0, n0 + c_begin, m_warp);
                }
                __syncwarp();
            } else if (has_c && rows_in && lane == 0 && n0 + c_begin < p.N) {
                bulk_wait_group_read<EB - 1>();
                load_c(eb, n0 + c_begin, m_warp);
            }
            ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_TFULL + buf), use & 1u, abort_flag, p.err));
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * BN);
            if constexpr (Cfg::kWholeTileStaging) {
                // Drain every chunk into its own staging buffer, release the
                // accumulator, then store: the MMAs of the next tile wait only for
                // the TMEM reads.
#pragma unroll 1
                for (int c = c_begin, b = 0; c < c_end; c += EC, ++b) {
                    if (n0 + c >= p.N) break;  // warp-uniform
                    uint32_t r[EC];
                    load_chunk<EC>(tacc, c, r);
                    tmem_ld_wait();
                    if (!rows_in) continue;
                    if constexpr (kSK) add_partials(r, b);
                    if (has_c) {
                        ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_CLOAD + e * EB + b), (cph >> b) & 1u,
                                                              abort_flag, p.err));
                        cph ^= 1u << b;
                        cpending &= ~(1u << b);
                        if (!ok) break;
                        stage_chunk<KIND, EC, true>(r, stg + b * Cfg::EPI_BUF_BYTES, lane);
                    } else {
                        stage_chunk<KIND, EC, false>(r, stg + b * Cfg::EPI_BUF_BYTES, lane);
                    }
                }
                if (!ok) break;
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_TEMPTY + buf));
                    else
                        mbar_arrive(bar(Cfg::BAR_TEMPTY + buf));
                }
                if (rows_in) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        for (int c = c_begin, b = 0; c < c_end && n0 + c < p.N; c += EC, ++b)
                            tma_store_2d_hint(&tmD, stg_u32 + b * Cfg::EPI_BUF_BYTES, n0 + c, m_warp, out_policy);
                        bulk_commit_group();
                    }
                }
            } else if constexpr (Cfg::kRegDrain) {
                // The warp's whole slice (BN_EPI fp32 columns) into registers with one
                // wait, release the accumulator, then per 64-column chunk: (C added from
                // the staging buffer) round, stage, TMA-store.
                static_assert(!kSK, "whole tiles only");
                uint32_t r[Cfg::BN_EPI];
#pragma unroll
                for (int h = 0; h < Cfg::BN_EPI / 32; ++h)
                    tmem_ld_32x32b_x32(tacc + static_cast<uint32_t>(c_begin + 32 * h),
                                       *reinterpret_cast<uint32_t(*)[32]>(r + 32 * h));
                tmem_ld_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_TEMPTY + buf));
                    else
                        mbar_arrive(bar(Cfg::BAR_TEMPTY + buf));
                }
                if (rows_in) {
#pragma unroll
                    for (int j = 0; j < Cfg::BN_EPI / EC; ++j) {
                        const int c = c_begin + j * EC;
                        if (n0 + c >= p.N) break;  // warp-uniform
                        if (j > 0) {
                            if (lane == 0) {
                                bulk_wait_group_read<0>();  // the previous chunk's store has read the buffer
                                if (has_c) load_c(0, n0 + c, m_warp);
                            }
                            __syncwarp();
                        }
                        if (has_c) {
                            ok = __all_sync(0xffffffffu,
                                            wait_bar(bar(Cfg::BAR_CLOAD + e * EB), cph & 1u, abort_flag, p.err));
                            cph ^= 1u;
                            cpending = 0;
                            if (!ok) break;
                            stage_chunk<KIND, EC, true>(r + j * EC, stg, lane);
                        } else {
                            stage_chunk<KIND, EC, false>(r + j * EC, stg, lane);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d_hint(&tmD, stg_u32, n0 + c, m_warp, out_policy);
                            bulk_commit_group();
                        }
                    }
                    if (!ok) break;
                }
            } else {
#pragma unroll 1
                for (int c = c_begin, b = 0; c < c_end; c += EC, ++b) {
                    if (n0 + c >= p.N) break;  // warp-uniform
                    uint32_t r[EC];
                    load_chunk<EC>(tacc, c, r);
                    tmem_ld_wait();
                    if (!rows_in) continue;  // no row of this warp lies inside D
                    if constexpr (kSK) add_partials(r, b);
                    const bool more = c + EC < c_end && n0 + c + EC < p.N;
                    if (has_c) {
                        if (EB == 2 && more && lane == 0) {
                            bulk_wait_group_read<0>();  // the other buffer's last store has read it
                            load_c(eb ^ 1, n0 + c + EC, m_warp);
                        }
                        ok = __all_sync(0xffffffffu, wait_bar(bar(Cfg::BAR_CLOAD + e * EB + eb), (cph >> eb) & 1u,
                                                              abort_flag, p.err));
                        cph ^= 1u << eb;
                        cpending &= ~(1u << eb);
                        if (!ok) break;
                        stage_chunk<KIND, EC, true>(r, stg + eb * Cfg::EPI_BUF_BYTES, lane);
                    } else {
                        // the staging buffer is free once the store issued from it has read it
                        if (lane == 0) bulk_wait_group_read<EB - 1>();
                        __syncwarp();
                        stage_chunk<KIND, EC, false>(r, stg + eb * Cfg::EPI_BUF_BYTES, lane);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d_hint(&tmD, stg_u32 + eb * Cfg::EPI_BUF_BYTES, n0 + c, m_warp, out_policy);
                        bulk_commit_group();
                        if (has_c && EB == 1 && more) {
                            bulk_wait_group_read<0>();
                            load_c(eb, n0 + c + EC, m_warp);
                        }
                    }
                    if constexpr (EB == 2) eb ^= 1;
                }
                if (!ok) break;
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)
                        mbar_arrive_cluster_relaxed(leader_bar(Cfg::BAR_TEMPTY + buf));
                    else
                        mbar_arrive(bar(Cfg::BAR_TEMPTY + buf));
                }
            }
        }
        if (lane == 0) {
            // Abandoning: let C loads still in flight land before the CTA exits.
            for (int b = 0; b < EB; ++b)
                if (cpending & (1u << b)) wait_bar_drain(bar(Cfg::BAR_CLOAD + e * EB + b), (cph >> b) & 1u);
            bulk_wait_group_all();
        }
        __syncwarp();
    };
    // Cluster split.  The tile's 32-row x EPI_COLS chunks u = 4g + q (q: lane quarter, g:
    // column chunk) are owned by the cluster's CTAs in turn: chunk u by CTA u % S (S =
    // cluster size), its (u / S)-th.  Each CTA owns at most ceil(UNITS / S) chunks and
    // keeps, in its idle operand stages, one fp32 slot per (owned chunk, source CTA):
    // slot (k, s) at k * S + s, [col/4][lane][4] inside.
    constexpr int UNIT_BYTES = 32 * Cfg::EPI_COLS * 4;
    // split_push (after every CTA of the cluster is past its mainloop), by every warp of
    // the CTA: warp w reads lane quarter w % 4 of the accumulator (the quarter a warp may
    // access) for the column chunks g with g % (warps / 4) == w / 4, and stores each
    // chunk into its owner's slot for this CTA -- through distributed shared memory, or
    // directly when this CTA owns the chunk.
    auto split_push = [&]() {
        if constexpr (Cfg::kSplit) {
            constexpr int EC = Cfg::EPI_COLS;
            constexpr int GROUPS = Cfg::THREADS / 128;  // warps per lane quarter
            const int q = warp & 3;
            const int S = p.split;
            const int r = static_cast<int>(blockIdx.x) % S;
            const int nkb = p.num_k_blocks;
            const bool none = nkb * r / S == nkb * (r + 1) / S;  // an empty k range contributes zeros
            tc_fence_after_sync();
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int g = warp >> 2; g < BN / EC; g += GROUPS) {
                const int u = 4 * g + q;
                const int owner = u % S, k = u / S;
                uint32_t v[EC];
                load_chunk<EC>(tacc, g * EC, v);
                tmem_ld_wait();
                if (none)
#pragma unroll
                    for (int i = 0; i < EC; ++i) v[i] = 0u;
                const uint32_t off = static_cast<uint32_t>(Cfg::OFF_A + (k * S + r) * UNIT_BYTES + lane * 16);
                if (owner == r) {
#pragma unroll
                    for (int i = 0; i < EC / 4; ++i)
                        *reinterpret_cast<uint4*>(smem + off + i * 512) =
                            make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                } else {
                    const uint32_t dst = mapa_shared(sbase + off, static_cast<uint32_t>(owner));
#pragma unroll
                    for (int i = 0; i < EC / 4; ++i)
                        st_shared_cluster_u4(dst + i * 512, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            }
        }
    };
    // split_reduce (after every slot has landed), by every warp of the CTA with a staging
    // buffer: the CTA's owned chunks are cut into P column parts (P = 1, 2 or 4, as many
    // as the warps allow), part j of owned chunk k going to warp kP + j.  Each warp adds
    // its columns of the chunk's S slots in rank order, adds C, rounds once and stages
    // them into the group's buffer; once the P warps of a group have staged (a named
    // barrier), the group's first warp stores the chunk.  With P = 1 each warp takes
    // whole chunks, round robin.
    auto split_reduce = [&]() {
        if constexpr (Cfg::kSplit) {
            constexpr int EC = Cfg::EPI_COLS;
            constexpr int UNITS = 4 * (BN / EC);
            constexpr int NBUF = Cfg::EPI_WARPS * Cfg::EPI_BUFS;  // staging buffers, one C barrier each
            constexpr int NW = (Cfg::THREADS / 32) < NBUF ? (Cfg::THREADS / 32) : NBUF;
            static_assert(NW % 4 == 0, "groups of up to four warps");
            if (warp >= NW) return;
            griddep_wait();  // C loads and D stores (returns at once: the previous grid is done)
            const uint64_t out_policy = l2_policy_evict_first();
            const int S = p.split;
            const int r = static_cast<int>(blockIdx.x) % S;
            const int owned = (UNITS - r + S - 1) / S;  // chunks u = r + kS < UNITS
            int mb, nb;
            tile_coords(static_cast<int>(blockIdx.x) / S, p.num_m_blocks, p.num_n_blocks, p.raster_group, mb, nb);
            const bool has_c = p.C != nullptr;
            auto run = [&](auto parts) {
                constexpr int P = decltype(parts)::value;
                constexpr int W = EC / P;  // columns of a part
                static_assert(W % 8 == 0, "whole 16-byte output vectors");
                const int grp = warp / P, part = warp % P;
                const bool first = part == 0 && lane == 0;  // issues the group's copies
                uint8_t* stg = smem + Cfg::OFF_EPI + grp * Cfg::EPI_BUF_BYTES;
                const uint32_t stg_u32 = sbase + Cfg::OFF_EPI + grp * Cfg::EPI_BUF_BYTES;
                const uint32_t cb = bar(Cfg::BAR_CLOAD + grp);
                uint32_t cph = 0;
                bool ok = *abort_flag == 0;
                // P > 1: owned * P <= NW, one round; P = 1: warp w takes chunks w, w + NW, ...
                for (int k = grp; ok && k < owned; k += NW / P) {
                    const int u = r + k * S;
                    const int q = u & 3, g = u >> 2;
                    const int m_warp = mb * Cfg::BM + q * 32;
                    const int nc = nb * BN + g * EC;
                    if (m_warp >= p.M || nc >= p.N) continue;  // uniform over the group
                    if (first) {
                        bulk_wait_group_read<0>();  // P = 1: the buffer's previous store has read it
                        if (has_c) {
                            mbar_arrive_expect_tx(cb, Cfg::EPI_BUF_BYTES);
                            tma_load_2d_hint(stg_u32, &tmC, cb, nc, m_warp, out_policy);
                        }
                    }
                    __syncwarp();
                    uint32_t acc[W];
#pragma unroll
                    for (int i = 0; i < W; ++i) acc[i] = 0u;  // +0.0f
                    const float4* slot =
                        reinterpret_cast<const float4*>(smem + Cfg::OFF_A + k * S * UNIT_BYTES) + part * (W / 4) * 32 + lane;
                    for (int src = 0; src < S; ++src, slot += UNIT_BYTES / 16) {
#pragma unroll
                        for (int i = 0; i < W / 4; ++i) {
                            const float4 v = slot[i * 32];
                            acc[4 * i] = __float_as_uint(__uint_as_float(acc[4 * i]) + v.x);
                            acc[4 * i + 1] = __float_as_uint(__uint_as_float(acc[4 * i + 1]) + v.y);
                            acc[4 * i + 2] = __float_as_uint(__uint_as_float(acc[4 * i + 2]) + v.z);
                            acc[4 * i + 3] = __float_as_uint(__uint_as_float(acc[4 * i + 3]) + v.w);
                        }
                    }
                    if (has_c) {
                        if constexpr (P == 1) {
                            ok = __all_sync(0xffffffffu, wait_bar(cb, cph, abort_flag, p.err));
                            if (!ok) {
                                if (first) wait_bar_drain(cb, cph);  // the C load lands before the CTA exits
                                break;
                            }
                        } else {
                            // every warp of the group must reach the named barrier below:
                            // a bounded wait that does not give up on the abort flag
                            wait_bar_drain(cb, cph);
                            __syncwarp();
                        }
                        cph ^= 1u;
                        stage_vectors<KIND, EC, W / 8, true>(acc, stg, lane, part * (W / 8));
                    } else {
                        stage_vectors<KIND, EC, W / 8, false>(acc, stg, lane, part * (W / 8));
                    }
                    fence_proxy_async_smem();
                    if constexpr (P > 1)
                        named_bar_sync(1 + grp, 32 * P);
                    else
                        __syncwarp();
                    if (first && *abort_flag == 0) {
                        tma_store_2d_hint(&tmD, stg_u32, nc, m_warp, out_policy);
                        bulk_commit_group();
                    }
                }
                if (first) bulk_wait_group_all();
                __syncwarp();
            };
            if (4 * owned <= NW)
                run(std::integral_constant<int, 4>{});
            else if (2 * owned <= NW)
                run(std::integral_constant<int, 2>{});
            else
                run(std::integral_constant<int, 1>{});
        }
    };

    if constexpr (Cfg::kRegDrain) {
        // Each warpgroup sets its register budget inside its own branch (all four
        // warps execute the same setmaxnreg, and the code after it is compiled to
        // that budget): issuers and MMA, then the scale writers, release registers;
        // the two epilogue warpgroups take them.
        const int wg = warp >> 2;
        if (wg == 0) {
            setmaxnreg_dec<Cfg::kRegsIssue>();
            if (warp == 1)
                mma_role();
            else if (lane == 0)
                warp == 3 ? scale_loop() : issue_loop(warp == 0 ? 0 : 1);
        } else if (wg == 2) {
            setmaxnreg_dec<Cfg::kRegsWriter>();
            writer_role();
        } else {
            setmaxnreg_inc<Cfg::kRegsEpi>();
            epilogue_role();
        }
    } else if (warp == 0 || warp == 2) {
        if (lane == 0) issue_loop(warp == 0 ? 0 : 1);
    } else if (warp == 1) {
        mma_role();
    } else if (kBS && warp == 3) {
        if (lane == 0) scale_loop();
    } else if (warp >= 8 && warp < 12) {
        writer_role();
    } else if (warp >= 4 && warp < 8) {
        epilogue_role();
    }
    __syncwarp();

    // Cluster split: the first barrier frees every CTA's operand stages for the pushed
    // partials (all mainloops are done), the second makes the pushed partials visible
    // to their owners.  No CTA touches another's shared memory after it, so each CTA
    // finishes on its own.
    if constexpr (Cfg::kSplit) {
        if (p.split > 1) {
            fence_proxy_async_smem();
            cluster_sync_all();
            if (*abort_flag == 0) split_push();
            __syncwarp();
            cluster_sync_all();
            split_reduce();
            __syncwarp();
        }
    }

    tc_fence_before_sync();
    if constexpr (kPair)
        cluster_sync_all();  // no CTA leaves while its peer may still signal it or read its memory
    else
        __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        if constexpr (kPair)
            tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace tn
