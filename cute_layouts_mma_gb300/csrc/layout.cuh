// Layout algebra of the two pages, as a header-only C++17 library usable from host
// code and from the kernels (every function is constexpr).
//
//   * "数据布局及其记号" (the data-layout chapter): S[(shape):(strides)] maps a flat
//     index, split with the LAST mode fastest ("Tile Layout" section), to offsets
//     along named axes (@m memory, @TLane/@TCol tensor memory, @laneid/@reg
//     fragments, @gpuid_x/@gpuid_y devices); R[n:s@axis] replicates and O[s@axis]
//     shifts ("Replication 与 Offset"); the block-scaled section places a 128 x 4
//     scale block into a 32-lane TMEM base tile (local_lane = m % 32, TCol = m / 32,
//     byte = sfk) replicated to the four lane quarters; the swizzle section XORs the
//     16-byte sector with the row inside an 8-row x 128-byte atom.
//   * "CuTe 中 A、B 如何加载到 MMA 寄存器": CuTe layouts (shape):(stride) with
//     nested modes whose flat coordinate runs with the FIRST mode fastest; the SM80
//     m16n8k16 thread-value layouts (section 2, section 5), ldmatrix.x4 (section 4),
//     make_fragment_like / make_ordered_layout (section 3 and the source appendix)
//     and retile (section 6).
//
// The kernels take their shared-memory swizzle, UMMA shared-memory descriptor and
// TMEM scale-factor placement from here; the SM80 and device-mesh parts reproduce the
// pages' worked examples and are host-side tools.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define TN_LAYOUT_HD __host__ __device__
#else
#define TN_LAYOUT_HD
#endif

namespace tn {
namespace layout {

// ------------------------------------------------------------------ named axes
enum Axis : int {
    AX_M = 0,      // linear memory
    AX_TLANE = 1,  // tensor-memory lane
    AX_TCOL = 2,   // tensor-memory column
    AX_LANEID = 3, // warp lane of a register fragment
    AX_REG = 4,    // register slot of a fragment
    AX_GPU_X = 5,  // device mesh
    AX_GPU_Y = 6,
    AX_COUNT = 7
};

// One mode of an S[(shape):(strides)] layout: extent, stride and the axis the stride
// runs along.
struct AxisMode {
    int shape;
    int stride;
    int axis;
};

// A point in the named-axis space: one offset per axis.
struct AxisPoint {
    int v[AX_COUNT];
    TN_LAYOUT_HD constexpr int operator[](int a) const { return v[a]; }
};

TN_LAYOUT_HD constexpr AxisPoint axis_origin() { return AxisPoint{{0, 0, 0, 0, 0, 0, 0}}; }

template <int R>
struct AxisLayout {
    AxisMode mode[R];
};

template <int R>
TN_LAYOUT_HD constexpr int size(const AxisLayout<R>& L) {
    int n = 1;
    for (int i = 0; i < R; ++i) n *= L.mode[i].shape;
    return n;
}

// f(coordinate) = sum over modes of coordinate * stride, accumulated per axis.
template <int R>
TN_LAYOUT_HD constexpr AxisPoint eval_coord(const AxisLayout<R>& L, const int (&c)[R]) {
    AxisPoint p = axis_origin();
    for (int i = 0; i < R; ++i) p.v[L.mode[i].axis] += c[i] * L.mode[i].stride;
    return p;
}

// f(x) for a flat index: the last mode varies fastest.
template <int R>
TN_LAYOUT_HD constexpr AxisPoint eval(const AxisLayout<R>& L, int x) {
    int c[R] = {};
    for (int i = R - 1; i >= 0; --i) {
        c[i] = x % L.mode[i].shape;
        x /= L.mode[i].shape;
    }
    return eval_coord(L, c);
}

// + O[s@axis]: a fixed shift along one axis.
TN_LAYOUT_HD constexpr AxisPoint offset(AxisPoint p, int s, int axis) {
    p.v[axis] += s;
    return p;
}

// + R[n:s@axis]: copy r (0 <= r < n) of a replicated element.
TN_LAYOUT_HD constexpr AxisPoint replica(AxisPoint p, int r, int s, int axis) {
    p.v[axis] += r * s;
    return p;
}

// ------------------------------------------------------------------ CuTe layouts
// A CuTe layout stored as its flattened modes (first fastest) plus the number of
// flat modes in each top-level mode, so that it can be evaluated at a flat index or
// at one flat coordinate per top-level mode.
constexpr int kMaxModes = 8;

struct CuteLayout {
    int rank;                   // top-level modes
    int nflat;                  // flat modes
    int group[kMaxModes];       // flat modes per top-level mode
    int shape[kMaxModes];
    int stride[kMaxModes];
};

TN_LAYOUT_HD constexpr int size(const CuteLayout& L) {
    int n = 1;
    for (int i = 0; i < L.nflat; ++i) n *= L.shape[i];
    return n;
}

// Evaluate flat modes [first, first + count) at the flat index x (first fastest).
TN_LAYOUT_HD constexpr int eval_run(const CuteLayout& L, int first, int count, int x) {
    int off = 0;
    for (int i = first; i < first + count; ++i) {
        off += (x % L.shape[i]) * L.stride[i];
        x /= L.shape[i];
    }
    return off;
}

TN_LAYOUT_HD constexpr int eval(const CuteLayout& L, int x) { return eval_run(L, 0, L.nflat, x); }

// One flat coordinate per top-level mode.
TN_LAYOUT_HD constexpr int eval_modes(const CuteLayout& L, const int* coord) {
    int off = 0, first = 0;
    for (int m = 0; m < L.rank; ++m) {
        off += eval_run(L, first, L.group[m], coord[m]);
        first += L.group[m];
    }
    return off;
}

TN_LAYOUT_HD constexpr int cosize(const CuteLayout& L) {
    int hi = 0;
    for (int i = 0; i < L.nflat; ++i)
        if (L.shape[i] > 1 && L.stride[i] > 0) hi += (L.shape[i] - 1) * L.stride[i];
    return hi + 1;
}

// SM80 m16n8k16, A operand ((4,8),(2,2,2)):((32,1),(16,8,128)): (lane, value) ->
// q = m + 16k of the 16 x 16 tile ("CuTe 中 A、B 如何加载到 MMA 寄存器", section 2).
TN_LAYOUT_HD constexpr CuteLayout sm80_a_tv() {
    return CuteLayout{2, 5, {2, 3}, {4, 8, 2, 2, 2}, {32, 1, 16, 8, 128}};
}
// B operand ((4,8),(2,2)):((16,1),(8,64)) over the 8 x 16 (n, k) tile, q = n + 8k
// (section 5: lane t holds n = t/4, k = 2(t%4) + v%2 + 8(v/2)).
TN_LAYOUT_HD constexpr CuteLayout sm80_b_tv() {
    return CuteLayout{2, 4, {2, 2}, {4, 8, 2, 2}, {16, 1, 8, 64}};
}
// ldmatrix.x4 (section 4): the copy source (32,8):(8,1) and the reference /
// destination (32,(2,4)):(2,(1,64)), both in half units of a 16 x 16 block of
// 8-element rows.
TN_LAYOUT_HD constexpr CuteLayout ldsm_x4_src() { return CuteLayout{2, 2, {1, 1}, {32, 8}, {8, 1}}; }
TN_LAYOUT_HD constexpr CuteLayout ldsm_x4_ref() { return CuteLayout{2, 3, {1, 2}, {32, 2, 4}, {2, 1, 64}}; }

// Inverse of a layout that is a bijection onto [0, size): the flat index i with
// eval(L, i) == e, or -1.  (Linear search: host-side and small layouts only.)
TN_LAYOUT_HD constexpr int inverse_at(const CuteLayout& L, int e) {
    const int n = size(L);
    for (int i = 0; i < n; ++i)
        if (eval(L, i) == e) return i;
    return -1;
}

// ------------------------------------------------------------------ make_fragment_like
// A stride tagged static (known at compile time) or dynamic (run time).
struct TaggedStride {
    int value;
    bool is_static;
};

// make_ordered_layout over flat modes: compact strides visiting the modes in
// increasing order of their `order` stride (static orders by value, dynamic ones
// after every static one, ties and dynamics in their order of appearance); a
// size-1 mode gets stride 0 and does not advance the running product.
TN_LAYOUT_HD constexpr void make_ordered(const int* shape, const TaggedStride* order, int n, int* out) {
    bool done[kMaxModes] = {};
    int cur = 1;
    for (int step = 0; step < n; ++step) {
        int best = -1;
        for (int i = 0; i < n; ++i) {
            if (done[i]) continue;
            if (best < 0) {
                best = i;
                continue;
            }
            const TaggedStride a = order[i], b = order[best];
            const bool better = a.is_static && (!b.is_static || a.value < b.value);
            if (better) best = i;
        }
        done[best] = true;
        if (shape[best] == 1) {
            out[best] = 0;
        } else {
            out[best] = cur;
            cur *= shape[best];
        }
    }
}

// The fragment block of an atom mode: modes whose stride is a static zero are
// broadcasts and collapse to extent 1; the remaining modes get compact strides with
// the first mode fastest (a size-1 mode gets stride 0).
TN_LAYOUT_HD constexpr void fragment_block(const int* shape, const TaggedStride* stride, int n, int* out) {
    int cur = 1;
    for (int i = 0; i < n; ++i) {
        const int extent = (stride[i].is_static && stride[i].value == 0) ? 1 : shape[i];
        if (extent == 1) {
            out[i] = 0;
        } else {
            out[i] = cur;
            cur *= extent;
        }
    }
}

// make_fragment_like of a partitioned tensor whose first top-level mode (the atom's
// values) has `atom_n` flat modes and whose other modes have `rest_n` flat modes:
// the atom block as fragment_block, the rest ordered by make_ordered and scaled by
// the block's cosize.  Shapes are unchanged; strides are written to `out`.
TN_LAYOUT_HD constexpr void make_fragment_like(const int* shape, const TaggedStride* stride, int atom_n, int rest_n,
                                               int* out) {
    fragment_block(shape, stride, atom_n, out);
    int block_cosize = 1;
    for (int i = 0; i < atom_n; ++i)
        if (out[i] > 0) block_cosize += (shape[i] - 1) * out[i];
    make_ordered(shape + atom_n, stride + atom_n, rest_n, out + atom_n);
    for (int i = atom_n; i < atom_n + rest_n; ++i) out[i] *= block_cosize;
}

// ------------------------------------------------------------------ swizzle
// CuTe Swizzle<B, M, S>: XOR the B bits starting at bit M + S into the B bits
// starting at bit M.
TN_LAYOUT_HD constexpr int swizzle(int B, int M, int S, int offset) {
    return offset ^ (((offset >> (M + S)) & ((1 << B) - 1)) << M);
}

// Byte offset of byte `col` of row `row` in a tile of `row_bytes`-byte rows stored
// with the matching TMA / UMMA swizzle: 128-byte rows use Swizzle<3,4,3> (16-byte
// sector XOR row % 8 inside a 1024-byte atom), 64-byte rows Swizzle<2,4,3> (sector
// XOR (row / 2) % 4 inside a 512-byte atom), 32-byte rows Swizzle<1,4,3>; 16-byte
// rows are not swizzled.
TN_LAYOUT_HD constexpr int swizzle_bits(int row_bytes) {
    return row_bytes == 128 ? 3 : row_bytes == 64 ? 2 : row_bytes == 32 ? 1 : 0;
}
TN_LAYOUT_HD constexpr int swizzled_offset(int row_bytes, int row, int col) {
    return swizzle(swizzle_bits(row_bytes), 4, 3, row * row_bytes + col);
}

// Shared-memory bank of a byte address (32 banks of 4 bytes).
TN_LAYOUT_HD constexpr int bank(int byte_addr) { return (byte_addr >> 2) & 31; }

// ------------------------------------------------------------------ tensor memory
// Accumulator of an M = 128 MMA: S[(128,N):(1@TLane,1@TCol)], element (row, col) at
// TMEM lane `row`, column `col`.
TN_LAYOUT_HD constexpr AxisLayout<2> tmem_accumulator(int n) {
    return AxisLayout<2>{{{128, 1, AX_TLANE}, {n, 1, AX_TCOL}}};
}

// Scale factor (m, sfk) of a 128-row x 4-scale block in the 32-lane base tile:
// local lane m % 32, column m / 32, byte sfk of the 32-bit column.  Copy p of the
// four-way lane replication (R[4 : 32@TLane]) sits at lane 32p + m % 32.
struct SfPlace {
    int lane;
    int col;
    int byte;
};
TN_LAYOUT_HD constexpr SfPlace sf_tmem(int m, int sfk, int copy = 0) {
    return SfPlace{32 * copy + m % 32, m / 32, sfk};
}
// Row of the 128-row block held at (local lane, column) of the base tile.
TN_LAYOUT_HD constexpr int sf_row(int local_lane, int col) { return local_lane + 32 * col; }
// Byte of (m, sfk) in the 512-byte base tile read as 16 bytes per local lane.
TN_LAYOUT_HD constexpr int sf_tile_byte(int m, int sfk) {
    return (m % 32) * 16 + (m / 32) * 4 + sfk;
}

// ------------------------------------------------------------------ UMMA descriptors
// Shared-memory matrix descriptor of a K-major operand tile whose rows are
// `row_bytes` long and swizzled as swizzled_offset() lays them out: start address
// / 16 (bits 0-13), leading byte offset / 16 (bits 16-29; unused by swizzled
// K-major tiles, 1 by convention), stride byte offset / 16 between 8-row groups
// (bits 32-45: 8 * row_bytes, the swizzle atom), version 1 (bit 46) and the
// swizzle mode (bits 61-63: 2 = 128-byte, 4 = 64-byte, 6 = 32-byte, 0 = none).
TN_LAYOUT_HD constexpr uint32_t umma_swizzle_mode(int row_bytes) {
    return row_bytes == 128 ? 2u : row_bytes == 64 ? 4u : row_bytes == 32 ? 6u : 0u;
}
TN_LAYOUT_HD constexpr uint64_t umma_smem_desc_kmajor(uint32_t saddr, int row_bytes) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | static_cast<uint64_t>(1) << 16 |
           static_cast<uint64_t>((8 * row_bytes) >> 4) << 32 | static_cast<uint64_t>(1) << 46 |
           static_cast<uint64_t>(umma_swizzle_mode(row_bytes)) << 61;
}

// Descriptor of an unswizzled K-major tile (layout type 0) of 8-row x 16-byte core
// matrices: start address / 16 (bits 0-13), leading byte offset / 16 (bits 16-29:
// between core matrices along K), stride byte offset / 16 (bits 32-45: between 8-row
// groups), version 1 (bit 46).  A 32-row x 16-byte tile stored row after row has
// stride 128 and a single core matrix along K.
TN_LAYOUT_HD constexpr uint64_t umma_smem_desc_noswizzle(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16 |
           static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32 | static_cast<uint64_t>(1) << 46;
}

}  // namespace layout
}  // namespace tn
