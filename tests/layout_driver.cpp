// Test driver for the layout library (cute_layouts_mma_gb300/csrc/layout.cuh):
// evaluates its maps over their whole domains and prints them as JSON, so that the
// CPU tests can hold them against the pages' values and the oracle.
//
//   layout_driver tables
//   layout_driver fragment <atom_flat_modes> <rest_flat_modes> <shape...> <stride...> <static 0/1...>
//   layout_driver ordered <flat_modes> <shape...> <order...> <static 0/1...>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "layout.cuh"

using namespace tn::layout;

static void list_begin(const char* name, bool& first) {
    std::printf("%s\"%s\": [", first ? "" : ",\n", name);
    first = false;
}

static void tables() {
    bool first = true;
    std::printf("{\n");
    // "Tile Layout": S[(4,2,2,4):(16,4,8,1)], element (i, j) at x = 8i + j
    {
        constexpr AxisLayout<4> tile{{{4, 16, AX_M}, {2, 4, AX_M}, {2, 8, AX_M}, {4, 1, AX_M}}};
        list_begin("tile_8x8", first);
        for (int x = 0; x < size(tile); ++x) std::printf("%s%d", x ? "," : "", eval(tile, x)[AX_M]);
        std::printf("]");
    }
    // m8n8 fragment S[(8,4,2):(4@laneid,1@laneid,1@reg)], element (r, c) at x = 8r + c
    {
        constexpr AxisLayout<3> frag{{{8, 4, AX_LANEID}, {4, 1, AX_LANEID}, {2, 1, AX_REG}}};
        list_begin("m8n8", first);
        for (int x = 0; x < 64; ++x) {
            const AxisPoint p = eval(frag, x);
            std::printf("%s[%d,%d]", x ? "," : "", p[AX_LANEID], p[AX_REG]);
        }
        std::printf("]");
    }
    // TMEM accumulator S[(128,256):(1@TLane,1@TCol)] at a few elements
    {
        const AxisLayout<2> acc = tmem_accumulator(256);
        const int pts[3][2] = {{0, 0}, {5, 200}, {127, 255}};
        list_begin("tmem_acc", first);
        for (int i = 0; i < 3; ++i) {
            const AxisPoint p = eval(acc, pts[i][0] * 256 + pts[i][1]);
            std::printf("%s[%d,%d]", i ? "," : "", p[AX_TLANE], p[AX_TCOL]);
        }
        std::printf("]");
    }
    // device mesh: base S[(2,4,8):(1@gpuid_y,8@m,1@m)]; + R[2:1@gpuid_x]; + O[1@gpuid_x]
    {
        constexpr AxisLayout<3> mesh{{{2, 1, AX_GPU_Y}, {4, 8, AX_M}, {8, 1, AX_M}}};
        list_begin("mesh", first);
        bool f = true;
        for (int y = 0; y < 2; ++y)
            for (int r = 0; r < 4; ++r)
                for (int c = 0; c < 8; ++c) {
                    const int crd[3] = {y, r, c};
                    const AxisPoint b = eval_coord(mesh, crd);
                    const AxisPoint r0 = replica(b, 0, 1, AX_GPU_X), r1 = replica(b, 1, 1, AX_GPU_X);
                    const AxisPoint o = offset(b, 1, AX_GPU_X);
                    std::printf("%s[[%d,%d,%d],[%d,%d,%d],[[%d,%d,%d],[%d,%d,%d]],[%d,%d,%d]]", f ? "" : ",", y, r,
                                c, b[AX_GPU_X], b[AX_GPU_Y], b[AX_M], r0[AX_GPU_X], r0[AX_GPU_Y], r0[AX_M],
                                r1[AX_GPU_X], r1[AX_GPU_Y], r1[AX_M], o[AX_GPU_X], o[AX_GPU_Y], o[AX_M]);
                    f = false;
                }
        std::printf("]");
    }
    // SM80 A and B thread-value layouts
    {
        constexpr CuteLayout a = sm80_a_tv();
        list_begin("sm80_a", first);
        for (int t = 0; t < 32; ++t)
            for (int v = 0; v < 8; ++v) {
                const int crd[2] = {t, v};
                const int q = eval_modes(a, crd);
                std::printf("%s[%d,%d]", (t || v) ? "," : "", q % 16, q / 16);
            }
        std::printf("]");
        constexpr CuteLayout b = sm80_b_tv();
        list_begin("sm80_b", first);
        for (int t = 0; t < 32; ++t)
            for (int v = 0; v < 4; ++v) {
                const int crd[2] = {t, v};
                const int q = eval_modes(b, crd);
                std::printf("%s[%d,%d]", (t || v) ? "," : "", q % 8, q / 8);
            }
        std::printf("]");
    }
    // ldmatrix.x4: source (t, v) -> element e -> reference (t, v) -> A q -> (m, k)
    {
        constexpr CuteLayout src = ldsm_x4_src(), ref = ldsm_x4_ref(), a = sm80_a_tv();
        list_begin("ldsm_x4", first);
        for (int t = 0; t < 32; ++t)
            for (int v = 0; v < 8; ++v) {
                const int crd[2] = {t, v};
                const int e = eval_modes(src, crd);
                const int tv = inverse_at(ref, e);
                const int q = eval(a, tv);
                std::printf("%s[%d,%d,%d,%d,%d]", (t || v) ? "," : "", e, tv, q, q % 16, q / 16);
            }
        std::printf("]");
    }
    // swizzles: 128-byte rows (bytes), Swizzle<3,3,3> on half offsets, 64- and 32-byte rows
    {
        list_begin("sw128", first);
        for (int r = 0; r < 16; ++r)
            for (int b = 0; b < 128; ++b) std::printf("%s%d", (r || b) ? "," : "", swizzled_offset(128, r, b));
        std::printf("]");
        list_begin("sw333_half", first);
        for (int o = 0; o < 1024; ++o) std::printf("%s%d", o ? "," : "", swizzle(3, 3, 3, o));
        std::printf("]");
        list_begin("sw64", first);
        for (int r = 0; r < 16; ++r)
            for (int b = 0; b < 64; ++b) std::printf("%s%d", (r || b) ? "," : "", swizzled_offset(64, r, b));
        std::printf("]");
        list_begin("sw32", first);
        for (int r = 0; r < 16; ++r)
            for (int b = 0; b < 32; ++b) std::printf("%s%d", (r || b) ? "," : "", swizzled_offset(32, r, b));
        std::printf("]");
        list_begin("bank", first);
        for (int a = 0; a < 256; a += 4) std::printf("%s%d", a ? "," : "", bank(a));
        std::printf("]");
    }
    // scale factors in TMEM: (m, sfk) -> four (lane, col, byte) copies and the base-tile byte
    {
        list_begin("sf", first);
        for (int m = 0; m < 128; ++m)
            for (int k = 0; k < 4; ++k) {
                std::printf("%s[", (m || k) ? "," : "");
                for (int p = 0; p < 4; ++p) {
                    const SfPlace s = sf_tmem(m, k, p);
                    std::printf("%s[%d,%d,%d]", p ? "," : "", s.lane, s.col, s.byte);
                }
                std::printf(",%d,%d]", sf_tile_byte(m, k), sf_row(m % 32, m / 32));
            }
        std::printf("]");
    }
    // UMMA shared-memory descriptors of K-major tiles
    {
        list_begin("umma_desc", first);
        const int rows[3] = {128, 64, 32};
        for (int i = 0; i < 3; ++i) {
            const uint64_t d = umma_smem_desc_kmajor(0x12400u, rows[i]);
            std::printf("%s[%d,%llu]", i ? "," : "", rows[i], static_cast<unsigned long long>(d));
        }
        std::printf("]");
    }
    std::printf("\n}\n");
}

int main(int argc, char** argv) {
    if (argc >= 2 && std::strcmp(argv[1], "tables") == 0) {
        tables();
        return 0;
    }
    if (argc >= 4 && std::strcmp(argv[1], "fragment") == 0) {
        const int an = std::atoi(argv[2]), rn = std::atoi(argv[3]), n = an + rn;
        if (n > kMaxModes || argc != 4 + 3 * n) return 2;
        int shape[kMaxModes], out[kMaxModes];
        TaggedStride st[kMaxModes];
        for (int i = 0; i < n; ++i) {
            shape[i] = std::atoi(argv[4 + i]);
            st[i] = TaggedStride{std::atoi(argv[4 + n + i]), std::atoi(argv[4 + 2 * n + i]) != 0};
        }
        make_fragment_like(shape, st, an, rn, out);
        for (int i = 0; i < n; ++i) std::printf("%s%d", i ? " " : "", out[i]);
        std::printf("\n");
        return 0;
    }
    if (argc >= 3 && std::strcmp(argv[1], "ordered") == 0) {
        const int n = std::atoi(argv[2]);
        if (n > kMaxModes || argc != 3 + 3 * n) return 2;
        int shape[kMaxModes], out[kMaxModes];
        TaggedStride st[kMaxModes];
        for (int i = 0; i < n; ++i) {
            shape[i] = std::atoi(argv[3 + i]);
            st[i] = TaggedStride{std::atoi(argv[3 + n + i]), std::atoi(argv[3 + 2 * n + i]) != 0};
        }
        make_ordered(shape, st, n, out);
        for (int i = 0; i < n; ++i) std::printf("%s%d", i ? " " : "", out[i]);
        std::printf("\n");
        return 0;
    }
    std::fprintf(stderr, "usage: layout_driver tables | fragment ... | ordered ...\n");
    return 2;
}
