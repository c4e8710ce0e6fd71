"""Pins of the oracle's layout functions against the pages' worked values (CPU only)."""
import itertools

import numpy as np
import pytest
import torch

from oracle import layouts as L
from oracle import emulate
import oracle


# ---- Shape:Stride and tiles ("数据布局及其记号") ---------------------------------

def test_row_major_and_torch_strides(page):
    lay = page["row_major_4x4"]
    for i, j in itertools.product(range(4), range(4)):
        assert L.S(lay["shape"], lay["strides"], i * 4 + j)["m"] == i * 4 + j
    t = torch.arange(12).reshape(3, 4)
    assert t.stride() == page["torch_strides_3x4"]
    assert t.T.stride() == page["torch_strides_3x4_T"]
    # the S[] of a torch view addresses the same storage element as torch does
    tt = t.T
    for i, j in itertools.product(range(4), range(3)):
        addr = L.S(tt.shape, tt.stride(), i * 3 + j)["m"]
        assert t.flatten()[addr] == tt[i, j]


def test_tile_layout_matches_tiles_described_in_prose(page):
    lay = page["tile_layout"]
    assert (lay["shape"], lay["strides"]) == ((4, 2, 2, 4), (16, 4, 8, 1))
    addrs = set()
    for i, j in itertools.product(range(8), range(8)):
        coords = L.unflatten_last_fastest(i * 8 + j, lay["shape"])
        assert coords == [eval(e, {"i": i, "j": j}) for e in page["tile_coords"]]
        a = L.tile_layout_8x8_in_2x4(i, j)
        # prose: 2x4 tiles laid out row-major, each tile's 8 elements row-major inside it
        tile = (i // 2) * 2 + (j // 4)
        assert a == tile * 8 + (i % 2) * 4 + (j % 4)
        addrs.add(a)
    assert addrs == set(range(64))


def test_m8n8_fragment(page):
    assert L.m8n8_fragment(*page["m8n8_element"]) == page["m8n8_lane_slot"]
    seen = set()
    for r, c in itertools.product(range(8), range(8)):
        lane, reg = L.m8n8_fragment(r, c)
        assert (lane, reg) == (r * 4 + c // 2, c % 2)
        seen.add((lane, reg))
    assert seen == {(l, s) for l in range(32) for s in range(2)}


def test_tmem_accumulator(page):
    assert page["tmem_lanes"] == 128 and page["tmem_max_cols"] == 512
    for r, c in [(0, 0), (5, 200), (127, 255)]:
        assert L.tmem_accumulator(r, c) == (r, c)


def test_mesh_replication_and_offset(page):
    y, r, c = page["mesh_element"]
    plain = L.mesh_element(y, r, c, "shard")
    assert plain == [((0, 1), page["mesh_local_offset"])]
    rep = L.mesh_element(y, r, c, "replica")
    assert sorted(d for d, _ in rep) == sorted(page["mesh_replica_devices"])
    assert all(off == page["mesh_local_offset"] for _, off in rep)
    off = L.mesh_element(y, r, c, "offset")
    assert [d for d, _ in off] == page["mesh_offset_devices"]
    assert off[0][1] == page["mesh_local_offset"]


# ---- SM80 fragments ("CuTe 中 A、B 如何加载到 MMA 寄存器") -----------------------

def test_lane0_A_fragment(page):
    elems = [L.sm80_A_tv_to_mk(0, v) for v in range(8)]
    assert elems == [tuple(e) for e in page["lane0_A_elements"]]
    offs, _ = L.partition_A_single_atom(0, 16)
    assert offs == page["lane0_A_smem_offsets"]
    assert L.sm80_A_mk_to_tv(0, 9) == page["A09_lane_value"]


def test_A_tv_layout_is_bijection_and_inverse_formula_agrees():
    seen = set()
    for t in range(32):
        for v in range(8):
            m, k = L.sm80_A_tv_to_mk(t, v)
            assert L.sm80_A_mk_to_tv(m, k) == (t, v)
            seen.add((m, k))
    assert seen == {(m, k) for m in range(16) for k in range(16)}


def test_B_operand_map(page):
    b = [L.sm80_B_tv_to_nk(0, v) for v in range(4)]
    assert b[:2] == [tuple(x) for x in page["lane0_b0"]]
    assert b[2:] == [tuple(x) for x in page["lane0_b1"]]
    seen = set()
    for t in range(32):
        for v in range(4):
            n, k = L.sm80_B_tv_to_nk(t, v)
            assert L.sm80_B_nk_to_tv(n, k) == (t, v)
            seen.add((n, k))
    assert seen == {(n, k) for n in range(8) for k in range(16)}


def test_partition_A_small_and_exercise1(page):
    _, strides = L.partition_A_single_atom(0, 16)
    assert tuple(strides) == page["tCsA_mma"]["strides"][0]
    # exercise 1: the row stride 16 -> 24 turns 128 into 192, the fragment is unchanged
    _, strides24 = L.partition_A_single_atom(0, 24)
    assert strides[1] == page["exercise1_partition_stride_before"]
    assert strides24[1] == page["exercise1_partition_stride_after"]
    st = lambda xs: tuple(L.S_(x) for x in xs)
    for sA in (strides, strides24):
        shape, stride = L.make_fragment_like(((2, 2, 2), 1, 1), (st(sA), L.S_(0), L.S_(0)))
        assert (shape, stride) == (page["tCrA_small"]["shape"], page["tCrA_small"]["strides"])


def test_make_fragment_like_block_and_broadcast(page):
    st = lambda xs, static=True: tuple(L.S_(x, static) for x in xs)
    blk = L.compact_major_left(L.filter_zeros(st((1, 128, 8)), (2, 2, 2)))
    assert blk == page["block_small"]["strides"]
    blk0 = L.compact_major_left(L.filter_zeros(st(page["broadcast_atom_stride_static"]), (2, 2, 2)))
    assert blk0 == page["broadcast_block_strides"]
    lay = L.Layout((2, 2, 2), blk0)
    assert lay(0, 0, 0) == 0 and lay(0, 1, 0) == 0
    assert lay.cosize() == 4
    # a run-time zero is not a broadcast
    dyn = (L.S_(1), L.S_(0, static=False), L.S_(8))
    assert L.compact_major_left(L.filter_zeros(dyn, (2, 2, 2))) == page["broadcast_dynamic_block_strides"]


def _tagged(strides):
    if isinstance(strides, tuple) and len(strides) == 2 and isinstance(strides[1], str):
        return L.S_(strides[0], strides[1] == "s")
    return tuple(_tagged(s) for s in strides)


def test_full_config_fragment_and_tensor_like(page):
    pa = page["full_partition_A"]
    stride = _tagged(pa["strides"])
    rest = L.make_ordered_layout(pa["shape"][1:], stride[1:])
    assert rest == page["full_rest"]["strides"]
    shape, frag = L.make_fragment_like(pa["shape"], stride)
    assert (shape, frag) == (page["full_tCrA"]["shape"], page["full_tCrA"]["strides"])
    _, like = L.make_tensor_like(pa["shape"], stride)
    assert like == page["full_make_tensor_like"]["strides"]
    # offset_A = v + 8m + 32k and offset_B = v + 4n + 32k (source appendix)
    for v, m, k in itertools.product(range(8), range(4), range(4)):
        assert L.offset_A_full(v, m, k) == v + 8 * m + 32 * k
    for v, n, k in itertools.product(range(4), range(8), range(4)):
        assert L.offset_B_full(v, n, k) == v + 4 * n + 32 * k
    assert (page["full_MMA_M"], page["full_MMA_N"], page["full_MMA_K"]) == (
        128 // (16 * 2), 128 // (8 * 2), 64 // 16)
    assert page["full_fragment_halves"]["tCrA"] == 8 * 4 * 4


def test_ldmatrix_x4_route_of_A09(page):
    e, tv, q, mk = L.ldsm_x4_route(*page["ldsm_src_tv"])
    assert (e, tv, q) == (page["ldsm_e"], page["ldsm_ref_tv"], page["ldsm_q"])
    assert mk == (0, 9)
    assert L.LDSM_X4_DST(*page["ldsm_dst_tv"]) == page["ldsm_e"]
    assert 16 * mk[0] + mk[1] == page["ldsm_smem_offset"]
    # each source lane supplies one contiguous, 16-byte aligned row of 8 halves
    # (section 4: source rows must be contiguous and 16-byte aligned); lane 16's row
    # is A(0, 8..15)
    rows = {}
    for ts in range(32):
        mks = [L.ldsm_x4_route(ts, vs)[3] for vs in range(8)]
        m0, k0 = mks[0]
        assert mks == [(m0, k0 + i) for i in range(8)]
        assert (16 * m0 + k0) % 8 == 0
        rows[ts] = (m0, k0)
    assert rows[16] == (0, 8)
    assert sorted(rows.values()) == sorted((m, k) for m in range(16) for k in (0, 8))


def test_retile_views(page):
    lay = page["tXrA_x4"]
    for mma_coord, copy_coord, slot in page["retile_pairs"]:
        frag = L.Layout(page["tCrA_small"]["shape"][0], page["tCrA_small"]["strides"][0])
        assert frag(*mma_coord) == slot
        assert L.Layout(lay["shape"][0], lay["strides"][0])(*copy_coord) == slot
    for v in range(8):
        assert L.retile_A_x4_group(v) == v
    c = L.retile_B_x4(*page["exercise2_copy"])
    assert c == page["exercise2_mma"]
    assert L.offset_B_full(*c) == page["exercise2_offset"]


# ---- swizzle ------------------------------------------------------------------

def test_swizzle128_row1_and_atom(page):
    assert [L.swizzle128_sector(1, s) for s in range(8)] == page["swizzle_row1_local"]
    assert [8 + L.swizzle128_sector(1, s) for s in range(8)] == page["swizzle_row1_global"]
    offs = {L.swizzle128_byte_offset(r, b) for r in range(8) for b in range(128)}
    assert offs == set(range(page["swizzle128_atom_bytes"]))
    # element-unit Swizzle<3,3,3> on fp16 agrees with the byte-level 128B pattern
    for r in range(16):
        for h in range(64):
            assert 2 * L.swizzle_333_half(r * 64 + h) == L.swizzle128_byte_offset(r, 2 * h)


def test_toy_bank_model_cycles(page):
    def cycles(mapping, col):
        banks = [mapping(r, col) for r in range(8)]
        return max(banks.count(b) for b in set(banks))
    assert all(cycles(lambda r, c: c, col) == page["toy_column_cycles_plain"] for col in range(8))
    assert all(cycles(L.toy_xor_swizzle, col) == page["toy_column_cycles_xor"] for col in range(8))


def test_swizzle128_column_read_conflict_free(page):
    # 8 lanes each read the same logical 16-byte sector of rows 0..7: one wavefront of
    # 16-byte accesses; with the swizzle the 8 sectors cover all 32 banks exactly once.
    assert page["wavefront_lanes"][16] == 8
    for sector in range(8):
        banks = []
        for r in range(8):
            off = L.swizzle128_byte_offset(r, sector * 16)
            banks.extend(L.bank_of(off + 4 * w) for w in range(4))
        assert sorted(banks) == list(range(32))
        plain = [L.bank_of(r * 128 + sector * 16) for r in range(8)]
        assert len(set(plain)) == 1


# ---- scale factors in TMEM ----------------------------------------------------

def test_sf_tmem_placement(page):
    assert L.sf_tmem_base_tile(64, 2) == page["sfa_64_2_base"]
    assert L.sf_tmem_locations(64, 2) == [tuple(x) for x in page["sfa_64_2_replicas"]]
    for (m, sfk), loc in page["sfa_col_examples"]:
        assert L.sf_tmem_base_tile(m, sfk) == tuple(loc)
    offs = {L.sf_base_tile_byte_offset(m, s) for m in range(128) for s in range(4)}
    assert offs == set(range(page["sf_tile_bytes"]))


# ---- emulations tied to the oracle GEMM ---------------------------------------

def test_sm80_fragment_emulation_equals_oracle_gemm():
    g = torch.Generator().manual_seed(11)
    A = torch.randint(-3, 4, (16, 16), generator=g).half()
    B = torch.randint(-3, 4, (8, 16), generator=g).half()
    C = torch.randint(-3, 4, (16, 8), generator=g).half()
    emu = emulate.sm80_m16n8k16_from_fragments(A.double().numpy(), B.double().numpy(),
                                                C.double().numpy())
    d16 = oracle.gemm_f16(A, B, C)
    assert np.array_equal(oracle.f16_bits_to_f64_array(d16), emu)


def test_block_scaled_tmem_emulation_equals_oracle_gemm():
    g = torch.Generator().manual_seed(12)
    K = 64  # one NVFP4 MMA: 4 scale blocks of 16
    a_codes = torch.randint(0, 16, (128, K), generator=g, dtype=torch.uint8)
    b_codes = torch.randint(0, 16, (128, K), generator=g, dtype=torch.uint8)
    sfa = (0x38 + 8 * torch.randint(-2, 3, (128, 4), generator=g)).to(torch.uint8)
    sfb = (0x38 + 8 * torch.randint(-2, 3, (128, 4), generator=g)).to(torch.uint8)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous()
    d16, d64 = oracle.gemm_block_scaled(oracle.NVFP4, pack(a_codes), sfa, pack(b_codes), sfb,
                                        exact=True)
    dec2 = np.vectorize(oracle.e2m1_to_f64)
    dec_sf = np.vectorize(oracle.e4m3_to_f64)
    emu = emulate.block_scaled_mma_via_tmem(dec2(a_codes.numpy()), dec_sf(sfa.numpy()),
                                            dec2(b_codes.numpy()), dec_sf(sfb.numpy()), 16)
    assert np.array_equal(emu, d64)
