"""The product's layout library (csrc/layout.cuh) against the pages and the oracle (CPU only).

The library is header-only C++; a small driver (tests/layout_driver.cpp) is built
with the host compiler and prints the library's maps over their whole domains.
Each map is held against the pages' worked values (tests/golden/page_layouts.txt)
and, element by element, against the oracle's independent restatement of the same
page (oracle/layouts.py).  The kernels take their shared-memory swizzle, UMMA
descriptor and TMEM scale placement from this library, so these checks also pin
the addressing the CUDA path uses.
"""
import itertools
import json
import os
import shutil
import subprocess

import pytest

from oracle import layouts as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("layout") / "layout_driver")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "cute_layouts_mma_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "layout_driver.cpp"), "-o", exe], check=True)
    return exe


@pytest.fixture(scope="module")
def tables(driver):
    out = subprocess.run([driver, "tables"], check=True, capture_output=True, text=True).stdout
    return json.loads(out)


def _run(driver, *args):
    out = subprocess.run([driver, *map(str, args)], check=True, capture_output=True, text=True).stdout
    return [int(x) for x in out.split()]


# ---- the data-layout chapter: S[...] with named axes ---------------------------

def test_tile_layout(tables, page):
    assert page["tile_layout"] == {"shape": (4, 2, 2, 4), "strides": (16, 4, 8, 1)}
    got = tables["tile_8x8"]
    for i, j in itertools.product(range(8), range(8)):
        assert got[8 * i + j] == L.tile_layout_8x8_in_2x4(i, j)
    assert sorted(got) == list(range(64))


def test_m8n8_fragment(tables, page):
    got = [tuple(x) for x in tables["m8n8"]]
    r, c = page["m8n8_element"]
    assert got[8 * r + c] == page["m8n8_lane_slot"]
    for r, c in itertools.product(range(8), range(8)):
        assert got[8 * r + c] == L.m8n8_fragment(r, c)


def test_tmem_accumulator(tables):
    for (r, c), got in zip([(0, 0), (5, 200), (127, 255)], tables["tmem_acc"]):
        assert tuple(got) == L.tmem_accumulator(r, c)


def test_mesh_replication_and_offset(tables, page):
    rows = {tuple(e[0]): e for e in tables["mesh"]}
    for y, r, c in itertools.product(range(2), range(4), range(8)):
        _, base, reps, off = rows[(y, r, c)]
        assert [((base[0], base[1]), base[2])] == L.mesh_element(y, r, c, "shard")
        assert [((x[0], x[1]), x[2]) for x in reps] == L.mesh_element(y, r, c, "replica")
        assert [((off[0], off[1]), off[2])] == L.mesh_element(y, r, c, "offset")
    _, base, reps, off = rows[tuple(page["mesh_element"])]
    assert base[2] == page["mesh_local_offset"]
    assert sorted((x[0], x[1]) for x in reps) == sorted(page["mesh_replica_devices"])
    assert [(off[0], off[1])] == page["mesh_offset_devices"]


# ---- CuTe layouts: SM80 fragments, ldmatrix, make_fragment_like -----------------

def test_sm80_a_and_b_thread_value_layouts(tables, page):
    a = [tuple(x) for x in tables["sm80_a"]]
    assert a[:8] == [tuple(e) for e in page["lane0_A_elements"]]
    for t, v in itertools.product(range(32), range(8)):
        assert a[8 * t + v] == L.sm80_A_tv_to_mk(t, v)
    assert a.index((0, 9)) == 8 * page["A09_lane_value"][0] + page["A09_lane_value"][1]
    b = [tuple(x) for x in tables["sm80_b"]]
    assert b[:2] == [tuple(x) for x in page["lane0_b0"]] and b[2:4] == [tuple(x) for x in page["lane0_b1"]]
    for t, v in itertools.product(range(32), range(4)):
        assert b[4 * t + v] == L.sm80_B_tv_to_nk(t, v)


def test_ldmatrix_x4_route(tables, page):
    rows = tables["ldsm_x4"]
    for t, v in itertools.product(range(32), range(8)):
        e, tv, q, m, k = rows[8 * t + v]
        assert (e, tv, q, (m, k)) == L.ldsm_x4_route(t, v)
    ts, vs = page["ldsm_src_tv"]
    e, tv, q, m, k = rows[8 * ts + vs]
    assert (e, tv, q) == (page["ldsm_e"], page["ldsm_ref_tv"], page["ldsm_q"])
    assert 16 * m + k == page["ldsm_smem_offset"]


def _flat(t):
    return [x for e in t for x in _flat(e)] if isinstance(t, tuple) else [t]


def test_make_fragment_like_small_and_broadcast(driver, page):
    # tCrA of the single-atom partition (section 3): ((2,2,2),1,1) from sA strides (1,128,8) or (1,192,8)
    for row_stride in (16, 24):
        _, st = L.partition_A_single_atom(0, row_stride)
        got = _run(driver, "fragment", 3, 2, 2, 2, 2, 1, 1, *st, 0, 0, 1, 1, 1, 1, 1)
        assert got == _flat(page["tCrA_small"]["strides"])
    # a static zero stride is a broadcast and collapses; a run-time zero does not
    assert _run(driver, "fragment", 3, 0, 2, 2, 2, *page["broadcast_atom_stride_static"], 1, 1, 1) == \
        list(page["broadcast_block_strides"])
    assert _run(driver, "fragment", 3, 0, 2, 2, 2, 1, 0, 8, 1, 0, 1) == list(page["broadcast_dynamic_block_strides"])
    assert _run(driver, "fragment", 3, 0, 2, 2, 2, 1, 128, 8, 1, 1, 1) == list(page["block_small"]["strides"])


def test_make_fragment_like_full_config(driver, page):
    pa = page["full_partition_A"]
    shape = _flat(pa["shape"])
    tagged = list(_walk_tagged(pa["strides"]))
    values = [v for v, _ in tagged]
    static = [1 if s == "s" else 0 for _, s in tagged]
    got = _run(driver, "fragment", 3, len(shape) - 3, *shape, *values, *static)
    assert got == _flat(page["full_tCrA"]["strides"])
    rest = _run(driver, "ordered", len(shape) - 3, *shape[3:], *values[3:], *static[3:])
    assert rest == _flat(page["full_rest"]["strides"])
    like = _run(driver, "ordered", len(shape), *shape, *values, *static)
    assert like == _flat(page["full_make_tensor_like"]["strides"])
    # and the oracle's reading of the same appendix agrees
    o_shape, o_frag = L.make_fragment_like(pa["shape"], _to_oracle(pa["strides"]))
    assert _flat(o_frag) == got


def _walk_tagged(t):
    if isinstance(t, tuple) and len(t) == 2 and isinstance(t[1], str):
        yield t
    else:
        for e in t:
            yield from _walk_tagged(e)


def _to_oracle(t):
    if isinstance(t, tuple) and len(t) == 2 and isinstance(t[1], str):
        return L.S_(t[0], t[1] == "s")
    return tuple(_to_oracle(e) for e in t)


# ---- swizzle ---------------------------------------------------------------------

def test_swizzle_128(tables, page):
    sw = tables["sw128"]
    for r, b in itertools.product(range(16), range(128)):
        assert sw[128 * r + b] == L.swizzle128_byte_offset(r, b)
    assert [(sw[128 + 16 * s] - 128) // 16 for s in range(8)] == page["swizzle_row1_local"]
    assert sorted(sw[:1024]) == list(range(page["swizzle128_atom_bytes"]))
    half = tables["sw333_half"]
    for o in range(1024):
        assert half[o] == L.swizzle_333_half(o)


def test_swizzle_64_and_32(tables):
    # 64-byte rows: 16-byte sector s of row r at sector s ^ ((r // 2) % 4) in a 512-byte
    # atom; 32-byte rows: s ^ ((r // 4) % 2) in a 256-byte atom.  Each atom is a
    # permutation of its bytes, and the same logical sector of the rows sharing one
    # 128-byte line lands in distinct sectors of that line.
    for width, table, atom in ((64, tables["sw64"], 512), (32, tables["sw32"], 256)):
        rows_per_line = 128 // width
        for r, b in itertools.product(range(16), range(width)):
            s, low = divmod(b, 16)
            want = r * width + ((s ^ ((r // rows_per_line) % (width // 16))) * 16) + low
            assert table[width * r + b] == want
        for a0 in range(0, 16 * width, atom):
            assert sorted(table[a0:a0 + atom]) == list(range(a0, a0 + atom))


def test_bank(tables):
    assert tables["bank"] == [L.bank_of(a) for a in range(0, 256, 4)]


# ---- scale factors in TMEM and the UMMA descriptor --------------------------------

def test_scale_factor_placement(tables, page):
    rows = tables["sf"]
    for m, k in itertools.product(range(128), range(4)):
        *copies, tile_byte, row = rows[4 * m + k]
        assert [tuple(c) for c in copies] == L.sf_tmem_locations(m, k)
        assert tuple(copies[0]) == L.sf_tmem_base_tile(m, k)
        assert tile_byte == L.sf_base_tile_byte_offset(m, k)
        assert row == m  # sf_row inverts the base-tile placement
    assert [tuple(c) for c in rows[4 * 64 + 2][:4]] == [tuple(x) for x in page["sfa_64_2_replicas"]]
    for (m, k), loc in page["sfa_col_examples"]:
        assert tuple(rows[4 * m + k][0]) == tuple(loc)
    assert sorted(r[4] for r in rows) == list(range(page["sf_tile_bytes"]))


def test_umma_descriptor_fields(tables):
    # PTX ISA shared-memory matrix descriptor: start >> 4 in bits 0-13, leading offset
    # >> 4 in 16-29, stride offset >> 4 in 32-45, version 1 at bit 46, swizzle mode in
    # 61-63 (2 = 128-byte, 4 = 64-byte, 6 = 32-byte).  The stride offset of a K-major
    # swizzled tile is one 8-row atom.
    for width, d in tables["umma_desc"]:
        assert d & 0x3FFF == 0x12400 >> 4
        assert (d >> 16) & 0x3FFF == 1
        assert (d >> 32) & 0x3FFF == 8 * width // 16
        assert (d >> 46) & 3 == 1
        assert (d >> 61) & 7 == {128: 2, 64: 4, 32: 6}[width]
