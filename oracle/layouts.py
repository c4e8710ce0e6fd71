"""The pages' layout functions, written out plainly.  TEST INFRASTRUCTURE ONLY.

These are the mappings the two pages work through by hand.  They pin the
oracle (and the reading of the data layouts the CUDA path relies on) against
the pages' printed values; nothing here is used by the product path.

Two indexing conventions appear on the pages and both are kept:
  * "数据布局及其记号" (the data-layout chapter) writes S[(shape):(strides)] and
    unflattens a flat index with the LAST mode fastest (section "Tile Layout":
    c0 = x // 16, ..., c3 = x % 4).  Strides may carry a named axis
    (@m, @TLane, @TCol, @laneid, @reg, @gpuid_x, @gpuid_y).
  * "CuTe 中 A、B 如何加载到 MMA 寄存器" writes CuTe layouts (shape):(stride)
    whose flat integer coordinate runs with the FIRST mode fastest
    (section 2: t = t0 + 4*t1, v = v0 + 2*v1 + 4*v2).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Sequence, Tuple, Union

# --------------------------------------------------------------------------
# Named-axis Shape:Stride layouts ("数据布局及其记号", sections "Shape-Stride 模型",
# "Tile Layout", "命名轴", "Replication 与 Offset")
# --------------------------------------------------------------------------

Axis = str
Stride = Union[int, Tuple[int, Axis]]  # plain int means the linear memory axis @m


def _as_axis(s: Stride) -> Tuple[int, Axis]:
    return (s, "m") if isinstance(s, int) else s


def unflatten_last_fastest(x: int, shape: Sequence[int]) -> List[int]:
    """Split a flat index into coordinates, last mode fastest (the "Tile Layout" section)."""
    coords = []
    for e in reversed(shape):
        coords.append(x % e)
        x //= e
    return list(reversed(coords))


def S(shape: Sequence[int], strides: Sequence[Stride], x: int) -> Dict[Axis, int]:
    """f_D(x) for S[(shape):(strides)]: unflatten x, then dot with the strides per axis."""
    assert len(shape) == len(strides)
    assert 0 <= x < _prod(shape)
    out: Dict[Axis, int] = {}
    for c, s in zip(unflatten_last_fastest(x, shape), strides):
        k, ax = _as_axis(s)
        out[ax] = out.get(ax, 0) + c * k
    return out


def S_coord(shape: Sequence[int], strides: Sequence[Stride], coord: Sequence[int]) -> Dict[Axis, int]:
    """Same as S() but taking the per-mode coordinates directly."""
    out: Dict[Axis, int] = {}
    for c, e, s in zip(coord, shape, strides):
        assert 0 <= c < e
        k, ax = _as_axis(s)
        out[ax] = out.get(ax, 0) + c * k
    return out


def with_replication(base: Dict[Axis, int], rshape: int, rstride: Stride) -> List[Dict[Axis, int]]:
    """base + R[n : s@axis]: one copy per replica coordinate r = 0..n-1, offset r*s@axis."""
    k, ax = _as_axis(rstride)
    outs = []
    for r in range(rshape):
        d = dict(base)
        d[ax] = d.get(ax, 0) + r * k
        outs.append(d)
    return outs


def with_offset(base: Dict[Axis, int], off: Stride) -> Dict[Axis, int]:
    """base + O[s@axis]: a fixed shift along one axis, no extra copy."""
    k, ax = _as_axis(off)
    d = dict(base)
    d[ax] = d.get(ax, 0) + k
    return d


def _prod(xs) -> int:
    p = 1
    for x in xs:
        p *= x
    return p


def tile_layout_8x8_in_2x4(i: int, j: int) -> int:
    """Address of element (i, j) under S[(4,2,2,4):(16,4,8,1)] with x = i*8 + j."""
    return S((4, 2, 2, 4), (16, 4, 8, 1), i * 8 + j)["m"]


def m8n8_fragment(row: int, col: int) -> Tuple[int, int]:
    """(laneid, reg) of element (row, col) under S[(8,4,2):(4@laneid,1@laneid,1@reg)]."""
    d = S((8, 4, 2), ((4, "laneid"), (1, "laneid"), (1, "reg")), row * 8 + col)
    return d["laneid"], d["reg"]


def tmem_accumulator(row: int, col: int) -> Tuple[int, int]:
    """(TLane, TCol) of accumulator element (row, col) under S[(128,256):(1@TLane,1@TCol)]."""
    d = S((128, 256), ((1, "TLane"), (1, "TCol")), row * 256 + col)
    return d["TLane"], d["TCol"]


def mesh_element(y: int, row: int, col: int, mode: str) -> List[Tuple[Tuple[int, int], int]]:
    """Devices (gpuid_x, gpuid_y) and local offset of element (y,row,col) of
    base = S[(2,4,8):(1@gpuid_y, 8@m, 1@m)], plain ("shard"), with + R[2:1@gpuid_x]
    ("replica") or with + O[1@gpuid_x] ("offset")."""
    base = S_coord((2, 4, 8), ((1, "gpuid_y"), (8, "m"), (1, "m")), (y, row, col))
    if mode == "replica":
        locs = with_replication(base, 2, (1, "gpuid_x"))
    elif mode == "offset":
        locs = [with_offset(base, (1, "gpuid_x"))]
    else:
        locs = [base]
    return [((d.get("gpuid_x", 0), d.get("gpuid_y", 0)), d["m"]) for d in locs]


# --------------------------------------------------------------------------
# CuTe layouts, first mode fastest ("CuTe 中 A、B 如何加载到 MMA 寄存器")
# --------------------------------------------------------------------------

Shape = Union[int, tuple]


def _flatten(t) -> list:
    if isinstance(t, tuple):
        out = []
        for e in t:
            out.extend(_flatten(e))
        return out
    return [t]


def size(shape: Shape) -> int:
    return _prod(_flatten(shape))


@dataclass(frozen=True)
class Layout:
    """A CuTe-style layout: nested shape and stride of the same profile."""
    shape: Shape
    stride: Shape

    def __call__(self, *coord) -> int:
        """Evaluate at a flat integer (first mode fastest) or per-mode coordinates.
        Each per-mode coordinate may itself be a flat integer over that mode."""
        if len(coord) == 1 and isinstance(coord[0], int):
            return _eval_flat(self.shape, self.stride, coord[0])
        shapes = self.shape if isinstance(self.shape, tuple) else (self.shape,)
        strides = self.stride if isinstance(self.stride, tuple) else (self.stride,)
        assert len(coord) == len(shapes)
        total = 0
        for c, sh, st in zip(coord, shapes, strides):
            if isinstance(c, int):
                total += _eval_flat(sh, st, c)
            else:
                total += Layout(sh, st)(*c)
        return total

    def size(self) -> int:
        return size(self.shape)

    def cosize(self) -> int:
        return max(self(i) for i in range(self.size())) + 1


def _eval_flat(shape, stride, x: int) -> int:
    shs, sts = _flatten(shape), _flatten(stride)
    total = 0
    for e, s in zip(shs, sts):
        total += (x % e) * s
        x //= e
    return total


# SM80 m16n8k16 A operand: (lane, value) -> q = m + 16*k, section 2.
SM80_A_TV = Layout(((4, 8), (2, 2, 2)), ((32, 1), (16, 8, 128)))


def sm80_A_tv_to_mk(t: int, v: int) -> Tuple[int, int]:
    """Matrix coordinate (m, k) held by lane t, value v of the 16x16 A operand."""
    q = SM80_A_TV(t, v)
    return q % 16, q // 16


def sm80_A_mk_to_tv(m: int, k: int) -> Tuple[int, int]:
    """Inverse map of section 2: lane = 4*(m%8) + (k%8)/2, v = k%2 + 2*(m/8) + 4*(k/8)."""
    return 4 * (m % 8) + (k % 8) // 2, k % 2 + 2 * (m // 8) + 4 * (k // 8)


def sm80_B_tv_to_nk(t: int, v: int) -> Tuple[int, int]:
    """B operand (N,K) indexing, section 5: n = t/4, k = 2*(t%4) + v%2 + 8*(v/2)."""
    return t // 4, 2 * (t % 4) + v % 2 + 8 * (v // 2)


def sm80_B_nk_to_tv(n: int, k: int) -> Tuple[int, int]:
    """Section 5 inverse: lane = 4*n + (k%8)/2, v = k%2 + 2*(k/8)."""
    return 4 * n + (k % 8) // 2, k % 2 + 2 * (k // 8)


def partition_A_single_atom(lane: int, row_stride: int) -> Tuple[List[int], List[int]]:
    """Shared-memory offsets of lane's 8 A values for a 16x16 sA with the given row
    stride (k contiguous), and the per-sub-mode strides of the (2,2,2) value mode."""
    offs = []
    for v in range(8):
        m, k = sm80_A_tv_to_mk(lane, v)
        offs.append(row_stride * m + k)
    base = offs[0]
    strides = [offs[1] - base, offs[2] - base, offs[4] - base]
    return offs, strides


# ldmatrix.x4 atoms in half units, section 4.
LDSM_X4_SRC = Layout((32, 8), (8, 1))
LDSM_X4_REF = Layout((32, (2, 4)), (2, (1, 64)))
LDSM_X4_DST = LDSM_X4_REF


def right_inverse_bijection(L: Layout) -> Dict[int, int]:
    """Inverse of a layout that is a bijection onto [0, size): element -> flat (t,v) index."""
    inv = {}
    for i in range(L.size()):
        e = L(i)
        assert e not in inv, "not injective"
        inv[e] = i
    assert sorted(inv) == list(range(L.size())), "not onto [0,size)"
    return inv


def ldsm_x4_route(src_lane: int, src_val: int):
    """Follow one element through ldmatrix.x4: source (t,v) -> copy element e ->
    reference tv -> matrix number q of the MMA A layout -> (m, k)."""
    e = LDSM_X4_SRC(src_lane, src_val)
    tv = right_inverse_bijection(LDSM_X4_REF)[e]
    q = SM80_A_TV(tv)
    return e, tv, q, (q % 16, q // 16)


# ---- make_fragment_like (section 3 and the source appendix) -----------------

@dataclass(frozen=True)
class S_:
    """A stride value tagged static (compile-time) or dynamic (run-time)."""
    value: int
    static: bool = True


def filter_zeros(stride, shape):
    """Replace the shape entries whose stride is a STATIC zero by 1."""
    if isinstance(shape, tuple):
        return tuple(filter_zeros(st, sh) for st, sh in zip(stride, shape))
    return 1 if (stride.static and stride.value == 0) else shape


def compact_major_left(shape):
    """Compact strides, first sub-mode fastest; a size-1 mode gets stride 0 and
    leaves the running product unchanged."""
    flat = _flatten(shape)
    out, cur = [], 1
    for e in flat:
        if e == 1:
            out.append(0)
        else:
            out.append(cur)
            cur *= e
    return _unflatten_like(out, shape)


def _unflatten_like(flat: list, profile):
    it = iter(flat)

    def rec(p):
        if isinstance(p, tuple):
            return tuple(rec(e) for e in p)
        return next(it)
    return rec(profile)


def make_ordered_layout(shape, order):
    """Compact strides visiting modes in increasing order: static orders compare
    by value, dynamic orders rank after all static ones and keep their order of
    appearance.  Size-1 modes get stride 0."""
    flat_shape = _flatten(shape)
    flat_order = _flatten(order)
    idx = list(range(len(flat_shape)))
    idx.sort(key=lambda i: (0, flat_order[i].value, i) if flat_order[i].static else (1, 0, i))
    strides = [0] * len(flat_shape)
    cur = 1
    for i in idx:
        if flat_shape[i] == 1:
            strides[i] = 0
        else:
            strides[i] = cur
            cur *= flat_shape[i]
    return _unflatten_like(strides, shape)


def make_fragment_like(shape, stride):
    """Fragment layout for a partitioned tensor of rank > 1 with static shape:
    mode 0 (the atom's values) compacted first-mode-fastest after filtering static
    zeros, the remaining modes ordered by make_ordered_layout, and the rest
    scaled by the atom block's cosize (tiled product)."""
    atom_shape, atom_stride = shape[0], stride[0]
    block_stride = compact_major_left(filter_zeros(atom_stride, atom_shape))
    block = Layout(atom_shape, block_stride)
    rest_shape = shape[1:]
    rest_stride = make_ordered_layout(rest_shape, stride[1:])
    cos = block.cosize()
    rest_scaled = _unflatten_like([s * cos for s in _flatten(rest_stride)], rest_stride)
    return (atom_shape,) + tuple(rest_shape), (block_stride,) + tuple(rest_scaled)


def make_tensor_like(shape, stride):
    """Ordered compact layout over all modes at once (the general make_tensor_like)."""
    return shape, make_ordered_layout(shape, stride)


def offset_A_full(v: int, m: int, k: int) -> int:
    """Full-config A fragment ((2,2,2),4,(2,2)):((1,2,4),8,(32,64)) with flat v and k."""
    return Layout(((2, 2, 2), 4, (2, 2)), ((1, 2, 4), 8, (32, 64)))(v, m, k)


def offset_B_full(v: int, n: int, k: int) -> int:
    """Full-config B fragment: 4 values, 8 N repeats, 4 K blocks -> v + 4n + 32k."""
    return Layout(((2, 2), 8, (2, 2)), ((1, 2), 4, (32, 64)))(v, n, k)


def retile_B_x4(v: int, j: int, k: int) -> Tuple[int, int, int]:
    """Copy-view coordinate (v, j, k) of tXrB -> MMA-view coordinate of tCrB (section 6)."""
    return v % 4, 2 * j + v // 4, k


def retile_A_x4_group(v: int) -> int:
    """A with ldmatrix.x4: copy view ((8,1),1,1):((1,0),0,0) -> the same slot v."""
    return Layout((8, 1), (1, 0))(v, 0)


# --------------------------------------------------------------------------
# Swizzle ("数据布局及其记号", section "Swizzle Layout")
# --------------------------------------------------------------------------

def bank_of(byte_addr: int) -> int:
    """bank = (addr // 4) % 32."""
    return (byte_addr // 4) % 32


def toy_xor_swizzle(row: int, col: int) -> int:
    """8-bank toy model: mapped_col = logical_col XOR row (bank = mapped_col)."""
    return col ^ row


def swizzle128_sector(row: int, sector: int) -> int:
    """SWIZZLE_128B, K-major: physical 16-byte sector of logical sector `sector`
    (0..7) in row `row` of an 8-row x 128-byte atom."""
    return sector ^ (row % 8)


def swizzle128_byte_offset(row: int, byte_in_row: int) -> int:
    """Byte offset inside a tile of 128-byte rows stored as 1024-byte atoms."""
    atom, r = divmod(row, 8)
    sector, b = divmod(byte_in_row, 16)
    return atom * 1024 + r * 128 + swizzle128_sector(r, sector) * 16 + b


def swizzle_333_half(offset: int) -> int:
    """CuTe Swizzle<3,3,3> on a half-element offset: bits [6,9) XOR into bits [3,6)."""
    return offset ^ (((offset >> 6) & 7) << 3)


# --------------------------------------------------------------------------
# Scale factors in TMEM ("数据布局及其记号", block-scaled MMA section)
# --------------------------------------------------------------------------

def sf_tmem_base_tile(m: int, sfk: int) -> Tuple[int, int, int]:
    """Packing of one 128 x 4 scale-factor block into the 32-lane base tile:
    local_lane = m % 32, TCol = m // 32, byte = sfk."""
    assert 0 <= m < 128 and 0 <= sfk < 4
    return m % 32, m // 32, sfk


def sf_tmem_locations(m: int, sfk: int) -> List[Tuple[int, int, int]]:
    """(TLane, TCol, byte) of SF[m, sfk] after the .warpx4 copy:
    S[(32, ...):(1@TLane, ...)] + R[4 : 32@TLane]."""
    lane, col, byte = sf_tmem_base_tile(m, sfk)
    return [(d["TLane"], col, byte) for d in with_replication({"TLane": lane}, 4, (32, "TLane"))]


def sf_base_tile_byte_offset(m: int, sfk: int) -> int:
    """Byte offset in the 512-byte base tile (16 bytes per local lane):
    local_lane*16 + TCol*4 + byte."""
    lane, col, byte = sf_tmem_base_tile(m, sfk)
    return lane * 16 + col * 4 + byte
