"""Plain CPU oracle for layout-driven data movement.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code,
header, table or helper with ``layout_driven_movement_gb300`` (the CUDA
path), and imports nothing from it.

What it computes, written as the plain definitions the three source pages
give, evaluated point by point with numpy int64 arithmetic (no blocking, no
fusion, no reordering):

* a layout is a shape:stride pair with arbitrary nesting; the offset of a
  logical coordinate is the inner product of the coordinate with the strides
  ("CUTLASS Layout可视化：从print_layout理解GPU内存映射与性能优化" §2.1, §3.2;
  "CUTE布局代数：GPU张量计算的内存优化革命" §2.1);
* a 1-D logical index is split into leaf coordinates first-leaf-fastest
  ("colex"); the pages never state the order, this is the reading the
  stripmined thread-map formula and the column-major example force (the
  tests check the generic evaluator against both);
* a 2-D coordinate (row, col) of a rank-2 layout addresses mode 0 with row
  and mode 1 with col ("CUTLASS Layout可视化" §3.3);
* Swizzle<B,M,S> XORs the B offset bits starting at bit M+S into the B bits
  starting at bit M, applied to the whole offset after the affine sum
  ("CUTLASS Layout可视化" §4.3; "CUTE布局代数" §4.2);
* composition R = A o B is the function i -> A(B(i)) ("CUTE布局代数" §2.2);
* zipped_divide splits every mode into a tile of the tiler's extent and the
  rest, tile modes first ("CUTE布局代数" §3.2);
* the inverse layout answers which logical index sits at an offset, and the
  largest common vector of two layouts is the longest prefix of offsets on
  which the two inverses agree ("CUTE布局代数" §2.3);
* the copy is out[dst(i)] = in[src(i)] for every logical index i, moving raw
  element bytes ("CUTE布局代数" §5.1, make_copy(gmem_layout, smem_layout));
* the thread maps are the pitch-linear map and the stripmined map of the
  PitchLinearStripminedThreadMap article (hotelren.com/news/5252042, §1.2
  and §2.2), the latter evaluated as the layout
  (Pitch, Strips, groups):(1, kRow, Pitch*Strips*kRow);
* a thread's part of a tile under local_partition is one element of every
  thread-layout-shaped block, at the thread's coordinate in the block
  ("CUTLASS Layout可视化" §5.3);
* a warp's shared-memory access costs one pass per distinct word that its
  busiest bank must serve, 32 banks of 4 bytes ("CUTLASS Layout可视化"
  §5.2).

Every function here is pinned by ``tests/test_oracle_pins.py`` against
values printed on the pages, closed forms, textbook special cases and
invariants.  Functions without such a pin say "parity unpinned".
"""

from __future__ import annotations

import ast
from math import prod
from typing import Iterable, Sequence

import numpy as np

__all__ = [
    "flatten", "Layout", "Swizzled", "Composed", "ZippedDivide", "Concat",
    "swizzle", "eval_leaf_coord", "eval_2d", "cosize", "is_injective",
    "inverse_map", "right_inverse_values", "max_common_vector",
    "pitch_linear_offset", "stripmined_offset", "copy", "copy_loop",
    "parse", "build", "image", "complement", "LogicalProduct",
    "BlockedProduct",
]


# ---------------------------------------------------------------------------
# shape:stride
# ---------------------------------------------------------------------------

def flatten(shape, stride) -> list[tuple[int, int]]:
    """Leaves (extent, stride) of a nested shape:stride pair, in the order the
    pair is written (so the first leaf of mode 0 comes first)."""
    if isinstance(shape, int):
        if not isinstance(stride, int):
            raise ValueError("shape and stride nest differently")
        if shape < 0:
            raise ValueError("extent must be >= 0 (0 makes an empty layout)")
        return [(shape, stride)]
    if isinstance(stride, int) or len(shape) != len(stride):
        raise ValueError("shape and stride nest differently")
    leaves: list[tuple[int, int]] = []
    for sh, st in zip(shape, stride):
        leaves.extend(flatten(sh, st))
    return leaves


def _as_index(i) -> np.ndarray:
    return np.asarray(i, dtype=np.int64)


def _affine_at(leaves: Sequence[tuple[int, int]], x: np.ndarray,
               extend_last: bool) -> np.ndarray:
    """Sum over leaves of (colex coordinate) * stride.

    With ``extend_last`` the last leaf takes the whole remaining quotient, i.e.
    the layout is read as a function on all non-negative integers by letting
    its last mode run past its extent (the way composition reads its outer
    layout)."""
    rem = x.copy()
    off = np.zeros_like(rem)
    for k, (extent, stride) in enumerate(leaves):
        if extent == 1 and not (extend_last and k == len(leaves) - 1):
            continue
        if extend_last and k == len(leaves) - 1:
            coord = rem
        else:
            coord = rem % extent
            rem = rem // extent
        off = off + coord * stride
    return off


class Layout:
    """An affine layout shape:stride (no swizzle).

    ``at(i)`` takes logical indices 0 <= i < size and returns offsets in
    elements ("CUTLASS Layout可视化" §2.1: offset = row*stride_row +
    col*stride_col, generalised to every leaf)."""

    def __init__(self, shape, stride):
        self.shape = shape
        self.stride = stride
        self.leaves = flatten(shape, stride)
        self.size = prod(e for e, _ in self.leaves)

    # top-level modes, each a Layout of its own
    def modes(self) -> list["Layout"]:
        if isinstance(self.shape, int):
            return [Layout(self.shape, self.stride)]
        return [Layout(sh, st) for sh, st in zip(self.shape, self.stride)]

    def at(self, i, extended: bool = False) -> np.ndarray:
        x = _as_index(i)
        if not extended and x.size and (x.min() < 0 or x.max() >= self.size):
            raise IndexError("logical index outside the layout's domain")
        return _affine_at(self.leaves, x, extend_last=extended)

    __call__ = at

    def __repr__(self) -> str:
        return f"Layout({self.shape!r}:{self.stride!r})"


def swizzle(offset, b: int, m: int, s: int):
    """Swizzle<B,M,S>: XOR bits [M+S, M+S+B) of the offset into bits
    [M, M+B) ("CUTLASS Layout可视化" §4.3: the low bits of the column are
    XORed with the low bits of the row)."""
    o = _as_index(offset)
    mask = ((1 << b) - 1) << m
    return o ^ ((o >> s) & mask)


class Swizzled:
    """Swz<B,M,S> o inner: the swizzle is applied to the whole offset after
    the affine sum."""

    def __init__(self, b: int, m: int, s: int, inner):
        if b < 0 or m < 0 or s < b:
            raise ValueError("Swizzle<B,M,S> needs B >= 0, M >= 0, S >= B")
        self.b, self.m, self.s = b, m, s
        self.inner = inner
        self.size = inner.size

    def at(self, i, extended: bool = False) -> np.ndarray:
        return swizzle(self.inner.at(i, extended), self.b, self.m, self.s)

    __call__ = at


class Composed:
    """R = A o B, R(i) = A(B(i)) ("CUTE布局代数" §2.2).  B's value is read by
    A as a 1-D logical index; A's last mode is extended past its extent when
    B reaches beyond A's domain.  size(R) = size(B)."""

    def __init__(self, outer, inner):
        self.outer, self.inner = outer, inner
        self.size = inner.size

    def at(self, i, extended: bool = False) -> np.ndarray:
        return self.outer.at(self.inner.at(i, extended), extended=True)

    __call__ = at


class ZippedDivide:
    """zipped_divide(L, tiler) ("CUTE布局代数" §3.2).

    Mode k of L (extent n_k) is cut into a tile of t_k consecutive mode-k
    coordinates and n_k/t_k tiles.  The result has two modes: the tile
    (t_0, t_1, ...) and the rest (n_0/t_0, n_1/t_1, ...), both colex.  The
    element e = (e_0, e_1, ...) of tile g = (g_0, g_1, ...) is L evaluated at
    mode coordinates x_k = e_k + t_k * g_k."""

    def __init__(self, layout, tiler: Sequence[int]):
        base = layout.inner if isinstance(layout, Swizzled) else layout
        if not isinstance(base, Layout):
            raise ValueError("zipped_divide takes a shape:stride layout")
        modes = base.modes()
        if len(tiler) != len(modes):
            raise ValueError("tiler rank must equal layout rank")
        for m, t in zip(modes, tiler):
            if t < 1 or m.size % t:
                raise ValueError("tiler must divide every mode")
        self.layout = layout
        self.modes = modes
        self.tiler = list(tiler)
        self.rest = [m.size // t for m, t in zip(modes, tiler)]
        self.size = base.size

    def at(self, i, extended: bool = False) -> np.ndarray:
        x = _as_index(i)
        if x.size and (x.min() < 0 or x.max() >= self.size):
            raise IndexError("logical index outside the layout's domain")
        tile_size = prod(self.tiler)
        e = x % tile_size
        g = x // tile_size
        off = np.zeros_like(x)
        for mode, t, r in zip(self.modes, self.tiler, self.rest):
            e_k = e % t
            e = e // t
            g_k = g % r
            g = g // r
            off = off + mode.at(e_k + t * g_k)
        if isinstance(self.layout, Swizzled):
            off = swizzle(off, self.layout.b, self.layout.m, self.layout.s)
        return off

    __call__ = at


class Concat:
    """(A, B, ...) as the modes of one layout: the logical index is split
    colex over the parts' sizes and the parts' offsets add (the batch mode of
    a batched layout)."""

    def __init__(self, *parts):
        self.parts = parts
        self.size = prod(p.size for p in parts)

    def at(self, i, extended: bool = False) -> np.ndarray:
        x = _as_index(i)
        if x.size and (x.min() < 0 or x.max() >= self.size):
            raise IndexError("logical index outside the layout's domain")
        off = np.zeros_like(x)
        rem = x
        for p in self.parts:
            off = off + p.at(rem % p.size)
            rem = rem // p.size
        return off

    __call__ = at


# ---------------------------------------------------------------------------
# coordinate forms
# ---------------------------------------------------------------------------

def eval_leaf_coord(layout, coord: Sequence[int]) -> int:
    """Inner product of a full leaf coordinate with the leaf strides, then
    the swizzle if any.  No bounds check: this is the bare offset formula
    ("CUTLASS Layout可视化" §2.1), which is how the blocked layout's printed
    values are read (see the R3 pin in the tests)."""
    sw = None
    base = layout
    if isinstance(layout, Swizzled):
        sw, base = layout, layout.inner
    if not isinstance(base, Layout):
        raise ValueError("leaf coordinates need a shape:stride layout")
    if len(coord) != len(base.leaves):
        raise ValueError("one coordinate per leaf")
    off = sum(int(c) * d for c, (_, d) in zip(coord, base.leaves))
    if sw is not None:
        off = int(swizzle(off, sw.b, sw.m, sw.s))
    return off


def eval_2d(layout, row, col) -> np.ndarray:
    """Offset of (row, col) of a rank-2 layout: row is a colex index into
    mode 0, col into mode 1 ("CUTLASS Layout可视化" §3.3: the outer print loop
    walks mode 0, the inner one mode 1)."""
    sw = None
    base = layout
    if isinstance(layout, Swizzled):
        sw, base = layout, layout.inner
    m0, m1 = base.modes()
    off = m0.at(row) + m1.at(col)
    if sw is not None:
        off = swizzle(off, sw.b, sw.m, sw.s)
    return off


def print_grid(layout) -> list[list[int]]:
    """The print_layout double loop: one row per mode-0 coordinate, one
    column per mode-1 coordinate ("CUTLASS Layout可视化" §3.1)."""
    base = layout.inner if isinstance(layout, Swizzled) else layout
    m0, m1 = base.modes()
    return [[int(eval_2d(layout, r, c)) for c in range(m1.size)]
            for r in range(m0.size)]


# ---------------------------------------------------------------------------
# whole-layout properties (brute force)
# ---------------------------------------------------------------------------

def image(layout) -> np.ndarray:
    """Offsets of all logical indices, in logical order."""
    return layout.at(np.arange(layout.size, dtype=np.int64))


def cosize(layout) -> int:
    """Largest offset plus one."""
    return int(image(layout).max()) + 1 if layout.size else 0


def is_injective(layout) -> bool:
    """No two logical indices share an offset."""
    v = image(layout)
    return np.unique(v).size == v.size


def inverse_map(layout, length: int | None = None) -> np.ndarray:
    """inv[j] = the logical index whose offset is j ("CUTE布局代数" §2.3);
    -1 where no index lands on j, -2 where several do."""
    v = image(layout)
    if length is None:
        length = int(v.max()) + 1 if v.size else 0
    inv = np.full(length, -1, dtype=np.int64)
    inside = v < length
    counts = np.bincount(v[inside], minlength=length)
    idx = np.arange(layout.size, dtype=np.int64)[inside]
    inv[v[inside]] = idx
    inv[counts > 1] = -2
    return inv


def right_inverse_values(layout) -> np.ndarray:
    """For a layout that is a bijection onto [0, size): the logical index at
    every offset, i.e. L^-1 as a table with L(L^-1(j)) = j."""
    inv = inverse_map(layout, layout.size)
    if (inv < 0).any():
        raise ValueError("layout is not a bijection onto [0, size)")
    return inv


def max_common_vector(a, b) -> int:
    """K = max{k : A^-1(j) = B^-1(j) for every j < k} ("CUTE布局代数" §2.3):
    the number of leading offsets at which both layouts hold the same logical
    element, so that a copy between them may move those K elements as one
    contiguous vector.  Offsets with no or several preimages end the run."""
    n = max(cosize(a), cosize(b))
    inv_a = inverse_map(a, n)
    inv_b = inverse_map(b, n)
    k = 0
    while k < n and inv_a[k] >= 0 and inv_a[k] == inv_b[k]:
        k += 1
    return k


# ---------------------------------------------------------------------------
# complement and products ("CUTE布局代数" §4.1)
# ---------------------------------------------------------------------------

def complement(layout: Layout, cotarget: int) -> Layout:
    """The layout that fills in what ``layout`` leaves out, up to cotarget.

    The pages name the products of §4.1 without defining them; the
    complement they rest on is taken as: walk the leaves by increasing
    stride; whenever the next stride d exceeds the span c reached so far,
    the gap contributes a leaf (d // c):c; the span becomes extent * d; a
    last leaf ceil(cotarget / c):c reaches cotarget.  Leaves of extent 1 or
    stride 0 add nothing.  A stride that is not a multiple of the span
    reached so far has no such complement (ValueError)."""
    leaves = sorted(((e, d) for e, d in layout.leaves if e > 1 and d > 0),
                    key=lambda ed: (ed[1], ed[0]))
    shape, stride = [], []
    span = 1
    for e, d in leaves:
        if d < span or d % span:
            raise ValueError("strides do not nest: no complement")
        if d // span > 1:
            shape.append(d // span)
            stride.append(span)
        span = e * d
    rest = -(-cotarget // span)
    if rest > 1:
        shape.append(rest)
        stride.append(span)
    if not shape:
        return Layout(1, 0)
    return Layout(tuple(shape), tuple(stride))


class LogicalProduct:
    """logical_product(A, B): the layout (A, complement(A, size(A) *
    cosize(B)) o B) -- A repeated at the positions B lists, each step of B
    skipping one whole copy of A."""

    def __init__(self, a: Layout, b: Layout):
        self.a = a
        self.rest = Composed(complement(a, a.size * cosize(b)), b)
        self.size = a.size * b.size

    def at(self, i, extended: bool = False) -> np.ndarray:
        x = _as_index(i)
        return self.a.at(x % self.a.size) + self.rest.at(x // self.a.size)

    __call__ = at


class BlockedProduct:
    """blocked_product(A, B) for layouts of equal rank r: mode k of the
    result is (mode k of A, mode k of complement(A, size(A)*cosize(B)) o B),
    so the tile A is laid out at every grid position of B.  The page's
    example, a 4x8 tile over a 2x5 grid, makes a layout of shape
    ((4,2),(8,5))."""

    def __init__(self, a: Layout, b: Layout):
        self.a_modes = a.modes()
        self.b_modes = b.modes()
        if len(self.a_modes) != len(self.b_modes):
            raise ValueError("blocked_product needs operands of equal rank")
        self.a = a
        self.c = complement(a, a.size * cosize(b))
        self.b = b
        self.size = a.size * b.size

    def at(self, i, extended: bool = False) -> np.ndarray:
        x = _as_index(i)
        a_idx = np.zeros_like(x)
        b_idx = np.zeros_like(x)
        a_w = b_w = 1
        for am, bm in zip(self.a_modes, self.b_modes):
            xk = x % (am.size * bm.size)        # this mode's coordinate
            x = x // (am.size * bm.size)
            a_idx = a_idx + (xk % am.size) * a_w   # A's part, colex in A
            b_idx = b_idx + (xk // am.size) * b_w  # B's part, colex in B
            a_w *= am.size
            b_w *= bm.size
        return self.a.at(a_idx) + self.c.at(self.b.at(b_idx), extended=True)

    __call__ = at


# ---------------------------------------------------------------------------
# thread maps (PitchLinearStripminedThreadMap article, hotelren.com)
# ---------------------------------------------------------------------------

def pitch_linear_offset(thread_id, k_row: int, pitch: int):
    """§1.2: the thread's row is thread_id / Pitch, its column
    thread_id % Pitch, and its offset column + row * kRow."""
    t = _as_index(thread_id)
    return (t % pitch) + (t // pitch) * k_row


def stripmined_offset(thread_id, k_row: int, pitch: int, strips: int):
    """§2.2's stripmined map, read as a layout: a thread id is a logical
    index into the three modes (Pitch, Strips, groups) -- a position inside
    the Pitch, a strip inside Strips, and the whole Pitch x Strips groups
    before it -- whose strides are 1 element, one kRow row per strip, and
    Pitch*Strips rows of kRow per group.  The offset is that layout
    evaluated by the generic colex evaluator (``Layout.at``), with as many
    groups as the largest thread id needs."""
    t = _as_index(thread_id)
    per_group = pitch * strips
    groups = int(t.max()) // per_group + 1 if t.size else 1
    L = Layout((pitch, strips, groups), (1, k_row, per_group * k_row))
    return L.at(t)


# ---------------------------------------------------------------------------
# thread partitions ("CUTLASS Layout可视化" §5.3)
# ---------------------------------------------------------------------------

def thread_coordinate(thr: Layout, thr_idx: int) -> list[int]:
    """§5.3: the thread layout maps a coordinate to a thread number; this
    is the per-mode coordinate (a 1-D index into each top mode of thr) that
    it maps to thread number thr_idx, found by trying every coordinate.
    thr must reach thr_idx exactly once."""
    hits = np.nonzero(thr.at(np.arange(thr.size)) == thr_idx)[0]
    if len(hits) != 1:
        raise ValueError("the thread layout must reach the thread once")
    i = int(hits[0])
    coord = []
    for m in thr.modes():
        coord.append(i % m.size)
        i //= m.size
    return coord


def local_partition(layout, thr: Layout, thr_idx: int) -> np.ndarray:
    """§5.3's local_partition(tile, thread_layout, thread_idx): the
    elements of `layout` that thread thr_idx owns.  With T_k the size of the
    thread layout's mode k (1 past its rank) and c the thread's coordinate,
    the thread owns, in every mode k, the coordinates x_k = c_k + T_k * r_k:
    one element of every T_0 x T_1 x ... block, at the thread's place in the
    block.  Returns their offsets, r taken colex (r_0 fastest); a swizzled
    layout's swizzle applies to each whole offset."""
    base = layout.inner if isinstance(layout, Swizzled) else layout
    modes = base.modes()
    tm = thr.modes()
    if len(tm) > len(modes):
        raise ValueError("thread layout of higher rank than the tile")
    c = thread_coordinate(thr, thr_idx) + [0] * (len(modes) - len(tm))
    t = [m.size for m in tm] + [1] * (len(modes) - len(tm))
    for m, tk in zip(modes, t):
        if m.size % tk:
            raise ValueError("thread layout extents must divide the tile")
    rest = [m.size // tk for m, tk in zip(modes, t)]
    out = []
    for r_flat in range(prod(rest)):
        off = 0
        for m, ck, tk, nk in zip(modes, c, t, rest):
            rk = r_flat % nk
            r_flat //= nk
            off += int(m.at(ck + tk * rk))
        out.append(off)
    off = np.array(out, dtype=np.int64)
    if isinstance(layout, Swizzled):
        off = swizzle(off, layout.b, layout.m, layout.s)
    return off


# ---------------------------------------------------------------------------
# shared-memory banks ("CUTLASS Layout可视化" §5.2, §6.4)
# ---------------------------------------------------------------------------

def smem_wavefronts(byte_addr, access_bytes: int) -> tuple[int, int]:
    """§5.2: shared memory is 32 banks of 4 bytes; lanes of one warp that
    touch different 4-byte words of the same bank are served one after the
    other, lanes that read the same word share it.  Accesses of 8 or 16
    bytes per lane are served 16 or 8 lanes at a time (128 bytes).  Access
    i belongs to warp i // 32.  Returns (wavefronts, conflict-free minimum)
    summed over every group of lanes served together."""
    addr = [int(a) for a in np.asarray(byte_addr, dtype=np.int64).ravel()]
    per_group = 32 if access_bytes <= 4 else 128 // access_bytes
    words_per_lane = max(1, access_bytes // 4)
    total = ideal = 0
    for w0 in range(0, len(addr), 32):
        warp = addr[w0:w0 + 32]
        for g0 in range(0, len(warp), per_group):
            group = warp[g0:g0 + per_group]
            words_in_bank = {}
            for a in group:
                for k in range(words_per_lane):
                    word = a // 4 + k
                    words_in_bank.setdefault(word % 32, set()).add(word)
            total += max(len(v) for v in words_in_bank.values())
            ideal += max(1, -(-len(group) * access_bytes // 128))
    return total, ideal


# ---------------------------------------------------------------------------
# the copy
# ---------------------------------------------------------------------------

def _element_view(buf: np.ndarray, elem_bytes: int) -> np.ndarray:
    if buf.dtype != np.uint8 or buf.ndim != 1:
        raise ValueError("buffers are flat uint8 arrays")
    if buf.size % elem_bytes:
        raise ValueError("buffer length is not a whole number of elements")
    return buf.view(np.dtype((np.void, elem_bytes)))


def copy(src, dst, inp: np.ndarray, out: np.ndarray, elem_bytes: int,
         indices: Iterable[int] | None = None) -> None:
    """out[dst(i)] = in[src(i)] for every logical index i (or only for the
    given ones), moving elem_bytes raw bytes per element, so no value is
    converted and NaN payloads survive.  Slots of ``out`` outside dst's image
    are left as they were.  A destination that two indices share is
    rejected: the pages define no order between such writes."""
    if src.size != dst.size:
        raise ValueError("source and destination layouts differ in size")
    if indices is None:
        idx = np.arange(src.size, dtype=np.int64)
    else:
        idx = _as_index(list(indices) if not isinstance(indices, np.ndarray)
                        else indices)
    s = src.at(idx)
    d = dst.at(idx)
    if indices is None and np.unique(d).size != d.size:
        raise ValueError("destination layout is not injective")
    vin = _element_view(inp, elem_bytes)
    vout = _element_view(out, elem_bytes)
    vout[d] = vin[s]


def copy_loop(src, dst, inp: np.ndarray, out: np.ndarray,
              elem_bytes: int) -> None:
    """The same copy as a plain Python loop, one element at a time (small
    cases only)."""
    if src.size != dst.size:
        raise ValueError("source and destination layouts differ in size")
    seen = set()
    for i in range(src.size):
        s = int(src.at(np.int64(i)))
        d = int(dst.at(np.int64(i)))
        if d in seen:
            raise ValueError("destination layout is not injective")
        seen.add(d)
        out[d * elem_bytes:(d + 1) * elem_bytes] = \
            inp[s * elem_bytes:(s + 1) * elem_bytes]


# ---------------------------------------------------------------------------
# building layouts from the workload descriptions
# ---------------------------------------------------------------------------

def parse(text: str) -> Layout:
    """"(4,2):(2,1)" -> Layout((4,2),(2,1)) (the notation the print_layout
    example prints, without the static-integer underscores)."""
    depth = 0
    split = None
    for pos, ch in enumerate(text):
        if ch == "(":
            depth += 1
        elif ch == ")":
            depth -= 1
        elif ch == ":" and depth == 0:
            split = pos
    if split is None:
        raise ValueError("expected shape:stride")
    clean = text.replace("_", "")
    shape = ast.literal_eval(clean[:split].strip())
    stride = ast.literal_eval(clean[split + 1:].strip())
    return Layout(shape, stride)


def build(spec):
    """Turn a workload description (nested tuples, see ``workloads``) into an
    oracle expression.

    ("layout", shape, stride) | ("swizzle", B, M, S, spec) |
    ("compose", outer, inner) | ("zipped_divide", spec, tiler) |
    ("concat", spec, spec, ...) | ("blocked_product", tile, grid) |
    ("logical_product", tile, grid); the products take plain layouts"""
    kind = spec[0]
    if kind == "layout":
        return Layout(spec[1], spec[2])
    if kind == "swizzle":
        return Swizzled(spec[1], spec[2], spec[3], build(spec[4]))
    if kind == "compose":
        return Composed(build(spec[1]), build(spec[2]))
    if kind == "zipped_divide":
        return ZippedDivide(build(spec[1]), spec[2])
    if kind == "concat":
        return Concat(*[build(s) for s in spec[1:]])
    if kind == "blocked_product":
        return BlockedProduct(build(spec[1]), build(spec[2]))
    if kind == "logical_product":
        return LogicalProduct(build(spec[1]), build(spec[2]))
    raise ValueError(f"unknown layout description {kind!r}")
