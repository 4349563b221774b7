"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (fixtures under tests/golden/, each with its citation), closed
forms derived by hand, textbook special cases (numpy transposes), and
invariants.  ``test_pins_catch_planted_mistakes`` plants plausible mistakes
in the oracle and checks that some pin fails for each.
"""

import itertools

import numpy as np
import pytest

from golden_io import load
from oracle import layout_oracle as lo
from workloads import WORKLOADS

TV = lo.Layout(((4, 8), 2), ((16, 1), 8))


# --------------------------------------------------------------------------
# shape:stride evaluation ("CUTLASS Layout可视化" §2.1, §3.3, §4.1)
# --------------------------------------------------------------------------

def pin_rowmajor_grid():
    g = load("rowmajor_4x2.txt")
    L = lo.parse(g["layout"])
    assert lo.print_grid(L) == g["grid"]
    for r, c, off in g["point"]:
        assert int(lo.eval_2d(L, r, c)) == off


def pin_colmajor_grid():
    g = load("colmajor_4x2.txt")
    assert lo.print_grid(lo.parse(g["layout"])) == g["grid"]


def test_rowmajor_grid():
    pin_rowmajor_grid()


def test_colmajor_grid():
    pin_colmajor_grid()


def test_parse_accepts_static_marks():
    # "RowMajor 4x2: (4,2):(_2,_1)" is how the example prints it (§3.2)
    L = lo.parse("(4,2):(_2,_1)")
    assert L.shape == (4, 2) and L.stride == (2, 1)


def pin_blocked_leaf_coordinates():
    """R3: the page's sample for ((4,2),(2,4)):((2,16),(1,8)) is the bare
    inner product of leaf coordinate (r, c, 0, 0) with the leaf strides,
    i.e. 2r + 16c; for c in {2,3} it lies outside mode 0's second leaf."""
    g = load("blocked_points.txt")
    L = lo.parse(g["layout"])
    for r, c, off in g["point"]:
        assert lo.eval_leaf_coord(L, (r, c, 0, 0)) == off


def test_blocked_leaf_coordinates():
    pin_blocked_leaf_coordinates()


def test_blocked_two_dimensional_reading():
    """The other reading of the same layout: (row, col) each a colex index
    into its mode.  Points worked by hand: mode 0 = (4,2):(2,16) takes row 3
    to 3*2 = 6, mode 1 = (2,4):(1,8) takes col 3 to 1*1 + 1*8 = 9."""
    L = lo.parse("((4,2),(2,4)):((2,16),(1,8))")
    assert int(lo.eval_2d(L, 0, 1)) == 1
    assert int(lo.eval_2d(L, 1, 0)) == 2
    assert int(lo.eval_2d(L, 3, 3)) == 6 + 9
    assert int(lo.eval_2d(L, 4, 0)) == 16      # row 4 = (0,1) of mode 0
    assert int(lo.eval_2d(L, 0, 2)) == 8       # col 2 = (0,1) of mode 1
    grid = np.array(lo.print_grid(L))
    # 64 coordinates, 48 distinct offsets, all below 48: the mode-1 stride 8
    # and mode-0 stride 16 collide (8*2 == 16), so the layout is no bijection
    assert grid.shape == (8, 8)
    assert np.unique(grid).size == 48
    assert grid.max() == 47 and lo.cosize(L) == 48
    assert not lo.is_injective(L)


# --------------------------------------------------------------------------
# colex order pinned by the stripmined formula and the column-major example
# --------------------------------------------------------------------------

def pin_stripmined_page_values():
    g = load("stripmined.txt")
    for k_row, pitch, strips, t0, t1, o0, o1 in g["range"]:
        t = np.arange(t0, t1 + 1)
        got = lo.stripmined_offset(t, k_row, pitch, strips)
        assert got.tolist() == list(range(o0, o1 + 1))


def test_stripmined_page_values():
    pin_stripmined_page_values()


def test_stripmined_host_program_listing_values():
    """The article's host simulator (§5.3) loops t = 0..63 with kPitch=8,
    kStrips=4, kRow=16.  Threads 32..63 are threads 0..31 shifted by 512."""
    t = np.arange(64)
    off = lo.stripmined_offset(t, 16, 8, 4)
    assert (off[32:] == off[:32] + 512).all()
    assert off[63] == 567 and off[8] == 16 and off[24] == 48


def _get_offset_by_hand(t, k_row, pitch, strips):
    """The article's §2.2 get_offset, worked as its three named parts: the
    position inside the Pitch, the strip inside Strips, the group of
    Pitch x Strips threads; each part times its step."""
    pos, strip, group = t % pitch, (t // pitch) % strips, t // (pitch * strips)
    return pos + strip * k_row + group * (pitch * strips * k_row)


def pin_stripmined_is_colex_layout():
    """R1: the page's get_offset arithmetic equals the oracle's generic
    evaluator on the layout (Pitch, Strips, G):(1, kRow, Pitch*Strips*kRow)
    only if that evaluator splits an index first-leaf-fastest, so this pins
    colex order (the oracle's stripmined map is that layout; the page's
    arithmetic lives only here)."""
    for pitch, strips, k_row in itertools.product((1, 2, 3, 8), (1, 2, 4, 5),
                                                  (1, 7, 16)):
        groups = 6
        L = lo.Layout((pitch, strips, groups),
                      (1, k_row, pitch * strips * k_row))
        t = np.arange(L.size)
        want = _get_offset_by_hand(t, k_row, pitch, strips)
        assert (L.at(t) == want).all()
        assert (lo.stripmined_offset(t, k_row, pitch, strips) == want).all()
        # one thread at a time sizes the groups from that thread alone
        assert lo.stripmined_offset(int(t[-1]), k_row, pitch,
                                    strips) == want[-1]


def test_stripmined_is_colex_layout():
    pin_stripmined_is_colex_layout()


def test_stripmined_reduces_to_pitch_linear():
    """R5: when one group of Pitch x Strips covers every thread
    (Pitch*Strips >= Threads) the stripmined map is the plain pitch-linear
    map row = t/Pitch, col = t%Pitch, offset = col + row*kRow (§1.2).  The
    article's Strips=1 claim holds only when Pitch is 1 or Threads <= Pitch:
    with Strips=1 the formula multiplies the row by Pitch*kRow."""
    for threads, pitch, strips, k_row in itertools.product(
            (8, 32, 64), (1, 4, 8), (1, 2, 4, 8, 64), (16, 33)):
        t = np.arange(threads)
        strip = lo.stripmined_offset(t, k_row, pitch, strips)
        plain = lo.pitch_linear_offset(t, k_row, pitch)
        if pitch * strips >= threads:
            assert (strip == plain).all()
        if strips == 1:
            same = bool((strip == plain).all())
            assert same == (pitch == 1 or threads <= pitch)
    # the article's own example: Strips=1, kRow=16, Pitch=8, thread 8
    assert lo.stripmined_offset(8, 16, 8, 1) == 128
    assert lo.pitch_linear_offset(8, 16, 8) == 16


def pin_column_major_composition_is_identity():
    """"CUTE布局代数" §3.1: composing the column-major 8x8 user layout with
    the thread-value layout.  (8,8):(1,8) is the identity on [0,64) only
    when the first mode runs fastest, so the result must equal TV."""
    user = lo.Layout((8, 8), (1, 8))
    R = lo.Composed(user, TV)
    i = np.arange(64)
    assert (R.at(i) == TV.at(i)).all()


def test_column_major_composition_is_identity():
    pin_column_major_composition_is_identity()


def test_thread_value_layout_is_bijection():
    """((4,8),2):((16,1),8) covers [0,64) once: thread stride 16 over 4,
    1 over 8, value stride 8 over 2 (§1, §3.1)."""
    assert sorted(lo.image(TV).tolist()) == list(range(64))


# --------------------------------------------------------------------------
# composition ("CUTE布局代数" §2.2)
# --------------------------------------------------------------------------

def pin_padded_composition_closed_form():
    """(8,8):(1,9) o ((4,8),2):((16,1),8).  Worked by hand: the thread mode
    4:16 steps over two whole columns of 8 per step, i.e. 2 columns of pitch
    9 = 18; the 8:1 mode walks inside a column (1); the value mode 2:8 steps
    one column (9).  Closed form ((4,8),2):((18,1),9)."""
    padded = lo.Layout((8, 8), (1, 9))
    R = lo.Composed(padded, TV)
    closed = lo.Layout(((4, 8), 2), ((18, 1), 9))
    i = np.arange(64)
    assert (R.at(i) == closed.at(i)).all()
    # "padding is skipped": no result lands on a pad slot (offset % 9 == 8)
    assert (R.at(i) % 9 != 8).all()
    assert np.unique(R.at(i)).size == 64


def test_padded_composition_closed_form():
    pin_padded_composition_closed_form()


def test_composition_invariants():
    """Identity on either side leaves a layout unchanged, and composition is
    associative (checked on small random layouts)."""
    rng = np.random.default_rng(7)
    for _ in range(40):
        n = int(rng.integers(1, 4))
        shape = tuple(int(v) for v in rng.integers(1, 5, size=n))
        stride = tuple(int(v) for v in rng.integers(0, 9, size=n))
        A = lo.Layout(shape, stride)
        size = A.size
        ident = lo.Layout(size, 1)
        i = np.arange(size)
        assert (lo.Composed(A, ident).at(i) == A.at(i)).all()
        cos = lo.cosize(A)
        big_ident = lo.Layout(max(cos, 1), 1)
        assert (lo.Composed(big_ident, A).at(i) == A.at(i)).all()
        B = lo.Layout((2, 3), (int(rng.integers(1, 4)), int(rng.integers(0, 5))))
        C = lo.Layout((3,), (int(rng.integers(0, 3)),))
        j = np.arange(C.size)
        left = lo.Composed(lo.Composed(A, B), C).at(j)
        right = lo.Composed(A, lo.Composed(B, C)).at(j)
        assert (left == right).all()


# --------------------------------------------------------------------------
# zipped_divide ("CUTE布局代数" §3.2)
# --------------------------------------------------------------------------

def pin_zipped_divide_closed_form():
    """zipped_divide((128,128):(1,128), (4,8)): tiles of 4 rows x 8 columns.
    Worked by hand: tile modes (4:1, 8:128); rest modes step one tile,
    4 rows = 4 and 8 columns = 8*128 = 1024, over 32 x 16 tiles."""
    Z = lo.ZippedDivide(lo.Layout((128, 128), (1, 128)), (4, 8))
    closed = lo.Layout(((4, 8), (32, 16)), ((1, 128), (4, 1024)))
    i = np.arange(Z.size)
    assert (Z.at(i) == closed.at(i)).all()


def test_zipped_divide_closed_form():
    pin_zipped_divide_closed_form()


def test_zipped_divide_tile_is_numpy_block():
    """The page's "take tile (3,5)": that tile is the numpy block
    rows 12..15, cols 40..47 of the 128x128 offset table, read column-major
    (tile modes are colex)."""
    L = lo.Layout((128, 128), (1, 128))
    Z = lo.ZippedDivide(L, (4, 8))
    table = np.array([[int(lo.eval_2d(L, r, c)) for c in range(128)]
                      for r in range(128)])
    g = 3 + 32 * 5
    got = Z.at(np.arange(32) + 32 * g)
    want = table[12:16, 40:48].flatten(order="F")
    assert (got == want).all()


def test_zipped_divide_c3_source_closed_form():
    """The bf16 8192x8192 source cut into 64x64 tiles:
    ((64,64),(128,128)):((8192,1),(524288,64)) (rows step 8192, a tile row
    of tiles steps 64 rows = 524288, a tile column steps 64 elements)."""
    Z = lo.build(WORKLOADS["C3"].src)
    closed = lo.Layout(((64, 64), (128, 128)), ((8192, 1), (524288, 64)))
    rng = np.random.default_rng(3)
    i = rng.integers(0, Z.size, size=200000)
    assert (Z.at(i) == closed.at(i)).all()


# --------------------------------------------------------------------------
# swizzle ("CUTLASS Layout可视化" §4.3)
# --------------------------------------------------------------------------

def pin_swizzle_page_formula():
    """Swizzle<3,0,3> on the row-major 8x8 block equals the page's
    row*8 + (col ^ row) for every (row, col), reproduces the worked values
    18 and 19, and maps every printed row onto the same set of offsets."""
    g = load("swizzle_8x8.txt")
    base = lo.parse(g["layout"])
    for r, *row in g["base_row"]:
        assert [int(lo.eval_2d(base, r, c)) for c in range(8)] == row
    S = lo.Swizzled(3, 0, 3, base)
    for r in range(8):
        for c in range(8):
            assert int(lo.eval_2d(S, r, c)) == r * 8 + (c ^ r)
    for r, c, off in g["worked"]:
        assert int(lo.eval_2d(S, r, c)) == off
    for r, *printed in g["printed_row"]:
        mine = [int(lo.eval_2d(S, r, c)) for c in range(8)]
        assert sorted(mine) == sorted(printed)
    # R4: the formula's rows (the printed rows contradict them)
    assert [int(lo.eval_2d(S, 1, c)) for c in range(8)] == \
        [9, 8, 11, 10, 13, 12, 15, 14]
    assert [int(lo.eval_2d(S, 2, c)) for c in range(8)] == \
        [18, 19, 16, 17, 22, 23, 20, 21]


def test_swizzle_page_formula():
    pin_swizzle_page_formula()


def test_swizzle_invariants():
    """Involution, bijection on aligned blocks of 2^(B+M+S), identity where
    bits [M+S, M+S+B) are zero, and 2^M-element atoms stay contiguous."""
    for b, m, s in [(3, 0, 3), (3, 4, 3), (2, 1, 4), (1, 3, 1), (0, 2, 2),
                    (3, 3, 5)]:
        n = 1 << (b + m + s + 1)
        o = np.arange(n)
        w = lo.swizzle(o, b, m, s)
        assert (lo.swizzle(w, b, m, s) == o).all()
        blk = 1 << (b + m + s)
        for start in range(0, n, blk):
            assert sorted(w[start:start + blk].tolist()) == \
                list(range(start, start + blk))
        quiet = ((o >> (m + s)) & ((1 << b) - 1)) == 0
        assert (w[quiet] == o[quiet]).all()
        atoms = w.reshape(-1, 1 << m)
        assert (np.diff(atoms, axis=1) == 1).all()
        assert (atoms[:, 0] % (1 << m) == 0).all()


# --------------------------------------------------------------------------
# inverse and common vector ("CUTE布局代数" §2.3)
# --------------------------------------------------------------------------

def test_right_inverse_of_transpose_is_transpose():
    """Row-major (m,n):(n,1) stores (r,c) at n*r+c; the element at offset j
    is r = j//n, c = j%n, logical index r + m*c = (j//n) + m*(j%n): the
    layout (n,m):(m,1)."""
    for m, n in [(4, 2), (3, 5), (8, 8), (1, 7)]:
        L = lo.Layout((m, n), (n, 1))
        want = lo.Layout((n, m), (m, 1))
        j = np.arange(m * n)
        assert (lo.right_inverse_values(L) == want.at(j)).all()


def test_right_inverse_round_trip():
    rng = np.random.default_rng(11)
    for _ in range(30):
        ext = [int(v) for v in rng.integers(1, 5, size=3)]
        perm = rng.permutation(3)
        stride = [0, 0, 0]
        acc = 1
        for k in perm:
            stride[k] = acc
            acc *= ext[k]
        L = lo.Layout(tuple(ext), tuple(stride))
        inv = lo.right_inverse_values(L)
        j = np.arange(L.size)
        assert (L.at(inv) == j).all()
        assert (inv[L.at(j)] == j).all()


def test_max_common_vector_cases():
    i64 = lo.Layout((8, 8), (1, 8))
    # identical compact layouts: every offset agrees
    assert lo.max_common_vector(i64, i64) == 64
    row = lo.Layout((4, 2), (2, 1))
    assert lo.max_common_vector(row, row) == 8
    # column- vs row-major 8x8: offset 1 holds logical 1 vs logical 8
    assert lo.max_common_vector(i64, lo.Layout((8, 8), (8, 1))) == 1
    # (4):(2) has no element at offset 1
    assert lo.max_common_vector(lo.Layout(4, 1), lo.Layout(4, 2)) == 1
    # the bf16 tiling: 64 elements of a tile row sit at offsets 0..63 on both
    # sides; offset 64 is the next tile on the source, the next row on the
    # destination.  The swizzle leaves offsets below 2^(M+S) = 128 alone.
    c3 = WORKLOADS["C3"]
    small_src = ("zipped_divide", ("layout", (256, 256), (256, 1)), (64, 64))
    small_dst = ("swizzle", 3, 4, 3,
                 ("layout", ((64, 64), (4, 4)), ((64, 1), (16384, 4096))))
    assert c3.dst[1:4] == small_dst[1:4]
    assert lo.max_common_vector(lo.build(small_src), lo.build(small_dst)) == 64


# --------------------------------------------------------------------------
# the copy ("CUTE布局代数" §5.1; closed forms of the workloads)
# --------------------------------------------------------------------------

def _run_copy(src, dst, eb, values, cos_out=None, fill=0xA5):
    n_in = lo.cosize(src)
    n_out = cos_out if cos_out is not None else lo.cosize(dst)
    rng = np.random.default_rng(5)
    inp = values if values is not None else rng.integers(
        0, 256, size=n_in * eb, dtype=np.uint8)
    out = np.full(n_out * eb, fill, dtype=np.uint8)
    lo.copy(src, dst, inp, out, eb)
    return inp, out


def pin_copy_transpose():
    """Column-major (m,n) -> row-major is numpy's transpose."""
    for m, n in [(5, 3), (64, 48), (200, 136)]:
        src = lo.Layout((m, n), (1, m))
        dst = lo.Layout((m, n), (n, 1))
        a = np.random.default_rng(m).random(m * n, dtype=np.float32)
        inp = a.view(np.uint8)
        _, out = _run_copy(src, dst, 4, inp)
        mat = a.reshape(n, m)            # column-major storage: [c][r]
        assert (out.view(np.float32) == mat.T.flatten()).all()


def test_copy_transpose():
    pin_copy_transpose()


def test_copy_nhwc_to_nchw():
    N, C, H, W = 2, 24, 5, 7
    src = lo.Layout((N, C, H, W), (H * W * C, 1, W * C, C))
    dst = lo.Layout((N, C, H, W), (C * H * W, H * W, W, 1))
    a = np.random.default_rng(1).standard_normal(N * H * W * C).astype(
        np.float16)
    _, out = _run_copy(src, dst, 2, a.view(np.uint8))
    want = a.reshape(N, H, W, C).transpose(0, 3, 1, 2).flatten()
    assert (out.view(np.float16).view(np.uint16) ==
            want.view(np.uint16)).all()


def test_copy_head_interleave():
    """Two heads of S x D, head-major -> head fastest (offset 2*(s*D+d)+h)."""
    S, D = 6, 8
    src = lo.Layout((2, S, D), (S * D, D, 1))
    dst = lo.Layout((2, S, D), (1, 2 * D, 2))
    a = np.arange(2 * S * D, dtype=np.uint16)
    _, out = _run_copy(src, dst, 2, a.view(np.uint8))
    want = np.stack([a[:S * D], a[S * D:]], axis=1).flatten()
    assert (out.view(np.uint16) == want).all()


def test_interleave_page_list():
    """The interleaved rule (head stride 1, the column-major strides
    doubled) reproduces the page's per-head list."""
    g = load("interleave_list.txt")
    L = lo.Layout((4, 2, 2), (2, 8, 1))            # (row, col, head)
    for head, r, c, off in g["entry"]:
        assert lo.eval_leaf_coord(L, (r, c, head)) == off


def test_copy_padded_tv_gather_closed_form():
    """R11: out[b*64 + t0 + 4*t1 + 32*v] = in[b*72 + 18*t0 + t1 + 9*v],
    written as explicit loops over b, t0, t1, v."""
    batch = 5
    src = lo.build(("concat", WORKLOADS["C4"].src[1], ("layout", batch, 72)))
    dst = lo.Layout((((4, 8), 2), batch), (((1, 4), 32), 64))
    a = np.random.default_rng(2).random(72 * batch)
    _, out = _run_copy(src, dst, 8, a.view(np.uint8))
    got = out.view(np.float64)
    for b in range(batch):
        for t0 in range(4):
            for t1 in range(8):
                for v in range(2):
                    assert got[b * 64 + t0 + 4 * t1 + 32 * v] == \
                        a[b * 72 + 18 * t0 + t1 + 9 * v]


def test_copy_c1_closed_form():
    w = WORKLOADS["C1"]
    src, dst = lo.build(w.src), lo.build(w.dst)
    a = np.arange(64, dtype=np.int32) * 1000 + 7
    _, out = _run_copy(src, dst, 4, a.view(np.uint8))
    got = out.view(np.int32)
    for r in range(8):
        for c in range(8):
            assert got[8 * r + (c ^ r)] == a[r + 8 * c]


def test_copy_matches_python_loop():
    rng = np.random.default_rng(9)
    cases = [(lo.build(WORKLOADS["C1"].src), lo.build(WORKLOADS["C1"].dst), 4),
             (lo.Layout((3, 4, 2), (8, 1, 4)), lo.Layout((3, 4, 2), (1, 3, 12)), 2),
             (lo.Composed(lo.Layout((8, 8), (1, 9)), TV),
              lo.Layout(((4, 8), 2), ((1, 4), 32)), 8)]
    for src, dst, eb in cases:
        inp = rng.integers(0, 256, size=lo.cosize(src) * eb, dtype=np.uint8)
        a = np.full(lo.cosize(dst) * eb, 0x5A, dtype=np.uint8)
        b = a.copy()
        lo.copy(src, dst, inp, a, eb)
        lo.copy_loop(src, dst, inp, b, eb)
        assert (a == b).all()


def test_copy_keeps_nan_payloads_and_untouched_slots():
    src = lo.Layout(4, 1)
    dst = lo.Layout(4, 3)                      # touches 0,3,6,9 of 10
    payload = np.array([0x7FF8DEADBEEF0001, 0xFFF0000000000123,
                        0x0000000000000001, 0x7FF0000000000000],
                       dtype=np.uint64)
    out = np.full(10 * 8, 0xA5, dtype=np.uint8)
    lo.copy(src, dst, payload.view(np.uint8), out, 8)
    got = out.view(np.uint64)
    assert got[[0, 3, 6, 9]].tolist() == payload.tolist()
    untouched = [k for k in range(10) if k % 3]
    assert (out.reshape(10, 8)[untouched] == 0xA5).all()


def test_copy_rejects_non_injective_destination():
    src = lo.Layout((8, 8), (1, 8))
    dst = lo.parse("((4,2),(2,4)):((2,16),(1,8))")
    with pytest.raises(ValueError):
        _run_copy(src, dst, 4, None)
    with pytest.raises(ValueError):
        lo.copy(lo.Layout(4, 1), lo.Layout(5, 1), np.zeros(16, np.uint8),
                np.zeros(20, np.uint8), 4)


def test_eval_rejects_out_of_domain():
    L = lo.Layout((4, 2), (2, 1))
    with pytest.raises(IndexError):
        L.at(8)
    with pytest.raises(IndexError):
        L.at(-1)


def test_workload_closed_forms_small_samples():
    """Spot checks of the full-size workload layouts at hand-worked points."""
    c2s, c2d = (lo.build(WORKLOADS["C2"].src), lo.build(WORKLOADS["C2"].dst))
    i = 5 + 4096 * 7                       # (row 5, col 7)
    assert int(c2s.at(i)) == 5 + 4096 * 7 and int(c2d.at(i)) == 5 * 4096 + 7
    c3d = lo.build(WORKLOADS["C3"].dst)
    # element (r=3, c=16) of tile (tr=0, tc=1) sits in tile 1 (base 4096),
    # row 3 (192); its 16-element chunk 1 is XORed with row//2 = 1 -> chunk 0
    i = 3 + 64 * 16 + 4096 * (0 + 128 * 1)
    assert int(c3d.at(i)) == 4096 + 192 + 0
    # (r=1, c=16): row//2 = 0 leaves the chunk alone
    i = 1 + 64 * 16 + 4096 * 128
    assert int(c3d.at(i)) == 4096 + 64 + 16
    c5s, c5d = (lo.build(WORKLOADS["C5a"].src), lo.build(WORKLOADS["C5a"].dst))
    n, c, h, w = 3, 17, 9, 40
    i = n + 64 * (c + 256 * (h + 56 * w))
    assert int(c5s.at(i)) == ((n * 56 + h) * 56 + w) * 256 + c
    assert int(c5d.at(i)) == ((n * 256 + c) * 56 + h) * 56 + w


# --------------------------------------------------------------------------
# complement and products ("CUTE布局代数" §4.1)
# --------------------------------------------------------------------------

def pin_complement_worked_examples():
    """Worked by hand from the definition (gap leaves in stride order, then
    a leaf up to the cotarget)."""
    cases = [((4, 1, 24), (6, 4)),              # 4:1 -> the other 6 copies
             ((6, 4, 24), (4, 1)),              # 6:4 -> the 4 inside
             ((4, 2, 16), ((2, 2), (1, 8)))]     # gap of 1 below 2, then 8
    for (e, d, m), (shape, stride) in cases:
        C = lo.complement(lo.Layout(e, d), m)
        want = lo.Layout(shape, stride)
        assert C.size == want.size
        assert (C.at(np.arange(C.size)) == want.at(np.arange(C.size))).all()
    C = lo.complement(lo.Layout((2, 2), (1, 6)), 24)
    assert (C.at(np.arange(6)) == lo.Layout((3, 2), (2, 12)).at(np.arange(6))).all()
    full = lo.complement(lo.Layout((4, 6), (1, 4)), 24)
    assert full.size == 1


def test_complement_worked_examples():
    pin_complement_worked_examples()


def test_complement_invariants():
    """(A, complement(A, M)) never repeats an offset, and covers [0, M)
    exactly when M is a multiple of A's span."""
    rng = np.random.default_rng(21)
    for _ in range(100):
        n = int(rng.integers(1, 4))
        ext = [int(v) for v in rng.integers(1, 5, n)]
        stride, span = [], 1
        for e in ext:                        # nested strides with gaps
            span *= int(rng.integers(1, 3))
            stride.append(span)
            span *= e
        A = lo.Layout(tuple(ext), tuple(stride))
        M = span * int(rng.integers(1, 4))
        C = lo.complement(A, M)
        both = lo.Concat(A, C)
        img = lo.image(both)
        assert np.unique(img).size == img.size
        assert sorted(img.tolist()) == list(range(M))
    with pytest.raises(ValueError):
        lo.complement(lo.Layout((2, 3), (1, 3)), 12)     # 3 is not 2-nested


def pin_blocked_product_page_example():
    """A 4x8 tile (column-major) over a 2x5 grid: the page's shape
    ((4,2),(8,5)).  Worked by hand: the complement of the 32-element tile is
    10:32, so grid coordinate (g0, g1) starts at 32*(g0 + 2*g1):
    ((4,2),(8,5)):((1,32),(4,64))."""
    T = lo.Layout((4, 8), (1, 4))
    G = lo.Layout((2, 5), (1, 2))
    P = lo.BlockedProduct(T, G)
    closed = lo.Layout(((4, 2), (8, 5)), ((1, 32), (4, 64)))
    i = np.arange(P.size)
    assert P.size == 320
    assert (P.at(i) == closed.at(i)).all()


def test_blocked_product_page_example():
    pin_blocked_product_page_example()


def test_logical_product_fills_the_gaps():
    """(2,2):(1,4) reaches {0,1,4,5}; its product with 2:1 repeats it at +2,
    giving ((2,2),2):((1,4),2), a bijection onto [0,8)."""
    P = lo.LogicalProduct(lo.Layout((2, 2), (1, 4)), lo.Layout(2, 1))
    closed = lo.Layout(((2, 2), 2), ((1, 4), 2))
    i = np.arange(8)
    assert (P.at(i) == closed.at(i)).all()
    assert sorted(P.at(i).tolist()) == list(range(8))
    # a contiguous tile repeated contiguously: (4):(1) x (3):(1) = (4,3):(1,4)
    Q = lo.LogicalProduct(lo.Layout(4, 1), lo.Layout(3, 1))
    assert (Q.at(np.arange(12)) == np.arange(12)).all()


# --------------------------------------------------------------------------
# shared-memory banks ("CUTLASS Layout可视化" §4.3, §5.2)
# --------------------------------------------------------------------------

def _column_read(rows, row_pitch, eb=4, swz=None):
    """Byte addresses of lanes 0..rows-1 reading column 0 of a row-major
    tile with `row_pitch` elements per row."""
    off = np.arange(rows, dtype=np.int64) * row_pitch
    if swz:
        off = lo.swizzle(off, *swz)
    return off * eb


def pin_bank_closed_forms():
    """Closed forms of the 32-bank model:
    * 32 lanes on consecutive fp32 words: one bank each, 1 wavefront;
    * all lanes on one word: a broadcast, 1;
    * a column of a 32-wide fp32 tile: every row in the column's bank, 32
      (the page's serialisation to 1/32);
    * a column of an 8-wide fp32 tile, 32 rows: banks c, c+8, c+16, c+24,
      eight rows each, so 8;
    * the same tile padded to 9 per row (the page's N -> N+1): 9 is odd, so
      the 32 rows land in 32 banks, 1;
    * 16-byte vectors on 32 consecutive chunks: 512 bytes, 4 passes of 128;
    * 8-byte lanes at a stride of 16 bytes: each half warp spans 256 bytes,
      so 2 passes per half, 4 in all (ideal 2);
    * Swizzle<3,0,3> on the 8-wide tile: rows r and r+4 share the bank
      group 8*(r mod 4) and differ in column bits, so 32 rows fall in 8
      banks, 4 deep; 8 rows of an 8x8 tile reach 8 banks, 1."""
    assert lo.smem_wavefronts(np.arange(32) * 4, 4) == (1, 1)
    assert lo.smem_wavefronts(np.zeros(32, np.int64), 4) == (1, 1)
    assert lo.smem_wavefronts(_column_read(32, 32), 4) == (32, 1)
    assert lo.smem_wavefronts(_column_read(32, 8), 4) == (8, 1)
    assert lo.smem_wavefronts(_column_read(32, 9), 4) == (1, 1)
    assert lo.smem_wavefronts(np.arange(32) * 16, 16) == (4, 4)
    assert lo.smem_wavefronts(np.arange(32) * 16, 8) == (4, 2)
    assert lo.smem_wavefronts(_column_read(32, 8, swz=(3, 0, 3)), 4) == (4, 1)
    assert lo.smem_wavefronts(_column_read(8, 8, swz=(3, 0, 3)), 4) == (1, 1)
    assert lo.smem_wavefronts(_column_read(8, 8), 4) == (2, 1)


def test_bank_closed_forms():
    pin_bank_closed_forms()


# --------------------------------------------------------------------------
# local_partition ("CUTLASS Layout可视化" §5.3)
# --------------------------------------------------------------------------

def pin_local_partition_closed_form():
    """8x8 row-major tile (8,8):(8,1) over a column-major 4x2 thread
    layout (4,2):(1,4).  Thread 5 sits at row 1, column 1 of the thread
    layout, so it owns rows 1, 5 and columns 1, 3, 5, 7: offsets 8*row+col
    with the row index fastest.  Thread 2 (row 2, column 0) owns rows 2, 6
    and columns 0, 2, 4, 6."""
    tile = lo.Layout((8, 8), (8, 1))
    thr = lo.Layout((4, 2), (1, 4))
    assert lo.local_partition(tile, thr, 5).tolist() == [
        9, 41, 11, 43, 13, 45, 15, 47]
    assert lo.local_partition(tile, thr, 2).tolist() == [
        16, 48, 18, 50, 20, 52, 22, 54]
    # a row-major thread layout (2,4):(4,1): thread 5 is row 1, column 1
    thr_r = lo.Layout((2, 4), (4, 1))
    assert lo.local_partition(tile, thr_r, 5).tolist() == [
        9, 25, 41, 57, 13, 29, 45, 61]


def test_local_partition_closed_form():
    pin_local_partition_closed_form()


def test_local_partition_tiles_the_layout():
    """The parts of all threads partition the tile's offsets; one thread
    owns the whole tile; a thread layout as large as the tile gives each
    thread the single element at its coordinate; the swizzle rides along."""
    cases = [
        (lo.Layout((16, 12), (12, 1)), lo.Layout((4, 3), (3, 1))),
        (lo.Layout(((2, 4), 6), ((1, 12), 2)), lo.Layout((8, 2), (1, 8))),
        (lo.Layout((32, 8), (8, 1)), lo.Layout(32, 1)),
        (lo.Layout((6, 10, 4), (40, 1, 10)), lo.Layout((3, 5), (5, 1))),
    ]
    for tile, thr in cases:
        parts = [lo.local_partition(tile, thr, t) for t in range(thr.size)]
        assert len({len(p) for p in parts}) == 1
        got = np.sort(np.concatenate(parts))
        want = np.sort(tile.at(np.arange(tile.size)))
        assert (got == want).all()
    tile = lo.Layout((8, 8), (8, 1))
    assert (lo.local_partition(tile, lo.Layout(1, 0), 0)
            == tile.at(np.arange(64))).all()
    full = lo.Layout((8, 8), (1, 8))
    for t in range(64):
        assert lo.local_partition(tile, full, t).tolist() == [
            8 * (t % 8) + t // 8]
    sw = lo.Swizzled(3, 0, 3, tile)
    thr = lo.Layout((4, 2), (1, 4))
    assert (lo.local_partition(sw, thr, 5)
            == lo.swizzle(lo.local_partition(tile, thr, 5), 3, 0, 3)).all()


# --------------------------------------------------------------------------
# the pins catch plausible mistakes planted in the oracle
# --------------------------------------------------------------------------

def _row_fastest_affine(leaves, x, extend_last):
    rem = x.copy()
    off = np.zeros_like(rem)
    for k, (e, d) in enumerate(reversed(leaves)):
        coord = rem % e
        rem = rem // e
        off = off + coord * d
    return off


def _dropped_term_affine(leaves, x, extend_last):
    rem = x.copy()
    off = np.zeros_like(rem)
    for k, (e, d) in enumerate(leaves[:-1] if len(leaves) > 1 else leaves):
        off = off + (rem % e) * d
        rem = rem // e
    return off


def _wrong_shift_swizzle(offset, b, m, s):
    o = np.asarray(offset, dtype=np.int64)
    return o ^ ((o >> (s + 1)) & (((1 << b) - 1) << m))


def _transposed_swizzle(offset, b, m, s):
    o = np.asarray(offset, dtype=np.int64)
    return o ^ ((o << s) & (((1 << b) - 1) << (m + s)))


def _complement_no_gap_leaf(layout, cotarget):
    # forgets the gap leaves: only the final leaf up to the cotarget
    span = 1
    for e, d in layout.leaves:
        span = max(span, e * d)
    return lo.Layout(-(-cotarget // span), span)


def _sixteen_banks(byte_addr, access_bytes):
    # banks taken mod 16 instead of mod 32
    addr = [int(a) for a in np.asarray(byte_addr, dtype=np.int64).ravel()]
    per = 32 if access_bytes <= 4 else 128 // access_bytes
    total = ideal = 0
    for w0 in range(0, len(addr), 32):
        warp = addr[w0:w0 + 32]
        for g0 in range(0, len(warp), per):
            banks = {}
            for a in warp[g0:g0 + per]:
                for k in range(max(1, access_bytes // 4)):
                    banks.setdefault((a // 4 + k) % 16, set()).add(a // 4 + k)
            total += max(len(v) for v in banks.values())
            ideal += max(1, -(-len(warp[g0:g0 + per]) * access_bytes // 128))
    return total, ideal


def _no_broadcast(byte_addr, access_bytes):
    # counts every lane, not every distinct word
    addr = [int(a) for a in np.asarray(byte_addr, dtype=np.int64).ravel()]
    total = ideal = 0
    for w0 in range(0, len(addr), 32):
        banks = {}
        for a in addr[w0:w0 + 32]:
            banks[(a // 4) % 32] = banks.get((a // 4) % 32, 0) + 1
        total += max(banks.values())
        ideal += 1
    return total, ideal



def _partition_blocked(layout, thr, thr_idx):
    # gives each thread a contiguous block instead of a strided share
    base = layout.inner if isinstance(layout, lo.Swizzled) else layout
    modes = base.modes()
    c = lo.thread_coordinate(thr, thr_idx) + [0] * (len(modes) - len(thr.modes()))
    t = [m.size for m in thr.modes()] + [1] * (len(modes) - len(thr.modes()))
    rest = [m.size // tk for m, tk in zip(modes, t)]
    out = []
    for r_flat in range(int(np.prod(rest))):
        off = 0
        for m, ck, nk in zip(modes, c, rest):
            off += int(m.at(ck * nk + r_flat % nk))
            r_flat //= nk
        out.append(off)
    return np.array(out, dtype=np.int64)


def _strips_times_pitch(thread_id, k_row, pitch, strips):
    t = np.asarray(thread_id, dtype=np.int64)
    div, mod = t // pitch, t % pitch
    return mod + (div % strips) * pitch + (div // strips) * (pitch * strips
                                                            * k_row)


PINS = [pin_rowmajor_grid, pin_colmajor_grid, pin_blocked_leaf_coordinates,
        pin_stripmined_page_values, pin_stripmined_is_colex_layout,
        pin_column_major_composition_is_identity,
        pin_padded_composition_closed_form, pin_zipped_divide_closed_form,
        pin_swizzle_page_formula, pin_copy_transpose,
        pin_complement_worked_examples, pin_blocked_product_page_example,
        pin_bank_closed_forms, pin_local_partition_closed_form]


@pytest.mark.parametrize("target,bad", [
    ("_affine_at", _row_fastest_affine),
    ("_affine_at", _dropped_term_affine),
    ("swizzle", _wrong_shift_swizzle),
    ("swizzle", _transposed_swizzle),
    ("stripmined_offset", _strips_times_pitch),
    ("complement", _complement_no_gap_leaf),
    ("smem_wavefronts", _sixteen_banks),
    ("smem_wavefronts", _no_broadcast),
    ("local_partition", _partition_blocked),
])
def test_pins_catch_planted_mistakes(monkeypatch, target, bad):
    monkeypatch.setattr(lo, target, bad)
    failures = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake in {target}"
