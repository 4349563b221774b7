"""Host side of the C ABI against the oracle (no GPU needed).

The library's layout algebra and its copy planner run on the host; these
tests compare them with the oracle on exhaustive tiny cases and seeded random
ones.  The planner is checked by expanding every piece of a plan into its
(src offset, dst offset) pairs and comparing the union with the oracle's
pairs {(src(i), dst(i))}: the pieces must partition the copy exactly.
"""

import itertools
import re

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import WORKLOADS

lm = pytest.importorskip("layout_driven_movement_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def fmt(x):
    return str(x) if isinstance(x, int) else "(" + ",".join(fmt(k) for k in x) + ")"


def random_layout(rng, max_modes=3, max_ext=5, max_stride=12, nest=True):
    n = int(rng.integers(1, max_modes + 1))
    shape, stride = [], []
    for _ in range(n):
        if nest and rng.random() < 0.3:
            k = int(rng.integers(2, 4))
            shape.append(tuple(int(v) for v in rng.integers(1, max_ext + 1, k)))
            stride.append(tuple(int(v) for v in rng.integers(0, max_stride + 1, k)))
        else:
            shape.append(int(rng.integers(1, max_ext + 1)))
            stride.append(int(rng.integers(0, max_stride + 1)))
    return tuple(shape), tuple(stride)


# --------------------------------------------------------------------------
# the ABI surface
# --------------------------------------------------------------------------

def test_library_exports_every_declared_symbol():
    import ctypes
    import os
    header = open(os.path.join(os.path.dirname(__file__), "..", "include",
                               "layoutmove.h")).read()
    names = set(re.findall(
        r"^(?:int|void|const char\*)\s+(lm_[a-z_]+)\s*\(", header, re.M))
    assert len(names) >= 25
    so = ctypes.CDLL(lm.LIB_PATH)
    for name in sorted(names):
        assert hasattr(so, name), name
    declared = {n for n, _, _ in lm.SIGNATURES}
    assert names == declared


def test_status_strings_and_version():
    L = lm.lib()
    assert L.lm_status_string(0) == b"LM_OK"
    assert L.lm_status_string(-4) == b"LM_E_NOT_INJECTIVE"
    assert L.lm_status_string(12345) == b"LM_E_UNKNOWN"
    assert re.match(rb"\d+\.\d+\.\d+", L.lm_version())


# --------------------------------------------------------------------------
# construction, printing, evaluation
# --------------------------------------------------------------------------

@pytest.mark.parametrize("text", [
    "(4,2):(2,1)", "((4,2),(2,4)):((2,16),(1,8))", "8:1", "(8):(3)",
    "Sw<3,4,3> o ((64,64),(128,128)):((64,1),(524288,4096))",
    "(((4,8),2),1048576):(((1,4),32),64)", "(0,3):(1,0)",
])
def test_parse_print_round_trip(text):
    assert str(lm.Layout.parse(text)) == text


def test_parse_static_marks_and_cute_swizzle_print():
    assert str(lm.Layout.parse("(4,2):(_2,_1)")) == "(4,2):(2,1)"
    L = lm.Layout.parse("Sw<3,0,3> o _0 o (8,8):(8,1)")
    assert str(L) == "Sw<3,0,3> o (8,8):(8,1)"


@pytest.mark.parametrize("bad", ["", "(4,2)", "(4,2):(1)", "(4,2):(1,2,3)",
                                 "((4,2):(1,2)", "(4,-2):(1,1)", "a:b",
                                 "Sw<3,0,2> o 8:1", "(4,2):(2,1) junk"])
def test_parse_rejects(bad):
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Layout.parse(bad)
    assert e.value.status == -1


def test_make_matches_parse():
    a = lm.Layout.make([4, 2, 2, 4], [2, 16, 1, 8], [2, 2])
    assert str(a) == "((4,2),(2,4)):((2,16),(1,8))"
    assert str(lm.Layout.make([8], [1])) == "8:1"
    with pytest.raises(lm.LayoutMoveError):
        lm.Layout.make([4, 2], [1, 4], [3])


def test_eval_matches_oracle_random():
    rng = np.random.default_rng(101)
    for _ in range(300):
        shape, stride = random_layout(rng)
        L = lm.Layout.of(shape, stride)
        O = lo.Layout(shape, stride)
        assert L.size == O.size
        i = np.arange(O.size)
        want = O.at(i)
        got = [L(int(k)) for k in i]
        assert got == want.tolist()
        if O.size:
            assert L.cosize == lo.cosize(O)
        # leaf-coordinate form
        coord = [int(rng.integers(0, 7)) for _ in O.leaves]
        assert L.eval_coord(coord) == lo.eval_leaf_coord(O, coord)


def test_eval_swizzled_matches_oracle():
    rng = np.random.default_rng(102)
    for _ in range(200):
        shape, stride = random_layout(rng, max_ext=6, max_stride=40)
        b = int(rng.integers(1, 4))
        m = int(rng.integers(0, 4))
        s = int(rng.integers(b, b + 4))
        L = lm.Layout.of(shape, stride).swizzle(b, m, s)
        O = lo.Swizzled(b, m, s, lo.Layout(shape, stride))
        i = np.arange(O.size)
        assert [L(int(k)) for k in i] == O.at(i).tolist()
        if O.size:
            assert L.cosize >= lo.cosize(O)
            assert L.cosize % (1 << (m + b)) == 0


def test_eval_rejects_out_of_range():
    L = lm.Layout.parse("(4,2):(2,1)")
    for bad in (-1, 8):
        with pytest.raises(lm.LayoutMoveError):
            L(bad)


def test_page_layouts_through_library():
    blocked = lm.Layout.parse("((4,2),(2,4)):((2,16),(1,8))")
    assert blocked.eval_coord([0, 1, 0, 0]) == 16
    assert blocked.eval_coord([1, 0, 0, 0]) == 2
    assert blocked.eval_coord([3, 3, 0, 0]) == 54
    assert blocked.cosize == 48
    sw = lm.Layout.parse("(8,8):(8,1)").swizzle(3, 0, 3)
    for r in range(8):
        for c in range(8):
            assert sw(r + 8 * c) == r * 8 + (c ^ r)


# --------------------------------------------------------------------------
# algebra
# --------------------------------------------------------------------------

def test_compose_page_example_closed_form():
    P = lm.Layout.parse("(8,8):(1,9)")
    TV = lm.Layout.parse("((4,8),2):((16,1),8)")
    assert str(P.compose(TV)) == "((4,8),2):((18,1),9)"
    col = lm.Layout.parse("(8,8):(1,8)")
    assert str(col.compose(TV)) == "((4,8),2):((16,1),8)"


def test_compose_matches_oracle_random():
    rng = np.random.default_rng(103)
    ok = 0
    for trial in range(600):
        if trial % 2:
            # compact outer layouts in random mode order: composable often
            ext = [int(v) for v in rng.integers(1, 5, int(rng.integers(1, 4)))]
            order = rng.permutation(len(ext))
            stride = [0] * len(ext)
            acc = 1
            for k in order:
                stride[k] = acc
                acc *= ext[k]
            a_shape, a_stride = tuple(ext), tuple(stride)
        else:
            a_shape, a_stride = random_layout(rng, max_stride=6, nest=False)
        b_shape, b_stride = random_layout(rng, max_ext=4, max_stride=6)
        A = lm.Layout.of(a_shape, a_stride)
        B = lm.Layout.of(b_shape, b_stride)
        OA, OB = lo.Layout(a_shape, a_stride), lo.Layout(b_shape, b_stride)
        if OA.size == 0:
            continue
        try:
            R = A.compose(B)
        except lm.LayoutMoveError as e:
            assert e.status == -3
            continue
        ok += 1
        want = lo.Composed(OA, OB).at(np.arange(OB.size))
        assert R.size == OB.size
        assert [R(int(k)) for k in range(OB.size)] == want.tolist(), \
            (a_shape, a_stride, b_shape, b_stride, str(R))
    assert ok > 250


def test_compose_swizzled_outer_and_rejects_swizzled_inner():
    A = lm.Layout.parse("(8,8):(8,1)").swizzle(3, 0, 3)
    B = lm.Layout.parse("(8,8):(1,8)")
    R = A.compose(B)
    OA = lo.Swizzled(3, 0, 3, lo.Layout((8, 8), (8, 1)))
    want = lo.Composed(OA, lo.Layout((8, 8), (1, 8))).at(np.arange(64))
    assert [R(k) for k in range(64)] == want.tolist()
    with pytest.raises(lm.LayoutMoveError) as e:
        B.compose(A)
    assert e.value.status == -3


def test_zipped_divide_page_example_and_c3():
    Z = lm.Layout.parse("(128,128):(1,128)").zipped_divide([4, 8])
    assert str(Z) == "((4,8),(32,16)):((1,128),(4,1024))"
    Z3 = lm.build_layout(WORKLOADS["C3"].src)
    assert str(Z3) == "((64,64),(128,128)):((8192,1),(524288,64))"


def test_zipped_divide_matches_oracle_random():
    rng = np.random.default_rng(104)
    ok = 0
    for _ in range(400):
        shape, stride = random_layout(rng, max_modes=3, max_ext=6)
        O = lo.Layout(shape, stride)
        modes = O.modes()
        tiler = []
        for m in modes:
            divs = [t for t in range(1, m.size + 1) if m.size % t == 0] or [1]
            tiler.append(int(rng.choice(divs)) if m.size else 1)
        if O.size == 0:
            continue
        L = lm.Layout.of(shape, stride)
        try:
            Z = L.zipped_divide(tiler)
        except lm.LayoutMoveError as e:
            assert e.status == -3
            continue
        ok += 1
        want = lo.ZippedDivide(O, tiler).at(np.arange(O.size))
        assert [Z(int(k)) for k in range(O.size)] == want.tolist(), \
            (shape, stride, tiler, str(Z))
    assert ok > 200


def test_zipped_divide_rejects_non_dividing_tiler():
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Layout.parse("(6,4):(1,6)").zipped_divide([4, 4])
    assert e.value.status == -3
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Layout.parse("(6,4):(1,6)").zipped_divide([2])
    assert e.value.status == -1


def test_coalesce_keeps_function():
    rng = np.random.default_rng(105)
    for _ in range(200):
        shape, stride = random_layout(rng)
        L = lm.Layout.of(shape, stride)
        C = L.coalesce()
        O = lo.Layout(shape, stride)
        assert [C(k) for k in range(O.size)] == O.at(np.arange(O.size)).tolist()
    assert str(lm.Layout.parse("(4,2,3):(1,4,8)").coalesce()) == "24:1"


def test_right_inverse_round_trip_and_oracle():
    rng = np.random.default_rng(106)
    for _ in range(150):
        ext = [int(v) for v in rng.integers(1, 6, int(rng.integers(1, 4)))]
        order = rng.permutation(len(ext))
        stride = [0] * len(ext)
        acc = 1
        for k in order:
            stride[k] = acc
            acc *= ext[k]
        L = lm.Layout.of(tuple(ext), tuple(stride))
        R = L.right_inverse()
        O = lo.Layout(tuple(ext), tuple(stride))
        assert R.size == O.size
        want = lo.right_inverse_values(O)
        assert [R(j) for j in range(R.size)] == want.tolist()
    assert str(lm.Layout.parse("(4,2):(2,1)").right_inverse()) == "(2,4):(4,1)"


def test_max_common_vector_matches_oracle():
    rng = np.random.default_rng(107)
    for _ in range(300):
        ext = [int(v) for v in rng.integers(1, 5, int(rng.integers(1, 4)))]
        def compact(perm, gap=0):
            stride = [0] * len(ext)
            acc = 1
            for k in perm:
                stride[k] = acc
                acc *= ext[k] + (gap if k == perm[-1] else 0)
            return tuple(stride)
        sa = compact(rng.permutation(len(ext)))
        sb = compact(rng.permutation(len(ext)), int(rng.integers(0, 2)))
        A = lm.Layout.of(tuple(ext), sa)
        B = lm.Layout.of(tuple(ext), sb)
        if rng.random() < 0.3:
            b = int(rng.integers(1, 3))
            m = int(rng.integers(0, 3))
            s = int(rng.integers(b, b + 3))
            B = B.swizzle(b, m, s)
            OB = lo.Swizzled(b, m, s, lo.Layout(tuple(ext), sb))
        else:
            OB = lo.Layout(tuple(ext), sb)
        OA = lo.Layout(tuple(ext), sa)
        assert A.max_common_vector(B) == lo.max_common_vector(OA, OB)
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Layout.parse("4:1").max_common_vector(lm.Layout.parse("5:1"))
    assert e.value.status == -2


def test_max_common_vector_large_uses_structure():
    # 2^22 elements: beyond the brute-force limit, answered from joint modes
    a = lm.Layout.parse("(64,65536):(1,64)")
    b = lm.Layout.parse("(64,65536):(1,128)")
    assert a.max_common_vector(b) == 64
    c = lm.build_layout(WORKLOADS["C3"].src)
    d = lm.build_layout(WORKLOADS["C3"].dst)
    assert c.max_common_vector(d) == 64


def test_complement_and_products_match_oracle():
    assert str(lm.Layout.parse("(2,2):(1,6)").complement(24)) == "(3,2):(2,12)"
    assert str(lm.Layout.parse("4:1").complement(24)) == "6:4"
    tile = lm.Layout.parse("(4,8):(1,4)")
    grid = lm.Layout.parse("(2,5):(1,2)")
    bp = tile.blocked_product(grid)
    assert str(bp) == "((4,2),(8,5)):((1,32),(4,64))"
    rng = np.random.default_rng(109)
    ok = 0
    for _ in range(200):
        n = int(rng.integers(1, 3))
        ext = [int(v) for v in rng.integers(1, 4, n)]
        stride, span = [], 1
        for e in ext:
            span *= int(rng.integers(1, 3))
            stride.append(span)
            span *= e
        A_spec = (tuple(ext), tuple(stride))
        B_spec = (tuple(int(v) for v in rng.integers(1, 4, n)),
                  tuple(int(v) for v in rng.integers(0, 3, n)))
        A, B = lm.Layout.of(*A_spec), lm.Layout.of(*B_spec)
        OA, OB = lo.Layout(*A_spec), lo.Layout(*B_spec)
        M = span * int(rng.integers(1, 3))
        C = A.complement(M)
        OC = lo.complement(OA, M)
        assert [C(k) for k in range(C.size)] == lo.image(OC).tolist()
        for fn, ofn in (("logical_product", lo.LogicalProduct),
                        ("blocked_product", lo.BlockedProduct)):
            try:
                R = getattr(A, fn)(B)
            except lm.LayoutMoveError as e:
                assert e.status == -3
                continue
            ok += 1
            O = ofn(OA, OB)
            assert R.size == O.size
            assert [R(k) for k in range(R.size)] == \
                O.at(np.arange(O.size)).tolist(), (A_spec, B_spec, fn, str(R))
    assert ok > 100
    with pytest.raises(lm.LayoutMoveError):
        lm.Layout.parse("(2,3):(1,3)").complement(12)


def test_stripmined_layout_matches_oracle():
    for threads, pitch, strips, k_row in itertools.product(
            (32, 64, 100), (1, 4, 8), (1, 2, 4), (16, 33)):
        L = lm.Layout.stripmined(threads, pitch, strips, k_row)
        t = np.arange(threads)
        want = lo.stripmined_offset(t, k_row, pitch, strips)
        assert [L(int(k)) for k in t] == want.tolist()


# --------------------------------------------------------------------------
# the planner
# --------------------------------------------------------------------------

def plan_pairs(plan: "lm.Plan", s_swz, d_swz):
    """Expand a joint plan's pieces into its (src, dst) offset pairs."""
    desc = plan.describe()
    assert desc["joint"]
    src, dst = [], []
    for pc in desc["pieces"]:
        ms = pc["modes"]
        n = int(np.prod([m[0] for m in ms])) if ms else 1
        i = np.arange(n)
        so = np.full(n, pc["s_base"], dtype=np.int64)
        do = np.full(n, pc["d_base"], dtype=np.int64)
        for e, s, d in ms:
            c = i % e
            i = i // e
            so += c * s
            do += c * d
        src.append(so)
        dst.append(do)
    so = np.concatenate(src) if src else np.zeros(0, np.int64)
    do = np.concatenate(dst) if dst else np.zeros(0, np.int64)
    if s_swz:
        so = lo.swizzle(so, *s_swz)
    if d_swz:
        do = lo.swizzle(do, *d_swz)
    return so, do


def check_plan_partition(src_spec, dst_spec, eb):
    S, D = lm.build_layout(src_spec), lm.build_layout(dst_spec)
    OS, OD = lo.build(src_spec), lo.build(dst_spec)
    plan = lm.Plan(S, D, eb)
    desc = plan.describe()
    if not desc["joint"]:
        return desc
    s_swz = (OS.b, OS.m, OS.s) if isinstance(OS, lo.Swizzled) else None
    d_swz = (OD.b, OD.m, OD.s) if isinstance(OD, lo.Swizzled) else None
    so, do = plan_pairs(plan, s_swz, d_swz)
    i = np.arange(OS.size)
    want = np.stack([OS.at(i), OD.at(i)], 1)
    got = np.stack([so, do], 1)
    assert got.shape == want.shape
    order_w = np.lexsort((want[:, 0], want[:, 1]))
    order_g = np.lexsort((got[:, 0], got[:, 1]))
    assert (want[order_w] == got[order_g]).all()
    n, sc, dc = plan.extent()
    assert n == OS.size and sc >= lo.cosize(OS) and dc >= lo.cosize(OD)
    assert plan.launches == len(desc["pieces"])
    return desc


def test_plan_paths_for_workloads():
    paths = {}
    for name, w in WORKLOADS.items():
        S, D = lm.build_layout(w.src), lm.build_layout(w.dst)
        paths[name] = [p["path"] for p in lm.Plan(S, D, w.elem_bytes).describe()["pieces"]]
    assert paths == {"C1": ["GENERIC"], "C2": ["STAGED"], "C3": ["VEC"],
                     "C4": ["STAGED"], "C5a": ["STAGED"], "C5b": ["ZIP"]}


def test_plan_partition_small_workload_shapes():
    cases = [
        (WORKLOADS["C1"].src, WORKLOADS["C1"].dst, 4),
        (("layout", (200, 136), (1, 200)), ("layout", (200, 136), (136, 1)), 4),
        (("zipped_divide", ("layout", (256, 192), (192, 1)), (64, 64)),
         ("swizzle", 3, 4, 3, ("layout", ((64, 64), (4, 3)), ((64, 1), (12288, 4096)))), 2),
        (("concat", WORKLOADS["C4"].src[1], ("layout", 100, 72)),
         ("layout", (((4, 8), 2), 100), (((1, 4), 32), 64)), 8),
        (("layout", (3, 40, 7, 9), (2520, 1, 360, 40)),
         ("layout", (3, 40, 7, 9), (2520, 63, 9, 1)), 2),
        (("layout", (2, 1000, 24), (24000, 24, 1)),
         ("layout", (2, 1000, 24), (1, 48, 2)), 2),
        (("layout", (97, 131), (1, 97)), ("layout", (97, 131), (131, 1)), 1),
        (("layout", (50, 60), (1, 50)), ("layout", (50, 60), (60, 1)), 16),
        (("layout", (4096,), (1,)), ("layout", (4096,), (1,)), 4),
        (("layout", (5000,), (1,)), ("layout", (5000,), (1,)), 2),
    ]
    for s, d, eb in cases:
        check_plan_partition(s, d, eb)


def test_plan_partition_random_bijections():
    rng = np.random.default_rng(108)
    for _ in range(120):
        nm = int(rng.integers(1, 5))
        ext = [int(v) for v in rng.integers(1, 40, nm)]
        def compact(perm, pad):
            stride = [0] * nm
            acc = 1
            for k in perm:
                stride[k] = acc
                acc *= ext[k] + (pad if k == perm[0] else 0)
            return tuple(stride)
        s = ("layout", tuple(ext), compact(rng.permutation(nm), int(rng.integers(0, 3))))
        d = ("layout", tuple(ext), compact(rng.permutation(nm), 0))
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        check_plan_partition(s, d, eb)


def test_plan_errors():
    a = lm.Layout.parse("(8,8):(1,8)")
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Plan(a, lm.Layout.parse("(8,4):(1,8)"), 4)
    assert e.value.status == -2
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Plan(a, lm.Layout.parse("((4,2),(2,4)):((2,16),(1,8))"), 4)
    assert e.value.status == -4
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Plan(a, a, 3)
    assert e.value.status == -1
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Plan(a, lm.Layout.parse("(8,8):(0,1)"), 4)
    assert e.value.status == -4


def test_plan_non_refinable_pair_is_generic_and_empty_plan():
    s = lm.Layout.parse("(2,3):(1,3)")
    d = lm.Layout.parse("(3,2):(2,1)")
    desc = lm.Plan(s, d, 4).describe()
    assert not desc["joint"] and desc["pieces"][0]["path"] == "GENERIC"
    # (2,3):(1,2) is the single run 6:1, which refines against (3,2)
    desc = lm.Plan(lm.Layout.parse("(2,3):(1,2)"), d, 4).describe()
    assert desc["joint"] and desc["pieces"][0]["modes"] == [[3, 1, 2],
                                                            [2, 3, 1]]
    e = lm.Plan(lm.Layout.parse("(0,4):(1,0)"), lm.Layout.parse("(0,4):(4,1)"), 4)
    assert e.describe()["pieces"] == [] and e.launches == 0


def test_copy_validation_without_gpu():
    """Host-side checks of lm_layout_copy fire before any CUDA call."""
    import ctypes as C
    L = lm.lib()
    p = lm.Plan(lm.Layout.parse("(64,64):(1,64)"), lm.Layout.parse("(64,64):(64,1)"), 4)
    assert L.lm_layout_copy(p.handle, C.c_void_p(4096), 4095, C.c_void_p(1 << 30), 4096, None) == -6
    assert L.lm_layout_copy(p.handle, C.c_void_p(4096), 4096, C.c_void_p(4096 + 100), 4096, None) == -7
    assert L.lm_layout_copy(p.handle, None, 4096, C.c_void_p(1 << 30), 4096, None) == -1
    assert L.lm_layout_eval_device(lm.Layout.parse("8:1").handle, C.c_void_p(4096), 3, 8, None) == -1
    assert L.lm_layout_eval_device(lm.Layout.parse("8:1").handle, C.c_void_p(4096), 4, 7, None) == -6
    big = lm.Layout.parse("(2,2):(1,4294967296)")
    assert L.lm_layout_eval_device(big.handle, C.c_void_p(4096), 4, 8, None) == -5


def test_local_partition_matches_oracle():
    """Thread parts from lm_layout_local_partition equal the oracle's, for
    nested tiles, thread layouts of lower rank, and a swizzled tile."""
    cases = [("(8,8):(8,1)", "(4,2):(1,4)"),
             ("(8,8):(8,1)", "(2,4):(4,1)"),
             ("(16,12):(12,1)", "(4,3):(3,1)"),
             ("((2,4),6):((1,12),2)", "(8,2):(1,8)"),
             ("(32,8):(8,1)", "32:1"),
             ("(6,10,4):(40,1,10)", "(3,5):(5,1)"),
             ("(64,64):(1,64)", "((8,4),(2,4)):((1,64),(8,16))")]
    for tile_t, thr_t in cases:
        tile, thr = lm.Layout.parse(tile_t), lm.Layout.parse(thr_t)
        ot, othr = lo.parse(tile_t), lo.parse(thr_t)
        for t in range(thr.size):
            part, base = tile.local_partition(thr, t)
            got = [base + part(v) for v in range(part.size)]
            assert got == lo.local_partition(ot, othr, t).tolist(), (tile_t, t)
    sw = lm.Layout.parse("(32,8):(8,1)").swizzle(3, 0, 3)
    thr = lm.Layout.parse("(8,4):(4,1)")
    osw = lo.Swizzled(3, 0, 3, lo.parse("(32,8):(8,1)"))
    for t in range(32):
        part, base = sw.local_partition(thr, t)
        got = lo.swizzle(np.array([base + part(v) for v in range(part.size)]),
                         3, 0, 3)
        assert got.tolist() == lo.local_partition(osw, lo.parse("(8,4):(4,1)"),
                                                  t).tolist()


def test_local_partition_rejects():
    tile = lm.Layout.parse("(8,8):(8,1)")
    bad = [("(4,2):(1,2)", 0, -1),        # not a bijection onto [0, 8)
           ("(4,2):(1,4)", 8, -1),        # thread out of range
           ("(4,2,2):(1,4,8)", 0, -1),    # rank above the tile's
           ("(3,2):(1,3)", 0, -3)]        # 3 does not divide 8
    for thr_t, t, code in bad:
        with pytest.raises(lm.LayoutMoveError) as e:
            tile.local_partition(lm.Layout.parse(thr_t), t)
        assert e.value.status == code, thr_t


def test_plans_beyond_2_to_31_elements_split_aligned():
    """A 70000x70000 byte transpose (4.9e9 elements): the plan splits into
    pieces under 2^31 elements each, at multiples of 64 coordinates, so
    every piece keeps the shared-memory path; together they cover the copy."""
    S = lm.Layout.parse("(70000,70000):(1,70000)")
    D = lm.Layout.parse("(70000,70000):(70000,1)")
    d = lm.Plan(S, D, 1).describe()
    total = 0
    for p in d["pieces"]:
        n = int(np.prod([m[0] for m in p["modes"]]))
        assert n < 2 ** 31
        assert p["path"] == "STAGED", p
        assert p["s_base"] % 16 == 0 and p["d_base"] % 16 == 0
        total += n
    assert total == 70000 * 70000


def _grid_ints(text):
    return [[int(v) for v in line.split()] for line in text.splitlines()]


def test_print_grid_matches_oracle_and_page_grids():
    """lm_layout_print_grid gives the oracle's print_layout grid (row =
    mode-0 coordinate) for the page's 4x2 grids, the swizzled 8x8 tile,
    nested and random rank-2 layouts; its bank view is every offset times
    the element size over 4, mod 32."""
    texts = ["(4,2):(2,1)", "(4,2):(1,4)", "((4,2),(2,4)):((2,16),(1,8))",
             "(8,8):(8,1)", "(16,12):(1,16)"]
    rng = np.random.default_rng(11)
    for _ in range(20):
        e0, e1 = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        d0, d1 = int(rng.integers(0, 40)), int(rng.integers(0, 40))
        texts.append(f"({e0},{e1}):({d0},{d1})")
    for t in texts:
        L, O = lm.Layout.parse(t), lo.parse(t)
        want = lo.print_grid(O)
        assert _grid_ints(L.print_grid()) == want, t
        for eb in (2, 4, 8):
            banks = [[(v * eb // 4) % 32 for v in row] for row in want]
            assert _grid_ints(L.print_grid(eb)) == banks, (t, eb)
    sw = lm.Layout.parse("(8,8):(8,1)").swizzle(3, 0, 3)
    osw = lo.Swizzled(3, 0, 3, lo.parse("(8,8):(8,1)"))
    assert _grid_ints(sw.print_grid()) == lo.print_grid(osw)
    assert _grid_ints(sw.print_grid())[1] == [9, 8, 11, 10, 13, 12, 15, 14]
    lines = lm.Layout.parse("(4,2):(2,1)").print_grid().splitlines()
    assert lines == ["0 1", "2 3", "4 5", "6 7"]
    for bad in ["8:1", "(2,2,2):(1,2,4)"]:
        with pytest.raises(lm.LayoutMoveError):
            lm.Layout.parse(bad).print_grid()


def test_product_built_copy_layouts_match_oracle():
    """The product-built layouts of the GPU product cases: the library's
    closed forms, and their offsets at seeded sample indices equal to the
    oracle's products."""
    from product_cases import PRODUCT_CASES
    rng = np.random.default_rng(31)
    for name, s, d, eb, built, _ in PRODUCT_CASES:
        spec = s if s[0].endswith("product") else d
        L, OL = lm.build_layout(spec), lo.build(spec)
        assert str(L) == built, name
        assert L.size == OL.size and L.cosize == lo.cosize(OL), name
        idx = np.concatenate([[0, L.size - 1], rng.integers(0, L.size, 2000)])
        assert [L(int(i)) for i in idx] == OL.at(idx).tolist(), name


def test_refinement_of_coalesced_sides():
    """Pairs whose raw leaves do not nest but whose coalesced leaves do are
    planned on the joint paths: the 6000x7000 fp32 matrix against the
    destination (7000,6000):(1,7000) (one run of 42,000,000) is a
    transpose; with a padded destination there is no refinement."""
    S = lm.Layout.parse("(6000,7000):(7000,1)")
    d = lm.Plan(S, lm.Layout.parse("(7000,6000):(1,7000)"), 4).describe()
    assert d["joint"] and [p["path"] for p in d["pieces"]] == ["STAGED"]
    assert d["pieces"][0]["modes"] == [[6000, 7000, 1], [7000, 1, 6000]]
    d = lm.Plan(S, lm.Layout.parse("(7000,6000):(1,7001)"), 4).describe()
    assert not d["joint"] and d["pieces"][0]["path"] == "GTILE"
    assert (d["pieces"][0]["outer"], d["pieces"][0]["u_extent"],
            d["pieces"][0]["v_extent"]) == ("src", 6000, 7000)
    # every accepted joint plan still maps each logical index like the two
    # layouts do (sampled against the oracle)
    rng = np.random.default_rng(77)
    for s_txt, d_txt in [("(6,5):(5,1)", "(5,6):(1,5)"),
                         ("(4,9,2):(18,2,1)", "(12,6):(1,12)"),
                         ("(10,21):(1,10)", "(6,35):(35,1)")]:
        plan = lm.Plan(lm.Layout.parse(s_txt), lm.Layout.parse(d_txt), 2)
        desc = plan.describe()
        assert desc["joint"], (s_txt, d_txt)
        OS, OD = lo.parse(s_txt), lo.parse(d_txt)
        i = np.arange(OS.size)
        ms = desc["pieces"][0]["modes"]
        so = np.zeros_like(i)
        do = np.zeros_like(i)
        rem = i.copy()
        for e, st, dt in ms:
            so += (rem % e) * st
            do += (rem % e) * dt
            rem //= e
        assert (so == OS.at(i)).all() and (do == OD.at(i)).all()


def _gtile_walk(leaves, step, x0, count):
    """The tiled kernels' walk over one part of a GTILE piece: the digits
    of x0 in the part's mixed radix and their byte offset, then `count`
    steps each adding the step's digits with carries and changing the
    offset by its precomputed amounts (the last leaf runs on, no carry out
    of it).  Returns the offsets visited, x0's included."""
    ext = [e for e, _ in leaves]
    st = [b for _, b in leaves]
    n = len(ext)
    c, q = [], x0
    for e in ext:
        c.append(q % e)
        q //= e
    off = sum(ck * sk for ck, sk in zip(c, st))
    out = [off]
    for _ in range(count):
        carry, delta = 0, step["dstep"]
        for k in range(n - 1):
            x = c[k] + step["digits"][k] + carry
            carry = 1 if x >= ext[k] else 0
            if carry:
                x -= ext[k]
                delta += step["cadj"][k]
            c[k] = x
        off += delta
        out.append(off)
    return out


def test_gtile_steps_reproduce_offsets():
    """The steps the tiled kernels take between a thread's elements, as the
    planner hands them over (each step's digits, its offset change without
    carries and the change of each carry): walking them from random starts
    visits exactly the byte offsets the oracle gives the logical indices
    they land on, for the inner side over the whole index and the outer
    side's lo leaves over u."""
    rng = np.random.default_rng(5)
    for s_txt, d_txt, eb in [("(6000,7000):(7000,1)", "(7000,6000):(1,7001)", 4),
                             ("(300,350):(350,1)", "(350,300):(1,351)", 4),
                             ("(350,300):(1,351)", "(300,350):(350,1)", 2),
                             ("(40,40,33):(40,1,1600)", "(33,1600):(1,35)", 8),
                             ("(3,14,37):(518,37,1)", "(37,42):(1,39)", 4),
                             ("(37,42):(1,39)", "(3,14,37):(518,37,1)", 2)]:
        pc = lm.Plan(lm.Layout.parse(s_txt), lm.Layout.parse(d_txt),
                     eb).describe()["pieces"][0]
        assert pc["path"] == "GTILE", (s_txt, pc)
        outer_src = pc["outer"] == "src"
        O = lo.parse(s_txt if outer_src else d_txt)
        I = lo.parse(d_txt if outer_src else s_txt)
        W, n = pc["u_extent"], I.size
        oleaves = lo.flatten(O.shape, O.stride)
        k = next(j for j, (e, st) in enumerate(oleaves) if st == 1)
        LO = lo.Layout(tuple(e for e, _ in oleaves[:k]),
                       tuple(st for _, st in oleaves[:k]))
        parts = [("in", pc["in_leaves"], n, I),
                 ("lo", pc["lo_leaves"], W, LO)]
        names = {"in": ["in", "in_next_v", "in_next_chunk"], "lo": ["lo"]}
        for part, leaves, size, L in parts:
            radix = np.cumprod([1] + [e for e, _ in leaves[:-1]])
            for name in names[part]:
                if name not in pc["steps"]:
                    continue
                step = pc["steps"][name]
                amount = int(sum(d * r for d, r in zip(step["digits"], radix)))
                assert 0 < amount < size, (s_txt, name, amount)
                count = min(12, (size - 1) // amount)
                for x0 in rng.integers(0, size - count * amount, 20):
                    got = _gtile_walk(leaves, step, int(x0), count)
                    xs = int(x0) + amount * np.arange(count + 1)
                    want = (L.at(xs) * eb).tolist()
                    assert got == want, (s_txt, name, int(x0))


def test_gtile_split_is_exact():
    """The tiled path for pairs without a common refinement reads the outer
    side as lo(u) + hi(v) with i = u + W*v: for every logical index of a
    few pairs, that split (its leaves before the unit-stride leaf over u,
    the rest over v) equals the oracle's offset, and the inner side's first
    leaf has unit stride."""
    for s_txt, d_txt, outer in [("(300,350):(350,1)", "(350,300):(1,351)", "src"),
                                ("(350,300):(1,351)", "(300,350):(350,1)", "dst"),
                                ("(40,40,33):(40,1,1600)", "(33,1600):(1,35)", "src")]:
        d = lm.Plan(lm.Layout.parse(s_txt), lm.Layout.parse(d_txt), 4).describe()
        pc = d["pieces"][0]
        assert pc["path"] == "GTILE" and pc["outer"] == outer, (s_txt, pc)
        W = pc["u_extent"]
        O = lo.parse(s_txt if outer == "src" else d_txt)
        leaves = lo.flatten(O.shape, O.stride)
        k = next(j for j, (e, st) in enumerate(leaves) if st == 1)
        assert int(np.prod([e for e, _ in leaves[:k]])) == W
        i = np.arange(O.size)
        u, v = i % W, i // W
        lo_off = lo.Layout(tuple(e for e, _ in leaves[:k]),
                           tuple(st for _, st in leaves[:k])).at(u)
        hi_off = lo.Layout(tuple(e for e, _ in leaves[k:]),
                           tuple(st for _, st in leaves[k:])).at(v)
        assert (lo_off + hi_off == O.at(i)).all()
        I = lo.parse(d_txt if outer == "src" else s_txt)
        assert lo.flatten(I.shape, I.stride)[0][1] == 1
