"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every comparison is byte-exact (tolerance 0: the copy moves raw bits).  The
destination is pre-filled with 0xA5 and framed by guard bands, so slots the
destination layout does not cover, and bytes outside the buffer, must come
back untouched.  Small cases span several tiles and ragged tails; the
full-size workloads run with the same plans (and so the same launch
configuration) that bench.py times and are compared with the oracle in
full.
"""

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import EVAL_C1, WORKLOADS, seeded_bytes
from product_cases import PRODUCT_CASES

torch = pytest.importorskip("torch")
lm = pytest.importorskip("layout_driven_movement_gb300")

pytestmark = pytest.mark.gpu

GUARD = 256
FILL = 0xA5
GUARD_FILL = 0x5C


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def device_buffer(nbytes, fill, offset=0):
    """A CUDA uint8 view of nbytes at byte `offset` past a 256-byte guard."""
    raw = torch.full((nbytes + 2 * GUARD + offset,), GUARD_FILL,
                     dtype=torch.uint8, device="cuda")
    view = raw[GUARD + offset:GUARD + offset + nbytes]
    view.fill_(fill)
    return raw, view


def run_case(src_spec, dst_spec, eb, values="bytes", dtype="uint8", seed=7,
             src_offset=0, dst_offset=0, stream=None, sentinel=None,
             expect_paths=None, src_round16=False):
    S, D = lm.build_layout(src_spec), lm.build_layout(dst_spec)
    OS, OD = lo.build(src_spec), lo.build(dst_spec)
    plan = lm.Plan(S, D, eb)
    if expect_paths is not None:
        assert [p["path"] for p in plan.describe()["pieces"]] == expect_paths
    n_src, n_dst = lo.cosize(OS), lo.cosize(OD)
    assert S.cosize >= n_src and D.cosize >= n_dst
    n_src_cap, n_dst_cap = S.cosize, D.cosize
    if src_round16:   # the source buffer rounded up to a 16-byte multiple
        n_src_cap = -(-(n_src_cap * eb) // 16) * 16 // eb
    if values == "bytes":
        inp = seeded_bytes("bytes", "uint8", n_src_cap * eb, seed)
    else:
        inp = seeded_bytes(values, dtype, n_src_cap, seed)
    if sentinel is not None:
        # slots of the source that no logical index reads
        touched = np.zeros(n_src_cap, dtype=bool)
        touched[lo.image(OS)] = True
        v = inp.view(np.dtype((np.void, eb)))
        pad = np.frombuffer(np.array([sentinel], dtype=np.uint64).tobytes(),
                            dtype=np.dtype((np.void, eb)))
        v[~touched] = pad[0]
    want = np.full(n_dst_cap * eb, FILL, dtype=np.uint8)
    lo.copy(OS, OD, inp, want, eb)

    s_raw, s_view = device_buffer(n_src_cap * eb, 0, src_offset)
    s_view.copy_(torch.from_numpy(inp))
    d_raw, d_view = device_buffer(n_dst_cap * eb, FILL, dst_offset)
    if stream is None:
        lm.layout_copy_ptr(plan, s_view.data_ptr(), n_src_cap,
                           d_view.data_ptr(), n_dst_cap)
    else:
        with torch.cuda.stream(stream):
            lm.layout_copy_ptr(plan, s_view.data_ptr(), n_src_cap,
                               d_view.data_ptr(), n_dst_cap, stream)
        stream.synchronize()
    torch.cuda.synchronize()
    # a bulk-path LM_OK holds only once no bounded wait gave up
    assert lm.device_status() == 0
    got = d_view.cpu().numpy()
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (
        f"{bad.size} bytes differ, first at byte {bad[:8].tolist()} "
        f"plan={plan.describe()}")
    g = d_raw.cpu().numpy()
    assert (g[:GUARD + dst_offset] == GUARD_FILL).all()
    assert (g[GUARD + dst_offset + n_dst_cap * eb:] == GUARD_FILL).all()
    if sentinel is not None:
        pat = np.frombuffer(np.array([sentinel], dtype=np.uint64).tobytes(),
                            dtype=np.uint8)[:eb]
        rows = got.reshape(-1, eb)
        assert not (rows == pat).all(axis=1).any()
    return plan


# --------------------------------------------------------------------------
# small cases: several tiles, ragged tails, every element size
# --------------------------------------------------------------------------

SMALL = [
    # (name, src, dst, eb)
    ("c1", WORKLOADS["C1"].src, WORKLOADS["C1"].dst, 4),
    ("transpose_ragged_f32", ("layout", (200, 136), (1, 200)),
     ("layout", (200, 136), (136, 1)), 4),
    ("transpose_1000x1000_f16", ("layout", (1000, 1000), (1, 1000)),
     ("layout", (1000, 1000), (1000, 1)), 2),
    ("transpose_prime_u8", ("layout", (97, 131), (1, 97)),
     ("layout", (97, 131), (131, 1)), 1),
    ("transpose_b128", ("layout", (50, 60), (1, 50)),
     ("layout", (50, 60), (60, 1)), 16),
    ("transpose_f64", ("layout", (300, 257), (1, 300)),
     ("layout", (300, 257), (257, 1)), 8),
    ("tiles_swizzled_bf16",
     ("zipped_divide", ("layout", (512, 384), (384, 1)), (64, 64)),
     ("swizzle", 3, 4, 3,
      ("layout", ((64, 64), (8, 6)), ((64, 1), (24576, 4096)))), 2),
    ("padded_tv_gather_f64",
     ("concat", WORKLOADS["C4"].src[1], ("layout", 3001, 72)),
     ("layout", (((4, 8), 2), 3001), (((1, 4), 32), 64)), 8),
    ("nhwc_to_nchw_f16", ("layout", (3, 40, 7, 9), (2520, 1, 360, 40)),
     ("layout", (3, 40, 7, 9), (2520, 63, 9, 1)), 2),
    ("nhwc_to_nchw_big_c", ("layout", (2, 256, 14, 14), (50176, 1, 3584, 256)),
     ("layout", (2, 256, 14, 14), (50176, 196, 14, 1)), 2),
    ("head_interleave_f16", ("layout", (2, 1000, 24), (24000, 24, 1)),
     ("layout", (2, 1000, 24), (1, 48, 2)), 2),
    ("head_interleave_full_rows", ("layout", (2, 4096, 128), (524288, 128, 1)),
     ("layout", (2, 4096, 128), (1, 256, 2)), 2),
    # in-register interleaves of 4 and 8 rows, fp32 pairs, a batch mode
    ("interleave_4_rows_f16", ("layout", (4, 3000, 8), (24000, 8, 1)),
     ("layout", (4, 3000, 8), (1, 32, 4)), 2),
    ("interleave_8_rows_u8", ("layout", (8, 5000), (5008, 1)),
     ("layout", (8, 5000), (1, 8)), 1),
    ("interleave_pairs_f32", ("layout", (2, 7, 1024), (1024, 2048, 1)),
     ("layout", (2, 7, 1024), (1, 2048, 2)), 4),
    ("interleave_ragged_run_f16", ("layout", (2, 5003), (5008, 1)),
     ("layout", (2, 5003), (1, 2)), 2),
    ("interleave_unaligned_rows_f16", ("layout", (2, 4000), (4001, 1)),
     ("layout", (2, 4000), (1, 2)), 2),
    # a swizzled destination keeps the 2-row interleave in shared memory
    ("interleave_swizzled_dst_f16", ("layout", (2, 4096), (4096, 1)),
     ("swizzle", 2, 3, 6, ("layout", (2, 4096), (1, 2))), 2),
    ("identity_vec", ("layout", 100003, 1), ("layout", 100003, 1), 4),
    ("run_then_transpose", ("layout", (8, 300, 70), (1, 8, 2400)),
     ("layout", (8, 300, 70), (1, 560, 8)), 2),
    ("gap_dst_untouched", ("layout", (64, 300), (1, 64)),
     ("layout", (64, 300), (301, 1)), 4),
    ("broadcast_src", ("layout", (512, 33), (1, 0)),
     ("layout", (512, 33), (33, 1)), 4),
    ("swizzled_src", ("swizzle", 2, 4, 4, ("layout", (128, 96), (96, 1))),
     ("layout", (128, 96), (1, 128)), 2),
    # 6 and 5 do not nest, and the padded strides keep both sides from
    # coalescing into one run: no common refinement, GENERIC
    ("non_refinable_generic", ("layout", (6, 5), (1, 7)),
     ("layout", (5, 6), (7, 1)), 4),
    # the same shapes refine once a side is seen as one run: the row-major
    # 600x700 matrix against the destination (700,600):(1,700) = 420000:1
    # is a transpose
    ("coalesced_refinement_f32", ("layout", (600, 700), (700, 1)),
     ("layout", (700, 600), (1, 700)), 4),
    ("coalesced_refinement_small_u8", ("layout", (6, 5), (5, 1)),
     ("layout", (5, 6), (1, 5)), 1),
    # no common refinement, tiled through shared memory (GTILE): the source
    # outer (its unit-stride leaf behind 300 indices), the destination
    # inner; then the other way round; ragged tiles on both axes
    ("gtile_outer_src_f32", ("layout", (300, 350), (350, 1)),
     ("layout", (350, 300), (1, 351)), 4),
    ("gtile_outer_dst_f16", ("layout", (350, 300), (1, 351)),
     ("layout", (300, 350), (350, 1)), 2),
    ("gtile_u8", ("layout", (100, 90), (90, 1)),
     ("layout", (90, 100), (1, 91)), 1),
    ("gtile_ragged_f64", ("layout", (1000, 77), (77, 1)),
     ("layout", (77, 1000), (1, 79)), 8),
    ("gtile_b128", ("layout", (40, 50), (50, 1)),
     ("layout", (50, 40), (1, 51)), 16),
    ("gtile_swizzled_src_f32",
     ("swizzle", 3, 0, 4, ("layout", (128, 100), (100, 1))),
     ("layout", (100, 128), (1, 101)), 4),
    ("gtile_three_leaves_f32", ("layout", (40, 40, 33), (40, 1, 1600)),
     ("layout", (33, 1600), (1, 35)), 4),
    # sources whose rows start on 16-byte boundaries: tensor-map loads of
    # 128-byte swizzled boxes (fp16, fp32, fp64; ragged on both axes; a
    # swizzled destination)
    ("gtma_f32", ("layout", (300, 352), (352, 1)),
     ("layout", (352, 300), (1, 353)), 4),
    ("gtma_f16", ("layout", (200, 136), (136, 1)),
     ("layout", (136, 200), (1, 137)), 2),
    ("gtma_f64", ("layout", (130, 100), (100, 1)),
     ("layout", (100, 130), (1, 101)), 8),
    ("gtma_dst_swizzled_f32", ("layout", (128, 96), (96, 1)),
     ("swizzle", 2, 0, 4, ("layout", (96, 128), (1, 97))), 4),
    # a destination of three leaves: the 4-leaf form with 64-bit offsets
    ("gtile_wide_leaves_f32", ("layout", (40, 40, 33), (40, 1, 1600)),
     ("layout", (33, 40, 40), (1, 35, 1401)), 4),
    ("transpose_tall_f32", ("layout", (2048, 96), (1, 2048)),
     ("layout", (2048, 96), (96, 1)), 4),
    ("vec_untiled_prime", ("layout", (8, 2053), (1, 8)),
     ("layout", (8, 2053), (1, 16)), 2),
    ("rank5_mixed", ("layout", (3, 4, 5, 6, 7), (1, 3, 12, 60, 360)),
     ("layout", (3, 4, 5, 6, 7), (840, 210, 42, 7, 1)), 2),
]


@pytest.mark.parametrize("name,src,dst,eb", SMALL, ids=[c[0] for c in SMALL])
def test_small_parity(name, src, dst, eb):
    run_case(src, dst, eb)


def test_small_parity_paths_cover_every_kernel():
    seen = set()
    for _, src, dst, eb in SMALL:
        p = lm.Plan(lm.build_layout(src), lm.build_layout(dst), eb)
        for pc in p.describe()["pieces"]:
            if pc["path"] == "STAGED":
                seen.add("STAGED/" + pc["store"] + str(pc["rows"]))
            elif pc["path"] == "GTILE" and pc["tma"]:
                seen.add("GTILE/tma")
            else:
                seen.add(pc["path"])
    assert {"GENERIC", "GTILE", "GTILE/tma", "VEC", "ZIP",
            "STAGED/gather0"} <= seen
    assert {"STAGED/transpose2", "STAGED/transpose4",
            "STAGED/transpose8"} <= seen, seen


@pytest.mark.parametrize("eb", [1, 2, 4, 8, 16])
def test_every_element_size_staged_and_vec(eb):
    run_case(("layout", (96, 80), (1, 96)), ("layout", (96, 80), (80, 1)), eb)
    run_case(("layout", (64, 90), (1, 70)), ("layout", (64, 90), (1, 64)), eb)


@pytest.mark.parametrize("src_off,dst_off", [(4, 0), (0, 8), (1, 3), (16, 16)])
def test_misaligned_pointers_fall_back(src_off, dst_off):
    run_case(("layout", (256, 96), (1, 256)), ("layout", (256, 96), (96, 1)),
             4, src_offset=src_off, dst_offset=dst_off)
    run_case(("layout", 50000, 1), ("layout", 50000, 1), 2,
             src_offset=src_off, dst_offset=dst_off)


def test_runs_on_side_stream():
    s = torch.cuda.Stream()
    run_case(("layout", (640, 320), (1, 640)), ("layout", (640, 320), (320, 1)),
             4, stream=s)


def test_random_bijections():
    rng = np.random.default_rng(2024)
    for trial in range(40):
        nm = int(rng.integers(1, 5))
        ext = [int(v) for v in rng.integers(1, 70, nm)]
        def compact(perm, pad):
            stride = [0] * nm
            acc = 1
            for k in perm:
                stride[k] = acc
                acc *= ext[k] + (pad if k == perm[0] else 0)
            return tuple(stride)
        s = ("layout", tuple(ext),
             compact(rng.permutation(nm), int(rng.integers(0, 3))))
        d = ("layout", tuple(ext), compact(rng.permutation(nm), 0))
        if rng.random() < 0.25:
            d = ("swizzle", int(rng.integers(1, 4)), int(rng.integers(2, 5)),
                 3, d)
        eb = int(rng.choice([1, 2, 4, 8, 16]))
        run_case(s, d, eb, seed=trial)


def test_empty_layout_is_a_no_op():
    plan = lm.Plan(lm.Layout.parse("(0,5):(1,0)"), lm.Layout.parse("(0,5):(5,1)"), 4)
    buf = torch.full((64,), FILL, dtype=torch.uint8, device="cuda")
    lm.layout_copy_ptr(plan, buf.data_ptr(), 0, buf.data_ptr() + 32, 0)
    torch.cuda.synchronize()
    assert (buf.cpu() == FILL).all()


def test_capacity_and_overlap_errors_on_device_buffers():
    plan = lm.Plan(lm.Layout.parse("(64,64):(1,64)"),
                   lm.Layout.parse("(64,64):(64,1)"), 4)
    a = torch.zeros(4096, dtype=torch.float32, device="cuda")
    b = torch.zeros(4095, dtype=torch.float32, device="cuda")
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.layout_copy(plan, a, b)
    assert e.value.status == -6
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.layout_copy(plan, a, a)
    assert e.value.status == -7


def test_src_capacity_exactly_cosize_staged_tail():
    """The padded gather loads whole 16-byte chunks; at the very end of the
    source the last chunk reaches past cosize and is clipped."""
    run_case(("concat", WORKLOADS["C4"].src[1], ("layout", 4096, 72)),
             ("layout", (((4, 8), 2), 4096), (((1, 4), 32), 64)), 8,
             sentinel=0x7FF8DEADBEEF0001)


# --------------------------------------------------------------------------
# layout_eval
# --------------------------------------------------------------------------

@pytest.mark.parametrize("spec", [
    EVAL_C1, WORKLOADS["C1"].dst, WORKLOADS["C3"].dst, WORKLOADS["C4"].src,
    ("layout", (7, 11, 13), (1, 1000, 7)),
    # tiles that cut a leaf: 6 x 500 of (6,1000,...), 15 x 256 of 2^22
    ("layout", (6, 1000, 7), (7000, 7, 1)),
    ("layout", (3, 5, 1 << 22), (5, 1, 15)),
    ("swizzle", 2, 3, 6, ("layout", (12, 64, 40), (64, 1, 768))),
])
@pytest.mark.parametrize("width", [4, 8])
def test_layout_eval_device(spec, width):
    L = lm.build_layout(spec)
    O = lo.build(spec)
    dt = torch.int32 if width == 4 else torch.int64
    table = torch.full((O.size + 3,), -7, dtype=dt, device="cuda")
    lm.layout_eval_device(L, table)
    torch.cuda.synchronize()
    got = table.cpu().numpy()
    assert (got[O.size:] == -7).all()
    n = O.size
    idx = np.arange(n) if n <= 1 << 22 else np.unique(np.concatenate([
        np.arange(4096), np.arange(n - 4096, n),
        np.random.default_rng(5).integers(0, n, 1 << 20)]))
    assert (got[idx] == O.at(idx)).all()


def test_layout_eval_c1_blocked_page_values():
    L = lm.build_layout(EVAL_C1)
    table = torch.empty(64, dtype=torch.int32, device="cuda")
    lm.layout_eval_device(L, table)
    t = table.cpu().numpy()
    assert sorted(set(t.tolist())) == sorted(set(lo.image(lo.build(EVAL_C1)).tolist()))
    assert len(set(t.tolist())) == 48 and t.max() == 47
    # (r=1, c=0) -> 2 and (r=3, c=1)? read as the leaf coordinate (3,0,1,0):
    # colex index 3 + 4*0 + 8*1 = 11 -> 6 + 1 = 7
    assert t[1] == 2 and t[3 + 8] == 7


# --------------------------------------------------------------------------
# layouts built by the products ("CUTE布局代数" §4.1), copied on the device
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", PRODUCT_CASES, ids=[c[0] for c in PRODUCT_CASES])
def test_product_built_layouts(case):
    """Copies whose source or destination the library builds with
    blocked_product / logical_product, compared in full with the oracle's
    products (BlockedProduct, LogicalProduct) through its copy."""
    name, s, d, eb, built, paths = case
    side = s if s[0].endswith("product") else d
    assert str(lm.build_layout(side)) == built
    run_case(s, d, eb, seed=900 + sum(map(ord, name)) % 97,
             expect_paths=paths)


# --------------------------------------------------------------------------
# full-size workloads (the bench's plans), compared in full
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5a", "C5b"])
def test_full_size_workload(name):
    w = WORKLOADS[name]
    sentinel = 0x7FF8DEADBEEF0001 if name == "C4" else None
    run_case(w.src, w.dst, w.elem_bytes, values=w.values, dtype=w.dtype,
             seed=w.seed, sentinel=sentinel, src_round16=True)
    assert lm.device_status() == 0


# --------------------------------------------------------------------------
# the two load paths of STAGED and the bounded waits of the bulk path
# --------------------------------------------------------------------------

VARIANT_CASES = ["transpose_ragged_f32", "transpose_1000x1000_f16",
                 "padded_tv_gather_f64", "head_interleave_full_rows",
                 "tiles_swizzled_bf16", "identity_vec", "transpose_tall_f32",
                 "interleave_4_rows_f16", "interleave_8_rows_u8"]


def test_bulk_path_is_planned_for_long_segments():
    """C4's 9 KiB segments load by one bulk copy each; the transposes (C2,
    C5a) keep per-thread cp.async loads (tensor-map boxes only with
    LM_TMA=1)."""
    for name, bulk, tma in (("C2", False, False), ("C4", True, False),
                            ("C5a", False, False)):
        w = WORKLOADS[name]
        d = lm.Plan(lm.build_layout(w.src), lm.build_layout(w.dst),
                    w.elem_bytes).describe()
        assert all(p["bulk"] == bulk and p["tma"] == tma
                   for p in d["pieces"]), (name, d)


def test_short_interleaves_plan_the_register_path():
    """The 2-head interleave and the small interleave cases move through
    registers (ZIP, no shared memory); rows not 16-byte aligned stay on the
    shared-memory transpose."""
    cases = {c[0]: c for c in SMALL}
    for name, rows in (("head_interleave_f16", 2), ("interleave_4_rows_f16", 4),
                       ("interleave_8_rows_u8", 8), ("interleave_pairs_f32", 2)):
        _, s, d, eb = cases[name]
        pieces = lm.Plan(lm.build_layout(s), lm.build_layout(d),
                         eb).describe()["pieces"]
        # a run that is not a whole number of vectors leaves a GENERIC tail
        assert pieces[0]["path"] == "ZIP", (name, pieces)
        assert all(p["path"] == "GENERIC" for p in pieces[1:]), (name, pieces)
        assert pieces[0]["rows"] == rows
    _, s, d, eb = cases["interleave_unaligned_rows_f16"]
    paths = [p["path"] for p in lm.Plan(lm.build_layout(s), lm.build_layout(d),
                                        eb).describe()["pieces"]]
    assert "ZIP" not in paths
    w = WORKLOADS["C5b"]
    pieces = lm.Plan(lm.build_layout(w.src), lm.build_layout(w.dst),
                     w.elem_bytes).describe()["pieces"]
    assert [p["path"] for p in pieces] == ["ZIP"]


@pytest.mark.parametrize("env", [{"LM_BULK": "0"},
                                 {"LM_BULK": "0", "LM_STAGES": "3"},
                                 {"LM_TMA": "1"},
                                 {"LM_TMA": "1", "LM_TMA_SWIZZLE": "0"},
                                 {"LM_TMA": "1", "LM_TMA_SWIZZLE": "0",
                                  "LM_TMA_ACFAST": "0"},
                                 {"LM_BULK_STAGES": "2", "LM_TMA": "1",
                                  "LM_TMA_STAGES": "2"},
                                 {"LM_BULK_STAGES": "4", "LM_TMA": "1",
                                  "LM_TMA_STAGES": "4", "LM_VEC_UNROLL": "8"},
                                 {"LM_ZIP": "0"}])
def test_pipeline_variants_parity(env):
    """The cp.async load path (LM_BULK=0, 2 or 3 stages), tensor-map tile
    loads for transposes (LM_TMA=1, both micro-tile orders) and other
    pipeline depths, in a fresh process since the knobs are read once."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import test_gpu_parity as t\n"
        "t.lm.lib()\n"
        "cases = {c[0]: c for c in t.SMALL}\n"
        "for n in %r:\n"
        "    _, s, d, eb = cases[n]\n"
        "    p = t.run_case(s, d, eb)\n"
        "    bulk = [pc.get('bulk') for pc in p.describe()['pieces']]\n"
        "    if %r == '0': assert not any(bulk), (n, bulk)\n"
        "print('ok')\n" % (here, os.path.dirname(here), VARIANT_CASES,
                           env.get("LM_BULK", "1")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, env={**os.environ, **env}, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


GTILE_CASES = ["gtile_outer_src_f32", "gtile_outer_dst_f16", "gtile_u8",
               "gtile_ragged_f64", "gtile_b128", "gtile_swizzled_src_f32",
               "gtile_three_leaves_f32", "gtma_f32", "gtma_f16", "gtma_f64",
               "gtma_dst_swizzled_f32", "gtile_wide_leaves_f32",
               "non_refinable_generic"]


@pytest.mark.parametrize("env", [{"LM_GTILE_TMA": "0"},
                                 {"LM_GTILE_TMA": "0", "LM_GTILE_U": "32"},
                                 {"LM_GTILE": "0"}])
def test_gtile_variants_parity(env):
    """The pairs without a common refinement in every form: tiles loaded by
    per-thread cp.async instead of tensor map (LM_GTILE_TMA=0), 32-row tiles
    (LM_GTILE_U=32), and one element per thread (LM_GTILE=0), each compared
    in full with the oracle, in a fresh process since the knobs are read
    once."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import test_gpu_parity as t\n"
        "t.lm.lib()\n"
        "cases = {c[0]: c for c in t.SMALL}\n"
        "for n in %r:\n"
        "    _, s, d, eb = cases[n]\n"
        "    p = t.run_case(s, d, eb)\n"
        "    paths = [pc['path'] for pc in p.describe()['pieces']]\n"
        "    if %r: assert 'GTILE' not in paths, (n, paths)\n"
        "print('ok')\n" % (here, os.path.dirname(here), GTILE_CASES,
                           env.get("LM_GTILE") == "0"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, env={**os.environ, **env}, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_tensor_map_transposes_full_size():
    """The opt-in tensor-map loads (LM_TMA=1) on the full-size fp32
    transpose and NHWC->NCHW, compared in full with the oracle, in a fresh
    process since the knob is read once."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import test_gpu_parity as t\n"
        "from workloads import WORKLOADS\n"
        "t.lm.lib()\n"
        "for n in ('C2', 'C5a'):\n"
        "    w = WORKLOADS[n]\n"
        "    p = t.run_case(w.src, w.dst, w.elem_bytes, values=w.values,\n"
        "                   dtype=w.dtype, seed=w.seed, src_round16=True)\n"
        "    assert all(pc['tma'] for pc in p.describe()['pieces']), n\n"
        "print('ok')\n" % (here, os.path.dirname(here)))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, env={**os.environ, "LM_TMA": "1"},
                       timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_bounded_wait_gives_up_and_reports():
    import ctypes as C
    st = C.c_int(123)
    L = lm.lib()
    assert L.lm_selftest_bounded_wait(1, None, C.byref(st)) == 0
    assert st.value == 0
    assert L.lm_selftest_bounded_wait(0, None, C.byref(st)) == 0
    assert st.value == -9                    # LM_E_TIMEOUT, after ~1 s
    assert lm.device_status() == 0           # the self-test cleared it
    # the context is still usable
    run_case(("layout", (96, 80), (1, 96)), ("layout", (96, 80), (80, 1)), 4)
    assert lm.device_status() == 0


@pytest.mark.parametrize("world", [2, 3])
def test_shards_compose_the_full_copy(world):
    """All shards of a copy, run one after another on the same buffers, give
    the oracle's full result (the shards of a multi-device run, on one)."""
    for name in ("C2", "C4", "C5b"):
        w = WORKLOADS[name]
        S, D = lm.build_layout(w.src), lm.build_layout(w.dst)
        OS, OD = lo.build(w.src), lo.build(w.dst)
        eb = w.elem_bytes
        n_src = -(-(S.cosize * eb) // 16) * 16 // eb
        inp = seeded_bytes(w.values, w.dtype, n_src, w.seed)
        want = np.full(D.cosize * eb, FILL, dtype=np.uint8)
        lo.copy(OS, OD, inp, want, eb)
        src = torch.from_numpy(inp).cuda()
        dst = torch.full((D.cosize * eb,), FILL, dtype=torch.uint8,
                         device="cuda")
        for r in range(world):
            lm.layout_copy(lm.Plan(S, D, eb, rank=r, world=world), src, dst)
        torch.cuda.synchronize()
        assert np.array_equal(dst.cpu().numpy(), want), name


@pytest.mark.parametrize("name", ["transpose_ragged_f32", "gap_dst_untouched",
                                  "head_interleave_f16", "padded_tv_gather_f64"])
def test_copy_host_buffers_round_trip(name):
    """lm_layout_copy_host: upload, copy and download on a side stream from
    and into pinned host tensors; destination slots outside the image (the
    gap case) come back with the host's own bytes."""
    _, s, d, eb = {c[0]: c for c in SMALL}[name]
    S, D = lm.build_layout(s), lm.build_layout(d)
    plan = lm.Plan(S, D, eb)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 31)
    host_dst = np.full(D.cosize * eb, 0x3C, dtype=np.uint8)
    want = host_dst.copy()
    lo.copy(lo.build(s), lo.build(d), inp, want, eb)
    hs = torch.from_numpy(inp).pin_memory()
    hd = torch.from_numpy(host_dst).pin_memory()
    sd = torch.full((S.cosize * eb,), 0x11, dtype=torch.uint8, device="cuda")
    dd = torch.full((D.cosize * eb,), 0x22, dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    lm.layout_copy_host(plan, hs, hd, sd, dd, st)
    st.synchronize()
    assert np.array_equal(hd.numpy(), want)


def test_copy_beyond_2_to_32_elements_sampled():
    """The 70000x70000 byte transpose (4.9e9 elements, 64-bit offsets,
    several pieces), checked at 300000 seeded logical indices computed one
    by one by the oracle, plus a guard band past the destination."""
    S = lm.Layout.parse("(70000,70000):(1,70000)")
    D = lm.Layout.parse("(70000,70000):(70000,1)")
    plan = lm.Plan(S, D, 1)
    n = 70000 * 70000
    inp = seeded_bytes("bytes", "uint8", n, 77)
    src = torch.from_numpy(inp).cuda()
    raw = torch.full((n + GUARD,), GUARD_FILL, dtype=torch.uint8, device="cuda")
    lm.layout_copy(plan, src, raw[:n])
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    i = np.concatenate([rng.integers(0, n, 300000), [0, n - 1, 2 ** 31,
                                                     2 ** 32 + 7]])
    OS, OD = lo.parse("(70000,70000):(1,70000)"), lo.parse(
        "(70000,70000):(70000,1)")
    so, do = OS.at(i), OD.at(i)
    got = raw[torch.from_numpy(do).cuda()].cpu().numpy()
    assert (got == inp[so]).all()
    assert (raw[n:].cpu().numpy() == GUARD_FILL).all()


def test_copy_host_buffers_by_shards_on_streams():
    """Shards of one copy (lm_plan_copy_shard), each through
    lm_layout_copy_host on its own stream over shared host and device
    buffers: each moves only its own ranges and together they give the
    oracle's result.  A shard whose destination range is not its own is
    refused."""
    _, s, d, eb = {c[0]: c for c in SMALL}["padded_tv_gather_f64"]
    S, D = lm.build_layout(s), lm.build_layout(d)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 41)
    want = np.full(D.cosize * eb, 0x3C, dtype=np.uint8)
    lo.copy(lo.build(s), lo.build(d), inp, want, eb)
    hs = torch.from_numpy(inp).pin_memory()
    hd = torch.from_numpy(np.full(D.cosize * eb, 0x3C, np.uint8)).pin_memory()
    sd = torch.full((S.cosize * eb,), 0x11, dtype=torch.uint8, device="cuda")
    dd = torch.full((D.cosize * eb,), 0x22, dtype=torch.uint8, device="cuda")
    plans = [lm.Plan(S, D, eb, rank=r, world=3) for r in range(3)]
    assert all(p.describe()["dst_own"] for p in plans)
    streams = [torch.cuda.Stream() for _ in plans]
    for p, st in zip(plans, streams):
        lm.layout_copy_host(p, hs, hd, sd, dd, st)
    torch.cuda.synchronize()
    assert np.array_equal(hd.numpy(), want)
    A = lm.Layout.parse("(4,100):(100,1)")
    shared = lm.Plan(A, A, 4, rank=1, world=8)
    assert not shared.describe()["dst_own"]
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.layout_copy_host(shared, torch.zeros(400).pin_memory(),
                            torch.zeros(400).pin_memory(),
                            torch.zeros(400, device="cuda"),
                            torch.zeros(400, device="cuda"))
    assert e.value.status == -1


@pytest.mark.parametrize("dst_t,path", [
    # no common refinement: 6000 and 7000 do not nest and the padded
    # destination does not coalesce; tiled through shared memory (GTILE)
    ("(7000,6000):(1,7001)", "GTILE"),
    # the destination is the single run 42000000:1: a transpose (STAGED)
    ("(7000,6000):(1,7000)", "STAGED"),
])
def test_generic_without_common_refinement_full_size_sampled(dst_t, path):
    """The 6000x7000 fp32 pairs bench.py times, checked at 200000 seeded
    logical indices computed one by one by the oracle, plus the guard
    band."""
    src_t = "(6000,7000):(7000,1)"
    S, D = lm.Layout.parse(src_t), lm.Layout.parse(dst_t)
    plan = lm.Plan(S, D, 4)
    assert [p["path"] for p in plan.describe()["pieces"]] == [path]
    n = S.size
    inp = seeded_bytes("bytes", "uint8", S.cosize * 4, 13)
    src = torch.from_numpy(inp).cuda()
    raw = torch.full((D.cosize * 4 + GUARD,), GUARD_FILL, dtype=torch.uint8,
                     device="cuda")
    lm.layout_copy(plan, src, raw[:D.cosize * 4])
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    i = np.concatenate([rng.integers(0, n, 200000), [0, n - 1]])
    so, do = lo.parse(src_t).at(i), lo.parse(dst_t).at(i)
    got = raw[:D.cosize * 4].view(torch.int32)[torch.from_numpy(do).cuda()]
    want = inp.view(np.int32)[so]
    assert (got.cpu().numpy() == want).all()
    assert (raw[D.cosize * 4:].cpu().numpy() == GUARD_FILL).all()


# --------------------------------------------------------------------------
# randomized: pairs without a common refinement, layout_eval tilings
# --------------------------------------------------------------------------

def _random_non_refinable(rng):
    """Matrices (a, b) and (c, d) of equal size whose extents do not nest
    (a and c do not divide each other), each side row- or column-major,
    padded so that no side coalesces into one run."""
    while True:
        a, c = int(rng.integers(33, 160)), int(rng.integers(33, 160))
        if a % c and c % a:
            break
    n = int(np.lcm(a, c)) * int(rng.integers(1, 3))
    while n < 2000:
        n *= 2
    b, d = n // a, n // c

    def side(r, k):
        pad = int(rng.integers(1, 4))
        if rng.integers(2):
            return ("layout", (r, k), (k + pad, 1))   # rows, padded
        return ("layout", (r, k), (1, r + pad))       # columns, padded

    src, dst = side(a, b), side(c, d)
    if rng.integers(4) == 0:
        src = ("swizzle", 2, 0, 5, src)
    return src, dst, int(rng.choice([1, 2, 4, 8, 16]))


def test_random_non_refinable_pairs():
    """Random pairs without a common refinement, on whichever path the
    planner picks (GTILE when a side runs along the logical index, else
    GENERIC), compared in full with the oracle."""
    rng = np.random.default_rng(4242)
    paths = set()
    for k in range(24):
        src, dst, eb = _random_non_refinable(rng)
        S, D = lm.build_layout(src), lm.build_layout(dst)
        try:
            plan = lm.Plan(S, D, eb)
        except lm.LayoutMoveError as e:       # a swizzle that collides
            assert e.status == -4
            continue
        d = plan.describe()
        assert not d["joint"], (src, dst)
        paths.update(p["path"] for p in d["pieces"])
        run_case(src, dst, eb, seed=300 + k)
    assert "GTILE" in paths


def test_random_layout_eval_tables():
    """Random layouts of 2-4 leaves (some swizzled) into int32 and int64
    tables, whichever kernel the shape gets (tiled or per element),
    compared in full with the oracle."""
    rng = np.random.default_rng(515)
    for k in range(16):
        nl = int(rng.integers(2, 5))
        ext = [int(v) for v in rng.integers(2, 40, nl)]
        perm = rng.permutation(nl)
        stride, span = [0] * nl, 1
        for j in perm:
            stride[j] = span
            span *= ext[j] + int(rng.integers(0, 3))
        spec = ("layout", tuple(ext), tuple(stride))
        if rng.integers(3) == 0:
            spec = ("swizzle", 2, 1, 6, spec)
        L, O = lm.build_layout(spec), lo.build(spec)
        dt = torch.int32 if k % 2 else torch.int64
        table = torch.full((O.size + 5,), -3, dtype=dt, device="cuda")
        lm.layout_eval_device(L, table)
        got = table.cpu().numpy()
        assert (got[:O.size] == lo.image(O)).all(), spec
        assert (got[O.size:] == -3).all()
