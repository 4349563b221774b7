"""GPU parity of the thread-value partitioned tile copy (lm_tv_copy).

Each tile goes global -> shared -> global through the device functions of
include/layoutmove_tv.cuh, every thread moving its local_partition of the
tile ("CUTLASS Layout可视化" §5.3).  The shared layout and the thread
layouts only decide who moves what and where it waits, so the result must
be the oracle's out[dst(i)] = in[src(i)], byte for byte, with untouched
destination slots and guard bands intact.
"""

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import WORKLOADS, seeded_bytes
from tv_cases import CASES, zd

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


def device_buffer(nbytes, fill):
    raw = torch.full((nbytes + 2 * GUARD,), GUARD_FILL, dtype=torch.uint8,
                     device="cuda")
    view = raw[GUARD:GUARD + nbytes]
    view.fill_(fill)
    return raw, view


def run_tv(src_spec, smem_spec, dst_spec, thr_l, thr_s, eb, vl=0, vs=0,
           seed=11, expect=None):
    S, D = lm.build_layout(src_spec), lm.build_layout(dst_spec)
    M = lm.build_layout(smem_spec)
    plan = lm.TVPlan(S, M, D,
                     lm.Layout.parse(thr_l) if thr_l is not None else None,
                     lm.Layout.parse(thr_s) if thr_s is not None else None,
                     eb, vl, vs)
    desc = plan.describe()
    if expect:
        for k, v in expect.items():
            phase, key = k.split(".")
            assert desc[phase][key] == v, (k, desc)
    OS, OD = lo.build(src_spec), lo.build(dst_spec)
    n_src, n_dst = S.cosize, D.cosize
    inp = seeded_bytes("bytes", "uint8", n_src * eb, seed)
    want = np.full(n_dst * eb, FILL, dtype=np.uint8)
    lo.copy(OS, OD, inp, want, eb)
    s_raw, s_view = device_buffer(n_src * eb, 0)
    s_view.copy_(torch.from_numpy(inp))
    d_raw, d_view = device_buffer(n_dst * eb, FILL)
    lm.tv_copy(plan, s_view, d_view)
    torch.cuda.synchronize()
    got = d_view.cpu().numpy()
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} bytes differ, first {bad[:8]} {desc}"
    g = d_raw.cpu().numpy()
    assert (g[:GUARD] == GUARD_FILL).all()
    assert (g[GUARD + n_dst * eb:] == GUARD_FILL).all()
    return desc


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tv_copy_matches_oracle(case):
    _, src, smem, dst, tl, ts, eb, expect = case
    run_tv(src, smem, dst, tl, ts, eb, expect=expect)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tv_copy_tuned_thread_layouts(case):
    """The same cases with no thread layouts: each phase runs the stripmined
    map whose Pitch and Strips the planner tuned (segments, then bank
    wavefronts); the result is the oracle's copy."""
    name, src, smem, dst, _, _, eb, _ = case
    if name == "nested_tile_modes":      # no tuned layout for nested modes
        return
    desc = run_tv(src, smem, dst, None, None, eb, seed=13)
    assert desc["load"]["tuned"] and desc["store"]["tuned"]


def test_tv_full_size_tuned_transpose_f32():
    """The 4096x4096 fp32 transpose in 64x64 tiles through the conflict-free
    5-bit-XOR shared tile, thread layouts tuned: the tune gives Pitch 64
    (one 256-byte column of the tile per 64 threads) in both phases and
    the bank model no conflicts; compared in full with the oracle."""
    w = WORKLOADS["C2"]
    src = ("zipped_divide", w.src, (64, 64))
    dst = ("zipped_divide", w.dst, (64, 64))
    smem = ("swizzle", 5, 0, 6, ("layout", (64, 64), (1, 64)))
    desc = run_tv(src, smem, dst, None, None, 4, seed=6,
                  expect={"load.pitch": 64, "store.pitch": 64,
                          "load.smem_wavefronts": 128,
                          "store.smem_wavefronts": 128})
    assert desc["n_tiles"] == 64 * 64


def test_tv_mbarrier_pipeline_parity():
    """The mbarrier-paced kernel (LM_TV_MBAR=1, 2 to 4 shared tiles) on every
    case with given and tuned thread layouts and on the full-size bf16
    tiling, in fresh processes since the knobs are read once."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import test_gpu_tv as t\n"
        "t.lm.lib()\n"
        "for c in t.CASES:\n"
        "    name, src, smem, dst, tl, ts, eb, expect = c\n"
        "    t.run_tv(src, smem, dst, tl, ts, eb, expect=expect)\n"
        "    if name != 'nested_tile_modes':\n"
        "        t.run_tv(src, smem, dst, None, None, eb, seed=13)\n"
        "t.test_tv_full_size_tiles_swizzled_bf16()\n"
        "assert t.lm.device_status() == 0\n"
        "print('ok')\n" % (here, os.path.dirname(here)))
    for stages in ("2", "3", "4"):
        r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                           text=True, timeout=900,
                           env={**os.environ, "LM_TV_MBAR": "1",
                                "LM_TV_STAGES": stages})
        assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr


def test_tv_forced_vector_widths():
    src = zd((128, 96), (1, 128), (32, 32))
    dst = zd((128, 96), (96, 1), (32, 32))
    smem = ("layout", (32, 32), (1, 32))
    for vl in (4, 8, 16):
        tl = {4: "(32,8):(1,32)", 8: "(16,16):(1,16)", 16: "(8,32):(1,8)"}[vl]
        run_tv(src, smem, dst, tl, "(32,8):(8,1)", 4, vl, 4,
               expect={"load.vec_bytes": vl})


def test_tv_empty_grid_is_a_no_op():
    S = lm.Layout.parse("((32,32),0):((1,32),1024)")
    M = lm.Layout.parse("(32,32):(1,32)")
    thr = lm.Layout.parse("(8,32):(1,8)")
    plan = lm.TVPlan(S, M, S, thr, thr, 4)
    assert plan.describe()["n_tiles"] == 0
    a = torch.zeros(16, device="cuda")
    b = torch.full((16,), 7.0, device="cuda")
    lm.tv_copy(plan, a, b)
    torch.cuda.synchronize()
    assert (b == 7.0).all()


def test_tv_rejects_on_device_buffers():
    src = lm.build_layout(zd((64, 64), (1, 64), (32, 32)))
    dst = lm.build_layout(zd((64, 64), (64, 1), (32, 32)))
    M = lm.Layout.parse("(32,32):(1,32)")
    plan = lm.TVPlan(src, M, dst, lm.Layout.parse("(8,32):(1,8)"),
                     lm.Layout.parse("(32,8):(8,1)"), 4)
    a = torch.zeros(4096, device="cuda")
    b = torch.zeros(4096, device="cuda")
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.tv_copy(plan, a[:4000], b)
    assert e.value.status == -6          # capacity
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.tv_copy(plan, a, a)
    assert e.value.status == -7          # overlap
    big = torch.zeros(4100, device="cuda")
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.tv_copy(plan, big[1:4097], b)  # 16-byte vectors need alignment
    assert e.value.status == -1


def test_tv_full_size_tiles_swizzled_bf16():
    """The 8192x8192 bf16 swizzled tiling through the building block, with
    the shapes bench.py times; compared in full with the oracle."""
    w = WORKLOADS["C3"]
    desc = run_tv(w.src, ("swizzle", 3, 3, 6, ("layout", (64, 64), (64, 1))),
                  w.dst, "(32,8):(8,1)", "(32,8):(8,1)", 2, seed=3,
                  expect={"load.vec_bytes": 16, "store.vec_bytes": 16})
    assert desc["n_tiles"] == 128 * 128


@pytest.mark.parametrize("smem,tl,ts", [
    (("swizzle", 5, 0, 6, ("layout", (64, 64), (1, 64))), "(32,8):(1,32)",
     "(8,32):(32,1)"),
    (("swizzle", 3, 2, 6, ("layout", (64, 64), (1, 64))), "(16,16):(1,16)",
     "(8,32):(32,1)"),
])
def test_tv_full_size_transpose_f32(smem, tl, ts):
    """The 4096x4096 fp32 transpose in 64x64 tiles, with the layouts
    bench.py times; compared in full with the oracle."""
    w = WORKLOADS["C2"]
    src = ("zipped_divide", w.src, (64, 64))
    dst = ("zipped_divide", w.dst, (64, 64))
    desc = run_tv(src, smem, dst, tl, ts, 4, seed=4)
    assert desc["n_tiles"] == 64 * 64


def test_consumer_kernel_built_apart_uses_the_building_block(tmp_path):
    """A kernel of its own (tests/consumer/tv_consumer.cu), compiled here
    against include/layoutmove_tv.cuh, takes the plan's argument block and
    stages bf16 tiles with load_tile / store_tile, complementing every byte
    in shared memory in between: the result is the oracle's copy of the
    complemented input."""
    import ctypes
    import os
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "tv_consumer.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a",
                    "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-cudart", "static", f"-I{root}/include",
                    os.path.join(root, "tests", "consumer", "tv_consumer.cu"),
                    "-o", so], check=True, capture_output=True, timeout=600)
    cons = ctypes.CDLL(so)
    cons.tv_consumer_launch.restype = ctypes.c_int
    cons.tv_consumer_launch.argtypes = [ctypes.c_void_p] * 3 + [
        ctypes.c_int, ctypes.c_void_p]
    src_spec = zd((512, 384), (384, 1), (64, 64))
    dst_spec = ("swizzle", 3, 4, 3,
                ("layout", ((64, 64), (8, 6)), ((64, 1), (24576, 4096))))
    S, D = lm.build_layout(src_spec), lm.build_layout(dst_spec)
    plan = lm.TVPlan(S, lm.Layout.parse("Sw<3,3,6> o (64,64):(64,1)"), D,
                     lm.Layout.parse("(32,8):(8,1)"),
                     lm.Layout.parse("(32,8):(8,1)"), 2)
    args = ctypes.create_string_buffer(plan.args_bytes(), 8192)
    inp = seeded_bytes("bytes", "uint8", S.cosize * 2, 21)
    want = np.full(D.cosize * 2, FILL, dtype=np.uint8)
    lo.copy(lo.build(src_spec), lo.build(dst_spec), ~inp, want, 2)
    src = torch.from_numpy(inp).cuda()
    dst = torch.full((D.cosize * 2,), FILL, dtype=torch.uint8, device="cuda")
    rc = cons.tv_consumer_launch(args, src.data_ptr(), dst.data_ptr(), 20,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy(), want)


def test_random_tv_cases_on_device():
    """The randomized cases of the host replay (random tiles, padded and
    swizzled shared layouts, thread layouts, element sizes), run on the
    device and compared byte for byte with the oracle."""
    import test_tv_plan as hp
    rng = np.random.default_rng(2024)
    ran = 0
    for _ in range(40):
        case = hp._random_tv_case(rng)
        src_t, dst_t, tile, smem_t, swz, tl, ts, eb = case
        smem = ("layout",) + _parse_pair(smem_t)
        if swz:
            smem = ("swizzle",) + tuple(swz) + (smem,)
        src = ("zipped_divide", ("layout",) + _parse_pair(src_t), tile)
        dst = ("zipped_divide", ("layout",) + _parse_pair(dst_t), tile)
        try:
            run_tv(src, smem, dst, tl, ts, eb, seed=ran)
        except lm.LayoutMoveError as e:
            assert e.status in (-1, -3)
            continue
        ran += 1
    assert ran >= 12


def _parse_pair(text):
    """'(a,b):(c,d)' -> ((a, b), (c, d))"""
    sh, st = text.split(":")
    return (tuple(int(v) for v in sh.strip("()").split(",")),
            tuple(int(v) for v in st.strip("()").split(",")))
