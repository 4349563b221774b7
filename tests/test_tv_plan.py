"""Host side of the thread-value partitioned tile copy (no GPU).

The plan's argument block (include/layoutmove_tv.h) is read back through a
ctypes mirror of the struct, and the device functions of layoutmove_tv.cuh
are replayed in numpy from their documented arithmetic: every address they
would form is checked against its buffer (global offsets inside the
layout's cosize, shared offsets inside the shared tile, both aligned to the
vector), every shared byte is written exactly once per tile before it is
read, and the replayed result must equal the oracle's copy.  The bank
figures of the plan are checked against the oracle's bank model applied to
the oracle's local_partition of the shared tile.
"""

import ctypes as C

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import seeded_bytes
from tv_cases import CASES

lm = pytest.importorskip("layout_driven_movement_gb300")

MAXL, MAXV, MAXG = 6, 128, 8


class Phase(C.Structure):
    _fields_ = [("n_thr", C.c_int32), ("n_val", C.c_int32),
                ("vec_bytes", C.c_int32), ("n_leaves", C.c_int32),
                ("leaf_ext", C.c_int32 * MAXL),
                ("leaf_stride", C.c_int32 * MAXL),
                ("from_step", C.c_int32 * MAXL),
                ("to_step", C.c_int32 * MAXL),
                ("from_val", C.c_int32 * MAXV), ("to_val", C.c_int32 * MAXV)]


class FastDiv(C.Structure):
    _fields_ = [("d", C.c_uint32), ("m", C.c_uint32), ("s1", C.c_uint32),
                ("s2", C.c_uint32)]


class Args(C.Structure):
    _fields_ = [("elem_bytes", C.c_int32), ("smem_bytes", C.c_int32),
                ("block_threads", C.c_int32), ("n_grid", C.c_int32),
                ("n_tiles", C.c_int64), ("grid_ext", C.c_int64 * MAXG),
                ("grid_src", C.c_int64 * MAXG), ("grid_dst", C.c_int64 * MAXG),
                ("grid_div", FastDiv * MAXG),
                ("src_swz", C.c_int32 * 3), ("smem_swz", C.c_int32 * 3),
                ("dst_swz", C.c_int32 * 3), ("grid_fast", C.c_int32),
                ("src_swz_tile", C.c_int32), ("dst_swz_tile", C.c_int32),
                ("offsets32", C.c_int32),
                ("load", Phase), ("store", Phase)]


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def args_of(plan):
    raw = plan.args_bytes()
    return Args.from_buffer_copy(raw[:C.sizeof(Args)])


def swz(o, z):
    return lo.swizzle(o, z[0], z[1], z[2]) if z[0] else o


def thread_bases(p, t):
    f = np.zeros_like(t)
    g = np.zeros_like(t)
    for j in range(p.n_leaves):
        c = (t // p.leaf_stride[j]) % p.leaf_ext[j]
        f = f + c * p.from_step[j]
        g = g + c * p.to_step[j]
    return f, g


def replay(a, src_bytes, dst_bytes, src_cos, dst_cos):
    """The kernel's loop over tiles, phase by phase, in numpy."""
    eb = a.elem_bytes
    for tile in range(a.n_tiles):
        sb = db = 0
        rem = tile
        for k in range(a.n_grid):
            if a.grid_fast:   # the device's 32-bit multiply-shift division
                f = a.grid_div[k]
                t = (f.m * rem) >> 32
                q = (t + ((rem - t) >> f.s1)) >> f.s2
                assert f.d == a.grid_ext[k] and q == rem // f.d
                c = rem - q * f.d
                rem = q
            else:
                c = rem % a.grid_ext[k]
                rem //= a.grid_ext[k]
            sb += c * a.grid_src[k]
            db += c * a.grid_dst[k]
        smem = np.zeros(a.smem_bytes, np.uint8)
        written = np.zeros(a.smem_bytes, np.int32)
        for phase, load in ((a.load, True), (a.store, False)):
            t = np.arange(phase.n_thr, dtype=np.int64)
            bf, bt = thread_bases(phase, t)
            vb = phase.vec_bytes
            assert vb % eb == 0
            for v in range(phase.n_val):
                if load:
                    g = swz((sb + bf + phase.from_val[v]).astype(np.int64),
                            a.src_swz)
                    if a.src_swz_tile:   # the swizzle commutes with the base
                        assert (g == sb + swz(
                            (bf + phase.from_val[v]).astype(np.int64),
                            a.src_swz)).all()
                    s = swz((bt + phase.to_val[v]).astype(np.int64),
                            a.smem_swz)
                    cos = src_cos
                else:
                    s = swz((bf + phase.from_val[v]).astype(np.int64),
                            a.smem_swz)
                    g = swz((db + bt + phase.to_val[v]).astype(np.int64),
                            a.dst_swz)
                    if a.dst_swz_tile:
                        assert (g == db + swz(
                            (bt + phase.to_val[v]).astype(np.int64),
                            a.dst_swz)).all()
                    cos = dst_cos
                # byte offsets
                assert (g >= 0).all() and ((g + vb) <= cos * eb).all()
                assert (s >= 0).all() and ((s + vb) <= a.smem_bytes).all()
                assert (g % vb == 0).all() and (s % vb == 0).all()
                for u in range(vb):
                    gi, si = g + u, s + u
                    if load:
                        smem[si] = src_bytes[gi]
                        np.add.at(written, si, 1)
                    else:
                        assert (written[si] == 1).all()
                        dst_bytes[gi] = smem[si]
        assert written.max() <= 1


TV_CASES = [
    ("(256,192):(1,256)", "(256,192):(192,1)", (32, 32), "(32,32):(1,32)",
     None, "(8,32):(1,8)", "(32,8):(8,1)", 4),
    ("(256,192):(1,256)", "(256,192):(192,1)", (32, 32), "(32,32):(1,33)",
     None, "(32,8):(1,32)", "(8,32):(32,1)", 4),
    ("(256,192):(1,256)", "(256,192):(192,1)", (32, 32), "(32,32):(1,32)",
     (3, 2, 5), "(8,32):(1,8)", "(32,8):(8,1)", 4),
    ("(512,384):(384,1)", "(512,384):(384,1)", (64, 64), "(64,64):(64,1)",
     (3, 3, 6), "(32,8):(8,1)", "(32,8):(8,1)", 2),
    ("(96,80):(1,96)", "(96,80):(80,1)", (32, 16), "(32,16):(16,1)", None,
     "(2,16):(16,1)", "(32,4):(1,32)", 1),
    ("(40,24):(24,1)", "(40,24):(1,40)", (8, 8), "(8,8):(8,1)", None,
     "(8,8):(8,1)", "(8,8):(1,8)", 16),
    ("(128,64):(1,128)", "(128,64):(64,1)", (32, 32), "(32,32):(1,32)", None,
     "(16,16):(1,16)", "(32,2):(2,1)", 8),
]


def build_case(src_t, dst_t, tile, smem_t, smem_swz, tl, ts, eb):
    S = lm.Layout.parse(src_t).zipped_divide(list(tile))
    D = lm.Layout.parse(dst_t).zipped_divide(list(tile))
    M = lm.Layout.parse(smem_t)
    OM = lo.parse(smem_t)
    if smem_swz:
        M = M.swizzle(*smem_swz)
        OM = lo.Swizzled(*smem_swz, OM)
    plan = lm.TVPlan(S, M, D, lm.Layout.parse(tl), lm.Layout.parse(ts), eb)
    OS = lo.ZippedDivide(lo.parse(src_t), tile)
    OD = lo.ZippedDivide(lo.parse(dst_t), tile)
    return plan, S, D, OS, OD, OM


@pytest.mark.parametrize("case", TV_CASES)
def test_replayed_kernel_matches_oracle(case):
    plan, S, D, OS, OD, _ = build_case(*case)
    eb = case[-1]
    a = args_of(plan)
    d = plan.describe()
    assert a.n_tiles == d["n_tiles"]
    assert a.load.vec_bytes == d["load"]["vec_bytes"]
    assert a.store.n_val == d["store"]["values"]
    assert a.block_threads % 32 == 0
    assert a.block_threads >= max(a.load.n_thr, a.store.n_thr)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 5)
    want = np.full(D.cosize * eb, 0xA5, np.uint8)
    lo.copy(OS, OD, inp, want, eb)
    got = np.full(D.cosize * eb, 0xA5, np.uint8)
    replay(a, inp, got, S.cosize, D.cosize)
    assert (got == want).all()


def test_args_block_size_is_checked():
    plan = build_case(*TV_CASES[0])[0]
    buf = C.create_string_buffer(C.sizeof(Args))
    assert lm.lib().lm_tv_plan_args(plan.handle, buf, C.sizeof(Args)) == 0
    assert lm.lib().lm_tv_plan_args(plan.handle, buf,
                                    C.sizeof(Args) - 1) == -11


@pytest.mark.parametrize("case", TV_CASES)
def test_bank_figures_match_oracle_partition(case):
    """Per phase, the shared side's offsets of lane l, value q are the
    oracle's local_partition of the shared tile (grouped into vectors along
    the phase's vector mode) for thread l; their bank wavefronts, summed over
    warps and values, must equal the plan's figure."""
    plan, S, D, OS, OD, OM = build_case(*case)
    eb = case[-1]
    d = plan.describe()
    base = OM.inner if isinstance(OM, lo.Swizzled) else OM
    for name, thr_t in (("load", case[5]), ("store", case[6])):
        ph = d[name]
        v = ph["vec_bytes"] // eb
        g = ph["vec_mode"]
        modes = base.modes()
        # the shared tile counted in vectors along mode g
        grouped = []
        for k, m in enumerate(modes):
            if k == g and v > 1:
                grouped.append(lo.Composed(m, lo.Layout(m.size // v, v)))
            else:
                grouped.append(m)
        unit = _Modes(grouped)
        thr = lo.parse(thr_t)
        parts = np.stack([lo.local_partition(unit, thr, t)
                          for t in range(thr.size)])  # (threads, values)
        if isinstance(OM, lo.Swizzled):
            parts = lo.swizzle(parts, OM.b, OM.m, OM.s)
        total = ideal = 0
        for w0 in range(0, thr.size, 32):
            for q in range(parts.shape[1]):
                wf, idl = lo.smem_wavefronts(parts[w0:w0 + 32, q] * eb,
                                             ph["vec_bytes"])
                total += wf
                ideal += idl
        assert (total, ideal) == (ph["smem_wavefronts"],
                                  ph["smem_wavefronts_ideal"]), name


class _Modes:
    """Oracle-side layout whose top modes are given objects (for grouping a
    mode into vectors); evaluated like the oracle's Layout."""

    def __init__(self, modes):
        self._modes = modes
        self.size = int(np.prod([m.size for m in modes]))

    def modes(self):
        return self._modes

    def at(self, i, extended=False):
        x = np.asarray(i, dtype=np.int64)
        off = np.zeros_like(x)
        for m in self._modes:
            off = off + m.at(x % m.size)
            x = x // m.size
        return off


def test_tv_plan_errors():
    S = lm.Layout.parse("(64,64):(1,64)").zipped_divide([32, 32])
    D = lm.Layout.parse("(64,64):(64,1)").zipped_divide([32, 32])
    M = lm.Layout.parse("(32,32):(1,32)")
    t = lm.Layout.parse("(8,32):(1,8)")
    cases = [
        ((S, M, D, t, t, 3), -1),                                  # elem size
        ((S, lm.Layout.parse("(32,16):(1,32)"), D, t, t, 4), -2),  # smem size
        ((S, lm.Layout.parse("(32,32):(1,16)"), D, t, t, 4), -4),  # smem overlap
        ((S, M, D, lm.Layout.parse("(8,32):(1,4)"), t, 4), -1),    # thr not bijective
        ((S, M, D, lm.Layout.parse("(3,32):(1,3)"), t, 4), -3),    # 3 does not divide
        ((S, M, D, lm.Layout.parse("(2048,1):(1,1)"), t, 4), -1),  # > 1024 threads
        ((S, M, D, lm.Layout.parse("(1,1):(1,1)"), t, 4), -1),     # > 128 values
        ((S, lm.Layout.parse("(256,256):(1,256)"), D, t, t, 4), -2),
    ]
    for (a, m, d, tl, ts, eb), code in cases:
        with pytest.raises(lm.LayoutMoveError) as e:
            lm.TVPlan(a, m, d, tl, ts, eb)
        assert e.value.status == code, (str(m), str(tl), e.value.status)
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.TVPlan(S, M, D, t, t, 4, vec_load_bytes=32)
    assert e.value.status == -1


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_replayed_gpu_cases_match_oracle(case):
    """The GPU parity cases, replayed on the host first."""
    _, src, smem, dst, tl, ts, eb, expect = case
    S, D = lm.build_layout(src), lm.build_layout(dst)
    plan = lm.TVPlan(S, lm.build_layout(smem), D, lm.Layout.parse(tl),
                     lm.Layout.parse(ts), eb)
    d = plan.describe()
    for k, v in (expect or {}).items():
        phase, key = k.split(".")
        assert d[phase][key] == v, (k, d)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 9)
    want = np.full(D.cosize * eb, 0xA5, np.uint8)
    lo.copy(lo.build(src), lo.build(dst), inp, want, eb)
    got = np.full(D.cosize * eb, 0xA5, np.uint8)
    replay(args_of(plan), inp, got, S.cosize, D.cosize)
    assert (got == want).all()


def _random_tv_case(rng):
    eb = int(rng.choice([1, 2, 4, 8]))
    n0, n1 = int(rng.choice([8, 16, 32])), int(rng.choice([8, 16, 32]))
    g0, g1 = int(rng.integers(1, 4)), int(rng.integers(1, 4))
    R, Cc = n0 * g0, n1 * g1

    def matrix(order):
        return f"({R},{Cc}):(1,{R})" if order else f"({R},{Cc}):({Cc},1)"

    src_t, dst_t = matrix(rng.integers(2)), matrix(rng.integers(2))
    pad = int(rng.choice([0, 0, 1, 4]))
    if rng.integers(2):
        smem_t = f"({n0},{n1}):(1,{n0 + pad})"
    else:
        smem_t = f"({n0},{n1}):({n1 + pad},1)"
    swz = None
    if pad == 0 and rng.integers(2):
        b = int(rng.integers(1, 4))
        swz = (b, int(rng.integers(0, 3)), int(rng.integers(b, 6)))
    threads = int(rng.choice([32, 64, 128]))
    t0 = int(rng.choice([1, 2, 4, 8, 16, 32]))
    t0 = min(t0, threads)
    t1 = threads // t0
    tl = f"({t0},{t1}):(1,{t0})" if rng.integers(2) else f"({t0},{t1}):({t1},1)"
    t0s = int(rng.choice([1, 2, 4, 8, 16, 32]))
    t0s = min(t0s, threads)
    ts = f"({t0s},{threads // t0s}):(1,{t0s})"
    return (src_t, dst_t, (n0, n1), smem_t, swz, tl, ts, eb)


def test_random_tv_plans_replay_exactly():
    """Random tiles, shared layouts (padded, swizzled), thread layouts and
    element sizes: every case the planner accepts replays to the oracle's
    copy with every address in bounds; rejections carry a status."""
    rng = np.random.default_rng(2024)
    planned = 0
    for _ in range(40):
        case = _random_tv_case(rng)
        try:
            plan, S, D, OS, OD, _ = build_case(*case)
        except lm.LayoutMoveError as e:
            assert e.status in (-1, -3), (case, e.status)
            continue
        eb = case[-1]
        inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 3)
        want = np.full(D.cosize * eb, 0xA5, np.uint8)
        lo.copy(OS, OD, inp, want, eb)
        got = np.full(D.cosize * eb, 0xA5, np.uint8)
        replay(args_of(plan), inp, got, S.cosize, D.cosize)
        assert (got == want).all(), case
        planned += 1
    assert planned >= 12


# --------------------------------------------------------------------------
# tuned thread layouts (no thread layout from the caller)
# --------------------------------------------------------------------------

def _tile_sizes(spec):
    """Sizes of the tile modes (mode 0's own modes) of a layout expression
    of the oracle."""
    L = lo.build(spec)
    base = L.inner if isinstance(L, lo.Swizzled) else L
    if isinstance(base, lo.ZippedDivide):
        return [int(t) for t in base.tiler]
    t = base.modes()[0]
    return [m.size for m in t.modes()] if not isinstance(t.shape, int) else [t.size]


def _tuned_by_oracle(glob_spec, smem_spec, n, eb, vec, threads):
    """The one-group search the planner documents, recomputed from the
    oracle: the phase's global side gives the row (its unit-stride tile mode
    a, else mode 0; ld = the other mode's step), Pitch x Strips == threads
    with both dividing the tile, cost = (128-byte global segments per warp,
    shared wavefronts of the same accesses, larger Pitch, larger Strips)."""
    G, M = lo.build(glob_spec), lo.build(smem_spec)
    r = len(n)
    weight = [1, n[0]]
    a = 0
    for k in range(r):
        if n[k] > 1 and int(G.at(weight[k])) - int(G.at(0)) == 1:
            a = k
            break
    b = 1 - a if r == 2 else None
    k_row, rows = n[a], (n[b] if b is not None else 1)
    ld = k_row if b is None else max(k_row, int(G.at(weight[b])) - int(G.at(0)))
    R = k_row // vec
    best = None
    P = 1
    while P <= R and P <= threads:
        S = threads // P
        if P * S == threads and R % P == 0 and rows % S == 0:
            t = np.arange(threads)
            row, col = t // P, (t % P) * vec
            g = (row * ld + col) * eb // 128
            if b is None:
                idx = col
            elif a == 0:
                idx = col + n[0] * row
            else:
                idx = row + n[0] * col
            s_off = M.at(idx)
            seg = wf = 0
            for w0 in range(0, threads, 32):
                seg += len(set(g[w0:w0 + 32].tolist()))
                wf += lo.smem_wavefronts(s_off[w0:w0 + 32] * eb, vec * eb)[0]
            key = (seg, wf, -P, -S)
            if best is None or key < best[0]:
                best = (key, P, S, seg)
        P *= 2
    return best[1], best[2], best[3]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tuned_thread_layouts(case):
    """With no thread layouts the planner tunes both phases: the plan replays
    to the oracle's copy with every address in bounds, and each phase's
    Pitch and Strips are the best one-group stripmined map by the oracle's
    own recomputation of the documented cost.  Tiles with nested modes may
    have no tuned layout (LM_E_NOT_REPRESENTABLE)."""
    name, src, smem, dst, _, _, eb, _ = case
    S, D = lm.build_layout(src), lm.build_layout(dst)
    try:
        plan = lm.TVPlan(S, lm.build_layout(smem), D, None, None, eb)
    except lm.LayoutMoveError as e:
        assert name == "nested_tile_modes" and e.status == -3
        return
    d = plan.describe()
    n = _tile_sizes(src)
    for phase, glob in (("load", src), ("store", dst)):
        p = d[phase]
        assert p["tuned"] is True
        vec = p["vec_bytes"] // eb
        pitch, strips, seg = _tuned_by_oracle(glob, smem, n, eb, vec,
                                              p["threads"])
        assert (p["pitch"], p["strips"], p["segments"]) == (pitch, strips,
                                                            seg), (phase, p)
        a = p["vec_mode"]
        want_thr = (f"({pitch},{strips}):(1,{pitch})" if a == 0
                    else f"({strips},{pitch}):({pitch},1)")
        if len(n) == 1:
            want_thr = f"{pitch}:1"
        assert p["thr"] == want_thr, (phase, p)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 19)
    want = np.full(D.cosize * eb, 0xA5, np.uint8)
    lo.copy(lo.build(src), lo.build(dst), inp, want, eb)
    got = np.full(D.cosize * eb, 0xA5, np.uint8)
    replay(args_of(plan), inp, got, S.cosize, D.cosize)
    assert (got == want).all()


def test_tuned_thread_layout_mixes_with_a_given_one():
    """One phase given, the other tuned; a tile of rank 3 cannot be tuned."""
    _, src, smem, dst, tl, _, eb, _ = CASES[0]
    S, D, M = lm.build_layout(src), lm.build_layout(dst), lm.build_layout(smem)
    d = lm.TVPlan(S, M, D, lm.Layout.parse(tl), None, eb).describe()
    assert d["load"]["tuned"] is False and d["load"]["thr"] == tl
    assert d["store"]["tuned"] is True
    S3 = lm.Layout.parse("((4,4,4),8):((1,4,16),64)")
    D3 = lm.Layout.parse("((4,4,4),8):((16,4,1),64)")
    M3 = lm.Layout.parse("(4,4,4):(1,4,16)")
    T3 = lm.Layout.parse("(4,4,4):(1,4,16)")
    lm.TVPlan(S3, M3, D3, T3, T3, 4)          # plans with given layouts
    for tl, ts in ((None, T3), (T3, None)):
        with pytest.raises(lm.LayoutMoveError) as e:
            lm.TVPlan(S3, M3, D3, tl, ts, 4)
        assert e.value.status == -1
