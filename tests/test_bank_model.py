"""The planner's shared-memory bank model (host only).

A STAGED tile passes through shared memory: 16-byte writes from the load
side, then the store side's reads.  The planner simulates both over every
warp of one tile (32 banks of 4 bytes; a 16-byte access is served eight
lanes at a time, an 8-byte one sixteen at a time) and picks the pad and XOR
swizzle with the fewest wavefronts.  These tests pin its figures to closed
forms for the bench workloads:

* the conflict-free minimum is the tile's bytes over 128 on each side;
* with the search on, both transposes are conflict-free;
* with the plain image (LM_SMEM_SEARCH=0: no pad, no swizzle) a transpose's
  eight lanes of a 16-byte phase read eight rows whose pitch is a multiple
  of 128 bytes, so every phase lands on one group of four banks: 8x;
* the fp64 TV gather reads a 2x-conflicted pattern that no pad can fix
  (its tile arrives as one contiguous bulk copy): lanes 2k and 2k+1 read
  source offsets 36 elements apart, whose banks overlap those of lanes
  2k+8 and 2k+9.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

from workloads import WORKLOADS, ELEM_BYTES

lm = pytest.importorskip("layout_driven_movement_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def staged_piece(name):
    w = WORKLOADS[name]
    d = lm.Plan(lm.build_layout(w.src), lm.build_layout(w.dst),
                ELEM_BYTES[w.dtype]).describe()
    (p,) = [p for p in d["pieces"] if p["path"] == "STAGED"]
    return p


def test_ideal_is_tile_bytes_over_128():
    for name in ["C2", "C4", "C5a"]:
        p = staged_piece(name)
        eb = ELEM_BYTES[WORKLOADS[name].dtype]
        assert p["bank_read_wavefronts_ideal"] == p["tile_elems"] * eb // 128
        write_ideal = p["bank_wavefronts_ideal"] - p["bank_read_wavefronts_ideal"]
        assert write_ideal == p["load_chunks"] * 16 // 128
        assert p["bank_wavefronts"] >= p["bank_wavefronts_ideal"]
        assert p["bank_read_wavefronts"] >= p["bank_read_wavefronts_ideal"]


def test_search_makes_transposes_conflict_free():
    for name in ["C2", "C5a"]:
        p = staged_piece(name)
        assert p["store"] == "transpose"
        assert p["bank_wavefronts"] == p["bank_wavefronts_ideal"], name


def test_tensor_map_images_read_conflict_free():
    """With tensor-map loads (LM_TMA=1) the tile lands densely (no pad, no
    swizzle); the micro-tiles then run along the row, 8 lanes reading 8
    consecutive chunks, which the model finds conflict-free."""
    code = (
        "import json, layout_driven_movement_gb300 as lm\n"
        "from workloads import WORKLOADS, ELEM_BYTES\n"
        "out = {}\n"
        "for n in ['C2', 'C5a']:\n"
        "    w = WORKLOADS[n]\n"
        "    d = lm.Plan(lm.build_layout(w.src), lm.build_layout(w.dst),\n"
        "                ELEM_BYTES[w.dtype]).describe()\n"
        "    out[n] = [p for p in d['pieces'] if p['path'] == 'STAGED'][0]\n"
        "print(json.dumps(out))\n")
    env = dict(os.environ, LM_TMA="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for name, p in got.items():
        assert p["tma"] and p["bulk"], name
        # fp32 (4 rows per micro-tile): 128-byte boxes in the hardware's
        # 128-byte swizzle; fp16 (8 rows): dense rows, micro-tiles along a
        want = [3, 4, 3] if name == "C2" else [0, 0, 0]
        assert p["tma_swizzle"] == (name == "C2"), name
        assert p["smem_swizzle"] == want, name
        assert p["bank_read_wavefronts"] == p["bank_read_wavefronts_ideal"]
    # by default the transposes keep the per-thread cp.async loads
    for name in ["C2", "C5a"]:
        p = staged_piece(name)
        assert not p["tma"] and not p["bulk"], name


def test_gather_of_tv_tiles_is_two_way():
    p = staged_piece("C4")
    assert p["store"] == "gather" and p["bulk"]
    assert p["bank_read_wavefronts"] == 2 * p["bank_read_wavefronts_ideal"]


def test_plain_image_predicts_eightfold_transpose_conflicts():
    code = (
        "import json, layout_driven_movement_gb300 as lm\n"
        "from workloads import WORKLOADS, ELEM_BYTES\n"
        "out = {}\n"
        "for n in ['C2', 'C5a']:\n"
        "    w = WORKLOADS[n]\n"
        "    d = lm.Plan(lm.build_layout(w.src), lm.build_layout(w.dst),\n"
        "                ELEM_BYTES[w.dtype]).describe()\n"
        "    out[n] = [p for p in d['pieces'] if p['path'] == 'STAGED'][0]\n"
        "print(json.dumps(out))\n")
    env = dict(os.environ, LM_SMEM_SEARCH="0", LM_TMA="0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for name, p in got.items():
        assert p["smem_swizzle"] == [0, 0, 0]
        assert p["bank_read_wavefronts"] == 8 * p["bank_read_wavefronts_ideal"], name
        # the 16-byte tile writes stay row-contiguous, so conflict-free
        assert (p["bank_wavefronts"] - p["bank_read_wavefronts"]
                == p["bank_wavefronts_ideal"] - p["bank_read_wavefronts_ideal"])


def test_smem_wavefronts_matches_oracle():
    from oracle import layout_oracle as lo
    rng = np.random.default_rng(7)
    cases = [("32:8", 4, 4), ("(32,8):(8,1)", 4, 4), ("(32,8):(9,1)", 4, 4),
             ("(8,32):(1,8)", 4, 16), ("(4,8,8):(2,64,8)", 8, 8),
             ("(2,16,8):(1,64,2)", 2, 2), ("100:3", 1, 1), ("77:2", 8, 16)]
    for _ in range(40):
        n = int(rng.integers(1, 4))
        shape = [int(rng.integers(1, 9)) for _ in range(n)]
        stride = [int(rng.integers(0, 70)) for _ in range(n)]
        text = "(" + ",".join(map(str, shape)) + "):(" + ",".join(
            map(str, stride)) + ")"
        eb = int(rng.choice([1, 2, 4, 8]))
        cases.append((text, eb, eb))
    for text, eb, ab in cases:
        L = lm.Layout.parse(text)
        O = lo.parse(text)
        off = O.at(np.arange(O.size)) * eb
        if (off % ab).any():
            with pytest.raises(lm.LayoutMoveError):
                L.smem_wavefronts(eb, ab)
            continue
        assert L.smem_wavefronts(eb, ab) == lo.smem_wavefronts(off, ab), text
    S = lm.Layout.parse("(32,8):(8,1)").swizzle(3, 0, 3)
    off = lo.swizzle(lo.parse("(32,8):(8,1)").at(np.arange(256)), 3, 0, 3) * 4
    assert S.smem_wavefronts(4) == lo.smem_wavefronts(off, 4)


def test_smem_wavefronts_rejects():
    L = lm.Layout.parse("32:1")
    for eb, ab in [(3, 4), (4, 32), (0, 4), (4, 0)]:
        with pytest.raises(lm.LayoutMoveError):
            L.smem_wavefronts(eb, ab)
    with pytest.raises(lm.LayoutMoveError):
        lm.Layout.parse("32:1").smem_wavefronts(4, 8)  # 4-byte aligned only
    with pytest.raises(lm.LayoutMoveError):
        lm.Layout.parse("(4096,4097):(1,4096)").smem_wavefronts(4)  # > 2^24


def _tune_by_oracle(threads, k_row, rows, ld, eb, vec, smem_text=None,
                    smem_swz=None):
    """The search lm_stripmined_tune documents, recomputed from the oracle's
    stripmined map, its layout evaluation and its bank model."""
    from oracle import layout_oracle as lo
    R = k_row // vec
    sm = None
    if smem_text:
        sm = lo.parse(smem_text)
        if smem_swz:
            sm = lo.Swizzled(*smem_swz, sm)
    best = None
    P = 1
    while P <= R and P <= threads:
        S = 1
        while S <= rows and P * S <= threads:
            t = np.arange(threads)
            off = lo.stripmined_offset(t, R, P, S)   # in vectors
            row, vcol = off // R, off % R
            if (row < rows).all():
                col = vcol * vec
                g = (row * ld + col) * eb // 128
                s_off = (sm.at(row + rows * col) if sm is not None
                         else row * k_row + col)
                seg = wf = 0
                for w0 in range(0, threads, 32):
                    seg += len(set(g[w0:w0 + 32].tolist()))
                    wf += lo.smem_wavefronts(s_off[w0:w0 + 32] * eb,
                                             vec * eb)[0]
                key = (seg, wf, -P, -S)
                if best is None or key < best[0]:
                    best = (key, P, S, seg, wf)
            S *= 2
        P *= 2
    return {"pitch": best[1], "strips": best[2], "segments": best[3],
            "wavefronts": best[4]}


@pytest.mark.parametrize("args", [
    (128, 64, 64, 64, 4, 4, None, None),
    (128, 32, 64, 32, 4, 4, "(64,32):(32,1)", None),
    (32, 16, 16, 16, 4, 1, None, None),
    (256, 64, 64, 4096, 4, 1, "(64,64):(64,1)", None),
    (256, 64, 64, 4096, 4, 1, "(64,64):(1,64)", None),
    (256, 64, 64, 4096, 4, 1, "(64,64):(1,64)", (5, 0, 6)),
    (128, 64, 32, 64, 2, 8, "(32,64):(64,1)", (3, 3, 6)),
    (96, 24, 96, 100, 8, 2, None, None),
    (64, 128, 8, 128, 1, 16, None, None),
])
def test_stripmined_tune_matches_oracle_search(args):
    threads, k_row, rows, ld, eb, vec, smem_text, swz = args
    smem = None
    if smem_text:
        smem = lm.Layout.parse(smem_text)
        if swz:
            smem = smem.swizzle(*swz)
    got = lm.stripmined_tune(threads, k_row, rows, eb, vec, ld=ld, smem=smem)
    assert got == _tune_by_oracle(threads, k_row, rows, ld, eb, vec,
                                  smem_text, swz)


def test_stripmined_tune_follows_the_article_in_closed_form():
    """fp32 with 16-byte vectors over 64-float rows: Pitch covers a row
    (16 vectors, 256 bytes), Strips = threads / Pitch, every access at the
    conflict-free and fully coalesced minimum ([TM] §4.2: Pitch from the
    vector width, Strips from threads over Pitch)."""
    got = lm.stripmined_tune(128, 64, 64, 4, 4)
    assert got == {"pitch": 16, "strips": 8, "segments": 16,
                   "wavefronts": 16}
    # a shared tile stored column-major: the same coalesced choice, and the
    # bank model charges the column-wise shared writes
    col = lm.stripmined_tune(256, 64, 64, 4, 1, ld=4096,
                             smem=lm.Layout.parse("(64,64):(1,64)"))
    assert col["pitch"] == 64 and col["segments"] == 8
    assert col["wavefronts"] == 8 * 32
    xor = lm.stripmined_tune(256, 64, 64, 4, 1, ld=4096,
                             smem=lm.Layout.parse("(64,64):(1,64)").swizzle(
                                 5, 0, 6))
    assert xor["pitch"] == 64 and xor["wavefronts"] == 8


def test_stripmined_tune_rejects():
    for a in [(0, 64, 64, 4, 4), (2048, 64, 64, 4, 4), (128, 63, 64, 4, 4),
              (128, 64, 64, 4, 8), (128, 64, 64, 3, 1)]:
        with pytest.raises(lm.LayoutMoveError):
            lm.stripmined_tune(*a)
    with pytest.raises(lm.LayoutMoveError):
        lm.stripmined_tune(128, 64, 64, 4, 4, ld=32)
    with pytest.raises(lm.LayoutMoveError):
        lm.stripmined_tune(128, 64, 64, 4, 4,
                           smem=lm.Layout.parse("(32,64):(64,1)"))
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.stripmined_tune(1024, 64, 2, 4, 4)   # no pass fits 2 rows
    assert e.value.status == -3
