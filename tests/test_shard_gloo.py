"""Sharded copies across ranks (CPU only).

Every logical index of a copy is independent, so a copy splits across
devices with no exchange: shard r of w (lm_plan_copy_shard) plans one range
of the joint mode with the largest destination stride.  These tests check,
on the host, that the shards of all ranks partition the copy exactly: the
union of their (src offset, dst offset) pairs is the oracle's set
{(src(i), dst(i))}, with no pair twice.  The multi-process test runs two
ranks over torch.distributed's gloo backend, gathers each rank's pairs and
checks them on rank 0.
"""

import os
import socket

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import WORKLOADS

lm = pytest.importorskip("layout_driven_movement_gb300")

CASES = [
    (("layout", (512, 384), (1, 512)), ("layout", (512, 384), (384, 1)), 4),
    (("concat", WORKLOADS["C4"].src[1], ("layout", 37, 72)),
     ("layout", (((4, 8), 2), 37), (((1, 4), 32), 64)), 8),
    (("layout", (3, 40, 7, 9), (2520, 1, 360, 40)),
     ("layout", (3, 40, 7, 9), (2520, 63, 9, 1)), 2),
    (("layout", (2, 300, 24), (7200, 24, 1)),
     ("layout", (2, 300, 24), (1, 48, 2)), 2),
    (("layout", (6, 5), (1, 6)), ("layout", (5, 6), (6, 1)), 4),  # no joint
    (WORKLOADS["C1"].src, WORKLOADS["C1"].dst, 4),
]


def shard_pairs(src_spec, dst_spec, eb, rank, world):
    """(src, dst) offset pairs of one shard, expanded from its plan."""
    S, D = lm.build_layout(src_spec), lm.build_layout(dst_spec)
    desc = lm.Plan(S, D, eb, rank=rank, world=world).describe()
    OS, OD = lo.build(src_spec), lo.build(dst_spec)
    if not desc["joint"]:
        out = []
        for pc in desc["pieces"]:
            i = np.arange(pc["index_begin"], pc["index_begin"] + pc["index_count"])
            out.append(np.stack([OS.at(i), OD.at(i)], 1))
        return np.concatenate(out) if out else np.zeros((0, 2), np.int64)
    src, dst = [], []
    for pc in desc["pieces"]:
        n = int(np.prod([m[0] for m in pc["modes"]])) if pc["modes"] else 1
        i = np.arange(n)
        so = np.full(n, pc["s_base"], dtype=np.int64)
        do = np.full(n, pc["d_base"], dtype=np.int64)
        for e, s, d in pc["modes"]:
            so += (i % e) * s
            do += (i % e) * d
            i = i // e
        src.append(so)
        dst.append(do)
    so = np.concatenate(src) if src else np.zeros(0, np.int64)
    do = np.concatenate(dst) if dst else np.zeros(0, np.int64)
    if isinstance(OS, lo.Swizzled):
        so = lo.swizzle(so, OS.b, OS.m, OS.s)
    if isinstance(OD, lo.Swizzled):
        do = lo.swizzle(do, OD.b, OD.m, OD.s)
    return np.stack([so, do], 1)


def check_partition(parts, src_spec, dst_spec):
    OS, OD = lo.build(src_spec), lo.build(dst_spec)
    i = np.arange(OS.size)
    want = np.stack([OS.at(i), OD.at(i)], 1)
    got = np.concatenate(parts)
    assert got.shape == want.shape
    w = want[np.lexsort((want[:, 0], want[:, 1]))]
    g = got[np.lexsort((got[:, 0], got[:, 1]))]
    assert (w == g).all()
    sizes = [len(p) for p in parts]
    return sizes


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_shards_partition_the_copy(world):
    for src, dst, eb in CASES:
        parts = [shard_pairs(src, dst, eb, r, world) for r in range(world)]
        sizes = check_partition(parts, src, dst)
        if world > 1 and lo.build(src).size >= 1000 * world:
            assert max(sizes) <= 2 * min(sizes) + 64, sizes


def test_shard_rejects_bad_rank():
    S = lm.Layout.parse("(8,8):(1,8)")
    D = lm.Layout.parse("(8,8):(8,1)")
    for rank, world in [(2, 2), (-1, 2), (0, 0)]:
        with pytest.raises(lm.LayoutMoveError) as e:
            lm.Plan(S, D, 4, rank=rank, world=world)
        assert e.value.status == -1


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                rank=rank, world_size=world)
        lm.lib()
        mine = [shard_pairs(s, d, eb, rank, world) for s, d, eb in CASES]
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            for c, (s, d, _) in enumerate(CASES):
                check_partition([gathered[r][c] for r in range(world)], s, d)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as exc:  # reported to the parent
        q.put((rank, repr(exc)))


def test_two_ranks_over_gloo():
    import torch.multiprocessing as mp
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert results == {0: "ok", 1: "ok"}, results


def test_shard_ranges_and_ownership():
    """A shard's described source and destination ranges hold every offset
    its pieces reach; where the shards own their destination ranges, those
    ranges are disjoint and tile [0, cosize)."""
    from workloads import WORKLOADS as W
    for name in ["C2", "C3", "C4", "C5a", "C5b"]:
        w = W[name]
        S, D = lm.build_layout(w.src), lm.build_layout(w.dst)
        descs = [lm.Plan(S, D, w.elem_bytes, rank=r, world=4).describe()
                 for r in range(4)]
        for r, d in enumerate(descs):
            pairs = shard_pairs(w.src, w.dst, w.elem_bytes, r, 4) \
                if name == "C2" else None
            if pairs is not None and len(pairs):
                assert d["src_range"][0] <= pairs[:, 0].min()
                assert pairs[:, 0].max() < d["src_range"][1]
                assert d["dst_range"][0] <= pairs[:, 1].min()
                assert pairs[:, 1].max() < d["dst_range"][1]
        if all(d["dst_own"] for d in descs):
            rng = sorted(tuple(d["dst_range"]) for d in descs)
            assert rng[0][0] == 0 and rng[-1][1] == D.cosize
            for a, b in zip(rng, rng[1:]):
                assert a[1] == b[0]
    whole = lm.Plan(lm.Layout.parse("(8,8):(1,8)"),
                    lm.Layout.parse("(8,8):(8,1)"), 4).describe()
    assert whole["src_range"] == [0, 64] and whole["dst_own"]


def test_random_shard_ranges_hold_their_pairs():
    """Random compact permutations split over 2-5 ranks: each shard's
    described source and destination ranges contain every offset it
    touches, and shards that own their destination ranges have disjoint
    ones."""
    rng = np.random.default_rng(17)
    for _ in range(50):
        n = int(rng.integers(2, 4))
        shape = tuple(int(rng.integers(2, 9)) for _ in range(n))

        def compact(order):
            st, w = [0] * n, 1
            for k in order:
                st[k] = w
                w *= shape[k]
            return tuple(st)

        src = ("layout", shape, compact(rng.permutation(n)))
        dst = ("layout", shape, compact(rng.permutation(n)))
        eb = int(rng.choice([1, 2, 4, 8]))
        world = int(rng.integers(2, 6))
        parts, owned = [], []
        for r in range(world):
            d = lm.Plan(lm.build_layout(src), lm.build_layout(dst), eb,
                        rank=r, world=world).describe()
            pr = shard_pairs(src, dst, eb, r, world)
            parts.append(pr)
            if len(pr):
                assert d["src_range"][0] <= pr[:, 0].min()
                assert pr[:, 0].max() < d["src_range"][1]
                assert d["dst_range"][0] <= pr[:, 1].min()
                assert pr[:, 1].max() < d["dst_range"][1]
            if d["dst_own"]:
                owned.append(tuple(d["dst_range"]))
        check_partition(parts, src, dst)
        owned.sort()
        for a, b in zip(owned, owned[1:]):
            assert a[1] <= b[0], owned
