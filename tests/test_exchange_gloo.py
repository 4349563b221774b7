"""Sharded relayouts with one all-to-all exchange (CPU).

lm_plan_exchange gives each rank the boxes it sends and receives.  Here
every rank cuts its shard of the source out of a seeded global source,
packs each outgoing box by the plan's description (numpy, the boxes'
modes and bases), exchanges the buffers with a real torch.distributed
all_to_all_single over gloo, unpacks them into its destination shard, and
checks the shard against the oracle's copy of the whole tensor: every
slot the rank owns holds the oracle's value, every other slot of its
buffer is untouched.  The device pack/unpack kernels are the layout copies
of the other tests; tests/test_gpu_exchange.py runs them for all ranks on
one GPU.
"""

import socket

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import WORKLOADS, seeded_bytes

lm = pytest.importorskip("layout_driven_movement_gb300")

FILL = 0xA5

CASES = [
    # row-sharded fp32 transpose: rows in, transposed rows out
    ("transpose_f32", ("layout", (96, 80), (80, 1)),
     ("layout", (96, 80), (1, 96)), 4),
    # NHWC -> NCHW sharded by N on both sides: no traffic between ranks
    ("nhwc_nchw_f16", ("layout", (6, 16, 5, 7), (560, 1, 112, 16)),
     ("layout", (6, 16, 5, 7), (560, 35, 7, 1)), 2),
    # batched padded TV gather, batch sharded on both sides
    ("tv_gather_f64", ("concat", WORKLOADS["C4"].src[1], ("layout", 37, 72)),
     ("layout", (((4, 8), 2), 37), (((1, 4), 32), 64)), 8),
    # 2-head interleave: heads in, positions out
    ("interleave_f16", ("layout", (2, 600), (600, 1)),
     ("layout", (2, 600), (1, 2)), 2),
    # a 3-D permutation whose slowest modes differ on the two sides
    ("permute_u8", ("layout", (12, 10, 9), (90, 9, 1)),
     ("layout", (12, 10, 9), (1, 108, 12)), 1),
]

# Cases whose largest-stride mode on one side is short: the most ranks that
# mode can be split over (more are refused with LM_E_INVALID).
MAX_WORLD = {"interleave_f16": 2}


def refused(name, S, D, eb, world):
    """True (after checking the refusal) when `world` ranks exceed what the
    case's slowest mode allows."""
    if world <= MAX_WORLD.get(name, world):
        return False
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.Exchange(S, D, eb, 0, world)
    assert e.value.status == -1
    return True


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def box_offsets(box, side):
    """Offsets of a box's elements (colex over its modes) on one side."""
    n = int(np.prod([m[0] for m in box])) if box else 1
    i = np.arange(n)
    off = np.zeros(n, dtype=np.int64)
    for e, s, d in box:
        off += (i % e) * (d if side == "d" else s)
        i //= e
    return off


def owned_dst(desc, rank):
    """Global destination offsets rank owns: its range of the out mode."""
    ms = [list(m) for m in desc["modes"]]
    k = desc["out_mode"]
    e = ms[k][0]
    lo_, hi = e * rank // desc["world"], e * (rank + 1) // desc["world"]
    ms[k][0] = hi - lo_
    return lo_ * ms[k][2] + box_offsets(ms, "d")


def global_problem(src, dst, eb):
    S, D = lm.build_layout(src), lm.build_layout(dst)
    inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 17)
    want = np.full(D.cosize * eb, FILL, np.uint8)
    lo.copy(lo.build(src), lo.build(dst), inp, want, eb)
    return S, D, inp, want


def pack(desc, src_local, peer, eb):
    b = desc["send"][peer]
    if b["count"] == 0:
        return np.zeros(0, np.uint8)
    idx = b["base"] + box_offsets(b["box"], "s")
    return src_local.reshape(-1, eb)[idx].reshape(-1)


def unpack(desc, buf, dst_local, peer, eb):
    b = desc["recv"][peer]
    if b["count"] == 0:
        return
    idx = b["base"] + box_offsets(b["box"], "d")
    dst_local.reshape(-1, eb)[idx] = buf.reshape(-1, eb)


def check_rank(desc, dst_local, want, eb, rank):
    own = owned_dst(desc, rank) - desc["dst_origin"]
    got = dst_local.reshape(-1, eb)
    exp = want.reshape(-1, eb)[own + desc["dst_origin"]]
    assert (got[own] == exp).all()
    mask = np.ones(len(got), bool)
    mask[own] = False
    assert (got[mask] == FILL).all()


@pytest.mark.parametrize("world", [1, 2, 3])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_boxes_partition_and_move_everything(case, world):
    """All ranks in one process: the send and receive descriptions agree,
    every logical index moves exactly once, the shards come out right."""
    name, src, dst, eb = case
    S, D, inp, want = global_problem(src, dst, eb)
    if refused(name, S, D, eb, world):
        return
    descs = [lm.Exchange(S, D, eb, r, world).describe() for r in range(world)]
    _assert_disjoint_shards(descs)
    total = sum(b["count"] for d in descs for b in d["send"])
    assert total == S.size
    for p in range(world):
        for q in range(world):
            assert descs[p]["send"][q]["count"] == descs[q]["recv"][p]["count"]
            assert descs[p]["send"][q]["box"] == descs[q]["recv"][p]["box"]
    src_local = [inp[d["src_origin"] * eb:(d["src_origin"] + d["src_local"]) * eb]
                 for d in descs]
    sent = [[pack(descs[p], src_local[p], q, eb) for q in range(world)]
            for p in range(world)]
    for q in range(world):
        dl = np.full(descs[q]["dst_local"] * eb, FILL, np.uint8)
        for p in range(world):
            unpack(descs[q], sent[p][q], dl, p, eb)
        check_rank(descs[q], dl, want, eb, q)


def test_exchange_rejects():
    S = lm.Layout.parse("(4,8):(8,1)")
    D = lm.Layout.parse("(4,8):(1,4)")
    for args, code in [((S, D, 3, 0, 2), -1), ((S, D, 4, 2, 2), -1),
                       ((S, D, 4, 0, 9), -1),   # no mode with 9 coordinates
                       ((S, lm.Layout.parse("(4,8):(1,4)").swizzle(1, 0, 2),
                         4, 0, 2), -3)]:
        with pytest.raises(lm.LayoutMoveError) as e:
            lm.Exchange(*args)
        assert e.value.status == code


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                                rank=rank, world_size=world)
        lm.lib()
        for name, src, dst, eb in CASES:
            if world > MAX_WORLD.get(name, world):
                continue            # refused; checked in one process
            S, D, inp, want = global_problem(src, dst, eb)
            desc = lm.Exchange(S, D, eb, rank, world).describe()
            o, n = desc["src_origin"], desc["src_local"]
            src_local = inp[o * eb:(o + n) * eb]
            send = np.concatenate([pack(desc, src_local, p, eb)
                                   for p in range(world)])
            sc = [b["count"] * eb for b in desc["send"]]
            rc = [b["count"] * eb for b in desc["recv"]]
            recv = torch.empty(sum(rc), dtype=torch.uint8)
            dist.all_to_all_single(recv, torch.from_numpy(send), rc, sc)
            dl = np.full(desc["dst_local"] * eb, FILL, np.uint8)
            off = 0
            for p in range(world):
                unpack(desc, recv[off:off + rc[p]].numpy(), dl, p, eb)
                off += rc[p]
            check_rank(desc, dl, want, eb, rank)
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as exc:  # reported to the parent
        q.put((rank, repr(exc)))


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_exchange_over_gloo(world):
    import torch.multiprocessing as mp
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q))
             for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
    assert results == {r: "ok" for r in range(world)}, results


def _random_permutation_case(rng):
    """A random compact permutation of a 2- or 3-mode tensor."""
    n = int(rng.integers(2, 4))
    shape = [int(rng.integers(2, 9)) for _ in range(n)]

    def compact(order):
        stride, w = [0] * n, 1
        for k in order:
            stride[k] = w
            w *= shape[k]
        return tuple(stride)

    src = ("layout", tuple(shape), compact(rng.permutation(n)))
    dst = ("layout", tuple(shape), compact(rng.permutation(n)))
    return src, dst, int(rng.choice([1, 2, 4, 8]))


def test_random_exchanges_move_everything():
    """Random permutations over 2-4 ranks: every plan the library accepts
    partitions the copy and the emulated exchange gives the oracle's
    shards."""
    rng = np.random.default_rng(99)
    done = 0
    for _ in range(60):
        src, dst, eb = _random_permutation_case(rng)
        world = int(rng.integers(2, 5))
        S, D, inp, want = global_problem(src, dst, eb)
        try:
            descs = [lm.Exchange(S, D, eb, r, world).describe()
                     for r in range(world)]
        except lm.LayoutMoveError as e:
            assert e.status == -1      # no mode with `world` coordinates
            continue
        assert sum(b["count"] for d in descs for b in d["send"]) == S.size
        _assert_disjoint_shards(descs)
        src_local = [inp[d["src_origin"] * eb:
                         (d["src_origin"] + d["src_local"]) * eb]
                     for d in descs]
        sent = [[pack(descs[p], src_local[p], q, eb) for q in range(world)]
                for p in range(world)]
        for q in range(world):
            dl = np.full(descs[q]["dst_local"] * eb, FILL, np.uint8)
            for p in range(world):
                unpack(descs[q], sent[p][q], dl, p, eb)
            check_rank(descs[q], dl, want, eb, q)
        done += 1
    assert done >= 30


def _assert_disjoint_shards(descs):
    """The ranks' source shards, and their destination shards, are
    disjoint ranges of the global buffers."""
    for org, n in (("src_origin", "src_local"), ("dst_origin", "dst_local")):
        spans = sorted((d[org], d[org] + d[n]) for d in descs)
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0, (org, spans)


@pytest.mark.parametrize("world", [3, 4, 8])
def test_short_slowest_mode_is_rejected(world):
    """The 2-head interleave sharded over more ranks than heads: the source's
    largest-stride mode (heads, 2 coordinates) cannot be split `world` ways,
    and sharding a faster mode instead would give overlapping source shards,
    so the plan is refused."""
    S = lm.Layout.parse("(2,1024):(1024,1)")
    D = lm.Layout.parse("(2,1024):(1,2)")
    for r in range(world):
        with pytest.raises(lm.LayoutMoveError) as ei:
            lm.Exchange(S, D, 2, r, world)
        assert ei.value.status == -1
    # two ranks split the heads, and the shards are disjoint
    descs = [lm.Exchange(S, D, 2, r, 2).describe() for r in range(2)]
    _assert_disjoint_shards(descs)
    assert sum(d["src_local"] for d in descs) == 2048


def test_short_destination_mode_is_rejected():
    """The same on the destination side: the interleave's reverse, whose
    destination's largest-stride mode has 2 coordinates."""
    S = lm.Layout.parse("(2,1024):(1,2)")
    D = lm.Layout.parse("(2,1024):(1024,1)")
    with pytest.raises(lm.LayoutMoveError) as ei:
        lm.Exchange(S, D, 2, 0, 4)
    assert ei.value.status == -1
