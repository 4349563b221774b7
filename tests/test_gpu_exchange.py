"""GPU parity of the sharded relayout's pack and unpack (lm_exchange_*).

All ranks of an exchange run one after another on one device: each packs
its boxes from its source shard with the library's copy kernels, the
"all-to-all" is a device-to-device copy of each box buffer to its
receiver (no collective, no rank waits on another), and each rank unpacks
what it received into its destination shard.  Every shard is compared
byte for byte with the oracle's copy of the whole tensor.
"""

import pytest

from test_exchange_gloo import (CASES, FILL, check_rank, global_problem,
                                refused)
from workloads import WORKLOADS

torch = pytest.importorskip("torch")
lm = pytest.importorskip("layout_driven_movement_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def run_exchange(src, dst, eb, world, name=""):
    S, D, inp, want = global_problem(src, dst, eb)
    if refused(name, S, D, eb, world):
        return
    xs = [lm.Exchange(S, D, eb, r, world) for r in range(world)]
    descs = [x.describe() for x in xs]
    g_src = torch.from_numpy(inp).cuda()
    sends = []
    for r, (x, d) in enumerate(zip(xs, descs)):
        o, n = d["src_origin"], d["src_local"]
        local = g_src[o * eb:(o + n) * eb].clone()
        bufs = []
        for q in range(world):
            c = d["send"][q]["count"]
            b = torch.full((c * eb,), 0x5C, dtype=torch.uint8, device="cuda")
            if c:
                x.pack(q, local, b)
            bufs.append(b)
        sends.append(bufs)
    for q, (x, d) in enumerate(zip(xs, descs)):
        dl = torch.full((d["dst_local"] * eb,), FILL, dtype=torch.uint8,
                        device="cuda")
        for p in range(world):
            recv = sends[p][q].clone()   # the exchange, on one device
            if recv.numel():
                x.unpack(p, recv, dl)
        torch.cuda.synchronize()
        assert lm.device_status() == 0
        check_rank(d, dl.cpu().numpy(), want, eb, q)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_exchange_on_one_device(case, world):
    name, src, dst, eb = case
    run_exchange(src, dst, eb, world, name)


def test_exchange_row_sharded_transpose_large():
    """The 4096x4096 fp32 transpose, rows sharded four ways on both sides:
    each rank's boxes are 1024x1024 transposes through the STAGED path."""
    w = WORKLOADS["C2"]
    # rows of a row-major source in, rows of the row-major result out
    src = ("layout", (4096, 4096), (4096, 1))
    dst = ("layout", (4096, 4096), (1, 4096))
    x = lm.Exchange(lm.build_layout(src), lm.build_layout(dst), 4, 0, 4)
    counts = {b["count"] for b in x.describe()["send"]}
    assert counts == {1024 * 1024}
    run_exchange(src, dst, w.elem_bytes, 4)


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_pack_all_and_unpack_all(case, world):
    """One buffer per rank for all peers: pack_all writes exactly the
    per-peer packs one after another (one copy when the boxes are equal),
    and unpack_all of the exchanged buffers gives the oracle's shards."""
    _, src, dst, eb = case
    S, D, inp, want = global_problem(src, dst, eb)
    try:
        xs = [lm.Exchange(S, D, eb, r, world) for r in range(world)]
    except lm.LayoutMoveError as e:      # no mode with `world` coordinates
        assert e.status == -1
        return
    descs = [x.describe() for x in xs]
    sizes = [x.sizes() for x in xs]
    g_src = torch.from_numpy(inp).cuda()
    packed = []
    for r, (x, d) in enumerate(zip(xs, descs)):
        o, n = d["src_origin"], d["src_local"]
        local = g_src[o * eb:(o + n) * eb].clone()
        total = sum(sizes[r]["send"]) * eb
        buf = torch.full((total,), 0x5C, dtype=torch.uint8, device="cuda")
        lm.exchange_pack_all(x, local, buf)
        ref = torch.full((total,), 0x5C, dtype=torch.uint8, device="cuda")
        off = 0
        for q in range(world):
            c = sizes[r]["send"][q] * eb
            if c:
                x.pack(q, local, ref[off:off + c])
            off += c
        torch.cuda.synchronize()
        assert torch.equal(buf, ref)
        packed.append(buf)
    for q, (x, d) in enumerate(zip(xs, descs)):
        parts, off = [], []
        for p in range(world):
            start = sum(sizes[p]["send"][:q]) * eb
            parts.append(packed[p][start:start + sizes[p]["send"][q] * eb])
        recv = torch.cat(parts)
        dl = torch.full((d["dst_local"] * eb,), FILL, dtype=torch.uint8,
                        device="cuda")
        lm.exchange_unpack_all(x, recv, dl)
        torch.cuda.synchronize()
        assert lm.device_status() == 0
        check_rank(d, dl.cpu().numpy(), want, eb, q)


def test_exchange_copy_single_rank_nccl():
    """exchange_copy end to end -- pack_all, torch.distributed's
    all_to_all_single, unpack_all -- in a one-rank NCCL group on this GPU
    (the whole copy is the rank's own box)."""
    import os
    import socket
    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("NCCL not available")
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}",
                            rank=0, world_size=1)
    try:
        _, src, dst, eb = CASES[0]
        S, D, inp, want = global_problem(src, dst, eb)
        x = lm.Exchange(S, D, eb, 0, 1)
        d = x.describe()
        local = torch.from_numpy(inp).cuda()[:d["src_local"] * eb].clone()
        out = torch.full((d["dst_local"] * eb,), FILL, dtype=torch.uint8,
                         device="cuda")
        lm.exchange_copy(x, local, out)
        torch.cuda.synchronize()
        assert lm.device_status() == 0
        check_rank(d, out.cpu().numpy(), want, eb, 0)
    finally:
        dist.destroy_process_group()
