"""lm_layout_copy_host_static: the host-buffer copy without device staging
buffers from the caller.

Some callers cannot allocate device memory -- a library inside a program
whose memory manager owns the device's memory, or a path that cannot afford
cudaMalloc/cudaFree -- so the library offers this variant, which stages
through its own fixed __device__ area.  Here it is called through the C ABI
twice in a row on one stream, each time with other host bytes, and every
result must equal, byte for byte, what lm_layout_copy_host gives for the
same inputs through caller-allocated staging buffers (copies move raw bytes:
the tolerance is zero).  A copy too large for the area is refused before
anything moves.

This file is collected last (its name sorts after every other test file) and
builds everything it needs itself, so it runs the same alone in a fresh
process and after the rest of the suite.
"""

import numpy as np
import pytest

from oracle import layout_oracle as lo
from workloads import WORKLOADS, seeded_bytes

torch = pytest.importorskip("torch")
lm = pytest.importorskip("layout_driven_movement_gb300")

pytestmark = pytest.mark.gpu

CASES = [
    # padded 8x8 fp64 tiles gathered into thread-value order, 8192 tiles:
    # the bulk-copy STAGED kernel
    ("padded_tv_gather_f64",
     ("concat", WORKLOADS["C4"].src[1], ("layout", 8192, 72)),
     ("layout", (((4, 8), 2), 8192), (((1, 4), 32), 64)), 8),
    # 1024x1024 fp32 transpose, 4 MiB each way: the shared-memory transpose
    ("transpose_f32", ("layout", (1024, 1024), (1, 1024)),
     ("layout", (1024, 1024), (1024, 1)), 4),
    # a destination with slots outside its image: they must come back with
    # the host's own bytes, whatever the area held from the call before
    ("gap_dst_f16", ("layout", (96, 80), (80, 1)),
     ("layout", (96, 80), (1, 100)), 2),
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from layout_driven_movement_gb300 import _build
    _build.build()
    lm.lib()


def _with_caller_staging(plan, S, D, eb, inp, host_dst, stream):
    """lm_layout_copy_host through device buffers this test allocates."""
    hs = torch.from_numpy(inp).pin_memory()
    hd = torch.from_numpy(host_dst.copy()).pin_memory()
    sd = torch.empty(S.cosize * eb, dtype=torch.uint8, device="cuda")
    dd = torch.empty(D.cosize * eb, dtype=torch.uint8, device="cuda")
    lm.layout_copy_host(plan, hs, hd, sd, dd, stream)
    stream.synchronize()
    return hd.numpy().copy()


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_static_staging_matches_caller_staging_twice(case):
    name, s, d, eb = case
    S, D = lm.build_layout(s), lm.build_layout(d)
    plan = lm.Plan(S, D, eb)
    OS, OD = lo.build(s), lo.build(d)
    st = torch.cuda.Stream()
    inputs = []
    for k in range(2):
        inp = seeded_bytes("bytes", "uint8", S.cosize * eb, 500 + k)
        host_dst = np.full(D.cosize * eb, 0x3C + k, dtype=np.uint8)
        inputs.append((inp, host_dst))
    # two calls in a row on one stream, nothing synchronised between them
    pinned = [(torch.from_numpy(inp).pin_memory(),
               torch.from_numpy(host_dst.copy()).pin_memory())
              for inp, host_dst in inputs]
    for hs, hd in pinned:
        lm.layout_copy_host_static(plan, hs, hd, st)
    st.synchronize()
    assert lm.device_status() == 0
    for (inp, host_dst), (_, hd) in zip(inputs, pinned):
        want = _with_caller_staging(plan, S, D, eb, inp, host_dst, st)
        got = hd.numpy()
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"{name}: {bad.size} bytes differ"
        # and both are the oracle's copy
        oracle = host_dst.copy()
        lo.copy(OS, OD, inp, oracle, eb)
        assert np.array_equal(got, oracle), name


def test_too_large_for_the_area_is_refused():
    """A copy whose source and destination together exceed the area is
    refused with LM_E_CAPACITY; the host destination is left as it was."""
    n = lm.HOST_COPY_STATIC_BYTES // 8          # fp64 elements of half the area
    S = lm.Layout.parse(f"({n // 1024 + 1},1024):(1024,1)")
    D = lm.Layout.parse(f"({n // 1024 + 1},1024):(1,{n // 1024 + 1})")
    plan = lm.Plan(S, D, 8)
    hs = torch.zeros(S.cosize * 8, dtype=torch.uint8).pin_memory()
    hd = torch.full((D.cosize * 8,), 0x5A, dtype=torch.uint8).pin_memory()
    with pytest.raises(lm.LayoutMoveError) as e:
        lm.layout_copy_host_static(plan, hs, hd)
    assert e.value.status == -6
    torch.cuda.synchronize()
    assert bool((hd == 0x5A).all())
