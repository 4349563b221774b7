"""Host helpers of bench.py (no GPU): CPU lists, the memory-policy call
behind the pinned-buffer placement, the CPU model, and the oracle windows
of the CPU baseline -- the all-cores leg must copy exactly what one thread
copies."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import WORKLOADS, seeded_bytes  # noqa: E402


def test_cpu_lists_round_trip():
    for cpus in ([0], [0, 1, 2, 3], [0, 2, 4], [5, 6, 7, 10, 11, 40]):
        text = bench._ranges(cpus)
        assert bench._cpulist(text) == sorted(cpus)
    assert bench._ranges([3, 1, 2, 9]) == "1-3,9"
    assert bench._cpulist("0-3,5,7-9") == [0, 1, 2, 3, 5, 7, 8, 9]
    assert bench._cpulist("") == []


def test_memory_policy_call_and_reset():
    """Preferring node 0 and going back to the default policy succeed on
    Linux (node 0 always exists); the call is per thread."""
    import threading
    res = {}

    def work():
        res["set"] = bench._set_mempolicy(0)
        res["reset"] = bench._set_mempolicy(None)

    th = threading.Thread(target=work)
    th.start()
    th.join()
    assert res == {"set": True, "reset": True}


def test_cpu_model_is_named():
    assert bench.cpu_model().strip()
    assert bench.host_cores() >= 1


def test_oracle_windows_threads_copy_the_same_bytes():
    """The same window of every workload copied by one thread and by four
    threads over contiguous index ranges gives identical outputs (small
    windows: the fraction is tiny)."""
    outs = []
    for threads in (1, 4):
        bufs = {}
        for name in ("C5b",):
            w = WORKLOADS[name]
            from oracle import layout_oracle as lo
            S, D = lo.build(w.src), lo.build(w.dst)
            bufs[name] = (seeded_bytes(w.values, w.dtype, lo.cosize(S), w.seed),
                          np.zeros(lo.cosize(D) * w.elem_bytes, np.uint8))
        ow = bench.OracleWindows(("C5b",), bufs)
        ow.run(2.0 ** -4, shift=3, threads=threads)
        outs.append({k: v[1].copy() for k, v in bufs.items()})
    for name in outs[0]:
        assert np.array_equal(outs[0][name], outs[1][name]), name
        assert outs[0][name].any()
