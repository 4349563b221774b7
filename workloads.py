"""Workload descriptions and seeded synthetic inputs.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``.  This
module holds data only: layout descriptions as nested tuples, element types
and value distributions, and seeded random buffers.  It computes no offsets,
no compositions and no copies; the oracle and the CUDA path each turn a
description into a layout with their own code.

A description is one of
    ("layout", shape, stride)
    ("swizzle", B, M, S, description)
    ("compose", outer_description, inner_description)
    ("zipped_divide", description, tiler)
    ("concat", description, description, ...)
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = ["Workload", "WORKLOADS", "BENCH_SUITE", "EVAL_C1", "seeded_bytes",
           "ELEM_BYTES"]

ELEM_BYTES = {"int32": 4, "float32": 4, "bfloat16": 2, "float64": 8,
              "float16": 2, "uint8": 1, "int64": 8, "complex128": 16}


@dataclass(frozen=True)
class Workload:
    name: str
    what: str
    dtype: str            # element type of the moved data
    values: str           # value distribution of the seeded input
    seed: int
    src: tuple
    dst: tuple

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.dtype]


_TV = ("layout", ((4, 8), 2), ((16, 1), 8))       # thread-value layout
_PADDED = ("layout", (8, 8), (1, 9))                # 8x8 tile, column pitch 9

WORKLOADS: dict[str, Workload] = {w.name: w for w in [
    Workload(
        "C1", "8x8 int32 tile, column-major -> row-major with the "
        "row*8+(col^row) XOR swizzle", "int32", "uniform_int32", 1001,
        src=("layout", (8, 8), (1, 8)),
        dst=("swizzle", 3, 0, 3, ("layout", (8, 8), (8, 1)))),
    Workload(
        "C2", "fp32 4096x4096 column-major -> row-major", "float32",
        "uniform_pm1", 1002,
        src=("layout", (4096, 4096), (1, 4096)),
        dst=("layout", (4096, 4096), (4096, 1))),
    Workload(
        "C3", "bf16 8192x8192 row-major -> 64x64 tiles, tile-major, "
        "Swizzle<3,4,3> inside each tile", "bfloat16", "normal", 1003,
        src=("zipped_divide", ("layout", (8192, 8192), (8192, 1)), (64, 64)),
        dst=("swizzle", 3, 4, 3,
             ("layout", ((64, 64), (128, 128)), ((64, 1), (524288, 4096))))),
    Workload(
        "C4", "fp64 batch of 2^20 padded 8x8 tiles (8,8):(1,9) gathered "
        "through the thread-value layout into dense TV order", "float64",
        "uniform01", 1004,
        src=("concat", ("compose", _PADDED, _TV),
             ("layout", 1048576, 72)),
        dst=("layout", (((4, 8), 2), 1048576), (((1, 4), 32), 64))),
    Workload(
        "C5a", "fp16 NHWC (N=64,H=56,W=56,C=256) -> NCHW, logical order "
        "(N,C,H,W)", "float16", "normal", 1005,
        src=("layout", (64, 256, 56, 56), (802816, 1, 14336, 256)),
        dst=("layout", (64, 256, 56, 56), (802816, 3136, 56, 1))),
    Workload(
        "C5b", "fp16 2-head (2,16384,128) head-major -> heads interleaved "
        "with stride 2", "float16", "normal", 1006,
        src=("layout", (2, 16384, 128), (2097152, 128, 1)),
        dst=("layout", (2, 16384, 128), (1, 256, 2))),
]}

# The eval-only part of the first workload: the blocked layout whose
# offset table the layout_eval kernel writes.
EVAL_C1 = ("layout", ((4, 2), (2, 4)), ((2, 16), (1, 8)))

# Relayouts timed together as one bench step.
BENCH_SUITE = ("C2", "C3", "C4", "C5a", "C5b")


def seeded_bytes(values: str, dtype: str, n_elems: int, seed: int
                 ) -> np.ndarray:
    """A flat uint8 buffer of n_elems seeded elements of ``dtype``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if values == "uniform_int32":
        arr = rng.integers(-(2 ** 31), 2 ** 31, size=n_elems, dtype=np.int64)
        arr = arr.astype(np.int32)
    elif values == "uniform_pm1":
        arr = rng.random(n_elems, dtype=np.float32) * 2.0 - 1.0
    elif values == "uniform01":
        arr = rng.random(n_elems, dtype=np.float64)
    elif values == "normal":
        arr = rng.standard_normal(n_elems, dtype=np.float32)
    elif values == "bytes":
        arr = rng.integers(0, 256, size=n_elems * ELEM_BYTES[dtype],
                           dtype=np.uint8)
        return arr
    else:
        raise ValueError(f"unknown value distribution {values!r}")
    if dtype == "bfloat16":
        import torch
        return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(
            torch.bfloat16).view(torch.uint8).numpy().copy()
    if dtype == "float16":
        arr = arr.astype(np.float16)
    elif dtype == "float32":
        arr = arr.astype(np.float32)
    elif dtype == "float64":
        arr = arr.astype(np.float64)
    elif dtype == "int32":
        arr = arr.astype(np.int32)
    else:
        raise ValueError(f"no {values!r} values for {dtype!r}")
    return np.ascontiguousarray(arr).view(np.uint8).reshape(-1).copy()
