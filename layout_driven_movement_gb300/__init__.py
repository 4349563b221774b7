"""Python binding of the layoutmove C ABI (``include/layoutmove.h``).

Argument marshalling only: every computation -- the layout algebra, the
copy planning and all device work -- happens in ``liblayoutmove.so``.  There
is no Python or CPU fallback: if the library is missing, every call raises.

Names follow the C ABI without the ``lm_`` prefix.  PyTorch is used only to
pass device pointers and streams (``tensor.data_ptr()``,
``torch.cuda.current_stream().cuda_stream``).
"""

from __future__ import annotations

import ctypes as C
import json
import os
from typing import Iterable, Sequence

__all__ = [
    "LayoutMoveError", "Layout", "Plan", "lib", "layout_copy",
    "layout_copy_host", "layout_copy_host_static", "HOST_COPY_STATIC_BYTES",
    "layout_eval_device", "build_layout", "device_status", "STATUS",
    "TVPlan", "tv_copy", "stripmined_tune", "Exchange", "exchange_copy",
    "exchange_pack_all", "exchange_unpack_all",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblayoutmove.so")

STATUS = {
    0: "LM_OK", -1: "LM_E_INVALID", -2: "LM_E_INCOMPATIBLE",
    -3: "LM_E_NOT_REPRESENTABLE", -4: "LM_E_NOT_INJECTIVE",
    -5: "LM_E_OVERFLOW", -6: "LM_E_CAPACITY", -7: "LM_E_OVERLAP",
    -8: "LM_E_CUDA", -9: "LM_E_TIMEOUT", -10: "LM_E_NOMEM",
    -11: "LM_E_BUFFER",
}

# (name, restype, argtypes) of every function include/layoutmove.h declares
_P = C.c_void_p
_I64 = C.c_int64
_I64P = C.POINTER(C.c_int64)
_IP = C.POINTER(C.c_int)
SIGNATURES = [
    ("lm_layout_make", C.c_int,
     [C.c_int, _I64P, _I64P, C.c_int, _IP, C.POINTER(_P)]),
    ("lm_layout_parse", C.c_int, [C.c_char_p, C.POINTER(_P)]),
    ("lm_layout_to_string", C.c_int, [_P, C.c_char_p, C.c_size_t]),
    ("lm_layout_print_grid", C.c_int, [_P, C.c_int, C.c_char_p, C.c_size_t]),
    ("lm_layout_size", C.c_int, [_P, _I64P]),
    ("lm_layout_cosize", C.c_int, [_P, _I64P]),
    ("lm_layout_rank", C.c_int, [_P, _IP, _IP]),
    ("lm_layout_leaves", C.c_int, [_P, _I64P, _I64P, _IP]),
    ("lm_layout_get_swizzle", C.c_int, [_P, _IP, _IP, _IP]),
    ("lm_layout_eval", C.c_int, [_P, _I64, _I64P]),
    ("lm_layout_eval_coord", C.c_int, [_P, C.c_int, _I64P, _I64P]),
    ("lm_layout_compose", C.c_int, [_P, _P, C.POINTER(_P)]),
    ("lm_layout_zipped_divide", C.c_int, [_P, C.c_int, _I64P, C.POINTER(_P)]),
    ("lm_layout_swizzle", C.c_int,
     [_P, C.c_int, C.c_int, C.c_int, C.POINTER(_P)]),
    ("lm_layout_concat", C.c_int, [_P, _P, C.POINTER(_P)]),
    ("lm_layout_coalesce", C.c_int, [_P, C.POINTER(_P)]),
    ("lm_layout_right_inverse", C.c_int, [_P, C.POINTER(_P)]),
    ("lm_layout_max_common_vector", C.c_int, [_P, _P, _I64P]),
    ("lm_layout_complement", C.c_int, [_P, _I64, C.POINTER(_P)]),
    ("lm_layout_logical_product", C.c_int, [_P, _P, C.POINTER(_P)]),
    ("lm_layout_blocked_product", C.c_int, [_P, _P, C.POINTER(_P)]),
    ("lm_layout_local_partition", C.c_int,
     [_P, _P, _I64, C.POINTER(_P), _I64P]),
    ("lm_layout_stripmined", C.c_int, [_I64, _I64, _I64, _I64, C.POINTER(_P)]),
    ("lm_smem_wavefronts", C.c_int, [_P, C.c_int, C.c_int, _I64P, _I64P]),
    ("lm_stripmined_tune", C.c_int,
     [_I64, _I64, _I64, _I64, C.c_int, C.c_int, _P, _I64P, _I64P, _I64P,
      _I64P]),
    ("lm_layout_destroy", None, [_P]),
    ("lm_plan_copy", C.c_int, [_P, _P, C.c_int, C.POINTER(_P)]),
    ("lm_plan_copy_shard", C.c_int,
     [_P, _P, C.c_int, C.c_int, C.c_int, C.POINTER(_P)]),
    ("lm_plan_describe", C.c_int, [_P, C.c_char_p, C.c_size_t]),
    ("lm_plan_extent", C.c_int, [_P, _I64P, _I64P, _I64P]),
    ("lm_layout_copy", C.c_int, [_P, _P, _I64, _P, _I64, _P]),
    ("lm_plan_launches", C.c_int, [_P, _IP]),
    ("lm_layout_copy_host", C.c_int, [_P, _P, _I64, _P, _I64, _P, _P, _P]),
    ("lm_layout_copy_host_static", C.c_int, [_P, _P, _I64, _P, _I64, _P]),
    ("lm_layout_eval_device", C.c_int, [_P, _P, C.c_int, _I64, _P]),
    ("lm_plan_destroy", None, [_P]),
    ("lm_plan_exchange", C.c_int,
     [_P, _P, C.c_int, C.c_int, C.c_int, C.POINTER(_P)]),
    ("lm_exchange_describe", C.c_int, [_P, C.c_char_p, C.c_size_t]),
    ("lm_exchange_sizes", C.c_int, [_P, _I64P, _I64P, _I64P, _I64P]),
    ("lm_exchange_pack", C.c_int, [_P, C.c_int, _P, _I64, _P, _I64, _P]),
    ("lm_exchange_unpack", C.c_int, [_P, C.c_int, _P, _I64, _P, _I64, _P]),
    ("lm_exchange_pack_all", C.c_int, [_P, _P, _I64, _P, _I64, _P]),
    ("lm_exchange_unpack_all", C.c_int, [_P, _P, _I64, _P, _I64, _P]),
    ("lm_exchange_destroy", None, [_P]),
    ("lm_tv_plan_create", C.c_int,
     [_P, _P, _P, _P, _P, C.c_int, C.c_int, C.c_int, C.POINTER(_P)]),
    ("lm_tv_plan_describe", C.c_int, [_P, C.c_char_p, C.c_size_t]),
    ("lm_tv_plan_args", C.c_int, [_P, _P, C.c_size_t]),
    ("lm_tv_copy", C.c_int, [_P, _P, _I64, _P, _I64, _P]),
    ("lm_tv_plan_destroy", None, [_P]),
    ("lm_status_string", C.c_char_p, [C.c_int]),
    ("lm_last_cuda_error", C.c_int, []),
    ("lm_device_status", C.c_int, [_P, C.c_int, _IP]),
    ("lm_selftest_bounded_wait", C.c_int, [C.c_int, _P, _IP]),
    ("lm_version", C.c_char_p, []),
]

_lib = None


def lib() -> C.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(no CPU fallback exists)")
        handle = C.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class LayoutMoveError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS.get(status, str(status))
        extra = ""
        if status == -8:
            extra = f" (cudaError {lib().lm_last_cuda_error()})"
        super().__init__(f"{what}: {name}{extra}")


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise LayoutMoveError(rc, what)


def _i64s(vals: Sequence[int]):
    return (C.c_int64 * max(len(vals), 1))(*vals)


def _fmt(x) -> str:
    if isinstance(x, int):
        return str(x)
    return "(" + ",".join(_fmt(k) for k in x) + ")"


class Layout:
    """A layout handle: shape:stride with nested modes, optionally swizzled."""

    __slots__ = ("_h",)

    def __init__(self, handle):
        if not handle:
            raise ValueError("null layout handle")
        self._h = C.c_void_p(handle)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.lm_layout_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    # -- construction ---------------------------------------------------
    @classmethod
    def parse(cls, text: str) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_parse(text.encode(), C.byref(out)),
               f"lm_layout_parse({text!r})")
        return cls(out.value)

    @classmethod
    def of(cls, shape, stride) -> "Layout":
        """From nested Python tuples, e.g. Layout.of((4, 2), (2, 1))."""
        return cls.parse(f"{_fmt(shape)}:{_fmt(stride)}")

    @classmethod
    def make(cls, shape: Sequence[int], stride: Sequence[int],
             leaves_per_mode: Sequence[int] | None = None) -> "Layout":
        out = C.c_void_p()
        n = len(shape)
        lpm = list(leaves_per_mode) if leaves_per_mode is not None else []
        arr = (C.c_int * max(len(lpm), 1))(*lpm)
        _check(lib().lm_layout_make(n, _i64s(shape), _i64s(stride), len(lpm),
                                    arr, C.byref(out)), "lm_layout_make")
        return cls(out.value)

    @classmethod
    def stripmined(cls, threads: int, pitch: int, strips: int,
                   k_row: int) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_stripmined(threads, pitch, strips, k_row,
                                          C.byref(out)), "lm_layout_stripmined")
        return cls(out.value)

    # -- inspection -----------------------------------------------------
    def __str__(self) -> str:
        cap = 256
        while True:
            buf = C.create_string_buffer(cap)
            rc = lib().lm_layout_to_string(self._h, buf, cap)
            if rc == -11:
                cap *= 4
                continue
            _check(rc, "lm_layout_to_string")
            return buf.value.decode()

    __repr__ = __str__

    def print_grid(self, bank_elem_bytes: int = 0) -> str:
        """print_layout's grid of a rank-2 layout (rows = mode 0); with
        bank_elem_bytes > 0, the shared-memory bank of every entry."""
        cap = 1 << 16
        while True:
            buf = C.create_string_buffer(cap)
            rc = lib().lm_layout_print_grid(self._h, int(bank_elem_bytes), buf,
                                            cap)
            if rc == -11:
                cap *= 4
                continue
            _check(rc, "lm_layout_print_grid")
            return buf.value.decode()

    @property
    def size(self) -> int:
        v = C.c_int64()
        _check(lib().lm_layout_size(self._h, C.byref(v)), "lm_layout_size")
        return v.value

    @property
    def cosize(self) -> int:
        v = C.c_int64()
        _check(lib().lm_layout_cosize(self._h, C.byref(v)), "lm_layout_cosize")
        return v.value

    def leaves(self) -> tuple[list[int], list[int], list[int]]:
        nm, nl = C.c_int(), C.c_int()
        _check(lib().lm_layout_rank(self._h, C.byref(nm), C.byref(nl)),
               "lm_layout_rank")
        sh = (C.c_int64 * max(nl.value, 1))()
        st = (C.c_int64 * max(nl.value, 1))()
        lpm = (C.c_int * max(nm.value, 1))()
        _check(lib().lm_layout_leaves(self._h, sh, st, lpm), "lm_layout_leaves")
        return (list(sh)[:nl.value], list(st)[:nl.value], list(lpm)[:nm.value])

    @property
    def swizzle_params(self) -> tuple[int, int, int]:
        b, m, s = C.c_int(), C.c_int(), C.c_int()
        _check(lib().lm_layout_get_swizzle(self._h, C.byref(b), C.byref(m),
                                           C.byref(s)), "lm_layout_get_swizzle")
        return b.value, m.value, s.value

    def __call__(self, index: int) -> int:
        v = C.c_int64()
        _check(lib().lm_layout_eval(self._h, int(index), C.byref(v)),
               "lm_layout_eval")
        return v.value

    def eval_coord(self, coord: Sequence[int]) -> int:
        v = C.c_int64()
        _check(lib().lm_layout_eval_coord(self._h, len(coord), _i64s(coord),
                                          C.byref(v)), "lm_layout_eval_coord")
        return v.value

    def local_partition(self, thr: "Layout",
                        thr_idx: int) -> tuple["Layout", int]:
        """(part, base): thread thr_idx's values sit at
        swizzle(base + part(v))."""
        out, base = C.c_void_p(), C.c_int64()
        _check(lib().lm_layout_local_partition(self._h, thr._h, int(thr_idx),
                                               C.byref(out), C.byref(base)),
               "lm_layout_local_partition")
        return Layout(out.value), base.value

    def smem_wavefronts(self, elem_bytes: int,
                        access_bytes: int | None = None) -> tuple[int, int]:
        """(wavefronts, conflict-free minimum) of warps reading shared
        memory at this layout's offsets, 32 consecutive indices a warp."""
        w, i = C.c_int64(), C.c_int64()
        ab = elem_bytes if access_bytes is None else access_bytes
        _check(lib().lm_smem_wavefronts(self._h, elem_bytes, ab, C.byref(w),
                                        C.byref(i)), "lm_smem_wavefronts")
        return w.value, i.value

    # -- algebra --------------------------------------------------------
    def _binary(self, fn, other, what) -> "Layout":
        out = C.c_void_p()
        _check(fn(self._h, other._h, C.byref(out)), what)
        return Layout(out.value)

    def compose(self, inner: "Layout") -> "Layout":
        """self o inner."""
        return self._binary(lib().lm_layout_compose, inner, "lm_layout_compose")

    def concat(self, other: "Layout") -> "Layout":
        return self._binary(lib().lm_layout_concat, other, "lm_layout_concat")

    def zipped_divide(self, tiler: Sequence[int]) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_zipped_divide(self._h, len(tiler), _i64s(tiler),
                                             C.byref(out)),
               "lm_layout_zipped_divide")
        return Layout(out.value)

    def swizzle(self, b: int, m: int, s: int) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_swizzle(self._h, b, m, s, C.byref(out)),
               "lm_layout_swizzle")
        return Layout(out.value)

    def coalesce(self) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_coalesce(self._h, C.byref(out)),
               "lm_layout_coalesce")
        return Layout(out.value)

    def complement(self, cotarget: int) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_complement(self._h, int(cotarget),
                                          C.byref(out)), "lm_layout_complement")
        return Layout(out.value)

    def logical_product(self, other: "Layout") -> "Layout":
        return self._binary(lib().lm_layout_logical_product, other,
                            "lm_layout_logical_product")

    def blocked_product(self, other: "Layout") -> "Layout":
        return self._binary(lib().lm_layout_blocked_product, other,
                            "lm_layout_blocked_product")

    def right_inverse(self) -> "Layout":
        out = C.c_void_p()
        _check(lib().lm_layout_right_inverse(self._h, C.byref(out)),
               "lm_layout_right_inverse")
        return Layout(out.value)

    def max_common_vector(self, other: "Layout") -> int:
        v = C.c_int64()
        _check(lib().lm_layout_max_common_vector(self._h, other._h,
                                                 C.byref(v)),
               "lm_layout_max_common_vector")
        return v.value


class Plan:
    """A lowered copy plan for out[dst(i)] = in[src(i)]."""

    __slots__ = ("_h", "elem_bytes")

    def __init__(self, src: Layout, dst: Layout, elem_bytes: int,
                 rank: int = 0, world: int = 1):
        """The copy plan, or with world > 1 the plan of shard `rank`."""
        out = C.c_void_p()
        if world == 1:
            _check(lib().lm_plan_copy(src.handle, dst.handle, int(elem_bytes),
                                      C.byref(out)), "lm_plan_copy")
        else:
            _check(lib().lm_plan_copy_shard(src.handle, dst.handle,
                                            int(elem_bytes), int(rank),
                                            int(world), C.byref(out)),
                   "lm_plan_copy_shard")
        self._h = out
        self.elem_bytes = int(elem_bytes)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.lm_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def describe(self) -> dict:
        cap = 4096
        while True:
            buf = C.create_string_buffer(cap)
            rc = lib().lm_plan_describe(self._h, buf, cap)
            if rc == -11:
                cap *= 4
                continue
            _check(rc, "lm_plan_describe")
            return json.loads(buf.value.decode())

    def extent(self) -> tuple[int, int, int]:
        n, sc, dc = C.c_int64(), C.c_int64(), C.c_int64()
        _check(lib().lm_plan_extent(self._h, C.byref(n), C.byref(sc),
                                    C.byref(dc)), "lm_plan_extent")
        return n.value, sc.value, dc.value

    @property
    def launches(self) -> int:
        v = C.c_int()
        _check(lib().lm_plan_launches(self._h, C.byref(v)), "lm_plan_launches")
        return v.value


class TVPlan:
    """A copy staged tile by tile through a caller-chosen shared layout,
    each phase a local_partition by a caller-chosen thread layout."""

    __slots__ = ("_h", "elem_bytes")

    def __init__(self, src: Layout, smem: Layout, dst: Layout,
                 thr_load: Layout | None, thr_store: Layout | None,
                 elem_bytes: int, vec_load_bytes: int = 0,
                 vec_store_bytes: int = 0):
        """thr_load / thr_store None: the library's tuned stripmined thread
        layout for that phase (see lm_tv_plan_create)."""
        out = C.c_void_p()
        tl = thr_load.handle if thr_load is not None else None
        ts = thr_store.handle if thr_store is not None else None
        _check(lib().lm_tv_plan_create(src.handle, smem.handle, dst.handle,
                                       tl, ts,
                                       int(elem_bytes), int(vec_load_bytes),
                                       int(vec_store_bytes), C.byref(out)),
               "lm_tv_plan_create")
        self._h = out
        self.elem_bytes = int(elem_bytes)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.lm_tv_plan_destroy(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def describe(self) -> dict:
        buf = C.create_string_buffer(4096)
        _check(lib().lm_tv_plan_describe(self._h, buf, 4096),
               "lm_tv_plan_describe")
        return json.loads(buf.value.decode())

    def args_bytes(self) -> bytes:
        """The lm_tv_args block (layoutmove_tv.h) for consumer kernels."""
        buf = C.create_string_buffer(8192)
        _check(lib().lm_tv_plan_args(self._h, buf, 8192), "lm_tv_plan_args")
        return buf.raw


class Exchange:
    """Rank `rank` of a relayout whose source and destination are both
    sharded over `world` ranks (see lm_plan_exchange)."""

    __slots__ = ("_h", "elem_bytes", "world")

    def __init__(self, src: Layout, dst: Layout, elem_bytes: int, rank: int,
                 world: int):
        out = C.c_void_p()
        _check(lib().lm_plan_exchange(src.handle, dst.handle, int(elem_bytes),
                                      int(rank), int(world), C.byref(out)),
               "lm_plan_exchange")
        self._h = out
        self.elem_bytes = int(elem_bytes)
        self.world = int(world)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.lm_exchange_destroy(h)
            self._h = None

    def describe(self) -> dict:
        cap = 4096
        while True:
            buf = C.create_string_buffer(cap)
            rc = lib().lm_exchange_describe(self._h, buf, cap)
            if rc == -11:
                cap *= 4
                continue
            _check(rc, "lm_exchange_describe")
            return json.loads(buf.value.decode())

    def sizes(self) -> dict:
        sl, dl = C.c_int64(), C.c_int64()
        sc = (C.c_int64 * self.world)()
        rc = (C.c_int64 * self.world)()
        _check(lib().lm_exchange_sizes(self._h, C.byref(sl), C.byref(dl), sc,
                                       rc), "lm_exchange_sizes")
        return {"src_local": sl.value, "dst_local": dl.value,
                "send": list(sc), "recv": list(rc)}

    def pack(self, peer: int, src_local, send, stream=None) -> None:
        sp, scap = _dev_buffer(src_local, self.elem_bytes)
        dp, dcap = _dev_buffer(send, self.elem_bytes)
        _check(lib().lm_exchange_pack(self._h, int(peer), C.c_void_p(sp),
                                      scap, C.c_void_p(dp), dcap,
                                      _stream_handle(stream)),
               "lm_exchange_pack")

    def unpack(self, peer: int, recv, dst_local, stream=None) -> None:
        sp, scap = _dev_buffer(recv, self.elem_bytes)
        dp, dcap = _dev_buffer(dst_local, self.elem_bytes)
        _check(lib().lm_exchange_unpack(self._h, int(peer), C.c_void_p(sp),
                                        scap, C.c_void_p(dp), dcap,
                                        _stream_handle(stream)),
               "lm_exchange_unpack")


def _exchange_all(fn, ex, a, b, stream, what):
    ap, acap = _dev_buffer(a, ex.elem_bytes)
    bp, bcap = _dev_buffer(b, ex.elem_bytes)
    _check(fn(ex._h, C.c_void_p(ap), acap, C.c_void_p(bp), bcap,
              _stream_handle(stream)), what)


def exchange_pack_all(ex: Exchange, src_local, send, stream=None) -> None:
    """Every peer's box into one buffer, peer after peer."""
    _exchange_all(lib().lm_exchange_pack_all, ex, src_local, send, stream,
                  "lm_exchange_pack_all")


def exchange_unpack_all(ex: Exchange, recv, dst_local, stream=None) -> None:
    """Every sender's box from one buffer, sender after sender."""
    _exchange_all(lib().lm_exchange_unpack_all, ex, recv, dst_local, stream,
                  "lm_exchange_unpack_all")


def exchange_copy(ex: Exchange, src_local, dst_local, group=None) -> None:
    """Pack every peer's box, exchange the buffers with one
    torch.distributed all_to_all_single, unpack: the sharded relayout of
    rank ex's shards (CUDA uint8 tensors)."""
    import torch
    import torch.distributed as dist
    sz = ex.sizes()
    eb = ex.elem_bytes
    send = torch.empty(sum(sz["send"]) * eb, dtype=torch.uint8,
                       device=src_local.device)
    recv = torch.empty(sum(sz["recv"]) * eb, dtype=torch.uint8,
                       device=dst_local.device)
    exchange_pack_all(ex, src_local, send)
    dist.all_to_all_single(recv, send, [n * eb for n in sz["recv"]],
                           [n * eb for n in sz["send"]], group=group)
    exchange_unpack_all(ex, recv, dst_local)


def _stream_handle(stream) -> C.c_void_p:
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _dev_buffer(t, elem_bytes: int) -> tuple[int, int]:
    """(device pointer, capacity in elements) of a CUDA tensor."""
    if not t.is_cuda:
        raise ValueError("layout_copy takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("buffers must be contiguous")
    nbytes = t.numel() * t.element_size()
    return t.data_ptr(), nbytes // elem_bytes


def layout_copy(plan: Plan, src, dst, stream=None) -> None:
    """Enqueue dst[dst_layout(i)] = src[src_layout(i)] on ``stream`` (default:
    torch's current stream).  src/dst are contiguous CUDA tensors viewed as
    flat arrays of plan.elem_bytes-byte elements."""
    sp, scap = _dev_buffer(src, plan.elem_bytes)
    dp, dcap = _dev_buffer(dst, plan.elem_bytes)
    _check(lib().lm_layout_copy(plan.handle, C.c_void_p(sp), scap,
                                C.c_void_p(dp), dcap, _stream_handle(stream)),
           "lm_layout_copy")


def stripmined_tune(threads: int, k_row: int, rows: int, elem_bytes: int,
                    vec_elems: int = 1, ld: int | None = None,
                    smem: Layout | None = None) -> dict:
    """Pitch and Strips of the stripmined map for one pass over a tile (see
    lm_stripmined_tune): {"pitch", "strips", "segments", "wavefronts"}."""
    p, s, g, w = C.c_int64(), C.c_int64(), C.c_int64(), C.c_int64()
    _check(lib().lm_stripmined_tune(int(threads), int(k_row), int(rows),
                                    int(k_row if ld is None else ld),
                                    int(elem_bytes), int(vec_elems),
                                    smem.handle if smem is not None else None,
                                    C.byref(p), C.byref(s), C.byref(g),
                                    C.byref(w)), "lm_stripmined_tune")
    return {"pitch": p.value, "strips": s.value, "segments": g.value,
            "wavefronts": w.value}


def tv_copy(plan: TVPlan, src, dst, stream=None) -> None:
    """Enqueue the tile-staged copy of ``plan`` (see TVPlan) on ``stream``."""
    sp, scap = _dev_buffer(src, plan.elem_bytes)
    dp, dcap = _dev_buffer(dst, plan.elem_bytes)
    _check(lib().lm_tv_copy(plan.handle, C.c_void_p(sp), scap,
                            C.c_void_p(dp), dcap, _stream_handle(stream)),
           "lm_tv_copy")


def layout_copy_host(plan: Plan, src_host, dst_host, src_dev, dst_dev,
                     stream=None) -> None:
    """Enqueue upload, copy and download for host tensors (pinned for
    asynchrony) through the device staging tensors src_dev / dst_dev, which
    must be at least as large as the host tensors."""
    for t in (src_host, dst_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors")
    sp, scap = _dev_buffer(src_dev, plan.elem_bytes)
    dp, dcap = _dev_buffer(dst_dev, plan.elem_bytes)
    hs = src_host.numel() * src_host.element_size() // plan.elem_bytes
    hd = dst_host.numel() * dst_host.element_size() // plan.elem_bytes
    if scap < hs or dcap < hd:
        raise ValueError("staging buffers smaller than the host buffers")
    _check(lib().lm_layout_copy_host(plan.handle,
                                     C.c_void_p(src_host.data_ptr()), hs,
                                     C.c_void_p(dst_host.data_ptr()), hd,
                                     C.c_void_p(sp), C.c_void_p(dp),
                                     _stream_handle(stream)),
           "lm_layout_copy_host")


# Size of the fixed device staging area of layout_copy_host_static (the
# header's LM_HOST_COPY_STATIC_BYTES).
HOST_COPY_STATIC_BYTES = 32 * 1024 * 1024


def layout_copy_host_static(plan: Plan, src_host, dst_host,
                            stream=None) -> None:
    """layout_copy_host without device staging buffers from the caller: for
    code that cannot allocate device memory (a program whose memory manager
    owns the device's memory, or a path that cannot afford cudaMalloc or
    cudaFree).  The library stages through its own fixed area of
    HOST_COPY_STATIC_BYTES on each device; larger copies are refused
    (LM_E_CAPACITY).  Calls share that area, so calls that overlap on the
    GPU race.  Nothing is allocated here either: the host tensors are
    passed by pointer."""
    for t in (src_host, dst_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous CPU tensors")
    hs = src_host.numel() * src_host.element_size() // plan.elem_bytes
    hd = dst_host.numel() * dst_host.element_size() // plan.elem_bytes
    _check(lib().lm_layout_copy_host_static(
        plan.handle, C.c_void_p(src_host.data_ptr()), hs,
        C.c_void_p(dst_host.data_ptr()), hd, _stream_handle(stream)),
        "lm_layout_copy_host_static")


def layout_copy_ptr(plan: Plan, src_ptr: int, src_cap: int, dst_ptr: int,
                    dst_cap: int, stream=None) -> None:
    """Raw-pointer form of layout_copy (capacities in elements)."""
    _check(lib().lm_layout_copy(plan.handle, C.c_void_p(src_ptr), src_cap,
                                C.c_void_p(dst_ptr), dst_cap,
                                _stream_handle(stream)), "lm_layout_copy")


def layout_eval_device(layout: Layout, table, stream=None) -> None:
    """Enqueue table[i] = layout(i) into an int32 or int64 CUDA tensor."""
    import torch
    if table.dtype not in (torch.int32, torch.int64) or not table.is_cuda:
        raise ValueError("table must be a CUDA int32 or int64 tensor")
    _check(lib().lm_layout_eval_device(layout.handle,
                                       C.c_void_p(table.data_ptr()),
                                       table.element_size(), table.numel(),
                                       _stream_handle(stream)),
           "lm_layout_eval_device")


def device_status(stream=None, reset: bool = False) -> int:
    """Synchronise the stream and return LM_OK (0) or LM_E_TIMEOUT (-9) if a
    kernel of the library gave up a bounded wait since the last reset."""
    st = C.c_int()
    _check(lib().lm_device_status(_stream_handle(stream), int(reset),
                                  C.byref(st)), "lm_device_status")
    return st.value


def build_layout(spec) -> Layout:
    """A layout from a workload description (see ``workloads``), built with
    the library's own algebra calls."""
    kind = spec[0]
    if kind == "layout":
        return Layout.of(spec[1], spec[2])
    if kind == "swizzle":
        return build_layout(spec[4]).swizzle(spec[1], spec[2], spec[3])
    if kind == "compose":
        return build_layout(spec[1]).compose(build_layout(spec[2]))
    if kind == "zipped_divide":
        return build_layout(spec[1]).zipped_divide(list(spec[2]))
    if kind == "blocked_product":
        return build_layout(spec[1]).blocked_product(build_layout(spec[2]))
    if kind == "logical_product":
        return build_layout(spec[1]).logical_product(build_layout(spec[2]))
    if kind == "concat":
        parts: Iterable = [build_layout(s) for s in spec[1:]]
        it = iter(parts)
        acc = next(it)
        for p in it:
            acc = acc.concat(p)
        return acc
    raise ValueError(f"unknown layout description {kind!r}")
