"""Thin Python binding of libq1gemv.so (see include/q1gemv.h).

Argument marshalling only: every function checks tensor dtypes, devices and
shapes, passes raw device pointers and the current CUDA stream to the C ABI,
and raises ``Q1Error`` with the library's message when a call fails.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.

Tensors:
  blocks  torch.uint8  [rows, n/128, 18]  Q1_0 blocks (see q1_0_pack)
  packed  torch.uint8  [q1_0_packed_bytes(rows, n)]
  x       torch.float32 [nvec, n]
  q       torch.int8   [nvec, n] (or [n])
  d       torch.int16/uint16 [nvec, n/32] (fp16 bit patterns; torch.float16 accepted)
  out     torch.float32 [nvec, rows] (or [rows])
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

Q1_OK = 0
Q1_ERR_ARG = -1
Q1_ERR_CUDA = -2
Q1_ERR_NOMEM = -3
Q1_MISMATCH = 2

# Every symbol include/q1gemv.h declares (checked by the tests).
EXPORTS = ("q1_last_error", "q1_0_packed_bytes", "q1_0_pack", "q1_0_unpack", "q8_quantize_act",
           "q1_0_gemv", "q1_0_gemv_multi", "q1_0_gemv_multi_plan", "q1_0_gemm_small", "q1_0_verify",
           "q1_device_status", "q2_0_packed_bytes", "q2_0_pack", "q2_0_unpack", "q2_0_gemv", "q2_0_gemv_multi",
           "q2_0_gemv_multi_plan", "q1_gemm_small_kernel", "q1_0_gemm_small_noalloc",
           "q1_0_gemv_multi_prefetch", "q2_0_gemv_multi_prefetch")

MAX_PRODUCTS = 256


class Product(ctypes.Structure):
    """Mirror of q1_product (include/q1gemv.h)."""
    _fields_ = [("packed", ctypes.c_void_p), ("rows", ctypes.c_int64), ("n", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("q", ctypes.c_void_p), ("d", ctypes.c_void_p),
                ("out", ctypes.c_void_p)]


class Range(ctypes.Structure):
    """Mirror of q1_range (include/q1gemv.h)."""
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_int64)]


MAX_PREFETCH_RANGES = 4


class MultiPlan(ctypes.Structure):
    """Mirror of q1_multi_plan (include/q1gemv.h)."""
    _fields_ = [("rows_per_thread", ctypes.c_int), ("grid", ctypes.c_int), ("total_cost", ctypes.c_int64),
                ("max_range_cost", ctypes.c_int64), ("panel_warps", ctypes.c_int),
                ("panel_unit_blocks", ctypes.c_int), ("panel_panels", ctypes.c_int)]


class Q1Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libq1gemv.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libq1gemv.so not found at {path}")
        lib = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.q1_last_error.argtypes = []
        lib.q1_last_error.restype = ctypes.c_char_p
        lib.q1_0_packed_bytes.argtypes = [I64, I64]
        lib.q1_0_packed_bytes.restype = I64
        lib.q1_0_pack.argtypes = [P, I64, I64, P, P]
        lib.q1_0_pack.restype = I
        lib.q1_0_unpack.argtypes = [P, I64, I64, P, P]
        lib.q1_0_unpack.restype = I
        lib.q8_quantize_act.argtypes = [P, I64, I64, P, P, P]
        lib.q8_quantize_act.restype = I
        lib.q1_0_gemv.argtypes = [P, I64, I64, P, P, P, P]
        lib.q1_0_gemv.restype = I
        lib.q1_0_gemv_multi.argtypes = [ctypes.POINTER(Product), I, P]
        lib.q1_0_gemv_multi.restype = I
        lib.q1_0_gemv_multi_plan.argtypes = [ctypes.POINTER(Product), I, I, ctypes.POINTER(MultiPlan),
                                             ctypes.POINTER(I64), I]
        lib.q1_0_gemv_multi_plan.restype = I
        lib.q2_0_gemv_multi_plan.argtypes = lib.q1_0_gemv_multi_plan.argtypes
        lib.q2_0_gemv_multi_plan.restype = I
        lib.q2_0_packed_bytes.argtypes = [I64, I64]
        lib.q2_0_packed_bytes.restype = I64
        lib.q2_0_pack.argtypes = [P, I64, I64, P, P]
        lib.q2_0_pack.restype = I
        lib.q2_0_unpack.argtypes = [P, I64, I64, P, P]
        lib.q2_0_unpack.restype = I
        lib.q2_0_gemv.argtypes = [P, I64, I64, P, P, P, P]
        lib.q2_0_gemv.restype = I
        lib.q2_0_gemv_multi.argtypes = [ctypes.POINTER(Product), I, P]
        lib.q2_0_gemv_multi.restype = I
        for fn in (lib.q1_0_gemv_multi_prefetch, lib.q2_0_gemv_multi_prefetch):
            fn.argtypes = [ctypes.POINTER(Product), I, ctypes.POINTER(Range), I, P]
            fn.restype = I
        lib.q1_0_gemm_small.argtypes = [P, I64, I64, I64, P, P, P, P]
        lib.q1_0_gemm_small.restype = I
        lib.q1_0_gemm_small_noalloc.argtypes = [P, I64, I64, I64, P, P, P, P]
        lib.q1_0_gemm_small_noalloc.restype = I
        lib.q1_gemm_small_kernel.argtypes = [I]
        lib.q1_gemm_small_kernel.restype = I
        lib.q1_device_status.argtypes = [I]
        lib.q1_device_status.restype = I
        lib.q1_0_verify.argtypes = [I, ctypes.c_char_p, ctypes.c_size_t]
        lib.q1_0_verify.restype = I
        _lib = lib
        return lib


def last_error() -> str:
    return load().q1_last_error().decode(errors="replace")


def _check(rc: int, what: str):
    if rc != Q1_OK:
        raise Q1Error(rc, f"{what}: {last_error()}")


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtypes, host_ok: bool = False) -> int:
    """Pointer of a contiguous CUDA tensor (or, where host_ok, of a pinned
    host tensor, which the kernels address directly)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or (host_ok and t.is_pinned())):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _packed_ptr(packed: torch.Tensor, rows: int, n: int, fmt: str) -> int:
    """Pointer of a packed weight buffer after checking that it holds the
    format's packed size for a rows x n matrix: the library reads that many
    bytes from the pointer, which it cannot check itself."""
    need = packed_bytes(rows, n) if fmt == "q1" else q2_packed_bytes(rows, n)
    if not isinstance(packed, torch.Tensor):
        raise TypeError("packed must be a torch.Tensor")
    if packed.numel() * packed.element_size() < need:
        raise ValueError(f"packed holds {packed.numel() * packed.element_size()} bytes; a {fmt.upper()}_0 "
                         f"{rows} x {n} matrix needs {need}")
    return _dev(packed, "packed", (torch.uint8,))


_SCALE_DTYPES = (torch.int16, torch.float16) + ((torch.uint16,) if hasattr(torch, "uint16") else ())


# ------------------------------------------------------------------ calls --
def packed_bytes(rows: int, n: int) -> int:
    v = load().q1_0_packed_bytes(int(rows), int(n))
    if v < 0:
        raise Q1Error(int(v), last_error())
    return int(v)


def pack(blocks: torch.Tensor, rows: int, n: int, packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    nbytes = packed_bytes(rows, n)
    if blocks.numel() != rows * (n // 128) * 18:
        raise ValueError("blocks must hold rows*(n/128) 18-byte blocks")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=blocks.device)
    if packed.numel() * packed.element_size() < nbytes:
        raise ValueError("packed buffer too small")
    _check(load().q1_0_pack(_dev(blocks, "blocks", (torch.uint8,)), rows, n,
                            _dev(packed, "packed", (torch.uint8,)), _stream_ptr(stream)), "q1_0_pack")
    return packed


def unpack(packed: torch.Tensor, rows: int, n: int, blocks: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    packed_bytes(rows, n)
    if blocks is None:
        blocks = torch.empty((rows, n // 128, 18), dtype=torch.uint8, device=packed.device)
    if blocks.numel() != rows * (n // 128) * 18:
        raise ValueError("blocks must hold rows*(n/128) 18-byte blocks")
    _check(load().q1_0_unpack(_packed_ptr(packed, rows, n, "q1"), rows, n,
                              _dev(blocks, "blocks", (torch.uint8,)), _stream_ptr(stream)), "q1_0_unpack")
    return blocks


def quantize(x: torch.Tensor, q: torch.Tensor | None = None, d: torch.Tensor | None = None, stream=None):
    """q8_0 quantization of x [nvec, n] (or [n]).  Returns (q int8, d int16 fp16 bits).
    x, q and d may be pinned host tensors (the kernel addresses them directly);
    q and d are allocated on the GPU when not given."""
    n = x.shape[-1]
    nvec = x.numel() // n if n else 0
    dev = x.device if x.is_cuda else torch.device("cuda")
    if q is None:
        q = torch.empty(x.shape, dtype=torch.int8, device=dev)
    if d is None:
        d = torch.empty(x.shape[:-1] + (n // 32,), dtype=torch.int16, device=dev)
    if q.numel() != nvec * n or d.numel() != nvec * (n // 32):
        raise ValueError("q/d sizes do not match x")
    _check(load().q8_quantize_act(_dev(x, "x", (torch.float32,), True), nvec, n,
                                  _dev(q, "q", (torch.int8,), True), _dev(d, "d", _SCALE_DTYPES, True),
                                  _stream_ptr(stream)), "q8_quantize_act")
    return q, d


def gemv(packed: torch.Tensor, rows: int, n: int, q: torch.Tensor, d: torch.Tensor,
         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if q.numel() != n or d.numel() != n // 32:
        raise ValueError("q must hold n quants and d n/32 scales")
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=q.device)
    if out.numel() != rows:
        raise ValueError("out must hold rows values")
    _check(load().q1_0_gemv(_packed_ptr(packed, rows, n, "q1"), rows, n, _dev(q, "q", (torch.int8,)),
                            _dev(d, "d", _SCALE_DTYPES), _dev(out, "out", (torch.float32,)),
                            _stream_ptr(stream)), "q1_0_gemv")
    return out


def product_array(items, fmt: str = "q1"):
    """Build a ctypes q1_product array from tuples
    (packed, rows, n, x_or_None, q_or_None, d_or_None, out) of CUDA tensors;
    x, q, d and out may also be pinned host tensors.  fmt ("q1" or "q2") is
    the weight format the array is for: each packed buffer is checked against
    that format's packed size."""
    if fmt not in ("q1", "q2"):
        raise ValueError("fmt must be 'q1' or 'q2'")
    arr = (Product * len(items))()
    for i, (packed, rows, n, x, q, d, out) in enumerate(items):
        if x is None and (q is None or d is None):
            raise ValueError("each product needs x, or q and d")
        if x is not None and x.numel() != n:
            raise ValueError("x must hold n values")
        if q is not None and (q.numel() != n or d.numel() != n // 32):
            raise ValueError("q must hold n quants and d n/32 scales")
        if out.numel() != rows:
            raise ValueError("out must hold rows values")
        arr[i] = Product(_packed_ptr(packed, int(rows), int(n), fmt), int(rows), int(n),
                         _dev(x, "x", (torch.float32,), True) if x is not None else None,
                         _dev(q, "q", (torch.int8,), True) if q is not None else None,
                         _dev(d, "d", _SCALE_DTYPES, True) if d is not None else None,
                         _dev(out, "out", (torch.float32,), True))
    return arr


def _one_range(r):
    if isinstance(r, torch.Tensor):
        if not r.is_cuda or not r.is_contiguous():
            raise ValueError("a prefetch range must be a contiguous CUDA tensor")
        return Range(r.data_ptr(), r.numel() * r.element_size())
    ptr, nbytes = r
    return Range(int(ptr) or None, int(nbytes))


def prefetch_ranges(prefetch):
    """A ctypes q1_range array from a prefetch argument: a CUDA tensor (its
    bytes), a (pointer, bytes) pair, or a list of those."""
    items = [prefetch] if isinstance(prefetch, (torch.Tensor, tuple)) else list(prefetch)
    arr = (Range * max(len(items), 1))()
    for i, r in enumerate(items):
        arr[i] = _one_range(r)
    return arr, len(items)


def gemv_multi(items=None, stream=None, array=None, prefetch=None):
    """One launch for several independent products.  `items` as product_array
    takes them, or a prebuilt `array` (to avoid rebuilding it per call).
    `prefetch` (a CUDA tensor, a (pointer, bytes) pair, or a list of up to
    four of those; or a prebuilt (q1_range array, count) from prefetch_ranges)
    is pulled into L2 while the launch runs, through q1_0_gemv_multi_prefetch."""
    arr = array if array is not None else product_array(items)
    if prefetch is None:
        _check(load().q1_0_gemv_multi(arr, len(arr), _stream_ptr(stream)), "q1_0_gemv_multi")
        return
    ranges, nr = prefetch if _is_range_array(prefetch) else prefetch_ranges(prefetch)
    _check(load().q1_0_gemv_multi_prefetch(arr, len(arr), ranges, nr, _stream_ptr(stream)),
           "q1_0_gemv_multi_prefetch")


def _is_range_array(p) -> bool:
    return isinstance(p, tuple) and len(p) == 2 and isinstance(p[0], ctypes.Array)


def multi_plan(shapes, sms: int = 0, fmt: str = "q1") -> dict:
    """The work split q1_0_gemv_multi (fmt "q1") or q2_0_gemv_multi ("q2")
    would make for products of the given (rows, n) shapes, in list order, on
    `sms` SMs (0 = the current device).  Nothing is launched; needs no GPU when
    sms > 0."""
    if fmt not in ("q1", "q2"):
        raise ValueError("fmt must be 'q1' or 'q2'")
    arr = (Product * len(shapes))()
    for i, (rows, n) in enumerate(shapes):
        arr[i] = Product(None, int(rows), int(n), None, None, None, None)
    plan = MultiPlan()
    cuts = (ctypes.c_int64 * (2 * max(int(sms), 4096) + 1))()
    fn = load().q1_0_gemv_multi_plan if fmt == "q1" else load().q2_0_gemv_multi_plan
    _check(fn(arr, len(arr), int(sms), ctypes.byref(plan), cuts, len(cuts)), f"{fmt}_0_gemv_multi_plan")
    return {"rows_per_thread": plan.rows_per_thread, "grid": plan.grid, "total_cost": plan.total_cost,
            "max_range_cost": plan.max_range_cost, "panel_warps": plan.panel_warps,
            "panel_unit_blocks": plan.panel_unit_blocks, "panel_panels": plan.panel_panels,
            "cuts": list(cuts[:plan.grid + 1]) if plan.panel_warps == 0 else []}


# ------------------------------------------------------- Q2_0 (ternary) --
def q2_packed_bytes(rows: int, n: int) -> int:
    v = load().q2_0_packed_bytes(int(rows), int(n))
    if v < 0:
        raise Q1Error(int(v), last_error())
    return int(v)


def q2_pack(blocks: torch.Tensor, rows: int, n: int, packed: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Pack Q2_0 blocks (uint8, rows*(n/128) 34-byte blocks) into the device layout."""
    nbytes = q2_packed_bytes(rows, n)
    if blocks.numel() != rows * (n // 128) * 34:
        raise ValueError("blocks must hold rows*(n/128) 34-byte blocks")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=blocks.device)
    if packed.numel() * packed.element_size() < nbytes:
        raise ValueError("packed buffer too small")
    _check(load().q2_0_pack(_dev(blocks, "blocks", (torch.uint8,)), rows, n,
                            _dev(packed, "packed", (torch.uint8,)), _stream_ptr(stream)), "q2_0_pack")
    return packed


def q2_unpack(packed: torch.Tensor, rows: int, n: int, blocks: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    q2_packed_bytes(rows, n)
    if blocks is None:
        blocks = torch.empty((rows, n // 128, 34), dtype=torch.uint8, device=packed.device)
    if blocks.numel() != rows * (n // 128) * 34:
        raise ValueError("blocks must hold rows*(n/128) 34-byte blocks")
    _check(load().q2_0_unpack(_packed_ptr(packed, rows, n, "q2"), rows, n,
                              _dev(blocks, "blocks", (torch.uint8,)), _stream_ptr(stream)), "q2_0_unpack")
    return blocks


def q2_gemv(packed: torch.Tensor, rows: int, n: int, q: torch.Tensor, d: torch.Tensor,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if q.numel() != n or d.numel() != n // 32:
        raise ValueError("q must hold n quants and d n/32 scales")
    if out is None:
        out = torch.empty(rows, dtype=torch.float32, device=q.device)
    if out.numel() != rows:
        raise ValueError("out must hold rows values")
    _check(load().q2_0_gemv(_packed_ptr(packed, rows, n, "q2"), rows, n, _dev(q, "q", (torch.int8,)),
                            _dev(d, "d", _SCALE_DTYPES), _dev(out, "out", (torch.float32,)),
                            _stream_ptr(stream)), "q2_0_gemv")
    return out


def q2_gemv_multi(items=None, stream=None, array=None, prefetch=None):
    """One launch for several independent Q2_0 products (items as product_array
    takes them, with packed buffers from q2_pack); `prefetch` as gemv_multi."""
    arr = array if array is not None else product_array(items, fmt="q2")
    if prefetch is None:
        _check(load().q2_0_gemv_multi(arr, len(arr), _stream_ptr(stream)), "q2_0_gemv_multi")
        return
    ranges, nr = prefetch if _is_range_array(prefetch) else prefetch_ranges(prefetch)
    _check(load().q2_0_gemv_multi_prefetch(arr, len(arr), ranges, nr, _stream_ptr(stream)),
           "q2_0_gemv_multi_prefetch")


def gemm_small(packed: torch.Tensor, rows: int, n: int, q: torch.Tensor, d: torch.Tensor,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    nvec = q.numel() // n
    if q.numel() != nvec * n or d.numel() != nvec * (n // 32):
        raise ValueError("q must be [nvec, n] and d [nvec, n/32]")
    if out is None:
        out = torch.empty((nvec, rows), dtype=torch.float32, device=q.device)
    if out.numel() != nvec * rows:
        raise ValueError("out must hold nvec*rows values")
    _check(load().q1_0_gemm_small(_packed_ptr(packed, rows, n, "q1"), rows, n, nvec,
                                  _dev(q, "q", (torch.int8,)), _dev(d, "d", _SCALE_DTYPES),
                                  _dev(out, "out", (torch.float32,)), _stream_ptr(stream)), "q1_0_gemm_small")
    return out


def gemm_small_noalloc(packed: torch.Tensor, rows: int, n: int, q: torch.Tensor, d: torch.Tensor,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gemm_small through q1_0_gemm_small_noalloc: the tensor-core kernel with
    the library's fixed scratch array, no allocation (see include/q1gemv.h)."""
    nvec = q.numel() // n
    if q.numel() != nvec * n or d.numel() != nvec * (n // 32):
        raise ValueError("q must be [nvec, n] and d [nvec, n/32]")
    if out is None:
        out = torch.empty((nvec, rows), dtype=torch.float32, device=q.device)
    if out.numel() != nvec * rows:
        raise ValueError("out must hold nvec*rows values")
    _check(load().q1_0_gemm_small_noalloc(_packed_ptr(packed, rows, n, "q1"), rows, n, nvec,
                                          _dev(q, "q", (torch.int8,)), _dev(d, "d", _SCALE_DTYPES),
                                          _dev(out, "out", (torch.float32,)), _stream_ptr(stream)),
           "q1_0_gemm_small_noalloc")
    return out


GEMM_KERNELS = {"auto": 0, "dp4a": 1, "tensor": 2}


def gemm_small_kernel(choice: str) -> str:
    """Select the kernel of gemm_small for the calls that follow in this
    process ("auto", "dp4a" or "tensor"); returns the previous choice."""
    if choice not in GEMM_KERNELS:
        raise ValueError(f"choice must be one of {sorted(GEMM_KERNELS)}")
    prev = load().q1_gemm_small_kernel(GEMM_KERNELS[choice])
    if prev < 0:
        raise Q1Error(prev, last_error())
    return {v: k for k, v in GEMM_KERNELS.items()}[prev]


def device_status(clear: bool = True) -> int:
    """The library's device status flags (0 = no kernel gave up a wait)."""
    v = load().q1_device_status(1 if clear else 0)
    if v < 0:
        raise Q1Error(v, last_error())
    return v


def verify(quick: bool = False, corrupt: bool = False, wait_probe: bool = False) -> tuple[int, str]:
    """Run the on-card self-check; returns (status, report text).  corrupt=True
    runs the negative control (one row's packed scales doubled per case);
    wait_probe=True first lets a bounded wait run out on purpose."""
    buf = ctypes.create_string_buffer(16384)
    flags = (1 if quick else 0) | (2 if corrupt else 0) | (4 if wait_probe else 0)
    rc = load().q1_0_verify(flags, buf, len(buf))
    return rc, buf.value.decode(errors="replace")


class Q1Linear:
    """A packed Q1_0 weight matrix resident on the GPU (convenience wrapper).

    ``Q1Linear(blocks)`` packs the 18-byte blocks once; ``__call__(q, d)`` runs
    q1_0_gemv for one activation vector and q1_0_gemm_small for several."""

    def __init__(self, blocks: torch.Tensor, stream=None):
        if blocks.dim() != 3 or blocks.shape[2] != 18:
            raise ValueError("blocks must be uint8 [rows, n/128, 18]")
        self.rows = int(blocks.shape[0])
        self.n = int(blocks.shape[1]) * 128
        self.packed = pack(blocks, self.rows, self.n, stream=stream)

    def __call__(self, q: torch.Tensor, d: torch.Tensor, out: torch.Tensor | None = None, stream=None):
        if q.dim() == 1 or q.shape[0] == 1:
            return gemv(self.packed, self.rows, self.n, q, d, out, stream)
        return gemm_small(self.packed, self.rows, self.n, q, d, out, stream)
