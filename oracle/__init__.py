"""CPU oracle for the Q1_0 x q8_0 product (ctypes wrapper over q1_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The library
(``decode_q1_gemv_gb300``) never imports it, and it never imports the library:
the two share no code.  See ``q1_oracle.c`` for the definition it implements
and the passages of bankML's "docs/modules/gpu.md" it follows.

Every function takes and returns numpy arrays:
  blocks  uint8  [rows, n/128, 18]   Q1_0 blocks (fp16 scale LE + 16 sign bytes)
  tblocks uint8  [rows, n/128, 34]   Q2_0 blocks (fp16 scale LE + 32 bytes of 2-bit
                                     codes 0/1/2 = -1/0/+1), the q2_* functions
  q       int8   [n] or [B, n]       q8_0 quants
  d       uint16 [n/32] or [B, n/32] fp16 scale bits
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q1_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libq1oracle.so")

# No contraction and no fast-math: the oracle's rounding must be the C
# source's rounding, on x86-64 and on aarch64 alike.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-pthread", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/libq1oracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.q1o_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q1o_f16_to_f32.restype = ctypes.c_float
        lib.q1o_f32_to_f16_rne.argtypes = [ctypes.c_float]
        lib.q1o_f32_to_f16_rne.restype = ctypes.c_uint16
        lib.q1o_f32_to_f16_rne_n.argtypes = [P, I64, P]
        lib.q1o_f32_to_f16_rne_n.restype = None
        lib.q1o_f16_to_f32_n.argtypes = [P, I64, P]
        lib.q1o_f16_to_f32_n.restype = None
        lib.q1o_q8_quantize.argtypes = [P, I64, P, P]
        lib.q1o_q8_quantize.restype = None
        lib.q1o_weight.argtypes = [P, I64, I64, I64]
        lib.q1o_weight.restype = ctypes.c_float
        lib.q1o_dot_row.argtypes = [P, I64, P, P]
        lib.q1o_dot_row.restype = ctypes.c_float
        lib.q1o_dot_row_variant.argtypes = [P, I64, P, P, ctypes.c_int]
        lib.q1o_dot_row_variant.restype = ctypes.c_float
        lib.q1o_dot_row_lanes.argtypes = [P, I64, P, P, P]
        lib.q1o_dot_row_lanes.restype = None
        lib.q1o_lane_sums.argtypes = [P, I64, P, P]
        lib.q1o_lane_sums.restype = None
        lib.q1o_gemv.argtypes = [P, I64, I64, P, P, P]
        lib.q1o_gemv.restype = None
        lib.q1o_gemm.argtypes = [P, I64, I64, I64, P, P, P]
        lib.q1o_gemm.restype = None
        lib.q1o_rows_sampled.argtypes = [P, I64, I64, P, P, P, P, P]
        lib.q1o_rows_sampled.restype = None
        lib.q1o_gemv_threaded.argtypes = [P, I64, I64, P, P, P, ctypes.c_int]
        lib.q1o_gemv_threaded.restype = ctypes.c_longlong
        lib.q1o_gemm_threaded.argtypes = [P, I64, I64, I64, P, P, P, ctypes.c_int]
        lib.q1o_gemm_threaded.restype = ctypes.c_longlong
        lib.q2o_gemv_threaded.argtypes = [P, I64, I64, P, P, P, ctypes.c_int]
        lib.q2o_gemv_threaded.restype = ctypes.c_longlong
        lib.q2o_weight.argtypes = [P, I64, I64, I64]
        lib.q2o_weight.restype = ctypes.c_float
        lib.q2o_dot_row.argtypes = [P, I64, P, P]
        lib.q2o_dot_row.restype = ctypes.c_float
        lib.q2o_lane_sums.argtypes = [P, I64, P, P]
        lib.q2o_lane_sums.restype = None
        lib.q2o_gemv.argtypes = [P, I64, I64, P, P, P]
        lib.q2o_gemv.restype = None
        lib.q2o_rows_sampled.argtypes = [P, I64, I64, P, P, P, P]
        lib.q2o_rows_sampled.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check_blocks(blocks: np.ndarray):
    if blocks.ndim != 3 or blocks.shape[2] != 18:
        raise ValueError("blocks must be uint8 [rows, n/128, 18]")
    return blocks.shape[0], blocks.shape[1] * 128


# ---------------------------------------------------------------- scalars --
def f16_to_f32(h: int) -> float:
    return float(_load().q1o_f16_to_f32(int(h)))


def f32_to_f16(x) -> int:
    return int(_load().q1o_f32_to_f16_rne(ctypes.c_float(float(np.float32(x)))))


def f32_to_f16_array(x: np.ndarray) -> np.ndarray:
    """fp16 RNE bit patterns of every element of a float32 array."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().q1o_f32_to_f16_rne_n(_ptr(x), x.size, _ptr(out))
    return out


def f16_to_f32_array(h: np.ndarray) -> np.ndarray:
    """float32 values of an array of fp16 bit patterns."""
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().q1o_f16_to_f32_n(_ptr(h), h.size, _ptr(out))
    return out


# ------------------------------------------------------------ activations --
def q8_quantize(x: np.ndarray):
    """q8_0 quantization of the last axis.  Returns (q int8, d uint16 fp16 bits)."""
    x = _c(x, np.float32)
    n = x.shape[-1]
    if n % 32:
        raise ValueError("n must be a multiple of 32")
    q = np.empty(x.shape, dtype=np.int8)
    d = np.empty(x.shape[:-1] + (n // 32,), dtype=np.uint16)
    lib = _load()
    xs = x.reshape(-1, n)
    qs = q.reshape(-1, n)
    ds = d.reshape(-1, n // 32)
    for v in range(xs.shape[0]):
        lib.q1o_q8_quantize(_ptr(xs[v]), n, _ptr(qs[v]), _ptr(ds[v]))
    return q, d


# ---------------------------------------------------------------- weights --
def weight(blocks: np.ndarray, r: int, j: int) -> float:
    rows, n = _check_blocks(blocks)
    blocks = _c(blocks, np.uint8)
    return float(_load().q1o_weight(_ptr(blocks), n, int(r), int(j)))


# ------------------------------------------------------------ dot products --
def dot_row(blocks_row: np.ndarray, q: np.ndarray, d: np.ndarray, variant: int = 0) -> np.float32:
    """One row: blocks_row uint8 [nb, 18]."""
    blocks_row = _c(blocks_row, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    nb = blocks_row.shape[0]
    if q.size != nb * 128 or d.size != nb * 4:
        raise ValueError("shape mismatch")
    lib = _load()
    if variant:
        return np.float32(lib.q1o_dot_row_variant(_ptr(blocks_row), nb, _ptr(q), _ptr(d), int(variant)))
    return np.float32(lib.q1o_dot_row(_ptr(blocks_row), nb, _ptr(q), _ptr(d)))


def dot_row_lanes(blocks_row: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    blocks_row = _c(blocks_row, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    out = np.empty(8, dtype=np.float32)
    _load().q1o_dot_row_lanes(_ptr(blocks_row), blocks_row.shape[0], _ptr(q), _ptr(d), _ptr(out))
    return out


def lane_sums(blocks_row: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Exact integer lane sums, int32 [nb, 4, 8]."""
    blocks_row = _c(blocks_row, np.uint8)
    q = _c(q, np.int8)
    nb = blocks_row.shape[0]
    out = np.empty((nb, 4, 8), dtype=np.int32)
    _load().q1o_lane_sums(_ptr(blocks_row), nb, _ptr(q), _ptr(out))
    return out


def gemv(blocks: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    rows, n = _check_blocks(blocks)
    blocks = _c(blocks, np.uint8)
    q = _c(q, np.int8).ravel()
    d = _c(d, np.uint16).ravel()
    if q.size != n or d.size != n // 32:
        raise ValueError("activation shape mismatch")
    out = np.empty(rows, dtype=np.float32)
    _load().q1o_gemv(_ptr(blocks), rows, n, _ptr(q), _ptr(d), _ptr(out))
    return out


def gemm(blocks: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Batched: q int8 [B, n], d uint16 [B, n/32] -> out float32 [B, rows]."""
    rows, n = _check_blocks(blocks)
    blocks = _c(blocks, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    nvec = q.shape[0]
    if q.shape != (nvec, n) or d.shape != (nvec, n // 32):
        raise ValueError("activation shape mismatch")
    out = np.empty((nvec, rows), dtype=np.float32)
    _load().q1o_gemm(_ptr(blocks), rows, n, nvec, _ptr(q), _ptr(d), _ptr(out))
    return out


def rows_sampled(blocks: np.ndarray, idx, q: np.ndarray, d: np.ndarray, vec_of=None) -> np.ndarray:
    """out[i] = dot(row idx[i], vector vec_of[i]) (vector 0 if vec_of is None)."""
    rows, n = _check_blocks(blocks)
    blocks = np.ascontiguousarray(blocks)
    if blocks.dtype != np.uint8:
        raise ValueError("blocks must be uint8")
    idx = _c(idx, np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= rows):
        raise ValueError("row index out of range")
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    nvec = q.size // n
    vptr = None
    if vec_of is not None:
        vec_of = _c(vec_of, np.int64)
        if vec_of.size != idx.size or (vec_of.size and (vec_of.min() < 0 or vec_of.max() >= nvec)):
            raise ValueError("vector index out of range")
        vptr = _ptr(vec_of)
    out = np.empty(idx.size, dtype=np.float32)
    _load().q1o_rows_sampled(_ptr(blocks), n, idx.size, _ptr(idx), vptr, _ptr(q), _ptr(d), _ptr(out))
    return out


def gemv_threaded(blocks: np.ndarray, q: np.ndarray, d: np.ndarray, threads: int,
                  out: np.ndarray | None = None):
    """Threaded oracle (16-row chunks from an atomic counter).

    Returns (out, rows_written).  ``out`` may be passed in (pre-filled with a
    sentinel) so a test can check that every row is written exactly once."""
    rows, n = _check_blocks(blocks)
    blocks = _c(blocks, np.uint8)
    q = _c(q, np.int8).ravel()
    d = _c(d, np.uint16).ravel()
    if out is None:
        out = np.empty(rows, dtype=np.float32)
    if out.dtype != np.float32 or not out.flags.c_contiguous or out.size < rows:
        raise ValueError("out must be contiguous float32 with at least `rows` elements")
    done = _load().q1o_gemv_threaded(_ptr(blocks), rows, n, _ptr(q), _ptr(d), _ptr(out), int(threads))
    return out, int(done)


def default_threads() -> int:
    return os.cpu_count() or 1


def gemm_threaded(blocks: np.ndarray, q: np.ndarray, d: np.ndarray, threads: int | None = None) -> np.ndarray:
    """Batched product on `threads` threads (16-row claims, every vector of a
    claimed row by the single-thread row function): float32 [B, rows],
    bit-identical to ``gemm``."""
    rows, n = _check_blocks(blocks)
    blocks = _c(blocks, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    if q.ndim == 1:
        q, d = q[None, :], d[None, :]
    nvec = q.shape[0]
    if q.shape != (nvec, n) or d.shape != (nvec, n // 32):
        raise ValueError("activation shape mismatch")
    out = np.empty((nvec, rows), dtype=np.float32)
    done = _load().q1o_gemm_threaded(_ptr(blocks), rows, n, nvec, _ptr(q), _ptr(d), _ptr(out),
                                     int(threads or default_threads()))
    if done != rows:
        raise RuntimeError("threaded oracle did not write every row")
    return out


# ------------------------------------------------------- Q2_0 (ternary) --
def _check_tblocks(tblocks: np.ndarray):
    if tblocks.ndim != 3 or tblocks.shape[2] != 34:
        raise ValueError("tblocks must be uint8 [rows, n/128, 34]")
    return tblocks.shape[0], tblocks.shape[1] * 128


def q2_weight(tblocks: np.ndarray, r: int, j: int) -> float:
    rows, n = _check_tblocks(tblocks)
    tblocks = _c(tblocks, np.uint8)
    return float(_load().q2o_weight(_ptr(tblocks), n, int(r), int(j)))


def q2_dot_row(tblocks_row: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.float32:
    """One Q2_0 row: tblocks_row uint8 [nb, 34]."""
    tblocks_row = _c(tblocks_row, np.uint8)
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    nb = tblocks_row.shape[0]
    if q.size != nb * 128 or d.size != nb * 4:
        raise ValueError("shape mismatch")
    return np.float32(_load().q2o_dot_row(_ptr(tblocks_row), nb, _ptr(q), _ptr(d)))


def q2_lane_sums(tblocks_row: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Exact integer lane sums of one Q2_0 row, int32 [nb, 4, 8]."""
    tblocks_row = _c(tblocks_row, np.uint8)
    q = _c(q, np.int8)
    nb = tblocks_row.shape[0]
    out = np.empty((nb, 4, 8), dtype=np.int32)
    _load().q2o_lane_sums(_ptr(tblocks_row), nb, _ptr(q), _ptr(out))
    return out


def q2_gemv(tblocks: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    rows, n = _check_tblocks(tblocks)
    tblocks = _c(tblocks, np.uint8)
    q = _c(q, np.int8).ravel()
    d = _c(d, np.uint16).ravel()
    if q.size != n or d.size != n // 32:
        raise ValueError("activation shape mismatch")
    out = np.empty(rows, dtype=np.float32)
    _load().q2o_gemv(_ptr(tblocks), rows, n, _ptr(q), _ptr(d), _ptr(out))
    return out


def q2_gemv_threaded(tblocks: np.ndarray, q: np.ndarray, d: np.ndarray, threads: int | None = None) -> np.ndarray:
    """Q2_0 matrix-vector product on `threads` threads, bit-identical to ``q2_gemv``."""
    rows, n = _check_tblocks(tblocks)
    tblocks = _c(tblocks, np.uint8)
    q = _c(q, np.int8).ravel()
    d = _c(d, np.uint16).ravel()
    if q.size != n or d.size != n // 32:
        raise ValueError("activation shape mismatch")
    out = np.empty(rows, dtype=np.float32)
    done = _load().q2o_gemv_threaded(_ptr(tblocks), rows, n, _ptr(q), _ptr(d), _ptr(out),
                                     int(threads or default_threads()))
    if done != rows:
        raise RuntimeError("threaded oracle did not write every row")
    return out


def q2_rows_sampled(tblocks: np.ndarray, idx, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """out[i] = dot(row idx[i], (q, d)) for a Q2_0 matrix."""
    rows, n = _check_tblocks(tblocks)
    tblocks = np.ascontiguousarray(tblocks)
    idx = _c(idx, np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= rows):
        raise ValueError("row index out of range")
    q = _c(q, np.int8).ravel()
    d = _c(d, np.uint16).ravel()
    out = np.empty(idx.size, dtype=np.float32)
    _load().q2o_rows_sampled(_ptr(tblocks), n, idx.size, _ptr(idx), _ptr(q), _ptr(d), _ptr(out))
    return out
