"""Ring all-reduce oracle — TEST INFRASTRUCTURE ONLY.

A plain CPU simulation of the ring schedule (one thread per rank, unbounded
channels between neighbours) written from the tirogla.com page "Ring
all-reduce", section "How it works", plus the plain per-element definition
(``fold_at``). Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package. It shares no code with
the CUDA library in ``ring_all_reduce_02_gb300``; the two meet only through
the seeded input generators.

Buffers are numpy arrays in the dtype's storage: float32, float16, int32, and
bf16 as uint16 bit patterns (numpy has no bfloat16), selected with
``dtype="bf16"``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.cpp")
_LIB = os.path.join(_HERE, "libring_oracle.so")

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}
OPS = {"sum": 0, "avg": 1, "min": 2, "max": 3, "prod": 4}
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i32": np.int32}
STATUS = {0: "ok", 1: "invalid", 2: "unsupported", 3: "timeout", 4: "protocol", 5: "faulted"}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: oracle status {code} ({STATUS.get(code, '?')})")
        self.code = code
        self.status = STATUS.get(code, "?")


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain IEEE arithmetic: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", _LIB + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P, U64, I = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
            PP = ctypes.POINTER(ctypes.c_void_p)
            lib.ra_oracle_chunk_range.argtypes = [U64, I, I, ctypes.POINTER(U64), ctypes.POINTER(U64)]
            lib.ra_oracle_allreduce.argtypes = [PP, PP, U64, I, I, I, I, P, P, I, I]
            lib.ra_oracle_reduce_scatter.argtypes = [PP, PP, U64, I, I, I, I, P]
            lib.ra_oracle_allgather.argtypes = [PP, PP, U64, I, I, I, P, P]
            lib.ra_oracle_fold_at.argtypes = [PP, U64, I, I, I, P, U64, P]
            lib.ra_oracle_allreduce_ex.argtypes = [PP, PP, U64, I, I, I, I, I, I, P]
            lib.ra_oracle_allreduce_ex.restype = ctypes.c_int
            lib.ra_oracle_hop.argtypes = [I, I, P, P, P, U64]
            lib.ra_oracle_round.argtypes = [I, P, P, U64]
            lib.ra_oracle_widen.argtypes = [I, P, P, U64]
            for f in (lib.ra_oracle_chunk_range, lib.ra_oracle_allreduce, lib.ra_oracle_reduce_scatter,
                      lib.ra_oracle_allgather, lib.ra_oracle_fold_at, lib.ra_oracle_hop,
                      lib.ra_oracle_round, lib.ra_oracle_widen):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check_inputs(xs, dtype, length=None):
    want = STORAGE[dtype]
    for x in xs:
        if x.dtype != want or not x.flags.c_contiguous or x.ndim != 1:
            raise TypeError(f"oracle input must be 1-D contiguous {want.__name__} for {dtype}")
        if length is not None and x.shape[0] != length:
            raise ValueError("all ranks' buffers must have the same length")


def chunk_range(length: int, n: int, c: int) -> tuple[int, int]:
    lib = _load()
    b, e = ctypes.c_uint64(), ctypes.c_uint64()
    st = lib.ra_oracle_chunk_range(length, n, c, ctypes.byref(b), ctypes.byref(e))
    if st:
        raise OracleError(st, "chunk_range")
    return b.value, e.value


def allreduce(xs, op: str, dtype: str, timeout_ms: int = 10000, snapshots: bool = False,
              fault_rank: int = -1, fault_step: int = -1, inplace: bool = False):
    """Ring all-reduce of the N arrays ``xs``. Returns (outs, bytes_sent[N], snaps).

    ``snaps`` (if requested) has shape [2(N-1), N, L]: every rank's buffer after
    every reduce-scatter step, then after every all-gather step.
    """
    lib = _load()
    n = len(xs)
    length = xs[0].shape[0] if n else 0
    _check_inputs(xs, dtype, length)
    outs = xs if inplace else [np.empty_like(x) for x in xs]
    sent = np.zeros(max(n, 1), dtype=np.uint64)
    snaps = np.zeros((max(2 * (n - 1), 0), n, length), dtype=STORAGE[dtype]) if snapshots else None
    st = lib.ra_oracle_allreduce(_ptrs(xs), _ptrs(outs), length, DTYPES[dtype], OPS[op], n, timeout_ms,
                                 sent.ctypes.data, snaps.ctypes.data if snapshots else None,
                                 fault_rank, fault_step)
    if st:
        raise OracleError(st, "allreduce")
    return outs, sent[:n], snaps


ORDERS = {"ring": 0, "tree": 1, "rabenseifner": 2}
ACCUMS = {"dtype": 0, "fp32": 1}


def allreduce_ex(xs, op: str, dtype: str, order: str = "ring", accum: str = "dtype", timeout_ms: int = 10000):
    """All-reduce by another algorithm or accumulation: order ring | tree (double binary tree) |
    rabenseifner (power-of-two N); accum dtype | fp32 (ring only). Returns (outs, bytes_sent)."""
    lib = _load()
    n = len(xs)
    length = xs[0].shape[0] if n else 0
    _check_inputs(xs, dtype, length)
    outs = [np.empty_like(x) for x in xs]
    sent = np.zeros(max(n, 1), dtype=np.uint64)
    st = lib.ra_oracle_allreduce_ex(_ptrs(xs), _ptrs(outs), length, DTYPES[dtype], OPS[op], n, ORDERS[order],
                                    ACCUMS[accum], timeout_ms, sent.ctypes.data)
    if st:
        raise OracleError(st, "allreduce_ex")
    return outs, sent[:n]


def reduce_scatter(xs, op: str, dtype: str, timeout_ms: int = 10000):
    """Ring reduce-scatter: returns (shards, bytes_sent); shards[r] is chunk r, compact."""
    lib = _load()
    n = len(xs)
    length = xs[0].shape[0]
    _check_inputs(xs, dtype, length)
    outs = []
    for r in range(n):
        b, e = chunk_range(length, n, r)
        outs.append(np.empty(e - b, dtype=STORAGE[dtype]))
    sent = np.zeros(n, dtype=np.uint64)
    # a zero-length shard still needs a valid host address for the ctypes array
    ptr_outs = [o if o.size else np.empty(1, dtype=o.dtype) for o in outs]
    st = lib.ra_oracle_reduce_scatter(_ptrs(xs), _ptrs(ptr_outs), length, DTYPES[dtype], OPS[op], n,
                                      timeout_ms, sent.ctypes.data)
    if st:
        raise OracleError(st, "reduce_scatter")
    return outs, sent


def allgather(shards, length: int, dtype: str, timeout_ms: int = 10000, snapshots: bool = False):
    """Standalone ring all-gather of compact shards (shard r = chunk r). Returns (outs, bytes_sent, snaps)."""
    lib = _load()
    n = len(shards)
    _check_inputs(shards, dtype)
    for r, s in enumerate(shards):
        b, e = chunk_range(length, n, r)
        if s.shape[0] != e - b:
            raise ValueError(f"shard {r} must hold {e - b} elements")
    outs = [np.empty(length, dtype=STORAGE[dtype]) for _ in range(n)]
    sent = np.zeros(n, dtype=np.uint64)
    snaps = np.zeros((max(n - 1, 0), n, length), dtype=STORAGE[dtype]) if snapshots else None
    ptr_in = [s if s.size else np.empty(1, dtype=s.dtype) for s in shards]
    st = lib.ra_oracle_allgather(_ptrs(ptr_in), _ptrs(outs), length, DTYPES[dtype], n, timeout_ms,
                                 sent.ctypes.data, snaps.ctypes.data if snapshots else None)
    if st:
        raise OracleError(st, "allgather")
    return outs, sent, snaps


def fold_at(xs, op: str, dtype: str, idx) -> np.ndarray:
    """The plain per-element definition (ring-order left fold) at indices ``idx``."""
    lib = _load()
    n = len(xs)
    length = xs[0].shape[0]
    _check_inputs(xs, dtype, length)
    idx = np.ascontiguousarray(idx, dtype=np.uint64)
    out = np.empty(idx.shape[0], dtype=STORAGE[dtype])
    st = lib.ra_oracle_fold_at(_ptrs(xs), length, DTYPES[dtype], OPS[op], n, idx.ctypes.data,
                               idx.shape[0], out.ctypes.data)
    if st:
        raise OracleError(st, "fold_at")
    return out


def hop(dtype: str, op: str, partial: np.ndarray, local: np.ndarray) -> np.ndarray:
    """One ring hop, element-wise, storage-typed (partial is the incoming operand)."""
    lib = _load()
    partial = np.ascontiguousarray(partial, dtype=STORAGE[dtype])
    local = np.ascontiguousarray(local, dtype=STORAGE[dtype])
    out = np.empty_like(partial)
    st = lib.ra_oracle_hop(DTYPES[dtype], OPS[op], partial.ctypes.data, local.ctypes.data,
                           out.ctypes.data, partial.size)
    if st:
        raise OracleError(st, "hop")
    return out


def round_f32(dtype: str, x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16/bf16 bit patterns, round to nearest even (the oracle's own code)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    st = lib.ra_oracle_round(DTYPES[dtype], x.ctypes.data, out.ctypes.data, x.size)
    if st:
        raise OracleError(st, "round")
    return out


def widen(dtype: str, h: np.ndarray) -> np.ndarray:
    """fp16/bf16 bit patterns -> fp32 (exact)."""
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    st = lib.ra_oracle_widen(DTYPES[dtype], h.ctypes.data, out.ctypes.data, h.size)
    if st:
        raise OracleError(st, "widen")
    return out
