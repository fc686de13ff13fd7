"""Python binding of libra.so: argument marshalling only.

The functions carry the C ABI's names (include/ra.h). Tensors supply device
pointers (``data_ptr()``) and the stream is torch's current CUDA stream unless
one is given; every step of the collective runs in the library's kernels.
The library must be built (``python -m ring_all_reduce_02_gb300.build``); if
it is missing, the first call raises instead of falling back to anything.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libra.so")

RA_SUCCESS, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_ALIAS, RA_ERR_CUDA, RA_ERR_SCRATCH_LIMIT = range(6)
RA_NOALLOC_STATUS_WORDS = 16
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}
OP_CODES = {"sum": 0, "avg": 1, "min": 2, "max": 3, "prod": 4}
ORDER_CODES = {"ring": 0, "tree": 1, "rabenseifner": 2}
ACCUM_CODES = {"dtype": 0, "fp32": 1}
RA_MAX_RANKS = 64

# every symbol include/ra.h declares
EXPORTS = ("ra_allreduce", "ra_reduce_scatter", "ra_allgather", "ra_allreduce_ex", "ra_reduce_scatter_ex",
           "ra_bucket_plan", "ra_allreduce_buckets", "ra_allreduce_ringsteps", "ra_chunk_range", "ra_plan_chunk",
           "ra_status_string", "ra_last_cuda_error", "ra_vector_bytes", "ra_selftest_bulk_timeout",
           "ra_allreduce_bulk_noalloc")
ENGINE_CODES = {"registers": 0, "bulk": 1}


class Options(ctypes.Structure):
    """ra_options_t."""

    _fields_ = [("order", ctypes.c_int), ("accum", ctypes.c_int), ("max_sms", ctypes.c_int),
                ("engine", ctypes.c_int), ("status", ctypes.c_void_p)]


def options(order: str = "ring", accum: str = "dtype", max_sms: int = 0, engine: str = "registers",
            status=None) -> Options:
    """ra_options_t; ``status`` is a device int32 tensor (or address) for the bulk engine."""
    st = status.data_ptr() if hasattr(status, "data_ptr") else status
    return Options(ORDER_CODES[order], ACCUM_CODES[accum], max_sms, ENGINE_CODES[engine], st or None)


class RaError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        name = lib().ra_status_string(status).decode()
        extra = f" (cudaError {lib().ra_last_cuda_error()})" if status == RA_ERR_CUDA else ""
        super().__init__(f"{call}: {name}{extra}")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m ring_all_reduce_02_gb300.build` (no fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            VP, SZ, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            PP = ctypes.POINTER(ctypes.c_void_p)
            PSZ = ctypes.POINTER(ctypes.c_size_t)
            POPT = ctypes.POINTER(Options)
            for name in ("ra_allreduce", "ra_reduce_scatter", "ra_allgather"):
                f = getattr(L, name)
                f.argtypes = [PP, PP, SZ, I, I, I, VP]
                f.restype = I
            for name in ("ra_allreduce_ex", "ra_reduce_scatter_ex"):
                f = getattr(L, name)
                f.argtypes = [PP, PP, SZ, I, I, I, POPT, VP]
                f.restype = I
            L.ra_bucket_plan.argtypes = [PSZ, I, SZ, I, PSZ, PSZ, I, ctypes.POINTER(I)]
            L.ra_bucket_plan.restype = I
            L.ra_allreduce_buckets.argtypes = [PP, PP, SZ, I, I, I, I, PSZ, PSZ, PP, POPT, VP]
            L.ra_allreduce_buckets.restype = I
            L.ra_allreduce_ringsteps.argtypes = [PP, PP, SZ, I, I, I, I, VP]
            L.ra_allreduce_ringsteps.restype = I
            L.ra_chunk_range.argtypes = [SZ, I, I, PSZ, PSZ]
            L.ra_chunk_range.restype = I
            L.ra_plan_chunk.argtypes = [SZ, I, I, I, I, I, PSZ, PSZ, PSZ, PSZ]
            L.ra_plan_chunk.restype = I
            L.ra_status_string.argtypes = [I]
            L.ra_status_string.restype = ctypes.c_char_p
            L.ra_last_cuda_error.argtypes = []
            L.ra_last_cuda_error.restype = I
            L.ra_vector_bytes.argtypes = []
            L.ra_vector_bytes.restype = I
            L.ra_selftest_bulk_timeout.argtypes = [PP, PP, SZ, I, I, I, I, VP, I, VP]
            L.ra_selftest_bulk_timeout.restype = I
            L.ra_allreduce_bulk_noalloc.argtypes = [PP, PP, SZ, I, I, I, I, VP, VP]
            L.ra_allreduce_bulk_noalloc.restype = I
            _lib = L
    return _lib


def ptr_array(ptrs) -> ctypes.Array:
    return (ctypes.c_void_p * len(ptrs))(*[int(p) if p else None for p in ptrs])


def dtype_code(t) -> int:
    import torch

    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.int32: 3}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _stream_ptr(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(tensors, what):
    dt = tensors[0].dtype
    for t in tensors:
        if not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
            raise ValueError(f"{what}: every buffer must be a CUDA tensor or pinned host memory")
        if t.dtype != dt:
            raise ValueError(f"{what}: all buffers must share one dtype")
        if not t.is_contiguous():
            raise ValueError(f"{what}: buffers must be contiguous")


def _check_full(sendbufs, recvbufs, what):
    _check(list(sendbufs) + list(recvbufs), what)
    count = sendbufs[0].numel()
    if any(t.numel() != count for t in list(sendbufs) + list(recvbufs)) or len(recvbufs) != len(sendbufs):
        raise ValueError(f"{what}: N send and N recv buffers of one length")
    return count


def _chunk_len(count: int, n: int, c: int) -> int:
    return (c + 1) * count // n - c * count // n


def call(name: str, send_ptrs, recv_ptrs, count: int, dtype: int, op: int, nranks: int, stream: int) -> int:
    """Raw C call with integer pointers; returns the ra_status_t."""
    f = getattr(lib(), name)
    return f(ptr_array(send_ptrs), ptr_array(recv_ptrs), count, dtype, op, nranks, ctypes.c_void_p(stream or None))


def call_ex(name: str, send_ptrs, recv_ptrs, count: int, dtype: int, op: int, nranks: int, order: int,
            accum: int, stream: int, max_sms: int = 0, engine: int = 0, status: int = 0) -> int:
    """Raw C call of ra_allreduce_ex / ra_reduce_scatter_ex; returns the ra_status_t."""
    f = getattr(lib(), name)
    opts = Options(order, accum, max_sms, engine, status or None)
    return f(ptr_array(send_ptrs), ptr_array(recv_ptrs), count, dtype, op, nranks, ctypes.byref(opts),
             ctypes.c_void_p(stream or None))


def ra_allreduce(sendbufs, recvbufs, op: str = "sum", stream=None) -> None:
    """All-reduce of N equal-length tensors into N tensors (recv may be send: in place)."""
    count = _check_full(sendbufs, recvbufs, "ra_allreduce")
    st = call("ra_allreduce", [t.data_ptr() for t in sendbufs], [t.data_ptr() for t in recvbufs], count,
              dtype_code(sendbufs[0]), OP_CODES[op], len(sendbufs), _stream_ptr(stream))
    if st:
        raise RaError(st, "ra_allreduce")


def ra_allreduce_ex(sendbufs, recvbufs, op: str = "sum", order: str = "ring", accum: str = "dtype",
                    max_sms: int = 0, engine: str = "registers", status=None, stream=None) -> None:
    """All-reduce with a reduction order (ring | tree | rabenseifner), accumulation (dtype | fp32),
    an SM budget (0 = all SMs) and an engine (registers | bulk; bulk needs a device int32 ``status``)."""
    count = _check_full(sendbufs, recvbufs, "ra_allreduce_ex")
    st_ptr = status.data_ptr() if status is not None else 0
    st = call_ex("ra_allreduce_ex", [t.data_ptr() for t in sendbufs], [t.data_ptr() for t in recvbufs], count,
                 dtype_code(sendbufs[0]), OP_CODES[op], len(sendbufs), ORDER_CODES[order], ACCUM_CODES[accum],
                 _stream_ptr(stream), max_sms, ENGINE_CODES[engine], st_ptr)
    if st:
        raise RaError(st, "ra_allreduce_ex")


def ra_reduce_scatter(sendbufs, recvbufs, op: str = "sum", stream=None) -> None:
    """Reduce-scatter: recvbufs[r] receives chunk r (compact) of the reduction."""
    _check(list(sendbufs) + [t for t in recvbufs if t.numel()], "ra_reduce_scatter")
    count, n = sendbufs[0].numel(), len(sendbufs)
    for r, t in enumerate(recvbufs):
        if t.numel() != _chunk_len(count, n, r):
            raise ValueError(f"ra_reduce_scatter: recvbufs[{r}] must hold chunk {r}")
    st = call("ra_reduce_scatter", [t.data_ptr() for t in sendbufs], [t.data_ptr() for t in recvbufs], count,
              dtype_code(sendbufs[0]), OP_CODES[op], n, _stream_ptr(stream))
    if st:
        raise RaError(st, "ra_reduce_scatter")


def ra_reduce_scatter_ex(sendbufs, recvbufs, op: str = "sum", order: str = "ring", accum: str = "dtype",
                         max_sms: int = 0, stream=None) -> None:
    """Reduce-scatter with a reduction order, accumulation and SM budget; recvbufs[r] receives chunk r."""
    _check(list(sendbufs) + [t for t in recvbufs if t.numel()], "ra_reduce_scatter_ex")
    count, n = sendbufs[0].numel(), len(sendbufs)
    for r, t in enumerate(recvbufs):
        if t.numel() != _chunk_len(count, n, r):
            raise ValueError(f"ra_reduce_scatter_ex: recvbufs[{r}] must hold chunk {r}")
    st = call_ex("ra_reduce_scatter_ex", [t.data_ptr() for t in sendbufs], [t.data_ptr() for t in recvbufs],
                 count, dtype_code(sendbufs[0]), OP_CODES[op], n, ORDER_CODES[order], ACCUM_CODES[accum],
                 _stream_ptr(stream), max_sms)
    if st:
        raise RaError(st, "ra_reduce_scatter_ex")


def ra_allgather(sendbufs, recvbufs, stream=None) -> None:
    """All-gather: sendbufs[r] is chunk r (compact); every recvbufs[r] receives all chunks."""
    _check([t for t in sendbufs if t.numel()] + list(recvbufs), "ra_allgather")
    count, n = recvbufs[0].numel(), len(recvbufs)
    for r, t in enumerate(sendbufs):
        if t.numel() != _chunk_len(count, n, r):
            raise ValueError(f"ra_allgather: sendbufs[{r}] must hold chunk {r}")
    st = call("ra_allgather", [t.data_ptr() for t in sendbufs], [t.data_ptr() for t in recvbufs], count,
              dtype_code(recvbufs[0]), OP_CODES["sum"], n, _stream_ptr(stream))
    if st:
        raise RaError(st, "ra_allgather")


def ra_allreduce_ringsteps(sendbufs, recvbufs, op: str = "sum", nsteps: int = -1, stream=None) -> None:
    """The literal ring schedule, one launch per step (first ``nsteps`` of 2(N-1); -1 = all)."""
    count = _check_full(sendbufs, recvbufs, "ra_allreduce_ringsteps")
    st = lib().ra_allreduce_ringsteps(ptr_array([t.data_ptr() for t in sendbufs]),
                                      ptr_array([t.data_ptr() for t in recvbufs]), count,
                                      dtype_code(sendbufs[0]), OP_CODES[op], len(sendbufs), nsteps,
                                      ctypes.c_void_p(_stream_ptr(stream) or None))
    if st:
        raise RaError(st, "ra_allreduce_ringsteps")


def ra_bucket_plan(param_counts, bucket_bytes: int, elem_size: int):
    """DDP-style buckets over a flat buffer: list of (begin, count) in the order they become ready."""
    n = len(param_counts)
    counts = (ctypes.c_size_t * max(n, 1))(*param_counts)
    nb = ctypes.c_int()
    st = lib().ra_bucket_plan(counts, n, bucket_bytes, elem_size, None, None, 0, ctypes.byref(nb))
    if st and not (st == RA_ERR_INVALID_ARG and nb.value > 0):
        raise RaError(st, "ra_bucket_plan")
    m = nb.value
    begin = (ctypes.c_size_t * max(m, 1))()
    cnt = (ctypes.c_size_t * max(m, 1))()
    st = lib().ra_bucket_plan(counts, n, bucket_bytes, elem_size, begin, cnt, m, ctypes.byref(nb))
    if st:
        raise RaError(st, "ra_bucket_plan")
    return [(begin[b], cnt[b]) for b in range(m)]


def ra_allreduce_buckets(sendbufs, recvbufs, buckets, op: str = "sum", ready_events=None, order: str = "ring",
                         accum: str = "dtype", max_sms: int = 0, engine: str = "registers", status=None,
                         stream=None) -> None:
    """All-reduce every bucket (begin, count) of the flat buffers, each after its ready event."""
    count = _check_full(sendbufs, recvbufs, "ra_allreduce_buckets")
    m = len(buckets)
    begin = (ctypes.c_size_t * max(m, 1))(*[b for b, _ in buckets])
    cnt = (ctypes.c_size_t * max(m, 1))(*[c for _, c in buckets])
    events = None
    if ready_events is not None:
        events = ptr_array([int(e.cuda_event) if e is not None else 0 for e in ready_events])
    opts = options(order, accum, max_sms, engine, status)
    st = lib().ra_allreduce_buckets(ptr_array([t.data_ptr() for t in sendbufs]),
                                    ptr_array([t.data_ptr() for t in recvbufs]), count, dtype_code(sendbufs[0]),
                                    OP_CODES[op], len(sendbufs), m, begin, cnt, events, ctypes.byref(opts),
                                    ctypes.c_void_p(_stream_ptr(stream) or None))
    if st:
        raise RaError(st, "ra_allreduce_buckets")


def ra_chunk_range(count: int, nranks: int, c: int) -> tuple[int, int]:
    b, e = ctypes.c_size_t(), ctypes.c_size_t()
    st = lib().ra_chunk_range(count, nranks, c, ctypes.byref(b), ctypes.byref(e))
    if st:
        raise RaError(st, "ra_chunk_range")
    return b.value, e.value


def ra_plan_chunk(count: int, nranks: int, c: int, elem_size: int, phase_bytes: int, align_bytes: int = 0):
    """(begin, end, vec_begin, vec_end) of chunk c: which part takes the vector path. ``align_bytes``
    is the grid's alignment (a power of two from ra_vector_bytes() to 512; 0: ra_vector_bytes())."""
    align_bytes = align_bytes or lib().ra_vector_bytes()
    out = [ctypes.c_size_t() for _ in range(4)]
    st = lib().ra_plan_chunk(count, nranks, c, elem_size, align_bytes, phase_bytes, *[ctypes.byref(o) for o in out])
    if st:
        raise RaError(st, "ra_plan_chunk")
    return tuple(o.value for o in out)


def ra_status_string(status: int) -> str:
    return lib().ra_status_string(status).decode()


def ra_selftest_bulk_timeout(sendbufs, recvbufs, status, op: str = "sum", withhold_chunk: int = 0,
                             per_chunk: bool = False, stream=None) -> None:
    """Run the bulk engine with chunk ``withhold_chunk``'s first tile withheld: that chunk's bounded
    wait must give up and set its status word. ``status``: a device int32 tensor, one word
    (``per_chunk`` False) or nranks words, word c for chunk c (``per_chunk`` True)."""
    count = _check_full(sendbufs, recvbufs, "ra_selftest_bulk_timeout")
    if status.numel() < (len(sendbufs) if per_chunk else 1):
        raise ValueError("ra_selftest_bulk_timeout: status is too small")
    st = lib().ra_selftest_bulk_timeout(ptr_array([t.data_ptr() for t in sendbufs]),
                                        ptr_array([t.data_ptr() for t in recvbufs]), count, dtype_code(sendbufs[0]),
                                        OP_CODES[op], len(sendbufs), withhold_chunk,
                                        ctypes.c_void_p(status.data_ptr()), 1 if per_chunk else 0,
                                        ctypes.c_void_p(_stream_ptr(stream) or None))
    if st:
        raise RaError(st, "ra_selftest_bulk_timeout")


def ra_vector_bytes() -> int:
    return lib().ra_vector_bytes()


def ra_allreduce_bulk_noalloc(sendbufs, recvbufs, op: str = "sum", max_sms: int = 0, chunk_status=None,
                              stream=None) -> None:
    """The bulk-engine all-reduce with the status words kept by the library, so no device memory
    beyond the buffers is needed. ``chunk_status``: optional int32 tensor of nranks words (device or
    host) that receives each chunk's wait code (0 = finished) once the stream has passed the call."""
    import torch

    count = _check_full(sendbufs, recvbufs, "ra_allreduce_bulk_noalloc")
    if chunk_status is not None and (chunk_status.dtype != torch.int32 or not chunk_status.is_contiguous()
                                     or chunk_status.numel() < len(sendbufs)):
        raise ValueError("ra_allreduce_bulk_noalloc: chunk_status must be a contiguous int32 tensor of nranks words")
    cs = chunk_status.data_ptr() if chunk_status is not None else None
    st = lib().ra_allreduce_bulk_noalloc(ptr_array([t.data_ptr() for t in sendbufs]),
                                         ptr_array([t.data_ptr() for t in recvbufs]), count,
                                         dtype_code(sendbufs[0]), OP_CODES[op], len(sendbufs), max_sms,
                                         ctypes.c_void_p(cs), ctypes.c_void_p(_stream_ptr(stream) or None))
    if st:
        raise RaError(st, "ra_allreduce_bulk_noalloc")
