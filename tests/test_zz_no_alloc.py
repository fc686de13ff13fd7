"""ra_allreduce_bulk_noalloc: the bulk-engine all-reduce whose status words are
kept by the library, so the caller hands in no device memory beyond its
buffers. Through the C ABI it must give the same bits as the existing
ra_allreduce_ex(engine=bulk) on two calls in a row (the second one finds the
library's words as the first left them), report zero codes for every chunk,
and reject a rank count beyond its fixed array before enqueuing anything.

The file is named to be collected last, after every other test has loaded
and used the library in the same process; it also passes alone."""

import ctypes

import pytest
import torch

import oracle
from helpers import assert_same_bits, to_device, to_host
from ring_all_reduce_02_gb300 import inputs


@pytest.fixture(scope="module")
def ra():
    from ring_all_reduce_02_gb300 import build, ra as binding

    build.build()
    return binding


def raw_call(ra, n, count, nranks, max_sms=0, chunk_status=None):
    ptrs = [4096 * (k + 1) for k in range(n)]
    return ra.lib().ra_allreduce_bulk_noalloc(ra.ptr_array(ptrs), ra.ptr_array(ptrs), count, 0, 0, nranks,
                                              max_sms, chunk_status, None)


def test_rejects_before_enqueuing(ra):
    # the size checks return before any CUDA call, so they run without a GPU
    assert ra.RA_NOALLOC_STATUS_WORDS == 16
    assert raw_call(ra, 17, 1 << 20, 17) == ra.RA_ERR_SCRATCH_LIMIT
    assert raw_call(ra, 64, 1 << 20, 64) == ra.RA_ERR_SCRATCH_LIMIT
    assert raw_call(ra, 1, 1 << 20, 0) == ra.RA_ERR_INVALID_ARG
    assert raw_call(ra, 65, 1 << 20, 65) == ra.RA_ERR_INVALID_ARG
    assert raw_call(ra, 4, 1 << 20, 4, max_sms=-1) == ra.RA_ERR_INVALID_ARG
    assert "RA_NOALLOC_STATUS_WORDS" in ra.ra_status_string(ra.RA_ERR_SCRATCH_LIMIT)
    # count 0: nothing enqueued, chunk_status untouched
    words = (ctypes.c_int * 4)(-7, -7, -7, -7)
    assert raw_call(ra, 4, 0, 4, chunk_status=ctypes.cast(words, ctypes.c_void_p)) == ra.RA_SUCCESS
    assert list(words) == [-7] * 4


CASES = [  # (dtype, op, nranks, length, max_sms, in_place, chunk_status memory)
    ("f32", "sum", 2, 1 << 16, 0, False, "device"),
    ("f32", "avg", 5, 5 * 4096 * 3 + 7, 0, False, "pinned"),
    ("bf16", "avg", 8, (1 << 20) + 13, 16, False, "device"),
    ("bf16", "max", 16, 16 * 2048 * 5 + 3, 0, True, "device"),
    ("f32", "sum", 8, (1 << 20) + 13, 0, False, None),
]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,op,n,length,max_sms,inplace,where", CASES)
def test_matches_bulk_entry_point_twice(ra, dtype, op, n, length, max_sms, inplace, where):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    oracle.build()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):  # two calls in a row, new inputs each time
        xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=40 + 10 * call + n)
        # the existing entry point, with a caller-owned status word
        ref_send = [to_device(x, dtype) for x in xs]
        ref_recv = ref_send if inplace else [torch.empty_like(s) for s in ref_send]
        ra.ra_allreduce_ex(ref_send, ref_recv, op, engine="bulk", status=status, max_sms=max_sms)
        # the no-alloc entry point on copies of the same inputs
        sends = [to_device(x, dtype) for x in xs]
        recvs = sends if inplace else [torch.full_like(s, 7) for s in sends]
        words = None
        if where == "device":
            words = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        elif where == "pinned":
            words = torch.full((n,), -7, dtype=torch.int32).pin_memory()
        ra.ra_allreduce_bulk_noalloc(sends, recvs, op, max_sms=max_sms, chunk_status=words)
        torch.cuda.synchronize()
        assert status.item() == 0
        if words is not None:
            assert words.cpu().tolist() == [0] * n, f"call {call}: chunk codes {words.cpu().tolist()}"
        want, _, _ = oracle.allreduce(xs, op, dtype)
        for r in range(n):
            assert torch.equal(recvs[r].view(torch.uint8), ref_recv[r].view(torch.uint8)), \
                f"call {call} rank {r}: differs from ra_allreduce_ex(engine=bulk)"
            assert_same_bits(to_host(recvs[r], dtype), want[r], dtype, f"call {call} rank {r} vs oracle")


@pytest.mark.gpu
def test_misaligned_phase_is_unsupported(ra):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    n, length = 4, 4096
    base = [torch.zeros(length + 4, dtype=torch.float32, device="cuda") for _ in range(n)]
    sends = [b[k % 2:k % 2 + length] for k, b in enumerate(base)]  # address phases 0 and 4 bytes
    recvs = [torch.empty(length, dtype=torch.float32, device="cuda") for _ in range(n)]
    with pytest.raises(ra.RaError, match="unsupported"):
        ra.ra_allreduce_bulk_noalloc(sends, recvs, "sum")


# A program that drives the GPU through the driver API alone, with no torch: it
# runs the no-alloc call in the device's primary context, then in a second
# context it created itself, then in the primary context again. The library's
# status words have one address per context, so an address remembered from an
# earlier call would point the second call's clear and kernel at memory that
# context does not map; a lookup per call gives each context its own words.
_CONTEXT_PROGRAM = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle
from ring_all_reduce_02_gb300 import inputs, ra

cu = ctypes.CDLL("libcuda.so.1")
def ck(res, what):
    if res != 0:
        raise SystemExit(f"{what}: CUresult {res}")
ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
primary, second = ctypes.c_void_p(), ctypes.c_void_p()
ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")

def one_call(tag, n, length, op, seed):
    xs = inputs.rank_buffers(n, length, "f32", ("normal", 1.0), seed_base=seed)
    nbytes = length * 4
    send, recv = [], []
    for x in xs:
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
        ck(cu.cuMemcpyHtoD_v2(p, x.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(nbytes)), "HtoD")
        send.append(p.value)
    for _ in xs:
        p = ctypes.c_uint64()
        ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
        recv.append(p.value)
    words = (ctypes.c_int * n)(*([-7] * n))
    st = ra.lib().ra_allreduce_bulk_noalloc(ra.ptr_array(send), ra.ptr_array(recv), length, 0,
                                            ra.OP_CODES[op], n, 0, ctypes.cast(words, ctypes.c_void_p), None)
    if st != 0:
        raise SystemExit(f"{tag}: status {st} ({ra.ra_status_string(st)}), cudaError {ra.lib().ra_last_cuda_error()}")
    ck(cu.cuCtxSynchronize(), f"{tag}: synchronize")
    want, _, _ = oracle.allreduce(xs, op, "f32")
    for r in range(n):
        got = np.empty(length, dtype=np.float32)
        ck(cu.cuMemcpyDtoH_v2(got.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(recv[r]),
                              ctypes.c_size_t(nbytes)), "DtoH")
        if got.tobytes() != want[r].tobytes():
            raise SystemExit(f"{tag}: rank {r} differs from the oracle")
    if list(words) != [0] * n:
        raise SystemExit(f"{tag}: chunk codes {list(words)}")
    for p in send + recv:
        ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
    print(tag, "ok", flush=True)

ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent(primary)")
one_call("primary", 4, 4 * 4096 * 3 + 5, "sum", 70)
ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "cuCtxCreate")  # also makes it current
one_call("second", 8, (1 << 18) + 3, "avg", 71)
one_call("second again", 3, 3 * 4096 * 2 + 1, "max", 72)
ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent(primary)")
one_call("primary again", 5, 5 * 4096 + 9, "sum", 73)
ck(cu.cuCtxDestroy_v2(second), "cuCtxDestroy")
ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
print("CONTEXTS OK", flush=True)
"""


@pytest.mark.gpu
def test_status_words_follow_the_current_context(ra):
    # A caller that manages contexts with the driver API (its own context per
    # library or per job, or a device reset between jobs) gets, in each context,
    # that context's copy of the status words: results and codes as in the first.
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import os
    import subprocess
    import sys

    oracle.build()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    proc = subprocess.run([sys.executable, "-c", _CONTEXT_PROGRAM, root], capture_output=True, text=True,
                          timeout=300)
    assert proc.returncode == 0 and "CONTEXTS OK" in proc.stdout, proc.stdout + proc.stderr
