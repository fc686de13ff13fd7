"""Stream order of back-to-back collectives.

The collective kernels are programmatic dependent launches: a launch's CTAs
may be resident while the previous kernel on the stream is still running, and
each kernel waits for that kernel to complete before it touches memory. These
tests chain calls whose inputs are the previous call's outputs, enqueued
behind a device sleep so that the whole chain is queued before the first
kernel starts, on buffers larger than L2 and with ragged chunk edges. Any
read that overtook the previous kernel's writes would break the closed form:
for int32 sum, k in-place all-reduces leave N^(k-1) * sum_r x_r on every rank
(wrapping), and a reduce-scatter then all-gather of an all-reduced buffer
gives N * sum_r x_r.
"""

import numpy as np
import pytest
import torch

from helpers import to_device, to_host
from ring_all_reduce_02_gb300 import inputs

pytestmark = pytest.mark.gpu

N = 8
L = (4 << 20) + 12347  # 16 MiB + a ragged tail per rank; chunk bounds off the line grid


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from ring_all_reduce_02_gb300 import build, ra as binding

    build.build()
    return binding


@pytest.fixture(scope="module")
def xs():
    return inputs.rank_buffers(N, L, "i32", ("int_uniform", -1000, 1000))


def wrap32(v: np.ndarray) -> np.ndarray:
    return ((v + 2**31) % 2**32 - 2**31).astype(np.int32)


def total(xs) -> np.ndarray:
    return np.sum(np.stack(xs).astype(np.int64), axis=0)


def check_all(bufs, want, what):
    for r, b in enumerate(bufs):
        got = to_host(b, "i32")
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"{what}: rank {r}: {bad.size} elements differ, first at {bad[:5]}"


CHAINS = ["ring", "bulk", "tree", "rabenseifner", "ringsteps"]


@pytest.mark.parametrize("how", CHAINS)
def test_chained_inplace_allreduce(ra, xs, how):
    k = 3
    bufs = [to_device(x, "i32") for x in xs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)
    for _ in range(k):
        if how == "ring":
            ra.ra_allreduce(bufs, bufs, "sum", stream=stream)
        elif how == "bulk":
            ra.ra_allreduce_ex(bufs, bufs, "sum", engine="bulk", status=status, stream=stream)
        elif how == "ringsteps":
            ra.ra_allreduce_ringsteps(bufs, bufs, "sum", stream=stream)
        else:
            ra.ra_allreduce_ex(bufs, bufs, "sum", order=how, stream=stream)
    torch.cuda.synchronize()
    if how == "bulk":
        assert int(status.item()) == 0
    check_all(bufs, wrap32(total(xs) * N ** (k - 1)), f"{k} chained in-place all-reduces ({how})")


def _chain_ar_rs_ag(ra, bufs, shards, outs, stream):
    ra.ra_allreduce(bufs, bufs, "sum", stream=stream)
    ra.ra_reduce_scatter(bufs, shards, "sum", stream=stream)
    ra.ra_allgather(shards, outs, stream=stream)


def _buffers(ra, xs):
    bufs = [to_device(x, "i32") for x in xs]
    shards = [torch.empty(e - b, dtype=torch.int32, device="cuda")
              for b, e in (ra.ra_chunk_range(L, N, c) for c in range(N))]
    outs = [torch.empty(L, dtype=torch.int32, device="cuda") for _ in range(N)]
    return bufs, shards, outs


def test_chained_allreduce_reducescatter_allgather(ra, xs):
    bufs, shards, outs = _buffers(ra, xs)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)
    _chain_ar_rs_ag(ra, bufs, shards, outs, stream)
    torch.cuda.synchronize()
    check_all(outs, wrap32(total(xs) * N), "all-reduce -> reduce-scatter -> all-gather")


def test_chain_captured_in_a_graph(ra, xs):
    bufs, shards, outs = _buffers(ra, xs)
    saved = [b.clone() for b in bufs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            _chain_ar_rs_ag(ra, bufs, shards, outs, side)
    torch.cuda.synchronize()
    for rep in range(2):
        for b, s in zip(bufs, saved):
            b.copy_(s)
        for o in outs:
            o.fill_(-1)
        torch.cuda._sleep(1_000_000)
        graph.replay()
        torch.cuda.synchronize()
        check_all(outs, wrap32(total(xs) * N), f"graph replay {rep}")
