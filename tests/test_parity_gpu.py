"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bar: bit-exact for every dtype and op (the ring order and per-hop rounding are
reproduced, so the tolerance is 0 ULP; any NaN equals any NaN). Every shape,
the full-size workloads included, is compared element by element, on every
rank, against the oracle's message-passing ring (or its tree, Rabenseifner
and fp32-message variants). Only the case past 2^32 elements per rank (48 GiB
on the device) is compared on sampled elements, against the oracle's
per-element definition. Guard regions around every small buffer ("canaries")
stand in for a bounds checker.
"""

import itertools

import numpy as np
import pytest
import torch

import oracle
from helpers import ELEM_SIZE, TORCH_DTYPE, assert_same_bits, to_device, to_host
from ring_all_reduce_02_gb300 import inputs

pytestmark = pytest.mark.gpu

DTYPES = ["f32", "f16", "bf16", "i32"]
OPS = ["sum", "avg", "min", "max", "prod"]


@pytest.fixture(scope="module")
def ra():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from ring_all_reduce_02_gb300 import build, ra as binding

    build.build()
    oracle.build()
    return binding


def dist_for(dtype, op):
    if dtype == "i32":
        return ("int_uniform", -2, 2) if op == "prod" else ("int_uniform", -1000, 1000)
    return ("normal", 1.0)


class Padded:
    """A device buffer with guard regions of a fixed byte pattern on both sides."""

    PAD = 256  # bytes on each side
    FILL = 0x5A

    def __init__(self, numel, dtype, offset_elems=0):
        es = ELEM_SIZE[dtype]
        self.dtype = dtype
        total = self.PAD * 2 + (numel + offset_elems) * es
        self.raw = torch.full((total,), self.FILL, dtype=torch.uint8, device="cuda")
        start = self.PAD + offset_elems * es
        self.view = self.raw[start:start + numel * es].view(TORCH_DTYPE[dtype])
        self.start, self.end = start, start + numel * es

    def fill(self, a: np.ndarray):
        if a.size:
            self.view.copy_(to_device(a, self.dtype))

    def canaries_intact(self) -> bool:
        raw = self.raw.cpu().numpy()
        return bool((raw[:self.start] == self.FILL).all() and (raw[self.end:] == self.FILL).all())


def run_allreduce(ra, xs, op, dtype, inplace=False, offsets=None):
    n = len(xs)
    offsets = offsets or [0] * (2 * n)
    sends = [Padded(x.size, dtype, offsets[r]) for r, x in enumerate(xs)]
    for b, x in zip(sends, xs):
        b.fill(x)
    recvs = sends if inplace else [Padded(xs[0].size, dtype, offsets[n + r]) for r in range(n)]
    ra.ra_allreduce([b.view for b in sends], [b.view for b in recvs], op)
    torch.cuda.synchronize()
    for b in sends + ([] if inplace else recvs):
        assert b.canaries_intact(), "write outside the buffers"
    return [to_host(b.view, dtype) for b in recvs]


def run_reduce_scatter(ra, xs, op, dtype, inplace=False):
    n, length = len(xs), xs[0].size
    sends = [Padded(length, dtype) for _ in xs]
    for b, x in zip(sends, xs):
        b.fill(x)
    bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
    if inplace:
        recvs = [s.view[b:e] for s, (b, e) in zip(sends, bounds)]
        ra.ra_reduce_scatter([s.view for s in sends], recvs, op)
        torch.cuda.synchronize()
        outs = [to_host(r, dtype) for r in recvs]
        pads = sends
    else:
        pads = [Padded(e - b, dtype) for b, e in bounds]
        ra.ra_reduce_scatter([s.view for s in sends], [p.view for p in pads], op)
        torch.cuda.synchronize()
        outs = [to_host(p.view, dtype) for p in pads]
        pads = pads + sends
    for p in pads:
        assert p.canaries_intact()
    return outs


def run_allgather(ra, shards, length, dtype, inplace=False):
    n = len(shards)
    bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
    recvs = [Padded(length, dtype) for _ in range(n)]
    if inplace:
        sends = []
        for r, (b, e) in enumerate(bounds):
            v = recvs[r].view[b:e]
            if e > b:
                v.copy_(to_device(shards[r], dtype))
            sends.append(v)
        ra.ra_allgather(sends, [p.view for p in recvs])
        pads = recvs
    else:
        sp = [Padded(e - b, dtype) for b, e in bounds]
        for p, s in zip(sp, shards):
            p.fill(s)
        ra.ra_allgather([p.view for p in sp], [p.view for p in recvs])
        pads = recvs + sp
    torch.cuda.synchronize()
    for p in pads:
        assert p.canaries_intact()
    return [to_host(p.view, dtype) for p in recvs]


def check_all(ra, xs, op, dtype, what):
    """AR, RS and AG against the oracle; AG(RS) == AR; every rank identical."""
    length = xs[0].size
    want, _, _ = oracle.allreduce(xs, op, dtype)
    got = run_allreduce(ra, xs, op, dtype)
    for r in range(len(xs)):
        assert_same_bits(got[r], want[r], dtype, f"{what} AR rank {r}")
    shards_want, _ = oracle.reduce_scatter(xs, op, dtype)
    shards = run_reduce_scatter(ra, xs, op, dtype)
    for r in range(len(xs)):
        assert_same_bits(shards[r], shards_want[r], dtype, f"{what} RS shard {r}")
    ag = run_allgather(ra, shards, length, dtype)
    ag_want, _, _ = oracle.allgather(shards_want, length, dtype)
    for r in range(len(xs)):
        assert_same_bits(ag[r], ag_want[r], dtype, f"{what} AG rank {r}")
        assert ag[r].tobytes() == got[0].tobytes(), f"{what}: AG(RS) != AR"


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------
def test_n4_f32_sum_4k(ra):
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n4_f32_sum_4k"]
    xs = inputs.rank_buffers(n, length, dtype, dist)
    check_all(ra, xs, op, dtype, "n4 f32 sum 4k")


@pytest.mark.parametrize("case", inputs.sweep_cases(), ids=lambda c: f"n{c[0]}-{c[2]}-{c[3]}")
def test_op_dtype_sweep_uneven_chunks(ra, case):
    n, length, dtype, op, dist = case
    xs = inputs.rank_buffers(n, length, dtype, dist)
    want, _, _ = oracle.allreduce(xs, op, dtype)
    got = run_allreduce(ra, xs, op, dtype)
    for r in range(n):
        assert_same_bits(got[r], want[r], dtype, f"rank {r}")
    shards = run_reduce_scatter(ra, xs, op, dtype)
    shards_want, _ = oracle.reduce_scatter(xs, op, dtype)
    for r in range(n):
        assert_same_bits(shards[r], shards_want[r], dtype, f"RS shard {r}")


# ---------------------------------------------------------------------------
# every dtype x op on small and ragged shapes, several tiles, edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,op", list(itertools.product(DTYPES, OPS)))
def test_small_and_ragged_shapes(ra, dtype, op):
    seed = 1000
    # every rank count with a launch shape of its own: 6 and 7 (the wide shape loading all ranks,
    # fp16/bf16 sum/avg/prod at 6 on two CTAs per SM), 9, 10, 12 and 14 (fp32 and fp16/bf16
    # min/max shapes, the flat all-gather)
    for n in (1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 12, 14, 16):
        for length in (0, 1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 64, 65, 100, 257, 1000, 4097):
            xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=seed)
            seed += 1
            if length == 0:
                outs = run_allreduce(ra, xs, op, dtype)
                assert all(o.size == 0 for o in outs)
                continue
            check_all(ra, xs, op, dtype, f"n={n} L={length}")


@pytest.mark.parametrize("n,length,dtype", [(8, (1 << 20) + 13, "f32"), (8, (1 << 24) + 7, "bf16"),
                                            (3, 3 * 600_001, "f16"), (16, 5_000_011, "f32")])
def test_many_tiles_and_trips(ra, n, length, dtype):
    # chunks of 10^5..2*10^6 elements: several CTAs per chunk, several trips per CTA,
    # and a ragged tail at every chunk boundary
    for op in ("sum", "avg"):
        xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=77)
        want, _, _ = oracle.allreduce(xs, op, dtype)
        got = run_allreduce(ra, xs, op, dtype)
        for r in range(n):
            assert_same_bits(got[r], want[r], dtype, f"{op} rank {r}")


def test_ring_order_is_reproduced(ra):
    # fp32: chunk c starts the fold at x_c. x_c = 1 and 2^-24 elsewhere: ties to even keep 1.0;
    # any other starting rank gives 1 + 2^-22. Bits must match the oracle exactly.
    n, length = 8, 8 * 1024 + 5
    tiny = np.float32(2.0 ** -24)
    for c in range(n):
        b, e = oracle.chunk_range(length, n, c)
        xs = [np.full(length, tiny, dtype=np.float32) for _ in range(n)]
        xs[c][b:e] = 1.0
        want, _, _ = oracle.allreduce(xs, "sum", "f32")
        got = run_allreduce(ra, xs, "sum", "f32")
        assert (got[0][b:e] == np.float32(1.0)).all()
        assert_same_bits(got[3], want[3], "f32", f"chunk {c}")


@pytest.mark.parametrize("length", [4 * 15 + 11, 5 * 4096 + 11, 8 * 16 * 100])
def test_special_values(ra, length):
    # NaN, infinities, signed zeros, subnormals in every float dtype; the short length runs on the
    # per-element edge path, the long ones on the vector path (paired 16-bit min/max, off-grid
    # compact reduce-scatter outputs and all-gather inputs; at 12800 every shard is on the vector
    # grid), at N = 2, 5 and 8 (the small-N, all-reduce and reduce-scatter launch shapes)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-40, 6e-8, -6e-8, 1e-39, 65504.0,
                         -65504.0, 3.4e38, 1.0, -1.0], dtype=np.float32)
    rng = np.random.default_rng(3)
    for dtype, op, n in itertools.product(("f32", "f16", "bf16"), OPS, (2, 5, 8)):
        xs = []
        for r in range(n):
            v = rng.choice(specials, size=length).astype(np.float32)
            if dtype == "f16":
                xs.append(v.astype(np.float16))
            elif dtype == "bf16":
                xs.append(oracle.round_f32("bf16", v))
            else:
                xs.append(v)
        check_all(ra, xs, op, dtype, f"specials {dtype} {op} N={n} L={length}")


def test_int32_wrap_and_avg(ra):
    n, length = 3, 1001
    big = [np.full(length, 2**31 - 5 - r, dtype=np.int32) for r in range(n)]
    for op in ("sum", "prod", "avg"):
        want, _, _ = oracle.allreduce(big, op, "i32")
        got = run_allreduce(ra, big, op, "i32")
        assert_same_bits(got[0], want[0], "i32", op)


# ---------------------------------------------------------------------------
# layouts: in place, offset views, mixed phases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", DTYPES)
def test_inplace_equals_out_of_place(ra, dtype):
    n, length = 5, 1003 * 17
    xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, "sum"), seed_base=5)
    a = run_allreduce(ra, xs, "sum", dtype)
    b = run_allreduce(ra, xs, "sum", dtype, inplace=True)
    for r in range(n):
        assert a[r].tobytes() == b[r].tobytes()
    s1 = run_reduce_scatter(ra, xs, "sum", dtype)
    s2 = run_reduce_scatter(ra, xs, "sum", dtype, inplace=True)
    for r in range(n):
        assert s1[r].tobytes() == s2[r].tobytes()
    g1 = run_allgather(ra, s1, length, dtype)
    g2 = run_allgather(ra, s1, length, dtype, inplace=True)
    for r in range(n):
        assert g1[r].tobytes() == g2[r].tobytes() == a[0].tobytes()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_inplace_small_n_on_grid(ra, dtype):
    # in place with every shard on the vector grid at small N: the one-trip launches of N <= 2
    # all-reduces and of on-grid reduce-scatters up to N = 7 read and write the same buffers
    per_vec = ra.ra_vector_bytes() // ELEM_SIZE[dtype]
    for n in (1, 2, 3, 4, 6, 7):
        length = n * per_vec * 300
        for op in ("sum", "max"):
            xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=170 + n)
            want, _, _ = oracle.allreduce(xs, op, dtype)
            got = run_allreduce(ra, xs, op, dtype, inplace=True)
            shards = run_reduce_scatter(ra, xs, op, dtype, inplace=True)
            bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
            for r, (b, e) in enumerate(bounds):
                assert_same_bits(got[r], want[r], dtype, f"AR in place n={n} {op} rank {r}")
                assert_same_bits(shards[r], want[0][b:e], dtype, f"RS in place n={n} {op} shard {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pinned_host_buffers(ra, dtype):
    # buffers in pinned host memory, read and written by the kernels over the host link (the bench's
    # end-to-end leg): all-reduce host -> host and host -> device, reduce-scatter into host shards,
    # all-gather from host shards into host buffers (plain stores, not the TMA tile kernel), every
    # element against the oracle; the paths built on TMA or cp.async refuse host memory up front
    td = TORCH_DTYPE[dtype]
    for n, length in ((2, 2 * 4096 * 3), (5, 5 * 1003 * 7 + 3), (8, (1 << 18) + 13)):
        xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=190 + n)
        want, _, _ = oracle.allreduce(xs, "avg", dtype)
        shards_want, _ = oracle.reduce_scatter(xs, "avg", dtype)
        sends = [to_device(x, dtype).cpu().pin_memory() for x in xs]
        host_out = [torch.empty(length, dtype=td).pin_memory() for _ in range(n)]
        dev_out = [torch.empty(length, dtype=td, device="cuda") for _ in range(n)]
        ra.ra_allreduce(sends, host_out, "avg")
        ra.ra_allreduce(sends, dev_out, "avg")
        bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
        shards = [torch.empty(e - b, dtype=td).pin_memory() for b, e in bounds]
        ra.ra_reduce_scatter(sends, shards, "avg")
        gathered = [torch.empty(length, dtype=td).pin_memory() for _ in range(n)]
        torch.cuda.synchronize()
        ra.ra_allgather(shards, gathered)
        torch.cuda.synchronize()
        for r in range(n):
            assert_same_bits(to_host(host_out[r], dtype), want[r], dtype, f"AR host->host n={n} rank {r}")
            assert_same_bits(to_host(dev_out[r], dtype), want[r], dtype, f"AR host->device n={n} rank {r}")
            assert_same_bits(to_host(shards[r], dtype), shards_want[r], dtype, f"RS host n={n} shard {r}")
            assert_same_bits(to_host(gathered[r], dtype), want[r], dtype, f"AG host n={n} rank {r}")
        # DDP-style buckets on the same host buffers: grouped launches, each bucket its own all-reduce
        plan = ra.ra_bucket_plan([length // 3, length // 3, length - 2 * (length // 3)], 4096, ELEM_SIZE[dtype])
        bucket_out = [torch.empty(length, dtype=td).pin_memory() for _ in range(n)]
        ra.ra_allreduce_buckets(sends, bucket_out, plan, "avg")
        torch.cuda.synchronize()
        for b, c in plan:
            bw, _, _ = oracle.allreduce([np.ascontiguousarray(x[b:b + c]) for x in xs], "avg", dtype)
            for r in range(n):
                assert_same_bits(to_host(bucket_out[r][b:b + c], dtype), bw[r], dtype, f"bucket {b}+{c} n={n} rank {r}")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(ra.RaError, match="unsupported"):
            ra.ra_allreduce_ex(sends, host_out, "avg", engine="bulk", status=status)
        with pytest.raises(ra.RaError, match="unsupported"):
            ra.ra_allreduce_ex(sends, host_out, "avg", order="tree")
        torch.cuda.synchronize()
        assert status.item() == 0


@pytest.mark.parametrize("n", [3, 5, 12])
def test_allgather_mixed_phases(ra, n):
    # destinations at different element offsets share no vector grid, so every element takes the
    # per-element path; at N = 5 and 12 the planner then keeps the row-per-chunk kernel instead
    # of the flat tile sequence
    dtype, length = "f32", 20_011
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=13)
    shards, _ = oracle.reduce_scatter(xs, "sum", dtype)
    want, _, _ = oracle.allreduce(xs, "sum", dtype)
    ins = []
    for c, (b, e) in enumerate(oracle.chunk_range(length, n, c) for c in range(n)):
        p = Padded(e - b, dtype, c % 2)
        p.fill(shards[c])
        ins.append(p)
    recvs = [Padded(length, dtype, r % 3) for r in range(n)]
    ra.ra_allgather([p.view for p in ins], [r.view for r in recvs])
    torch.cuda.synchronize()
    for r in range(n):
        assert recvs[r].canaries_intact()
        assert_same_bits(to_host(recvs[r].view, dtype), want[r], dtype, f"rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_offset_views(ra, dtype):
    # every buffer at the same element offset (vector path with a head), then at different
    # offsets (per-element path); compact sides of RS/AG at arbitrary offsets
    n, length = 4, 10_007
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=9)
    want, _, _ = oracle.allreduce(xs, "avg", dtype)
    es = ELEM_SIZE[dtype]
    per_vec = ra.ra_vector_bytes() // es
    for offsets in ([1] * 8, [per_vec - 1] * 8, [0, 1, 2, 3, 0, 1, 2, 3], [0] * 4 + [1] * 4):
        got = run_allreduce(ra, xs, "avg", dtype, offsets=offsets)
        for r in range(n):
            assert_same_bits(got[r], want[r], dtype, f"offsets {offsets} rank {r}")
    # reduce-scatter into compact buffers of every phase; all-gather from them
    shards_want, _ = oracle.reduce_scatter(xs, "avg", dtype)
    bounds = [oracle.chunk_range(length, n, c) for c in range(n)]
    for off in range(per_vec):
        sends = [Padded(length, dtype) for _ in range(n)]
        for s, x in zip(sends, xs):
            s.fill(x)
        outs = [Padded(e - b, dtype, off + c) for c, (b, e) in enumerate(bounds)]
        ra.ra_reduce_scatter([s.view for s in sends], [o.view for o in outs], "avg")
        recvs = [Padded(length, dtype, off) for _ in range(n)]
        ra.ra_allgather([o.view for o in outs], [r.view for r in recvs])
        torch.cuda.synchronize()
        for c in range(n):
            assert outs[c].canaries_intact() and recvs[c].canaries_intact()
            assert_same_bits(to_host(outs[c].view, dtype), shards_want[c], dtype, f"RS off {off}")
            assert_same_bits(to_host(recvs[c].view, dtype), want[c], dtype, f"AG off {off}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [3, 4, 6, 8, 12])
def test_offgrid_compact_buffers_many_tiles(ra, dtype, n):
    # compact RS outputs / AG inputs at every phase against the vector grid, with chunks several
    # all-gather tiles (256 vectors) long: the unit-wise tile loads of the all-gather, the 4-byte
    # per-lane and 2-byte cooperative reduce-scatter stores (one resident wave below N = 8 for
    # 2-byte types, a CTA per trip from there)
    es = ELEM_SIZE[dtype]
    per_vec = ra.ra_vector_bytes() // es
    length = n * 256 * per_vec * 3 + 13
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=70 + n)
    want, _, _ = oracle.allreduce(xs, "avg", dtype)
    shards_want, _ = oracle.reduce_scatter(xs, "avg", dtype)
    bounds = [oracle.chunk_range(length, n, c) for c in range(n)]
    for off in range(per_vec):
        sends = [Padded(length, dtype) for _ in range(n)]
        for b, x in zip(sends, xs):
            b.fill(x)
        outs = [Padded(e - b, dtype, off) for b, e in bounds]
        ra.ra_reduce_scatter([b.view for b in sends], [o.view for o in outs], "avg")
        recvs = [Padded(length, dtype) for _ in range(n)]
        ra.ra_allgather([o.view for o in outs], [r.view for r in recvs])
        torch.cuda.synchronize()
        for c in range(n):
            assert outs[c].canaries_intact() and recvs[c].canaries_intact(), f"off {off} chunk {c}"
            assert_same_bits(to_host(outs[c].view, dtype), shards_want[c], dtype, f"RS off {off} chunk {c}")
            assert_same_bits(to_host(recvs[c].view, dtype), want[c], dtype, f"AG off {off} rank {c}")


@pytest.mark.parametrize("dtype,op", list(itertools.product(DTYPES, OPS)))
def test_ongrid_shards_small_n(ra, dtype, op):
    # reduce-scatters whose shards all sit on the vector grid (L a multiple of N vectors, shards in
    # their own allocations) at N = 1..8: the small-N one-trip launches (N <= 4, and up to 7 for
    # 16-bit types and float min/max), several trips per chunk plus a partial one
    per_vec = ra.ra_vector_bytes() // ELEM_SIZE[dtype]
    for n in range(1, 9):
        length = n * per_vec * (2 * 256 + 37)
        xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=150 + n)
        shards_want, _ = oracle.reduce_scatter(xs, op, dtype)
        sends = [to_device(x, dtype) for x in xs]
        bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
        assert all((b * ELEM_SIZE[dtype]) % ra.ra_vector_bytes() == 0 for b, _ in bounds)
        shards = [Padded(e - b, dtype) for b, e in bounds]
        ra.ra_reduce_scatter(sends, [s.view for s in shards], op)
        torch.cuda.synchronize()
        for c in range(n):
            assert shards[c].canaries_intact(), f"n={n} chunk {c}"
            assert_same_bits(to_host(shards[c].view, dtype), shards_want[c], dtype, f"n={n} shard {c}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("op", ["min", "max"])
@pytest.mark.parametrize("n", [3, 9, 12])
def test_offgrid_shards_min_max(ra, dtype, op, n):
    # min/max reduce-scatters into 16-bit shards at odd and even phases against the vector grid,
    # several trips per chunk: the min/max launch shapes with the realigned off-grid stores
    per_vec = ra.ra_vector_bytes() // ELEM_SIZE[dtype]
    length = n * 512 * per_vec + 29
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=110 + n)
    shards_want, _ = oracle.reduce_scatter(xs, op, dtype)
    bounds = [oracle.chunk_range(length, n, c) for c in range(n)]
    for off in (0, 1, 2, 5, per_vec - 1):
        sends = [Padded(length, dtype) for _ in range(n)]
        for b, x in zip(sends, xs):
            b.fill(x)
        outs = [Padded(e - b, dtype, (off + c) % per_vec) for c, (b, e) in enumerate(bounds)]
        ra.ra_reduce_scatter([b.view for b in sends], [o.view for o in outs], op)
        torch.cuda.synchronize()
        for c in range(n):
            assert outs[c].canaries_intact(), f"off {off} chunk {c}"
            assert_same_bits(to_host(outs[c].view, dtype), shards_want[c], dtype, f"off {off} chunk {c}")


@pytest.mark.parametrize("n", [3, 8, 12])
def test_offgrid_shards_fp32_partials(ra, n):
    # reduce-scatter with fp32 partials into bf16 shards at every 2-byte phase against the vector
    # grid: the off-grid stores realigned in registers, on the one-wave kernel
    dtype = "bf16"
    per_vec = ra.ra_vector_bytes() // ELEM_SIZE[dtype]
    length = n * 128 * per_vec * 3 + 13
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=90 + n)
    want, _ = oracle.allreduce_ex(xs, "avg", dtype, accum="fp32")
    bounds = [oracle.chunk_range(length, n, c) for c in range(n)]
    for off in (0, 1, 2, 3, per_vec - 1):
        sends = [Padded(length, dtype) for _ in range(n)]
        for b, x in zip(sends, xs):
            b.fill(x)
        outs = [Padded(e - b, dtype, off + c) for c, (b, e) in enumerate(bounds)]
        ra.ra_reduce_scatter_ex([b.view for b in sends], [o.view for o in outs], "avg", accum="fp32")
        torch.cuda.synchronize()
        for c, (b, e) in enumerate(bounds):
            assert outs[c].canaries_intact(), f"off {off} chunk {c}"
            assert_same_bits(to_host(outs[c].view, dtype), want[0][b:e], dtype, f"off {off} chunk {c}")


def test_fewer_elements_than_ranks(ra):
    # empty chunks: L < N (infra-guide 3.4 example: 3 elements over 4 ranks)
    for n, length in ((4, 3), (16, 5), (64, 63), (7, 1)):
        for dtype in ("f32", "i32"):
            xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, "sum"), seed_base=n)
            check_all(ra, xs, "sum", dtype, f"n={n} L={length}")


def test_max_ranks(ra):
    n, length = 64, 64 * 129 + 7
    xs = inputs.rank_buffers(n, length, "f32", ("normal", 1.0), seed_base=2)
    check_all(ra, xs, "sum", "f32", "64 ranks")


def test_errors_enqueue_nothing(ra):
    x = torch.ones(100, device="cuda")
    y = torch.zeros(100, device="cuda")
    with pytest.raises(ra.RaError):
        ra.ra_allreduce([x, x], [y, y], "sum")  # two ranks writing one buffer
    torch.cuda.synchronize()
    assert (y == 0).all()


# ---------------------------------------------------------------------------
# full-size workloads in the benchmark's launch configuration: every element against the oracle
# ---------------------------------------------------------------------------
def _host_ram_gb():
    with open("/proc/meminfo") as f:
        for ln in f:
            if ln.startswith("MemAvailable"):
                return int(ln.split()[1]) / 2**20
    return 0.0


def sample_indices(length, n, k=1 << 17, seed=0):
    rng = np.random.default_rng(seed)
    idx = [rng.integers(0, length, size=k, dtype=np.int64), np.arange(min(64, length)),
           np.arange(max(0, length - 64), length)]
    for c in range(1, n):
        b = c * length // n
        idx.append(np.arange(max(0, b - 4), min(length, b + 5)))
    return np.unique(np.concatenate(idx)).astype(np.int64)


def test_more_than_2_pow_32_elements(ra):
    # L = 2^32 + 1,000,003 bf16 per rank: element indices and byte offsets past 32 bits in every
    # kernel the call reaches (all-reduce on both engines, reduce-scatter, all-gather). Inputs
    # are drawn on the device; the oracle gets them at the sampled indices only, in host arrays
    # that are otherwise untouched zero pages.
    n, length, dtype = 2, (1 << 32) + 1_000_003, "bf16"
    need = 5 * n * length * 2 + (1 << 30)
    if torch.cuda.mem_get_info()[0] < need:
        pytest.skip("not enough free device memory")
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    sends = []
    for _ in range(n):
        x = torch.empty(length, dtype=torch.bfloat16, device="cuda")
        step = 1 << 28
        for a in range(0, length, step):
            b = min(length, a + step)
            x[a:b] = torch.randn(b - a, generator=g, device="cuda").to(torch.bfloat16)
        sends.append(x)
    recvs = [torch.empty_like(x) for x in sends]
    ra.ra_allreduce(sends, recvs, "sum")
    torch.cuda.synchronize()
    assert torch.equal(recvs[0].view(torch.int16), recvs[1].view(torch.int16))

    idx = sample_indices(length, n, k=1 << 16)
    near = np.concatenate([np.arange((1 << 31) - 8, (1 << 31) + 8), np.arange((1 << 32) - 8, (1 << 32) + 8)])
    idx = np.unique(np.concatenate([idx, near])).astype(np.int64)
    idx_dev = torch.from_numpy(idx).cuda()
    xs = []
    for x in sends:
        h = np.zeros(length, dtype=np.uint16)  # zero pages, touched only at the samples
        h[idx] = x[idx_dev].view(torch.int16).cpu().numpy().view(np.uint16)
        xs.append(h)
    want = oracle.fold_at(xs, "sum", dtype, idx)
    assert_same_bits(to_host(recvs[0][idx_dev], dtype), want, dtype, "AR sampled past 2^32")

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bulk = [torch.empty_like(x) for x in sends]
    ra.ra_allreduce_ex(sends, bulk, "sum", engine="bulk", status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(bulk[0].view(torch.int16), recvs[0].view(torch.int16)), "bulk engine differs"
    del bulk

    bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
    shards = [torch.empty(e - b, dtype=torch.bfloat16, device="cuda") for b, e in bounds]
    ra.ra_reduce_scatter(sends, shards, "sum")
    torch.cuda.synchronize()
    for c, (b, e) in enumerate(bounds):
        assert torch.equal(shards[c].view(torch.int16), recvs[0][b:e].view(torch.int16)), f"RS chunk {c}"
    del sends
    gathered = [torch.empty(length, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    ra.ra_allgather(shards, gathered)
    torch.cuda.synchronize()
    for r in range(n):
        assert torch.equal(gathered[r].view(torch.int16), recvs[0].view(torch.int16)), f"AG rank {r}"


ORACLE_TIMEOUT_MS = 600_000  # a full-size ring step moves up to 1 GiB per message on the host


def same_bits_fast(got, want, dtype, what):
    """Byte equality first (one pass); the NaN-aware comparison only to explain a difference."""
    if got.shape == want.shape and np.array_equal(got.view(np.uint8), want.view(np.uint8)):
        return
    assert_same_bits(got, want, dtype, what)


def compare_ranks(recvs, want, dtype, what):
    """Every element of every rank's device result against the oracle's, one rank at a time."""
    for r, t in enumerate(recvs):
        same_bits_fast(to_host(t, dtype), want[r], dtype, f"{what} rank {r}")


def check_full_size(ra, n, length, dtype, op, dist, rs_ag=False):
    """The workload in the bench's launch configuration, all N x L outputs against the oracle's
    message-passing ring run on the same full inputs (in place, so the host holds N x S once).
    With rs_ag, the reduce-scatter and the all-gather of its shards too: shard c must equal
    chunk c of the all-reduce and the gathered buffers the all-reduce (AG o RS = AR, pinned on
    the oracle), every element."""
    es = ELEM_SIZE[dtype]
    need_gb = (n + 2) * length * es / 2**30
    if _host_ram_gb() < need_gb + 4:
        pytest.skip(f"host RAM below {need_gb + 4:.0f} GB")
    xs = inputs.rank_buffers(n, length, dtype, dist)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    ra.ra_allreduce(sends, recvs, op)
    torch.cuda.synchronize()
    shards = gathered = None
    if rs_ag:
        bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
        shards = [torch.empty(e - b, dtype=TORCH_DTYPE[dtype], device="cuda") for b, e in bounds]
        ra.ra_reduce_scatter(sends, shards, op)
        del sends
        gathered = [torch.empty(length, dtype=TORCH_DTYPE[dtype], device="cuda") for _ in range(n)]
        ra.ra_allgather(shards, gathered)
        torch.cuda.synchronize()
    else:
        del sends
    want, _, _ = oracle.allreduce(xs, op, dtype, timeout_ms=ORACLE_TIMEOUT_MS, inplace=True)
    compare_ranks(recvs, want, dtype, f"AR n={n} L={length}")
    if rs_ag:
        for c, (b, e) in enumerate(bounds):
            same_bits_fast(to_host(shards[c], dtype), want[0][b:e], dtype, f"RS n={n} L={length} shard {c}")
        compare_ranks(gathered, want, dtype, f"AG(RS) n={n} L={length}")
    del recvs, shards, gathered
    torch.cuda.empty_cache()


def test_full_size_n8_f32_avg_64m(ra):
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_f32_avg_64m"]
    check_full_size(ra, n, length, dtype, op, dist, rs_ag=True)


def test_full_size_n8_bf16_avg_gpt2m(ra):
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_bf16_avg_gpt2m"]
    check_full_size(ra, n, length, dtype, op, dist, rs_ag=True)


@pytest.mark.parametrize("n,dtype,op", [(6, "bf16", "avg"), (7, "f16", "sum")])
def test_offgrid_16bit_reduce_scatter_from_512_mib(ra, n, dtype, op):
    # 16-bit reduce-scatters with shards off the vector grid at N = 5..7 take a one-trip launch
    # from 320 MiB over all ranks: every element of every shard against the oracle's ring
    length = (512 << 20) // ELEM_SIZE[dtype] // n + 5
    if _host_ram_gb() < 3 * n * length * ELEM_SIZE[dtype] / 2**30 + 4:
        pytest.skip("host RAM too small")
    xs = inputs.rank_buffers(n, length, dtype, ("normal", 1.0), seed_base=130 + n)
    sends = [to_device(x, dtype) for x in xs]
    bounds = [ra.ra_chunk_range(length, n, c) for c in range(n)]
    shards = [torch.empty(e - b, dtype=TORCH_DTYPE[dtype], device="cuda") for b, e in bounds]
    ra.ra_reduce_scatter(sends, shards, op)
    torch.cuda.synchronize()
    del sends
    assert any((b * ELEM_SIZE[dtype]) % ra.ra_vector_bytes() for b, _ in bounds), "no shard off the grid"
    want, _ = oracle.reduce_scatter(xs, op, dtype, timeout_ms=ORACLE_TIMEOUT_MS)
    del xs
    for c in range(n):
        same_bits_fast(to_host(shards[c], dtype), want[c], dtype, f"n={n} shard {c}")


def test_full_size_n8_bf16_avg_gpt2m_fp32_partials(ra):
    # the same bucket with fp32 partials, rounded once: every element against the oracle's ring
    # whose messages are fp32
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_bf16_avg_gpt2m"]
    if _host_ram_gb() < 2 * n * length * 2 / 2**30 + 6:
        pytest.skip("host RAM too small for the inputs and the oracle's outputs")
    xs = inputs.rank_buffers(n, length, dtype, dist)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    ra.ra_allreduce_ex(sends, recvs, op, accum="fp32")
    torch.cuda.synchronize()
    del sends
    want, _ = oracle.allreduce_ex(xs, op, dtype, accum="fp32", timeout_ms=ORACLE_TIMEOUT_MS)
    del xs
    compare_ranks(recvs, want, dtype, "fp32 partials, full bucket")
    del recvs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,length", [(n, 1 << p) for n in (8, 16) for p in (8, 10, 12, 14, 16, 18, 20)])
def test_size_sweep_small(ra, n, length):
    xs = inputs.rank_buffers(n, length, "f32", ("uniform", -1.0, 1.0))
    check_all(ra, xs, "sum", "f32", f"sweep n={n} L={length}")


@pytest.mark.parametrize("n,length", [(8, 1 << 24), (16, 1 << 26), (16, 1 << 28)])
def test_size_sweep_large(ra, n, length):
    check_full_size(ra, n, length, "f32", "sum", ("uniform", -1.0, 1.0))


# ---------------------------------------------------------------------------
# the literal schedule (one launch per ring step) against the oracle's steps
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("f16", "prod"), ("i32", "max"),
                                      ("f32", "avg"), ("bf16", "min")])
def test_ringsteps_final_result(ra, dtype, op):
    for n, length in ((1, 100), (2, 1001), (3, 1000), (4, 4096), (5, 1003), (8, 65536 + 3), (16, 999)):
        xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=n)
        want, _, _ = oracle.allreduce(xs, op, dtype)
        fused = run_allreduce(ra, xs, op, dtype)
        for inplace in (False, True):
            sends = [to_device(x, dtype) for x in xs]
            recvs = sends if inplace else [torch.empty_like(s) for s in sends]
            ra.ra_allreduce_ringsteps(sends, recvs, op)
            torch.cuda.synchronize()
            for r in range(n):
                got = to_host(recvs[r], dtype)
                assert_same_bits(got, want[r], dtype, f"n={n} L={length} rank {r} inplace={inplace}")
                assert got.tobytes() == fused[r].tobytes()


def test_ringsteps_intermediate_states(ra):
    # after k steps, every chunk a step has written holds the oracle's state at step k-1
    n, length, dtype, op = 5, 1003, "i32", "sum"
    xs = [np.full(length, 1 << r, dtype=np.int32) for r in range(n)]  # tags: partial = set of ranks
    _, _, snaps = oracle.allreduce(xs, op, dtype, snapshots=True)
    for k in range(1, 2 * (n - 1) + 1):
        sends = [to_device(x, dtype) for x in xs]
        recvs = [torch.zeros_like(s) for s in sends]
        ra.ra_allreduce_ringsteps(sends, recvs, op, nsteps=k)
        torch.cuda.synchronize()
        s = k - 1
        for r in range(n):
            c = (r - s - 1) % n if s < n - 1 else (r - (s - (n - 1))) % n
            b, e = oracle.chunk_range(length, n, c)
            assert (to_host(recvs[r], dtype)[b:e] == snaps[s, r, b:e]).all(), (k, r, c)


# ---------------------------------------------------------------------------
# fp32 accumulation (partials kept in fp32, rounded once) against the oracle's fp32-message ring
# ---------------------------------------------------------------------------
def _run_ex(ra, xs, op, dtype, order="ring", accum="dtype"):
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    ra.ra_allreduce_ex(sends, recvs, op, order=order, accum=accum)
    n, length = len(xs), xs[0].size
    shards = [torch.empty((c + 1) * length // n - c * length // n, dtype=TORCH_DTYPE[dtype], device="cuda")
              for c in range(n)]
    ra.ra_reduce_scatter_ex(sends, shards, op, order=order, accum=accum)
    torch.cuda.synchronize()
    return [to_host(r, dtype) for r in recvs], [to_host(s, dtype) for s in shards]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", OPS)
def test_fp32_accumulation(ra, dtype, op):
    # ragged lengths, and lengths whose shards all sit on the vector grid (the reduce-scatter then takes
    # a CTA per trip from N = 3)
    for n, length in ((1, 100), (2, 1001), (3, 4097), (6, 6 * 4099 + 5), (7, 30_011), (8, 65536 + 5), (16, 1003),
                      (64, 64 * 33 + 1), (3, 3 * 16 * 300), (4, 4 * 16 * 257), (5, 5 * 16 * 300), (7, 7 * 16 * 250),
                      (12, 12 * 16 * 100)):
        xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=n + 17)
        want, _ = oracle.allreduce_ex(xs, op, dtype, accum="fp32")
        got, shards = _run_ex(ra, xs, op, dtype, accum="fp32")
        for r in range(n):
            assert_same_bits(got[r], want[r], dtype, f"n={n} L={length} rank {r}")
            b, e = oracle.chunk_range(length, n, r)
            assert_same_bits(shards[r], want[0][b:e], dtype, f"RS n={n} shard {r}")


def test_fp32_accumulation_closed_form(ra):
    # rank 0 holds 256, 63 ranks hold 1: per-hop bf16 rounding stalls chunk 0 at 256, fp32 partials give 320
    n, length = 64, 64 * 64
    xs = [np.full(length, 0x3F80, dtype=np.uint16) for _ in range(n)]
    xs[0][:] = 0x4380
    hop, _ = _run_ex(ra, xs, "sum", "bf16", accum="dtype")
    acc, _ = _run_ex(ra, xs, "sum", "bf16", accum="fp32")
    b0, e0 = oracle.chunk_range(length, n, 0)
    assert (oracle.widen("bf16", hop[0][b0:e0]) == 256.0).all()
    assert (oracle.widen("bf16", acc[7]) == 320.0).all()


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_fp32_accumulation_is_identity_for_wide_types(ra, dtype):
    xs = inputs.rank_buffers(5, 10_003, dtype, dist_for(dtype, "sum"), seed_base=3)
    a, _ = _run_ex(ra, xs, "sum", dtype, accum="fp32")
    b = run_allreduce(ra, xs, "sum", dtype)
    assert all(x.tobytes() == y.tobytes() for x, y in zip(a, b))


# ---------------------------------------------------------------------------
# other reduction orders (double binary tree, Rabenseifner) against the oracle's
# message-passing simulations of those algorithms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("order", ["tree", "rabenseifner"])
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("f32", "avg"), ("bf16", "sum"), ("bf16", "avg"),
                                      ("f16", "prod"), ("f16", "max"), ("i32", "sum"), ("i32", "min"),
                                      ("bf16", "min"), ("f32", "prod")])
def test_other_orders(ra, order, dtype, op):
    ns = (1, 2, 4, 8, 16, 64) if order == "rabenseifner" else (1, 2, 3, 5, 7, 8, 16, 64)
    for n in ns:
        for length in (1, 13, 1003, 65536 + 7):
            xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=n + length)
            want, _ = oracle.allreduce_ex(xs, op, dtype, order=order)
            got, shards = _run_ex(ra, xs, op, dtype, order=order)
            for r in range(n):
                assert_same_bits(got[r], want[r], dtype, f"{order} n={n} L={length} rank {r}")
                b, e = oracle.chunk_range(length, n, r)
                assert_same_bits(shards[r], want[0][b:e], dtype, f"{order} RS n={n} shard {r}")


def test_other_orders_differ_from_ring_only_by_rounding(ra):
    # same values, different association: fp32 results agree with the ring to 1e-6 relative
    n, length = 8, 1 << 20
    xs = inputs.rank_buffers(n, length, "f32", ("uniform", 0.5, 1.0), seed_base=1)
    ring = run_allreduce(ra, xs, "sum", "f32")[0]
    for order in ("tree", "rabenseifner"):
        got, _ = _run_ex(ra, xs, "sum", "f32", order=order)
        np.testing.assert_allclose(got[0], ring, rtol=1e-6)
        assert not np.array_equal(got[0], ring)  # the order is observable


def test_rabenseifner_rejects_non_power_of_two(ra):
    xs = [torch.ones(10, device="cuda") for _ in range(3)]
    with pytest.raises(ra.RaError):
        ra.ra_allreduce_ex(xs, [torch.empty_like(x) for x in xs], "sum", order="rabenseifner")


@pytest.mark.parametrize("order", ["tree", "rabenseifner"])
def test_other_orders_full_size(ra, order):
    # the bench workload in tree / Rabenseifner order: every element of every rank against the
    # oracle's message-passing simulation of that algorithm on the same full inputs
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_f32_avg_64m"]
    if _host_ram_gb() < 2 * n * length * 4 / 2**30 + 6:
        pytest.skip("host RAM too small for the inputs and the oracle's outputs")
    xs = inputs.rank_buffers(n, length, dtype, dist)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    ra.ra_allreduce_ex(sends, recvs, op, order=order)
    torch.cuda.synchronize()
    del sends
    want, _ = oracle.allreduce_ex(xs, op, dtype, order=order, timeout_ms=ORACLE_TIMEOUT_MS)
    del xs
    compare_ranks(recvs, want, dtype, f"{order} full size")


# ---------------------------------------------------------------------------
# bucketed all-reduce (each bucket is its own all-reduce) and the SM budget
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("bf16", "avg"), ("i32", "max")])
def test_bucketed_allreduce(ra, dtype, op):
    counts = [1000, 3, 77, 4096, 10, 2048, 5, 65536, 1, 333]
    n, length = 5, sum(counts)
    es = ELEM_SIZE[dtype]
    plan = ra.ra_bucket_plan(counts, 3000 * es, es)
    assert len(plan) == 5
    xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=11)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.zeros_like(s) for s in sends]
    # gradients "become ready" on a producer stream; the collective waits on each bucket's event
    producer = torch.cuda.Stream()
    events = []
    with torch.cuda.stream(producer):
        for _ in plan:
            torch.cuda._sleep(20000)
            ev = torch.cuda.Event()
            ev.record(producer)
            events.append(ev)
    ra.ra_allreduce_buckets(sends, recvs, plan, op, ready_events=events)
    torch.cuda.synchronize()
    for b, c in plan:
        want, _, _ = oracle.allreduce([np.ascontiguousarray(x[b:b + c]) for x in xs], op, dtype)
        for r in range(n):
            assert_same_bits(to_host(recvs[r][b:b + c], dtype), want[r], dtype, f"bucket {b} rank {r}")


def _bucket_want(xs, b, c, op, dtype, accum):
    part = [np.ascontiguousarray(x[b:b + c]) for x in xs]
    if accum == "fp32":
        return oracle.allreduce_ex(part, op, dtype, accum="fp32")[0]
    return oracle.allreduce(part, op, dtype)[0]


@pytest.mark.parametrize("dtype,op,accum", [("f32", "sum", "dtype"), ("bf16", "avg", "dtype"), ("bf16", "avg", "fp32"),
                                            ("i32", "max", "dtype"), ("f16", "prod", "dtype"), ("f32", "avg", "dtype")])
def test_grouped_buckets(ra, dtype, op, accum):
    # buckets that need no wait between them go out as one grouped launch; a ready event on a
    # bucket starts a new group. Every bucket must equal its own all-reduce (own chunk bounds).
    counts = [1000, 3, 77, 4096, 10, 2048, 5, 65536, 1, 333, 70001, 12345, 7]
    es = ELEM_SIZE[dtype]
    plan = ra.ra_bucket_plan(counts, 5000 * es, es)
    length = sum(counts)
    for n in (1, 2, 3, 5, 6, 8, 16):
        xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=31 + n)
        for every in (0, 3):  # 0: no events (one group); 3: an event on every third bucket
            sends = [to_device(x, dtype) for x in xs]
            recvs = [torch.zeros_like(s) for s in sends]
            events = None
            if every:
                events = []
                for k in range(len(plan)):
                    ev = None
                    if k % every == 0:
                        ev = torch.cuda.Event()
                        ev.record()
                    events.append(ev)
            ra.ra_allreduce_buckets(sends, recvs, plan, op, ready_events=events, accum=accum)
            torch.cuda.synchronize()
            for b, c in plan:
                want = _bucket_want(xs, b, c, op, dtype, accum)
                for r in range(n):
                    assert_same_bits(to_host(recvs[r][b:b + c], dtype), want[r], dtype,
                                     f"n={n} every={every} bucket {b}+{c} rank {r}")


def test_grouped_buckets_many_and_empty(ra):
    # more buckets than one grouped launch holds (so the group is split), zero-length buckets, in
    # place, and ascending order
    n, dtype, op = 4, "f32", "sum"
    sizes = [(k * 37) % 211 for k in range(150)]  # includes zeros
    begins, at = [], 0
    for c in sizes:
        begins.append(at)
        at += c
    length = at
    plan = list(zip(begins, sizes))
    xs = inputs.rank_buffers(n, length, dtype, ("uniform", -1.0, 1.0), seed_base=5)
    sends = [to_device(x, dtype) for x in xs]
    ra.ra_allreduce_buckets(sends, sends, plan, op)
    torch.cuda.synchronize()
    for b, c in plan:
        if c == 0:
            continue
        want = _bucket_want(xs, b, c, op, dtype, "dtype")
        for r in range(n):
            assert_same_bits(to_host(sends[r][b:b + c], dtype), want[r], dtype, f"bucket {b}+{c} rank {r}")


def test_grouped_buckets_full_size_gpt2m(ra):
    # the 33 DDP buckets (25 MB cap) of the bf16 GPT-2-medium gradient, no ready events: grouped
    # launches; every element of every bucket against the oracle's ring run on that bucket
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_bf16_avg_gpt2m"]
    counts = [int(np.prod(s)) for _, s in inputs.gpt2_medium_param_shapes()]
    plan = ra.ra_bucket_plan(counts, 25 * 1000 * 1000, 2)
    assert len(plan) == 33
    if _host_ram_gb() < 2 * n * length * 2 / 2**30 + 6:
        pytest.skip("host RAM too small")
    xs = inputs.rank_buffers(n, length, dtype, dist)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    ra.ra_allreduce_buckets(sends, recvs, plan, op)
    torch.cuda.synchronize()
    del sends
    got = [to_host(r, dtype) for r in recvs]
    del recvs
    for b, c in plan:
        want = _bucket_want(xs, b, c, op, dtype, "dtype")
        for r in range(n):
            same_bits_fast(got[r][b:b + c], want[r], dtype, f"bucket {b}+{c} rank {r}")


def test_sm_budget_changes_nothing_but_speed(ra):
    n, length = 8, (1 << 22) + 5
    xs = inputs.rank_buffers(n, length, "bf16", ("normal", 1.0), seed_base=4)
    base = run_allreduce(ra, xs, "avg", "bf16")
    for max_sms in (1, 8, 76):
        sends = [to_device(x, "bf16") for x in xs]
        recvs = [torch.empty_like(s) for s in sends]
        ra.ra_allreduce_ex(sends, recvs, "avg", max_sms=max_sms)
        torch.cuda.synchronize()
        assert all(to_host(r, "bf16").tobytes() == b.tobytes() for r, b in zip(recvs, base))


# ---------------------------------------------------------------------------
# the bulk engine (TMA-staged loads): same bits as the register engine, bounded waits
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,op", [("f32", "sum"), ("f32", "avg"), ("bf16", "avg"), ("f16", "prod"),
                                      ("i32", "max"), ("bf16", "min")])
def test_bulk_engine(ra, dtype, op):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 384 consumer threads on an SM budget or below N = 8, else 128; from N = 9 on a budget the tiles
    # shrink below one vector per consumer so that two stages fit
    for n, length in ((1, 100), (2, 1 << 16), (3, 3 * 4096 * 7 + 11), (5, 1003), (8, (1 << 20) + 13),
                      (12, 12 * 4096 * 5 + 7), (16, 16 * 2048 * 5 + 3)):
        xs = inputs.rank_buffers(n, length, dtype, dist_for(dtype, op), seed_base=n + 90)
        want, _, _ = oracle.allreduce(xs, op, dtype)
        for max_sms, inplace in ((0, False), (16, False), (0, True)):
            sends = [to_device(x, dtype) for x in xs]
            recvs = sends if inplace else [torch.empty_like(s) for s in sends]
            ra.ra_allreduce_ex(sends, recvs, op, engine="bulk", status=status, max_sms=max_sms)
            torch.cuda.synchronize()
            for r in range(n):
                assert_same_bits(to_host(recvs[r], dtype), want[r], dtype,
                                 f"bulk n={n} L={length} sms={max_sms} inplace={inplace} rank {r}")
    assert status.item() == 0


def test_bulk_engine_full_size(ra):
    n, length, dtype, op, dist = inputs.WORKLOADS["ar_n8_f32_avg_64m"]
    xs = inputs.rank_buffers(n, length, dtype, dist)
    sends = [to_device(x, dtype) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ra.ra_allreduce_ex(sends, recvs, op, engine="bulk", status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    del sends
    want, _, _ = oracle.allreduce(xs, op, dtype, timeout_ms=ORACLE_TIMEOUT_MS, inplace=True)
    compare_ranks(recvs, want, dtype, "bulk full size")


def test_bulk_wait_runs_out_and_reports(ra):
    # one tile's bulk copies are withheld: the consumers' bounded wait gives up after 1 s, the kernel
    # records the code in the status word and finishes; the context stays usable
    n, length = 4, 4 * 1024 * 8
    xs = inputs.rank_buffers(n, length, "f32", ("normal", 1.0), seed_base=3)
    sends = [to_device(x, "f32") for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ra.ra_selftest_bulk_timeout(sends, recvs, status)
    torch.cuda.synchronize()
    assert status.item() in (1, 2)
    want, _, _ = oracle.allreduce(xs, "sum", "f32")
    status.zero_()
    ra.ra_allreduce_ex(sends, recvs, "sum", engine="bulk", status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_same_bits(to_host(recvs[1], "f32"), want[1], "f32", "after the self-test")


def test_bulk_wait_reports_in_the_withheld_chunks_word(ra):
    # per-chunk status words (the layout of the no-alloc entry point): chunk c's first tile is
    # withheld, so word c alone turns nonzero; every other chunk finishes and reports 0
    n, length, c = 4, 4 * 1024 * 8, 2
    xs = inputs.rank_buffers(n, length, "f32", ("normal", 1.0), seed_base=5)
    sends = [to_device(x, "f32") for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    words = torch.zeros(n, dtype=torch.int32, device="cuda")
    ra.ra_selftest_bulk_timeout(sends, recvs, words, withhold_chunk=c, per_chunk=True)
    torch.cuda.synchronize()
    codes = words.cpu().tolist()
    assert codes[c] in (1, 2) and all(codes[k] == 0 for k in range(n) if k != c), codes
    want, _, _ = oracle.allreduce(xs, "sum", "f32")
    for k in range(n):  # the chunks that finished hold their results
        if k == c:
            continue
        b, e = oracle.chunk_range(length, n, k)
        assert_same_bits(to_host(recvs[0], "f32")[b:e], want[0][b:e], "f32", f"chunk {k} beside the withheld one")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ra.ra_allreduce_ex(sends, recvs, "sum", engine="bulk", status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert_same_bits(to_host(recvs[3], "f32"), want[3], "f32", "after the self-test")
