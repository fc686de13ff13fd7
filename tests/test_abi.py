"""The C-ABI library on the host, without a GPU: it loads, exports every symbol
include/ra.h declares, plans chunks as the tirogla.com page defines them, and
rejects bad arguments and overlapping buffers before launching anything."""

import ctypes
import os
import re

import numpy as np

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def ra():
    from ring_all_reduce_02_gb300 import build, ra as binding

    build.build()
    return binding


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ra.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?(ra_[a-z_0-9]+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol(ra):
    names = declared_symbols()
    assert "ra_allreduce" in names and "ra_reduce_scatter" in names and "ra_allgather" in names
    lib = ctypes.CDLL(ra.LIB_PATH)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ra.h but not exported"
    assert set(ra.EXPORTS) == set(names)


def test_stream_probes_build_and_export(ra):
    # the measurement kernels behind bench.py --roofs (not the collective path)
    from ring_all_reduce_02_gb300 import build

    probe = ctypes.CDLL(build.build_probe())
    for name in ("rp_store", "rp_load", "rp_copy", "rp_copy_sms", "rp_copy_n", "rp_read_n"):
        assert hasattr(probe, name), name


def test_chunk_range_is_floor_definition(ra):
    for n in range(1, 65):
        for count in list(range(0, 40)) + [1003, 1_000_003, 354_823_168, 1 << 28, (1 << 57) - 1]:
            for c in range(n):
                assert ra.ra_chunk_range(count, n, c) == (c * count // n, (c + 1) * count // n)


@pytest.mark.parametrize("es", [2, 4])
@pytest.mark.parametrize("align", [16, 32, 128, 512])
def test_plan_splits_each_chunk_exactly_once(ra, es, align):
    vb_bytes = ra.ra_vector_bytes()
    assert vb_bytes in (16, 32)
    if align < vb_bytes:
        pytest.skip(f"the grid is at least one {vb_bytes}-byte vector")
    v, a = vb_bytes // es, align // es
    for n in (1, 2, 3, 5, 7, 8, 16, 64):
        for count in list(range(0, 70, 3)) + [1003, 4096, 1_000_003]:
            for phase in range(0, align, max(es, align // 8)):
                covered = 0
                head = ((align - phase) % align) // es
                for c in range(n):
                    b, e, vb, ve = ra.ra_plan_chunk(count, n, c, es, phase, align)
                    assert (b, e) == (c * count // n, (c + 1) * count // n)
                    assert b <= vb <= ve <= e
                    # the first aligned grid point at or after b
                    first = head if b <= head else head + -(-(b - head) // a) * a
                    if ve > vb:
                        assert vb == first and (ve - vb) % v == 0
                        assert e - ve < v  # runs to the last whole vector
                    else:
                        assert vb == ve == b
                        assert first + v > e  # no whole vector fits after the aligned start
                    covered += e - b
                assert covered == count


def test_plan_rejects_bad_phase(ra):
    # the default alignment (one vector) is accepted
    b, e, vb, ve = ra.ra_plan_chunk(1000, 4, 1, 4, 0)
    assert (b, e) == (250, 500) and b <= vb <= ve <= e and (ve - vb) % (ra.ra_vector_bytes() // 4) == 0
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 4, 0, ra.ra_vector_bytes() // 2)  # alignment below one vector
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 4, 2)  # phase not a multiple of the element size
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 3, 0)
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 4, 0, 48)  # alignment not a power of two
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 4, 16, 16)  # phase beyond the alignment


# Fake, never-dereferenced device addresses: every case below is rejected on the
# host before any CUDA call, so no GPU is needed.
BASE = 0x7F0000000000
MB = 1 << 20


def bufs(n, stride=MB, base=BASE, offset=0):
    return [base + offset + r * stride for r in range(n)]


@pytest.mark.parametrize("name", ["ra_allreduce", "ra_reduce_scatter", "ra_allgather"])
def test_invalid_arguments(ra, name):
    call = ra.call
    s, d = bufs(4), bufs(4, base=BASE + 64 * MB)
    assert call(name, s, d, 1000, 0, 0, 0, 0) == ra.RA_ERR_INVALID_ARG       # nranks 0
    assert call(name, bufs(65), bufs(65, base=BASE + 256 * MB), 10, 0, 0, 65, 0) == ra.RA_ERR_INVALID_ARG
    assert call(name, s, d, 1000, 7, 0, 4, 0) == ra.RA_ERR_INVALID_ARG       # dtype
    if name != "ra_allgather":
        assert call(name, s, d, 1000, 0, 9, 4, 0) == ra.RA_ERR_INVALID_ARG   # op
    assert call(name, s, d, 1 << 57, 0, 0, 4, 0) == ra.RA_ERR_INVALID_ARG    # count too big
    assert call(name, [s[0], 0, s[2], s[3]], d, 1000, 0, 0, 4, 0) == ra.RA_ERR_INVALID_ARG  # null
    assert call(name, s, [d[0] + 2] + d[1:], 1000, 0, 0, 4, 0) == ra.RA_ERR_INVALID_ARG  # misaligned f32
    assert call(name, s, d, 0, 0, 0, 4, 0) == ra.RA_SUCCESS                   # nothing to do
    f = getattr(ra.lib(), name)
    assert f(None, ra.ptr_array(d), 10, 0, 0, 4, None) == ra.RA_ERR_INVALID_ARG


def test_ex_options(ra):
    s, d = bufs(4), bufs(4, base=BASE + 64 * MB)
    for name in ("ra_allreduce_ex", "ra_reduce_scatter_ex"):
        assert ra.call_ex(name, s, d, 1000, 0, 0, 4, 7, 0, 0) == ra.RA_ERR_INVALID_ARG   # order
        assert ra.call_ex(name, s, d, 1000, 0, 0, 4, 0, 5, 0) == ra.RA_ERR_INVALID_ARG   # accum
        assert ra.call_ex(name, s, d, 1000, 0, 0, 4, 0, 0, 0, max_sms=-1) == ra.RA_ERR_INVALID_ARG
        assert ra.call_ex(name, s[:3], d[:3], 1000, 0, 0, 3, 2, 0, 0) == ra.RA_ERR_UNSUPPORTED  # halving, N=3
        assert ra.call_ex(name, s, d, 1000, 2, 0, 4, 1, 1, 0) == ra.RA_ERR_UNSUPPORTED  # fp32 accum + tree
        assert ra.call_ex(name, s, d, 0, 0, 0, 4, 0, 1, 0) == ra.RA_SUCCESS
    # the bulk engine: needs a status word, covers the ring all-reduce with dtype accumulation up to 16 ranks
    status = BASE + 512 * MB
    assert ra.call_ex("ra_allreduce_ex", s, d, 1000, 0, 0, 4, 0, 0, 0, engine=1) == ra.RA_ERR_INVALID_ARG
    assert ra.call_ex("ra_allreduce_ex", s, d, 1000, 0, 0, 4, 0, 0, 0, engine=5, status=status) == ra.RA_ERR_INVALID_ARG
    assert ra.call_ex("ra_reduce_scatter_ex", s, d, 1000, 0, 0, 4, 0, 0, 0, engine=1, status=status) == \
        ra.RA_ERR_UNSUPPORTED
    assert ra.call_ex("ra_allreduce_ex", s, d, 1000, 2, 0, 4, 1, 0, 0, engine=1, status=status) == ra.RA_ERR_UNSUPPORTED
    assert ra.call_ex("ra_allreduce_ex", s, d, 1000, 2, 0, 4, 0, 1, 0, engine=1, status=status) == ra.RA_ERR_UNSUPPORTED
    s20, d20 = bufs(20), bufs(20, base=BASE + 128 * MB)
    assert ra.call_ex("ra_allreduce_ex", s20, d20, 1000, 0, 0, 20, 0, 0, 0, engine=1, status=status) == \
        ra.RA_ERR_UNSUPPORTED
    # NULL options = defaults
    f = ra.lib().ra_allreduce_ex
    assert f(ra.ptr_array(s), ra.ptr_array(d), 0, 0, 0, 4, None, None) == ra.RA_SUCCESS


def test_zero_length_shards_may_be_null(ra):
    # count 3 over 4 ranks: chunk 0 is empty, so its compact buffer may be NULL; the call
    # then passes every host check and only fails at the CUDA step (no GPU here)
    s = bufs(4)
    d = [0] + bufs(3, base=BASE + 64 * MB)
    st = ra.call("ra_reduce_scatter", s, d, 3, 0, 0, 4, 0)
    assert st in (ra.RA_SUCCESS, ra.RA_ERR_CUDA)


def test_alias_rules(ra):
    call = ra.call
    n, count, es = 4, 1000, 4
    s = bufs(n)
    # all-reduce: exact in place is fine (reaches the CUDA step), any other overlap is rejected
    assert call("ra_allreduce", s, s, count, 0, 0, n, 0) in (ra.RA_SUCCESS, ra.RA_ERR_CUDA)
    assert call("ra_allreduce", s, [s[0] + 4] + s[1:], count, 0, 0, n, 0) == ra.RA_ERR_ALIAS
    assert call("ra_allreduce", s, [s[1]] + s[1:], count, 0, 0, n, 0) == ra.RA_ERR_ALIAS
    d = bufs(n, base=BASE + 64 * MB)
    assert call("ra_allreduce", s, [d[0], d[0] + 16, d[2], d[3]], count, 0, 0, n, 0) == ra.RA_ERR_ALIAS
    # send buffers may overlap each other (only read)
    assert call("ra_allreduce", [s[0]] * n, d, count, 0, 0, n, 0) in (ra.RA_SUCCESS, ra.RA_ERR_CUDA)
    # reduce-scatter in place: recv[r] = send[r] + begin_r
    b = [r * count // n for r in range(n)]
    rs_inplace = [s[r] + b[r] * es for r in range(n)]
    assert call("ra_reduce_scatter", s, rs_inplace, count, 0, 0, n, 0) in (ra.RA_SUCCESS, ra.RA_ERR_CUDA)
    assert call("ra_reduce_scatter", s, [s[r] for r in range(n)], count, 0, 0, n, 0) in (
        ra.RA_ERR_ALIAS,) or b[1] == 0
    # all-gather in place: send[r] = recv[r] + begin_r
    r_full = bufs(n, base=BASE + 128 * MB)
    ag_inplace = [r_full[r] + b[r] * es for r in range(n)]
    assert call("ra_allgather", ag_inplace, r_full, count, 0, 0, n, 0) in (ra.RA_SUCCESS, ra.RA_ERR_CUDA)
    wrong = list(ag_inplace)
    wrong[1] = r_full[1]  # overlaps its own recv buffer at the wrong place
    assert call("ra_allgather", wrong, r_full, count, 0, 0, n, 0) == ra.RA_ERR_ALIAS


def test_status_strings(ra):
    for st in range(5):
        assert isinstance(ra.ra_status_string(st), str) and ra.ra_status_string(st)
    assert ra.ra_status_string(99) == "unknown status"


def test_product_path_has_no_fallback(ra, monkeypatch):
    # the binding refuses to run without the library rather than computing anything itself
    import ring_all_reduce_02_gb300.ra as binding

    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", "/nonexistent/libra.so")
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def _ddp_buckets(counts, cap_bytes, es):
    """The DDP packing rule written out: reverse order, close a bucket before it would exceed the cap."""
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    out, cur, cur_bytes = [], [], 0
    for p in reversed(range(len(counts))):
        if cur and cur_bytes + counts[p] * es > cap_bytes:
            out.append((offs[cur[-1]], offs[cur[0] + 1] - offs[cur[-1]]))
            cur, cur_bytes = [], 0
        cur.append(p)
        cur_bytes += counts[p] * es
    if cur:
        out.append((offs[cur[-1]], offs[cur[0] + 1] - offs[cur[-1]]))
    return out


def test_bucket_plan_gpt2_medium(ra):
    from ring_all_reduce_02_gb300 import inputs

    counts = [int(np.prod(s)) for _, s in inputs.gpt2_medium_param_shapes()]
    cap = 25 * 1000 * 1000
    plan = ra.ra_bucket_plan(counts, cap, 2)
    assert plan == _ddp_buckets(counts, cap, 2)
    # buckets tile the flat buffer from its end to its start, each within the cap unless it is one parameter
    assert plan[0][0] + plan[0][1] == sum(counts) and plan[-1][0] == 0
    for (b0, c0), (b1, c1) in zip(plan, plan[1:]):
        assert b1 + c1 == b0
    big = {c for c in counts if c * 2 > cap}
    for b, c in plan:
        assert c * 2 <= cap or c in big
    assert len(plan) > 10


def test_bucket_plan_edge_cases(ra):
    assert ra.ra_bucket_plan([], 100, 4) == []
    assert ra.ra_bucket_plan([10], 4, 4) == [(0, 10)]        # larger than the cap: its own bucket
    assert ra.ra_bucket_plan([1, 1, 1, 1], 8, 4) == [(2, 2), (0, 2)]
    rng = np.random.default_rng(0)
    for _ in range(200):
        counts = [int(x) for x in rng.integers(0, 50, size=rng.integers(1, 30))]
        cap = int(rng.integers(1, 300))
        assert ra.ra_bucket_plan(counts, cap, 4) == _ddp_buckets(counts, cap, 4)


def test_bucketed_allreduce_checks_buckets(ra):
    s, d = bufs(2), bufs(2, base=BASE + 64 * MB)
    f = ra.lib().ra_allreduce_buckets
    C = ctypes.c_size_t

    def run(begins, counts):
        m = len(begins)
        return f(ra.ptr_array(s), ra.ptr_array(d), 1000, 0, 0, 2, m, (C * m)(*begins), (C * m)(*counts), None, None,
                 None)

    assert run([0, 400], [500, 100]) == ra.RA_ERR_INVALID_ARG      # overlapping
    assert run([900], [200]) == ra.RA_ERR_INVALID_ARG              # past the end
    assert run([0, 600, 300], [100, 100, 100]) == ra.RA_ERR_INVALID_ARG  # not monotonic
