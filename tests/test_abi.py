"""The C-ABI library on the host, without a GPU: it loads, exports every symbol
include/ra.h declares, plans chunks as the tirogla.com page defines them, and
rejects bad arguments and overlapping buffers before launching anything."""

import ctypes
import os
import re

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


def test_chunk_range_is_floor_definition(ra):
    for n in range(1, 65):
        for count in list(range(0, 40)) + [1003, 1_000_003, 354_823_168, 1 << 28, (1 << 57) - 1]:
            for c in range(n):
                assert ra.ra_chunk_range(count, n, c) == (c * count // n, (c + 1) * count // n)


@pytest.mark.parametrize("es", [2, 4])
def test_plan_splits_each_chunk_exactly_once(ra, es):
    v = 16 // es
    for n in (1, 2, 3, 5, 7, 8, 16, 64):
        for count in list(range(0, 70)) + [1003, 4096, 1_000_003]:
            for phase in range(0, 16, es):
                covered = 0
                head = ((16 - phase) % 16) // es
                for c in range(n):
                    b, e, vb, ve = ra.ra_plan_chunk(count, n, c, es, phase)
                    assert (b, e) == (c * count // n, (c + 1) * count // n)
                    assert b <= vb <= ve <= e
                    if ve > vb:
                        assert (vb - head) % v == 0 and (ve - vb) % v == 0 and vb >= head
                        # maximal: fewer than V elements at either end of the chunk
                        assert vb - b < v and e - ve < v
                    else:
                        assert vb == ve == b
                        # no whole vector fits on the grid inside the chunk
                        first = head if b <= head else head + -(-(b - head) // v) * v
                        assert first + v > e
                    covered += e - b
                assert covered == count


def test_plan_rejects_bad_phase(ra):
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 4, 2)  # phase not a multiple of the element size
    with pytest.raises(ra.RaError):
        ra.ra_plan_chunk(100, 4, 0, 3, 0)


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
