"""Pins for the CPU oracle: it is checked against what the pages print and what
the mathematics fixes, never against itself or the CUDA path.

* values the pages print (golden fixtures under tests/golden, each cited);
* the step-by-step traces of the pages (ring all-gather, ring reduce-scatter,
  the chunk-0 journey), compared through per-step snapshots;
* the closed form of the tirogla.com self-test;
* invariants (ownership of chunk (r+1) after reduce-scatter, bytes sent,
  identical results on every rank, all-reduce == all-gather after
  reduce-scatter);
* a brute-force fold in ring order built from numpy / torch CPU arithmetic
  (a different implementation of every hop) on all small shapes;
* the rounding of one fp16/bf16 hop against the exact result rounded once;
* IEEE minimum/maximum special cases, int32 wrap, host-side fault injection.
"""

import itertools
import time

import numpy as np
import pytest
import torch

from conftest import golden_lines
from ring_all_reduce_02_gb300 import inputs

DTYPES = ["f32", "f16", "bf16", "i32"]
OPS = ["sum", "avg", "min", "max", "prod"]


# ---------------------------------------------------------------------------
# helpers: NaN-aware bit comparison and an independent brute-force fold
# ---------------------------------------------------------------------------
def is_nan_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype in ("f32", "f16"):
        return np.isnan(a)
    if dtype == "bf16":
        return ((a & 0x7F80) == 0x7F80) & ((a & 0x007F) != 0)
    return np.zeros(a.shape, dtype=bool)


def assert_same_bits(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    assert got.shape == want.shape, what
    gn, wn = is_nan_bits(got, dtype), is_nan_bits(want, dtype)
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    ok = gn | (got.view(np.uint8).reshape(got.shape[0], -1) == want.view(np.uint8).reshape(
        want.shape[0], -1)).all(axis=1) if got.size else gn
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, f"{what}: {bad.size} elements differ, first at {bad[:5]}: got {got[bad[:5]]} want {want[bad[:5]]}"


def _bf16_t(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


def _bf16_np(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def lib_hop(dtype, op, a, b):
    """One hop with library arithmetic: numpy for f32/f16/i32, torch CPU for bf16."""
    if dtype == "bf16":
        ta, tb = _bf16_t(a), _bf16_t(b)
        f = {"sum": torch.add, "avg": torch.add, "prod": torch.mul,
             "min": torch.minimum, "max": torch.maximum}[op]
        return _bf16_np(f(ta, tb))
    f = {"sum": np.add, "avg": np.add, "prod": np.multiply, "min": np.minimum, "max": np.maximum}[op]
    with np.errstate(all="ignore"):
        return f(a, b)


def lib_avg(dtype, n, a):
    if dtype == "f32":
        return a * (np.float32(1.0) / np.float32(n))
    if dtype == "f16":
        return (a.astype(np.float32) * (np.float32(1.0) / np.float32(n))).astype(np.float16)
    if dtype == "bf16":
        inv = float(np.float32(1.0) / np.float32(n))
        return _bf16_np((_bf16_t(a).float() * torch.tensor(inv, dtype=torch.float32)).to(torch.bfloat16))
    a64 = a.astype(np.int64)
    return (np.sign(a64) * (np.abs(a64) // n)).astype(np.int32)


def brute_fold(xs, op, dtype):
    """Element i of chunk c = floor bounds c*L//N: left fold x_c, x_{c+1}, ... (mod N)."""
    n, length = len(xs), xs[0].shape[0]
    x = np.stack(xs)
    cidx = np.empty(length, dtype=np.int64)
    for c in range(n):
        cidx[c * length // n:(c + 1) * length // n] = c
    cols = np.arange(length)
    acc = x[cidx, cols]
    for k in range(1, n):
        acc = lib_hop(dtype, op, acc, x[(cidx + k) % n, cols])
    if op == "avg":
        acc = lib_avg(dtype, n, acc)
    return acc


def small_inputs(n, length, dtype, op, seed):
    if dtype == "i32":
        dist = ("int_uniform", -2, 2) if op == "prod" else ("int_uniform", -1000, 1000)
    else:
        dist = ("normal", 1.0)
    return inputs.rank_buffers(n, length, dtype, dist, seed_base=seed)


# ---------------------------------------------------------------------------
# chunk bounds
# ---------------------------------------------------------------------------
def test_chunk_bounds_floor_definition(oracle):
    # tirogla "Ring all-reduce", section "Code": chunk c = [c*len/n, (c+1)*len/n)
    for n in range(1, 65):
        for length in list(range(0, 70)) + [1003, 1_000_003, 354_823_168, (1 << 40) - 3]:
            for c in range(n):
                assert oracle.chunk_range(length, n, c) == (c * length // n, (c + 1) * length // n)


def test_chunk_bounds_selftest_shape(oracle):
    # the page's self-test: 5 ranks x 1003 elements -> chunks 200/201/200/201/201
    sizes = [e - b for b, e in (oracle.chunk_range(1003, 5, c) for c in range(5))]
    assert sizes == [200, 201, 200, 201, 201]


def test_chunk_bounds_64bit(oracle):
    # c*L overflows 32 (and near 2^40 would overflow 64 without care) bits
    for length, n in [(1 << 28, 16), (354_823_168, 8), ((1 << 40) - 1, 64)]:
        bounds = [oracle.chunk_range(length, n, c) for c in range(n)]
        assert bounds[0][0] == 0 and bounds[-1][1] == length
        for (b0, e0), (b1, _) in zip(bounds, bounds[1:]):
            assert e0 == b1
        sizes = {e - b for b, e in bounds}
        assert max(sizes) - min(sizes) <= 1


# ---------------------------------------------------------------------------
# values and traces printed on the pages
# ---------------------------------------------------------------------------
def test_tirogla_selftest_closed_form(oracle):
    kv = dict(ln.split() for ln in golden_lines("tirogla_selftest.txt"))
    n, length = int(kv["ranks"]), int(kv["length"])
    xs = [np.arange(length, dtype=np.float64).astype(np.float32) + np.float32(r * length) for r in range(n)]
    outs, _, _ = oracle.allreduce(xs, "sum", "f32")
    want = (int(kv["expect_offset"]) + int(kv["expect_slope"]) * np.arange(length)).astype(np.float32)
    for o in outs:
        assert np.array_equal(o, want)


def _parse_row(s):
    return [list(map(int, part.split(","))) for part in s.split("|")]


def test_infra_guide_examples(oracle):
    for ln in golden_lines("infra_guide_examples.txt"):
        case, op, rest = ln.split(None, 2)
        lhs, rhs = rest.split("->")
        ins, want = _parse_row(lhs.replace(" ", "")), _parse_row(rhs.replace(" ", ""))
        n = len(ins)
        if case == "allreduce":
            xs = [np.array(v, dtype=np.int32) for v in ins]
            outs, _, _ = oracle.allreduce(xs, op, "i32")
            # the same example in fp32 gives the same exact values
            outs_f, _, _ = oracle.allreduce([x.astype(np.float32) for x in xs], op, "f32")
            for o, of, w in zip(outs, outs_f, want):
                assert o.tolist() == w and of.tolist() == w
        elif case == "reduce_scatter":
            xs = [np.array(v, dtype=np.int32) for v in ins]
            outs, _ = oracle.reduce_scatter(xs, op, "i32")
            assert [o.tolist() for o in outs] == want
        elif case == "allgather":
            length = sum(len(v) for v in ins)
            shards = [np.array(v, dtype=np.int32) for v in ins]
            outs, _, _ = oracle.allgather(shards, length, "i32")
            assert [o.tolist() for o in outs] == want
        else:
            raise AssertionError(case)
        assert n == 4


def test_ramchalamkr_examples(oracle):
    for ln in golden_lines("ramchalamkr_examples.txt"):
        lhs, rhs = ln.split("->")
        case, n, m, fills = lhs.split()
        n, m = int(n), int(m)
        fills = list(map(int, fills.split(",")))
        if case == "allreduce":
            xs = [np.full(m, f, dtype=np.float32) for f in fills]
            outs, _, _ = oracle.allreduce(xs, "sum", "f32")
            want = float(rhs.split()[1])
            assert all((o == want).all() for o in outs)
        else:
            shards = [np.full(m, f, dtype=np.float32) for f in fills]
            outs, _, _ = oracle.allgather(shards, n * m, "f32")
            want = list(map(float, rhs.split(",")))
            assert all(o.tolist() == want for o in outs)


def test_bitfern_example(oracle):
    lhs, rhs = golden_lines("bitfern_example.txt")[0].split("->")
    xs = [np.array([v], dtype=np.float32) for v in map(float, lhs.split())]
    outs, _, _ = oracle.allreduce(xs, "sum", "f32")
    assert all(o[0] == float(rhs) for o in outs)


def test_ramchalamkr_allgather_trace(oracle):
    tag = {"A": 1, "B": 2, "C": 3, "D": 4, "_": 0}
    rows = {}
    for ln in golden_lines("ramchalamkr_allgather_trace.txt"):
        step, gpu, *slots = ln.split()
        rows[(int(step), int(gpu))] = [tag[s] for s in slots]
    shards = [np.array([tag["ABCD"[r]]], dtype=np.int32) for r in range(4)]
    outs, _, snaps = oracle.allgather(shards, 4, "i32", snapshots=True)
    for (step, gpu), want in rows.items():
        if step == 0:
            continue  # the initial placement: checked through the first step's carry-over
        assert snaps[step - 1, gpu].tolist() == want, (step, gpu)
    assert all(o.tolist() == [1, 2, 3, 4] for o in outs)


def _contributors(term: str) -> int:
    mask = 0
    for t in term.split("+"):
        mask |= 1 << int(t[1:] if t[0].isalpha() else t)
    return mask


def test_ramchalamkr_reduce_scatter_trace(oracle):
    # tag rank r's value with the bit 1<<r: an int32 sum of distinct tags is the set of ranks
    n = 4
    xs = [np.full(4, 1 << r, dtype=np.int32) for r in range(n)]
    outs, _, snaps = oracle.allreduce(xs, "sum", "i32", snapshots=True)
    for ln in golden_lines("ramchalamkr_reduce_scatter_trace.txt"):
        f = ln.split()
        if f[0] == "final":
            gpu, chunk, terms = int(f[1]), int(f[2]), f[3]
            assert snaps[n - 2, gpu, chunk] == _contributors(terms)
            continue
        step, gpu = int(f[0]), int(f[1])
        want = [_contributors(t) for t in f[2:]]
        assert snaps[step - 1, gpu].tolist() == want, (step, gpu)
    assert all((o == 15).all() for o in outs)


def test_arjunsriva_chunk0_journey(oracle):
    n = 4
    xs = [np.full(8, 1 << r, dtype=np.int32) for r in range(n)]  # 2 elements per chunk
    _, _, snaps = oracle.allreduce(xs, "sum", "i32", snapshots=True)
    b, e = oracle.chunk_range(8, n, 0)
    for ln in golden_lines("arjunsriva_chunk0_trace.txt"):
        frame, holder, terms = ln.split()
        frame, holder = int(frame), int(holder)
        want = _contributors(terms)
        if frame == 0:
            assert (xs[holder][b:e] == want).all()
        else:
            assert (snaps[frame - 1, holder, b:e] == want).all(), frame


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", range(2, 17))
def test_ownership_after_reduce_scatter(oracle, n):
    # tirogla "How it works": after N-1 steps rank r holds the complete chunk (r+1) mod N
    length = 3 * n + 2
    xs = [np.full(length, 1 << r, dtype=np.int32) for r in range(n)]
    _, _, snaps = oracle.allreduce(xs, "sum", "i32", snapshots=True)
    full = (1 << n) - 1
    for r in range(n):
        for c in range(n):
            b, e = oracle.chunk_range(length, n, c)
            complete = (snaps[n - 2, r, b:e] == full).all()
            assert complete == (c == (r + 1) % n), (r, c)


@pytest.mark.parametrize("n,length", [(2, 10), (3, 1000), (4, 4096), (5, 1003), (7, 64), (8, 4096), (16, 999)])
def test_bytes_sent(oracle, n, length):
    # per-rank bytes 2(N-1)/N*S when N | L; exactly 2S - |C_{r+1}| - |C_{r+2}| in general;
    # the ring moves 2(N-1)*S bytes in total (tirogla "How it works"; infra-guide 4.3)
    xs = small_inputs(n, length, "f32", "sum", 3)
    _, sent, _ = oracle.allreduce(xs, "sum", "f32")
    es = 4
    size = [oracle.chunk_range(length, n, c) for c in range(n)]
    size = [(e - b) * es for b, e in size]
    s_bytes = length * es
    for r in range(n):
        assert sent[r] == 2 * s_bytes - size[(r + 1) % n] - size[(r + 2) % n]
        if length % n == 0:
            assert sent[r] * n == 2 * (n - 1) * s_bytes
    assert int(sent.sum()) == 2 * (n - 1) * s_bytes
    # standalone all-gather: (N-1)/N * S per rank (ramchalamkr section 1)
    shards = [np.zeros((oracle.chunk_range(length, n, c)[1] - oracle.chunk_range(length, n, c)[0]),
                       dtype=np.float32) for c in range(n)]
    _, sent_ag, _ = oracle.allgather(shards, length, "f32")
    for r in range(n):
        assert sent_ag[r] == s_bytes - size[(r + 1) % n]


# ---------------------------------------------------------------------------
# brute force on every small shape, all dtypes and ops
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,op", list(itertools.product(DTYPES, OPS)))
def test_brute_force_small(oracle, dtype, op):
    seed = 11
    for n in range(1, 8):
        for length in list(range(0, 18)) + [31, 64]:
            xs = small_inputs(n, length, dtype, op, seed)
            seed += 1
            outs, _, _ = oracle.allreduce(xs, op, dtype)
            want = brute_fold(xs, op, dtype) if length else np.empty(0, dtype=xs[0].dtype)
            for r, o in enumerate(outs):
                assert_same_bits(o, want, dtype, f"n={n} L={length} rank {r}")
            if length == 0:
                continue
            # every rank byte-identical (tirogla "Implementation notes": replicas do not drift)
            for o in outs[1:]:
                assert o.tobytes() == outs[0].tobytes()
            # the per-element definition agrees
            fa = oracle.fold_at(xs, op, dtype, np.arange(length))
            assert_same_bits(fa, want, dtype, "fold_at")
            # reduce-scatter gives chunk r to rank r, and all-gather of those is the all-reduce
            # (infra-guide 3.8: AllReduce = ReduceScatter + AllGather)
            shards, _ = oracle.reduce_scatter(xs, op, dtype)
            for c in range(n):
                b, e = oracle.chunk_range(length, n, c)
                assert_same_bits(shards[c], want[b:e], dtype, f"rs shard {c}")
            ag, _, _ = oracle.allgather(shards, length, dtype)
            for o in ag:
                assert o.tobytes() == outs[0].tobytes()


@pytest.mark.parametrize("op", ["sum", "prod", "min", "max"])
def test_int_ops_order_free(oracle, op):
    # integer sum/prod (mod 2^32), min and max do not depend on the order of the fold
    for n in (2, 3, 5, 7):
        xs = small_inputs(n, 257, "i32", op, 100 + n)
        outs, _, _ = oracle.allreduce(xs, op, "i32")
        x = np.stack(xs).astype(np.int64)
        want = {"sum": x.sum(0), "prod": x.prod(0), "min": x.min(0), "max": x.max(0)}[op]
        want = ((want + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)
        assert np.array_equal(outs[0], want)


def test_ring_order_is_observable(oracle):
    # fp32: the ring fold of chunk c starts at x_c. With x_c = 1 and every other rank
    # 2^-24, each hop 1 + 2^-24 ties back to 1 (round half to even), while a fold that
    # starts elsewhere accumulates 2^-23 first and ends at 1 + 2^-22.
    n, length = 4, 8
    tiny = np.float32(2.0 ** -24)
    for c in range(n):
        b, e = oracle.chunk_range(length, n, c)
        xs = [np.full(length, tiny, dtype=np.float32) for _ in range(n)]
        xs[c][b:e] = 1.0
        outs, _, _ = oracle.allreduce(xs, "sum", "f32")
        assert (outs[0][b:e] == np.float32(1.0)).all()
        other = np.float32(0)
        for k in range(1, n + 1):  # a fold starting at x_{c+1}
            other = np.float32(other + xs[(c + k) % n][b])
        assert other == np.float32(1.0 + 2.0 ** -22)


# ---------------------------------------------------------------------------
# rounding of one hop and of the conversions
# ---------------------------------------------------------------------------
def test_widen_exhaustive(oracle):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got16 = oracle.widen("f16", h)
    want16 = h.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(got16), np.isnan(want16))
    m = ~np.isnan(want16)
    assert np.array_equal(got16[m].view(np.uint32), want16[m].view(np.uint32))
    gotb = oracle.widen("bf16", h)
    wantb = _bf16_t(h).float().numpy()
    assert np.array_equal(np.isnan(gotb), np.isnan(wantb))
    m = ~np.isnan(wantb)
    assert np.array_equal(gotb[m].view(np.uint32), wantb[m].view(np.uint32))


def _f32_sample(rng):
    # every 251st fp32 bit pattern (all exponents, both signs), the neighbourhood of every
    # fp16/bf16 rounding boundary in a few binades, and random patterns
    strided = np.arange(0, 1 << 32, 251, dtype=np.uint64).astype(np.uint32)
    ties = []
    for e in list(range(-30, 20)) + [120, 126, 127]:
        base = int(np.float32(2.0 ** e).view(np.uint32))
        for low in (1 << 12, 1 << 13, 1 << 15, 1 << 16):  # half-ulp positions for fp16 / bf16
            for k in range(8):
                mid = base + k * 2 * low + low
                ties += [mid - 1, mid, mid + 1]
    ties = np.array(ties, dtype=np.uint32)
    ties = np.concatenate([ties, ties | np.uint32(0x80000000)])
    rand = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([strided, ties, rand]).view(np.float32)


def test_round_f32_to_f16_against_numpy(oracle):
    x = _f32_sample(np.random.default_rng(5))
    got = oracle.round_f32("f16", x)
    want = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert ((got[nan] & 0x7C00) == 0x7C00).all() and ((got[nan] & 0x03FF) != 0).all()


def test_round_f32_to_bf16_against_torch(oracle):
    x = _f32_sample(np.random.default_rng(6))
    got = oracle.round_f32("bf16", x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], want[~nan])
    assert ((got[nan] & 0x7F80) == 0x7F80).all() and ((got[nan] & 0x007F) != 0).all()


def _round_double_to_bits(x: np.ndarray, p: int) -> np.ndarray:
    """Round doubles (normal range of the target, no overflow) to p significant bits,
    ties to even, with numpy's frexp / rint (rint rounds halves to even)."""
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, p)), e - p)


@pytest.mark.parametrize("op", ["sum", "prod"])
def test_f16_hop_is_correctly_rounded(oracle, op):
    # one fp16 hop = the exact result (exact in float64) rounded once to fp16
    rng = np.random.default_rng(7)
    a = rng.integers(0, 1 << 16, size=1 << 21, dtype=np.uint32).astype(np.uint16)
    b = rng.integers(0, 1 << 16, size=1 << 21, dtype=np.uint32).astype(np.uint16)
    # near-ties: b chosen so a+b lands half an fp16 ulp off a representable value
    fa, fb = a.view(np.float16), b.view(np.float16)
    keep = np.isfinite(fa) & np.isfinite(fb)
    fa, fb = fa[keep], fb[keep]
    exact = fa.astype(np.float64) + fb.astype(np.float64) if op == "sum" else fa.astype(np.float64) * fb.astype(np.float64)
    got = oracle.hop("f16", op, fa, fb)
    with np.errstate(over="ignore"):
        want = exact.astype(np.float16)  # numpy rounds the double once, to nearest even
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint16), want[~nan].view(np.uint16))


@pytest.mark.parametrize("op", ["sum", "prod"])
def test_bf16_hop_is_correctly_rounded(oracle, op):
    # one bf16 hop = the exact result rounded once to 8 significant bits; operands are drawn so
    # the exact result is a float64 and stays in bf16's normal range
    rng = np.random.default_rng(8)
    n = 1 << 20
    sign = rng.integers(0, 2, size=(2, n), dtype=np.uint32) << 15
    exps = rng.integers(110, 141, size=(2, n), dtype=np.uint32)  # 2^-17 .. 2^13: sums exact in float64
    mant = rng.integers(0, 128, size=(2, n), dtype=np.uint32)
    bits = (sign | (exps << 7) | mant).astype(np.uint16)
    a, b = bits[0], bits[1]
    fa = oracle.widen("bf16", a).astype(np.float64)
    fb = oracle.widen("bf16", b).astype(np.float64)
    assert np.array_equal(fa, _bf16_t(a).double().numpy())  # decoding agrees with torch
    exact = fa + fb if op == "sum" else fa * fb
    nz = exact != 0
    want = np.zeros_like(exact)
    want[nz] = _round_double_to_bits(exact[nz], 8)
    got = oracle.widen("bf16", oracle.hop("bf16", op, a, b)).astype(np.float64)
    assert np.array_equal(got, want)


def test_minimum_maximum_special_values(oracle):
    # IEEE 754-2019 minimum/maximum: NaN propagates, -0 < +0
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    a = np.array([0.0, -0.0, nan, 1.0, -inf, 3.0], dtype=np.float32)
    b = np.array([-0.0, 0.0, 1.0, nan, 5.0, 3.0], dtype=np.float32)
    mn, mx = oracle.hop("f32", "min", a, b), oracle.hop("f32", "max", a, b)
    assert np.signbit(mn[0]) and np.signbit(mn[1]) and mn[0] == 0 and mn[1] == 0
    assert not np.signbit(mx[0]) and not np.signbit(mx[1])
    assert np.isnan(mn[2]) and np.isnan(mn[3]) and np.isnan(mx[2]) and np.isnan(mx[3])
    assert mn[4] == -inf and mx[4] == 5.0 and mn[5] == 3.0 and mx[5] == 3.0
    for dt in ("f16", "bf16"):
        bits_a = oracle.round_f32(dt, a)
        bits_b = oracle.round_f32(dt, b)
        if dt == "f16":
            bits_a, bits_b = bits_a.view(np.float16), bits_b.view(np.float16)
        mn16 = oracle.widen(dt, oracle.hop(dt, "min", bits_a, bits_b).view(np.uint16))
        mx16 = oracle.widen(dt, oracle.hop(dt, "max", bits_a, bits_b).view(np.uint16))
        assert np.signbit(mn16[0]) and np.signbit(mn16[1]) and not np.signbit(mx16[0]) and not np.signbit(mx16[1])
        assert np.isnan(mn16[2]) and np.isnan(mx16[3])


def test_int32_wraps(oracle):
    a = np.array([2**31 - 1, -2**31, 65536, -7], dtype=np.int32)
    b = np.array([1, -1, 65536, 2], dtype=np.int32)
    assert oracle.hop("i32", "sum", a, b).tolist() == [-2**31, 2**31 - 1, 131072, -5]
    assert oracle.hop("i32", "prod", a, b).tolist() == [2**31 - 1, -2**31, 0, -14]
    # int32 avg: wrapped sum, then C division (toward zero)
    xs = [np.array([-7, 7], dtype=np.int32), np.array([0, 0], dtype=np.int32)]
    outs, _, _ = oracle.allreduce(xs, "avg", "i32")
    assert outs[0].tolist() == [-3, 3]


def test_avg_epilogue_exact_for_power_of_two(oracle):
    # avg at N = 8 multiplies by 0.125: exact, so avg == sum / 8 bit for bit
    for dt in ("f32", "f16", "bf16"):
        xs = small_inputs(8, 100, dt, "sum", 40)
        s, _, _ = oracle.allreduce(xs, "sum", dt)
        a, _, _ = oracle.allreduce(xs, "avg", dt)
        if dt == "bf16":
            want = oracle.round_f32("bf16", oracle.widen("bf16", s[0]) / np.float32(8))
        else:
            want = (s[0].astype(np.float32) / np.float32(8)).astype(s[0].dtype)
        assert a[0].tobytes() == want.tobytes()


def test_single_rank_is_identity(oracle):
    for dt in DTYPES:
        for op in OPS:
            xs = small_inputs(1, 33, dt, op, 9)
            outs, sent, _ = oracle.allreduce(xs, op, dt)
            assert outs[0].tobytes() == xs[0].tobytes() and int(sent.sum()) == 0


def test_inplace_matches_out_of_place(oracle):
    xs = small_inputs(5, 1003, "bf16", "sum", 21)
    outs, _, _ = oracle.allreduce([x.copy() for x in xs], "sum", "bf16")
    ins = [x.copy() for x in xs]
    inpl, _, _ = oracle.allreduce(ins, "sum", "bf16", inplace=True)
    for a, b in zip(outs, inpl):
        assert a.tobytes() == b.tobytes()


# ---------------------------------------------------------------------------
# host-side fault injection: a rank that stops sending becomes a timeout, not a hang
# (tirogla "Pitfalls": mismatched collective order across ranks hangs with no error)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fault_step", [0, 2, 5])
def test_missing_rank_times_out(oracle, fault_step):
    n = 4
    xs = small_inputs(n, 64, "f32", "sum", 1)
    t0 = time.time()
    with pytest.raises(oracle.OracleError) as ei:
        oracle.allreduce(xs, "sum", "f32", timeout_ms=200, fault_rank=1, fault_step=fault_step)
    assert ei.value.status == "timeout"
    assert time.time() - t0 < n * 0.2 + 5


def test_invalid_args(oracle):
    xs = small_inputs(2, 8, "f32", "sum", 1)
    with pytest.raises(oracle.OracleError):
        oracle.chunk_range(8, 0, 0)
    with pytest.raises(oracle.OracleError):
        oracle.chunk_range(8, 4, 4)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.allreduce(xs * 40, "sum", "f32")  # 80 ranks > 64
    assert ei.value.status == "invalid"
