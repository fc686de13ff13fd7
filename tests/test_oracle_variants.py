"""Pins for the oracle's other algorithms and accumulation (no GPU).

* fp32 accumulation (tirogla.com "Ring all-reduce", "Implementation notes":
  bf16 sums lose bits, accumulate in fp32): a closed form where per-hop bf16
  rounding stalls and fp32 accumulation does not; a numpy/torch fold in ring
  order over widened values; identity for fp32/int32 buffers.
* Rabenseifner (recursive halving / doubling, power-of-two N) and the double
  binary tree: integer results equal an order-free fold; float results equal
  a direct evaluation of the association each algorithm implies, written
  independently of the message passing; bytes sent match the pages' cost
  models (2(N-1)/N*S per rank for Rabenseifner, 2(N-1)*S in total for both).
"""

import numpy as np
import pytest
import torch

from test_oracle import _bf16_np, _bf16_t, assert_same_bits, lib_avg, lib_hop, small_inputs


# ---------------------------------------------------------------------------
# fp32 accumulation
# ---------------------------------------------------------------------------
def test_fp32_accumulation_closed_form(oracle):
    # 64 ranks, rank 0 holds 256 and every other rank 1. Chunk 0 starts its fold at 256:
    # with bf16 hops 256 + 1 ties back to 256 every time (ulp 2 at 256), so the ring gives 256.
    # Chunk 1 adds the 63 ones first (exact) and 256 last: 319 ties to 320. With fp32 partials
    # every chunk sums to 319 exactly, rounded once to bf16: 320.
    n, length = 64, 128
    xs = [np.full(length, 0x3F80, dtype=np.uint16) for _ in range(n)]  # 1.0
    xs[0][:] = 0x4380  # 256.0
    per_hop, _ = oracle.allreduce_ex(xs, "sum", "bf16", accum="dtype")
    acc32, _ = oracle.allreduce_ex(xs, "sum", "bf16", accum="fp32")
    b0, e0 = oracle.chunk_range(length, n, 0)
    b1, e1 = oracle.chunk_range(length, n, 1)
    w_hop, w_32 = oracle.widen("bf16", per_hop[5]), oracle.widen("bf16", acc32[5])
    assert (w_hop[b0:e0] == 256.0).all() and (w_hop[b1:e1] == 320.0).all()
    assert (w_32 == 320.0).all()


def _fp32_ring_fold(xs, op, dtype, n):
    length = xs[0].shape[0]
    wide = [(_bf16_t(x).float().numpy() if dtype == "bf16" else x.astype(np.float32)) for x in xs]
    w = np.stack(wide)
    cidx = np.empty(length, dtype=np.int64)
    for c in range(n):
        cidx[c * length // n:(c + 1) * length // n] = c
    cols = np.arange(length)
    acc = w[cidx, cols]
    for k in range(1, n):
        acc = lib_hop("f32", op, acc, w[(cidx + k) % n, cols])
    if op == "avg":
        acc = lib_avg("f32", n, acc)
    if dtype == "bf16":
        return _bf16_np(torch.from_numpy(acc).to(torch.bfloat16))
    return acc.astype(np.float16)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("op", ["sum", "avg", "prod", "min", "max"])
def test_fp32_accumulation_matches_widened_fold(oracle, dtype, op):
    for n in (1, 2, 3, 5, 8):
        for length in (1, 7, 64, 1003):
            xs = small_inputs(n, length, dtype, op, 300 + n)
            got, _ = oracle.allreduce_ex(xs, op, dtype, accum="fp32")
            want = _fp32_ring_fold(xs, op, dtype, n)
            for r in range(n):
                assert_same_bits(got[r], want, dtype, f"n={n} L={length} rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "i32"])
def test_fp32_accumulation_is_identity_for_wide_types(oracle, dtype):
    xs = small_inputs(5, 1003, dtype, "sum", 9)
    a, _ = oracle.allreduce_ex(xs, "sum", dtype, accum="fp32")
    b, _, _ = oracle.allreduce(xs, "sum", dtype)
    assert all(x.tobytes() == y.tobytes() for x, y in zip(a, b))


# ---------------------------------------------------------------------------
# Rabenseifner and double binary tree
# ---------------------------------------------------------------------------
def _pairwise_high_bit_first(vals, dtype, op):
    """Rabenseifner's association: level d = N/2, ..., 1 combines v[r] with v[r + d]."""
    v = list(vals)
    d = len(v) // 2
    while d >= 1:
        v = [lib_hop(dtype, op, v[r], v[r + d]) for r in range(d)]
        d //= 2
    return v[0]


def _inorder(seq, vals, dtype, op):
    """Double binary tree association: fold(left subtree), own value, fold(right subtree)."""
    if not seq:
        return None
    m = (len(seq) - 1) // 2
    left = _inorder(seq[:m], vals, dtype, op)
    right = _inorder(seq[m + 1:], vals, dtype, op)
    acc = vals[seq[m]] if left is None else lib_hop(dtype, op, left, vals[seq[m]])
    return acc if right is None else lib_hop(dtype, op, acc, right)


def _tree_fold(xs, op, dtype):
    n, length = len(xs), xs[0].shape[0]
    split = (n // 2) * length // n
    out = np.empty_like(xs[0])
    fwd, bwd = list(range(n)), list(range(n - 1, -1, -1))
    for seq, lo, hi in ((fwd, 0, split), (bwd, split, length)):
        if hi > lo:
            out[lo:hi] = _inorder(seq, [x[lo:hi] for x in xs], dtype, op)
    return lib_avg(dtype, n, out) if op == "avg" else out


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "avg", "prod", "min", "max"])
def test_rabenseifner_association(oracle, dtype, op):
    for n in (1, 2, 4, 8, 16):
        for length in (1, 5, 64, 1000):
            xs = small_inputs(n, length, dtype, op, 500 + n)
            got, _ = oracle.allreduce_ex(xs, op, dtype, order="rabenseifner")
            want = _pairwise_high_bit_first(xs, dtype, op)
            if op == "avg":
                want = lib_avg(dtype, n, want)
            for r in range(n):
                assert_same_bits(got[r], want, dtype, f"n={n} L={length} rank {r}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16", "i32"])
@pytest.mark.parametrize("op", ["sum", "avg", "prod", "min", "max"])
def test_double_tree_association(oracle, dtype, op):
    for n in (1, 2, 3, 4, 5, 7, 8, 16):
        for length in (1, 5, 64, 1000):
            xs = small_inputs(n, length, dtype, op, 700 + n)
            got, _ = oracle.allreduce_ex(xs, op, dtype, order="tree")
            want = _tree_fold(xs, op, dtype)
            for r in range(n):
                assert_same_bits(got[r], want, dtype, f"n={n} L={length} rank {r}")


@pytest.mark.parametrize("order", ["tree", "rabenseifner"])
@pytest.mark.parametrize("op", ["sum", "prod", "min", "max"])
def test_other_orders_integer_results_are_order_free(oracle, order, op):
    for n in (2, 4, 8):
        xs = small_inputs(n, 999, "i32", op, 40 + n)
        got, _ = oracle.allreduce_ex(xs, op, "i32", order=order)
        x = np.stack(xs).astype(np.int64)
        want = {"sum": x.sum(0), "prod": x.prod(0), "min": x.min(0), "max": x.max(0)}[op]
        want = ((want + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32)
        assert np.array_equal(got[0], want)


@pytest.mark.parametrize("n", [2, 4, 8, 16])
def test_rabenseifner_bytes(oracle, n):
    # recursive halving sends S/2 + S/4 + ... + S/N, doubling the same again: 2(N-1)/N*S per rank
    length = 64 * n
    xs = small_inputs(n, length, "f32", "sum", 2)
    _, sent = oracle.allreduce_ex(xs, "sum", "f32", order="rabenseifner")
    s_bytes = length * 4
    assert all(int(b) * n == 2 * (n - 1) * s_bytes for b in sent)


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_double_tree_bytes(oracle, n):
    # every tree edge carries its half once up and once down: 2(N-1) * S in total over both trees
    length = 60 * n
    xs = small_inputs(n, length, "f32", "sum", 2)
    _, sent = oracle.allreduce_ex(xs, "sum", "f32", order="tree")
    assert int(sent.sum()) == 2 * (n - 1) * length * 4


def test_rabenseifner_needs_power_of_two(oracle):
    xs = small_inputs(3, 10, "f32", "sum", 1)
    with pytest.raises(oracle.OracleError) as ei:
        oracle.allreduce_ex(xs, "sum", "f32", order="rabenseifner")
    assert ei.value.status == "unsupported"


def test_fp32_accumulation_only_for_the_ring(oracle):
    xs = small_inputs(4, 10, "bf16", "sum", 1)
    with pytest.raises(oracle.OracleError):
        oracle.allreduce_ex(xs, "sum", "bf16", order="tree", accum="fp32")
