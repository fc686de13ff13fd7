"""Seeded synthetic inputs for the ring all-reduce workloads.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It holds no part of the reduction: it only draws per-rank buffers from
numpy's ``default_rng`` (seed = base + rank) and stores them in the buffer
dtype. Every returned array is 1-D and contiguous in the dtype's storage:
float32, float16, int32, or bf16 as uint16 bit patterns.

Recipes (value distributions of the workloads described on the pages and in
the benchmark configuration):

* ``int_uniform(lo, hi)``: integers in [lo, hi], stored exactly in the dtype;
* ``normal(sigma)``: N(0, sigma) drawn in float32, rounded to the dtype;
* ``uniform(lo, hi)``: U(lo, hi) drawn in float32, rounded to the dtype.

Rounding float32 to float16 uses numpy's cast, to bf16 torch's CPU cast (both
round to nearest even); which converter made the inputs does not matter for
parity, since both sides receive the same bits.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i32": np.int32}
ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}

# chunk of draws per call, to bound host memory for very large buffers
_BLOCK = 1 << 24


def _f32_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return x.astype(np.float32, copy=False)
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        import torch

        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    if dtype == "i32":
        return x.astype(np.int32)
    raise ValueError(dtype)


def rank_buffer(rank: int, length: int, dtype: str, dist: tuple, seed_base: int = 0) -> np.ndarray:
    """One rank's buffer: ``dist`` is ("int_uniform", lo, hi) | ("normal", sigma) | ("uniform", lo, hi)."""
    rng = np.random.default_rng(seed_base + rank)
    out = np.empty(length, dtype=STORAGE[dtype])
    kind = dist[0]
    for s in range(0, length, _BLOCK):
        m = min(_BLOCK, length - s)
        if kind == "int_uniform":
            v = rng.integers(dist[1], dist[2] + 1, size=m, dtype=np.int64)
            if dtype == "i32":
                out[s:s + m] = v.astype(np.int32)
            else:
                out[s:s + m] = _f32_to_storage(v.astype(np.float32), dtype)
        elif kind == "normal":
            v = rng.standard_normal(m, dtype=np.float32) * np.float32(dist[1])
            out[s:s + m] = _f32_to_storage(v, dtype)
        elif kind == "uniform":
            v = rng.uniform(dist[1], dist[2], size=m).astype(np.float32)
            out[s:s + m] = _f32_to_storage(v, dtype)
        else:
            raise ValueError(f"unknown distribution {dist!r}")
    return out


def rank_buffers(n: int, length: int, dtype: str, dist: tuple, seed_base: int = 0,
                 workers: int | None = None) -> list[np.ndarray]:
    """All ranks' buffers. Ranks are drawn on ``workers`` threads (default: one per rank up to
    the host's cores) once a buffer is large; each rank has its own generator, so the bits do
    not depend on the thread count."""
    if workers is None:
        workers = min(n, os.cpu_count() or 1) if length >= _BLOCK else 1
    if workers <= 1 or n <= 1:
        return [rank_buffer(r, length, dtype, dist, seed_base) for r in range(n)]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(lambda r: rank_buffer(r, length, dtype, dist, seed_base), range(n)))


# ---- the named workloads ---------------------------------------------------
# GPT-2-medium-like parameter list (24 layers, d = 1024, vocab 50257, 1024
# positions): the flat gradient bucket of the bf16 workload is their
# concatenation. Only the total length matters to the collective.
def gpt2_medium_param_shapes() -> list[tuple[str, tuple[int, ...]]]:
    d, v, t, layers = 1024, 50257, 1024, 24
    shapes = [("wte", (v, d)), ("wpe", (t, d))]
    for i in range(layers):
        shapes += [
            (f"h{i}.ln_1.weight", (d,)), (f"h{i}.ln_1.bias", (d,)),
            (f"h{i}.attn.c_attn.weight", (d, 3 * d)), (f"h{i}.attn.c_attn.bias", (3 * d,)),
            (f"h{i}.attn.c_proj.weight", (d, d)), (f"h{i}.attn.c_proj.bias", (d,)),
            (f"h{i}.ln_2.weight", (d,)), (f"h{i}.ln_2.bias", (d,)),
            (f"h{i}.mlp.c_fc.weight", (d, 4 * d)), (f"h{i}.mlp.c_fc.bias", (4 * d,)),
            (f"h{i}.mlp.c_proj.weight", (4 * d, d)), (f"h{i}.mlp.c_proj.bias", (d,)),
        ]
    shapes += [("ln_f.weight", (d,)), ("ln_f.bias", (d,))]
    return shapes


def gpt2_medium_numel() -> int:
    total = 0
    for _, shp in gpt2_medium_param_shapes():
        k = 1
        for s in shp:
            k *= s
        total += k
    return total


# name -> (nranks, length, dtype, op, distribution)
WORKLOADS = {
    # 4 ranks x 4096 fp32, integer-valued in [-8, 8]: every sum is exact
    "ar_n4_f32_sum_4k": (4, 4096, "f32", "sum", ("int_uniform", -8, 8)),
    # 8 ranks x 64 Mi fp32 gradient-like values, averaged
    "ar_n8_f32_avg_64m": (8, 64 * 1024 * 1024, "f32", "avg", ("normal", 1e-3)),
    # 8 ranks x one flat bf16 bucket of a GPT-2-medium-like model, averaged
    "ar_n8_bf16_avg_gpt2m": (8, 354_823_168, "bf16", "avg", ("normal", 1e-2)),
}


def sweep_cases():
    """The op/dtype sweep with uneven chunk bounds: 1,000,003 elements per rank."""
    cases = []
    for n in (2, 3, 5, 7):
        for op in ("sum", "min", "max", "prod"):
            cases.append((n, 1_000_003, "i32", op, ("int_uniform", -2, 2) if op == "prod"
                          else ("int_uniform", -1000, 1000)))
            cases.append((n, 1_000_003, "f16", op, ("normal", 1.0)))
    return cases


def size_sweep():
    """Message sizes 1 KiB .. 1 GiB per rank (fp32, powers of two) at 8 and 16 ranks."""
    out = []
    for n in (8, 16):
        for p in range(8, 29):
            out.append((n, 1 << p, "f32", "sum", ("uniform", -1.0, 1.0)))
    return out
