// Fused ring collectives of N virtual ranks held in one GPU's HBM.
//
// The ring of the tirogla.com page "Ring all-reduce" ("How it works") moves
// chunk c from rank c to c+1, ..., c+N-1 during reduce-scatter, combining it
// with each rank's own copy; the finished chunk is then copied to every rank
// by all-gather. On one GPU every "message" of that schedule would be a round
// trip through HBM. Here the 2(N-1) steps collapse into one pass per element:
// a thread loads x_0[i] .. x_{N-1}[i] once, folds them in the ring's order for
// the chunk that holds i (x_c first), rounds at every hop exactly as the
// message would be rounded, and stores the result once per destination. The
// partial sums stay in registers, so HBM sees only the algorithmic bytes:
// all-reduce N*S read + N*S written, reduce-scatter N*S + S, all-gather S + N*S.
//
// Work mapping: blockIdx.y = chunk c, so every CTA of a row folds in the same
// rank order and derives the chunk's bounds once; blockIdx.x splits the
// chunk's vectors among the row's CTAs (the shape's kUnroll vectors per thread
// per trip, loads of up to kBatch ranks issued back to back before they are
// folded). The elements of each chunk before its first line boundary and
// after its last whole vector, and every element when the buffers do not
// share one address phase, go through the per-element path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ra_ops.cuh"
#include "ra_plan.h"

#ifndef RA_MAX_RANKS
#define RA_MAX_RANKS 64
#endif

namespace ra {

// Launch shapes of the fused AR/RS kernels. How many bytes a thread keeps in
// flight is N loads x kUnroll vectors, so the rank count decides how many
// threads per SM and vectors per thread keep HBM busiest; the host planner
// picks the shape from N. Measured on GB300 with 32-byte vectors (fraction of
// the copy bandwidth, fp32, 1 GiB over all ranks): all-reduce N <= 2: 99% with
// 128 threads x 2 vectors at 4 CTAs/SM, loads of 2 ranks at a time (95% with
// 128 x 1 at 8 CTAs/SM); N = 3: 98% with 256 x 4 at 1 CTA/SM;
// N = 4..7: 95-99% with 256 x 1 at 2 CTAs/SM (the wide shape: 90-92% at
// N = 6, 7); N >= 8: 256 x 2 at 1 CTA/SM (99.5% at N = 8, 97% at N = 12 and
// 16). Reduce-scatter reads N values per element and writes one. Up to N = 3
// loads of 2 ranks at a time suit it (max at N = 3 98% against 89% with 4):
// 128 x 1 with registers for 6 CTAs/SM (98-101%), except fp16/bf16
// sum/avg/prod at 8 CTAs/SM (97-98%, against 88% at 6); from N = 4 sum/avg
// keep batches of 4 (96-102%) and min/max take 128 x 2 with batches of 2
// (96-103%, against 91-99%).
// How a chunk's vectors are dealt to the CTAs of its row. Every warp moves 32
// consecutive vectors (1 KB with 32-byte vectors) per unroll slot and trip.
//  0: grid-stride by CTA: trip k of CTA x covers the CTA-sized block x of the
//     trip; the last, partial trip then falls on the row's first CTAs only.
//     Since CTA x of every chunk lands on the same SM, those SMs run it while
//     the rest idle.
//  1: each CTA streams one contiguous slab of the chunk.
//  2: grid-stride by warp: the warps of a trip are dealt across the row's CTAs
//     (warp slot s of CTA x takes block s * gridDim.x + x), so the partial last
//     trip is spread over every CTA, and every SM, of the row.
#ifndef RA_SCHEDULE
#define RA_SCHEDULE 2
#endif

// Programmatic dependent launch. With RA_PDL set (the default), the
// collective kernels are launched with programmatic stream serialization, so
// the driver prepares a launch while the kernel before it on the stream is
// still running and starts it as that kernel's last CTA exits, instead of
// after the usual gap between kernels. Each kernel's threads wait
// (griddepcontrol.wait) until the previous grid has completed and its writes
// are visible before any global load or store, so the stream order is kept.
// On GB300, 16-32 MiB all-reduces launched back to back gained 2-4 points of
// the copy bandwidth, and the 33 DDP buckets of a GPT-2-medium gradient ran
// 1.6% faster. The kernels do not signal their dependents early
// (griddepcontrol.launch_dependents): CTAs of the next launch then sat on the
// SMs beside a running kernel that left registers free, and the fp32
// reduce-scatter at N = 3 ran at half speed.
#ifndef RA_PDL
#define RA_PDL 1
#endif

__device__ __forceinline__ void pdl_enter() {
#if RA_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Launch `kernel` on `s`, as a programmatic dependent launch when RA_PDL is
// set; returns the launch error (and consumes it).
template <typename... P, typename... A>
cudaError_t launch_programmatic(void (*kernel)(P...), dim3 grid, unsigned threads, size_t smem, cudaStream_t s,
                                A&&... args) {
#if RA_PDL
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<A&&>(args)...);
  const cudaError_t last = cudaGetLastError();
  return err != cudaSuccess ? err : last;
#else
  kernel<<<grid, threads, smem, s>>>(static_cast<A&&>(args)...);
  return cudaGetLastError();
#endif
}

template <int THREADS, int MIN_BLOCKS, int UNROLL, int BATCH>
struct Shape {
  static constexpr int kThreads = THREADS;       // threads per CTA
  static constexpr int kMinBlocks = MIN_BLOCKS;  // resident CTAs per SM the registers are budgeted for
  static constexpr int kUnroll = UNROLL;         // vectors per thread per trip
  static constexpr int kBatch = BATCH;           // ranks whose loads are in flight together
};
#ifndef RA_TUNE_SHAPE
using ShapeS = Shape<128, 8, 1, 4>;   // sum/avg/prod reduce-scatter nranks >= 4; fp16/bf16 sum/avg/prod
                                      // all-reduce and fp32 partials at nranks 1..2
using ShapeS4 = Shape<128, 4, 2, 2>;  // other all-reduces at nranks 1..2
using ShapeRS2 = Shape<128, 8, 1, 2>; // fp16/bf16 sum/avg/prod reduce-scatter nranks 1..3; fp32 partials below 8
using ShapeRS6 = Shape<128, 6, 1, 2>; // other reduce-scatters at nranks 1..3
using ShapeRS = Shape<128, 8, 2, 2>;  // min/max reduce-scatter nranks >= 4
using ShapeN3 = Shape<256, 1, 4, 4>;  // all-reduce nranks 3
using ShapeM = Shape<256, 2, 1, 4>;   // all-reduce nranks 4..5, fp16/bf16 sum/avg/prod at 8..15; fp32 partials
using ShapeW = Shape<256, 1, 2, 4>;   // all-reduce nranks >= 8
using ShapeM3 = Shape<256, 3, 1, 4>;  // fp16/bf16 at nranks 3 and min/max at 12..15; fp32 partials at 3
using ShapeMB8 = Shape<256, 2, 1, 8>; // fp16/bf16 sum/avg/prod at nranks 6: all six ranks' loads at once
using ShapeW8 = Shape<256, 1, 2, 8>;  // all-reduce nranks 6..7 (not fp16/bf16 sum/avg/prod at 6)
#else  // tuning sweeps: one shape (RA_TUNE_T, _MB, _U, _B) for every rank count
using ShapeS = Shape<RA_TUNE_T, RA_TUNE_MB, RA_TUNE_U, RA_TUNE_B>;
using ShapeN3 = ShapeS;
using ShapeM = ShapeS;
using ShapeW = ShapeS;
using ShapeM3 = ShapeS;
using ShapeS4 = ShapeS;
using ShapeRS2 = ShapeS;
using ShapeRS6 = ShapeS;
using ShapeRS = ShapeS;
using ShapeMB8 = ShapeS;
using ShapeW8 = ShapeS;
#endif
// Shapes of one-trip launches (a CTA per trip of the chunk; each CTA does one
// trip and exits). Short-lived CTAs stream HBM faster on GB300 than resident
// ones that grid-stride, and with one trip per CTA the occupancy the registers
// allow is what keeps bytes in flight, so these shapes are small. From sweeps
// of seven shapes (fp32 and bf16, avg and max, 128 MiB and 1 GiB over all
// ranks, back to back): all-reduce N = 3..16 103-105% of the copy bandwidth at
// 1 GiB with 128 x 1 at 8 CTAs/SM and loads of 4 ranks (the one-wave shapes:
// 96-100%), 91-98% at 128 MiB (85-94%); reduce-scatter from N = 8 104-107%
// (100-104%), min/max on 128 x 2 at 4 CTAs/SM.
// fp32 partials take TripS for the all-reduce (bf16 avg: 102.5-104.8% at 1 GiB,
// N = 3..16, against 95.9-99.5% one-wave) and TripAccRS (below) for the
// reduce-scatter (TripS, with loads of 4 ranks, would spill there).
using TripS = Shape<128, 8, 1, 4>;
using TripRS2 = Shape<128, 4, 2, 4>;
// N <= 2 has too few loads per thread on TripS to keep HBM busy; 128 x 2 at 8
// CTAs/SM with loads of 2 ranks, from five candidates (fp32 and bf16, avg and
// max, N = 1, 2, back to back): all-reduce 104-105.5% at 1 GiB over all ranks,
// 101.5-104% at 256 MiB, 94-102.5% at 64 MiB, against 98-100%, 96-96.6% and
// 86-90% on the one-wave shapes; reduce-scatter 104.7-106.9% at 1 GiB against
// 95.7-100%. At N = 3 the all-reduce already takes TripS, and a reduce-scatter
// on this shape lost 20 points to one wave (fp32, shards off the vector grid);
// with every shard on the grid, reduce-scatters take it up to N = 4, and up to
// N = 7 for 16-bit types and float min/max (106-108.7% at 1 GiB).
using TripW = Shape<128, 8, 2, 2>;
// fp32 partials in the reduce-scatter: 128 x 1 at 8 CTAs/SM with loads of 2
// ranks (bf16 avg, shards on the vector grid, N = 3..16): 100.4-103.9% at 1 GiB
// over all ranks, 94.5-95.6% at 256 MiB and 86.6-89.1% at 128 MiB from N = 6,
// against 98.9-103.8%, 76.7-96.7% and 79.7-91.8% on TripRS2 (128 x 2 at 4
// CTAs/SM, loads of 4 ranks); 128 x 2 at 4 CTAs/SM with loads of 2 measured
// between the two.
using TripAccRS = Shape<128, 8, 1, 2>;
// SHAPE_RS_OFFGRID(_B2, _M): a reduce-scatter with some compact output off the
// vector grid at a 2-byte offset, on ShapeS, or on ShapeRS2 (where the plain
// call would take loads of 2 ranks at a time; _M: with fp32 partials).
enum ShapeId {
  SHAPE_S = 0,
  SHAPE_N3 = 1,
  SHAPE_M = 2,
  SHAPE_W = 3,
  SHAPE_RS_OFFGRID = 4,
  SHAPE_STEP = 5,
  SHAPE_RS_OFFGRID_M = 6,
  SHAPE_M3 = 7,
  SHAPE_S4 = 8,
  SHAPE_RS2 = 9,
  SHAPE_RS = 10,
  SHAPE_RS_OFFGRID_B2 = 11,
  SHAPE_MB8 = 12,
  SHAPE_RS6 = 13,
  SHAPE_W8 = 14,
  SHAPE_TRIP_S = 15,    // TripS, one trip per CTA (all-reduce; reduce-scatter sum/avg/prod)
  SHAPE_TRIP_RS2 = 16,  // TripRS2, one trip per CTA (reduce-scatter min/max)
  SHAPE_TRIP_ACC = 17,  // TripS, one trip per CTA, fp32 partials (all-reduce)
  SHAPE_TRIP_ACC_RS2 = 18,  // TripAccRS, one trip per CTA, fp32 partials (reduce-scatter)
  SHAPE_TRIP_RS_OFFGRID = 19,  // TripS, one trip per CTA, reduce-scatter with 2-byte-offset shards
  SHAPE_TRIP_W = 20,           // TripW, one trip per CTA (small N)
  SHAPE_TRIP_RS2_OFFGRID = 21,  // TripRS2, one trip per CTA, min/max reduce-scatter with 2-byte-offset shards
  SHAPE_TRIP_W_OFFGRID = 22     // TripW, one trip per CTA, 16-bit reduce-scatter with 2-byte-offset shards
};
// A launch that takes a CTA per trip instead of one resident wave.
__host__ __device__ constexpr bool is_trip_shape(int shape) {
  return shape == SHAPE_TRIP_S || shape == SHAPE_TRIP_RS2 || shape == SHAPE_TRIP_ACC || shape == SHAPE_TRIP_ACC_RS2 ||
         shape == SHAPE_TRIP_RS_OFFGRID || shape == SHAPE_TRIP_W || shape == SHAPE_TRIP_RS2_OFFGRID ||
         shape == SHAPE_TRIP_W_OFFGRID;
}

enum Kind {
  KIND_ALLREDUCE = 0,       // fused: one launch per call
  KIND_REDUCE_SCATTER = 1,  // fused
  KIND_ALLGATHER = 2,       // fused
  KIND_RING_RS_STEP = 3,    // one reduce-scatter step of the literal schedule, all ranks
  KIND_RING_AG_STEP = 4,    // one all-gather step of the literal schedule, all ranks
};

// Kernel parameters, passed by value (no device allocation, no state).
struct Args {
  const void* src[RA_MAX_RANKS];
  void* dst[RA_MAX_RANKS];
  uint64_t count;            // elements per rank (the full vector length L)
  uint64_t compact_aligned;  // bit c: the compact buffer of chunk c shares the vector phase
  int nranks;
  int head;        // first element index whose address is on the common line-aligned grid
  int align_elems; // elements per line-alignment step (a multiple of V)
  int vec_ok;  // the N-way side (AR/RS: sources and AR destinations; AG: destinations) shares one phase
  float inv_n; // 1.0f / nranks, rounded in fp32
  int step;    // ring step of a KIND_RING_* launch
  int acc32;   // fp16/bf16: partials stay in fp32 and are rounded once
  int shape;   // ShapeId of the fused AR/RS launch
};

// The walk of one CTA over a chunk's nv vectors: trip bases run over
// [begin, end) in steps of stride; in each trip this warp takes the 32
// vectors base + slot0 + u * uslot + lane (u < kUnroll); vectors at or past
// `end` are skipped. Trip bases are the same for every thread of the CTA.
// TRIP: the grid has a CTA per trip of the chunk, and CTA x takes the x-th
// CTA-sized block of it, whatever the schedule.
struct Walk {
  uint64_t begin, end, stride;
  uint32_t slot0, uslot;  // offsets inside one trip (less than stride)
};
template <class SH, bool TRIP>
__device__ __forceinline__ Walk cta_walk(uint64_t nv) {
  constexpr uint32_t kThreads = SH::kThreads, kUnroll = SH::kUnroll, kWarps = kThreads / 32;
  const uint32_t wid = threadIdx.x / 32;
  Walk w;
  w.begin = 0;
  w.end = nv;
  w.stride = (uint64_t)gridDim.x * kThreads * kUnroll;
  w.slot0 = blockIdx.x * kThreads * kUnroll + wid * 32;
  w.uslot = kThreads;
  if constexpr (!TRIP) {
#if RA_SCHEDULE == 1
    const uint64_t trip = (uint64_t)kThreads * kUnroll;
    const uint64_t per = ((nv + gridDim.x - 1) / gridDim.x + trip - 1) / trip * trip;
    w.begin = (uint64_t)blockIdx.x * per;
    w.end = w.begin + per < nv ? w.begin + per : nv;
    w.stride = trip;
    w.slot0 = wid * 32;
#elif RA_SCHEDULE == 2
    w.slot0 = (wid * gridDim.x + blockIdx.x) * 32;
    w.uslot = kWarps * gridDim.x * 32;
#endif
  }
  return w;
}

// ---------------------------------------------------------------------------
// the ring fold of kUnroll vectors at byte offsets off[] of every source
// ---------------------------------------------------------------------------
template <int DT, int OP, int kUnroll, int kBatch>
__device__ __forceinline__ void fold_vectors(const Args& a, int c, int n, const uint64_t (&off)[kUnroll],
                                             const bool (&ok)[kUnroll], Vec (&acc)[kUnroll]) {
  {
    const char* p = static_cast<const char*>(a.src[c]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (ok[u]) acc[u] = ld_vec(p + off[u]);
  }
  for (int k0 = 1; k0 < n; k0 += kBatch) {
    Vec x[kBatch][kUnroll];
#pragma unroll
    for (int kb = 0; kb < kBatch; ++kb) {
      const int k = k0 + kb;
      if (k < n) {
        int r = c + k;
        if (r >= n) r -= n;
        const char* p = static_cast<const char*>(a.src[r]);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (ok[u]) x[kb][u] = ld_vec(p + off[u]);
      }
    }
#pragma unroll
    for (int kb = 0; kb < kBatch; ++kb) {
      if (k0 + kb < n) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc[u] = vec_hop<DT, OP>(acc[u], x[kb][u]);
      }
    }
  }
  if constexpr (OP == OP_AVG) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc[u] = vec_avg<DT>(acc[u], a.inv_n, n);
  }
}

// The same fold with fp32 partials for fp16/bf16 buffers (one rounding at the end).
template <int DT, int OP, int kUnroll, int kBatch>
__device__ __forceinline__ void fold_vectors_acc32(const Args& a, int c, int n, const uint64_t (&off)[kUnroll],
                                                   const bool (&ok)[kUnroll], Vec (&out)[kUnroll]) {
  VecF acc[kUnroll];
  {
    const char* p = static_cast<const char*>(a.src[c]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (ok[u]) acc[u] = vec_widen<DT>(ld_vec(p + off[u]));
  }
  for (int k0 = 1; k0 < n; k0 += kBatch) {
    Vec x[kBatch][kUnroll];
#pragma unroll
    for (int kb = 0; kb < kBatch; ++kb) {
      const int k = k0 + kb;
      if (k < n) {
        int r = c + k;
        if (r >= n) r -= n;
        const char* p = static_cast<const char*>(a.src[r]);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (ok[u]) x[kb][u] = ld_vec(p + off[u]);
      }
    }
#pragma unroll
    for (int kb = 0; kb < kBatch; ++kb) {
      if (k0 + kb < n) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc[u] = vecf_hop<OP>(acc[u], vec_widen<DT>(x[kb][u]));
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    if constexpr (OP == OP_AVG) {
#pragma unroll
      for (int k = 0; k < kVecHalves; ++k) acc[u].f[k] = __fmul_rn(acc[u].f[k], a.inv_n);
    }
    out[u] = vec_narrow<DT>(acc[u]);
  }
}

template <int DT, int OP, bool ACC32, int kUnroll, int kBatch>
__device__ __forceinline__ void fold(const Args& a, int c, int n, const uint64_t (&off)[kUnroll],
                                     const bool (&ok)[kUnroll], Vec (&acc)[kUnroll]) {
  if constexpr (ACC32) fold_vectors_acc32<DT, OP, kUnroll, kBatch>(a, c, n, off, ok, acc);
  else fold_vectors<DT, OP, kUnroll, kBatch>(a, c, n, off, ok, acc);
}

// the ring fold of one element i of chunk c. The loads of up to kElemBatch
// ranks are issued before any of them is folded, so an element waits about one
// memory latency per kElemBatch ranks instead of one per rank.
constexpr int kElemBatch = 8;
template <int DT, int OP, bool ACC32>
__device__ __forceinline__ uint32_t fold_elem(const Args& a, int c, int n, uint64_t i) {
  uint32_t acc = 0;
  float accf = 0.0f;
  for (int k0 = 0; k0 < n; k0 += kElemBatch) {
    uint32_t x[kElemBatch];
#pragma unroll
    for (int kb = 0; kb < kElemBatch; ++kb) {
      const int k = k0 + kb;
      if (k < n) {
        int r = c + k;
        if (r >= n) r -= n;
        x[kb] = ld_elem<DT>(a.src[r], i);
      }
    }
#pragma unroll
    for (int kb = 0; kb < kElemBatch; ++kb) {
      const int k = k0 + kb;
      if (k < n) {
        if constexpr (ACC32) accf = k == 0 ? widen16<DT>(x[kb]) : f32_hop<OP>(accf, widen16<DT>(x[kb]));
        else acc = k == 0 ? x[kb] : elem_hop<DT, OP>(acc, x[kb]);
      }
    }
  }
  if constexpr (ACC32) {
    if constexpr (OP == OP_AVG) accf = __fmul_rn(accf, a.inv_n);
    return round16<DT>(accf);
  } else {
    if constexpr (OP == OP_AVG) acc = elem_avg<DT>(acc, a.inv_n, n);
    return acc;
  }
}

// Per-element path over [b0, vb) and [ve, b1), shared by the chunk's CTAs
// from the row's last CTA down: the vector loops leave those with the fewest
// trips, so the edge elements do not lengthen the longest CTA.
template <int kThreads, typename F>
__device__ __forceinline__ void for_each_edge_elem(uint64_t b0, uint64_t vb, uint64_t ve, uint64_t b1, F&& f) {
  const uint64_t n_lo = vb - b0, total = n_lo + (b1 - ve);
  for (uint64_t k = (uint64_t)(gridDim.x - 1 - blockIdx.x) * kThreads + threadIdx.x; k < total;
       k += (uint64_t)gridDim.x * kThreads) {
    f(k < n_lo ? b0 + k : ve + (k - n_lo));
  }
}

// ---------------------------------------------------------------------------
// all-reduce: every destination receives the fold
// ---------------------------------------------------------------------------
// The all-reduce of the element range [b0, b1), one chunk of one collective,
// folded in ring order from rank c: whole vectors, then the edge elements.
template <int DT, int OP, bool ACC32, class SH, bool TRIP>
__device__ __forceinline__ void ar_range(const Args& a, int c, int n, uint64_t b0, uint64_t b1) {
  constexpr int kThreads = SH::kThreads, kUnroll = SH::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const Walk w = cta_walk<SH, TRIP>((ve - vb) / V);
  // a thread's first vector of each trip; its later unroll slots lie further on
  for (uint64_t j0 = w.begin + w.slot0 + (threadIdx.x & 31u); j0 < w.end; j0 += w.stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * w.uslot;
      ok[u] = j < w.end;
      off[u] = (vb + j * V) * ES;
    }
    Vec acc[kUnroll];
    fold<DT, OP, ACC32, kUnroll, SH::kBatch>(a, c, n, off, ok, acc);
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.dst[r]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (ok[u]) st_vec(q + off[u], acc[u]);
    }
  }
  for_each_edge_elem<kThreads>(b0, vb, ve, b1, [&](uint64_t i) {
    const uint32_t v = fold_elem<DT, OP, ACC32>(a, c, n, i);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, v);
  });
}

// TRIP: launched with a CTA per trip of the chunk (each CTA does one trip and
// exits) instead of one resident wave.
template <int DT, int OP, bool ACC32, class SH, bool TRIP>
__global__ void __launch_bounds__(SH::kThreads, SH::kMinBlocks) ar_fused_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  const int n = a.nranks, c = blockIdx.y;
  ar_range<DT, OP, ACC32, SH, TRIP>(a, c, n, chunk_begin(c, n, a.count), chunk_begin(c + 1, n, a.count));
}

// ---------------------------------------------------------------------------
// grouped all-reduce: several independent all-reduces of element ranges of the
// same N buffers in one launch (gradient buckets that need no wait between
// them). Bucket b is the all-reduce of elements [begin[b], begin[b] + count[b])
// with its own chunk bounds, so each bucket's bits are those of a launch of its
// own. Row c of CTAs folds chunk c of every bucket in turn; a CTA goes on to
// the next bucket as soon as its share of one is done, so the buckets' partial
// last trips overlap instead of each paying a launch's ramp and tail.
// ---------------------------------------------------------------------------
constexpr int kMaxGroup = 64;
struct GroupArgs {
  Args a;             // the N whole buffers; a.count = the group's total elements
  uint32_t nbuckets;  // 1..kMaxGroup
  uint64_t begin[kMaxGroup];
  uint64_t count[kMaxGroup];
  // one-trip launches: bucket b owns the CTAs [trip_begin[b], trip_begin[b + 1]) of every row
  uint32_t trip_begin[kMaxGroup + 1];
};

template <int DT, int OP, bool ACC32, class SH>
__global__ void __launch_bounds__(SH::kThreads, SH::kMinBlocks) ar_group_kernel(const __grid_constant__ GroupArgs g) {
  pdl_enter();
  const Args& a = g.a;
  const int n = a.nranks, c = blockIdx.y;
  for (uint32_t b = 0; b < g.nbuckets; ++b) {
    const uint64_t at = g.begin[b], len = g.count[b];
    ar_range<DT, OP, ACC32, SH, false>(a, c, n, at + chunk_begin(c, n, len), at + chunk_begin(c + 1, n, len));
  }
}

// ---------------------------------------------------------------------------
// reduce-scatter: chunk c's fold goes to dst[c], compact (element i -> i - b0)
// ---------------------------------------------------------------------------
template <int DT, int OP, bool ACC32, class SH, bool OFFGRID = false, bool TRIP = false>
__global__ void __launch_bounds__(SH::kThreads, SH::kMinBlocks) rs_fused_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  constexpr int kThreads = SH::kThreads, kUnroll = SH::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const Walk w = cta_walk<SH, TRIP>((ve - vb) / V);
  void* out = a.dst[c];
  const bool out_vec = (a.compact_aligned >> c) & 1u;
  // Off the vector grid the plain kernel stores each lane's vector in 4-byte
  // units. OFFGRID (chosen when some chunk's output is only 2-byte aligned
  // against the grid) realigns such a chunk's results in registers instead:
  // the warp's 32 consecutive results are one run of bytes that starts 2 bytes
  // past a 4-byte boundary, so the 4-byte word that starts in lane l's 32
  // bytes takes its upper half from the lane's next word, and the word that
  // starts in its first 2 bytes takes its lower half from lane l-1's last word
  // (a shuffle). Each lane then writes 8 aligned 4-byte words; only the run's
  // first and last 2 bytes take 2-byte stores.
  const uint32_t lane = threadIdx.x & 31u;
  // trips are warp-uniform (the warp synchronises on the off-grid path)
  for (uint64_t base = w.begin; base < w.end; base += w.stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = base + w.slot0 + (uint64_t)u * w.uslot + lane;
      ok[u] = j < w.end;
      off[u] = (vb + j * V) * ES;
    }
    Vec acc[kUnroll];
    fold<DT, OP, ACC32, kUnroll, SH::kBatch>(a, c, n, off, ok, acc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (out_vec) {
        if (ok[u]) st_vec(static_cast<char*>(out) + off[u] - b0 * ES, acc[u]);
      } else if constexpr (OFFGRID) {
        const uint64_t jw = base + w.slot0 + (uint64_t)u * w.uslot;  // the warp's first vector this trip
        char* wdst = static_cast<char*>(out) + (vb + jw * V - b0) * ES;
        if ((reinterpret_cast<uintptr_t>(wdst) & 3u) == 0) {  // the chunk allows 4-byte units
          if (ok[u]) st_vec_units(static_cast<char*>(out) + off[u] - b0 * ES, acc[u]);
        } else {  // 2-byte offset: realign in registers (the branch is warp-uniform: jw is)
          const uint32_t nvalid = jw >= w.end ? 0u : (w.end - jw < 32 ? (uint32_t)(w.end - jw) : 32u);
          const Vec& v = acc[u];
          const uint32_t prev = __shfl_up_sync(0xffffffffu, v.w[kVecWords - 1], 1);
          if (lane < nvalid) {
            char* mine = wdst + lane * kVecBytes;  // this lane's 32 bytes start here, 2 bytes past a word
            unsigned int* q = reinterpret_cast<unsigned int*>(mine - 2);
            if (lane == 0) __stcs(reinterpret_cast<unsigned short*>(mine), (unsigned short)(v.w[0] & 0xffffu));
            else __stcs(q, (prev >> 16) | (v.w[0] << 16));
#pragma unroll
            for (int k = 1; k < kVecWords; ++k) __stcs(q + k, (v.w[k - 1] >> 16) | (v.w[k] << 16));
            if (lane == nvalid - 1)
              __stcs(reinterpret_cast<unsigned short*>(mine + kVecBytes - 2), (unsigned short)(v.w[kVecWords - 1] >> 16));
          }
        }
      } else if (ok[u]) {
        st_vec_units(static_cast<char*>(out) + off[u] - b0 * ES, acc[u]);
      }
    }
  }
  for_each_edge_elem<kThreads>(b0, vb, ve, b1, [&](uint64_t i) {
    st_elem<DT>(out, i - b0, fold_elem<DT, OP, ACC32>(a, c, n, i));
  });
}

// ---------------------------------------------------------------------------
// all-gather: src[c] (chunk c, compact) goes to every dst at [b0, b1)
// ---------------------------------------------------------------------------
template <int DT, class SH>
__global__ void __launch_bounds__(SH::kThreads, SH::kMinBlocks) ag_copy_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  constexpr int kThreads = SH::kThreads, kUnroll = SH::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const Walk w = cta_walk<SH, false>((ve - vb) / V);
  const void* in = a.src[c];
  const bool in_vec = (a.compact_aligned >> c) & 1u;
  for (uint64_t j0 = w.begin + w.slot0 + (threadIdx.x & 31u); j0 < w.end; j0 += w.stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
    Vec v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * w.uslot;
      ok[u] = j < w.end;
      off[u] = (vb + j * V) * ES;
      if (!ok[u]) continue;
      if (in_vec) {
        v[u] = ld_vec(static_cast<const char*>(in) + off[u] - b0 * ES);
      } else {
        const uint64_t i = off[u] / ES - b0;
#pragma unroll
        for (int k = 0; k < kVecWords; ++k) {
          if constexpr (ES == 4) {
            v[u].w[k] = ld_elem<DT>(in, i + k);
          } else {
            v[u].w[k] = ld_elem<DT>(in, i + 2 * k) | (ld_elem<DT>(in, i + 2 * k + 1) << 16);
          }
        }
      }
    }
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.dst[r]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (ok[u]) st_vec(q + off[u], v[u]);
    }
  }
  for_each_edge_elem<kThreads>(b0, vb, ve, b1, [&](uint64_t i) {
    const uint32_t x = ld_elem<DT>(in, i - b0);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, x);
  });
}

// ---------------------------------------------------------------------------
// host-side launch for one dtype (instantiated once per dtype translation unit)
// ---------------------------------------------------------------------------
template <int DT, int OP, bool ACC32, class SH, bool TRIP = false>
cudaError_t launch_ar(const Args& a, dim3 grid, cudaStream_t s) {
  return launch_programmatic(ar_fused_kernel<DT, OP, ACC32, SH, TRIP>, grid, SH::kThreads, 0, s, a);
}
template <int DT, int OP, bool ACC32, class SH, bool OFFGRID = false, bool TRIP = false>
cudaError_t launch_rs(const Args& a, dim3 grid, cudaStream_t s) {
  return launch_programmatic(rs_fused_kernel<DT, OP, ACC32, SH, OFFGRID, TRIP>, grid, SH::kThreads, 0, s, a);
}
template <int DT, int OP, bool ACC32, class SH>
cudaError_t launch_fused_shape(int kind, const Args& a, dim3 grid, cudaStream_t s) {
  return kind == KIND_ALLREDUCE ? launch_ar<DT, OP, ACC32, SH>(a, grid, s) : launch_rs<DT, OP, ACC32, SH>(a, grid, s);
}

// The grouped all-reduce with a CTA per trip: CTA x of row c finds its bucket
// b (the last with trip_begin[b] <= x), takes trip x - trip_begin[b] of chunk
// c of that bucket (a CTA-sized block of its vectors), and the bucket's last
// CTA also takes the chunk's edge elements. Each bucket keeps its own chunk
// bounds, so its bits are those of a launch of its own.
template <int DT, int OP, bool ACC32, class SH>
__global__ void __launch_bounds__(SH::kThreads, SH::kMinBlocks)
    ar_group_trip_kernel(const __grid_constant__ GroupArgs g) {
  pdl_enter();
  constexpr int kThreads = SH::kThreads, kUnroll = SH::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const Args& a = g.a;
  const int n = a.nranks, c = blockIdx.y;
  const uint32_t x = blockIdx.x;
  uint32_t lo = 0, hi = g.nbuckets;  // trip_begin[lo] <= x < trip_begin[hi]
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) / 2;
    if (g.trip_begin[mid] <= x) lo = mid;
    else hi = mid;
  }
  const uint32_t b = lo;
  const uint64_t t = x - g.trip_begin[b];
  const uint64_t at = g.begin[b], len = g.count[b];
  const uint64_t b0 = at + chunk_begin(c, n, len), b1 = at + chunk_begin(c + 1, n, len);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t j0 = t * kThreads * kUnroll + threadIdx.x;
  if (j0 < nv) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      ok[u] = j < nv;
      off[u] = (vb + j * V) * ES;
    }
    Vec acc[kUnroll];
    fold<DT, OP, ACC32, kUnroll, SH::kBatch>(a, c, n, off, ok, acc);
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.dst[r]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (ok[u]) st_vec(q + off[u], acc[u]);
    }
  }
  if (x + 1 == g.trip_begin[b + 1]) {  // the bucket's last CTA: the chunk's edge elements
    const uint64_t n_lo = vb - b0, total = n_lo + (b1 - ve);
    for (uint64_t k = threadIdx.x; k < total; k += kThreads) {
      const uint64_t i = k < n_lo ? b0 + k : ve + (k - n_lo);
      const uint32_t v = fold_elem<DT, OP, ACC32>(a, c, n, i);
      for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, v);
    }
  }
}

template <int DT, int OP, bool ACC32, class SH>
cudaError_t launch_group_shape(const GroupArgs& g, dim3 grid, cudaStream_t s) {
  return launch_programmatic(ar_group_kernel<DT, OP, ACC32, SH>, grid, SH::kThreads, 0, s, g);
}

// The grouped all-reduce on the all-reduce shapes shape_for() can choose, but
// for the two whose register budget the bucket loop would overflow (ShapeS,
// ShapeM3): the planner sends those groups to ShapeM.
template <int DT, int OP, bool ACC32>
cudaError_t launch_group_fused(const GroupArgs& g, dim3 grid, cudaStream_t s) {
  switch (g.a.shape) {
    case SHAPE_S4:
      if constexpr (!ACC32) return launch_group_shape<DT, OP, false, ShapeS4>(g, grid, s);
      break;
    case SHAPE_N3:
      if constexpr (!ACC32 && Elem<DT>::kSize == 4) return launch_group_shape<DT, OP, false, ShapeN3>(g, grid, s);
      break;
    case SHAPE_M: return launch_group_shape<DT, OP, ACC32, ShapeM>(g, grid, s);
    case SHAPE_W: return launch_group_shape<DT, OP, ACC32, ShapeW>(g, grid, s);
    case SHAPE_MB8:
      if constexpr (!ACC32 && (DT == DT_F16 || DT == DT_BF16) && OP != OP_MIN && OP != OP_MAX)
        return launch_group_shape<DT, OP, false, ShapeMB8>(g, grid, s);
      break;
    case SHAPE_W8: return launch_group_shape<DT, OP, ACC32, ShapeW8>(g, grid, s);
    case SHAPE_TRIP_S:
    case SHAPE_TRIP_ACC:
      return launch_programmatic(ar_group_trip_kernel<DT, OP, ACC32, TripS>, grid, TripS::kThreads, 0, s, g);
    case SHAPE_TRIP_W:
      if constexpr (!ACC32)
        return launch_programmatic(ar_group_trip_kernel<DT, OP, false, TripW>, grid, TripW::kThreads, 0, s, g);
      break;
  }
  return cudaErrorInvalidValue;
}

template <int DT, int OP>
cudaError_t launch_group_op(const GroupArgs& g, dim3 grid, cudaStream_t s) {
  constexpr bool kPartials = (DT == DT_F16 || DT == DT_BF16) && OP != OP_MIN && OP != OP_MAX;
  if constexpr (kPartials) {
    if (g.a.acc32) return launch_group_fused<DT, OP, true>(g, grid, s);
  }
  if (g.a.acc32) return cudaErrorInvalidValue;
  return launch_group_fused<DT, OP, false>(g, grid, s);
}

// Only the (kind, accumulation, shape) combinations shape_for() can choose are
// instantiated; any other is refused.
template <int DT, int OP, bool ACC32>
cudaError_t launch_fused(int kind, const Args& a, dim3 grid, cudaStream_t s) {
  const bool rs = kind == KIND_REDUCE_SCATTER;
  switch (a.shape) {
    case SHAPE_S:
      if constexpr (!ACC32) return launch_fused_shape<DT, OP, false, ShapeS>(kind, a, grid, s);
      if constexpr (ACC32 && OP != OP_MIN && OP != OP_MAX) {
        if (!rs) return launch_ar<DT, OP, true, ShapeS>(a, grid, s);
      }
      break;
    case SHAPE_S4:
      if constexpr (!ACC32) {
        if (!rs) return launch_ar<DT, OP, false, ShapeS4>(a, grid, s);
      }
      break;
    case SHAPE_RS2:  // fp16/bf16 sum/avg/prod, with or without fp32 partials
      if constexpr (Elem<DT>::kSize == 2 && OP != OP_MIN && OP != OP_MAX) {
        if (rs) return launch_rs<DT, OP, ACC32, ShapeRS2>(a, grid, s);
      }
      break;
    case SHAPE_RS6:
      if constexpr (!ACC32 && (Elem<DT>::kSize == 4 || OP == OP_MIN || OP == OP_MAX)) {
        if (rs) return launch_rs<DT, OP, false, ShapeRS6>(a, grid, s);
      }
      break;
    case SHAPE_RS:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, ShapeRS>(a, grid, s);
      }
      break;
    case SHAPE_N3:  // 4-byte types only: fp16/bf16 take ShapeM3 at N = 3
      if constexpr (!ACC32 && Elem<DT>::kSize == 4) {
        if (!rs) return launch_ar<DT, OP, false, ShapeN3>(a, grid, s);
      }
      break;
    case SHAPE_M: return launch_fused_shape<DT, OP, ACC32, ShapeM>(kind, a, grid, s);
    case SHAPE_W:
      if (!rs) return launch_ar<DT, OP, ACC32, ShapeW>(a, grid, s);
      break;
    case SHAPE_RS_OFFGRID:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, ShapeS, true>(a, grid, s);
      }
      break;
    case SHAPE_RS_OFFGRID_B2:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, ShapeRS2, true>(a, grid, s);
      }
      break;
    case SHAPE_RS_OFFGRID_M:  // fp32 partials, shards off the vector grid
      if (rs) return launch_rs<DT, OP, ACC32, ShapeRS2, true>(a, grid, s);
      break;
    case SHAPE_M3:
      if (!rs) return launch_ar<DT, OP, ACC32, ShapeM3>(a, grid, s);
      break;
    case SHAPE_MB8:
      if constexpr (!ACC32 && (DT == DT_F16 || DT == DT_BF16) && OP != OP_MIN && OP != OP_MAX) {
        if (!rs) return launch_ar<DT, OP, false, ShapeMB8>(a, grid, s);
      }
      break;
    case SHAPE_W8:
      if (!rs) return launch_ar<DT, OP, ACC32, ShapeW8>(a, grid, s);
      break;
    case SHAPE_TRIP_S:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, TripS, false, true>(a, grid, s);
        return launch_ar<DT, OP, false, TripS, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_RS2:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, TripRS2, false, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_ACC:
      if constexpr (ACC32) {
        if (!rs) return launch_ar<DT, OP, true, TripS, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_ACC_RS2:
      if constexpr (ACC32) {
        if (rs) return launch_rs<DT, OP, true, TripAccRS, false, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_RS_OFFGRID:
      if constexpr (!ACC32 && Elem<DT>::kSize == 2) {
        if (rs) return launch_rs<DT, OP, false, TripS, true, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_RS2_OFFGRID:
      if constexpr (!ACC32 && Elem<DT>::kSize == 2 && (OP == OP_MIN || OP == OP_MAX)) {
        if (rs) return launch_rs<DT, OP, false, TripRS2, true, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_W_OFFGRID:
      if constexpr (!ACC32 && Elem<DT>::kSize == 2 && OP != OP_MIN && OP != OP_MAX) {
        if (rs) return launch_rs<DT, OP, false, TripW, true, true>(a, grid, s);
      }
      break;
    case SHAPE_TRIP_W:
      if constexpr (!ACC32) {
        if (rs) return launch_rs<DT, OP, false, TripW, false, true>(a, grid, s);
        return launch_ar<DT, OP, false, TripW, true>(a, grid, s);
      }
      break;
  }
  return cudaErrorInvalidValue;
}

// The fused all-reduce / reduce-scatter of one (dtype, op) pair.
template <int DT, int OP>
cudaError_t launch_op(int kind, const Args& a, dim3 grid, cudaStream_t s) {
  // fp32 partials exist for fp16/bf16 sum, avg and prod; min and max are exact
  // in the buffer dtype, and the planner never asks for partials there
  constexpr bool kPartials = (DT == DT_F16 || DT == DT_BF16) && OP != OP_MIN && OP != OP_MAX;
  if constexpr (kPartials) {
    if (a.acc32) return launch_fused<DT, OP, true>(kind, a, grid, s);
  }
  if (a.acc32) return cudaErrorInvalidValue;
  return launch_fused<DT, OP, false>(kind, a, grid, s);
}

template <class SH>
inline void shape_params_of(int* threads, int* unroll, int* min_blocks) {
  *threads = SH::kThreads, *unroll = SH::kUnroll, *min_blocks = SH::kMinBlocks;
}
inline void shape_params(int shape, int* threads, int* unroll, int* min_blocks) {
  switch (shape) {
    case SHAPE_S: return shape_params_of<ShapeS>(threads, unroll, min_blocks);
    case SHAPE_N3: return shape_params_of<ShapeN3>(threads, unroll, min_blocks);
    case SHAPE_M: return shape_params_of<ShapeM>(threads, unroll, min_blocks);
    case SHAPE_W: return shape_params_of<ShapeW>(threads, unroll, min_blocks);
    case SHAPE_RS_OFFGRID: return shape_params_of<ShapeS>(threads, unroll, min_blocks);
    case SHAPE_RS_OFFGRID_B2: return shape_params_of<ShapeRS2>(threads, unroll, min_blocks);
    case SHAPE_RS_OFFGRID_M: return shape_params_of<ShapeRS2>(threads, unroll, min_blocks);
    case SHAPE_M3: return shape_params_of<ShapeM3>(threads, unroll, min_blocks);
    case SHAPE_S4: return shape_params_of<ShapeS4>(threads, unroll, min_blocks);
    case SHAPE_RS2: return shape_params_of<ShapeRS2>(threads, unroll, min_blocks);
    case SHAPE_RS6: return shape_params_of<ShapeRS6>(threads, unroll, min_blocks);
    case SHAPE_RS: return shape_params_of<ShapeRS>(threads, unroll, min_blocks);
    case SHAPE_MB8: return shape_params_of<ShapeMB8>(threads, unroll, min_blocks);
    case SHAPE_W8: return shape_params_of<ShapeW8>(threads, unroll, min_blocks);
    case SHAPE_TRIP_S: return shape_params_of<TripS>(threads, unroll, min_blocks);
    case SHAPE_TRIP_RS2: return shape_params_of<TripRS2>(threads, unroll, min_blocks);
    case SHAPE_TRIP_ACC: return shape_params_of<TripS>(threads, unroll, min_blocks);
    case SHAPE_TRIP_ACC_RS2: return shape_params_of<TripAccRS>(threads, unroll, min_blocks);
    case SHAPE_TRIP_RS_OFFGRID: return shape_params_of<TripS>(threads, unroll, min_blocks);
    case SHAPE_TRIP_W: return shape_params_of<TripW>(threads, unroll, min_blocks);
    case SHAPE_TRIP_RS2_OFFGRID: return shape_params_of<TripRS2>(threads, unroll, min_blocks);
    case SHAPE_TRIP_W_OFFGRID: return shape_params_of<TripW>(threads, unroll, min_blocks);
    default: return shape_params_of<ShapeS>(threads, unroll, min_blocks);
  }
}

}  // namespace ra
