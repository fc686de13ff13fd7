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
// rank order and derives the chunk's bounds once; blockIdx.x strides over the
// chunk's 16-byte vectors (kUnroll vectors per thread per trip, loads of up to
// kBatch ranks issued back to back before they are folded). The at most 2(V-1)
// elements at the ends of each chunk, and every element when the buffers do
// not share a 16-byte phase, go through the per-element path.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ra_ops.cuh"
#include "ra_plan.h"

#ifndef RA_MAX_RANKS
#define RA_MAX_RANKS 64
#endif

namespace ra {

// Launch shape (build-time overridable for tuning sweeps; these defaults are the
// measured choice on GB300).
#ifndef RA_THREADS
#define RA_THREADS 256
#endif
#ifndef RA_MIN_BLOCKS
#define RA_MIN_BLOCKS 2
#endif
#ifndef RA_UNROLL
#define RA_UNROLL 2
#endif
#ifndef RA_BATCH
#define RA_BATCH 8
#endif
constexpr int kThreads = RA_THREADS;       // threads per CTA
constexpr int kMinBlocks = RA_MIN_BLOCKS;  // resident CTAs per SM the register budget is set for
constexpr int kUnroll = RA_UNROLL;         // 16-byte vectors per thread per trip
constexpr int kBatch = RA_BATCH;           // ranks whose loads are in flight together

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
  uint64_t compact_aligned;  // bit c: the compact buffer of chunk c shares the 16-byte phase
  int nranks;
  int head;    // first element index on the common 16-byte grid, in [0, V)
  int vec_ok;  // the N-way side (AR/RS: sources and AR destinations; AG: destinations) shares one phase
  float inv_n; // 1.0f / nranks, rounded in fp32
  int step;    // ring step of a KIND_RING_* launch
};

// ---------------------------------------------------------------------------
// the ring fold of kUnroll vectors at byte offsets off[] of every source
// ---------------------------------------------------------------------------
template <int DT, int OP>
__device__ __forceinline__ void fold_vectors(const Args& a, int c, int n, const uint64_t (&off)[kUnroll],
                                             const bool (&ok)[kUnroll], uint4 (&acc)[kUnroll]) {
  {
    const char* p = static_cast<const char*>(a.src[c]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (ok[u]) acc[u] = ld_vec(p + off[u]);
  }
  for (int k0 = 1; k0 < n; k0 += kBatch) {
    uint4 x[kBatch][kUnroll];
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

// the ring fold of one element i of chunk c
template <int DT, int OP>
__device__ __forceinline__ uint32_t fold_elem(const Args& a, int c, int n, uint64_t i) {
  uint32_t acc = ld_elem<DT>(a.src[c], i);
  for (int k = 1; k < n; ++k) {
    int r = c + k;
    if (r >= n) r -= n;
    acc = elem_hop<DT, OP>(acc, ld_elem<DT>(a.src[r], i));
  }
  if constexpr (OP == OP_AVG) acc = elem_avg<DT>(acc, a.inv_n, n);
  return acc;
}

// Per-element path over [b0, vb) and [ve, b1), shared by the chunk's CTAs.
template <typename F>
__device__ __forceinline__ void for_each_edge_elem(uint64_t b0, uint64_t vb, uint64_t ve, uint64_t b1, F&& f) {
  const uint64_t n_lo = vb - b0, total = n_lo + (b1 - ve);
  for (uint64_t k = (uint64_t)blockIdx.x * kThreads + threadIdx.x; k < total;
       k += (uint64_t)gridDim.x * kThreads) {
    f(k < n_lo ? b0 + k : ve + (k - n_lo));
  }
}

// ---------------------------------------------------------------------------
// all-reduce: every destination receives the fold
// ---------------------------------------------------------------------------
template <int DT, int OP>
__global__ void __launch_bounds__(kThreads, kMinBlocks) ar_fused_kernel(const __grid_constant__ Args a) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads * kUnroll;
  for (uint64_t j0 = (uint64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; j0 < nv; j0 += stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      ok[u] = j < nv;
      off[u] = (vb + j * V) * ES;
    }
    uint4 acc[kUnroll];
    fold_vectors<DT, OP>(a, c, n, off, ok, acc);
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.dst[r]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (ok[u]) st_vec(q + off[u], acc[u]);
    }
  }
  for_each_edge_elem(b0, vb, ve, b1, [&](uint64_t i) {
    const uint32_t v = fold_elem<DT, OP>(a, c, n, i);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, v);
  });
}

// ---------------------------------------------------------------------------
// reduce-scatter: chunk c's fold goes to dst[c], compact (element i -> i - b0)
// ---------------------------------------------------------------------------
template <int DT, int OP>
__global__ void __launch_bounds__(kThreads, kMinBlocks) rs_fused_kernel(const __grid_constant__ Args a) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads * kUnroll;
  void* out = a.dst[c];
  const bool out_vec = (a.compact_aligned >> c) & 1u;
  for (uint64_t j0 = (uint64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; j0 < nv; j0 += stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      ok[u] = j < nv;
      off[u] = (vb + j * V) * ES;
    }
    uint4 acc[kUnroll];
    fold_vectors<DT, OP>(a, c, n, off, ok, acc);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (!ok[u]) continue;
      if (out_vec) {
        st_vec(static_cast<char*>(out) + off[u] - b0 * ES, acc[u]);
      } else {
        const uint64_t i = off[u] / ES - b0;
#pragma unroll
        for (int l = 0; l < V; ++l) st_elem<DT>(out, i + l, vec_lane<DT>(acc[u], l));
      }
    }
  }
  for_each_edge_elem(b0, vb, ve, b1, [&](uint64_t i) {
    st_elem<DT>(out, i - b0, fold_elem<DT, OP>(a, c, n, i));
  });
}

// ---------------------------------------------------------------------------
// all-gather: src[c] (chunk c, compact) goes to every dst at [b0, b1)
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) ag_copy_kernel(const __grid_constant__ Args a) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads * kUnroll;
  const void* in = a.src[c];
  const bool in_vec = (a.compact_aligned >> c) & 1u;
  for (uint64_t j0 = (uint64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; j0 < nv; j0 += stride) {
    uint64_t off[kUnroll];
    bool ok[kUnroll];
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      ok[u] = j < nv;
      off[u] = (vb + j * V) * ES;
      if (!ok[u]) continue;
      if (in_vec) {
        v[u] = ld_vec(static_cast<const char*>(in) + off[u] - b0 * ES);
      } else {
        const uint64_t i = off[u] / ES - b0;
        uint32_t w[4];
        if constexpr (ES == 4) {
#pragma unroll
          for (int l = 0; l < 4; ++l) w[l] = ld_elem<DT>(in, i + l);
        } else {
#pragma unroll
          for (int l = 0; l < 4; ++l) w[l] = ld_elem<DT>(in, i + 2 * l) | (ld_elem<DT>(in, i + 2 * l + 1) << 16);
        }
        v[u] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    for (int r = 0; r < n; ++r) {
      char* q = static_cast<char*>(a.dst[r]);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (ok[u]) st_vec(q + off[u], v[u]);
    }
  }
  for_each_edge_elem(b0, vb, ve, b1, [&](uint64_t i) {
    const uint32_t x = ld_elem<DT>(in, i - b0);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, x);
  });
}

// ---------------------------------------------------------------------------
// The literal schedule, one launch per ring step (for checking and measuring
// the fused kernels against it). blockIdx.y = rank r.
//
// reduce-scatter step s: rank r receives chunk C = (r - s - 1) mod N from rank
// r-1 and combines it with its own copy: dst[r][C] = hop(in, src[r][C]), where
// `in` is rank r-1's partial of C from step s-1 (dst[r-1][C]) or, at s = 0,
// its input (src[r-1][C]). Each chunk of rank r is touched once in this phase,
// so its own operand is still its input, read from src[r]; in place
// (dst == src) this is the same memory. At s = N-2 rank r finishes chunk
// (r+1) mod N and applies the avg epilogue to it.
// all-gather step s: dst[r][C] = dst[r-1][C] with C = (r - s) mod N.
// ---------------------------------------------------------------------------
template <int DT, int OP>
__global__ void __launch_bounds__(kThreads, kMinBlocks) ring_rs_step_kernel(const __grid_constant__ Args a) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, r = blockIdx.y, s = a.step;
  const int prev = r == 0 ? n - 1 : r - 1;
  const int cc = ((r - s - 1) % n + n) % n;
  const void* in = s == 0 ? a.src[prev] : a.dst[prev];
  const void* own = a.src[r];
  void* out = a.dst[r];
  const bool finish = (OP == OP_AVG) && (s == n - 2);
  const uint64_t b0 = chunk_begin(cc, n, a.count), b1 = chunk_begin(cc + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < nv; j += (uint64_t)gridDim.x * kThreads) {
    const uint64_t off = (vb + j * V) * ES;
    uint4 v = vec_hop<DT, OP>(ld_vec(static_cast<const char*>(in) + off), ld_vec(static_cast<const char*>(own) + off));
    if (finish) v = vec_avg<DT>(v, a.inv_n, n);
    st_vec(static_cast<char*>(out) + off, v);
  }
  for_each_edge_elem(b0, vb, ve, b1, [&](uint64_t i) {
    uint32_t v = elem_hop<DT, OP>(ld_elem<DT>(in, i), ld_elem<DT>(own, i));
    if (finish) v = elem_avg<DT>(v, a.inv_n, n);
    st_elem<DT>(out, i, v);
  });
}

template <int DT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) ring_ag_step_kernel(const __grid_constant__ Args a) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, r = blockIdx.y, s = a.step;
  const int prev = r == 0 ? n - 1 : r - 1;
  const int cc = ((r - s) % n + n) % n;
  const void* in = a.dst[prev];
  void* out = a.dst[r];
  const uint64_t b0 = chunk_begin(cc, n, a.count), b1 = chunk_begin(cc + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  for (uint64_t j = (uint64_t)blockIdx.x * kThreads + threadIdx.x; j < nv; j += (uint64_t)gridDim.x * kThreads) {
    const uint64_t off = (vb + j * V) * ES;
    st_vec(static_cast<char*>(out) + off, ld_vec(static_cast<const char*>(in) + off));
  }
  for_each_edge_elem(b0, vb, ve, b1, [&](uint64_t i) { st_elem<DT>(out, i, ld_elem<DT>(in, i)); });
}

// ---------------------------------------------------------------------------
// host-side launch for one dtype (instantiated once per dtype translation unit)
// ---------------------------------------------------------------------------
template <int DT>
cudaError_t launch_dtype(int kind, int op, const Args& a, dim3 grid, cudaStream_t s) {
  const dim3 block(kThreads);
  if (kind == KIND_ALLGATHER) {
    ag_copy_kernel<DT><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
  }
  if (kind == KIND_RING_AG_STEP) {
    ring_ag_step_kernel<DT><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
  }
#define RA_LAUNCH_OP(OPV)                                                            \
  case OPV:                                                                          \
    if (kind == KIND_ALLREDUCE) ar_fused_kernel<DT, OPV><<<grid, block, 0, s>>>(a);  \
    else if (kind == KIND_REDUCE_SCATTER) rs_fused_kernel<DT, OPV><<<grid, block, 0, s>>>(a); \
    else ring_rs_step_kernel<DT, OPV><<<grid, block, 0, s>>>(a);                     \
    break;
  switch (op) {
    RA_LAUNCH_OP(OP_SUM)
    RA_LAUNCH_OP(OP_AVG)
    RA_LAUNCH_OP(OP_MIN)
    RA_LAUNCH_OP(OP_MAX)
    RA_LAUNCH_OP(OP_PROD)
    default: return cudaErrorInvalidValue;
  }
#undef RA_LAUNCH_OP
  return cudaGetLastError();
}

}  // namespace ra
