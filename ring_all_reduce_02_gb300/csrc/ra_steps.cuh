// The literal ring schedule, one launch per ring step, for checking and
// measuring the fused kernels against it (tirogla.com "Ring all-reduce", "How
// it works": N-1 reduce-scatter steps, then N-1 all-gather steps).
// blockIdx.y = rank r.
//
// reduce-scatter step s: rank r receives chunk C = (r - s - 1) mod N from rank
// r-1 and combines it with its own copy: dst[r][C] = hop(in, src[r][C]), where
// `in` is rank r-1's partial of C from step s-1 (dst[r-1][C]) or, at s = 0,
// its input (src[r-1][C]). Each chunk of rank r is touched once in this phase,
// so its own operand is still its input, read from src[r]; in place
// (dst == src) this is the same memory. At s = N-2 rank r finishes chunk
// (r+1) mod N and applies the avg epilogue to it.
// all-gather step s: dst[r][C] = dst[r-1][C] with C = (r - s) mod N.
//
// Per step the reduce-scatter reads 2 and writes 1 chunk per rank (3 S over
// all ranks), the all-gather reads and writes 1 (2 S): 5 (N-1) S for the whole
// schedule, against 2 N S for the fused kernel.
//
// The steps are plain launches, each after the previous one has completed:
// as programmatic dependent launches whose CTAs also signalled the next step
// early, the schedule measured 1.5% slower on GB300.
#pragma once

#include "ra_kernels.cuh"

#ifndef RA_STEP_THREADS
#define RA_STEP_THREADS 256
#endif
#ifndef RA_STEP_MIN_BLOCKS
#define RA_STEP_MIN_BLOCKS 2
#endif
#ifndef RA_STEP_UNROLL
#define RA_STEP_UNROLL 2
#endif

namespace ra {

// 2 vectors per thread per trip, all of a trip's loads issued before its stores
// (on GB300 the schedule then runs at 95% of the copy bandwidth for its own
// traffic at N = 8, against 86% with 1 vector and 93% with 4)
using StepShape = Shape<RA_STEP_THREADS, RA_STEP_MIN_BLOCKS, RA_STEP_UNROLL, 1>;

template <int DT, int OP>
__global__ void __launch_bounds__(StepShape::kThreads, StepShape::kMinBlocks)
    ring_rs_step_kernel(const __grid_constant__ Args a) {
  constexpr int kThreads = StepShape::kThreads, kUnroll = StepShape::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, r = blockIdx.y, s = a.step;
  const int prev = r == 0 ? n - 1 : r - 1;
  const int cc = ((r - s - 1) % n + n) % n;
  const char* in = static_cast<const char*>(s == 0 ? a.src[prev] : a.dst[prev]);
  const char* own = static_cast<const char*>(a.src[r]);
  char* out = static_cast<char*>(a.dst[r]);
  const bool finish = (OP == OP_AVG) && (s == n - 2);
  const uint64_t b0 = chunk_begin(cc, n, a.count), b1 = chunk_begin(cc + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  for (uint64_t j0 = (uint64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; j0 < nv;
       j0 += (uint64_t)gridDim.x * kThreads * kUnroll) {
    Vec x[kUnroll], y[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      if (j < nv) {
        const uint64_t off = (vb + j * V) * ES;
        x[u] = ld_vec(in + off);
        y[u] = ld_vec(own + off);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      if (j < nv) {
        Vec v = vec_hop<DT, OP>(x[u], y[u]);
        if (finish) v = vec_avg<DT>(v, a.inv_n, n);
        st_vec(out + (vb + j * V) * ES, v);
      }
    }
  }
  for_each_edge_elem<kThreads>(b0, vb, ve, b1, [&](uint64_t i) {
    uint32_t v = elem_hop<DT, OP>(ld_elem<DT>(in, i), ld_elem<DT>(own, i));
    if (finish) v = elem_avg<DT>(v, a.inv_n, n);
    st_elem<DT>(out, i, v);
  });
}

template <int DT>
__global__ void __launch_bounds__(StepShape::kThreads, StepShape::kMinBlocks)
    ring_ag_step_kernel(const __grid_constant__ Args a) {
  constexpr int kThreads = StepShape::kThreads, kUnroll = StepShape::kUnroll;
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks, r = blockIdx.y, s = a.step;
  const int prev = r == 0 ? n - 1 : r - 1;
  const int cc = ((r - s) % n + n) % n;
  const char* in = static_cast<const char*>(a.dst[prev]);
  char* out = static_cast<char*>(a.dst[r]);
  const uint64_t b0 = chunk_begin(cc, n, a.count), b1 = chunk_begin(cc + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  for (uint64_t j0 = (uint64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; j0 < nv;
       j0 += (uint64_t)gridDim.x * kThreads * kUnroll) {
    Vec x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      if (j < nv) x[u] = ld_vec(in + (vb + j * V) * ES);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint64_t j = j0 + (uint64_t)u * kThreads;
      if (j < nv) st_vec(out + (vb + j * V) * ES, x[u]);
    }
  }
  for_each_edge_elem<kThreads>(b0, vb, ve, b1, [&](uint64_t i) { st_elem<DT>(out, i, ld_elem<DT>(in, i)); });
}

template <int DT, int OP>
cudaError_t launch_ring_rs_step(const Args& a, dim3 grid, cudaStream_t s) {
  ring_rs_step_kernel<DT, OP><<<grid, StepShape::kThreads, 0, s>>>(a);
  return cudaGetLastError();
}
template <int DT>
cudaError_t launch_ring_ag_step(const Args& a, dim3 grid, cudaStream_t s) {
  ring_ag_step_kernel<DT><<<grid, StepShape::kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace ra
