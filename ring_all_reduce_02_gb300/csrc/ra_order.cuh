// All-reduce / reduce-scatter in the association of another algorithm the
// pages describe (tirogla.com "Ring all-reduce", "How it works", cost model):
// Rabenseifner's recursive halving (power-of-two N) or the double binary tree.
// On one GPU these move the same bytes as the ring; only the order in which
// each element's N values are combined differs, and that order fixes the
// rounding.
//
// The host planner turns the algorithm into a reduction program of N-1 steps
// "slot[a] = op(slot[a], slot[b])" over the N rank slots (at most two
// programs, chosen per chunk: the double binary tree reduces the first N/2
// chunks with one tree and the rest with the other). Each thread stages the N
// vectors of its element range into its own shared-memory slots with cp.async
// (16-byte global-to-shared copies, no registers held while they fly), waits
// for its own copies only, runs the program on its slots and stores the
// result. No thread reads another thread's slots, so no CTA barrier is needed.
#pragma once

#include "ra_kernels.cuh"

namespace ra {

// The ordered kernel stages 16-byte vectors (the grid of the plan is laid on
// lines of at least 32 bytes, so 16-byte vectors tile it too): with 32-byte
// slots it measured 85-87% of the copy bandwidth against 91% with 16-byte ones.
constexpr int kOrdVecBytes = 16;
using OVec = VecT<kOrdVecBytes / 4>;
#ifndef RA_ORD_THREADS
#define RA_ORD_THREADS (2048 / 16)  // 2 KB of vectors per CTA and rank slot
#endif
constexpr int kOrdThreads = RA_ORD_THREADS;
constexpr int kMaxProgSteps = RA_MAX_RANKS - 1;

struct OrderArgs {
  Args base;
  uint8_t prog[2][kMaxProgSteps][2];  // (a, b) per step
  uint8_t prog_len[2];
  uint8_t root[2];          // slot holding the result after the program
  uint64_t chunk_prog;      // bit c: chunk c runs program 1, else program 0
};

__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int DT, int OP>
__device__ __forceinline__ uint32_t run_prog_elem(const OrderArgs& o, int pr, int n, uint64_t i) {
  // One load per rank in turn. Issuing them in batches before the stores to
  // the slot array (as the ring's per-element fold does) changed the code
  // generated for the vector path and cost it 8 points of the copy bandwidth.
  uint32_t v[RA_MAX_RANKS];
  for (int r = 0; r < n; ++r) v[r] = ld_elem<DT>(o.base.src[r], i);
  for (int t = 0; t < o.prog_len[pr]; ++t) {
    const int a = o.prog[pr][t][0], b = o.prog[pr][t][1];
    v[a] = elem_hop<DT, OP>(v[a], v[b]);
  }
  uint32_t acc = v[o.root[pr]];
  if constexpr (OP == OP_AVG) acc = elem_avg<DT>(acc, o.base.inv_n, n);
  return acc;
}

// IS_RS: reduce-scatter (chunk c to dst[c], compact) instead of all-reduce.
template <int DT, int OP, bool IS_RS>
__global__ void __launch_bounds__(kOrdThreads, 6) ordered_kernel(const __grid_constant__ OrderArgs o) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t slots[];  // [rank][thread] vectors
  constexpr int ES = Elem<DT>::kSize;
  constexpr int V = kOrdVecBytes / ES;  // elements per staged vector
  const Args& a = o.base;
  const int n = a.nranks, c = blockIdx.y;
  const int pr = (int)((o.chunk_prog >> c) & 1u);
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  OVec* my = reinterpret_cast<OVec*>(slots) + threadIdx.x;  // slot r at my[r * kOrdThreads]
  void* out = a.dst[c];
  const bool out_vec = !IS_RS || ((a.compact_aligned >> c) & 1u);
  // A warp stages its 32 consecutive vectors of each rank as one contiguous run of
  // 16-byte pieces, lane l copying pieces l, l + 32, ...: every cp.async instruction
  // covers 512 contiguous bytes. A lane's slots are thus filled by other lanes, so
  // the warp synchronises after the copies land and before the slots are refilled.
  constexpr uint32_t kPieces = kOrdVecBytes / 16;
  const uint32_t lane = threadIdx.x & 31u, wbase = threadIdx.x & ~31u;
  for (uint64_t jw = (uint64_t)blockIdx.x * kOrdThreads + wbase; jw < nv;
       jw += (uint64_t)gridDim.x * kOrdThreads) {
    const uint64_t j = jw + lane;
    const uint64_t off0 = (vb + jw * V) * ES;  // the warp's first vector
    for (int r = 0; r < n; ++r) {
      const char* g = static_cast<const char*>(a.src[r]) + off0;
      char* sw = reinterpret_cast<char*>(reinterpret_cast<OVec*>(slots) + r * kOrdThreads + wbase);
#pragma unroll
      for (uint32_t h = 0; h < kPieces; ++h) {
        const uint32_t p = h * 32u + lane;
        if (jw + p / kPieces < nv) cp_async_16(sw + 16u * p, g + 16u * p);
      }
    }
    cp_async_wait_all();
    __syncwarp();
    if (j < nv) {
      const uint64_t off = (vb + j * V) * ES;
      for (int t = 0; t < o.prog_len[pr]; ++t) {
        OVec* sa = my + o.prog[pr][t][0] * kOrdThreads;
        const OVec* sb = my + o.prog[pr][t][1] * kOrdThreads;
        *sa = vec_hop<DT, OP>(*sa, *sb);
      }
      OVec v = my[o.root[pr] * kOrdThreads];
      if constexpr (OP == OP_AVG) v = vec_avg<DT>(v, a.inv_n, n);
      if constexpr (IS_RS) {
        if (out_vec) st_vec(static_cast<char*>(out) + off - b0 * ES, v);
        else my[0] = v;  // slot 0 of this lane is no longer read: it stages the result
      } else {
        for (int r = 0; r < n; ++r) st_vec(static_cast<char*>(a.dst[r]) + off, v);
      }
    }
    if constexpr (IS_RS) {
      if (!out_vec) {  // off the vector grid: the warp writes its results in address-suited units
        __syncwarp();
        const uint32_t nw = nv - jw < 32 ? (uint32_t)(nv - jw) : 32u;
        copy_out_units(static_cast<char*>(out) + (vb + jw * V - b0) * ES,
                       reinterpret_cast<const char*>(reinterpret_cast<OVec*>(slots) + wbase), nw * kOrdVecBytes,
                       lane, 32);
      }
    }
    __syncwarp();
  }
  const uint64_t n_lo = vb - b0, total = n_lo + (b1 - ve);
  for (uint64_t k = (uint64_t)blockIdx.x * kOrdThreads + threadIdx.x; k < total;
       k += (uint64_t)gridDim.x * kOrdThreads) {
    const uint64_t i = k < n_lo ? b0 + k : ve + (k - n_lo);
    const uint32_t v = run_prog_elem<DT, OP>(o, pr, n, i);
    if constexpr (IS_RS) {
      st_elem<DT>(out, i - b0, v);
    } else {
      for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, v);
    }
  }
}

template <int DT, int OP, bool IS_RS>
cudaError_t launch_ordered_kind(const OrderArgs& o, dim3 grid, cudaStream_t s) {
  const size_t smem = (size_t)o.base.nranks * kOrdThreads * kOrdVecBytes;
  const cudaError_t err =
      cudaFuncSetAttribute(ordered_kernel<DT, OP, IS_RS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_programmatic(ordered_kernel<DT, OP, IS_RS>, grid, kOrdThreads, smem, s, o);
}

template <int DT, int OP>
cudaError_t launch_ordered_op(bool is_rs, const OrderArgs& o, dim3 grid, cudaStream_t s) {
  return is_rs ? launch_ordered_kind<DT, OP, true>(o, grid, s) : launch_ordered_kind<DT, OP, false>(o, grid, s);
}

}  // namespace ra
