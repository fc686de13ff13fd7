// The fused all-reduce with its loads staged through shared memory by the
// Tensor Memory Accelerator (cp.async.bulk), for running on a subset of the
// SMs beside other work (arjunsriva.com "AllReduce, All the Way Down":
// communication kernels compete with compute for SMs).
//
// The register kernel keeps every load in flight in registers and in the
// SM's outstanding-miss slots, which caps one SM at roughly 50 GB/s. Here one
// producer thread per CTA streams tiles of all N ranks into a ring of
// shared-memory stages with bulk copies (up to ~200 KB in flight per SM,
// tracked by mbarrier transaction counts instead of per-thread misses); the
// consumer warps fold each tile in the ring's order from shared memory and
// store the result to the N destinations. Same fold, same rounding, same
// result bits as ar_fused_kernel.
//
// Every wait is bounded: a wait that has not completed after kWaitNs of the
// global timer records an error code in the caller's status word and the
// kernel winds down (waiting, again bounded, for its own bulk copies still in
// flight) instead of hanging.
#pragma once

#include "ra_kernels.cuh"

namespace ra {

// Folding threads per CTA, chosen per launch (BulkArgs::consumers). More
// consumers keep more stores in flight, which is what bounds an SM budget: N = 8
// fp32 avg, 256 MiB per rank, on 16 / 32 / 64 SMs, GB/s per SM with 128 / 256 /
// 384 / 512 consumers: 87 / 89 / 92 / 91, 88 / 89 / 89 / 90, 87 / 89 / 87 / 87;
// at N = 2: 54 / 83 / 89 / 104; at N = 3: 59 / 84 / 98 / 99; at N = 4: 78 / 104
// / 105 / 100; at N = 16: 88 / 95 / 95 / 94 on 16 SMs and 86-88 on 64. On all
// SMs 384 gained at N <= 4 (37-42 against 42-43 GB/s per SM) and lost 1.5% at
// N = 8 and 16. So: 384 on an SM budget or below N = 8, else 128.
// The two counts are separate instantiations: 384 as a launch-time value
// measured 9 points below the instantiated 384 at N = 16 on SM budgets.
constexpr int kBulkConsumersWide = 384, kBulkConsumersNarrow = 128;
inline int bulk_consumers_for(int nranks, bool sm_budget) {
  return (sm_budget || nranks < 8) ? kBulkConsumersWide : kBulkConsumersNarrow;
}
constexpr uint64_t kWaitNs = 1000000000ull;       // 1 s per wait
constexpr int kBulkErrFull = 1;                    // a stage's bulk copies did not land in time
constexpr int kBulkErrEmpty = 2;                   // the consumers did not release a stage in time

struct BulkArgs {
  Args base;
  int* status;        // device words; 0 = fine, else the first error code seen
  uint32_t status_stride;  // 0: every chunk reports into status[0]; 1: chunk c into status[c]
  uint32_t tile_vecs;  // vectors per rank per stage (a multiple of 32)
  uint32_t consumers;  // folding threads: kBulkConsumersWide or kBulkConsumersNarrow; the CTA has
                       // consumers + 32 threads (the last warp is the producer's)
  uint32_t stages;     // stages in the shared-memory ring
  int withhold_chunk;  // self-test of the bounded waits: -1 none, else CTA (0, c) never issues its
                       // first tile's copies for c = withhold_chunk
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// true once the barrier's phase with this parity has completed, false on timeout
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t start = global_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (global_ns() - start > kWaitNs) return false;
  }
}
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void record_error(int* status, int code) { atomicCAS(status, 0, code); }

template <int DT, int OP, int NC>
__global__ void __launch_bounds__(NC + 32, 1) ar_bulk_kernel(const __grid_constant__ BulkArgs ba) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const Args& a = ba.base;
  const int n = a.nranks, c = blockIdx.y;
  constexpr uint32_t NT = NC + 32;
  const uint32_t S = ba.stages, TV = ba.tile_vecs;
  const uint32_t tile_bytes = TV * kVecBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);  // [S]: bulk copies of a stage landed
  uint64_t* empty = full + S;                          // [S]: consumers done with a stage
  uint8_t* data = smem + 128 * ((2 * S * 8 + 127) / 128);  // [S][n][tile_bytes]

  int* const status = ba.status + (size_t)c * ba.status_stride;

  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t ntiles = nv / TV;  // whole tiles; the rest of the chunk takes the direct path

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC / 32);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  const uint64_t first = blockIdx.x, step = gridDim.x;
  if (threadIdx.x >= NC) {
    // ---- producer warp: one elected thread issues the bulk copies --------------
    if (threadIdx.x == NC) {
      uint32_t issued = 0;
      for (uint64_t t = first; t < ntiles; t += step, ++issued) {
        const uint32_t s = issued % S;
        if (issued >= S && !mbar_wait(&empty[s], ((issued / S) - 1) & 1)) {
          record_error(status, kBulkErrEmpty);
          break;
        }
        mbar_arrive_expect_tx(&full[s], tile_bytes * (uint32_t)n);
        if (issued == 0 && blockIdx.x == 0 && (int)blockIdx.y == ba.withhold_chunk) continue;
        const uint64_t off = (vb + t * TV * V) * ES;
        for (int k = 0; k < n; ++k) {
          int r = c + k;
          if (r >= n) r -= n;
          bulk_load(data + ((size_t)s * n + k) * tile_bytes, static_cast<const char*>(a.src[r]) + off,
                    tile_bytes, &full[s]);
        }
      }
      // Never leave with bulk copies into this CTA's shared memory still in
      // flight: wait (bounded) on every stage that may still be filling, also
      // after one of these waits has run out, and keep the first error code.
      const uint32_t lo = issued > S ? issued - S : 0;
      for (uint32_t i = lo; i < issued; ++i) {
        if (!mbar_wait(&full[i % S], (i / S) & 1)) record_error(status, kBulkErrFull);
      }
    }
  } else {
    // ---- consumers: fold each landed tile in ring order, store to every rank ----
    uint32_t used = 0;
    for (uint64_t t = first; t < ntiles; t += step, ++used) {
      const uint32_t s = used % S;
      if (!mbar_wait(&full[s], (used / S) & 1)) {
        record_error(status, kBulkErrFull);
        break;
      }
      const uint8_t* tile = data + (size_t)s * n * tile_bytes;
      for (uint32_t j = threadIdx.x; j < TV; j += NC) {
        Vec acc = *reinterpret_cast<const Vec*>(tile + (size_t)j * kVecBytes);  // slot 0 = rank c
        for (int k = 1; k < n; ++k)
          acc = vec_hop<DT, OP>(acc, *reinterpret_cast<const Vec*>(tile + (size_t)k * tile_bytes + j * kVecBytes));
        if constexpr (OP == OP_AVG) acc = vec_avg<DT>(acc, a.inv_n, n);
        const uint64_t off = (vb + (t * TV + j) * V) * ES;
        for (int r = 0; r < n; ++r) st_vec(static_cast<char*>(a.dst[r]) + off, acc);
      }
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s]);
    }
  }

  // the part of the chunk outside whole tiles, read directly: leftover vectors, then edge elements
  const uint64_t tail_beg = ntiles * TV;
  for (uint64_t j = tail_beg + (uint64_t)blockIdx.x * NT + threadIdx.x; j < nv; j += (uint64_t)gridDim.x * NT) {
    const uint64_t off = (vb + j * V) * ES;
    Vec acc = ld_vec(static_cast<const char*>(a.src[c]) + off);
    for (int k = 1; k < n; ++k) {
      int r = c + k;
      if (r >= n) r -= n;
      acc = vec_hop<DT, OP>(acc, ld_vec(static_cast<const char*>(a.src[r]) + off));
    }
    if constexpr (OP == OP_AVG) acc = vec_avg<DT>(acc, a.inv_n, n);
    for (int r = 0; r < n; ++r) st_vec(static_cast<char*>(a.dst[r]) + off, acc);
  }
  const uint64_t n_lo = vb - b0, n_edge = n_lo + (b1 - ve);  // edge elements (the CTA width is per launch)
  for (uint64_t k = (uint64_t)(gridDim.x - 1 - blockIdx.x) * NT + threadIdx.x; k < n_edge;
       k += (uint64_t)gridDim.x * NT) {
    const uint64_t i = k < n_lo ? b0 + k : ve + (k - n_lo);
    const uint32_t v = fold_elem<DT, OP, false>(a, c, n, i);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, v);
  }
}

// Raises both instances' dynamic shared-memory limit to `smem`; enqueues nothing.
template <int DT, int OP>
cudaError_t configure_bulk_op(size_t smem) {
  const cudaError_t err = cudaFuncSetAttribute(ar_bulk_kernel<DT, OP, kBulkConsumersWide>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute(ar_bulk_kernel<DT, OP, kBulkConsumersNarrow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

// Launches the kernel; configure_bulk_op(smem) must have succeeded on this device.
template <int DT, int OP>
cudaError_t launch_bulk_op(const BulkArgs& b, dim3 grid, size_t smem, cudaStream_t s) {
  if (b.consumers == (uint32_t)kBulkConsumersWide)
    return launch_programmatic(ar_bulk_kernel<DT, OP, kBulkConsumersWide>, grid, kBulkConsumersWide + 32, smem, s, b);
  if (b.consumers == (uint32_t)kBulkConsumersNarrow)
    return launch_programmatic(ar_bulk_kernel<DT, OP, kBulkConsumersNarrow>, grid, kBulkConsumersNarrow + 32, smem, s,
                               b);
  return cudaErrorInvalidValue;
}

}  // namespace ra
