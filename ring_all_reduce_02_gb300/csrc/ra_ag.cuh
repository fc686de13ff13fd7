// The all-gather kernels and their plan: compact chunk c (src[c]) goes to
// every destination at [b0, b1) — one read and N writes per element
// (infra-guide "All-Gather"; tirogla "How it works", the all-gather phase).
//
// HBM writes bound this kernel. On GB300 a pure stream of stores from the SMs
// peaks near 6.4 TB/s (94% of the copy bandwidth) whatever the store width or
// cache hint, against about 7.2 TB/s for reads. The library's all-gather is
// ag_tma_store_kernel (below): the threads load a tile into shared memory and
// one thread hands it to the Tensor Memory Accelerator as N bulk stores
// (cp.async.bulk shared -> global, 8 or 16 KB contiguous per destination),
// double-buffered so the next tile loads while the last one is written. The
// planner picks the tile, the CTAs per SM and the grid from N: a row of CTAs
// per chunk, or ag_tma_flat_kernel's single tile sequence over all SMs. ag_copy_kernel
// (ra_kernels.cuh: every thread loads vectors into registers and stores each
// to the N destinations) measured 84-91% at its best shape; it is kept for
// comparison sweeps (RA_AG_TUNE_KERNEL=0).
#pragma once

#include "ra_bulk.cuh"
#include "ra_kernels.cuh"

namespace ra {

constexpr int kAgThreads = 256;
using AgShape = Shape<kAgThreads, 2, 1, 1>;  // the register kernel

#ifndef RA_AG_STAGES
#define RA_AG_STAGES 2
#endif
constexpr uint32_t kAgStages = RA_AG_STAGES;  // tiles in shared memory per CTA

enum AgKernel { AG_REGISTERS = 0, AG_TMA_STORE = 1, AG_TMA_FLAT = 2 };
constexpr int kShapeAgBase = 100;  // Args::shape of an all-gather launch: kShapeAgBase + AgKernel

struct AgPlan {
  int kernel;         // AgKernel
  int unroll;         // AG_TMA_STORE: vectors per thread per tile (1 or 2: 8 or 16 KB tiles at 32-byte vectors)
  int blocks_per_sm;  // resident CTAs per SM the grid is sized for
};

// Chosen from sweeps on GB300 (fp32, 1 GiB over all ranks, fraction of the
// copy bandwidth): the tiles in flight per SM that keep HBM busiest shrink as
// N grows, because the reads are 1/(N+1) of the traffic. 32 KB per SM at
// N <= 3 (98.6% at N = 2, 92% at N = 3), 16 KB at N = 4..7, 8 KB from N = 8.
// Up to N = 4 and at N = 8 a row of CTAs per chunk fills the SMs (95.7% at
// N = 4, 93.5% at N = 8). Elsewhere the rows leave SMs idle, and one tile
// sequence over all SMs does better: 95.2 / 92.0 / 88.8% at N = 5 / 6 / 7
// against 92.6 / 90.8 / 86.5%, 92.0 / 89.4% at N = 12 / 16 against
// 90.2 / 88.4%. The register kernel measured 84-91% at its best shape.
inline AgPlan ag_plan_for(int nranks) {
#ifdef RA_AG_TUNE_KERNEL  // tuning sweeps: one plan for every rank count
  (void)nranks;
  return {RA_AG_TUNE_KERNEL, RA_AG_TUNE_UNROLL, RA_AG_TUNE_BPS};
#else
  if (nranks <= 2) return {AG_TMA_STORE, 1, 4};
  if (nranks == 3) return {AG_TMA_STORE, 2, 2};
  if (nranks == 4) return {AG_TMA_STORE, 1, 2};
  if (nranks <= 7) return {AG_TMA_FLAT, 2, 1};
  if (nranks == 8) return {AG_TMA_STORE, 1, 1};
  return {AG_TMA_FLAT, 1, 1};
#endif
}

template <int kUnroll>
__host__ __device__ constexpr uint32_t ag_tile_bytes() {
  return (uint32_t)kAgThreads * kUnroll * kVecBytes;  // per destination
}

__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Vector at byte offset off (of the destination layout) from the compact
// chunk that starts at element b0: one vector load when the chunk shares the
// destinations' phase, element loads otherwise.
template <int DT>
__device__ __forceinline__ Vec ag_load(const void* in, bool in_vec, uint64_t off, uint64_t b0) {
  constexpr int ES = Elem<DT>::kSize;
  if (in_vec) return ld_vec(static_cast<const char*>(in) + off - b0 * ES);
  Vec v;
  const uint64_t i = off / ES - b0;
#pragma unroll
  for (int k = 0; k < kVecWords; ++k) {
    if constexpr (ES == 4) {
      v.w[k] = ld_elem<DT>(in, i + k);
    } else {
      v.w[k] = ld_elem<DT>(in, i + 2 * k) | (ld_elem<DT>(in, i + 2 * k + 1) << 16);
    }
  }
  return v;
}

// The CTA's whole tiles of one chunk: t0, t0 + tstride, ... below ntiles; `it`
// counts the CTA's tiles so far and picks the stage. G = 0: the compact chunk
// is on the destinations' vector grid and a thread loads kUnroll vectors;
// G = 2..16: it is off the grid and the CTA reads the tile in G-byte units,
// consecutive threads on consecutive units. Either way the loads are issued
// before the wait for the stage, and the stage holds the tile in destination
// order.
template <int DT, int kUnroll, uint32_t G>
__device__ __forceinline__ void ag_tiles(const Args& a, uint8_t* smem, const char* in, uint64_t vb, uint64_t b0,
                                         uint64_t ntiles, uint64_t t0, uint64_t tstride, uint32_t& it) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  constexpr uint32_t TV = (uint32_t)kAgThreads * kUnroll;  // vectors per tile
  constexpr uint32_t TB = ag_tile_bytes<kUnroll>();
  using T = typename UnitT<G == 0 ? 16 : G>::T;
  constexpr uint32_t K = G == 0 ? kUnroll : TB / (G * kAgThreads);  // loads per thread per tile
  const int n = a.nranks;
  for (uint64_t t = t0; t < ntiles; t += tstride, ++it) {
    const char* src = in + (vb + t * TV * V - b0) * ES;  // the tile in the compact chunk
    Vec v[G == 0 ? kUnroll : 1];
    T w[G == 0 ? 1 : K];
    if constexpr (G == 0) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = ld_vec(src + ((uint32_t)u * kAgThreads + threadIdx.x) * kVecBytes);
    } else {
#pragma unroll
      for (uint32_t k = 0; k < K; ++k) w[k] = __ldcs(reinterpret_cast<const T*>(src) + threadIdx.x + k * kAgThreads);
    }
    uint8_t* stage = smem + (it % kAgStages) * TB;
    // the stage was last handed to bulk stores kAgStages tiles ago: wait until they have read it
    if (it >= kAgStages && threadIdx.x == 0)
      asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kAgStages - 1) : "memory");
    __syncthreads();
    if constexpr (G == 0) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        *reinterpret_cast<Vec*>(stage + ((uint32_t)u * kAgThreads + threadIdx.x) * kVecBytes) = v[u];
    } else {
#pragma unroll
      for (uint32_t k = 0; k < K; ++k) reinterpret_cast<T*>(stage)[threadIdx.x + k * kAgThreads] = w[k];
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic-proxy writes -> bulk copies
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint64_t off = (vb + t * TV * V) * ES;
      for (int r = 0; r < n; ++r) bulk_store(static_cast<char*>(a.dst[r]) + off, stage, TB);
      bulk_commit();
    }
  }
}

// The CTA's whole tiles of one chunk (t0, t0 + tstride, ...), loaded by vectors
// when the compact chunk is on the destinations' grid, else in the widest unit
// its address allows.
template <int DT, int kUnroll>
__device__ __forceinline__ void ag_chunk_tiles(const Args& a, uint8_t* smem, const char* in, bool in_vec, uint64_t vb,
                                               uint64_t b0, uint64_t ntiles, uint64_t t0, uint64_t tstride,
                                               uint32_t& it) {
  constexpr int ES = Elem<DT>::kSize;
  if (t0 >= ntiles) return;
  if (in_vec) {
    ag_tiles<DT, kUnroll, 0>(a, smem, in, vb, b0, ntiles, t0, tstride, it);
  } else {
    switch (unit_bytes(in + (vb - b0) * ES)) {
      case 16: ag_tiles<DT, kUnroll, 16>(a, smem, in, vb, b0, ntiles, t0, tstride, it); break;
      case 8: ag_tiles<DT, kUnroll, 8>(a, smem, in, vb, b0, ntiles, t0, tstride, it); break;
      case 4: ag_tiles<DT, kUnroll, 4>(a, smem, in, vb, b0, ntiles, t0, tstride, it); break;
      default: ag_tiles<DT, kUnroll, 2>(a, smem, in, vb, b0, ntiles, t0, tstride, it); break;
    }
  }
}

// Whole tiles per chunk can differ by one between chunks; this bound holds
// for every chunk (a chunk has at most count / n + 1 elements).
template <int kUnroll>
__host__ __device__ inline uint64_t ag_tiles_per_chunk_bound(uint64_t count, int n, int v) {
  return (count / (uint64_t)n + 1) / (uint64_t)v / ((uint64_t)kAgThreads * kUnroll) + 1;
}

// grid (CTAs, 1), the same threads and shared memory as below. The tiles of
// all chunks form one sequence (tile k of chunk c at c * tpc + k) dealt to the
// CTAs in turn, so each CTA (one per SM on the budget) gets an equal share
// whatever N is; with a row of CTAs per chunk, N that do not divide the SM
// count leave SMs idle (8 of 152 at N = 12 and 16). Chunk c's leftover vectors
// and edge elements go to CTA c mod gridDim.x.
template <int DT, int kUnroll>
__global__ void __launch_bounds__(kAgThreads) ag_tma_flat_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  constexpr uint32_t TV = (uint32_t)kAgThreads * kUnroll;  // vectors per tile
  const int n = a.nranks;
  const uint64_t tpc = ag_tiles_per_chunk_bound<kUnroll>(a.count, n, V);
  const uint64_t g = gridDim.x;
  uint32_t it = 0;
  for (int c = 0; c < n; ++c) {
    const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
    uint64_t vb = b0, ve = b0;
    if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
    const uint64_t nv = (ve - vb) / V;
    const uint64_t ntiles = nv / TV;
    const char* in = static_cast<const char*>(a.src[c]);
    const bool in_vec = (a.compact_aligned >> c) & 1u;
    // this CTA's first tile of the chunk: the sequence index c * tpc + t0 is blockIdx.x mod g
    const uint64_t t0 = ((uint64_t)blockIdx.x + g - ((uint64_t)c * tpc) % g) % g;
    ag_chunk_tiles<DT, kUnroll>(a, smem, in, in_vec, vb, b0, ntiles, t0, g, it);
    if ((uint64_t)c % g == blockIdx.x) {
      for (uint64_t j = ntiles * TV + threadIdx.x; j < nv; j += kAgThreads) {
        const uint64_t off = (vb + j * V) * ES;
        const Vec x = ag_load<DT>(in, in_vec, off, b0);
        for (int r = 0; r < n; ++r) st_vec(static_cast<char*>(a.dst[r]) + off, x);
      }
      const uint64_t n_lo = vb - b0, total = n_lo + (b1 - ve);
      for (uint64_t k = threadIdx.x; k < total; k += kAgThreads) {
        const uint64_t i = k < n_lo ? b0 + k : ve + (k - n_lo);
        const uint32_t x = ld_elem<DT>(in, i - b0);
        for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, x);
      }
    }
  }
  // shared memory must outlive the bulk stores that read it
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// grid (CTAs per chunk, N), kAgThreads threads, kAgStages * ag_tile_bytes<kUnroll>()
// of dynamic shared memory. The chunk's whole tiles go through shared memory and
// bulk stores; the leftover vectors and the edge elements take plain stores.
template <int DT, int kUnroll>
__global__ void __launch_bounds__(kAgThreads) ag_tma_store_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  constexpr uint32_t TV = (uint32_t)kAgThreads * kUnroll;  // vectors per tile
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t nv = (ve - vb) / V;
  const uint64_t ntiles = nv / TV;
  const char* in = static_cast<const char*>(a.src[c]);
  const bool in_vec = (a.compact_aligned >> c) & 1u;

  uint32_t it = 0;
  ag_chunk_tiles<DT, kUnroll>(a, smem, in, in_vec, vb, b0, ntiles, blockIdx.x, gridDim.x, it);

  for (uint64_t j = ntiles * TV + (uint64_t)blockIdx.x * kAgThreads + threadIdx.x; j < nv;
       j += (uint64_t)gridDim.x * kAgThreads) {
    const uint64_t off = (vb + j * V) * ES;
    const Vec x = ag_load<DT>(in, in_vec, off, b0);
    for (int r = 0; r < n; ++r) st_vec(static_cast<char*>(a.dst[r]) + off, x);
  }
  for_each_edge_elem<kAgThreads>(b0, vb, ve, b1, [&](uint64_t i) {
    const uint32_t x = ld_elem<DT>(in, i - b0);
    for (int r = 0; r < n; ++r) st_elem<DT>(a.dst[r], i, x);
  });
  // shared memory must outlive the bulk stores that read it
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace ra
