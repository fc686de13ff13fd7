// The all-gather kernel and its plan: compact chunk c (src[c]) goes to every
// destination at [b0, b1) — one read and N writes per element (infra-guide
// "All-Gather"; tirogla "How it works", the all-gather phase).
//
// HBM writes bound this kernel: N of its N+1 bytes are writes. On GB300 the
// write stream depends on how long the writing CTAs live. Persistent CTAs that
// grid-stride over a buffer write 6.66-6.81 TB/s whatever the store width,
// cache hint or order (cyclic, contiguous slabs, scrambled), and so do TMA bulk
// stores from persistent CTAs; CTAs that each write 4-64 KB and exit write
// 7.38-7.48 TB/s (CUDA events, 4 GiB, clean or back to back). So the library's
// all-gather gives every CTA one tile: its 256 threads read the tile (8 KB) of
// the compact chunk into shared memory, one thread hands it to the Tensor
// Memory Accelerator as N bulk stores (cp.async.bulk shared -> global, one per
// destination), waits until they have read the tile and the CTA exits.
// Measured, fraction of the copy bandwidth, fp32, 1 GiB over all ranks, back
// to back: 100.4-104.1% for N = 2..16, against 89.4-98.7% for the persistent
// TMA kernels this replaced. ag_copy_kernel (ra_kernels.cuh: persistent
// threads load vectors into registers and store each to the N destinations) is
// kept for comparison sweeps (RA_AG_TUNE_KERNEL=0).
#pragma once

#include "ra_bulk.cuh"
#include "ra_kernels.cuh"

namespace ra {

constexpr int kAgThreads = 256;
using AgShape = Shape<kAgThreads, 2, 1, 1>;  // the register kernel

enum AgKernel { AG_REGISTERS = 0, AG_TILE = 1 };
constexpr int kShapeAgBase = 100;  // Args::shape of an all-gather launch: kShapeAgBase + AgKernel

struct AgPlan {
  int kernel;         // AgKernel
  int unroll;         // vectors per thread per tile (1: 8 KB tiles at 32-byte vectors; 2: 16 KB; 4: 32 KB)
  int blocks_per_sm;  // AG_REGISTERS: resident CTAs per SM the grid is sized for
};

// One 8 KB tile per CTA for every N: 8 KB measured best or within half a point
// of 16 KB everywhere but N = 6 at 256 MiB over all ranks (95.0 against 96.5%),
// and 32 KB tiles lost 1-8 points at 256 MiB.
inline AgPlan ag_plan_for(int nranks) {
#ifdef RA_AG_TUNE_KERNEL  // tuning sweeps: one plan for every rank count
  (void)nranks;
  return {RA_AG_TUNE_KERNEL, RA_AG_TUNE_UNROLL, RA_AG_TUNE_BPS};
#else
  (void)nranks;
  return {AG_TILE, 1, 1};
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

// Whole tiles per chunk can differ by one between chunks; this bound holds
// for every chunk (a chunk has at most count / n + 1 elements).
template <int kUnroll>
__host__ __device__ inline uint64_t ag_tiles_per_chunk_bound(uint64_t count, int n, int v) {
  return (count / (uint64_t)n + 1) / (uint64_t)v / ((uint64_t)kAgThreads * kUnroll) + 1;
}

// ---------------------------------------------------------------------------
// One tile per CTA. grid (tiles per chunk bound + 1, N): CTA (x, c) copies
// whole tile x of chunk c to the N destinations and exits; CTA x == ntiles of
// the chunk takes its leftover vectors and edge elements; CTAs past that exit
// at once. A stream of stores from short-lived CTAs writes HBM faster than the
// same stores from persistent, grid-striding CTAs.
// ---------------------------------------------------------------------------
template <int kUnroll>
__host__ __device__ inline uint64_t ag_tile_grid_x(uint64_t count, int n, int v) {
  return ag_tiles_per_chunk_bound<kUnroll>(count, n, v) + 1;
}

// the leftover vectors and the edge elements of chunk c, by one CTA
template <int DT>
__device__ __forceinline__ void ag_chunk_rest(const Args& a, const char* in, bool in_vec, uint64_t b0, uint64_t b1,
                                              uint64_t vb, uint64_t ve, uint64_t from_vec) {
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  const int n = a.nranks;
  const uint64_t nv = (ve - vb) / V;
  for (uint64_t j = from_vec + threadIdx.x; j < nv; j += kAgThreads) {
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

// Tile t of a compact chunk (src = its first byte) into shared memory in
// destination order. G = 0: the chunk is on the destinations' vector grid and a
// thread loads kUnroll vectors; G = 2..16: it is off the grid and the CTA reads
// it in G-byte units, consecutive threads on consecutive units. All of a
// thread's loads are issued before the first shared-memory store.
template <int kUnroll, uint32_t G>
__device__ __forceinline__ void ag_stage_tile(const char* src, uint8_t* smem) {
  constexpr uint32_t TB = ag_tile_bytes<kUnroll>();
  if constexpr (G == 0) {
    Vec v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_vec(src + ((uint32_t)u * kAgThreads + threadIdx.x) * kVecBytes);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      *reinterpret_cast<Vec*>(smem + ((uint32_t)u * kAgThreads + threadIdx.x) * kVecBytes) = v[u];
  } else {
    using T = typename UnitT<G>::T;
    constexpr uint32_t K = TB / (G * kAgThreads);  // loads per thread
    T w[K];
#pragma unroll
    for (uint32_t k = 0; k < K; ++k) w[k] = __ldcs(reinterpret_cast<const T*>(src) + threadIdx.x + k * kAgThreads);
#pragma unroll
    for (uint32_t k = 0; k < K; ++k) reinterpret_cast<T*>(smem)[threadIdx.x + k * kAgThreads] = w[k];
  }
}

// grid (ag_tile_grid_x, N), kAgThreads threads, ag_tile_bytes<kUnroll>() of
// dynamic shared memory.
template <int DT, int kUnroll>
__global__ void __launch_bounds__(kAgThreads) ag_tile_kernel(const __grid_constant__ Args a) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int V = Elem<DT>::kPerVec;
  constexpr int ES = Elem<DT>::kSize;
  constexpr uint32_t TV = (uint32_t)kAgThreads * kUnroll;
  constexpr uint32_t TB = ag_tile_bytes<kUnroll>();
  const int n = a.nranks, c = blockIdx.y;
  const uint64_t b0 = chunk_begin(c, n, a.count), b1 = chunk_begin(c + 1, n, a.count);
  uint64_t vb = b0, ve = b0;
  if (a.vec_ok) vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, V, &vb, &ve);
  const uint64_t ntiles = (ve - vb) / V / TV, t = blockIdx.x;
  const char* in = static_cast<const char*>(a.src[c]);
  const bool in_vec = (a.compact_aligned >> c) & 1u;
  if (t < ntiles) {
    const char* first = in + (vb - b0) * ES;  // the chunk's first whole vector, compact side
    const char* src = first + t * TB;
    if (in_vec) {
      ag_stage_tile<kUnroll, 0>(src, smem);
    } else {
      switch (unit_bytes(first)) {  // every tile of the chunk shares this alignment (TB % 16 == 0)
        case 16: ag_stage_tile<kUnroll, 16>(src, smem); break;
        case 8: ag_stage_tile<kUnroll, 8>(src, smem); break;
        case 4: ag_stage_tile<kUnroll, 4>(src, smem); break;
        default: ag_stage_tile<kUnroll, 2>(src, smem); break;
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic-proxy writes -> bulk copies
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint64_t off = (vb + t * TV * V) * ES;
      for (int r = 0; r < n; ++r) bulk_store(static_cast<char*>(a.dst[r]) + off, smem, TB);
      bulk_commit();
      // shared memory must outlive the bulk stores that read it (a hardware wait, no spin)
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
  } else if (t == ntiles) {
    ag_chunk_rest<DT>(a, in, in_vec, b0, b1, vb, ve, ntiles * TV);
  }
}

}  // namespace ra
