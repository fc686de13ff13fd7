// The C ABI of libra.so: argument checks, the alias rules, the chunk-schedule
// planner (grid sizing, launch shape and vector-path selection, the reduction
// programs of the other orders, gradient buckets) and dispatch to the kernels.
// Declarations and the contract of every entry point: include/ra.h.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "../../include/ra.h"
#include "ra_ag.cuh"
#include "ra_bulk.cuh"
#include "ra_kernels.cuh"
#include "ra_order.cuh"
#include "ra_steps.cuh"

namespace ra {
cudaError_t launch_kernel(int kind, int dtype, int op, const Args& a, dim3 grid, cudaStream_t s);
cudaError_t launch_ordered_kernel(bool is_rs, int dtype, int op, const OrderArgs& o, dim3 grid, cudaStream_t s);
cudaError_t launch_bulk_kernel(int dtype, int op, const BulkArgs& b, dim3 grid, size_t smem, cudaStream_t s);
cudaError_t configure_bulk_kernel(int dtype, int op, size_t smem);
cudaError_t launch_group_kernel(int dtype, int op, const GroupArgs& g, dim3 grid, cudaStream_t s);
}  // namespace ra

namespace {

thread_local int g_last_cuda_error = 0;

int elem_size(int dtype) {
  switch (dtype) {
    case RA_FLOAT32: return 4;
    case RA_FLOAT16: return 2;
    case RA_BFLOAT16: return 2;
    case RA_INT32: return 4;
    default: return 0;
  }
}

ra_status_t cuda_failed(cudaError_t err) {
  g_last_cuda_error = (int)err;
  return RA_ERR_CUDA;
}

struct Range {
  uintptr_t lo = 0, hi = 0;  // [lo, hi) in bytes; empty if lo == hi
};
bool overlaps(const Range& a, const Range& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// ---- launch shapes of the fused kernels ------------------------------------
// The fused shape for a call, from sweeps on GB300 (fraction of the copy
// bandwidth, 1 GiB over all ranks; the shapes themselves are in ra_kernels.cuh):
//  - reduce-scatter: loads of 2 ranks at a time up to N = 3, with registers for
//    8 CTAs/SM for fp16/bf16 sum/avg/prod (ShapeRS2) and for 6 otherwise
//    (ShapeRS6: fp32 N = 3 avg 101% against 90%, bf16 max 100-101% against
//    98-99%; bf16 avg 88% against 97-98%), and for min/max from N = 4
//    (ShapeRS); of 4 for sum/avg/prod from N = 4 (ShapeS); fp32 partials on
//    ShapeM;
//  - all-reduce N <= 2: ShapeS4 (99%), except fp16/bf16 sum/avg/prod and fp32
//    partials (sum/avg/prod only), which keep ShapeS (98.5-99%);
//  - N = 3: ShapeN3 for fp32/int32, ShapeM3 for fp16/bf16 and for fp32
//    partials, which ShapeN3 cannot hold (97% against 85%);
//  - fp16/bf16 min/max (one paired min/max per word, less ALU work than fp32):
//    ShapeW8 at N = 6, 7 (98.7 / 96.9% against 95.0 / 96.2% on ShapeM3), ShapeW at
//    N = 8, 9 (100.0 / 96.5% against 95.3 / 91.9% on ShapeM), ShapeM3 at
//    N = 10..15 (96.4-96.8% at 10, 11, 12, 14, 15 against 93.3-93.8% on ShapeW at
//    10, 11; 94.3% at 13, where ShapeW gave 95.7%), ShapeW from N = 16 (98.9%);
//  - every other call at N = 6, 7 loads all ranks at once on the wide shape
//    (ShapeW8: fp32 99% / 97% against 95% / 96.5% on ShapeM and ShapeM3; bf16
//    sum/avg at N = 7 96% against 95%), except fp16/bf16 sum/avg/prod at N = 6,
//    which do better at 2 CTAs/SM (ShapeMB8, 97-98% against 95% on ShapeW8);
//    fp32 partials there 97-98% against 94-96% on ShapeM;
//  - fp32 partials at N = 8: ShapeW (99% against 96.5% on ShapeM);
//  - otherwise ShapeM up to N = 7 and, for fp16/bf16 (more ALU work per byte),
//    up to N = 15 (98.9% at N = 8 against 93.4%); ShapeW from N = 8, but
//    ShapeM at N = 10, 11, 14 (fp32: 96.1-97.1% against 92.5-93.8%; ShapeW is
//    ahead at 9, 12, 13, 15 by 0.4-3 points).
int shape_for(int nranks, bool reduce_scatter = false, bool acc32 = false, bool narrow = false,
              bool minmax = false) {
  if (reduce_scatter) {
    // fp32 partials: 128 x 1 at 8 CTAs/SM with loads of 2 ranks (bf16 avg, 1 GiB over all
    // ranks, N = 3..7: 96.5-99.5% of the copy bandwidth against 72-90% on ShapeM)
    if (acc32) return ra::SHAPE_RS2;
    if (nranks <= 3) return (narrow && !minmax) ? ra::SHAPE_RS2 : ra::SHAPE_RS6;
    return minmax ? ra::SHAPE_RS : ra::SHAPE_S;
  }
  if (nranks <= 2) {
    if (acc32) return ra::SHAPE_S;
    return (narrow && !minmax) ? ra::SHAPE_S : ra::SHAPE_S4;
  }
  if (nranks == 3) return (acc32 || narrow) ? ra::SHAPE_M3 : ra::SHAPE_N3;
  if (narrow && minmax && nranks >= 6) {
    if (nranks <= 7) return ra::SHAPE_W8;
    if (nranks <= 9) return ra::SHAPE_W;
    if (nranks <= 15) return ra::SHAPE_M3;
    return ra::SHAPE_W;
  }
  if (nranks == 6 || nranks == 7) return (narrow && !acc32 && nranks == 6) ? ra::SHAPE_MB8 : ra::SHAPE_W8;
  if (acc32 && nranks == 8) return ra::SHAPE_W;
  if (nranks <= 7 || (narrow && nranks < 16)) return ra::SHAPE_M;
  if (nranks == 10 || nranks == 11 || nranks == 14) return ra::SHAPE_M;
  return ra::SHAPE_W;
}

// Checks shared by the three collectives; on success fills the kernel args.
ra_status_t prepare(int kind, const void* const* sendbufs, void* const* recvbufs, size_t count,
                    int dtype, int op, int nranks, ra::Args* a) {
  if (nranks < 1 || nranks > RA_MAX_RANKS) return RA_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  if (es == 0) return RA_ERR_INVALID_ARG;
  if (op < RA_SUM || op > RA_PROD) return RA_ERR_INVALID_ARG;
  if ((uint64_t)count > RA_MAX_COUNT) return RA_ERR_INVALID_ARG;
  if (sendbufs == nullptr || recvbufs == nullptr) return RA_ERR_INVALID_ARG;
  if (count == 0) return RA_SUCCESS;

  Range send[RA_MAX_RANKS], recv[RA_MAX_RANKS];
  for (int r = 0; r < nranks; ++r) {
    const uint64_t b = ra::chunk_begin(r, nranks, count), e = ra::chunk_begin(r + 1, nranks, count);
    const uint64_t full = count * (uint64_t)es, part = (e - b) * (uint64_t)es;
    const uint64_t send_bytes = kind == ra::KIND_ALLGATHER ? part : full;
    const uint64_t recv_bytes = kind == ra::KIND_REDUCE_SCATTER ? part : full;
    const uintptr_t s = reinterpret_cast<uintptr_t>(sendbufs[r]);
    const uintptr_t d = reinterpret_cast<uintptr_t>(recvbufs[r]);
    if ((send_bytes && s == 0) || (recv_bytes && d == 0)) return RA_ERR_INVALID_ARG;
    if (s % (uintptr_t)es || d % (uintptr_t)es) return RA_ERR_INVALID_ARG;
    if (s + send_bytes < s || d + recv_bytes < d) return RA_ERR_INVALID_ARG;  // wraps the address space
    send[r] = {s, s + (uintptr_t)send_bytes};
    recv[r] = {d, d + (uintptr_t)recv_bytes};
  }
  // A receive buffer may overlap nothing but its own rank's send buffer, and
  // that only in the exact in-place layout of the call.
  for (int r = 0; r < nranks; ++r) {
    const uintptr_t b_bytes = (uintptr_t)(ra::chunk_begin(r, nranks, count) * (uint64_t)es);
    for (int q = 0; q < nranks; ++q) {
      if (overlaps(recv[r], send[q])) {
        bool inplace = false;
        if (q == r) {
          if (kind == ra::KIND_ALLREDUCE) inplace = recv[r].lo == send[r].lo;
          if (kind == ra::KIND_REDUCE_SCATTER) inplace = recv[r].lo == send[r].lo + b_bytes;
          if (kind == ra::KIND_ALLGATHER) inplace = send[r].lo == recv[r].lo + b_bytes;
        }
        if (!inplace) return RA_ERR_ALIAS;
      }
      if (q != r && overlaps(recv[r], recv[q])) return RA_ERR_ALIAS;
    }
  }

  // Address phases: the N-way side must share one phase for the vector path
  // (AR: all sources and destinations; RS: the sources; AG: the destinations).
  // The grid is laid on the largest alignment, up to a 512-byte line, at
  // which every such buffer shares its phase.
  const Range* wide = kind == ra::KIND_ALLGATHER ? recv : send;
  unsigned align = ra::kLineAlignMax;
  for (; align >= (unsigned)ra::kVecBytes; align /= 2) {
    const unsigned ph = (unsigned)(wide[0].lo % align);
    bool same_here = true;
    for (int r = 0; r < nranks; ++r) {
      same_here = same_here && (wide[r].lo % align) == ph;
      if (kind == ra::KIND_ALLREDUCE) same_here = same_here && (recv[r].lo % align) == ph;
    }
    if (same_here) break;
  }
  const bool same = align >= (unsigned)ra::kVecBytes;
  if (!same) align = ra::kVecBytes;
  const unsigned phase_a = (unsigned)(wide[0].lo % align);
  const unsigned phase = (unsigned)(wide[0].lo % ra::kVecBytes);
  uint64_t compact_aligned = 0;
  if (kind != ra::KIND_ALLREDUCE) {
    const Range* compact = kind == ra::KIND_ALLGATHER ? send : recv;
    for (int c = 0; c < nranks; ++c) {
      const uint64_t b_bytes = ra::chunk_begin(c, nranks, count) * (uint64_t)es;
      const unsigned p = (unsigned)((compact[c].lo - (uintptr_t)b_bytes) % ra::kVecBytes);
      if (p == phase) compact_aligned |= (uint64_t)1 << c;
    }
  }
  for (int r = 0; r < nranks; ++r) {
    a->src[r] = sendbufs[r];
    a->dst[r] = recvbufs[r];
  }
  a->count = count;
  a->compact_aligned = compact_aligned;
  a->nranks = nranks;
  a->head = (int)(((align - phase_a) % align) / (unsigned)es);
  a->align_elems = (int)(align / (unsigned)es);
  a->vec_ok = same ? 1 : 0;
  a->inv_n = 1.0f / (float)nranks;
  a->step = 0;
  a->acc32 = 0;
  a->shape = shape_for(nranks);
  return RA_SUCCESS;
}

// A reduce-scatter whose compact output for some chunk sits off the vector
// grid at a 2-byte (odd-element) offset: its stores need the cooperative
// OFFGRID kernel. Offsets of 4 bytes or more are stored per lane in 4-byte
// units.
bool rs_needs_offgrid(const ra::Args& a, void* const* recvbufs, int es) {
  const int n = a.nranks;
  const uint64_t v = (uint64_t)(ra::kVecBytes / es);
  for (int c = 0; c < n; ++c) {
    if ((a.compact_aligned >> c) & 1u) continue;
    const uint64_t b0 = ra::chunk_begin(c, n, a.count), b1 = ra::chunk_begin(c + 1, n, a.count);
    uint64_t vb = b0, ve = b0;
    ra::vec_range(b0, b1, (uint64_t)a.head, (uint64_t)a.align_elems, v, &vb, &ve);
    if (ve == vb) continue;  // no whole vectors: element path only
    const uintptr_t addr = reinterpret_cast<uintptr_t>(recvbufs[c]) + (uintptr_t)((vb - b0) * (uint64_t)es);
    if ((addr & 3u) != 0) return true;
  }
  return false;
}

// SMs the launch may fill: all of them, or the caller's budget (max_sms > 0)
// when other work runs beside the collective.
ra_status_t sm_budget(int max_sms, int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return cuda_failed(err);
  if (max_sms > 0 && max_sms < *sms) *sms = max_sms;
  return RA_SUCCESS;
}

// Grid: blockIdx.y = chunk (or rank, for the ring steps); blockIdx.x = CTAs
// sharing it, enough to cover its vectors but no more than one resident wave
// of the launch shape on the SM budget; a one-trip shape takes a CTA per trip.
ra_status_t grid_for(const ra::Args& a, int dtype, int shape, int max_sms, dim3* grid, bool step_trip = false) {
  int threads, per_thread, min_blocks, sms = 0;
  if (shape == ra::kShapeAgBase + ra::AG_TILE) {
    // one CTA per whole tile of the longest chunk, plus one per chunk for its leftovers
    const ra::AgPlan p = ra::ag_plan_for(a.nranks);
    const int v = ra::kVecBytes / elem_size(dtype);
    const uint64_t gx = p.unroll == 1 ? ra::ag_tile_grid_x<1>(a.count, a.nranks, v)
                                      : (p.unroll == 2 ? ra::ag_tile_grid_x<2>(a.count, a.nranks, v)
                                                       : ra::ag_tile_grid_x<4>(a.count, a.nranks, v));
    if (gx > 0x7fffffffull) return RA_ERR_UNSUPPORTED;
    *grid = dim3((unsigned)gx, (unsigned)a.nranks);
    return RA_SUCCESS;
  }
  if (shape >= ra::kShapeAgBase) {  // the register all-gather
    const ra::AgPlan p = ra::ag_plan_for(a.nranks);
    threads = ra::AgShape::kThreads, per_thread = ra::AgShape::kUnroll;
    min_blocks = p.kernel == ra::AG_REGISTERS ? p.blocks_per_sm : ra::AgShape::kMinBlocks;
  } else if (shape == ra::SHAPE_STEP) {
    threads = ra::StepShape::kThreads, per_thread = ra::StepShape::kUnroll, min_blocks = ra::StepShape::kMinBlocks;
  } else {
    ra::shape_params(shape, &threads, &per_thread, &min_blocks);
  }
  const ra_status_t st = sm_budget(max_sms, &sms);
  if (st != RA_SUCCESS) return st;
  const uint64_t v = (uint64_t)(ra::kVecBytes / elem_size(dtype));
  const uint64_t n = (uint64_t)a.nranks;
  const uint64_t per_chunk = (a.count + n - 1) / n;
  const uint64_t work = a.vec_ok ? (per_chunk / v + 1) : per_chunk;  // vectors, or elements
  const uint64_t per_cta = a.vec_ok ? (uint64_t)threads * per_thread : (uint64_t)threads;
  uint64_t gx = (work + per_cta - 1) / per_cta;
  const uint64_t cap = (uint64_t)sms * min_blocks / n;
  const bool one_trip = ra::is_trip_shape(shape) || (shape == ra::SHAPE_STEP && step_trip && max_sms == 0);
  if (!one_trip && gx > cap) gx = cap;
  if (gx > 0x7fffffffull) return RA_ERR_UNSUPPORTED;
  if (gx < 1) gx = 1;
  *grid = dim3((unsigned)gx, (unsigned)a.nranks);
  return RA_SUCCESS;
}

ra_status_t launch(int kind, int dtype, int op, const ra::Args& a, dim3 grid, void* stream) {
  const cudaError_t err = ra::launch_kernel(kind, dtype, op, a, grid, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? RA_SUCCESS : cuda_failed(err);
}

const ra_options_t kDefaultOptions = {RA_ORDER_RING, RA_ACCUM_DTYPE, 0, RA_ENGINE_REGISTERS, nullptr};

// Memory the device reaches over the host link: pinned host memory, or pageable
// host memory on a system whose GPU reads system memory coherently (the
// runtime reports them as registered and unregistered host memory). Device and
// managed memory are not. A pointer the runtime cannot describe counts as
// device memory; its launch then reports any failure of its own.
bool on_host(const void* p) {
  if (p == nullptr) return false;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}
bool any_on_host(const ra::Args& a) {
  for (int r = 0; r < a.nranks; ++r)
    if (on_host(a.src[r]) || on_host(a.dst[r])) return true;
  return false;
}

// The bulk engine: tiles of tile_vecs vectors per rank, as many stages as fit
// in about 200 KB of shared memory (2..8), one CTA per SM on the budget.
#ifndef RA_BULK_SMEM_KB
#define RA_BULK_SMEM_KB 200
#endif
constexpr size_t kBulkSmemBudget = (size_t)RA_BULK_SMEM_KB * 1024;
#ifndef RA_BULK_MAX_STAGES
#define RA_BULK_MAX_STAGES 8
#endif
constexpr int kBulkMaxStages = RA_BULK_MAX_STAGES;

// A planned bulk-engine launch: kernel arguments, grid and shared memory.
struct BulkLaunch {
  ra::BulkArgs args;
  dim3 grid;
  size_t smem = 0;
};

// Plans a bulk-engine launch and raises the kernel's shared-memory limit to
// what it needs. Enqueues nothing: every error the bulk path can report before
// its launch is reported here.
ra_status_t plan_bulk(const ra::Args& a, int dtype, int op, int max_sms, BulkLaunch* p) {
  // the bulk engine's loads are TMA bulk copies, which the library issues on device memory only
  if (any_on_host(a)) return RA_ERR_UNSUPPORTED;
  ra::BulkArgs& b = p->args;
  b.base = a;
  b.status = nullptr;
  b.status_stride = 0;
  b.withhold_chunk = -1;
  const int n = a.nranks;
  int sms = 0, all_sms = 0;
  ra_status_t st = sm_budget(max_sms, &sms);
  if (st == RA_SUCCESS) st = sm_budget(0, &all_sms);
  if (st != RA_SUCCESS) return st;
  const uint32_t nc = (uint32_t)ra::bulk_consumers_for(n, sms < all_sms);
  b.consumers = nc;
  // about 32 KB per stage: 32 KB / N per rank, between 4 and 16 KB (fewer, longer tiles when N
  // is small, so the per-tile barrier work is spread over more bytes), and one vector per consumer
  // thread where two stages still fit
  uint32_t tile_bytes = 32768u / (uint32_t)n;
  if (tile_bytes < 4096u) tile_bytes = 4096u;
  if (tile_bytes > 16384u) tile_bytes = 16384u;
  uint32_t tv = tile_bytes / (uint32_t)ra::kVecBytes;
  tv = tv / nc * nc;
  if (tv < nc) tv = nc;
  // keep at least two stages: shrink the tile to a multiple of a warp's vectors (some consumer
  // threads then idle on each tile)
  while (tv > 32 && 2 * (size_t)n * tv * ra::kVecBytes > kBulkSmemBudget) tv -= 32;
  b.tile_vecs = tv;
  const size_t stage_bytes = (size_t)n * b.tile_vecs * ra::kVecBytes;
  size_t stages = kBulkSmemBudget / stage_bytes;
  if (stages > (size_t)kBulkMaxStages) stages = kBulkMaxStages;
  if (stages < 2) return RA_ERR_UNSUPPORTED;
  b.stages = (uint32_t)stages;
  p->smem = 128 * ((2 * stages * 8 + 127) / 128) + stages * stage_bytes;
  const uint64_t v = (uint64_t)(ra::kVecBytes / elem_size(dtype));
  const uint64_t tiles = ((a.count + n - 1) / n / v) / b.tile_vecs + 1;
  uint64_t gx = (uint64_t)sms / (uint64_t)n;
  if (gx > tiles) gx = tiles;
  if (gx < 1) gx = 1;
  p->grid = dim3((unsigned)gx, (unsigned)n);
  const cudaError_t err = ra::configure_bulk_kernel(dtype, op, p->smem);
  return err == cudaSuccess ? RA_SUCCESS : cuda_failed(err);
}

// Enqueues a planned bulk-engine launch. status: the device words the CTAs of
// chunk c report into (word c * status_stride); withhold_chunk >= 0 runs the
// self-test that leaves that chunk's first tile uncopied.
ra_status_t launch_bulk(BulkLaunch p, int dtype, int op, int* status, uint32_t status_stride,
                        int withhold_chunk, void* stream) {
  p.args.status = status;
  p.args.status_stride = status_stride;
  p.args.withhold_chunk = withhold_chunk;
  const cudaError_t err =
      ra::launch_bulk_kernel(dtype, op, p.args, p.grid, p.smem, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? RA_SUCCESS : cuda_failed(err);
}

ra_status_t run_bulk(const ra::Args& a, int dtype, int op, int max_sms, int* status, void* stream) {
  BulkLaunch p;
  const ra_status_t st = plan_bulk(a, dtype, op, max_sms, &p);
  if (st != RA_SUCCESS) return st;
  return launch_bulk(p, dtype, op, status, 0, -1, stream);
}

// ---- reduction programs of the other orders --------------------------------
// A program is a list of steps slot[a] = op(slot[a], slot[b]) over the N rank
// slots; after it runs, slot `root` holds the element's result.
void emit(ra::OrderArgs& o, int pr, int a, int b) {
  const int t = o.prog_len[pr]++;
  o.prog[pr][t][0] = (uint8_t)a;
  o.prog[pr][t][1] = (uint8_t)b;
}

// Recursive halving with distance d = N/2, ..., 1: the rank with the d bit
// clear combines its partial (left operand) with its partner's, so level by
// level slot r absorbs slot r + d.
void rabenseifner_program(ra::OrderArgs& o, int pr, int n) {
  for (int d = n / 2; d >= 1; d /= 2)
    for (int r = 0; r < d; ++r) emit(o, pr, r, r + d);
  o.root[pr] = 0;
}

// A binary tree laid over the rank sequence seq[lo..hi] in order (the middle
// position is the root): a node folds its left subtree's partial, its own
// value, then its right subtree's partial. Returns the slot of the result.
int inorder_program(ra::OrderArgs& o, int pr, const int* seq, int lo, int hi) {
  if (lo > hi) return -1;
  const int m = (lo + hi) / 2, v = seq[m];
  const int left = inorder_program(o, pr, seq, lo, m - 1);
  const int right = inorder_program(o, pr, seq, m + 1, hi);
  int acc = v;
  if (left >= 0) {
    emit(o, pr, left, v);
    acc = left;
  }
  if (right >= 0) emit(o, pr, acc, right);
  return acc;
}

// Double binary tree: tree 0 over ranks 0..N-1 reduces chunks [0, N/2),
// tree 1 over ranks N-1..0 reduces the rest.
void tree_programs(ra::OrderArgs& o, int n) {
  int fwd[RA_MAX_RANKS], bwd[RA_MAX_RANKS];
  for (int i = 0; i < n; ++i) {
    fwd[i] = i;
    bwd[i] = n - 1 - i;
  }
  o.root[0] = (uint8_t)inorder_program(o, 0, fwd, 0, n - 1);
  o.root[1] = (uint8_t)inorder_program(o, 1, bwd, 0, n - 1);
  for (int c = n / 2; c < n; ++c) o.chunk_prog |= (uint64_t)1 << c;
}

ra_status_t run_ordered(int kind, const ra::Args& a, int dtype, int op, int order, int max_sms, void* stream) {
  // the ordered kernel stages its loads with cp.async, which the library issues on device memory only
  if (any_on_host(a)) return RA_ERR_UNSUPPORTED;
  ra::OrderArgs o;
  memset(&o, 0, sizeof(o));
  o.base = a;
  const int n = a.nranks;
  if (order == RA_ORDER_RABENSEIFNER) rabenseifner_program(o, 0, n);
  else tree_programs(o, n);
  int sms = 0;
  const ra_status_t st = sm_budget(max_sms, &sms);
  if (st != RA_SUCCESS) return st;
  // resident CTAs per SM: shared memory (N slots per thread) and at most 1024 threads
  const uint64_t smem = (uint64_t)n * ra::kOrdThreads * ra::kOrdVecBytes;
  uint64_t per_sm = (uint64_t)(220 * 1024) / smem;
  if (per_sm > 1024 / ra::kOrdThreads) per_sm = 1024 / ra::kOrdThreads;
  if (per_sm < 1) per_sm = 1;
  const uint64_t v = (uint64_t)(ra::kOrdVecBytes / elem_size(dtype));
  const uint64_t per_chunk = (a.count + n - 1) / n;
  const uint64_t work = a.vec_ok ? per_chunk / v + 1 : per_chunk;
  uint64_t gx = (work + ra::kOrdThreads - 1) / ra::kOrdThreads;
  const uint64_t cap = (uint64_t)sms * per_sm / (uint64_t)n;
  // From N = 4 a CTA per trip (each CTA stages, folds and stores one trip and
  // exits) instead of one resident wave: fp32 avg, 1-2 GiB over all ranks, back
  // to back, 102-105% of the copy bandwidth at N = 4..16 against 93-96%; at
  // N = 2 and 3 it measured 76% and 94% against 92% and 98%.
  const bool one_trip = max_sms == 0 && n >= 4;
  if (!one_trip && gx > cap) gx = cap;
  if (gx > 0x7fffffffull) return RA_ERR_UNSUPPORTED;
  if (gx < 1) gx = 1;
  const dim3 grid((unsigned)gx, (unsigned)n);
  const cudaError_t err = ra::launch_ordered_kernel(kind == ra::KIND_REDUCE_SCATTER, dtype, op, o, grid,
                                                    static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? RA_SUCCESS : cuda_failed(err);
}

// The one-trip shape for a fused call, or -1 to keep the one-wave shape, on
// every SM (an SM budget caps the grid by definition). minmax: a float min/max
// (int32 min/max fold as cheaply as sums and take the sum shapes). Each rule
// below is the measured winner (back to back, 1 GiB and 256 MiB over all ranks):
// - TripW at small N: all-reduces at N <= 2; reduce-scatters whose shards all
//   sit on the vector grid at N <= 4, and at N = 5..7 for 16-bit types and
//   float min/max (shards stored in 4-byte units lost up to 25 points on it);
// - TripS for all-reduces from N = 3, and for reduce-scatters from N = 8 and,
//   for 4-byte types, from N = 4 (fp32 avg at 1 GiB: 105-107% against 101-105%;
//   bf16 lost 3-4 points there); TripRS2 for float min/max reduce-scatters,
//   on and off the grid (bf16 with 2-byte-offset shards, N = 9..15: 102.3-104.5%
//   against 94.6-100.3% on TripS);
// - fp32 partials and shards off the vector grid take trips too, but not both
//   at once (bf16 avg at N = 12: 96.7% one-wave against 90.0%); reduce-scatters
//   with fp32 partials from N = 3 when every shard is on the grid (TripAccRS);
// - large 16-bit off-grid sums at N = 5..7 (below).
// RA_GRID_MODE, a build-time tunable for sweeps: -1 these rules, 0 never, 1
// wherever a trip shape exists.
#ifndef RA_GRID_MODE
#define RA_GRID_MODE -1
#endif
int trip_shape_for(int kind, int nranks, int elem_bytes, bool acc32, bool minmax, bool offgrid, bool shards_on_grid,
                   uint64_t total_bytes, int max_sms) {
  if (max_sms > 0 || kind == ra::KIND_ALLGATHER) return -1;
  const bool rs = kind == ra::KIND_REDUCE_SCATTER;
  if (rs && offgrid && acc32) return -1;
  // TripW: all-reduces at N <= 2; reduce-scatters whose shards all sit on the vector grid at
  // N <= 4, and at N = 5..7 for 16-bit types and float min/max (1 GiB over all ranks: 106-108.7%
  // against 100.4-104.8%; 256 MiB: 97.7-103% against 96-102.7%). 4-byte sums at N = 5..7 measured
  // the same at 1 GiB and up to 4 points lower at 256 MiB, and every call from N = 8 up to 5 points
  // lower at 256 MiB, so those keep TripS / TripRS2.
  const bool small_n =
      !acc32 && (rs ? shards_on_grid && (nranks <= 4 || (nranks <= 7 && (elem_bytes == 2 || minmax))) : nranks <= 2);
  int trip;
  if (small_n) trip = ra::SHAPE_TRIP_W;
  else if (rs && offgrid) trip = minmax ? ra::SHAPE_TRIP_RS2_OFFGRID : ra::SHAPE_TRIP_RS_OFFGRID;
  else if (acc32) trip = rs ? ra::SHAPE_TRIP_ACC_RS2 : ra::SHAPE_TRIP_ACC;
  else trip = (rs && minmax) ? ra::SHAPE_TRIP_RS2 : ra::SHAPE_TRIP_S;
#if RA_GRID_MODE >= 0
  (void)nranks, (void)elem_bytes, (void)total_bytes;
  return RA_GRID_MODE == 1 ? trip : -1;
#else
  if (small_n) return trip;
  // 16-bit sum/avg/prod with 2-byte-offset shards at N = 5..7 stream best on TripW from about
  // 384 MiB over all ranks (bf16 avg / fp16 sum at 1 GiB: 102.5-104.8% against 97.2-100.5%; at
  // 512 MiB +2.8-4.6 points at N = 6, 7 and level at 5; at 384 MiB +0.3-1.8), one wave below that
  // (at 256 MiB TripW lost 4 points at N = 5, at 128 MiB 3-6 points) and at N = 3 (it lost 2-16
  // points at every size)
  if (rs && offgrid && elem_bytes == 2 && !minmax && nranks >= 5 && nranks <= 7 && total_bytes >= (320ull << 20))
    return ra::SHAPE_TRIP_W_OFFGRID;
  // fp32 partials take a trip from N = 3 when every shard is on the vector grid (TripAccRS: +0.6-3.8
  // points at 256 MiB - 1 GiB over all ranks against one wave)
  if (rs && acc32 && shards_on_grid && nranks >= 3) return trip;
  if (rs) return (nranks >= 8 || (elem_bytes == 4 && nranks >= 4)) ? trip : -1;
  return nranks >= 3 ? trip : -1;
#endif
}

ra_status_t run(int kind, const void* const* sendbufs, void* const* recvbufs, size_t count, ra_dtype_t dtype,
                ra_op_t op, int nranks, void* stream, const ra_options_t* options = &kDefaultOptions) {
  ra::Args a;
  if (kind == ra::KIND_ALLGATHER) op = RA_SUM;  // no reduction; any valid op is accepted
  if (options == nullptr) options = &kDefaultOptions;
  const int order = options->order, accum = options->accum, max_sms = options->max_sms;
  const int engine = options->engine;
  if (accum != RA_ACCUM_DTYPE && accum != RA_ACCUM_FP32) return RA_ERR_INVALID_ARG;
  if (order < RA_ORDER_RING || order > RA_ORDER_RABENSEIFNER || max_sms < 0) return RA_ERR_INVALID_ARG;
  if (engine != RA_ENGINE_REGISTERS && engine != RA_ENGINE_BULK) return RA_ERR_INVALID_ARG;
  if (engine == RA_ENGINE_BULK && options->status == nullptr) return RA_ERR_INVALID_ARG;
  ra_status_t st = prepare(kind, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS) return st;
  if (order == RA_ORDER_RABENSEIFNER && (nranks & (nranks - 1))) return RA_ERR_UNSUPPORTED;
  if (order != RA_ORDER_RING && accum == RA_ACCUM_FP32) return RA_ERR_UNSUPPORTED;
  if (engine == RA_ENGINE_BULK &&
      (kind != ra::KIND_ALLREDUCE || order != RA_ORDER_RING || accum != RA_ACCUM_DTYPE || nranks > 16))
    return RA_ERR_UNSUPPORTED;
  if (count == 0) return RA_SUCCESS;
  if (engine == RA_ENGINE_BULK) {
    if (!a.vec_ok) return RA_ERR_UNSUPPORTED;
    return run_bulk(a, dtype, op, max_sms, options->status, stream);
  }
  if (order != RA_ORDER_RING) return run_ordered(kind, a, dtype, op, order, max_sms, stream);
  // fp32 partials for fp16/bf16 sum, avg and prod. min and max are exact in
  // any precision: partials would give the same bits (any NaN for any NaN),
  // so those calls take the buffer-dtype kernels.
  a.acc32 = (accum == RA_ACCUM_FP32 && (dtype == RA_FLOAT16 || dtype == RA_BFLOAT16) && op != RA_MIN &&
             op != RA_MAX)
                ? 1
                : 0;
  // the tile all-gather gives a chunk's per-element work to one CTA: with mixed
  // address phases (every element on the per-element path) the register
  // kernel's rows of CTAs spread it instead
  int ag_kernel = ra::ag_plan_for(nranks).kernel;
  if (!a.vec_ok) ag_kernel = ra::AG_REGISTERS;
  // the tile kernel writes with TMA bulk stores, which the library issues on device memory only;
  // buffers in host memory take the register kernel's plain stores
  if (kind == ra::KIND_ALLGATHER && ag_kernel == ra::AG_TILE && any_on_host(a)) ag_kernel = ra::AG_REGISTERS;
  a.shape = kind == ra::KIND_ALLGATHER ? ra::kShapeAgBase + ag_kernel
                                       : shape_for(nranks, kind == ra::KIND_REDUCE_SCATTER, a.acc32 != 0,
                                                   dtype == RA_FLOAT16 || dtype == RA_BFLOAT16,
                                                   op == RA_MIN || op == RA_MAX);
  const bool offgrid =
      kind == ra::KIND_REDUCE_SCATTER && a.vec_ok && rs_needs_offgrid(a, recvbufs, elem_size(dtype));
  if (offgrid)
    a.shape = a.acc32 ? ra::SHAPE_RS_OFFGRID_M
                      : (a.shape == ra::SHAPE_S ? ra::SHAPE_RS_OFFGRID : ra::SHAPE_RS_OFFGRID_B2);
  const uint64_t all_chunks = nranks >= 64 ? ~0ull : ((1ull << nranks) - 1);
  const bool shards_on_grid = a.vec_ok && (a.compact_aligned & all_chunks) == all_chunks;
  // int32 min/max folds are as light as sums and stream best on the sum shapes (reduce-scatter at
  // 1 GiB over all ranks, N = 4..16: 104.7-107.9% on TripS against 99.5-106.9% on TripRS2); the
  // IEEE minimum/maximum of the float types keeps TripRS2 (TripS: 92.5-105.4% against 99.0-106.8%)
  const bool minmax_shape = (op == RA_MIN || op == RA_MAX) && dtype != RA_INT32;
  const uint64_t rank_bytes = (uint64_t)count * (uint64_t)elem_size(dtype);  // <= 2^59
  const uint64_t total_bytes = rank_bytes > UINT64_MAX / (uint64_t)nranks ? UINT64_MAX : rank_bytes * (uint64_t)nranks;
  const int trip = trip_shape_for(kind, nranks, elem_size(dtype), a.acc32 != 0, minmax_shape, offgrid,
                                  shards_on_grid, total_bytes, max_sms);
  // buffers in host memory stream over the host link faster from one resident wave (8 x 256 MiB fp32
  // avg on pinned host buffers: 335.5 GB/s of link traffic, the rate of concurrent copy-engine
  // transfers, against 326.9 GB/s with a CTA per trip)
  const bool host_side = on_host(sendbufs[0]) || on_host(recvbufs[0]);
  if (trip >= 0 && !host_side) a.shape = trip;
  dim3 grid;
  st = grid_for(a, dtype, a.shape, max_sms, &grid);
  if (st != RA_SUCCESS) return st;
  return launch(kind, dtype, op, a, grid, stream);
}

ra_status_t run_ringsteps(const void* const* sendbufs, void* const* recvbufs, size_t count, ra_dtype_t dtype,
                          ra_op_t op, int nranks, int nsteps, void* stream) {
  ra::Args a;
  ra_status_t st = prepare(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS || count == 0) return st;
  const int total = 2 * (nranks - 1);
  if (nsteps < 0 || nsteps > total) nsteps = total;
  dim3 grid;
  if (nranks == 1) {  // no ring steps: the result is the (avg-scaled) copy
    a.shape = shape_for(1);
    st = grid_for(a, dtype, a.shape, 0, &grid);
    return st != RA_SUCCESS ? st : launch(ra::KIND_ALLREDUCE, dtype, op, a, grid, stream);
  }
  // A CTA per trip from 64 MiB per rank: 8 x 256 MiB fp32 avg 1.336 ms (103.6% of the copy
  // bandwidth for the schedule's own bytes) against 1.465 ms (94.5%) as one resident wave,
  // 4 x 256 MiB 101.6 against 94.1%, 16 x 64 MiB 89.9 against 85.4%; at 8 x 32 MiB bf16 it lost
  // (78.6 against 87.9%).
  const bool step_trip = (uint64_t)count * (uint64_t)elem_size(dtype) >= (64ull << 20);
  st = grid_for(a, dtype, ra::SHAPE_STEP, 0, &grid, step_trip);
  if (st != RA_SUCCESS) return st;
  for (int k = 0; k < nsteps; ++k) {
    const bool rs = k < nranks - 1;
    a.step = rs ? k : k - (nranks - 1);
    st = launch(rs ? ra::KIND_RING_RS_STEP : ra::KIND_RING_AG_STEP, dtype, op, a, grid, stream);
    if (st != RA_SUCCESS) return st;
  }
  return RA_SUCCESS;
}

// Gradient buckets (bitfern.com "AllReduce Explained", "PyTorch DDP and
// Gradient Synchronization"; tirogla.com "Ring all-reduce", "Implementation
// notes"): parameters are visited in the order backward produces their
// gradients (reverse registration order) and packed into buckets of at most
// bucket_bytes; a parameter larger than that gets a bucket of its own. With the
// parameters laid out contiguously in registration order, every bucket is one
// contiguous element range of the flat gradient buffer.
ra_status_t bucket_plan(const size_t* counts, int nparams, size_t bucket_bytes, int elem_size_bytes,
                        size_t* begin, size_t* count, int max_buckets, int* nbuckets) {
  if (nparams < 0 || (nparams > 0 && counts == nullptr) || nbuckets == nullptr || bucket_bytes == 0 ||
      (elem_size_bytes != 2 && elem_size_bytes != 4) || max_buckets < 0)
    return RA_ERR_INVALID_ARG;
  uint64_t end = 0;
  for (int p = 0; p < nparams; ++p) end += counts[p];
  int nb = 0;
  uint64_t cur_begin = end, cur_bytes = 0;
  bool open = false;
  for (int p = nparams - 1; p >= 0; --p) {
    const uint64_t bytes = (uint64_t)counts[p] * (uint64_t)elem_size_bytes;
    if (open && cur_bytes + bytes > bucket_bytes) {  // close the current bucket
      if (nb < max_buckets && begin && count) {
        begin[nb] = (size_t)cur_begin;
        count[nb] = (size_t)(end - cur_begin);
      }
      ++nb;
      end = cur_begin;
      cur_bytes = 0;
      open = false;
    }
    cur_begin -= counts[p];
    cur_bytes += bytes;
    open = true;
  }
  if (open) {
    if (nb < max_buckets && begin && count) {
      begin[nb] = (size_t)cur_begin;
      count[nb] = (size_t)(end - cur_begin);
    }
    ++nb;
  }
  *nbuckets = nb;
  return nb <= max_buckets ? RA_SUCCESS : RA_ERR_INVALID_ARG;
}

// The all-reduces of buckets [first, first + k) of the table in one launch (k >= 2):
// ring order, register engine; `whole` holds the checked N whole buffers. From
// N = 3 on all SMs the group takes a CTA per trip of every bucket's chunk, like
// a single all-reduce; otherwise one resident wave walks the buckets in turn.
ra_status_t launch_group(const ra::Args& whole, int dtype, int op, int accum, int max_sms, const size_t* bucket_begin,
                         const size_t* bucket_count, const int* members, int k, void* stream) {
  ra::GroupArgs g;
  g.a = whole;
  g.nbuckets = (uint32_t)k;
  uint64_t total = 0;
  for (int i = 0; i < k; ++i) {
    g.begin[i] = bucket_begin[members[i]];
    g.count[i] = bucket_count[members[i]];
    total += g.count[i];
  }
  ra::Args& a = g.a;
  a.acc32 = (accum == RA_ACCUM_FP32 && (dtype == RA_FLOAT16 || dtype == RA_BFLOAT16) && op != RA_MIN &&
             op != RA_MAX)
                ? 1
                : 0;
  const int n = a.nranks;
  const int trip = trip_shape_for(ra::KIND_ALLREDUCE, n, elem_size(dtype), a.acc32 != 0,
                                  op == RA_MIN || op == RA_MAX, false, true, 0, max_sms);
  dim3 grid;
  if (trip >= 0) {
    // every trip is threads x vectors of a chunk (TripS: 128, TripW: 256); a bucket's chunks have
    // at most len / n + 1 elements, and its last CTA also takes the edge elements, so it has at
    // least one
    const uint64_t per_trip = trip == ra::SHAPE_TRIP_W ? (uint64_t)ra::TripW::kThreads * ra::TripW::kUnroll
                                                       : (uint64_t)ra::TripS::kThreads * ra::TripS::kUnroll;
    const uint64_t v = (uint64_t)(ra::kVecBytes / elem_size(dtype));
    uint64_t trips = 0;
    for (int i = 0; i < k; ++i) {
      g.trip_begin[i] = (uint32_t)trips;
      trips += (g.count[i] / (uint64_t)n + 1) / v / per_trip + 1;
      if (trips > 0x7fffffffull) return RA_ERR_UNSUPPORTED;
    }
    g.trip_begin[k] = (uint32_t)trips;
    a.shape = trip;
    grid = dim3((unsigned)trips, (unsigned)n);
  } else {
    a.shape = shape_for(n, false, a.acc32 != 0, dtype == RA_FLOAT16 || dtype == RA_BFLOAT16,
                        op == RA_MIN || op == RA_MAX);
    // the bucket loop needs a few more registers than ShapeS and ShapeM3 budget (a shape
    // changes how fast, never which bits)
    if (a.shape == ra::SHAPE_S || a.shape == ra::SHAPE_M3) a.shape = ra::SHAPE_M;
    a.count = total;  // sizes the grid like one all-reduce of the group's elements
    const ra_status_t st = grid_for(a, dtype, a.shape, max_sms, &grid);
    if (st != RA_SUCCESS) return st;
  }
  const cudaError_t err = ra::launch_group_kernel(dtype, op, g, grid, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? RA_SUCCESS : cuda_failed(err);
}

ra_status_t run_buckets(const void* const* sendbufs, void* const* recvbufs, size_t count, ra_dtype_t dtype,
                        ra_op_t op, int nranks, int nbuckets, const size_t* bucket_begin,
                        const size_t* bucket_count, void* const* ready_events, const ra_options_t* options,
                        void* stream) {
  ra::Args whole;
  ra_status_t st = prepare(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, &whole);
  if (st != RA_SUCCESS) return st;
  if (nbuckets < 0 || (nbuckets > 0 && (bucket_begin == nullptr || bucket_count == nullptr)))
    return RA_ERR_INVALID_ARG;
  // buckets inside [0, count), disjoint, listed in ascending or descending order
  int dir = 0;
  for (int b = 0; b < nbuckets; ++b) {
    if (bucket_begin[b] > count || bucket_count[b] > count - bucket_begin[b]) return RA_ERR_INVALID_ARG;
    if (b > 0) {
      const size_t pb = bucket_begin[b - 1], pe = pb + bucket_count[b - 1];
      const size_t cb = bucket_begin[b], ce = cb + bucket_count[b];
      const int d = cb >= pe ? 1 : (ce <= pb ? -1 : 0);
      if (d == 0 || (dir != 0 && d != dir)) return RA_ERR_INVALID_ARG;
      dir = d;
    }
  }
  if (options == nullptr) options = &kDefaultOptions;
  // the per-bucket path checks the options; the grouped one takes the defaults' engine and order only
  const bool groupable = count > 0 && options->engine == RA_ENGINE_REGISTERS && options->order == RA_ORDER_RING &&
                         (options->accum == RA_ACCUM_DTYPE || options->accum == RA_ACCUM_FP32) &&
                         options->max_sms >= 0;
  const int es = elem_size(dtype);
  const void* s_ptr[RA_MAX_RANKS];
  void* d_ptr[RA_MAX_RANKS];
  auto one_bucket = [&](int b) -> ra_status_t {
    const size_t off = bucket_begin[b] * (size_t)es;
    for (int r = 0; r < nranks; ++r) {
      s_ptr[r] = static_cast<const char*>(sendbufs[r]) + off;
      d_ptr[r] = static_cast<char*>(recvbufs[r]) + off;
    }
    return run(ra::KIND_ALLREDUCE, s_ptr, d_ptr, bucket_count[b], dtype, op, nranks, stream, options);
  };
  // Buckets with no ready event of their own follow the previous bucket without a
  // wait; a run of such buckets goes out as one grouped launch.
  int members[ra::kMaxGroup];
  int k = 0;
  auto flush = [&]() -> ra_status_t {
    ra_status_t r = RA_SUCCESS;
    if (k == 1) r = one_bucket(members[0]);
    else if (k > 1)
      r = launch_group(whole, dtype, op, options->accum, options->max_sms, bucket_begin, bucket_count, members, k,
                       stream);
    k = 0;
    return r;
  };
  for (int b = 0; b < nbuckets; ++b) {
    if (ready_events && ready_events[b]) {
      st = flush();
      if (st != RA_SUCCESS) return st;
      const cudaError_t err = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream),
                                                  static_cast<cudaEvent_t>(ready_events[b]), 0);
      if (err != cudaSuccess) return cuda_failed(err);
    }
    if (bucket_count[b] == 0) continue;
    if (!groupable) {
      st = one_bucket(b);
      if (st != RA_SUCCESS) return st;
      continue;
    }
    members[k++] = b;
    if (k == ra::kMaxGroup) {
      st = flush();
      if (st != RA_SUCCESS) return st;
    }
  }
  return flush();
}

}  // namespace

extern "C" {

ra_status_t ra_allreduce(const void* const* sendbufs, void* const* recvbufs, size_t count,
                         ra_dtype_t dtype, ra_op_t op, int nranks, void* stream) {
  return run(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, stream);
}

ra_status_t ra_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, size_t count,
                              ra_dtype_t dtype, ra_op_t op, int nranks, void* stream) {
  return run(ra::KIND_REDUCE_SCATTER, sendbufs, recvbufs, count, dtype, op, nranks, stream);
}

ra_status_t ra_allgather(const void* const* sendbufs, void* const* recvbufs, size_t count,
                         ra_dtype_t dtype, ra_op_t op, int nranks, void* stream) {
  return run(ra::KIND_ALLGATHER, sendbufs, recvbufs, count, dtype, op, nranks, stream);
}

ra_status_t ra_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, size_t count, ra_dtype_t dtype,
                            ra_op_t op, int nranks, const ra_options_t* options, void* stream) {
  return run(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, stream, options);
}

ra_status_t ra_reduce_scatter_ex(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                 ra_dtype_t dtype, ra_op_t op, int nranks, const ra_options_t* options,
                                 void* stream) {
  return run(ra::KIND_REDUCE_SCATTER, sendbufs, recvbufs, count, dtype, op, nranks, stream, options);
}

ra_status_t ra_bucket_plan(const size_t* param_counts, int nparams, size_t bucket_bytes, int elem_size,
                           size_t* bucket_begin, size_t* bucket_count, int max_buckets, int* nbuckets) {
  return bucket_plan(param_counts, nparams, bucket_bytes, elem_size, bucket_begin, bucket_count, max_buckets,
                     nbuckets);
}

ra_status_t ra_allreduce_buckets(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                 ra_dtype_t dtype, ra_op_t op, int nranks, int nbuckets, const size_t* bucket_begin,
                                 const size_t* bucket_count, void* const* ready_events,
                                 const ra_options_t* options, void* stream) {
  return run_buckets(sendbufs, recvbufs, count, dtype, op, nranks, nbuckets, bucket_begin, bucket_count,
                     ready_events, options, stream);
}

ra_status_t ra_allreduce_ringsteps(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                   ra_dtype_t dtype, ra_op_t op, int nranks, int nsteps, void* stream) {
  return run_ringsteps(sendbufs, recvbufs, count, dtype, op, nranks, nsteps, stream);
}

ra_status_t ra_chunk_range(size_t count, int nranks, int c, size_t* begin, size_t* end) {
  if (nranks < 1 || nranks > RA_MAX_RANKS || c < 0 || c >= nranks) return RA_ERR_INVALID_ARG;
  if ((uint64_t)count > RA_MAX_COUNT || begin == nullptr || end == nullptr) return RA_ERR_INVALID_ARG;
  *begin = (size_t)ra::chunk_begin(c, nranks, count);
  *end = (size_t)ra::chunk_begin(c + 1, nranks, count);
  return RA_SUCCESS;
}

ra_status_t ra_plan_chunk(size_t count, int nranks, int c, int elem_size_bytes, int align_bytes, int phase_bytes,
                          size_t* begin, size_t* end, size_t* vec_begin, size_t* vec_end) {
  if (elem_size_bytes != 2 && elem_size_bytes != 4) return RA_ERR_INVALID_ARG;
  if (align_bytes < ra::kVecBytes || align_bytes > ra::kLineAlignMax || (align_bytes & (align_bytes - 1)))
    return RA_ERR_INVALID_ARG;
  if (phase_bytes < 0 || phase_bytes >= align_bytes || phase_bytes % elem_size_bytes) return RA_ERR_INVALID_ARG;
  if (vec_begin == nullptr || vec_end == nullptr) return RA_ERR_INVALID_ARG;
  const ra_status_t st = ra_chunk_range(count, nranks, c, begin, end);
  if (st != RA_SUCCESS) return st;
  const uint64_t head = (uint64_t)((align_bytes - phase_bytes) % align_bytes) / elem_size_bytes;
  uint64_t vb, ve;
  ra::vec_range(*begin, *end, head, (uint64_t)(align_bytes / elem_size_bytes),
                (uint64_t)(ra::kVecBytes / elem_size_bytes), &vb, &ve);
  *vec_begin = (size_t)vb;
  *vec_end = (size_t)ve;
  return RA_SUCCESS;
}

const char* ra_status_string(ra_status_t status) {
  switch (status) {
    case RA_SUCCESS: return "success";
    case RA_ERR_INVALID_ARG: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported dtype/op/order";
    case RA_ERR_ALIAS: return "buffers overlap outside the in-place layout";
    case RA_ERR_CUDA: return "CUDA launch failed";
    case RA_ERR_SCRATCH_LIMIT: return "nranks exceeds the library's status words (RA_NOALLOC_STATUS_WORDS)";
  }
  return "unknown status";
}

int ra_last_cuda_error(void) { return g_last_cuda_error; }

int ra_vector_bytes(void) { return ra::kVecBytes; }

ra_status_t ra_selftest_bulk_timeout(const void* const* sendbufs, void* const* recvbufs, size_t count,
                                     ra_dtype_t dtype, ra_op_t op, int nranks, int withhold_chunk, int* status,
                                     int status_per_chunk, void* stream) {
  if (status == nullptr || (status_per_chunk != 0 && status_per_chunk != 1)) return RA_ERR_INVALID_ARG;
  if (withhold_chunk < 0 || withhold_chunk >= nranks) return RA_ERR_INVALID_ARG;
  ra::Args a;
  ra_status_t st = prepare(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS) return st;
  if (nranks > 16 || !a.vec_ok || count == 0) return RA_ERR_UNSUPPORTED;
  BulkLaunch p;
  st = plan_bulk(a, dtype, op, 0, &p);
  if (st != RA_SUCCESS) return st;
  return launch_bulk(p, dtype, op, status, (uint32_t)status_per_chunk, withhold_chunk, stream);
}

}  // extern "C"

// ---- the bulk all-reduce without caller scratch ------------------------------
// The status words of ra_allreduce_bulk_noalloc: one per chunk, part of the
// module's device image, so no call allocates them. One copy per context that
// has loaded the module; calls in flight at once in one context share it (see
// the declaration in ra.h).
namespace {

static __device__ __align__(256) int g_noalloc_status[RA_NOALLOC_STATUS_WORDS];

// The array's device address in the current context. Looked up on every call
// rather than kept: an address from an earlier call may belong to another
// context (the caller switched contexts, or reset the device since), and the
// lookup is a table search once the module is loaded.
ra_status_t noalloc_status_words(int** out) {
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_status);
  if (err != cudaSuccess) return cuda_failed(err);
  *out = static_cast<int*>(p);
  return RA_SUCCESS;
}

}  // namespace

extern "C" ra_status_t ra_allreduce_bulk_noalloc(const void* const* sendbufs, void* const* recvbufs,
                                                 size_t count, ra_dtype_t dtype, ra_op_t op, int nranks,
                                                 int max_sms, int* chunk_status, void* stream) {
  if (nranks < 1 || nranks > RA_MAX_RANKS || max_sms < 0) return RA_ERR_INVALID_ARG;
  if (nranks > RA_NOALLOC_STATUS_WORDS) return RA_ERR_SCRATCH_LIMIT;
  ra::Args a;
  ra_status_t st = prepare(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS) return st;
  if (count == 0) return RA_SUCCESS;
  if (!a.vec_ok) return RA_ERR_UNSUPPORTED;
  // everything that can fail short of an enqueue failing happens before the first enqueue
  BulkLaunch p;
  st = plan_bulk(a, dtype, op, max_sms, &p);
  if (st != RA_SUCCESS) return st;
  int* words = nullptr;
  st = noalloc_status_words(&words);
  if (st != RA_SUCCESS) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)nranks * sizeof(int);
  cudaError_t err = cudaMemsetAsync(words, 0, bytes, s);
  if (err != cudaSuccess) return cuda_failed(err);
  st = launch_bulk(p, dtype, op, words, /*status_stride=*/1, /*withhold_chunk=*/-1, stream);
  if (st != RA_SUCCESS) return st;
  if (chunk_status != nullptr) {
    err = cudaMemcpyAsync(chunk_status, words, bytes, cudaMemcpyDefault, s);
    if (err != cudaSuccess) return cuda_failed(err);
  }
  return RA_SUCCESS;
}
