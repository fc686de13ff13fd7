// The C ABI of libra.so: argument checks, the alias rules, the chunk-schedule
// planner (grid sizing and vector-path selection) and dispatch to the fused
// kernels. Declarations and the contract of every entry point: include/ra.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ra.h"
#include "ra_kernels.cuh"

namespace ra {
cudaError_t launch_f32(int kind, int op, const Args& a, dim3 grid, cudaStream_t s);
cudaError_t launch_f16(int kind, int op, const Args& a, dim3 grid, cudaStream_t s);
cudaError_t launch_bf16(int kind, int op, const Args& a, dim3 grid, cudaStream_t s);
cudaError_t launch_i32(int kind, int op, const Args& a, dim3 grid, cudaStream_t s);
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

struct Range {
  uintptr_t lo = 0, hi = 0;  // [lo, hi) in bytes; empty if lo == hi
};
bool overlaps(const Range& a, const Range& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
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

  // 16-byte phases: the N-way side must share one phase for the vector path
  // (AR: all sources and destinations; RS: the sources; AG: the destinations).
  const Range* wide = kind == ra::KIND_ALLGATHER ? recv : send;
  const unsigned phase = (unsigned)(wide[0].lo % ra::kVecBytes);
  bool same = true;
  for (int r = 0; r < nranks; ++r) {
    same = same && (wide[r].lo % ra::kVecBytes) == phase;
    if (kind == ra::KIND_ALLREDUCE) same = same && (recv[r].lo % ra::kVecBytes) == phase;
  }
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
  a->head = (int)(((ra::kVecBytes - phase) % ra::kVecBytes) / (unsigned)es);
  a->vec_ok = same ? 1 : 0;
  a->inv_n = 1.0f / (float)nranks;
  a->step = 0;
  return RA_SUCCESS;
}

// Grid: blockIdx.y = chunk (or rank, for the ring steps); blockIdx.x = CTAs
// sharing it, enough to cover its vectors (per_thread of them per thread) but
// no more than one resident wave in total.
ra_status_t grid_for(const ra::Args& a, int dtype, int per_thread, dim3* grid) {
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    return RA_ERR_CUDA;
  }
  const int es = elem_size(dtype);
  const uint64_t v = (uint64_t)(ra::kVecBytes / es);
  const uint64_t n = (uint64_t)a.nranks;
  const uint64_t per_chunk = (a.count + n - 1) / n;
  const uint64_t work = a.vec_ok ? (per_chunk / v + 1) : per_chunk;  // vectors, or elements
  const uint64_t per_cta = a.vec_ok ? (uint64_t)ra::kThreads * per_thread : (uint64_t)ra::kThreads;
  uint64_t gx = (work + per_cta - 1) / per_cta;
  const uint64_t cap = (uint64_t)sms * ra::kMinBlocks / n;
  if (gx > cap) gx = cap;
  if (gx < 1) gx = 1;
  *grid = dim3((unsigned)gx, (unsigned)a.nranks);
  return RA_SUCCESS;
}

ra_status_t launch(int kind, int dtype, int op, const ra::Args& a, dim3 grid, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  switch (dtype) {
    case RA_FLOAT32: err = ra::launch_f32(kind, op, a, grid, s); break;
    case RA_FLOAT16: err = ra::launch_f16(kind, op, a, grid, s); break;
    case RA_BFLOAT16: err = ra::launch_bf16(kind, op, a, grid, s); break;
    case RA_INT32: err = ra::launch_i32(kind, op, a, grid, s); break;
    default: return RA_ERR_UNSUPPORTED;
  }
  if (err != cudaSuccess) {
    g_last_cuda_error = (int)err;
    return RA_ERR_CUDA;
  }
  return RA_SUCCESS;
}

ra_status_t run(int kind, const void* const* sendbufs, void* const* recvbufs, size_t count,
                ra_dtype_t dtype, ra_op_t op, int nranks, void* stream) {
  ra::Args a;
  if (kind == ra::KIND_ALLGATHER) op = RA_SUM;  // no reduction; any valid op is accepted
  ra_status_t st = prepare(kind, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS || count == 0) return st;
  dim3 grid;
  st = grid_for(a, dtype, ra::kUnroll, &grid);
  if (st != RA_SUCCESS) return st;
  return launch(kind, dtype, op, a, grid, stream);
}

ra_status_t run_ringsteps(const void* const* sendbufs, void* const* recvbufs, size_t count,
                          ra_dtype_t dtype, ra_op_t op, int nranks, int nsteps, void* stream) {
  ra::Args a;
  ra_status_t st = prepare(ra::KIND_ALLREDUCE, sendbufs, recvbufs, count, dtype, op, nranks, &a);
  if (st != RA_SUCCESS || count == 0) return st;
  const int total = 2 * (nranks - 1);
  if (nsteps < 0 || nsteps > total) nsteps = total;
  dim3 grid;
  if (nranks == 1) {  // no ring steps: the result is the (avg-scaled) copy
    st = grid_for(a, dtype, ra::kUnroll, &grid);
    return st != RA_SUCCESS ? st : launch(ra::KIND_ALLREDUCE, dtype, op, a, grid, stream);
  }
  st = grid_for(a, dtype, 1, &grid);
  if (st != RA_SUCCESS) return st;
  for (int k = 0; k < nsteps; ++k) {
    const bool rs = k < nranks - 1;
    a.step = rs ? k : k - (nranks - 1);
    st = launch(rs ? ra::KIND_RING_RS_STEP : ra::KIND_RING_AG_STEP, dtype, op, a, grid, stream);
    if (st != RA_SUCCESS) return st;
  }
  return RA_SUCCESS;
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

ra_status_t ra_plan_chunk(size_t count, int nranks, int c, int elem_size_bytes, int phase_bytes,
                          size_t* begin, size_t* end, size_t* vec_begin, size_t* vec_end) {
  if (elem_size_bytes != 2 && elem_size_bytes != 4) return RA_ERR_INVALID_ARG;
  if (phase_bytes < 0 || phase_bytes >= ra::kVecBytes || phase_bytes % elem_size_bytes) return RA_ERR_INVALID_ARG;
  if (vec_begin == nullptr || vec_end == nullptr) return RA_ERR_INVALID_ARG;
  const ra_status_t st = ra_chunk_range(count, nranks, c, begin, end);
  if (st != RA_SUCCESS) return st;
  const uint64_t head = (uint64_t)((ra::kVecBytes - phase_bytes) % ra::kVecBytes) / elem_size_bytes;
  uint64_t vb, ve;
  ra::vec_range(*begin, *end, head, (uint64_t)(ra::kVecBytes / elem_size_bytes), &vb, &ve);
  *vec_begin = (size_t)vb;
  *vec_end = (size_t)ve;
  return RA_SUCCESS;
}

const char* ra_status_string(ra_status_t status) {
  switch (status) {
    case RA_SUCCESS: return "success";
    case RA_ERR_INVALID_ARG: return "invalid argument";
    case RA_ERR_UNSUPPORTED: return "unsupported dtype/op";
    case RA_ERR_ALIAS: return "buffers overlap outside the in-place layout";
    case RA_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

int ra_last_cuda_error(void) { return g_last_cuda_error; }

}  // extern "C"
