// Stream probes: the HBM read and write rates that the collective kernels are
// measured against. Not part of the collective path; `bench.py --roofs` runs
// them with CUDA events.
//
// Two launch styles for the same 32-byte accesses:
//  - persistent: kPersistPerSm CTAs per SM grid-stride over the buffer, the
//    style of a one-wave kernel;
//  - one-shot: one CTA per 16 KB piece, which it reads or writes and exits,
//    the style of the library's one-trip kernels and of its all-gather.
// The store probes write the same piece to each of n destinations (n = 1: a
// plain store stream; n > 1: the all-gather's write pattern without its reads);
// the copy probes read a piece and write it elsewhere (the 1:1 mix of an
// all-reduce's traffic). The SM-share copy runs on a given number of CTAs, one
// per SM, to show how many bytes a share of the SMs can move.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr int kThreads = 256;
constexpr int kPersistPerSm = 4;
constexpr uint64_t kPiece = 16384;  // bytes per one-shot CTA: 256 threads x 2 x 32 B
constexpr int kMaxBuffers = 64;

struct Dsts {
  char* p[kMaxBuffers];
};

__device__ __forceinline__ void st32(char* p, uint32_t v) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v), "r"(v ^ 1u), "r"(v ^ 2u),
               "r"(v ^ 3u), "r"(v ^ 4u), "r"(v ^ 5u), "r"(v ^ 6u), "r"(v ^ 7u)
               : "memory");
}
__device__ __forceinline__ uint32_t ld32(const char* p) {
  uint32_t a, b, c, d, e, f, g, h;
  asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d), "=r"(e), "=r"(f), "=r"(g), "=r"(h)
               : "l"(p));
  return a ^ b ^ c ^ d ^ e ^ f ^ g ^ h;
}

__global__ void __launch_bounds__(kThreads) store_persistent(const __grid_constant__ Dsts d, int n, uint64_t nvec) {
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += stride) {
    const uint32_t v = 0x9e3779b9u * (uint32_t)i;
    for (int r = 0; r < n; ++r) st32(d.p[r] + i * 32, v);
  }
}

__global__ void __launch_bounds__(kThreads) store_one_shot(const __grid_constant__ Dsts d, int n) {
  const uint64_t i0 = (uint64_t)blockIdx.x * (kPiece / 32) + threadIdx.x, i1 = i0 + kThreads;
  for (int r = 0; r < n; ++r) {
    st32(d.p[r] + i0 * 32, 0x9e3779b9u * (uint32_t)i0);
    st32(d.p[r] + i1 * 32, 0x9e3779b9u * (uint32_t)i1);
  }
}

__global__ void __launch_bounds__(kThreads) load_persistent(const char* src, uint64_t nvec, uint32_t* sink) {
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  uint32_t acc = 0;
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += stride) acc ^= ld32(src + i * 32);
  if (acc == 0x5bd1e995u) *sink = acc;  // keeps the loads alive; the value is irrelevant
}

__global__ void __launch_bounds__(kThreads) load_one_shot(const char* src, uint32_t* sink) {
  const uint64_t i0 = (uint64_t)blockIdx.x * (kPiece / 32) + threadIdx.x;
  const uint32_t acc = ld32(src + i0 * 32) ^ ld32(src + (i0 + kThreads) * 32);
  if (acc == 0x5bd1e995u) *sink = acc;
}

__global__ void __launch_bounds__(kThreads) copy_persistent(const char* src, char* dst, uint64_t nvec) {
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  for (uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += stride) {
    uint32_t a, b, c, d, e, f, g, h;
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d), "=r"(e), "=r"(f), "=r"(g), "=r"(h)
                 : "l"(src + i * 32));
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + i * 32), "r"(a), "r"(b), "r"(c),
                 "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
                 : "memory");
  }
}

__global__ void __launch_bounds__(kThreads) copy_one_shot(const char* src, char* dst) {
  const uint64_t i0 = (uint64_t)blockIdx.x * (kPiece / 32) + threadIdx.x;
  uint32_t v[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[h][0]), "=r"(v[h][1]), "=r"(v[h][2]), "=r"(v[h][3]), "=r"(v[h][4]), "=r"(v[h][5]),
                   "=r"(v[h][6]), "=r"(v[h][7])
                 : "l"(src + (i0 + h * kThreads) * 32));
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + (i0 + h * kThreads) * 32),
                 "r"(v[h][0]), "r"(v[h][1]), "r"(v[h][2]), "r"(v[h][3]), "r"(v[h][4]), "r"(v[h][5]), "r"(v[h][6]),
                 "r"(v[h][7])
                 : "memory");
}

// one CTA of kShareThreads per SM-share slot: CTA b copies bytes [b * slab, (b + 1) * slab)
constexpr int kShareThreads = 1024;
__global__ void __launch_bounds__(kShareThreads) copy_share(const char* src, char* dst, uint64_t slab) {
  const char* s = src + blockIdx.x * slab;
  char* d = dst + blockIdx.x * slab;
  const uint64_t nvec = slab / 32;
  for (uint64_t i = threadIdx.x; i < nvec; i += 4 * kShareThreads) {
    uint32_t v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                   : "=r"(v[u][0]), "=r"(v[u][1]), "=r"(v[u][2]), "=r"(v[u][3]), "=r"(v[u][4]), "=r"(v[u][5]),
                     "=r"(v[u][6]), "=r"(v[u][7])
                   : "l"(s + (i + (uint64_t)u * kShareThreads) * 32));
#pragma unroll
    for (int u = 0; u < 4; ++u)
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d + (i + (uint64_t)u * kShareThreads) * 32),
                   "r"(v[u][0]), "r"(v[u][1]), "r"(v[u][2]), "r"(v[u][3]), "r"(v[u][4]), "r"(v[u][5]), "r"(v[u][6]),
                   "r"(v[u][7])
                   : "memory");
  }
}

// one CTA per 16 KB piece: read it once and write it to each of n destinations
// (the all-gather's traffic: one read, n writes)
__global__ void __launch_bounds__(kThreads) copy_n_one_shot(const char* src, const __grid_constant__ Dsts d, int n) {
  const uint64_t i0 = (uint64_t)blockIdx.x * (kPiece / 32) + threadIdx.x;
  uint32_t v[2][8];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[h][0]), "=r"(v[h][1]), "=r"(v[h][2]), "=r"(v[h][3]), "=r"(v[h][4]), "=r"(v[h][5]),
                   "=r"(v[h][6]), "=r"(v[h][7])
                 : "l"(src + (i0 + h * kThreads) * 32));
  for (int r = 0; r < n; ++r) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d.p[r] + (i0 + h * kThreads) * 32),
                   "r"(v[h][0]), "r"(v[h][1]), "r"(v[h][2]), "r"(v[h][3]), "r"(v[h][4]), "r"(v[h][5]),
                   "r"(v[h][6]), "r"(v[h][7])
                   : "memory");
  }
}

// one CTA per 16 KB piece: read it from each of n sources and write one
// combination of them (the reduce-scatter's traffic: n reads, one write)
struct Srcs {
  const char* p[kMaxBuffers];
};
__global__ void __launch_bounds__(kThreads) read_n_one_shot(const __grid_constant__ Srcs sr, int n, char* dst) {
  const uint64_t i0 = (uint64_t)blockIdx.x * (kPiece / 32) + threadIdx.x;
  uint32_t acc[2][8] = {};
  for (int r = 0; r < n; ++r) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[8];
      asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                   : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                   : "l"(sr.p[r] + (i0 + h * kThreads) * 32));
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[h][k] ^= v[k];
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + (i0 + h * kThreads) * 32),
                 "r"(acc[h][0]), "r"(acc[h][1]), "r"(acc[h][2]), "r"(acc[h][3]), "r"(acc[h][4]), "r"(acc[h][5]),
                 "r"(acc[h][6]), "r"(acc[h][7])
                 : "memory");
}

int persistent_grid() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n * kPersistPerSm;
}

}  // namespace

extern "C" {

// Writes `bytes` (a nonzero multiple of 16 KB) to each of the n (1..64) device
// buffers dst[0..n). one_shot: 0 persistent CTAs, 1 one CTA per 16 KB piece.
// Returns a cudaError_t (0 on success).
int rp_store(int one_shot, void* const* dst, int n, size_t bytes, void* stream) {
  if (dst == nullptr || n < 1 || n > kMaxBuffers || bytes == 0 || bytes % kPiece) return (int)cudaErrorInvalidValue;
  Dsts d{};
  for (int r = 0; r < n; ++r) {
    if (dst[r] == nullptr) return (int)cudaErrorInvalidValue;
    d.p[r] = static_cast<char*>(dst[r]);
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (one_shot) {
    const uint64_t pieces = bytes / kPiece;
    if (pieces > 0x7fffffffull) return (int)cudaErrorInvalidValue;
    store_one_shot<<<(unsigned)pieces, kThreads, 0, s>>>(d, n);
  } else {
    const int grid = persistent_grid();
    if (grid <= 0) return (int)cudaErrorUnknown;
    store_persistent<<<grid, kThreads, 0, s>>>(d, n, bytes / 32);
  }
  return (int)cudaGetLastError();
}

// Reads `bytes` (a nonzero multiple of 16 KB) of the device buffer src; sink is
// one device word the kernels may write. Returns a cudaError_t.
int rp_load(int one_shot, const void* src, size_t bytes, void* sink, void* stream) {
  if (src == nullptr || sink == nullptr || bytes == 0 || bytes % kPiece) return (int)cudaErrorInvalidValue;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* p = static_cast<const char*>(src);
  uint32_t* k = static_cast<uint32_t*>(sink);
  if (one_shot) {
    const uint64_t pieces = bytes / kPiece;
    if (pieces > 0x7fffffffull) return (int)cudaErrorInvalidValue;
    load_one_shot<<<(unsigned)pieces, kThreads, 0, s>>>(p, k);
  } else {
    const int grid = persistent_grid();
    if (grid <= 0) return (int)cudaErrorUnknown;
    load_persistent<<<grid, kThreads, 0, s>>>(p, bytes / 32, k);
  }
  return (int)cudaGetLastError();
}

// Copies `bytes` (a nonzero multiple of 16 KB) from device buffer src to dst (not
// overlapping): the 1:1 mix of reads and writes. Returns a cudaError_t.
int rp_copy(int one_shot, const void* src, void* dst, size_t bytes, void* stream) {
  if (src == nullptr || dst == nullptr || bytes == 0 || bytes % kPiece) return (int)cudaErrorInvalidValue;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* p = static_cast<const char*>(src);
  char* q = static_cast<char*>(dst);
  if (one_shot) {
    const uint64_t pieces = bytes / kPiece;
    if (pieces > 0x7fffffffull) return (int)cudaErrorInvalidValue;
    copy_one_shot<<<(unsigned)pieces, kThreads, 0, s>>>(p, q);
  } else {
    const int grid = persistent_grid();
    if (grid <= 0) return (int)cudaErrorUnknown;
    copy_persistent<<<grid, kThreads, 0, s>>>(p, q, bytes / 32);
  }
  return (int)cudaGetLastError();
}

// Reads `bytes` (a nonzero multiple of 16 KB) of src once and writes them to
// each of the n (1..64) device buffers dst[0..n), one CTA per 16 KB piece: the
// traffic mix of an all-gather. Returns a cudaError_t.
int rp_copy_n(const void* src, void* const* dst, int n, size_t bytes, void* stream) {
  if (src == nullptr || dst == nullptr || n < 1 || n > kMaxBuffers || bytes == 0 || bytes % kPiece)
    return (int)cudaErrorInvalidValue;
  Dsts d{};
  for (int r = 0; r < n; ++r) {
    if (dst[r] == nullptr) return (int)cudaErrorInvalidValue;
    d.p[r] = static_cast<char*>(dst[r]);
  }
  const uint64_t pieces = bytes / kPiece;
  if (pieces > 0x7fffffffull) return (int)cudaErrorInvalidValue;
  copy_n_one_shot<<<(unsigned)pieces, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const char*>(src), d, n);
  return (int)cudaGetLastError();
}

// Reads `bytes` (a nonzero multiple of 16 KB) from each of the n (1..64)
// device buffers src[0..n) and writes one combination of them to dst, one CTA
// per 16 KB piece: the traffic mix of a reduce-scatter. Returns a cudaError_t.
int rp_read_n(const void* const* src, int n, void* dst, size_t bytes, void* stream) {
  if (src == nullptr || dst == nullptr || n < 1 || n > kMaxBuffers || bytes == 0 || bytes % kPiece)
    return (int)cudaErrorInvalidValue;
  Srcs sr{};
  for (int r = 0; r < n; ++r) {
    if (src[r] == nullptr) return (int)cudaErrorInvalidValue;
    sr.p[r] = static_cast<const char*>(src[r]);
  }
  const uint64_t pieces = bytes / kPiece;
  if (pieces > 0x7fffffffull) return (int)cudaErrorInvalidValue;
  read_n_one_shot<<<(unsigned)pieces, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(sr, n, static_cast<char*>(dst));
  return (int)cudaGetLastError();
}

// Copies `bytes` from src to dst on `ctas` CTAs of 1024 threads (one per SM
// while ctas <= the SM count): the copy rate an SM share reaches. bytes must be
// a nonzero multiple of ctas * 128 KB. Returns a cudaError_t.
int rp_copy_sms(const void* src, void* dst, size_t bytes, int ctas, void* stream) {
  if (src == nullptr || dst == nullptr || ctas < 1 || bytes == 0 || bytes % ((size_t)ctas * 4 * kShareThreads * 32))
    return (int)cudaErrorInvalidValue;
  copy_share<<<ctas, kShareThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const char*>(src), static_cast<char*>(dst), bytes / (size_t)ctas);
  return (int)cudaGetLastError();
}

}  // extern "C"
