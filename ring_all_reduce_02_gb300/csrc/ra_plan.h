// Chunk-schedule planner arithmetic, shared by the host planner (grid sizing,
// introspection) and the kernels (each CTA derives its chunk and vector range).
//
// Chunk c of a count-element buffer over n ranks is [c*count/n, (c+1)*count/n)
// with floor division (tirogla.com "Ring all-reduce", section "Code"). The
// library accepts count < 2^57, so c*count (c <= 64) never leaves 63 bits.
//
// Within a chunk, elements whose byte address lies on the common 16-byte grid
// of all buffers are moved as 16-byte vectors: the grid is {head + k*V}, with
// V = 16 / elem_size and head the first element index whose address is 16-byte
// aligned. A chunk's vector part is the largest run of whole vectors inside it;
// the at most 2(V-1) elements at its two ends take the per-element path.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

constexpr int kVecBytes = 16;

RA_HD uint64_t chunk_begin(int c, int n, uint64_t count) {
  return ((uint64_t)c * count) / (uint64_t)n;
}

// [vb, ve): whole 16-byte vectors of the grid {head + k*V} inside [b0, b1).
// vb == ve when the chunk holds no whole vector.
RA_HD void vec_range(uint64_t b0, uint64_t b1, uint64_t head, uint64_t v, uint64_t* vb,
                     uint64_t* ve) {
  const uint64_t lo = b0 <= head ? head : head + ((b0 - head + v - 1) / v) * v;
  if (b1 < lo + v) {
    *vb = *ve = b0;
    return;
  }
  *vb = lo;
  *ve = head + ((b1 - head) / v) * v;
}

}  // namespace ra
