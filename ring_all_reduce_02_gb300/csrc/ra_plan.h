// Chunk-schedule planner arithmetic, shared by the host planner (grid sizing,
// introspection) and the kernels (each CTA derives its chunk and vector range).
//
// Chunk c of a count-element buffer over n ranks is [c*count/n, (c+1)*count/n)
// with floor division (tirogla.com "Ring all-reduce", section "Code"). The
// library accepts count < 2^57, so c*count (c <= 64) never leaves 63 bits.
//
// Within a chunk, elements whose byte address lies on the common kVecBytes grid
// of all buffers are moved as whole vectors: the grid is {head + k*V}, with
// V = kVecBytes / elem_size and head the first element index whose address is
// aligned to the common line alignment (16..512 bytes, see vec_range). A chunk's
// vector part runs from the first line-aligned element to its last whole vector;
// the elements before and after it take the per-element path.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

// Bytes per vector access: 32 (the 256-bit ld/st.global.v8.b32 of sm_100 and
// later; on GB300 a stream of them reads HBM about 5% faster than 16-byte
// accesses) or 16 (ld/st.global.v4.b32). Build-time choice.
#ifndef RA_VEC_BYTES
#define RA_VEC_BYTES 32
#endif
constexpr int kVecBytes = RA_VEC_BYTES;

RA_HD uint64_t chunk_begin(int c, int n, uint64_t count) {
  return ((uint64_t)c * count) / (uint64_t)n;
}

// [vb, ve): whole vectors of the chunk [b0, b1), starting at the first element
// of the alignment grid {head + k*align} at or after b0 (align is a multiple of
// v, so the start is also on the vector grid) and ending at the last whole
// vector. Starting on a line-aligned boundary keeps every warp's contiguous
// access inside whole cache lines and DRAM sectors. vb == ve (== b0) when no
// whole vector fits.
RA_HD void vec_range(uint64_t b0, uint64_t b1, uint64_t head, uint64_t align, uint64_t v, uint64_t* vb,
                     uint64_t* ve) {
  const uint64_t lo = b0 <= head ? head : head + ((b0 - head + align - 1) / align) * align;
  if (b1 < lo + v) {
    *vb = *ve = b0;
    return;
  }
  *vb = lo;
  *ve = lo + ((b1 - lo) / v) * v;
}

// Largest alignment (bytes) the vector grid is laid on: every buffer's address
// shares its phase modulo this.
constexpr int kLineAlignMax = 512;

}  // namespace ra
