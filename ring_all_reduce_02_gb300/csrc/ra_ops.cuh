// Element and 16-byte-vector reduction ops of one ring hop, on sm_103a.
//
// One hop combines the partial arriving from the left neighbour with the local
// value and rounds the result to the buffer dtype (every hop of the ring is
// rounded: the message between ranks is stored in the buffer dtype):
//   fp32       fp32 add / multiply (round to nearest even, no FMA contraction);
//   fp16/bf16  both operands widened to fp32 (exact), one fp32 add / multiply,
//              one conversion back with round to nearest even. fp32 has at
//              least 2p+2 significand bits for p = 11 (fp16) and p = 8 (bf16),
//              so this equals the correctly rounded fp16/bf16 operation;
//   int32      add / multiply modulo 2^32;
//   min / max  IEEE 754-2019 minimum / maximum: a NaN operand gives NaN,
//              -0 < +0; the result is one of the operands, bits unchanged.
// avg = sum over the ring, then one multiply by inv_n = 1.0f/N (fp32) rounded
// to the dtype (bitfern.com "AllReduce Explained": gradients summed, then
// divided by the number of workers); int32 avg = wrapped sum / N, truncated.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace ra {

enum Dtype { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_I32 = 3 };
enum Op { OP_SUM = 0, OP_AVG = 1, OP_MIN = 2, OP_MAX = 3, OP_PROD = 4 };

template <int DT>
struct Elem {
  static constexpr int kSize = (DT == DT_F16 || DT == DT_BF16) ? 2 : 4;
  static constexpr int kPerVec = 16 / kSize;  // elements per 16-byte vector
};

// ---- scalar helpers on storage bits (held in the low bits of a uint32) ----
__device__ __forceinline__ float fminimum(float a, float b) {
  if (a != a) return a;
  if (b != b) return b;
  if (a < b) return a;
  if (b < a) return b;
  return __int_as_float(__float_as_int(a) | __float_as_int(b));  // equal: -0 wins
}
__device__ __forceinline__ float fmaximum(float a, float b) {
  if (a != a) return a;
  if (b != b) return b;
  if (a > b) return a;
  if (b > a) return b;
  return __int_as_float(__float_as_int(a) & __float_as_int(b));  // equal: +0 wins
}

template <int DT>
__device__ __forceinline__ float widen16(uint32_t h) {
  if constexpr (DT == DT_F16) {
    return __half2float(__ushort_as_half((unsigned short)h));
  } else {
    return __uint_as_float(h << 16);  // bf16 is the top half of an fp32
  }
}
template <int DT>
__device__ __forceinline__ uint32_t round16(float f) {
  if constexpr (DT == DT_F16) {
    return __half_as_ushort(__float2half_rn(f));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
  }
}

template <int DT, bool IS_MAX>
__device__ __forceinline__ uint32_t minmax16(uint32_t a, uint32_t b) {
  const float fa = widen16<DT>(a), fb = widen16<DT>(b);
  if (fa != fa) return a;
  if (fb != fb) return b;
  if (IS_MAX ? (fa > fb) : (fa < fb)) return a;
  if (IS_MAX ? (fb > fa) : (fb < fa)) return b;
  return IS_MAX ? (a & b) : (a | b);  // equal values: only the sign of zero can differ
}

// One hop on one element: `partial` (incoming) on the left, `local` on the right.
template <int DT, int OP>
__device__ __forceinline__ uint32_t elem_hop(uint32_t partial, uint32_t local) {
  if constexpr (DT == DT_F32) {
    const float a = __uint_as_float(partial), b = __uint_as_float(local);
    float r;
    if constexpr (OP == OP_SUM || OP == OP_AVG) r = __fadd_rn(a, b);
    else if constexpr (OP == OP_PROD) r = __fmul_rn(a, b);
    else if constexpr (OP == OP_MIN) r = fminimum(a, b);
    else r = fmaximum(a, b);
    return __float_as_uint(r);
  } else if constexpr (DT == DT_I32) {
    if constexpr (OP == OP_SUM || OP == OP_AVG) return partial + local;
    else if constexpr (OP == OP_PROD) return partial * local;
    else if constexpr (OP == OP_MIN) return (uint32_t)min((int32_t)partial, (int32_t)local);
    else return (uint32_t)max((int32_t)partial, (int32_t)local);
  } else {
    if constexpr (OP == OP_MIN) return minmax16<DT, false>(partial, local);
    else if constexpr (OP == OP_MAX) return minmax16<DT, true>(partial, local);
    else {
      const float a = widen16<DT>(partial), b = widen16<DT>(local);
      return round16<DT>(OP == OP_PROD ? __fmul_rn(a, b) : __fadd_rn(a, b));
    }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t elem_avg(uint32_t v, float inv_n, int n) {
  if constexpr (DT == DT_F32) {
    return __float_as_uint(__fmul_rn(__uint_as_float(v), inv_n));
  } else if constexpr (DT == DT_I32) {
    return (uint32_t)((int32_t)v / n);
  } else {
    return round16<DT>(__fmul_rn(widen16<DT>(v), inv_n));
  }
}

// ---- 16-byte vectors ------------------------------------------------------
template <int DT, int OP>
__device__ __forceinline__ uint32_t word_hop(uint32_t a, uint32_t b) {
  if constexpr (DT == DT_F32 || DT == DT_I32) {
    return elem_hop<DT, OP>(a, b);
  } else if constexpr (OP == OP_SUM || OP == OP_AVG || OP == OP_PROD) {
    // two 16-bit lanes: widen the pair, two fp32 ops, one paired RNE conversion
    if constexpr (DT == DT_F16) {
      const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&a));
      const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&b));
      const float2 r = (OP == OP_PROD) ? make_float2(__fmul_rn(fa.x, fb.x), __fmul_rn(fa.y, fb.y))
                                       : make_float2(__fadd_rn(fa.x, fb.x), __fadd_rn(fa.y, fb.y));
      const __half2 h = __float22half2_rn(r);
      return *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b));
      const float2 r = (OP == OP_PROD) ? make_float2(__fmul_rn(fa.x, fb.x), __fmul_rn(fa.y, fb.y))
                                       : make_float2(__fadd_rn(fa.x, fb.x), __fadd_rn(fa.y, fb.y));
      const __nv_bfloat162 h = __float22bfloat162_rn(r);
      return *reinterpret_cast<const uint32_t*>(&h);
    }
  } else {
    const uint32_t lo = elem_hop<DT, OP>(a & 0xffffu, b & 0xffffu);
    const uint32_t hi = elem_hop<DT, OP>(a >> 16, b >> 16);
    return lo | (hi << 16);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t word_avg(uint32_t v, float inv_n, int n) {
  if constexpr (DT == DT_F32 || DT == DT_I32) {
    return elem_avg<DT>(v, inv_n, n);
  } else {
    return elem_avg<DT>(v & 0xffffu, inv_n, n) | (elem_avg<DT>(v >> 16, inv_n, n) << 16);
  }
}

template <int DT, int OP>
__device__ __forceinline__ uint4 vec_hop(uint4 a, uint4 b) {
  return make_uint4(word_hop<DT, OP>(a.x, b.x), word_hop<DT, OP>(a.y, b.y),
                    word_hop<DT, OP>(a.z, b.z), word_hop<DT, OP>(a.w, b.w));
}
template <int DT>
__device__ __forceinline__ uint4 vec_avg(uint4 v, float inv_n, int n) {
  return make_uint4(word_avg<DT>(v.x, inv_n, n), word_avg<DT>(v.y, inv_n, n),
                    word_avg<DT>(v.z, inv_n, n), word_avg<DT>(v.w, inv_n, n));
}

// lane l of a 16-byte vector, as storage bits
template <int DT>
__device__ __forceinline__ uint32_t vec_lane(const uint4& v, int l) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (Elem<DT>::kSize == 4) {
    return w[l];
  } else {
    return (w[l >> 1] >> ((l & 1) * 16)) & 0xffffu;
  }
}

// ---- global memory ----------------------------------------------------------
// Streaming (evict-first) 16-byte loads and stores: every byte is touched once.
// RA_LD_MODE / RA_ST_MODE select other cache hints for tuning sweeps
// (0 = evict-first streaming, 1 = default caching).
#ifndef RA_LD_MODE
#define RA_LD_MODE 0
#endif
#ifndef RA_ST_MODE
#define RA_ST_MODE 0
#endif
__device__ __forceinline__ uint4 ld_vec(const void* p) {
#if RA_LD_MODE == 0
  return __ldcs(reinterpret_cast<const uint4*>(p));
#else
  return *reinterpret_cast<const uint4*>(p);
#endif
}
__device__ __forceinline__ void st_vec(void* p, uint4 v) {
#if RA_ST_MODE == 0
  __stcs(reinterpret_cast<uint4*>(p), v);
#else
  *reinterpret_cast<uint4*>(p) = v;
#endif
}
template <int DT>
__device__ __forceinline__ uint32_t ld_elem(const void* base, uint64_t i) {
  if constexpr (Elem<DT>::kSize == 4) {
    return __ldcs(reinterpret_cast<const unsigned int*>(base) + i);
  } else {
    return __ldcs(reinterpret_cast<const unsigned short*>(base) + i);
  }
}
template <int DT>
__device__ __forceinline__ void st_elem(void* base, uint64_t i, uint32_t v) {
  if constexpr (Elem<DT>::kSize == 4) {
    __stcs(reinterpret_cast<unsigned int*>(base) + i, v);
  } else {
    __stcs(reinterpret_cast<unsigned short*>(base) + i, (unsigned short)v);
  }
}

}  // namespace ra
