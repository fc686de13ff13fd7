// Element and vector reduction ops of one ring hop, on sm_103a.
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
//   min / max  IEEE 754-2019 minimum / maximum: a NaN operand gives NaN
//              (the canonical one on the vector path), -0 < +0; otherwise
//              the result is one of the operands, bits unchanged.
// avg = sum over the ring, then one multiply by inv_n = 1.0f/N (fp32) rounded
// to the dtype (bitfern.com "AllReduce Explained": gradients summed, then
// divided by the number of workers); int32 avg = wrapped sum / N, truncated.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ra_plan.h"

namespace ra {

enum Dtype { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2, DT_I32 = 3 };
enum Op { OP_SUM = 0, OP_AVG = 1, OP_MIN = 2, OP_MAX = 3, OP_PROD = 4 };

template <int DT>
struct Elem {
  static constexpr int kSize = (DT == DT_F16 || DT == DT_BF16) ? 2 : 4;
  static constexpr int kPerVec = kVecBytes / kSize;  // elements per vector
};

// ---- scalar helpers on storage bits (held in the low bits of a uint32) ----
// IEEE 754-2019 minimum / maximum: a NaN operand gives NaN, -0 < +0. The PTX
// min.NaN / max.NaN instructions compute exactly this on sm_103a (checked on
// GB300: max(-0, +0) = +0 and min = -0 in either order, NaN in either operand
// gives the canonical NaN, subnormals kept), one instruction per hop.
__device__ __forceinline__ float fminimum(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float fmaximum(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
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

// The same minimum / maximum on the two 16-bit lanes of a word at once
// (min.NaN / max.NaN on f16x2 or bf16x2: the same semantics per lane).
template <int DT, bool IS_MAX>
__device__ __forceinline__ uint32_t minmax16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (DT == DT_F16) {
    if constexpr (IS_MAX) asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  } else {
    if constexpr (IS_MAX) asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    else asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  }
  return r;
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

// ---- word-level ops (one fp32/int32 lane, or two fp16/bf16 lanes) ----------
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
    return minmax16x2<DT, OP == OP_MAX>(a, b);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t word_avg(uint32_t v, float inv_n, int n) {
  if constexpr (DT == DT_F32 || DT == DT_I32) {
    return elem_avg<DT>(v, inv_n, n);
  } else if constexpr (DT == DT_F16) {
    // two lanes: widen the pair, two fp32 multiplies, one paired RNE conversion
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    const __half2 h = __float22half2_rn(make_float2(__fmul_rn(f.x, inv_n), __fmul_rn(f.y, inv_n)));
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
    const __nv_bfloat162 h = __float22bfloat162_rn(make_float2(__fmul_rn(f.x, inv_n), __fmul_rn(f.y, inv_n)));
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// A vector of W 32-bit words (16 or 32 bytes): fp32/int32 lanes are words,
// fp16/bf16 lanes are half-words (lane l in word l/2, low half first). Vec is
// the width of the fused kernels: kVecBytes (16, or 32 with the sm_100+
// 256-bit accesses).
template <int W>
struct __align__(16) VecT {
  uint32_t w[W];
};
constexpr int kVecWords = kVecBytes / 4;
using Vec = VecT<kVecWords>;

template <int DT, int OP, int W>
__device__ __forceinline__ VecT<W> vec_hop(const VecT<W>& a, const VecT<W>& b) {
  VecT<W> r;
#pragma unroll
  for (int k = 0; k < W; ++k) r.w[k] = word_hop<DT, OP>(a.w[k], b.w[k]);
  return r;
}
template <int DT, int W>
__device__ __forceinline__ VecT<W> vec_avg(const VecT<W>& v, float inv_n, int n) {
  VecT<W> r;
#pragma unroll
  for (int k = 0; k < W; ++k) r.w[k] = word_avg<DT>(v.w[k], inv_n, n);
  return r;
}

// lane l of a vector, as storage bits
template <int DT, int W>
__device__ __forceinline__ uint32_t vec_lane(const VecT<W>& v, int l) {
  if constexpr (Elem<DT>::kSize == 4) {
    return v.w[l];
  } else {
    return (v.w[l >> 1] >> ((l & 1) * 16)) & 0xffffu;
  }
}

// ---- fp32 accumulation for fp16/bf16 buffers ----------------------------------
// The partial of every lane stays in fp32 from hop to hop; it is rounded to
// the dtype once, after the avg multiply (tirogla.com "Ring all-reduce",
// "Implementation notes": accumulate bf16 in fp32 at large N).
constexpr int kVecHalves = kVecBytes / 2;
struct VecF {
  float f[kVecHalves];
};
template <int DT>
__device__ __forceinline__ VecF vec_widen(const Vec& v) {
  VecF r;
#pragma unroll
  for (int k = 0; k < kVecWords; ++k) {
    r.f[2 * k] = widen16<DT>(v.w[k] & 0xffffu);
    r.f[2 * k + 1] = widen16<DT>(v.w[k] >> 16);
  }
  return r;
}
template <int DT>
__device__ __forceinline__ Vec vec_narrow(const VecF& a) {
  Vec r;
#pragma unroll
  for (int k = 0; k < kVecWords; ++k) {
    const float2 p = make_float2(a.f[2 * k], a.f[2 * k + 1]);
    if constexpr (DT == DT_F16) {
      const __half2 h = __float22half2_rn(p);
      r.w[k] = *reinterpret_cast<const uint32_t*>(&h);
    } else {
      const __nv_bfloat162 h = __float22bfloat162_rn(p);
      r.w[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
  }
  return r;
}
template <int OP>
__device__ __forceinline__ float f32_hop(float a, float b) {
  if constexpr (OP == OP_SUM || OP == OP_AVG) return __fadd_rn(a, b);
  else if constexpr (OP == OP_PROD) return __fmul_rn(a, b);
  else if constexpr (OP == OP_MIN) return fminimum(a, b);
  else return fmaximum(a, b);
}
template <int OP>
__device__ __forceinline__ VecF vecf_hop(const VecF& a, const VecF& b) {
  VecF r;
#pragma unroll
  for (int k = 0; k < kVecHalves; ++k) r.f[k] = f32_hop<OP>(a.f[k], b.f[k]);
  return r;
}

// ---- global memory ----------------------------------------------------------
// Streaming (evict-first) vector loads and stores: every byte is touched once.
// RA_LD_MODE / RA_ST_MODE select other cache hints for tuning sweeps
// (0 = evict-first streaming, 1 = default caching).
#ifndef RA_LD_MODE
#define RA_LD_MODE 0
#endif
#ifndef RA_ST_MODE
#define RA_ST_MODE 0
#endif
#if RA_LD_MODE == 0
#define RA_LD_HINT ".cs"
#else
#define RA_LD_HINT ""
#endif
#if RA_ST_MODE == 0
#define RA_ST_HINT ".cs"
#else
#define RA_ST_HINT ""
#endif

template <int W>
__device__ __forceinline__ VecT<W> ld_vec_w(const void* p) {
  static_assert(W == 4 || W == 8, "16- or 32-byte vectors");
  VecT<W> v;
  if constexpr (W == 4) {
    asm volatile("ld.global" RA_LD_HINT ".v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
  } else {
    asm volatile("ld.global" RA_LD_HINT ".v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                   "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
  }
  return v;
}
__device__ __forceinline__ Vec ld_vec(const void* p) { return ld_vec_w<kVecWords>(p); }
template <int W>
__device__ __forceinline__ void st_vec(void* p, const VecT<W>& v) {
  static_assert(W == 4 || W == 8, "16- or 32-byte vectors");
  if constexpr (W == 4) {
    asm volatile("st.global" RA_ST_HINT ".v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
  } else {
    asm volatile("st.global" RA_ST_HINT ".v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
  }
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

// ---- compact buffers off the vector grid -----------------------------------
// A compact RS output or AG input whose address phase differs from the vector
// grid's is moved in g-byte units, g the largest power of two up to 16 that
// divides its address. With consecutive threads on consecutive units every
// warp access covers whole sectors; each lane storing its own vector in
// 2-byte pieces would scatter them over 32 sectors per instruction.
__device__ __forceinline__ uint32_t unit_bytes(const void* p) {
  const uint32_t a = (uint32_t)reinterpret_cast<uintptr_t>(p) & 15u;
  return a == 0 ? 16u : (a & (0u - a));
}
// `bytes` (a multiple of 16) from 16-byte-aligned shared memory s to global g;
// thread t of nt takes units t, t + nt, ...
__device__ __forceinline__ void copy_out_units(char* g, const char* s, uint32_t bytes, uint32_t t, uint32_t nt) {
  const uint32_t u = unit_bytes(g);
  if (u == 16) {
    for (uint32_t o = t * 16u; o < bytes; o += nt * 16u)
      __stcs(reinterpret_cast<uint4*>(g + o), *reinterpret_cast<const uint4*>(s + o));
  } else if (u == 8) {
    for (uint32_t o = t * 8u; o < bytes; o += nt * 8u)
      __stcs(reinterpret_cast<uint2*>(g + o), *reinterpret_cast<const uint2*>(s + o));
  } else if (u == 4) {
    for (uint32_t o = t * 4u; o < bytes; o += nt * 4u)
      __stcs(reinterpret_cast<unsigned int*>(g + o), *reinterpret_cast<const unsigned int*>(s + o));
  } else {
    for (uint32_t o = t * 2u; o < bytes; o += nt * 2u)
      __stcs(reinterpret_cast<unsigned short*>(g + o), *reinterpret_cast<const unsigned short*>(s + o));
  }
}
template <uint32_t G> struct UnitT;
template <> struct UnitT<16> { using T = uint4; };
template <> struct UnitT<8> { using T = uint2; };
template <> struct UnitT<4> { using T = unsigned int; };
template <> struct UnitT<2> { using T = unsigned short; };
// One thread's vector to global p off the vector grid: 4-byte units when p's
// address allows (the reduce-scatter's per-lane store), else 2-byte ones. The
// planner sends calls with 2-byte offsets to the cooperative OFFGRID kernel,
// so the 2-byte branch is a fallback that keeps any launch correct.
template <int W>
__device__ __forceinline__ void st_vec_units(char* p, const VecT<W>& v) {
  if ((reinterpret_cast<uintptr_t>(p) & 3u) == 0) {
#pragma unroll
    for (int k = 0; k < W; ++k) __stcs(reinterpret_cast<unsigned int*>(p) + k, v.w[k]);
  } else {
#pragma unroll
    for (int k = 0; k < W; ++k) {
      __stcs(reinterpret_cast<unsigned short*>(p) + 2 * k, (unsigned short)(v.w[k] & 0xffffu));
      __stcs(reinterpret_cast<unsigned short*>(p) + 2 * k + 1, (unsigned short)(v.w[k] >> 16));
    }
  }
}

}  // namespace ra
