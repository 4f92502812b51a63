// device.cuh -- device primitives shared by the relay kernels (passes.cu, chain_kernel.cu): the
// loads and stores with the cache hints each kernel needs, the payload traits (fp32, bf16,
// int32: widen, add, scale, round to nearest-even, narrow) and the funnel shift that
// realigns a 16-byte vector out of the two aligned blocks it straddles.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "program.h"

namespace relay {
namespace {

// ---------------------------------------------------------------- memory access --

// Loads. The per-pass kernels read only what earlier launches wrote, so they use the
// non-coherent path without allocating in L1. The fused small-call kernel reads, after a
// grid barrier, what other CTAs of the same launch wrote: it loads through L2 only
// (.cg), which is coherent across SMs.
template <bool COH>
struct Mem;
template <>
struct Mem<false> {
  static __device__ __forceinline__ uint4 v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
  }
  static __device__ __forceinline__ uint32_t u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
  }
  static __device__ __forceinline__ uint16_t u16(const void* p) {
    uint16_t r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
  }
};
template <>
struct Mem<true> {
  static __device__ __forceinline__ uint4 v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
  }
  static __device__ __forceinline__ uint32_t u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
  }
  static __device__ __forceinline__ uint16_t u16(const void* p) {
    uint16_t r;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
  }
};
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) { return Mem<false>::v4(p); }
// 16-byte stores are streaming (.cs, evict first): no pass re-reads its own output, and
// on GB300 this measured 0.4-2.7% faster than default stores with one CTA per tile.
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// Default-policy 16-byte store, for data the storing CTA reads back (chained launch).
__device__ __forceinline__ void st_v4_keep(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_u32(void* p, uint32_t v) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_u16(void* p, uint16_t v) {
  asm volatile("st.global.u16 [%0], %1;" ::"l"(p), "h"(v) : "memory");
}
// Invalidate the 128-byte L2 line at p (128-byte aligned, device memory) without writing
// it back: for dead data only, whose bytes are unspecified afterwards.
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(__cvta_generic_to_global(p)) : "memory");
}

// ------------------------------------------------------------- payload traits --
// bf16 is the upper half of a binary32, so widening is a shift; narrowing rounds to
// nearest-even in one cvt instruction (two lanes at a time).

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

struct TF32 {
  static constexpr int kE = 4, kLanes = 4;
  using Acc = float;
  static __device__ __forceinline__ void unpack(uint4 v, float* a) {
    a[0] = __uint_as_float(v.x); a[1] = __uint_as_float(v.y);
    a[2] = __uint_as_float(v.z); a[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* a) {
    return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                      __float_as_uint(a[3]));
  }
  static __device__ __forceinline__ float add(float x, float y) { return __fadd_rn(x, y); }
  static __device__ __forceinline__ float scale(float x, float s) { return __fmul_rn(x, s); }
  template <bool COH>
  static __device__ __forceinline__ float load1(const void* p) {
    return __uint_as_float(Mem<COH>::u32(p));
  }
  static __device__ __forceinline__ void store1(void* p, float v) { st_u32(p, __float_as_uint(v)); }
};

struct TBF16 {
  static constexpr int kE = 2, kLanes = 8;
  using Acc = float;
  static __device__ __forceinline__ void unpack(uint4 v, float* a) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a[2 * i] = __uint_as_float(w[i] << 16);
      a[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* a) {
    return make_uint4(bf16x2_rn(a[0], a[1]), bf16x2_rn(a[2], a[3]), bf16x2_rn(a[4], a[5]),
                      bf16x2_rn(a[6], a[7]));
  }
  static __device__ __forceinline__ float add(float x, float y) { return __fadd_rn(x, y); }
  static __device__ __forceinline__ float scale(float x, float s) { return __fmul_rn(x, s); }
  template <bool COH>
  static __device__ __forceinline__ float load1(const void* p) {
    return __uint_as_float((uint32_t)Mem<COH>::u16(p) << 16);
  }
  static __device__ __forceinline__ void store1(void* p, float v) {
    st_u16(p, (uint16_t)(bf16x2_rn(v, 0.0f) & 0xffffu));
  }
};

struct TI32 {
  static constexpr int kE = 4, kLanes = 4;
  using Acc = uint32_t;  // two's-complement sums wrap modulo 2^32
  static __device__ __forceinline__ void unpack(uint4 v, uint32_t* a) {
    a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
  }
  static __device__ __forceinline__ uint4 pack(const uint32_t* a) {
    return make_uint4(a[0], a[1], a[2], a[3]);
  }
  static __device__ __forceinline__ uint32_t add(uint32_t x, uint32_t y) { return x + y; }
  static __device__ __forceinline__ uint32_t scale(uint32_t x, float) { return x; }
  template <bool COH>
  static __device__ __forceinline__ uint32_t load1(const void* p) { return Mem<COH>::u32(p); }
  static __device__ __forceinline__ void store1(void* p, uint32_t v) { st_u32(p, v); }
};

// ------------------------------------------------------------------ realignment --
// The 16 bytes that start sigma bytes into `lo`, continuing into `hi` (lo and hi are
// consecutive aligned blocks of a source), by funnel shifts of 32-bit words.
__device__ __forceinline__ uint4 shift_pair(uint4 lo, uint4 hi, unsigned sigma) {
  const unsigned r = (sigma & 3u) * 8u;
  uint32_t w0 = lo.x, w1 = lo.y, w2 = lo.z, w3 = lo.w, w4 = hi.x, w5 = hi.y, w6 = hi.z, w7 = hi.w;
  uint4 o;
  switch (sigma >> 2) {
    case 0:
      o.x = __funnelshift_r(w0, w1, r); o.y = __funnelshift_r(w1, w2, r);
      o.z = __funnelshift_r(w2, w3, r); o.w = __funnelshift_r(w3, w4, r);
      break;
    case 1:
      o.x = __funnelshift_r(w1, w2, r); o.y = __funnelshift_r(w2, w3, r);
      o.z = __funnelshift_r(w3, w4, r); o.w = __funnelshift_r(w4, w5, r);
      break;
    case 2:
      o.x = __funnelshift_r(w2, w3, r); o.y = __funnelshift_r(w3, w4, r);
      o.z = __funnelshift_r(w4, w5, r); o.w = __funnelshift_r(w5, w6, r);
      break;
    default:
      o.x = __funnelshift_r(w3, w4, r); o.y = __funnelshift_r(w4, w5, r);
      o.z = __funnelshift_r(w5, w6, r); o.w = __funnelshift_r(w6, w7, r);
      break;
  }
  return o;
}

}  // namespace
}  // namespace relay
