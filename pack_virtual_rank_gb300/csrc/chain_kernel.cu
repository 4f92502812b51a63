// chain_kernel.cu -- the chained launch's kernel and its launcher (the analysis that groups the
// pieces is chain.cpp).
//
// One ordinary launch for a whole call: CTA t runs tile t of one group of pieces in pass
// order, with a block barrier between passes where a dependency crosses threads, so every
// dependency of the schedule stays inside one CTA and no CTA ever waits for another; then it
// drops the group's dead scratch lines from L2.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "device.cuh"

namespace relay {
namespace {

// A piece is any element range of a segment (chain.cpp); its alignment is sorted out here:
// a scalar head until the destinations sit on a 16-byte boundary, then 16-byte vectors
// (sources realigned from two aligned blocks when only they are off the grid), then a
// scalar tail.

// The small tables come first and the segment table last, so that every table the kernel
// indexes by a run-time value starts within the block's first 2 KiB. With the drop table
// at parameter offsets 31,890-32,274 of the 384-piece block, the kernel on GB300 did not
// see its values (no line of those programs was ever dropped), although a probe kernel
// read every byte of a 32,752-byte parameter correctly by index from offset 0.
template <int CAP>
struct ChainArgs {
  int32_t ngroup;
  int32_t ntask;
  float scale;
  int32_t tile;               // elements per task
  int32_t mult;               // CTA b runs task (b * mult) mod ntask (mult coprime to ntask)
  uint8_t level[CAP];         // pass of each piece
  uint8_t drop[CAP];          // sources whose lines go dead after this piece (program.h)
  uint8_t local[CAP];         // per group: dependencies stay inside each thread (program.h)
  int16_t gfirst[CAP + 1];    // first piece of each group, then one past the last
  Seg seg[CAP];               // tile0: first task of the piece's group
};
static_assert(sizeof(ChainArgs<kChainMaxPieces>) <= 32764, "kernel parameter space");

// Elements [b, e) of a piece one at a time (copies move raw bits), U elements per thread
// per batch: each source's loads of a batch are issued together, then combined in source
// order. The general executor of the 4-source build takes U = 4 (off-grid 4-active calls
// 13-25% faster); the others keep U = 1, which their register limits fit better.
template <class P, bool COH, bool COPY = false, int U = 1>
__device__ __forceinline__ void piece_scalar(const Seg& s, int64_t b, int64_t e, float scale) {
  using Acc = typename P::Acc;
  const bool copy = COPY || s.op == kOpCopy;
  const bool do_scale = (s.flags & kFlagScale) != 0;
#pragma unroll 1
  for (int64_t i0 = b + threadIdx.x; i0 < e; i0 += (int64_t)kThreads * U) {
    if (copy) {
      uint32_t x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        const char* q = static_cast<const char*>(s.src[0]) + i * P::kE;
        x[u] = i >= e ? 0u : P::kE == 4 ? Mem<COH>::u32(q) : (uint32_t)Mem<COH>::u16(q);
      }
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t i = i0 + (int64_t)u * kThreads;
          if (i >= e) break;
          char* q = static_cast<char*>(s.dst[d]) + i * P::kE;
          if (P::kE == 4) st_u32(q, x[u]);
          else st_u16(q, (uint16_t)x[u]);
        }
      }
      continue;
    }
    Acc acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * kThreads;
      acc[u] = i >= e ? Acc(0) : P::template load1<COH>(static_cast<const char*>(s.src[0]) + i * P::kE);
    }
#pragma unroll 1
    for (int k = 1; k < s.nsrc; ++k) {
      Acc w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        w[u] = i >= e ? Acc(0) : P::template load1<COH>(static_cast<const char*>(s.src[k]) + i * P::kE);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = P::add(acc[u], w[u]);
    }
    if (do_scale) {
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = P::scale(acc[u], scale);
    }
#pragma unroll 1
    for (int d = 0; d < s.ndst; ++d) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        if (i >= e) break;
        P::store1(static_cast<char*>(s.dst[d]) + i * P::kE, acc[u]);
      }
    }
  }
}

// A batch's results r[u] (vector vi0 + u * kThreads of the piece from byte offset `off`)
// to every destination: kept in L2 when a later pass of this CTA reads them, else
// streamed. Each destination pointer is read once per batch: the stores' memory clobbers
// would otherwise make the compiler reload it from parameter space for every vector.
// CHECK: vectors at or past nvec are skipped.
template <int UB, bool CHECK>
__device__ __forceinline__ void store_batch(const Seg& s, int ndst, int64_t off, int vi0, int nvec,
                                            const uint4 (&r)[UB], bool keep) {
#pragma unroll
  for (int d = 0; d < kMaxDst; ++d) {
    if (d >= ndst) break;
    uint4* q = reinterpret_cast<uint4*>(static_cast<char*>(s.dst[d]) + off);
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      const int vi = vi0 + u * kThreads;
      if (CHECK && vi >= nvec) break;
      if (keep) st_v4_keep(q + vi, r[u]);
      else st_v4(q + vi, r[u]);
    }
  }
}

// r = the sum of v[0..NSRC) lane by lane, scaled if asked, rounded to the payload type.
template <class P, int NSRC>
__device__ __forceinline__ uint4 reduce_vec(const uint4 (&v)[NSRC], bool do_scale, float scale) {
  constexpr int L = P::kLanes;
  using Acc = typename P::Acc;
  Acc acc[L], w[L];
  P::unpack(v[0], acc);
#pragma unroll
  for (int k = 1; k < NSRC; ++k) {
    P::unpack(v[k], w);
#pragma unroll
    for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], w[i]);
  }
  if (do_scale) {
#pragma unroll
    for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], scale);
  }
  return P::pack(acc);
}

// A whole 16 KiB tile from element b on, every pointer 16-byte aligned there: each thread
// takes kUnroll vectors (batches of 2 past two sources), no bounds to check.
template <class P, int NSRC, bool COH, bool COPY = false>
__device__ __forceinline__ void piece_full(const Seg& s, int64_t b, float scale) {
  constexpr int UB = NSRC <= 2 ? kUnroll : kUnroll / 2;
  const bool reduce = !COPY && s.op != kOpCopy;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool keep = (s.flags & kFlagKeep) != 0;
  const int ndst = s.ndst;
  const int64_t off = b * P::kE;
  const int t = (int)threadIdx.x;
  const uint4* src[NSRC];
#pragma unroll
  for (int k = 0; k < NSRC; ++k)
    src[k] = reinterpret_cast<const uint4*>(static_cast<const char*>(s.src[k]) + off) + t;
#pragma unroll
  for (int u0 = 0; u0 < kUnroll; u0 += UB) {
    uint4 v[UB][NSRC];
#pragma unroll
    for (int u = 0; u < UB; ++u)
#pragma unroll
      for (int k = 0; k < NSRC; ++k) v[u][k] = Mem<COH>::v4(src[k] + (u0 + u) * kThreads);
    uint4 r[UB];
#pragma unroll
    for (int u = 0; u < UB; ++u) r[u] = reduce ? reduce_vec<P, NSRC>(v[u], do_scale, scale) : v[u][0];
    store_batch<UB, false>(s, ndst, off, t + u0 * kThreads, 0, r, keep);
  }
}

// nvec 16-byte vectors from element b on, every pointer 16-byte aligned there. Loads of a
// batch are issued together (4 vectors per thread per source, 2 past two sources).
template <class P, int NSRC, bool COH, bool COPY = false>
__device__ __forceinline__ void piece_vec(const Seg& s, int64_t b, int nvec, float scale) {
  constexpr int UB = NSRC <= 2 ? kUnroll : kUnroll / 2;
  const bool reduce = !COPY && s.op != kOpCopy;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool keep = (s.flags & kFlagKeep) != 0;
  const int ndst = s.ndst;
  const uint4* src[NSRC];
#pragma unroll
  for (int k = 0; k < NSRC; ++k)
    src[k] = reinterpret_cast<const uint4*>(static_cast<const char*>(s.src[k]) + b * P::kE);
#pragma unroll 1
  for (int v0 = (int)threadIdx.x; v0 < nvec; v0 += kThreads * UB) {
    uint4 v[UB][NSRC];
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      const int vi = v0 + u * kThreads;
#pragma unroll
      for (int k = 0; k < NSRC; ++k)
        v[u][k] = vi < nvec ? Mem<COH>::v4(src[k] + vi) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint4 r[UB];
#pragma unroll
    for (int u = 0; u < UB; ++u) r[u] = reduce ? reduce_vec<P, NSRC>(v[u], do_scale, scale) : v[u][0];
    store_batch<UB, true>(s, ndst, b * P::kE, v0, nvec, r, keep);
  }
}

// The same with the destinations aligned at element b but one or two sources off the
// 16-byte grid: each vector of such a source is funnel-shifted out of the two aligned
// blocks it straddles (both hold bytes of the piece's own source range).
template <class P, int NSRC, bool COH, bool COPY = false>
__device__ __forceinline__ void piece_realign(const Seg& s, int64_t b, int nvec, float scale) {
  constexpr int UB = NSRC <= 2 ? 2 : 1;
  const bool reduce = !COPY && s.op != kOpCopy;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool keep = (s.flags & kFlagKeep) != 0;
  const int ndst = s.ndst;
  unsigned sig[NSRC];
  const uint4* a[NSRC];
#pragma unroll
  for (int k = 0; k < NSRC; ++k) {
    const char* p = static_cast<const char*>(s.src[k]) + b * P::kE;
    sig[k] = (unsigned)(reinterpret_cast<uintptr_t>(p) & 15u);
    a[k] = reinterpret_cast<const uint4*>(p - sig[k]);
  }
#pragma unroll 1
  for (int v0 = (int)threadIdx.x; v0 < nvec; v0 += kThreads * UB) {
    uint4 v[UB][NSRC];
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      const int vi = v0 + u * kThreads;
#pragma unroll
      for (int k = 0; k < NSRC; ++k) {
        if (vi < nvec) {
          v[u][k] = Mem<COH>::v4(a[k] + vi);
          if (sig[k] != 0) v[u][k] = shift_pair(v[u][k], Mem<COH>::v4(a[k] + vi + 1), sig[k]);
        } else {
          v[u][k] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    uint4 r[UB];
#pragma unroll
    for (int u = 0; u < UB; ++u) r[u] = reduce ? reduce_vec<P, NSRC>(v[u], do_scale, scale) : v[u][0];
    store_batch<UB, true>(s, ndst, b * P::kE, v0, nvec, r, keep);
  }
}

// A mixed-width piece of a bf16 payload: the helper summing its bf16 slots into an fp32
// partial (kFlagOutF32), or an owner adding its own bf16 value and the fp32 partial,
// scaled once and rounded to bf16 (kFlagSrc1F32). 8 elements per step (one 16-byte bf16
// vector, two fp32 vectors) when the destinations and an fp32 source are 16-byte aligned at
// `base` (a bf16 source off that grid is funnel-shifted out of the two aligned blocks it
// straddles, both holding bytes of its own range), else one element at a time.
template <bool COH>
__device__ __noinline__ void piece_mixed(const Seg& s, int64_t base, int64_t len, float scale) {
  const bool out_f32 = (s.flags & kFlagOutF32) != 0;
  const bool src1_f32 = (s.flags & kFlagSrc1F32) != 0;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool keep = (s.flags & kFlagKeep) != 0;
  auto sw = [&](int k) { return (k == 1 && src1_f32) ? 4 : 2; };
  const int dw = out_f32 ? 4 : 2;
  bool al = true;
  for (int k = 0; k < s.nsrc; ++k)
    if (sw(k) == 4) al &= ((reinterpret_cast<uintptr_t>(s.src[k]) + (uintptr_t)(base * 4)) & 15u) == 0;
  for (int d = 0; d < s.ndst; ++d)
    al &= ((reinterpret_cast<uintptr_t>(s.dst[d]) + (uintptr_t)(base * dw)) & 15u) == 0;
  // the 8 bf16 elements of source k from element e on, whatever its alignment
  auto bf16_vec = [&](int k, int64_t e) {
    const char* p = static_cast<const char*>(s.src[k]) + e * 2;
    const unsigned sig = (unsigned)(reinterpret_cast<uintptr_t>(p) & 15u);
    const uint4* q = reinterpret_cast<const uint4*>(p - sig);
    const uint4 lo = Mem<COH>::v4(q);
    return sig ? shift_pair(lo, Mem<COH>::v4(q + 1), sig) : lo;
  };
  int64_t done = 0;
  if (al) {
    const int nvec = (int)(len / 8);
#pragma unroll 1
    for (int v = (int)threadIdx.x; v < nvec; v += kThreads) {
      const int64_t e = base + 8 * (int64_t)v;
      float acc[8], t[8];
      TBF16::unpack(bf16_vec(0, e), acc);
#pragma unroll 1
      for (int k = 1; k < s.nsrc; ++k) {
        if (k == 1 && src1_f32) {
          const char* q = static_cast<const char*>(s.src[1]) + e * 4;
          const uint4 lo = Mem<COH>::v4(q), hi = Mem<COH>::v4(q + 16);
          t[0] = __uint_as_float(lo.x); t[1] = __uint_as_float(lo.y);
          t[2] = __uint_as_float(lo.z); t[3] = __uint_as_float(lo.w);
          t[4] = __uint_as_float(hi.x); t[5] = __uint_as_float(hi.y);
          t[6] = __uint_as_float(hi.z); t[7] = __uint_as_float(hi.w);
        } else {
          TBF16::unpack(bf16_vec(k, e), t);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], t[i]);
      }
      if (do_scale) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fmul_rn(acc[i], scale);
      }
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) {
        if (out_f32) {
          char* q = static_cast<char*>(s.dst[d]) + e * 4;
          const uint4 lo = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                      __float_as_uint(acc[2]), __float_as_uint(acc[3]));
          const uint4 hi = make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                      __float_as_uint(acc[6]), __float_as_uint(acc[7]));
          if (keep) { st_v4_keep(q, lo); st_v4_keep(q + 16, hi); }
          else { st_v4(q, lo); st_v4(q + 16, hi); }
        } else {
          char* q = static_cast<char*>(s.dst[d]) + e * 2;
          if (keep) st_v4_keep(q, TBF16::pack(acc)); else st_v4(q, TBF16::pack(acc));
        }
      }
    }
    done = 8 * (int64_t)nvec;
  }
  // The rest one element at a time, U elements per thread per batch: each source's loads
  // of a batch are issued together, then added in source order as above.
  constexpr int U = 4;
  const int64_t end = base + len;
#pragma unroll 1
  for (int64_t i0 = base + done + threadIdx.x; i0 < end; i0 += (int64_t)kThreads * U) {
    float acc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + (int64_t)u * kThreads;
      acc[u] = i < end ? TBF16::template load1<COH>(static_cast<const char*>(s.src[0]) + i * 2) : 0.f;
    }
#pragma unroll 1
    for (int k = 1; k < s.nsrc; ++k) {
      float w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        w[u] = i >= end ? 0.f
               : (k == 1 && src1_f32)
                   ? TF32::template load1<COH>(static_cast<const char*>(s.src[1]) + i * 4)
                   : TBF16::template load1<COH>(static_cast<const char*>(s.src[k]) + i * 2);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = __fadd_rn(acc[u], w[u]);
    }
    if (do_scale) {
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = __fmul_rn(acc[u], scale);
    }
#pragma unroll 1
    for (int d = 0; d < s.ndst; ++d) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * kThreads;
        if (i >= end) break;
        if (out_f32) TF32::store1(static_cast<char*>(s.dst[d]) + i * 4, acc[u]);
        else TBF16::store1(static_cast<char*>(s.dst[d]) + i * 2, acc[u]);
      }
    }
  }
}

// The whole 128-byte lines of this tile's part of each source in `mask`: scratch that no
// later pass reads, dropped from L2 so that it is never written back to memory. Partial
// lines at the ends may hold a neighbour's live bytes and stay. A tile's part of one
// source is at most 32 KiB (an fp32 partial beside a 16 KiB bf16 tile): one line per
// thread; the loop only guards that bound.
template <class P>
__device__ __forceinline__ void drop_lines(const Seg& s, unsigned mask, int64_t base, int64_t len) {
#pragma unroll 1
  for (int k = 0; k < kMaxSrc; ++k) {
    if (!((mask >> k) & 1u)) continue;
    const int64_t w = (k == 1 && (s.flags & kFlagSrc1F32)) ? 4 : P::kE;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(s.src[k]) + (uintptr_t)(base * w);
    const uintptr_t hi = lo + (uintptr_t)(len * w);
#pragma unroll 1
    for (uintptr_t q = ((lo + 127) & ~(uintptr_t)127) + (uintptr_t)threadIdx.x * 128; q + 128 <= hi;
         q += (uintptr_t)kThreads * 128)
      discard_l2(reinterpret_cast<const void*>(q));
  }
}

// Elements [base, base + len) of segment s, whatever the alignment of its pointers there.
// MAXSRC: the most sources a reduction of the launch has (1: copies only); the paths for
// more are compiled out.
template <class P, bool COH, int MAXSRC>
__device__ __noinline__ void run_piece(const Seg& s, int64_t base, int64_t len, float scale) {
  constexpr int E = P::kE, L = P::kLanes;
  constexpr bool COPY = MAXSRC == 1;
  constexpr int SU = MAXSRC > 2 ? 4 : 1;  // elements per thread per batch, one at a time
  auto mis = [&](const void* p) {
    return (unsigned)((reinterpret_cast<uintptr_t>(p) + (uintptr_t)(base * E)) & 15u);
  };
  const int nsrc = COPY || s.op == kOpCopy ? 1 : s.nsrc;
  const unsigned md = mis(s.dst[0]);
  bool dsame = md % E == 0;
  for (int d = 1; d < s.ndst; ++d) dsame &= mis(s.dst[d]) == md;
  if (dsame && md == 0 && len * E == kTileBytes) {
    bool sal = true;
    for (int k = 0; k < nsrc; ++k) sal &= mis(s.src[k]) == 0;
    if (sal) {
      if (COPY || nsrc == 1) piece_full<P, 1, COH, COPY>(s, base, scale);
      else if constexpr (MAXSRC >= 2) {
        if (nsrc == 2) piece_full<P, 2, COH>(s, base, scale);
        else if constexpr (MAXSRC > 2) {
          if (nsrc == 3) piece_full<P, 3, COH>(s, base, scale);
          else piece_full<P, 4, COH>(s, base, scale);
        }
      }
      return;
    }
  }
  if (!dsame) {
    piece_scalar<P, COH, COPY, SU>(s, base, base + len, scale);
    return;
  }
  const int64_t head = min((int64_t)(((16u - md) & 15u) / E), len);
  piece_scalar<P, COH, COPY, SU>(s, base, base + head, scale);
  const int64_t b1 = base + head;
  const int nvec = (int)((len - head) / L);
  if (nvec > 0) {
    bool sal = true;
    for (int k = 0; k < nsrc; ++k)
      sal &= ((reinterpret_cast<uintptr_t>(s.src[k]) + (uintptr_t)(b1 * E)) & 15u) == 0;
    if (sal) {
      if (COPY || nsrc == 1) piece_vec<P, 1, COH, COPY>(s, b1, nvec, scale);
      else if constexpr (MAXSRC >= 2) {
        if (nsrc == 2) piece_vec<P, 2, COH>(s, b1, nvec, scale);
        else if constexpr (MAXSRC > 2) {
          if (nsrc == 3) piece_vec<P, 3, COH>(s, b1, nvec, scale);
          else piece_vec<P, 4, COH>(s, b1, nvec, scale);
        }
      }
    } else if (COPY || nsrc == 1) {
      piece_realign<P, 1, COH, COPY>(s, b1, nvec, scale);
    } else if (nsrc == 2) {
      if constexpr (MAXSRC >= 2) piece_realign<P, 2, COH>(s, b1, nvec, scale);
    } else if constexpr (MAXSRC > 2) {
      if (nsrc == 3) piece_realign<P, 3, COH>(s, b1, nvec, scale);
      else piece_realign<P, 4, COH>(s, b1, nvec, scale);
    }
  }
  piece_scalar<P, COH, COPY, SU>(s, b1 + nvec * L, base + len, scale);
}

// MAXSRC: the most sources any reduction of the launch has, 4 for any program (fp32
// partials included). MINB: CTAs per SM the build is held to. Programs of copies only
// (all-gather, all-to-all) take MAXSRC = 1 and run 8 CTAs per SM at 32 registers; those
// whose reductions have at most two sources (the 2-active collectives) take MAXSRC = 2 and
// run 6 at 40. Of the rest, programs with fp32 partials (the 4-active bf16 reduce-scatter,
// whose mixed-width executor stays spill-free at 40 registers) run 6, 3-12% faster than at
// 5; the others (the 4-active allreduce) run 5 at 48, 2.4% faster than at 6.
template <class P, int CAP, int MAXSRC, int MINB>
__global__ void __launch_bounds__(kThreads, MINB)
    relay_chain_kernel(const __grid_constant__ ChainArgs<CAP> a) {
  // the task of this CTA (a permutation of the grid; see the launcher)
  const int t = (int)(((int64_t)blockIdx.x * a.mult) % a.ntask);
  // the last group whose first task is <= t (uniform across the CTA)
  int lo = 0, hi = a.ngroup - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.seg[a.gfirst[mid]].tile0 <= t) lo = mid; else hi = mid - 1;
  }
  const int f = a.gfirst[lo], l = a.gfirst[lo + 1];
  const int64_t base = (int64_t)(t - a.seg[f].tile0) * a.tile;
  const int64_t len = min((int64_t)a.tile, a.seg[f].n - base);
  // in a group whose dependencies stay inside each thread, program order alone puts a
  // thread's loads of the next pass after its own stores of this one
  const bool local = a.local[lo] != 0;
  // every piece of an aligned group is 16-byte aligned at every tile base
  const bool full = local && len * P::kE == kTileBytes;
  int lvl = a.level[f];
  for (int i = f; i < l; ++i) {
    if (a.level[i] != lvl) {
      // the previous pass's stores of this tile are visible to the whole CTA after this
      if (!local) __syncthreads();
      lvl = a.level[i];
    }
    // the first pass reads only memory written before the launch; later passes read what
    // this CTA has just written, through L2. fp32 partials exist only next to a bf16
    // payload (the host refuses anything else).
    const bool first = lvl == a.level[f];
    if (MAXSRC > 2 && P::kE == 2 && seg_mixed(a.seg[i])) {
      if (first) piece_mixed<false>(a.seg[i], base, len, a.scale);
      else piece_mixed<true>(a.seg[i], base, len, a.scale);
    } else if (MAXSRC >= 2 && full) {
      // A whole aligned tile, inline in the kernel: apart from the general executor (which
      // spills under these register limits) it gets a spill-free allocation, measured 3-9%
      // faster than the executor's own fast path on every reducing program. Copy-only
      // programs gained nothing from it and keep the executor.
      const Seg& sg = a.seg[i];
      const int ns = sg.op == kOpCopy ? 1 : sg.nsrc;
      if (first) {
        if (ns == 1) piece_full<P, 1, false>(sg, base, a.scale);
        else if (ns == 2) piece_full<P, 2, false>(sg, base, a.scale);
        else if constexpr (MAXSRC > 2) {
          if (ns == 3) piece_full<P, 3, false>(sg, base, a.scale);
          else piece_full<P, 4, false>(sg, base, a.scale);
        }
      } else {
        if (ns == 1) piece_full<P, 1, true>(sg, base, a.scale);
        else if (ns == 2) piece_full<P, 2, true>(sg, base, a.scale);
        else if constexpr (MAXSRC > 2) {
          if (ns == 3) piece_full<P, 3, true>(sg, base, a.scale);
          else piece_full<P, 4, true>(sg, base, a.scale);
        }
      }
    } else if (first) {
      run_piece<P, false, MAXSRC>(a.seg[i], base, len, a.scale);
    } else {
      run_piece<P, true, MAXSRC>(a.seg[i], base, len, a.scale);
    }
  }
  // Scratch whose last reader has run: once every thread's reads are done, its lines are
  // dead, and dropping them spares the write-back of bytes nothing will read.
  unsigned any = 0;
  for (int i = f; i < l; ++i) any |= a.drop[i];
  if (any) {
    __syncthreads();
    for (int i = f; i < l; ++i)
      if (a.drop[i]) drop_lines<P>(a.seg[i], a.drop[i], base, len);
  }
}

template <class P, int CAP>
cudaError_t launch_chain_cap(const ChainPlan& c, float scale, int64_t tile, cudaStream_t stream,
                             int* ntask_out, int max_src, bool mixed) {
  static thread_local ChainArgs<CAP> a;  // up to ~32 KiB: keep it off the stack
  const int G = (int)c.gn.size();
  int64_t tasks = 0;
  for (int g = 0; g < G; ++g) {
    a.gfirst[g] = (int16_t)c.gfirst[g];
    for (int i = c.gfirst[g]; i < c.gfirst[g + 1]; ++i) {
      a.seg[i] = c.segs[i];
      a.seg[i].tile0 = (int32_t)tasks;
      a.level[i] = c.level[i];
      a.drop[i] = c.drop[i];
    }
    tasks += (c.gn[g] + tile - 1) / tile;
  }
  a.gfirst[G] = (int16_t)c.gfirst[G];
  for (int g = 0; g < G; ++g) a.local[g] = c.local[g];
  a.ngroup = G;
  a.ntask = (int32_t)tasks;
  a.scale = scale;
  a.tile = (int32_t)tile;
  // Programs whose chains span three or more passes (the 4-active all-to-all and
  // reduce-scatter) spread each wave of CTAs over every group: tasks about a resident CTA's
  // share of the grid apart, the step coprime to the task count. The all-to-all's
  // latency-bound chains then share each SM with its streaming copies (4.5-4.9% faster; the
  // reduce-scatter 0.7%). Two-pass programs lost 1-6% that way, to DRAM locality, and keep
  // their tasks in group order.
  int levels = 0;
  for (uint8_t l : c.level) levels = std::max(levels, (int)l + 1);
  int64_t m = 1;
  if (levels >= 3) {
    const int64_t resident = (int64_t)sm_count() * (max_src == 1 ? 8 : max_src == 2 || mixed ? 6 : 5);
    m = std::max<int64_t>(1, tasks / resident);
    auto gcd = [](int64_t x, int64_t y) {
      while (y) {
        const int64_t r = x % y;
        x = y;
        y = r;
      }
      return x;
    };
    while (gcd(m, tasks) != 1) ++m;
  }
  a.mult = (int32_t)m;
  *ntask_out = (int)tasks;
  if (max_src == 1) relay_chain_kernel<P, CAP, 1, 8><<<(unsigned)tasks, kThreads, 0, stream>>>(a);
  else if (max_src == 2) relay_chain_kernel<P, CAP, 2, 6><<<(unsigned)tasks, kThreads, 0, stream>>>(a);
  else if (mixed) relay_chain_kernel<P, CAP, 4, 6><<<(unsigned)tasks, kThreads, 0, stream>>>(a);
  else relay_chain_kernel<P, CAP, 4, 5><<<(unsigned)tasks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <class P>
cudaError_t launch_chain_typed(const ChainPlan& c, float scale, int64_t tile, cudaStream_t stream,
                               int* ntask) {
  const size_t n = c.segs.size();
  int max_src = 1;
  bool mixed = false;
  for (const Seg& sg : c.segs) {
    if (sg.op != kOpCopy) max_src = std::max<int>(max_src, seg_mixed(sg) ? kMaxSrc : sg.nsrc);
    mixed |= seg_mixed(sg);
  }
  if (n <= 32) return launch_chain_cap<P, 32>(c, scale, tile, stream, ntask, max_src, mixed);
  if (n <= 128) return launch_chain_cap<P, 128>(c, scale, tile, stream, ntask, max_src, mixed);
  return launch_chain_cap<P, kChainMaxPieces>(c, scale, tile, stream, ntask, max_src, mixed);
}

}  // namespace

// Tiles of 16 KiB, halved (down to 4 KiB, one 16-byte vector per thread) while the call
// has fewer tasks than twice the SMs: in the latency-bound regime more, smaller tasks
// spread the same bytes over more SMs.
bool launch_chain(int dtype, const ChainPlan& c, float scale, cudaStream_t stream,
                  cudaError_t* err) {
  *err = cudaSuccess;
  if (c.segs.empty() || c.segs.size() > (size_t)kChainMaxPieces) return false;
  const int E = esize_of(dtype);
  int64_t tile_bytes = kTileBytes;
  auto tasks = [&](int64_t tb) {
    int64_t t = 0;
    for (int64_t n : c.gn) t += (n + tb / E - 1) / (tb / E);
    return t;
  };
  while (tile_bytes > (int64_t)kThreads * kVecBytes && tasks(tile_bytes) < 2 * sm_count())
    tile_bytes /= 2;
  if (tasks(tile_bytes) > INT32_MAX) return false;
  const int64_t tile = tile_bytes / E;
  int ntask = 0;
  switch (dtype) {
    case RELAY_F32: *err = launch_chain_typed<TF32>(c, scale, tile, stream, &ntask); break;
    case RELAY_BF16: *err = launch_chain_typed<TBF16>(c, scale, tile, stream, &ntask); break;
    default: *err = launch_chain_typed<TI32>(c, scale, tile, stream, &ntask); break;
  }
  return true;
}

}  // namespace relay
