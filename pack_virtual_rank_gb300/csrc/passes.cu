// passes.cu -- the one streaming kernel behind every relay pass (sm_103a).
//
// A pass is a table of segments (program.h) executed by one launch. Each segment is
// cut into tiles of 16 KiB of payload and the grid has one CTA per tile of the whole
// table, so one launch covers every transfer and reduction of a schedule group
// regardless of how many there are (the page
// "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)", item 5, blames the
// per-op launch overhead of many small groups; here a group costs one launch).
//
// Per tile a CTA of 256 threads issues all its 16-byte loads first (4 per thread per
// source), then reduces in fp32 (int32: wrapping uint32) in ascending source order,
// scales once, rounds to nearest-even into the payload type and stores the result to
// each destination. Copies move raw 16-byte vectors. Segments whose pointers are not
// 16-byte aligned (after a host-side prologue split) take a per-element path.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <type_traits>

#include "device.cuh"
#include "program.h"

namespace relay {
namespace {

template <int CAP>
struct PassArgs {
  int32_t nseg;
  int32_t ntiles;
  float scale;
  int32_t extra_tx;  // staged kernel: bytes its barrier expects beyond the copies (0; a test
                     // sets it to make a wait run out)
  Seg seg[CAP];
};

// ---------------------------------------------------------------- tile bodies --

// Whole tile on the 16-byte vector path: every thread loads kUnroll vectors per
// source (in batches that keep at most 8 loads in flight per thread), reduces and
// stores them. base is the tile's first element.
template <class P, int NSRC, bool COH, int U = kUnroll>
__device__ __forceinline__ void reduce_full_tile(const Seg& s, int64_t base, float scale) {
  constexpr int L = P::kLanes;
  constexpr int UB = (NSRC <= 2 || U < 2) ? U : U / 2;
  using Acc = typename P::Acc;
  const int64_t v0 = base / L + threadIdx.x;
  const bool do_scale = (s.flags & kFlagScale) != 0;
#pragma unroll
  for (int u0 = 0; u0 < U; u0 += UB) {
    uint4 v[NSRC][UB];
#pragma unroll
    for (int u = 0; u < UB; ++u)
#pragma unroll
      for (int k = 0; k < NSRC; ++k)
        v[k][u] = Mem<COH>::v4(static_cast<const uint4*>(s.src[k]) + v0 + (u0 + u) * kThreads);
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      Acc acc[L], t[L];
      P::unpack(v[0][u], acc);
#pragma unroll
      for (int k = 1; k < NSRC; ++k) {
        P::unpack(v[k][u], t);
#pragma unroll
        for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], t[i]);
      }
      if (do_scale) {
#pragma unroll
        for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], scale);
      }
      const uint4 r = P::pack(acc);
#pragma unroll
      for (int d = 0; d < kMaxDst; ++d)
        if (d < s.ndst) st_v4(static_cast<uint4*>(s.dst[d]) + v0 + (u0 + u) * kThreads, r);
    }
  }
}

template <bool COH, int U = kUnroll>
__device__ __forceinline__ void copy_full_tile(const Seg& s, int64_t vbase) {
  const int64_t v0 = vbase + threadIdx.x;
  uint4 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u)
    v[u] = Mem<COH>::v4(static_cast<const uint4*>(s.src[0]) + v0 + u * kThreads);
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int d = 0; d < kMaxDst; ++d)
      if (d < s.ndst) st_v4(static_cast<uint4*>(s.dst[d]) + v0 + u * kThreads, v[u]);
}

template <class P, bool COH, int U = kUnroll>
__device__ __forceinline__ void run_full_tile(const Seg& s, int64_t base, float scale) {
  if (s.op == kOpCopy) {
    copy_full_tile<COH, U>(s, base / P::kLanes);
    return;
  }
  switch (s.nsrc) {
    case 1: reduce_full_tile<P, 1, COH, U>(s, base, scale); break;
    case 2: reduce_full_tile<P, 2, COH, U>(s, base, scale); break;
    case 3: reduce_full_tile<P, 3, COH, U>(s, base, scale); break;
    default: reduce_full_tile<P, 4, COH, U>(s, base, scale); break;
  }
}

// ---------------------------------------------------------- realigned sources --
// Destinations 16-byte aligned, sources at any element offset (an all-to-all whose
// segmentCount is not a multiple of the vector width, an odd recvCount): each lane loads
// the aligned 16-byte vector that holds the start of its source range, takes the next
// one from its right neighbour by a warp shuffle, and funnel-shifts the pair by the
// source's byte offset (shift_pair, device.cuh; the one-launch kernel loads both blocks
// itself). Reads stay inside the 16-byte blocks that hold the segment's own bytes.

// TAIL: a segment's last, partial tile. Only its first `nvec` whole vectors are stored; a
// block is loaded only if it holds bytes of those vectors (the block after the last one
// holds its final bytes when the source is misaligned), so every read stays inside the
// segment's own 16-byte blocks. The shuffles still run on every lane.
template <class P, int NSRC, bool TAIL = false>
__device__ __forceinline__ void realign_full_tile(const Seg& s, int64_t base, float scale,
                                                  int nvec = 0) {
  constexpr int L = P::kLanes;
  // vectors per source in flight: all kUnroll for one source, 2 at a time for two
  constexpr int NB = NSRC == 1 ? kUnroll : 2;
  using Acc = typename P::Acc;
  // Warp w covers the tile's vectors [w, w + 1) x 32 * kUnroll, lane l takes l + 32 * j:
  // the block after lane 31's j-th is lane 0's (j+1)-th, so a warp loads only one extra
  // block (lane 31's last neighbour) per batch instead of one per vector.
  const unsigned lane = threadIdx.x & 31u;
  const bool last_lane = lane == 31u;
  const int lv0 = (int)(threadIdx.x >> 5) * (32 * kUnroll) + (int)lane;  // within the tile
  const int64_t v0 = base / L + lv0;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  unsigned sig[NSRC];
  const uint4* a[NSRC];
  int last_blk[NSRC];  // TAIL: last block index (within the tile) that may be read
#pragma unroll
  for (int k = 0; k < NSRC; ++k) {
    sig[k] = (unsigned)(reinterpret_cast<uintptr_t>(s.src[k]) & 15u);
    a[k] = reinterpret_cast<const uint4*>(static_cast<const char*>(s.src[k]) - sig[k]);
    last_blk[k] = sig[k] != 0 ? nvec : nvec - 1;
  }
#pragma unroll
  for (int u = 0; u < kUnroll; u += NB) {
    uint4 cur[NSRC][NB], ext[NSRC];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int k = 0; k < NSRC; ++k) {
        if (!TAIL || lv0 + (u + j) * 32 <= last_blk[k])
          cur[k][j] = ld_stream_v4(a[k] + v0 + (u + j) * 32);
        else
          cur[k][j] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
    for (int k = 0; k < NSRC; ++k)
      if (sig[k] != 0 && last_lane && (!TAIL || lv0 + (u + NB - 1) * 32 + 1 <= last_blk[k]))
        ext[k] = ld_stream_v4(a[k] + v0 + (u + NB - 1) * 32 + 1);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      uint4 v[NSRC];
#pragma unroll
      for (int k = 0; k < NSRC; ++k) {
        v[k] = cur[k][j];
        if (sig[k] != 0) {
          // every lane reads its right neighbour's block; lane 0 offers its next one,
          // which is what lane 31 needs
          uint4 send = cur[k][j];
          if (j + 1 < NB && lane == 0) send = cur[k][j + 1];
          const int from = (int)((lane + 1) & 31u);
          uint4 nxt;
          nxt.x = __shfl_sync(0xffffffffu, send.x, from);
          nxt.y = __shfl_sync(0xffffffffu, send.y, from);
          nxt.z = __shfl_sync(0xffffffffu, send.z, from);
          nxt.w = __shfl_sync(0xffffffffu, send.w, from);
          if (j + 1 == NB && last_lane) nxt = ext[k];
          v[k] = shift_pair(cur[k][j], nxt, sig[k]);
        }
      }
      uint4 r = v[0];
      if (s.op != kOpCopy) {
        Acc acc[L], t[L];
        P::unpack(v[0], acc);
#pragma unroll
        for (int k = 1; k < NSRC; ++k) {
          P::unpack(v[k], t);
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], t[i]);
        }
        if (do_scale) {
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], scale);
        }
        r = P::pack(acc);
      }
      const int64_t vi = v0 + (u + j) * 32;
      if (TAIL && lv0 + (u + j) * 32 >= nvec) continue;
#pragma unroll
      for (int d = 0; d < kMaxDst; ++d)
        if (d < s.ndst) st_v4(static_cast<uint4*>(s.dst[d]) + vi, r);
    }
  }
}

// One or two sources (the host sends segments with more sources to the per-element
// path when their sources need realigning).
template <class P>
__device__ __forceinline__ void run_realign_tile(const Seg& s, int64_t base, float scale) {
  if (s.nsrc == 1) realign_full_tile<P, 1>(s, base, scale);
  else realign_full_tile<P, 2>(s, base, scale);
}

// The last, partial tile of a realigned segment: its whole vectors on the shuffle path,
// then the last < L elements one at a time (copies move raw bits).
template <class P>
__device__ __forceinline__ void run_realign_tail(const Seg& s, int64_t base, int64_t len,
                                                 float scale) {
  using Acc = typename P::Acc;
  const int nvec = (int)(len / P::kLanes);
  if (s.nsrc == 1) realign_full_tile<P, 1, true>(s, base, scale, nvec);
  else realign_full_tile<P, 2, true>(s, base, scale, nvec);
  const bool copy = s.op == kOpCopy;
#pragma unroll 1
  for (int64_t e = (int64_t)nvec * P::kLanes + threadIdx.x; e < len; e += kThreads) {
    const int64_t off = (base + e) * P::kE;
    if (copy) {
      if (P::kE == 4) {
        const uint32_t x = Mem<false>::u32(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
        for (int d = 0; d < s.ndst; ++d) st_u32(static_cast<char*>(s.dst[d]) + off, x);
      } else {
        const uint16_t x = Mem<false>::u16(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
        for (int d = 0; d < s.ndst; ++d) st_u16(static_cast<char*>(s.dst[d]) + off, x);
      }
      continue;
    }
    Acc acc = P::template load1<false>(static_cast<const char*>(s.src[0]) + off);
    if (s.nsrc == 2) acc = P::add(acc, P::template load1<false>(static_cast<const char*>(s.src[1]) + off));
    if (s.flags & kFlagScale) acc = P::scale(acc, scale);
#pragma unroll 1
    for (int d = 0; d < s.ndst; ++d) P::store1(static_cast<char*>(s.dst[d]) + off, acc);
  }
}

// The last, partial tile of a segment and every tile of a segment whose pointers are
// not 16-byte aligned: one vector (or one element) per source at a time, with the
// source count read at run time. Rare, so it is kept small rather than fast.
template <class P, bool COH>
__device__ __noinline__ void run_partial_tile(const Seg& s, int64_t base, int64_t len,
                                              float scale) {
  using Acc = typename P::Acc;
  constexpr int L = P::kLanes;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool copy = s.op == kOpCopy;
  int64_t done = 0;
  if (s.flags & kFlagVector) {
    const int64_t vb = base / L, nvec = len / L;
#pragma unroll 1
    for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) {
      uint4 r = Mem<COH>::v4(static_cast<const uint4*>(s.src[0]) + vb + vi);
      if (!copy) {
        Acc acc[L], t[L];
        P::unpack(r, acc);
#pragma unroll 1
        for (int k = 1; k < s.nsrc; ++k) {
          P::unpack(Mem<COH>::v4(static_cast<const uint4*>(s.src[k]) + vb + vi), t);
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], t[i]);
        }
        if (do_scale) {
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], scale);
        }
        r = P::pack(acc);
      }
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) st_v4(static_cast<uint4*>(s.dst[d]) + vb + vi, r);
    }
    done = nvec * L;
  }
#pragma unroll 1
  for (int64_t e = done + threadIdx.x; e < len; e += kThreads) {
    const int64_t off = (base + e) * P::kE;
    if (copy) {
      if (P::kE == 4) {
        const uint32_t x = Mem<COH>::u32(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
        for (int d = 0; d < s.ndst; ++d) st_u32(static_cast<char*>(s.dst[d]) + off, x);
      } else {
        const uint16_t x = Mem<COH>::u16(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
        for (int d = 0; d < s.ndst; ++d) st_u16(static_cast<char*>(s.dst[d]) + off, x);
      }
      continue;
    }
    Acc acc = P::template load1<COH>(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
    for (int k = 1; k < s.nsrc; ++k)
      acc = P::add(acc, P::template load1<COH>(static_cast<const char*>(s.src[k]) + off));
    if (do_scale) acc = P::scale(acc, scale);
#pragma unroll 1
    for (int d = 0; d < s.ndst; ++d) P::store1(static_cast<char*>(s.dst[d]) + off, acc);
  }
}

// Every tile of a realigned segment in the one-launch kernel: each thread takes whole
// vectors, loads the two aligned blocks a vector's source bytes straddle and funnel-shifts
// them (no shuffles, since any subset of lanes may hold a vector), then finishes the tail
// per element.
template <class P, bool COH>
__device__ __noinline__ void run_partial_realign_tile(const Seg& s, int64_t base, int64_t len,
                                                      float scale) {
  using Acc = typename P::Acc;
  constexpr int L = P::kLanes;
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool copy = s.op == kOpCopy;
  {
    const int64_t vb = base / L, nvec = len / L;
#pragma unroll 1
    for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) {
      uint4 v[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        if (k >= s.nsrc) break;
        const unsigned sig = (unsigned)(reinterpret_cast<uintptr_t>(s.src[k]) & 15u);
        const uint4* a = reinterpret_cast<const uint4*>(static_cast<const char*>(s.src[k]) - sig);
        v[k] = Mem<COH>::v4(a + vb + vi);
        if (sig != 0) v[k] = shift_pair(v[k], Mem<COH>::v4(a + vb + vi + 1), sig);
      }
      uint4 r = v[0];
      if (!copy) {
        Acc acc[L], t[L];
        P::unpack(v[0], acc);
        if (s.nsrc == 2) {
          P::unpack(v[1], t);
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], t[i]);
        }
        if (do_scale) {
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], scale);
        }
        r = P::pack(acc);
      }
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) st_v4(static_cast<uint4*>(s.dst[d]) + vb + vi, r);
    }
    // the last < L elements one at a time (copies move raw bits)
#pragma unroll 1
    for (int64_t e = nvec * L + threadIdx.x; e < len; e += kThreads) {
      const int64_t off = (base + e) * P::kE;
      if (copy) {
        if (P::kE == 4) {
          const uint32_t x = Mem<COH>::u32(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
          for (int d = 0; d < s.ndst; ++d) st_u32(static_cast<char*>(s.dst[d]) + off, x);
        } else {
          const uint16_t x = Mem<COH>::u16(static_cast<const char*>(s.src[0]) + off);
#pragma unroll 1
          for (int d = 0; d < s.ndst; ++d) st_u16(static_cast<char*>(s.dst[d]) + off, x);
        }
        continue;
      }
      Acc acc = P::template load1<COH>(static_cast<const char*>(s.src[0]) + off);
      if (s.nsrc == 2) acc = P::add(acc, P::template load1<COH>(static_cast<const char*>(s.src[1]) + off));
      if (do_scale) acc = P::scale(acc, scale);
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) P::store1(static_cast<char*>(s.dst[d]) + off, acc);
    }
  }
}

// Mixed-width segments of the wide-partial reduce-scatter (bf16 payload): a helper
// summing bf16 slots into an fp32 partial (kFlagOutF32), and an owner adding its bf16 value
// and the fp32 partial (kFlagSrc1F32). 8 elements per step: one 16-byte bf16 vector or
// two 16-byte fp32 vectors per operand. Rare and optional, so one vector at a time.
__device__ __forceinline__ void unpack_f32x8(uint4 a, uint4 b, float* v) {
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
  v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}

// Whole tiles of the two mixed-width segment kinds, with the same batching as the main
// path (loads of a batch issued together). bf16 payload only: 8 elements per step.
template <int NSRC>
__device__ __forceinline__ void mixed_partial_full(const Seg& s, int64_t base) {
  // NSRC bf16 slots summed in order into an fp32 partial (no scale)
  constexpr int UB = NSRC <= 2 ? 4 : 2;
  const int64_t v0 = base / 8 + threadIdx.x;
#pragma unroll
  for (int u0 = 0; u0 < kUnroll; u0 += UB) {
    uint4 v[NSRC][UB];
#pragma unroll
    for (int u = 0; u < UB; ++u)
#pragma unroll
      for (int k = 0; k < NSRC; ++k)
        v[k][u] = Mem<false>::v4(static_cast<const uint4*>(s.src[k]) + v0 + (u0 + u) * kThreads);
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      float acc[8], t[8];
      TBF16::unpack(v[0][u], acc);
#pragma unroll
      for (int k = 1; k < NSRC; ++k) {
        TBF16::unpack(v[k][u], t);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], t[i]);
      }
      const uint4 lo = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                                  __float_as_uint(acc[2]), __float_as_uint(acc[3]));
      const uint4 hi = make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                  __float_as_uint(acc[6]), __float_as_uint(acc[7]));
      const int64_t q = 2 * (v0 + (u0 + u) * kThreads);
#pragma unroll
      for (int d = 0; d < kMaxDst; ++d)
        if (d < s.ndst) {
          st_v4(static_cast<uint4*>(s.dst[d]) + q, lo);
          st_v4(static_cast<uint4*>(s.dst[d]) + q + 1, hi);
        }
    }
  }
}

__device__ __forceinline__ void mixed_final_full(const Seg& s, int64_t base, float scale) {
  // a bf16 value plus an fp32 partial, scaled once, rounded to bf16
  const int64_t v0 = base / 8 + threadIdx.x;
  const bool do_scale = (s.flags & kFlagScale) != 0;
#pragma unroll
  for (int u0 = 0; u0 < kUnroll; u0 += 2) {
    uint4 x[2], p0[2], p1[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t vi = v0 + (u0 + u) * kThreads;
      x[u] = Mem<false>::v4(static_cast<const uint4*>(s.src[0]) + vi);
      p0[u] = Mem<false>::v4(static_cast<const uint4*>(s.src[1]) + 2 * vi);
      p1[u] = Mem<false>::v4(static_cast<const uint4*>(s.src[1]) + 2 * vi + 1);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float acc[8], t[8];
      TBF16::unpack(x[u], acc);
      unpack_f32x8(p0[u], p1[u], t);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], t[i]);
      if (do_scale) {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fmul_rn(acc[i], scale);
      }
      const uint4 r = TBF16::pack(acc);
      const int64_t vi = v0 + (u0 + u) * kThreads;
#pragma unroll
      for (int d = 0; d < kMaxDst; ++d)
        if (d < s.ndst) st_v4(static_cast<uint4*>(s.dst[d]) + vi, r);
    }
  }
}

template <class P>
__device__ __noinline__ void run_mixed_tile(const Seg& s, int64_t base, int64_t len, float scale) {
  const bool do_scale = (s.flags & kFlagScale) != 0;
  const bool out_f32 = (s.flags & kFlagOutF32) != 0;
  const bool src1_f32 = (s.flags & kFlagSrc1F32) != 0;
  int64_t done = 0;
  if (P::kE == 2 && (s.flags & kFlagVector)) {
    const int64_t vb = base / 8, nvec = len / 8;
#pragma unroll 1
    for (int64_t vi = threadIdx.x; vi < nvec; vi += kThreads) {
      float acc[8], t[8];
      TBF16::unpack(Mem<false>::v4(static_cast<const uint4*>(s.src[0]) + vb + vi), acc);
#pragma unroll 1
      for (int k = 1; k < s.nsrc; ++k) {
        if (k == 1 && src1_f32) {
          const uint4* q = static_cast<const uint4*>(s.src[1]) + 2 * (vb + vi);
          unpack_f32x8(Mem<false>::v4(q), Mem<false>::v4(q + 1), t);
        } else {
          TBF16::unpack(Mem<false>::v4(static_cast<const uint4*>(s.src[k]) + vb + vi), t);
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
          uint4* q = static_cast<uint4*>(s.dst[d]) + 2 * (vb + vi);
          st_v4(q, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]),
                              __float_as_uint(acc[2]), __float_as_uint(acc[3])));
          st_v4(q + 1, make_uint4(__float_as_uint(acc[4]), __float_as_uint(acc[5]),
                                  __float_as_uint(acc[6]), __float_as_uint(acc[7])));
        } else {
          st_v4(static_cast<uint4*>(s.dst[d]) + vb + vi, TBF16::pack(acc));
        }
      }
    }
    done = nvec * 8;
  }
#pragma unroll 1
  for (int64_t e = done + threadIdx.x; e < len; e += kThreads) {
    const int64_t i = base + e;
    float acc = TBF16::template load1<false>(static_cast<const char*>(s.src[0]) + i * 2);
#pragma unroll 1
    for (int k = 1; k < s.nsrc; ++k) {
      const float v = (k == 1 && src1_f32)
                          ? TF32::template load1<false>(static_cast<const char*>(s.src[1]) + i * 4)
                          : TBF16::template load1<false>(static_cast<const char*>(s.src[k]) + i * 2);
      acc = __fadd_rn(acc, v);
    }
    if (do_scale) acc = __fmul_rn(acc, scale);
#pragma unroll 1
    for (int d = 0; d < s.ndst; ++d) {
      if (out_f32) TF32::store1(static_cast<char*>(s.dst[d]) + i * 4, acc);
      else TBF16::store1(static_cast<char*>(s.dst[d]) + i * 2, acc);
    }
  }
}

// MODE selects the segments a launch runs: kModeMain (aligned and per-element paths),
// kModeRealign (realigned sources), kModeMixed (the main paths plus fp32 partials next to
// bf16, so that a pass with wide partials stays one launch). Each is its own kernel so
// that the rarer variants' register needs do not cost the main path occupancy. Main and
// mixed run 5 CTAs per SM (48 registers). The realign kernel runs 4 (64 registers): with
// its vectorized partial tiles it spilled at 48, and on GB300 the 4-CTA build ran 1 GiB
// all-to-alls as fast as the spill-free 5-CTA one without them, and misaligned 54-135 MiB
// all-to-alls 10-22% faster.
// kModeRealignAll runs a whole misaligned copy pass in one launch: its aligned copies take
// the realigning path with a zero shift. It runs 3 CTAs per SM (4 spilled) and is used only
// for passes of at most kRealignAllBytes: on GB300 the one launch ran a 54 MiB-per-rank
// misaligned all-to-all 14% faster than two, but 1 GiB ones 7% slower.
constexpr int kModeMain = 0, kModeRealign = 1, kModeMixed = 2, kModeRealignAll = 3,
              kModeStaged = 4;
constexpr int64_t kRealignAllBytes = 256ll << 20;

template <class P, int CAP, int MODE>
__global__ void __launch_bounds__(kThreads, MODE == kModeRealignAll ? 3 : MODE == kModeRealign ? 4 : 5)
    relay_pass_kernel(const __grid_constant__ PassArgs<CAP> args) {
  constexpr int64_t kTile = kTileBytes / P::kE;
  for (int t = blockIdx.x; t < args.ntiles; t += gridDim.x) {
    // last segment whose first tile is <= t (uniform across the CTA)
    int lo = 0, hi = args.nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (args.seg[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    const Seg& s = args.seg[lo];
    const int64_t base = (int64_t)(t - s.tile0) * kTile;
    const int64_t len = min(kTile, s.n - base);
    if (MODE == kModeMixed && seg_mixed(s)) {
      const bool full = P::kE == 2 && (s.flags & kFlagVector) && len == kTile;
      if (full && (s.flags & kFlagOutF32) && s.nsrc == 3 && s.ndst == 1) mixed_partial_full<3>(s, base);
      else if (full && (s.flags & kFlagOutF32) && s.nsrc == 2 && s.ndst == 1) mixed_partial_full<2>(s, base);
      else if (full && (s.flags & kFlagSrc1F32) && s.nsrc == 2) mixed_final_full(s, base, args.scale);
      else run_mixed_tile<P>(s, base, len, args.scale);
    }
    else if ((MODE == kModeMain || MODE == kModeMixed) && (s.flags & kFlagVector) && len == kTile)
      run_full_tile<P, false>(s, base, args.scale);
    else if (MODE == kModeRealign && len == kTile) run_realign_tile<P>(s, base, args.scale);
    else if (MODE == kModeRealign) run_realign_tail<P>(s, base, len, args.scale);
    else if (MODE == kModeRealignAll && (s.flags & kFlagRealign) && len == kTile)
      run_realign_tile<P>(s, base, args.scale);
    else if (MODE == kModeRealignAll && (s.flags & kFlagRealign))
      run_realign_tail<P>(s, base, len, args.scale);
    else run_partial_tile<P, false>(s, base, len, args.scale);
  }
}

// ------------------------------------------------- TMA-staged realignment kernel --
// A pass whose sources sit off the 16-byte grid (an all-to-all with an odd segmentCount, an
// odd recvCount) in one launch: per 16 KiB tile of destination, one thread bulk-copies the
// 16-byte blocks that hold the tile's source bytes into shared memory (cp.async.bulk, an
// mbarrier counting the bytes), and the CTA then funnel-shifts each vector out of two
// adjacent shared blocks and stores it 16-byte aligned. Copies and two-source reductions
// whose pointers are already aligned take the same path with a zero shift, so the whole
// pass is one launch. Data in flight sits in shared memory rather than registers, so the
// kernel runs 6 CTAs per SM where the register-realigning one ran 3-4.

// A tile's source bytes plus the block they spill into, per source.
constexpr uint32_t kStageBytes = (uint32_t)kTileBytes + 16;
// Bound of one mbarrier wait, in nanoseconds of the global timer. A bulk copy of 16 KiB
// lands in microseconds; a wait that runs out records a fault and gives up.
constexpr uint64_t kStageWaitNs = 200ull * 1000 * 1000;

// Set (bit 0) when a bounded wait of the staged kernel gave up; read and cleared on the
// host by relay_device_status().
__device__ unsigned g_relay_fault;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of the barrier, for at most `limit_ns`. False when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, unsigned parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(a));
  return r;
}

// The 16 bytes at shared byte offset sig + 16 v of a staged source.
__device__ __forceinline__ uint4 staged_vec(uint32_t base, unsigned sig, int v) {
  const uint4 lo = lds_v4(base + 16u * (uint32_t)v);
  return sig == 0 ? lo : shift_pair(lo, lds_v4(base + 16u * (uint32_t)(v + 1)), sig);
}

// One element of a staged source, widened like P::load1.
template <class P>
__device__ __forceinline__ typename P::Acc staged_elem(uint32_t a) {
  uint32_t w;
  if (P::kE == 4) {
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(a));
  } else {
    uint16_t h;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
    w = (uint32_t)h << 16;
  }
  if constexpr (std::is_same<typename P::Acc, float>::value) return __uint_as_float(w);
  else return (typename P::Acc)w;
}

template <class P, int CAP>
__global__ void __launch_bounds__(kThreads, 6) relay_staged_kernel(const __grid_constant__ PassArgs<CAP> args) {
  extern __shared__ __align__(16) unsigned char stage[];
  using Acc = typename P::Acc;
  constexpr int L = P::kLanes;
  constexpr int64_t kTile = kTileBytes / P::kE;
  // dynamic shared memory: one slot of kStageBytes per source (a launch of copies holds
  // one, of two-source reductions two); the barrier counting the copied bytes is static
  __shared__ __align__(8) uint64_t bar_word;
  const uint32_t bar = smem_u32(&bar_word);
  const uint32_t s0 = smem_u32(stage);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  unsigned phase = 0;
  for (int t = blockIdx.x; t < args.ntiles; t += gridDim.x, phase ^= 1u) {
    int lo = 0, hi = args.nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (args.seg[mid].tile0 <= t) lo = mid; else hi = mid - 1;
    }
    const Seg& s = args.seg[lo];
    const int64_t base = (int64_t)(t - s.tile0) * kTile;
    const int len = (int)min(kTile, s.n - base);
    const int nsrc = s.op == kOpCopy ? 1 : s.nsrc;
    unsigned sig[2] = {0u, 0u};
    uintptr_t a0[2] = {0, 0};
    uint32_t bytes[2] = {0u, 0u};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (k >= nsrc) break;
      // the 16-byte blocks holding the tile's source bytes
      const uintptr_t p = reinterpret_cast<uintptr_t>(s.src[k]) + (uintptr_t)(base * P::kE);
      sig[k] = (unsigned)(p & 15u);
      a0[k] = p & ~(uintptr_t)15;
      bytes[k] = (uint32_t)(((p + (uintptr_t)len * P::kE + 15) & ~(uintptr_t)15) - a0[k]);
    }
    if (threadIdx.x == 0) {
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                   "r"(bytes[0] + bytes[1] + (uint32_t)args.extra_tx)
                   : "memory");
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < nsrc)
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
                  "r"(s0 + (uint32_t)k * kStageBytes), "l"(a0[k]), "r"(bytes[k]), "r"(bar)
              : "memory");
    }
    const bool landed = mbar_wait_bounded(bar, phase, kStageWaitNs);
    if (__syncthreads_or(!landed)) {
      // a copy did not land in time: record it, give the copies one more bounded wait so
      // that nothing is still writing this CTA's shared memory, and leave (every thread)
      if (threadIdx.x == 0) atomicOr(&g_relay_fault, 1u);
      mbar_wait_bounded(bar, phase, kStageWaitNs);
      return;
    }
    const int nvec = len / L;
    const bool do_scale = (s.flags & kFlagScale) != 0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = (int)threadIdx.x + u * kThreads;
      if (v >= nvec) break;
      uint4 r = staged_vec(s0, sig[0], v);
      if (s.op != kOpCopy) {
        Acc acc[L], t2[L];
        P::unpack(r, acc);
        if (nsrc == 2) {
          P::unpack(staged_vec(s0 + kStageBytes, sig[1], v), t2);
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::add(acc[i], t2[i]);
        }
        if (do_scale) {
#pragma unroll
          for (int i = 0; i < L; ++i) acc[i] = P::scale(acc[i], args.scale);
        }
        r = P::pack(acc);
      }
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d)
        st_v4(reinterpret_cast<uint4*>(static_cast<char*>(s.dst[d]) + base * P::kE) + v, r);
    }
    // the last < L elements of a segment's final tile, one at a time from shared memory
    for (int e = nvec * L + (int)threadIdx.x; e < len; e += kThreads) {
      const uint32_t o0 = s0 + sig[0] + (uint32_t)(e * P::kE);
      if (s.op == kOpCopy) {
        if (P::kE == 4) {
          uint32_t x;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x) : "r"(o0));
#pragma unroll 1
          for (int d = 0; d < s.ndst; ++d) st_u32(static_cast<char*>(s.dst[d]) + (base + e) * P::kE, x);
        } else {
          uint16_t x;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(x) : "r"(o0));
#pragma unroll 1
          for (int d = 0; d < s.ndst; ++d) st_u16(static_cast<char*>(s.dst[d]) + (base + e) * P::kE, x);
        }
        continue;
      }
      Acc acc = staged_elem<P>(o0);
      if (nsrc == 2)
        acc = P::add(acc, staged_elem<P>(s0 + kStageBytes + sig[1] + (uint32_t)(e * P::kE)));
      if (do_scale) acc = P::scale(acc, args.scale);
#pragma unroll 1
      for (int d = 0; d < s.ndst; ++d) P::store1(static_cast<char*>(s.dst[d]) + (base + e) * P::kE, acc);
    }
    // every thread is done with this tile's shared bytes before the next copy lands there
    __syncthreads();
  }
}

// ----------------------------------------------------- fused small-call kernel --
// A whole call in one cooperative launch: the passes run one after another, separated
// by grid-wide barriers (every CTA takes part in every barrier: the pass loop is
// uniform). For calls small enough that the fixed cost of a launch per pass dominates.

constexpr int kMaxFusedPasses = 4;
// The one-launch kernel's tiles hold U vectors per thread: 4 (16 KiB), or 2 (8 KiB) for a
// call whose 16 KiB tiles number at most twice its grid, so that CTAs have a tile each.
// On GB300 8 KiB tiles took 4 MiB-per-rank 4-active calls 13-16% faster (allreduce 14.5 ->
// 12.6 us, reduce-scatter 12.4 -> 10.4 us) and made larger ones up to 14% slower.
constexpr int kFusedUnrollSmall = 2;
constexpr int kFusedCap = 384;  // 48 + 384 * 80 bytes of parameters, under the 32 KiB limit
// Calls with more segments than this fuse only when some of them need realigning (whose
// per-pass form costs a second launch per pass) and their traffic is at most
// kFusedManyBytes. On GB300 (CUDA-graph replays, warm L2) 4-active all-to-alls of 172
// segments (sizes are the workload count per rank; the input is a third of it) ran: aligned,
// 13.5 MiB, 14.5 us pass by pass and 16.5 us fused; misaligned, 13 MiB (55 MiB of
// traffic), 22.7 us either way in bf16 and 24.7 vs 22.7 us in int32; misaligned, 27 MiB
// (110 MiB of traffic), 30.8 vs 35.9 us; 54 MiB, 51.5 vs 70 us.
constexpr int kFusedPlainCap = 128;
constexpr int64_t kFusedManyBytes = 64ll << 20;

struct FusedArgs {
  int32_t npass;
  float scale;
  int32_t seg0[kMaxFusedPasses + 1];  // segments of pass p: [seg0[p], seg0[p+1])
  int32_t ntiles[kMaxFusedPasses];
  Seg seg[kFusedCap];                  // tile0 counts from the start of its pass
};

// 4 CTAs per SM (64 registers): with its realigning path the kernel spills at 48, and on
// GB300 the 4-CTA build was as fast or faster on every small call measured (a 16 MiB
// 2-active allreduce 22.7 -> 20.6 us).
template <class P, int U>
__global__ void __launch_bounds__(kThreads, 4) relay_fused_kernel(const __grid_constant__ FusedArgs args) {
  namespace cg = cooperative_groups;
  constexpr int64_t kTile = (int64_t)kThreads * U * kVecBytes / P::kE;
  for (int p = 0; p < args.npass; ++p) {
    for (int t = blockIdx.x; t < args.ntiles[p]; t += gridDim.x) {
      int lo = args.seg0[p], hi = args.seg0[p + 1] - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (args.seg[mid].tile0 <= t) lo = mid; else hi = mid - 1;
      }
      const Seg& s = args.seg[lo];
      const int64_t base = (int64_t)(t - s.tile0) * kTile;
      const int64_t len = min(kTile, s.n - base);
      if ((s.flags & kFlagVector) && len == kTile) run_full_tile<P, true, U>(s, base, args.scale);
      else if (s.flags & kFlagRealign) run_partial_realign_tile<P, true>(s, base, len, args.scale);
      else run_partial_tile<P, true>(s, base, len, args.scale);
    }
    if (p + 1 < args.npass) cg::this_grid().sync();
  }
}

// ------------------------------------------------------------------- host side --

// Split segments so that as much as possible takes a 16-byte path. When every pointer
// of a segment sits at the same offset modulo 16 bytes, that many bytes are peeled off
// the front as a per-element segment and the rest is vectorized. When only the
// destinations share an offset, the head is peeled so that they are aligned and the
// sources are realigned in registers. Destinations at different offsets leave the
// segment to the per-element path.
void split_for_alignment(const std::vector<Seg>& in, int E, std::vector<Seg>* out) {
  out->clear();
  out->reserve(in.size() + 8);
  auto mis = [](const void* p) { return (unsigned)(reinterpret_cast<uintptr_t>(p) & 15u); };
  for (const Seg& s0 : in) {
    Seg s = s0;
    s.flags &= ~(kFlagVector | kFlagRealign);
    const unsigned md = mis(s.dst[0]);
    bool dst_same = true, src_same = true;
    for (int d = 0; d < s.ndst; ++d) dst_same &= mis(s.dst[d]) == md;
    for (int k = 0; k < s.nsrc; ++k) src_same &= mis(s.src[k]) == md;
    if (!dst_same || md % E != 0) {
      out->push_back(s);
      continue;
    }
    const int64_t head = md == 0 ? 0 : std::min<int64_t>((16 - md) / E, s.n);
    if (head > 0) {
      Seg h = s;
      h.n = head;
      out->push_back(h);
      for (int k = 0; k < s.nsrc; ++k) s.src[k] = static_cast<const char*>(s.src[k]) + head * E;
      for (int d = 0; d < s.ndst; ++d) s.dst[d] = static_cast<char*>(s.dst[d]) + head * E;
      s.n -= head;
    }
    if (s.n > 0) {
      if (src_same) s.flags |= kFlagVector;
      else if (s.nsrc <= 2) s.flags |= kFlagRealign;
      out->push_back(s);
    }
  }
}


template <class P, int CAP, int MODE>
cudaError_t launch_cap(const Seg* segs, int nseg, float scale, cudaStream_t stream,
                       int max_ctas, int extra_tx = 0) {
  static thread_local PassArgs<CAP> a;  // up to ~30 KiB: keep it off the stack
  constexpr int64_t kTile = kTileBytes / P::kE;
  int64_t tiles = 0;
  int max_src = 1;
  for (int i = 0; i < nseg; ++i) {
    a.seg[i] = segs[i];
    a.seg[i].tile0 = (int32_t)tiles;
    tiles += (segs[i].n + kTile - 1) / kTile;
    if (segs[i].op != kOpCopy) max_src = std::max<int>(max_src, segs[i].nsrc);
  }
  if (tiles > INT32_MAX) return cudaErrorInvalidValue;
  a.nseg = nseg;
  a.ntiles = (int32_t)tiles;
  a.scale = scale;
  a.extra_tx = extra_tx;
  // one CTA per tile: the block scheduler starts a new tile on an SM the moment one of
  // its 5 resident CTAs finishes, which on GB300 streams ~11% faster than a persistent
  // grid walking the tiles (that grid's CTAs load, then store, tile after tile in step).
  // A capped grid (copies over the host link) walks the tiles instead.
  const int64_t want = max_ctas > 0 ? std::min<int64_t>(tiles, max_ctas) : tiles;
  const int grid = (int)std::max<int64_t>(1, want);
  if constexpr (MODE == kModeStaged) {
    if (max_src > 2) return cudaErrorInvalidValue;  // the staged kernel holds two sources
    relay_staged_kernel<P, CAP><<<grid, kThreads, (size_t)max_src * kStageBytes, stream>>>(a);
  } else {
    relay_pass_kernel<P, CAP, MODE><<<grid, kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

template <class P, int MODE>
cudaError_t launch_typed(const std::vector<Seg>& segs, float scale, cudaStream_t stream,
                         int max_ctas) {
  constexpr int kMaxCap = 384;  // 16 + 384 * 80 bytes of parameters, under the 32 KiB limit
  size_t i = 0;
  while (i < segs.size()) {
    const int n = (int)std::min<size_t>(segs.size() - i, kMaxCap);
    cudaError_t e;
    if (n <= 8) e = launch_cap<P, 8, MODE>(segs.data() + i, n, scale, stream, max_ctas);
    else if (n <= 32) e = launch_cap<P, 32, MODE>(segs.data() + i, n, scale, stream, max_ctas);
    else if (n <= 128) e = launch_cap<P, 128, MODE>(segs.data() + i, n, scale, stream, max_ctas);
    else e = launch_cap<P, kMaxCap, MODE>(segs.data() + i, n, scale, stream, max_ctas);
    if (e != cudaSuccess) return e;
    i += n;
  }
  return cudaSuccess;
}

// Resident CTAs per SM of the one-launch kernel on the current device (the cooperative
// grid must fit), cached per device.
template <class P, int U>
int fused_blocks_per_sm() {
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  if (dev >= 0 && dev < kMaxDevices && cached[dev] > 0) return cached[dev];
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, relay_fused_kernel<P, U>, kThreads, 0) !=
          cudaSuccess ||
      nb <= 0)
    nb = 1;
  if (dev >= 0 && dev < kMaxDevices) cached[dev] = nb;
  return nb;
}

bool cooperative_supported() {
  static int cached[kMaxDevices] = {0};  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  if (dev < kMaxDevices && cached[dev] != 0) return cached[dev] == 1;
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev);
  if (dev < kMaxDevices) cached[dev] = v ? 1 : 2;
  return v != 0;
}

// Fill the tile counts of `a` for tiles of U vectors per thread; returns the largest
// phase's tile count, or -1 if a count would overflow.
int fused_tiles(FusedArgs& a, int E, int U) {
  const int64_t tile = (int64_t)kThreads * U * kVecBytes / E;
  int max_tiles = 0;
  for (int p = 0; p < a.npass; ++p) {
    int64_t tiles = 0;
    for (int i = a.seg0[p]; i < a.seg0[p + 1]; ++i) {
      a.seg[i].tile0 = (int32_t)tiles;
      tiles += (a.seg[i].n + tile - 1) / tile;
    }
    if (tiles > INT32_MAX) return -1;
    a.ntiles[p] = (int32_t)tiles;
    max_tiles = std::max<int>(max_tiles, (int)tiles);
  }
  return max_tiles;
}

template <class P>
cudaError_t launch_fused_typed(FusedArgs& a, cudaStream_t stream, bool* ok) {
  *ok = true;
  const int64_t cap = (int64_t)sm_count() * fused_blocks_per_sm<P, kUnroll>();
  int max_tiles = fused_tiles(a, P::kE, kUnroll);
  int64_t total = 0;
  for (int p = 0; p < a.npass; ++p) total += a.ntiles[p];
  const bool small = total <= 2 * cap;
  if (small) max_tiles = fused_tiles(a, P::kE, kFusedUnrollSmall);
  if (max_tiles < 0) {
    *ok = false;
    return cudaSuccess;
  }
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, cap));
  void* params[] = {&a};
  const void* fn = small ? reinterpret_cast<const void*>(relay_fused_kernel<P, kFusedUnrollSmall>)
                         : reinterpret_cast<const void*>(relay_fused_kernel<P, kUnroll>);
  cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kThreads), params, 0, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int sm_count() {
  static int cached[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDevices && cached[dev] > 0) return cached[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices) cached[dev] = n;
  return n;
}

bool launch_fused(int dtype, const std::vector<Pass>& passes, float scale, cudaStream_t stream,
                  cudaError_t* err, bool forced) {
  *err = cudaSuccess;
  static thread_local std::vector<Pass> phases;
  fused_phases(passes, &phases);
  if (passes.size() < 2 || phases.size() > (size_t)kMaxFusedPasses || !cooperative_supported())
    return false;
  static thread_local FusedArgs a;
  static thread_local std::vector<Seg> segs;
  const int E = esize_of(dtype);
  int n = 0;
  bool realign = false;
  int64_t traffic = 0;
  a.npass = (int32_t)phases.size();
  a.scale = scale;
  for (size_t p = 0; p < phases.size(); ++p) {
    split_for_alignment(phases[p].segs, E, &segs);
    a.seg0[p] = n;
    for (const Seg& sg : segs) {
      if (seg_mixed(sg) || n >= kFusedCap) return false;
      realign |= (sg.flags & kFlagRealign) != 0;
      traffic += sg.n * E * (sg.nsrc + sg.ndst);
      a.seg[n++] = sg;
    }
  }
  if (!forced && n > kFusedPlainCap && (!realign || traffic > kFusedManyBytes)) return false;
  a.seg0[phases.size()] = n;
  bool ok = true;
  switch (dtype) {
    case RELAY_F32: *err = launch_fused_typed<TF32>(a, stream, &ok); break;
    case RELAY_BF16: *err = launch_fused_typed<TBF16>(a, stream, &ok); break;
    default: *err = launch_fused_typed<TI32>(a, stream, &ok); break;
  }
  return ok;
}

namespace {

template <class P>
cudaError_t launch_split(const std::vector<Seg>& direct, const std::vector<Seg>& realigned,
                         const std::vector<Seg>& mixed, float scale, cudaStream_t stream,
                         int max_ctas, bool staged) {
  cudaError_t e = cudaSuccess;
  bool realigned_reduce = false;
  for (const Seg& sg : realigned) realigned_reduce |= sg.op != kOpCopy;
  if (!realigned.empty() && staged && realigned_reduce) {
    // A pass with realigned reductions: the TMA-staged kernel takes the realigned segments
    // and, for a pass of at most kRealignAllBytes, also its aligned copies and one- or
    // two-source reductions (with a zero shift), so that such a pass is one launch; the
    // rest stay on the main kernel. On GB300 this ran an odd-count 2-active reduce-scatter
    // at 32 MB per rank 8-11% faster than the register-realigning kernel; passes of
    // realigned copies only (the all-to-all's pack and unpack) ran 3-30% slower staged at
    // 13.5-135 MB (a few waves each, where every CTA's barrier set-up and bulk-copy latency
    // shows) and level at 512 MB-1 GiB, so they keep the register path below.
    int64_t bytes = 0;
    for (const Seg& sg : direct) bytes += sg.n * P::kE * (sg.nsrc + sg.ndst);
    for (const Seg& sg : realigned) bytes += sg.n * P::kE * (sg.nsrc + sg.ndst);
    static thread_local std::vector<Seg> st, rest;
    st.assign(realigned.begin(), realigned.end());
    rest.clear();
    for (const Seg& sg : direct) {
      const bool fits = (sg.flags & kFlagVector) && (sg.op == kOpCopy || sg.nsrc <= 2);
      (fits && bytes <= kRealignAllBytes ? st : rest).push_back(sg);
    }
    if (!rest.empty()) e = launch_typed<P, kModeMain>(rest, scale, stream, max_ctas);
    if (e == cudaSuccess) e = launch_typed<P, kModeStaged>(st, scale, stream, max_ctas);
    if (e == cudaSuccess && !mixed.empty()) e = launch_typed<P, kModeMixed>(mixed, scale, stream, max_ctas);
    return e;
  }
  if (!realigned.empty() && !direct.empty()) {
    bool copies_only = true;
    int64_t bytes = 0;
    for (const Seg& sg : direct) {
      copies_only &= sg.op == kOpCopy;
      bytes += sg.n * P::kE * (sg.nsrc + sg.ndst);
    }
    for (const Seg& sg : realigned) bytes += sg.n * P::kE * (sg.nsrc + sg.ndst);
    if (copies_only && bytes <= kRealignAllBytes) {
      // one launch: an aligned copy is a realigned one with a zero shift
      static thread_local std::vector<Seg> all;
      all.assign(realigned.begin(), realigned.end());
      for (Seg sg : direct) {
        if (sg.flags & kFlagVector) sg.flags = (uint8_t)((sg.flags & ~kFlagVector) | kFlagRealign);
        all.push_back(sg);
      }
      return launch_typed<P, kModeRealignAll>(all, scale, stream, max_ctas);
    }
  }
  if (!direct.empty()) e = launch_typed<P, kModeMain>(direct, scale, stream, max_ctas);
  if (e == cudaSuccess && !realigned.empty())
    e = launch_typed<P, kModeRealign>(realigned, scale, stream, max_ctas);
  if (e == cudaSuccess && !mixed.empty()) e = launch_typed<P, kModeMixed>(mixed, scale, stream, max_ctas);
  return e;
}

}  // namespace

// Segments with realigned sources, and mixed-width segments, go to their own launches
// after the others; the launches of one pass touch disjoint memory, so their order does
// not matter.
cudaError_t launch_pass(int dtype, const Pass& pass, float scale, cudaStream_t stream,
                        int max_ctas, bool staged) {
  static thread_local std::vector<Seg> plain, segs, direct, realigned, mixed;
  plain.clear();
  mixed.clear();
  for (const Seg& sg : pass.segs) {
    if (!seg_mixed(sg)) {
      plain.push_back(sg);
      continue;
    }
    // only bf16 payloads widen, and every fp32 operand must be 4-byte aligned: never
    // launch anything else
    if (dtype != RELAY_BF16 || !seg_operands_aligned(sg, 2)) return cudaErrorInvalidValue;
    Seg m = sg;
    bool aligned = true;
    for (int k = 0; k < m.nsrc; ++k) aligned &= (reinterpret_cast<uintptr_t>(m.src[k]) & 15u) == 0;
    for (int d = 0; d < m.ndst; ++d) aligned &= (reinterpret_cast<uintptr_t>(m.dst[d]) & 15u) == 0;
    m.flags = (uint8_t)((m.flags & ~(kFlagVector | kFlagRealign)) | (aligned ? kFlagVector : 0));
    mixed.push_back(m);
  }
  split_for_alignment(plain, esize_of(dtype), &segs);
  direct.clear();
  realigned.clear();
  for (const Seg& sg : segs) (sg.flags & kFlagRealign ? realigned : direct).push_back(sg);
  if (!mixed.empty()) {
    // one launch for the pass: the mixed-mode kernel also runs the plain segments
    mixed.insert(mixed.end(), direct.begin(), direct.end());
    direct.clear();
  }
  switch (dtype) {
    case RELAY_F32: return launch_split<TF32>(direct, realigned, mixed, scale, stream, max_ctas, staged);
    case RELAY_BF16: return launch_split<TBF16>(direct, realigned, mixed, scale, stream, max_ctas, staged);
    default: return launch_split<TI32>(direct, realigned, mixed, scale, stream, max_ctas, staged);
  }
}

cudaError_t launch_staged_wait_test(void* dst, const void* src, int64_t count, int dtype,
                                    int extra_bytes, cudaStream_t stream) {
  Seg sg{};
  sg.src[0] = src;
  sg.dst[0] = dst;
  sg.n = count;
  sg.op = kOpCopy;
  sg.nsrc = sg.ndst = 1;
  switch (dtype) {
    case RELAY_F32: return launch_cap<TF32, 8, kModeStaged>(&sg, 1, 1.0f, stream, 0, extra_bytes);
    case RELAY_BF16: return launch_cap<TBF16, 8, kModeStaged>(&sg, 1, 1.0f, stream, 0, extra_bytes);
    default: return launch_cap<TI32, 8, kModeStaged>(&sg, 1, 1.0f, stream, 0, extra_bytes);
  }
}

cudaError_t read_device_fault(unsigned* fault) {
  // reads and clears the word (synchronous copies on the default stream)
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_relay_fault, sizeof *fault);
  if (e != cudaSuccess || *fault == 0) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_relay_fault, &zero, sizeof zero);
}

}  // namespace relay
