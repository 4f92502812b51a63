/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Plain loops, one element at a time, no blocking and no reordering beyond what the
 * definitions state.  Built with -ffp-contract=off so that no multiply-add is fused.
 *
 * Citations name the page "Link-balance the sharded relay schedules (up to 3.2x vs
 * NCCL)" (torchrec pull request #4570): "Sk" = item k of its summary, "cost model" =
 * the paragraph before item 1, "Dnnnnnnnnn" = the commit of its stack with that
 * Differential Revision number.
 */
#include "oracle.h"

#include <string.h>

/* ======================================================================= */
/* bfloat16                                                                 */
/* ======================================================================= */

/* IEEE-754 round-to-nearest, ties-to-even, from binary32 to bfloat16.  bfloat16 is
 * the upper half of a binary32 (sign, 8 exponent bits, 7 fraction bits).  The lower
 * 16 bits are the discarded tail: above half an ulp rounds up, below rounds down, and
 * exactly half rounds to the neighbour whose last kept bit is 0.  A carry out of the
 * fraction correctly bumps the exponent (up to infinity).  NaN stays NaN (quiet bit
 * set so that the truncation cannot turn it into infinity). */
uint16_t orc_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u) {
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  uint32_t kept = u >> 16;
  uint32_t tail = u & 0xffffu;
  if (tail > 0x8000u || (tail == 0x8000u && (kept & 1u) != 0u)) {
    kept += 1u;
  }
  return (uint16_t)kept;
}

float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

void orc_bf16_rne_array(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(in[i]);
}

/* ======================================================================= */
/* element access                                                           */
/* ======================================================================= */

static float load_f(int dtype, const void* base, int64_t i) {
  if (dtype == ORC_F32) return ((const float*)base)[i];
  return orc_bf16_to_f32(((const uint16_t*)base)[i]);
}

/* Q: the value as it is stored in (and carried over a link in) the payload type */
static float quantize(int dtype, float v) {
  if (dtype == ORC_BF16) return orc_bf16_to_f32(orc_bf16_rne(v));
  return v;
}

static void store_q(int dtype, void* base, int64_t i, float v) {
  if (dtype == ORC_F32) {
    ((float*)base)[i] = v;
  } else {
    ((uint16_t*)base)[i] = orc_bf16_rne(v);
  }
}

/* ======================================================================= */
/* collective semantics                                                     */
/* ======================================================================= */

/* Allreduce (S2, D115998369): every active rank ends with scale * sum over the A
 * actives of their inputs; SUM is scale 1 and AVG is scale 1/A (D115998376).
 *   ref64: the sum accumulated in double, times scale  (fp32 tolerance reference)
 *   ref32: the sum accumulated in float in ascending rank order, times scale in float
 *   refq : ref32 stored in the payload type (RNE for bf16); int32 sums wrap. */
void orc_allreduce(int dtype, int A, const void* const* x, int64_t i0, int64_t i1,
                   float scale, double* ref64, float* ref32, void* refq) {
  for (int64_t i = i0; i < i1; ++i) {
    int64_t o = i - i0;
    if (dtype == ORC_I32) {
      uint32_t acc = 0u;
      int64_t exact = 0;
      for (int k = 0; k < A; ++k) {
        int32_t v = ((const int32_t*)x[k])[i];
        acc += (uint32_t)v;
        exact += v;
      }
      if (ref64) ref64[o] = (double)exact;
      if (ref32) ref32[o] = (float)exact;
      if (refq) ((int32_t*)refq)[o] = (int32_t)acc;
      continue;
    }
    /* the sums start from their first term, as IEEE addition of the terms would
     * (a sum of negative zeros stays -0) */
    double acc64 = (double)load_f(dtype, x[0], i);
    float acc32 = load_f(dtype, x[0], i);
    for (int k = 1; k < A; ++k) {
      float v = load_f(dtype, x[k], i);
      acc64 += (double)v;
      acc32 = acc32 + v;
    }
    float r32 = acc32 * scale;
    if (ref64) ref64[o] = acc64 * (double)scale;
    if (ref32) ref32[o] = r32;
    if (refq) store_q(dtype, refq, o, r32);
  }
}

/* Reduce-scatter (D115998376): each active's input holds A blocks of m elements,
 * block k destined for active k; owner o ends with scale * sum over sources s of
 * block o of x_s.
 *
 * helper_span > 0 restates the 4-active flat reduce-at-helper (S6): positions
 * [0, helper_span) of every block are summed at a helper over the A-1 non-owner
 * sources, and that partial travels back to the owner as ONE payload-typed chunk
 * (A-1 chunks come in, one goes out), so it is rounded to the payload type before
 * the owner adds its own contribution and applies the scale.  Positions past helper_span are
 * reduced at the owner from all A sources, ascending. */
static void reduce_scatter_impl(int dtype, int A, const void* const* x, int64_t m, int owner,
                                int64_t i0, int64_t i1, float scale, int64_t helper_span,
                                int round_partial, double* ref64, float* ref32, void* refq) {
  for (int64_t i = i0; i < i1; ++i) {
    int64_t o = i - i0;
    int64_t p = (int64_t)owner * m + i;
    if (dtype == ORC_I32) {
      uint32_t acc = 0u;
      int64_t exact = 0;
      for (int k = 0; k < A; ++k) {
        int32_t v = ((const int32_t*)x[k])[p];
        acc += (uint32_t)v;
        exact += v;
      }
      if (ref64) ref64[o] = (double)exact;
      if (ref32) ref32[o] = (float)exact;
      if (refq) ((int32_t*)refq)[o] = (int32_t)acc;
      continue;
    }
    double acc64 = (double)load_f(dtype, x[0], p);
    for (int k = 1; k < A; ++k) acc64 += (double)load_f(dtype, x[k], p);
    float acc32;
    if (i < helper_span) {
      int first = owner == 0 ? 1 : 0;
      float partial = load_f(dtype, x[first], p);
      for (int s = first + 1; s < A; ++s) {
        if (s == owner) continue;
        partial = partial + load_f(dtype, x[s], p);
      }
      if (round_partial) partial = quantize(dtype, partial);
      acc32 = load_f(dtype, x[owner], p) + partial;
    } else {
      acc32 = load_f(dtype, x[0], p);
      for (int s = 1; s < A; ++s) acc32 = acc32 + load_f(dtype, x[s], p);
    }
    float r32 = acc32 * scale;
    if (ref64) ref64[o] = acc64 * (double)scale;
    if (ref32) ref32[o] = r32;
    if (refq) store_q(dtype, refq, o, r32);
  }
}

void orc_reduce_scatter(int dtype, int A, const void* const* x, int64_t m, int owner,
                        int64_t i0, int64_t i1, float scale, int64_t helper_span,
                        double* ref64, float* ref32, void* refq) {
  reduce_scatter_impl(dtype, A, x, m, owner, i0, i1, scale, helper_span, 1, ref64, ref32, refq);
}

/* The same flat reduce-at-helper with the helper's partial carried back in fp32 instead
 * of the payload type (a reading the page leaves open: it does not state the precision
 * of the returned chunk).  The owner still adds its own value first, then the partial. */
void orc_reduce_scatter_wide(int dtype, int A, const void* const* x, int64_t m, int owner,
                             int64_t i0, int64_t i1, float scale, int64_t helper_span,
                             double* ref64, float* ref32, void* refq) {
  reduce_scatter_impl(dtype, A, x, m, owner, i0, i1, scale, helper_span, 0, ref64, ref32, refq);
}

/* All-gather (D115998385): every active's output is the A inputs of S elements laid
 * end to end in rank order. */
void orc_all_gather(int esize, int A, const void* const* x, int64_t S, void* out) {
  for (int k = 0; k < A; ++k) {
    const unsigned char* src = (const unsigned char*)x[k];
    unsigned char* dst = (unsigned char*)out + (int64_t)k * S * esize;
    for (int64_t b = 0; b < S * esize; ++b) dst[b] = src[b];
  }
}

/* All-to-all (D115998370): input of s is A segments, segment d destined for d;
 * output of d is A segments, segment s received from s. */
void orc_all_to_all(int esize, int A, const void* const* x, int64_t seg, int dst, void* out) {
  for (int s = 0; s < A; ++s) {
    const unsigned char* src = (const unsigned char*)x[s] + (int64_t)dst * seg * esize;
    unsigned char* o = (unsigned char*)out + (int64_t)s * seg * esize;
    for (int64_t b = 0; b < seg * esize; ++b) o[b] = src[b];
  }
}

/* ======================================================================= */
/* planner restatement                                                      */
/* ======================================================================= */

/* chunk sizes are aligned down to 128 elements (D115998394, D115998370) */
int64_t orc_align_down(int64_t x) { return x - x % 128; }

#define MB (1024LL * 1024LL)

/* Per-active-rank input bytes, the quantity every crossover is stated in (D115998363:
 * the swept size is the per-active-rank input). */
static int64_t input_bytes(int coll, int A, int64_t count, int esize) {
  if (coll == ORC_RS || coll == ORC_A2A) return (int64_t)A * count * esize;
  return count * esize;
}

/* Default crossovers.  S7: reduce-scatter A=2 fused relays from 2 MB; A=4
 * reduce-scatter offload only past 48 MB; A=4 all-gather past 12 MB (fused).  S4: A=4
 * allreduce 2 MB pure-direct floor.  The page gives no value for the A=2 allreduce
 * full-exchange crossover (S3), the A=2 all-gather / all-to-all paths, or the A=4
 * all-to-all relay; these take 2 MB, 2 MB and 12 MB (readings). */
static int wants_relay(int coll, int A, int64_t bytes) {
  if (A == 2) return bytes >= 2 * MB;
  switch (coll) {
    case ORC_AR: return bytes >= 2 * MB;
    case ORC_RS: return bytes > 48 * MB;
    case ORC_AG: return bytes > 12 * MB;
    default: return bytes > 12 * MB;
  }
}

int orc_plan(int coll, int A, int R, int64_t count, int esize, int permille, int force,
             int64_t* g) {
  for (int i = 0; i < ORC_G_NFIELDS; ++i) g[i] = 0;
  if (A != 2 && A != 4) return -1;
  if (R <= A || count < 0 || coll < 0 || coll > 3) return -1;
  if (esize != 2 && esize != 4) return -1;
  if (permille < 0 || permille > 1000) return -1;
  int H = R - A;
  g[ORC_G_COLL] = coll;
  g[ORC_G_A] = A;
  g[ORC_G_R] = R;
  g[ORC_G_H] = H;
  g[ORC_G_ESIZE] = esize;
  g[ORC_G_COUNT] = count;
  g[ORC_G_KIND] = ORC_KIND_DIRECT;
  if (count == 0) return 0;

  int relay;
  if (force == ORC_FORCE_RELAY || force == ORC_FORCE_LEGACY) relay = 1;
  else if (force == ORC_FORCE_DIRECT) relay = 0;
  else relay = wants_relay(coll, A, input_bytes(coll, A, count, esize));

  int64_t n = count;
  if (A == 2) {
    if (force == ORC_FORCE_LEGACY) {
      /* S1, before: numChunks = H+1, three serialized groups -- scatter, forward,
       * then a separate active<->active exchange of what the relay chunks leave. */
      int64_t c = orc_align_down(n / (H + 1));
      if (c == 0) return -1;
      g[ORC_G_KIND] = ORC_KIND_LEGACY;
      g[ORC_G_GROUPS] = 3;
      g[ORC_G_CHUNK] = c;
      g[ORC_G_DIRA_OFF] = (int64_t)H * c;
      g[ORC_G_DIRA] = n - (int64_t)H * c;
      g[ORC_G_DIRB] = 0;
      return 0;
    }
    if (!relay) {
      /* S3: below the crossover one full direct exchange (one group). */
      g[ORC_G_KIND] = ORC_KIND_DIRECT;
      g[ORC_G_GROUPS] = 1;
      g[ORC_G_DIRA] = n;
      return 0;
    }
    /* S1: numChunks = H+2; relay chunk h goes to helper h; one direct chunk rides
     * each of the two relay groups; the second direct region absorbs the remainder. */
    int64_t c = orc_align_down(n / (H + 2));
    g[ORC_G_GROUPS] = 2;
    if (c == 0) {
      /* D115998367: chunk aligned down to zero -> dirA takes half, dirB the rest,
       * both over the active<->active link; no helper work. */
      g[ORC_G_KIND] = ORC_KIND_ZERO_CHUNK;
      g[ORC_G_DIRA] = n / 2;
      g[ORC_G_DIRA_OFF] = 0;
      g[ORC_G_DIRB] = n - n / 2;
      return 0;
    }
    g[ORC_G_KIND] = ORC_KIND_RELAY;
    g[ORC_G_CHUNK] = c;
    g[ORC_G_DIRA_OFF] = (int64_t)H * c;
    g[ORC_G_DIRA] = c;
    g[ORC_G_DIRB] = n - (int64_t)(H + 1) * c;
    return 0;
  }

  /* A = 4 */
  if (force == ORC_FORCE_LEGACY) return -1;
  int64_t oc = 0;
  if (relay) {
    if (coll == ORC_A2A) {
      /* offload geometry that balances both groups' cross links ((A-1)*oc per group)
       * against the intra links (d1, d2); reproduces the 1.67x that item 7's link
       * model predicted */
      oc = orc_align_down(n / (2 * (A - 1) + H));
    } else {
      /* S4: offload fraction in permille of the region, split evenly over helpers */
      oc = orc_align_down((permille * n) / (1000LL * H));
    }
  }
  g[ORC_G_CHUNK] = oc;
  g[ORC_G_KIND] = oc > 0 ? ORC_KIND_RELAY : ORC_KIND_DIRECT;
  int64_t pD = n - (int64_t)H * oc;
  g[ORC_G_PD] = pD;
  switch (coll) {
    case ORC_AR: {
      /* S4: direct region reduce-scattered over owners then all-gathered; offload
       * region reduced at helpers and broadcast.  Two groups either way. */
      int64_t s = orc_align_down(pD / A);
      g[ORC_G_OWNER_SLICE] = s;
      g[ORC_G_OWNER_LAST] = pD - (int64_t)(A - 1) * s;
      g[ORC_G_GROUPS] = 2;
      break;
    }
    case ORC_RS:
      if (oc == 0) {
        g[ORC_G_D1] = pD;
        g[ORC_G_GROUPS] = 1;
      } else {
        /* S6: direct part split so that G1's intra links balance the (A-1)*oc cross
         * load and G2's the single returned chunk */
        g[ORC_G_D1] = orc_align_down(((int64_t)(A - 1) * pD) / A);
        g[ORC_G_D2] = pD - g[ORC_G_D1];
        g[ORC_G_GROUPS] = 2;
      }
      break;
    case ORC_AG:
      if (oc == 0) {
        g[ORC_G_D1] = pD;
        g[ORC_G_GROUPS] = 1;
      } else {
        /* S5: direct region split 1:(A-1) across the two groups */
        g[ORC_G_D1] = orc_align_down(pD / A);
        g[ORC_G_D2] = pD - g[ORC_G_D1];
        g[ORC_G_GROUPS] = 2;
      }
      break;
    default:
      if (oc == 0) {
        g[ORC_G_D1] = pD;
        g[ORC_G_GROUPS] = 1;
      } else {
        g[ORC_G_D1] = (int64_t)(A - 1) * oc;
        g[ORC_G_D2] = pD - g[ORC_G_D1];
        g[ORC_G_GROUPS] = 2;
      }
      break;
  }
  return 0;
}

static void add(uint64_t* t, int R, int grp, int s, int d, int64_t v) {
  t[((int64_t)grp * R + s) * R + d] += (uint64_t)v;
}

/* Cost model: a group's time is the most any (link, direction) carries in it; the
 * schedule's time is the sum over its serialized groups.  This enumerates what each
 * (group, sender, receiver) carries, straight from the schedules as the page states
 * them.  Ranks 0..A-1 are the actives, A+h is helper h (D115998382: actives are
 * consecutive local ranks). */
int orc_link_elems(const int64_t* g, uint64_t* t, int64_t cap) {
  int coll = (int)g[ORC_G_COLL], A = (int)g[ORC_G_A], R = (int)g[ORC_G_R];
  int H = (int)g[ORC_G_H], G = (int)g[ORC_G_GROUPS], kind = (int)g[ORC_G_KIND];
  if ((int64_t)G * R * R > cap) return -1;
  for (int64_t i = 0; i < (int64_t)G * R * R; ++i) t[i] = 0;
  if (G == 0) return 0;
  int64_t n = g[ORC_G_COUNT], c = g[ORC_G_CHUNK];

  if (A == 2) {
    for (int a = 0; a < 2; ++a) {
      int other = 1 - a;
      if (kind == ORC_KIND_DIRECT) {
        add(t, R, 0, a, other, n);
      } else if (kind == ORC_KIND_LEGACY) {
        for (int h = 0; h < H; ++h) {
          add(t, R, 0, a, A + h, c);    /* scatter */
          add(t, R, 1, A + h, a, c);    /* forward */
        }
        add(t, R, 2, a, other, g[ORC_G_DIRA]);  /* separate direct exchange */
      } else {
        if (kind == ORC_KIND_RELAY) {
          for (int h = 0; h < H; ++h) {
            add(t, R, 0, a, A + h, c);  /* G1: chunk h to helper h */
            add(t, R, 1, A + h, a, c);  /* G2: one chunk back to each active */
          }
        }
        add(t, R, 0, a, other, g[ORC_G_DIRA]);  /* direct chunk riding G1 */
        add(t, R, 1, a, other, g[ORC_G_DIRB]);  /* direct chunk riding G2 */
      }
    }
    return G;
  }

  int64_t d1 = g[ORC_G_D1], d2 = g[ORC_G_D2];
  for (int s = 0; s < A; ++s) {
    for (int h = 0; h < H && c > 0; ++h) {
      switch (coll) {
        case ORC_AR:
          add(t, R, 0, s, A + h, c);    /* slice h of the offload region */
          add(t, R, 1, A + h, s, c);    /* reduced slice broadcast back */
          break;
        case ORC_RS:
          add(t, R, 0, s, A + h, (int64_t)(A - 1) * c);  /* slice h of each non-own block */
          add(t, R, 1, A + h, s, c);                     /* one reduced chunk to the owner */
          break;
        case ORC_AG:
          add(t, R, 0, s, A + h, c);
          add(t, R, 1, A + h, s, (int64_t)(A - 1) * c);  /* the other sources' slice h */
          break;
        default:
          add(t, R, 0, s, A + h, (int64_t)(A - 1) * c);  /* coalesced per helper */
          add(t, R, 1, A + h, s, (int64_t)(A - 1) * c);  /* coalesced per destination */
          break;
      }
    }
    for (int d = 0; d < A; ++d) {
      if (d == s) continue;
      if (coll == ORC_AR) {
        int64_t len_d = (d == A - 1) ? g[ORC_G_OWNER_LAST] : g[ORC_G_OWNER_SLICE];
        int64_t len_s = (s == A - 1) ? g[ORC_G_OWNER_LAST] : g[ORC_G_OWNER_SLICE];
        add(t, R, 0, s, d, len_d);  /* s sends owner d its direct slice */
        add(t, R, 1, s, d, len_s);  /* owner s returns its reduced slice */
      } else {
        add(t, R, 0, s, d, d1);
        if (G > 1) add(t, R, 1, s, d, d2);
      }
    }
  }
  return G;
}

uint64_t orc_cost_elems(const int64_t* g) {
  int R = (int)g[ORC_G_R];
  int G = (int)g[ORC_G_GROUPS];
  static uint64_t t[3 * 64 * 64];
  if (R > 64 || orc_link_elems(g, t, 3 * 64 * 64) < 0) return 0;
  uint64_t total = 0;
  for (int grp = 0; grp < G; ++grp) {
    uint64_t mx = 0;
    for (int s = 0; s < R; ++s)
      for (int d = 0; d < R; ++d) {
        uint64_t v = t[((int64_t)grp * R + s) * R + d];
        if (v > mx) mx = v;
      }
    total += mx;
  }
  return total;
}

/* ======================================================================= */
/* helper-buffer contracts                                                  */
/* ======================================================================= */

/* The passthrough helper size (D115998394, D115998388, D115998370):
 * min(count_g, A * align_down(count_g / num_chunks, 128)) -- A slots, each a whole
 * number of 128-element chunks.  Below one chunk the page only says the fallback
 * errs only towards allocating too much; this returns count_g there (a reading). */
int64_t orc_passthrough_helper_size(int64_t count_g, int A, int num_chunks) {
  int64_t c = orc_align_down(count_g / num_chunks);
  if (c == 0) return count_g;
  int64_t s = (int64_t)A * c;
  return s < count_g ? s : count_g;
}

/* Helper contracts at A > 2: 2*recvCount for reduce-scatter (S6, D115998367),
 * 2*total for allreduce (D115998382), A*send_count for all-gather (D115998397), a
 * size-1 placeholder for the pure-direct all-to-all (D115998358).  A = 2 uses the
 * passthrough size with num_chunks = (R - A) + 1, i.e. 7 on an 8-rank node
 * (D115998370). */
int64_t orc_relay_helper_contract(int coll, int A, int R, int64_t count) {
  if (A == 2) return orc_passthrough_helper_size(count, 2, (R - A) + 1);
  switch (coll) {
    case ORC_RS: return 2 * count;
    case ORC_AR: return 2 * count;
    case ORC_AG: return (int64_t)A * count;
    default: return 1;
  }
}
