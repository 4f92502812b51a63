// plan.cpp -- schedule geometry of the sharded relay collectives (host, integers only).
//
// Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)" (torchrec pull
// request #4570). "item k" is item k of its summary; "Dnnnnnnnnn" a commit of its
// stack by Differential Revision number.
#include <string.h>

#include <limits>
#include <string>

#include "program.h"

namespace relay {
namespace {

constexpr int64_t kMiB = int64_t(1) << 20;

// chunk sizes are whole multiples of 128 elements (D115998394, D115998370)
inline int64_t align128(int64_t v) { return (v / RELAY_ALIGN_ELEMS) * RELAY_ALIGN_ELEMS; }

// Bytes of one active rank's input: the quantity the crossovers are quoted in
// (D115998363 sweeps the per-active-rank input size).
int64_t active_input_bytes(const relay_plan_t& p) { return p.input_elems * p.esize; }

// Default crossover, relay on (true) or pure-direct. Item 7: reduce-scatter A=2 relays
// from 2 MB; the A=4 reduce-scatter offload only pays past 48 MB; A=4 all-gather past
// 12 MB (fused). Item 4: a 2 MB pure-direct floor for the A=4 allreduce. The page has
// no figure for the A=2 allreduce full-exchange crossover (item 3), the A=2 all-gather
// and all-to-all, or the coalesced A=4 all-to-all; they take 2, 2, 2 and 12 MB.
bool default_relay(const relay_plan_t& p) {
  const int64_t b = active_input_bytes(p);
  if (p.A == 2) return b >= 2 * kMiB;
  if (p.coll == RELAY_ALLREDUCE) return b >= 2 * kMiB;
  if (p.coll == RELAY_REDUCE_SCATTER) return b > 48 * kMiB;
  return b > 12 * kMiB;
}

bool overflows(int64_t elems, int64_t factor, int esize) {
  const int64_t lim = std::numeric_limits<int64_t>::max() / 8;
  return elems > lim / factor / esize;
}

}  // namespace

relay_status_t make_plan(relay_coll_t coll, int64_t count, relay_dtype_t dtype, int A, int R,
                         const relay_opts_t* opts, relay_plan_t* out, std::string* why) {
  auto fail = [&](const char* msg) {
    if (why) *why = msg;
    return RELAY_ERR_INVALID_ARGUMENT;
  };
  if (out == nullptr) return fail("plan output pointer is NULL");
  memset(out, 0, sizeof *out);
  if (coll < RELAY_ALLREDUCE || coll > RELAY_ALL_TO_ALL) return fail("unknown collective");
  if (dtype < RELAY_F32 || dtype > RELAY_I32) return fail("unknown dtype");
  // D115998382: A in {2, 4}, at least one helper (local size > A)
  if (A != 2 && A != 4) return fail("A must be 2 or 4");
  if (R <= A) return fail("R must exceed A (at least one helper)");
  if (R > RELAY_MAX_RANKS) return fail("R exceeds RELAY_MAX_RANKS");
  if (count < 0) return fail("count does not fit int64");

  relay_opts_t o;
  relay_opts_init(&o);
  if (opts) o = *opts;
  const int permille = o.offload_permille < 0 ? 500 : o.offload_permille;
  if (permille > 1000) return fail("offload_permille must be in [0, 1000]");
  if (o.schedule < RELAY_SCHEDULE_AUTO || o.schedule > RELAY_SCHEDULE_LEGACY)
    return fail("unknown schedule request");

  relay_plan_t& p = *out;
  p.coll = coll;
  p.dtype = dtype;
  p.A = A;
  p.R = R;
  p.H = R - A;
  p.esize = esize_of(dtype);
  p.count = count;
  p.offload_permille = permille;

  const bool blocked_in = coll == RELAY_REDUCE_SCATTER || coll == RELAY_ALL_TO_ALL;
  const bool blocked_out = coll == RELAY_ALL_GATHER || coll == RELAY_ALL_TO_ALL;
  if (overflows(count, A * int64_t(1000), p.esize)) return fail("count too large");
  p.input_elems = blocked_in ? A * count : count;
  p.output_elems = blocked_out ? A * count : count;

  p.kind = RELAY_KIND_DIRECT;
  if (count == 0) return RELAY_OK;

  bool relay;
  switch (o.schedule) {
    case RELAY_SCHEDULE_RELAY:
    case RELAY_SCHEDULE_LEGACY: relay = true; break;
    case RELAY_SCHEDULE_DIRECT: relay = false; break;
    default:
      relay = o.relay_threshold_bytes >= 0 ? active_input_bytes(p) >= o.relay_threshold_bytes
                                           : default_relay(p);
  }
  const int H = p.H;
  const int64_t n = count;

  if (A == 2) {
    if (o.schedule == RELAY_SCHEDULE_LEGACY) {
      // item 1, before: numChunks = H+1; scatter, forward, then a separate direct
      // exchange of everything the relay chunks leave
      const int64_t c = align128(n / (H + 1));
      if (c == 0) return fail("legacy schedule needs a nonzero chunk");
      p.kind = RELAY_KIND_LEGACY;
      p.num_groups = 3;
      p.chunk = c;
      p.relay_total = H * c;
      p.dirA_offset = H * c;
      p.dirA_size = n - H * c;
      p.helper_elems = 2 * c;
    } else if (!relay) {
      // item 3: one full direct exchange, one group
      p.kind = RELAY_KIND_DIRECT;
      p.num_groups = 1;
      p.dirA_size = n;
    } else {
      // item 1: numChunks = H+2, one direct chunk rides each of the two relay groups
      const int64_t c = align128(n / (H + 2));
      p.num_groups = 2;
      if (c == 0) {
        // D115998367: direct halves over the active<->active link, no helper work
        p.kind = RELAY_KIND_ZERO_CHUNK;
        p.dirA_offset = 0;
        p.dirA_size = n / 2;
        p.dirB_size = n - n / 2;
      } else {
        p.kind = RELAY_KIND_RELAY;
        p.chunk = c;
        p.relay_total = H * c;
        p.dirA_offset = H * c;
        p.dirA_size = c;
        p.dirB_size = n - (H + 1) * c;
        p.helper_elems = 2 * c;  // one slot per active
      }
    }
    // what an active receives from the other active, staged for its reduction
    if (coll == RELAY_ALLREDUCE) {
      p.active_scratch_elems = n - p.relay_total;
      if (p.kind == RELAY_KIND_LEGACY) p.active_scratch_elems = n;
    } else if (coll == RELAY_REDUCE_SCATTER) {
      p.active_scratch_elems = n;
    }
    return RELAY_OK;
  }

  // A = 4
  if (o.schedule == RELAY_SCHEDULE_LEGACY) return fail("legacy schedule exists for A=2 only");
  int64_t oc = 0;
  if (relay) {
    if (coll == RELAY_ALL_TO_ALL) {
      // both groups' cross links carry (A-1)*oc; balancing them against the direct
      // links gives count/(2(A-1)+H) -- the geometry behind item 7's 1.67x model
      oc = align128(n / (2 * (A - 1) + H));
    } else {
      oc = align128((int64_t)permille * n / (1000 * (int64_t)H));
    }
  }
  p.kind = oc > 0 ? RELAY_KIND_RELAY : RELAY_KIND_DIRECT;
  p.chunk = oc;
  p.relay_total = H * oc;
  const int64_t pD = n - H * oc;
  p.direct_total = pD;
  switch (coll) {
    case RELAY_ALLREDUCE: {
      // item 4: direct region reduce-scattered to owners and all-gathered back, the
      // offload region reduced at helpers and broadcast; two groups either way
      p.num_groups = 2;
      p.owner_slice = align128(pD / A);
      p.owner_slice_last = pD - (A - 1) * p.owner_slice;
      p.helper_elems = A * oc;
      p.active_scratch_elems = (A - 1) * p.owner_slice_last;
      break;
    }
    case RELAY_REDUCE_SCATTER: {
      // item 6: flat reduce-at-helper; helper holds one chunk per (owner, source)
      if (oc == 0) {
        p.num_groups = 1;
        p.direct_g1 = pD;
      } else {
        p.num_groups = 2;
        p.direct_g1 = align128((A - 1) * pD / A);
        p.direct_g2 = pD - p.direct_g1;
      }
      p.helper_elems = (int64_t)A * (A - 1) * oc;
      p.active_scratch_elems = H * oc + (A - 1) * pD;
      // a bf16 partial crosses in fp32 unless the caller asks for the payload type; an
      // fp32 partial takes two bf16 elements of the owner's scratch
      if (!(o.flags & RELAY_FLAG_PAYLOAD_PARTIAL) && dtype == RELAY_BF16 && oc > 0) {
        p.wide_partial = 1;
        p.active_scratch_elems += H * oc + kWideSlackElems;
      }
      break;
    }
    case RELAY_ALL_GATHER: {
      // item 5: two balanced groups, direct region split 1:(A-1)
      if (oc == 0) {
        p.num_groups = 1;
        p.direct_g1 = pD;
      } else {
        p.num_groups = 2;
        p.direct_g1 = align128(pD / A);
        p.direct_g2 = pD - p.direct_g1;
      }
      p.helper_elems = A * oc;
      break;
    }
    default: {
      // item 7's open lead: helper sends coalesced per destination
      if (oc == 0) {
        p.num_groups = 1;
        p.direct_g1 = pD;
      } else {
        p.num_groups = 2;
        p.direct_g1 = (A - 1) * oc;
        p.direct_g2 = pD - p.direct_g1;
      }
      p.helper_elems = (int64_t)A * (A - 1) * oc;
      p.active_scratch_elems = (int64_t)H * (A - 1) * oc;
      break;
    }
  }
  return RELAY_OK;
}

}  // namespace relay
