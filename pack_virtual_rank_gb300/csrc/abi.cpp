// abi.cpp -- the extern "C" entry points declared in relay.h: validation, planning,
// the link-byte accountant, and the pass-by-pass execution of a collective.
//
// Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)" (torchrec pull
// request #4570): "item k" of its summary, "Dnnnnnnnnn" a commit of its stack.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <string>
#include <vector>

#include "program.h"

namespace relay {
namespace {

thread_local std::string g_last_error;
thread_local std::string g_last_launch = "none";

relay_status_t fail(relay_status_t st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

// Fake, widely spaced, 256-byte aligned buffer addresses: enough to build a program
// whose segment lengths and ranks can be counted without touching memory.
struct FakeBuffers {
  std::vector<void*> send, recv, scratch;
  FakeBuffers(const relay_plan_t& p, bool in_place, int salt = 0) {
    send.resize(p.R);
    recv.resize(p.R);
    scratch.resize(p.R);
    for (int r = 0; r < p.R; ++r) {
      auto base = [&](int k) {
        return reinterpret_cast<void*>(((uintptr_t)(4 * r + k + 1) << 42) +
                                       ((uintptr_t)salt << 36));
      };
      send[r] = base(0);
      recv[r] = base(1);
      scratch[r] = base(2);
      if (in_place && r < p.A) {
        const int64_t E = p.esize;
        switch (p.coll) {
          case RELAY_ALLREDUCE: recv[r] = send[r]; break;
          case RELAY_REDUCE_SCATTER: recv[r] = (char*)send[r] + r * p.count * E; break;
          case RELAY_ALL_GATHER: send[r] = (char*)recv[r] + r * p.count * E; break;
          default: break;
        }
      }
    }
  }
  Buffers view() const { return Buffers{send.data(), recv.data(), scratch.data()}; }
};

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
  std::string what;
  bool scratch = false;  // a scratch buffer of the call (its contents afterwards: unspecified)
};

bool overlaps(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

// Two segments of one launch must not write what the other reads or writes: nothing
// orders CTAs within a launch.
bool find_hazard(const Pass& pass, int E, std::string* why) {
  const auto& s = pass.segs;
  auto rng = [&](const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + (uintptr_t)bytes, ""};
  };
  for (size_t i = 0; i < s.size(); ++i)
    for (int d = 0; d < s[i].ndst; ++d) {
      const Range w = rng(s[i].dst[d], seg_dst_bytes(s[i], E));
      for (size_t j = 0; j < s.size(); ++j) {
        if (j == i) continue;
        for (int k = 0; k < s[j].nsrc; ++k)
          if (overlaps(w, rng(s[j].src[k], seg_src_bytes(s[j], k, E)))) {
            *why = "segment " + std::to_string(i) + " writes what segment " + std::to_string(j) +
                   " reads in pass " + relay_pass_name(pass.kind);
            return true;
          }
        for (int k = 0; k < s[j].ndst; ++k)
          if (overlaps(w, rng(s[j].dst[k], seg_dst_bytes(s[j], E)))) {
            *why = "segments " + std::to_string(i) + " and " + std::to_string(j) +
                   " write the same bytes in pass " + relay_pass_name(pass.kind);
            return true;
          }
      }
    }
  return false;
}

// Every range a segment reads or writes must lie inside one declared buffer.
bool find_out_of_bounds(const Pass& pass, int E, const std::vector<Range>& bufs,
                        std::string* why) {
  auto inside = [&](const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p), hi = lo + (uintptr_t)bytes;
    for (const Range& b : bufs)
      if (lo >= b.lo && hi <= b.hi) return true;
    return false;
  };
  for (size_t i = 0; i < pass.segs.size(); ++i) {
    const Seg& s = pass.segs[i];
    bool ok = true;
    for (int k = 0; k < s.nsrc; ++k) ok &= inside(s.src[k], seg_src_bytes(s, k, E));
    for (int d = 0; d < s.ndst; ++d) ok &= inside(s.dst[d], seg_dst_bytes(s, E));
    if (!ok) {
      *why = "segment " + std::to_string(i) + " of pass " + relay_pass_name(pass.kind) +
             " leaves the declared buffers";
      return true;
    }
    if (!seg_operands_aligned(s, E)) {
      *why = "segment " + std::to_string(i) + " of pass " + relay_pass_name(pass.kind) +
             " has an operand not aligned to its element width";
      return true;
    }
  }
  return false;
}

// Validate one group's buffers (R local entries: actives first, then its helpers) and
// append their ranges. In-place forms are recognised and not counted twice.
relay_status_t validate_group(const relay_plan_t& p, void* const* send, void* const* recv,
                              void* const* scratch, const int* global_rank,
                              std::vector<Range>* ranges) {
  const int A = p.A;
  const int64_t E = p.esize;
  auto name = [&](const char* what, int local) {
    return std::string(what) + "[" + std::to_string(global_rank[local]) + "]";
  };
  auto add = [&](const void* ptr, int64_t elems, const std::string& what) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(ptr);
    ranges->push_back(Range{lo, lo + (uintptr_t)(elems * E), what});
  };
  for (int a = 0; a < A; ++a) {
    if (send[a] == nullptr || recv[a] == nullptr)
      return fail(RELAY_ERR_INVALID_ARGUMENT, "active " + name("rank", a) + ": send/recv is NULL");
    if ((reinterpret_cast<uintptr_t>(send[a]) | reinterpret_cast<uintptr_t>(recv[a])) % E)
      return fail(RELAY_ERR_INVALID_ARGUMENT,
                  "active " + name("rank", a) + ": buffer not element-aligned");
    const char* s = static_cast<const char*>(send[a]);
    const char* r = static_cast<const char*>(recv[a]);
    bool send_in_recv = false, recv_in_send = false;
    switch (p.coll) {
      case RELAY_ALLREDUCE: recv_in_send = r == s; break;                          // D115998369
      case RELAY_REDUCE_SCATTER: recv_in_send = r == s + a * p.count * E; break;  // D115998376
      case RELAY_ALL_GATHER: send_in_recv = s == r + a * p.count * E; break;      // D115998385
      default: break;                                                               // D115998370
    }
    if (!send_in_recv) add(send[a], p.input_elems, name("send", a));
    if (!recv_in_send) add(recv[a], p.output_elems, name("recv", a));
  }
  for (int l = 0; l < p.R; ++l) {
    const int64_t need = l < A ? p.active_scratch_elems : p.helper_elems;
    if (need <= 0) continue;
    if (scratch[l] == nullptr)
      return fail(RELAY_ERR_INVALID_ARGUMENT,
                  std::string(l < A ? "active " : "helper ") + name("rank", l) + " needs scratch");
    if (reinterpret_cast<uintptr_t>(scratch[l]) % E)
      return fail(RELAY_ERR_INVALID_ARGUMENT, name("scratch", l) + " not element-aligned");
    add(scratch[l], need, name("scratch", l));
    ranges->back().scratch = true;
  }
  return RELAY_OK;
}

relay_status_t check_disjoint(const std::vector<Range>& ranges) {
  for (size_t i = 0; i < ranges.size(); ++i)
    for (size_t j = i + 1; j < ranges.size(); ++j)
      if (overlaps(ranges[i], ranges[j]))
        return fail(RELAY_ERR_INVALID_ARGUMENT,
                    ranges[i].what + " overlaps " + ranges[j].what + " (not an in-place form)");
  return RELAY_OK;
}

// The chained-launch analysis of the last few distinct programs this thread ran, keyed by
// the exact bytes of their segment tables: a call repeated on the same buffers (the usual
// case) skips the analysis, which costs more host time than a small call's kernel.
struct ChainMemo {
  std::vector<unsigned char> key;
  std::vector<ByteRange> scratch;  // the scratch whose dead lines the plan drops
  ChainPlan plan;
  bool ok = false;
  bool checked = false;
  std::string why;
};
constexpr size_t kChainMemoSize = 8;
thread_local std::vector<ChainMemo> g_chain_memo;

// Scratch ranges whose dead lines the chained launch may drop: device memory only (the
// collectives take device pointers; anything else keeps every line). A dry run launches
// nothing and queries nothing: it takes every scratch buffer as device memory.
std::vector<ByteRange> droppable(const std::vector<ByteRange>& scratch, bool dry) {
  std::vector<ByteRange> out;
  for (const ByteRange& r : scratch) {
    if (!dry) {
      cudaPointerAttributes at{};
      if (cudaPointerGetAttributes(&at, reinterpret_cast<const void*>(r.lo)) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      if (at.type != cudaMemoryTypeDevice) continue;
    }
    out.push_back(r);
  }
  return out;
}

// scratch: the call's scratch buffers (empty when every line is to be kept).
ChainMemo& chain_for(const std::vector<Pass>& passes, int E, const std::vector<ByteRange>& scratch,
                     bool dry) {
  thread_local std::vector<unsigned char> key;
  key.clear();
  auto put = [&](const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    key.insert(key.end(), b, b + n);
  };
  put(&E, sizeof E);
  put(&dry, sizeof dry);
  const size_t ns = scratch.size();
  put(&ns, sizeof ns);
  if (ns) put(scratch.data(), ns * sizeof(ByteRange));
  for (const Pass& ps : passes) {
    const size_t n = ps.segs.size();
    put(&n, sizeof n);
    if (n) put(ps.segs.data(), n * sizeof(Seg));
  }
  for (size_t i = g_chain_memo.size(); i-- > 0;)
    if (g_chain_memo[i].key == key) {
      if (i + 1 != g_chain_memo.size()) {
        ChainMemo hit = std::move(g_chain_memo[i]);
        g_chain_memo.erase(g_chain_memo.begin() + (long)i);
        g_chain_memo.push_back(std::move(hit));
      }
      return g_chain_memo.back();
    }
  if (g_chain_memo.size() >= kChainMemoSize) g_chain_memo.erase(g_chain_memo.begin());
  g_chain_memo.emplace_back();
  ChainMemo& m = g_chain_memo.back();
  m.key = key;
  m.scratch = droppable(scratch, dry);
  m.ok = build_chain(passes, E, m.scratch, &m.plan, &m.why);
  return m;
}

// Optional host checks, then the passes in order on `stream`.
relay_status_t execute(const std::vector<Pass>& passes, const std::vector<Range>& ranges,
                       relay_dtype_t dtype, float scale, const relay_opts_t* opts,
                       cudaStream_t stream) {
  const int E = esize_of(dtype);
  std::string why;
  const int flags = opts ? opts->flags : 0;
  if (flags & RELAY_FLAG_CHECK_HAZARDS) {
    for (const Pass& ps : passes) {
      if (find_out_of_bounds(ps, E, ranges, &why) || find_hazard(ps, E, &why))
        return fail(RELAY_ERR_UNSUPPORTED, "internal: " + why);
    }
    // the one-launch kernel's phases run segments of several passes side by side
    std::vector<Pass> phases;
    fused_phases(passes, &phases);
    for (const Pass& ps : phases)
      if (find_hazard(ps, E, &why))
        return fail(RELAY_ERR_UNSUPPORTED, "internal (one-launch phase): " + why);
  }
  // Launch policy. Pass events need the per-pass launches. Otherwise a call runs as one
  // chained launch where its program allows it; else a call of at most
  // RELAY_FUSED_MAX_BYTES of pass traffic runs as one cooperative launch; else pass by pass.
  const bool events_wanted = opts && opts->pass_events;
  const bool one_launch = !events_wanted && !(flags & RELAY_FLAG_SEPARATE_PASSES);
  int64_t bytes = 0;
  for (const Pass& ps : passes)
    for (const Seg& sg : ps.segs) {
      for (int k = 0; k < sg.nsrc; ++k) bytes += seg_src_bytes(sg, k, E);
      bytes += seg_dst_bytes(sg, E) * sg.ndst;
    }
  const bool small = bytes <= RELAY_FUSED_MAX_BYTES;
  const bool try_chain = one_launch && passes.size() > 1 && !(flags & RELAY_FLAG_FUSED_PASSES);
  const ChainPlan* chain = nullptr;
  bool chained = false;
  if (try_chain) {
    std::vector<ByteRange> scratch;
    if (!(flags & RELAY_FLAG_KEEP_SCRATCH))
      for (const Range& r : ranges)
        if (r.scratch) scratch.push_back(ByteRange{r.lo, r.hi});
    ChainMemo& m = chain_for(passes, E, scratch, (flags & RELAY_FLAG_DRY_RUN) != 0);
    chained = m.ok;
    chain = &m.plan;
    if (chained && (flags & RELAY_FLAG_CHECK_HAZARDS) && !m.checked) {
      if (!check_chain(m.plan, E, m.scratch, &why))
        return fail(RELAY_ERR_UNSUPPORTED, "internal (chained launch): " + why);
      m.checked = true;
    }
  }
  std::string chain_desc;
  if (chained) {
    int dropped = 0;
    for (uint8_t d : chain->drop)
      for (unsigned m = d; m; m &= m - 1) ++dropped;
    chain_desc = "chained: " + std::to_string(chain->gn.size()) + " groups, " +
                 std::to_string(chain->segs.size()) + " pieces, " + std::to_string(dropped) +
                 " dropped";
  }
  if (flags & RELAY_FLAG_DRY_RUN) {
    g_last_launch = chained ? chain_desc : "dry run";
    return RELAY_OK;
  }
  if (chained) {
    cudaError_t e = cudaSuccess;
    if (launch_chain(dtype, *chain, scale, stream, &e)) {
      if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
      g_last_launch = chain_desc;
      return RELAY_OK;
    }
  }
  if (one_launch && ((flags & RELAY_FLAG_FUSED_PASSES) || small)) {
    cudaError_t e = cudaSuccess;
    if (launch_fused(dtype, passes, scale, stream, &e, (flags & RELAY_FLAG_FUSED_PASSES) != 0)) {
      if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
      g_last_launch = "cooperative";
      return RELAY_OK;
    }
  }
  g_last_launch = "passes";

  cudaEvent_t* events = nullptr;
  unsigned record_flags = cudaEventRecordDefault;
  if (opts && opts->pass_events) {
    if (opts->n_pass_events < (int)passes.size() + 1)
      return fail(RELAY_ERR_INVALID_ARGUMENT, "pass_events holds fewer than passes + 1 events");
    events = static_cast<cudaEvent_t*>(opts->pass_events);
    // under stream capture the records must become event nodes of the graph, so that
    // the events can still be timed after a replay
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess)
      return fail(RELAY_ERR_CUDA, "cudaStreamIsCapturing failed");
    if (cs == cudaStreamCaptureStatusActive) record_flags = cudaEventRecordExternal;
  }
  for (size_t i = 0; i < passes.size(); ++i) {
    if (events && cudaEventRecordWithFlags(events[i], stream, record_flags) != cudaSuccess)
      return fail(RELAY_ERR_CUDA, "cudaEventRecord failed");
    const cudaError_t e = launch_pass(dtype, passes[i], scale, stream);
    if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
  }
  if (events && cudaEventRecordWithFlags(events[passes.size()], stream, record_flags) != cudaSuccess)
    return fail(RELAY_ERR_CUDA, "cudaEventRecord failed");
  return RELAY_OK;
}

relay_status_t check_scale(relay_coll_t coll, relay_dtype_t dtype, float scale) {
  // D115998376: SUM (scale 1) and AVG (scale 1/A) only; an integer average is not
  // defined on the page, so int32 takes scale 1 only
  const bool reduces = coll == RELAY_ALLREDUCE || coll == RELAY_REDUCE_SCATTER;
  if (reduces && dtype == RELAY_I32 && scale != 1.0f)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "int32 reductions take scale == 1 only");
  return RELAY_OK;
}

// The prepared form (validated buffer ranges and the program) of the last few distinct
// calls this thread made, keyed by every argument that shapes them: the collective, count,
// dtype, A, R, the options other than the pass events, and every buffer pointer. A call
// repeated on the same buffers skips planning, validation and the program build.
struct CallMemo {
  std::vector<unsigned char> key;
  std::vector<Pass> passes;
  std::vector<Range> ranges;
};
constexpr size_t kCallMemoSize = 8;
thread_local std::vector<CallMemo> g_call_memo;

void call_key(relay_coll_t coll, void* const* send, void* const* recv, void* const* scratch,
              size_t count, relay_dtype_t dtype, int A, int R, const relay_opts_t* opts,
              std::vector<unsigned char>* key) {
  key->clear();
  auto put = [&](const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    key->insert(key->end(), b, b + n);
  };
  const int32_t head[4] = {(int32_t)coll, (int32_t)dtype, A, R};
  put(head, sizeof head);
  put(&count, sizeof count);
  const unsigned char has_opts = opts != nullptr;
  put(&has_opts, 1);
  if (opts) {
    put(&opts->offload_permille, sizeof opts->offload_permille);
    put(&opts->schedule, sizeof opts->schedule);
    put(&opts->relay_threshold_bytes, sizeof opts->relay_threshold_bytes);
    put(&opts->flags, sizeof opts->flags);
  }
  put(send, (size_t)A * sizeof(void*));
  put(recv, (size_t)A * sizeof(void*));
  put(scratch, (size_t)R * sizeof(void*));
}

relay_status_t run_collective(relay_coll_t coll, void* const* send, void* const* recv,
                              void* const* scratch, size_t count, relay_dtype_t dtype, int A,
                              int R, float scale, const relay_opts_t* opts, cudaStream_t stream) {
  if (count > (size_t)INT64_MAX) return fail(RELAY_ERR_INVALID_ARGUMENT, "count too large");
  thread_local std::vector<unsigned char> key;
  const bool keyable = count > 0 && send != nullptr && recv != nullptr && scratch != nullptr &&
                       A >= 1 && A <= R && R <= RELAY_MAX_RANKS;
  if (keyable) {
    call_key(coll, send, recv, scratch, count, dtype, A, R, opts, &key);
    for (size_t i = g_call_memo.size(); i-- > 0;)
      if (g_call_memo[i].key == key) {
        relay_status_t st = check_scale(coll, dtype, scale);
        if (st != RELAY_OK) return st;
        if (i + 1 != g_call_memo.size()) {
          CallMemo hit = std::move(g_call_memo[i]);
          g_call_memo.erase(g_call_memo.begin() + (long)i);
          g_call_memo.push_back(std::move(hit));
        }
        const CallMemo& m = g_call_memo.back();
        return execute(m.passes, m.ranges, dtype, scale, opts, stream);
      }
  }
  relay_plan_t p;
  std::string why;
  relay_status_t st = make_plan(coll, (int64_t)count, dtype, A, R, opts, &p, &why);
  if (st != RELAY_OK) return fail(st, why);
  if ((st = check_scale(coll, dtype, scale)) != RELAY_OK) return st;
  if (p.count == 0) return RELAY_OK;
  if (send == nullptr || recv == nullptr || scratch == nullptr)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "pointer arrays must not be NULL");
  std::vector<int> ident(R);
  for (int r = 0; r < R; ++r) ident[r] = r;
  std::vector<Range> ranges;
  if ((st = validate_group(p, send, recv, scratch, ident.data(), &ranges)) != RELAY_OK) return st;
  if ((st = check_disjoint(ranges)) != RELAY_OK) return st;
  std::vector<Pass> passes;
  build_program(p, Buffers{send, recv, scratch}, false, &passes);
  if (!keyable) return execute(passes, ranges, dtype, scale, opts, stream);
  if (g_call_memo.size() >= kCallMemoSize) g_call_memo.erase(g_call_memo.begin());
  g_call_memo.push_back(CallMemo{key, std::move(passes), std::move(ranges)});
  const CallMemo& m = g_call_memo.back();
  return execute(m.passes, m.ranges, dtype, scale, opts, stream);
}

// Fused multi-group call (D115998367, D115998376): R/A sparse groups of A consecutive
// ranks; every rank is active in its own group and a helper in every other group.
// send/recv are indexed by global rank; scratch[g*R + r] is rank r's scratch for group
// g. Each group plans its own schedule from its own count.
relay_status_t run_multi(relay_coll_t coll, int num_groups, const size_t* counts,
                         void* const* send, void* const* recv, void* const* scratch,
                         relay_dtype_t dtype, int A, float scale, const relay_opts_t* opts,
                         cudaStream_t stream) {
  if (num_groups < 2 || counts == nullptr)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "a fused call needs at least 2 groups and counts");
  const int R = num_groups * A;
  if (A != 2 && A != 4) return fail(RELAY_ERR_INVALID_ARGUMENT, "A must be 2 or 4");
  if (R > RELAY_MAX_RANKS) return fail(RELAY_ERR_INVALID_ARGUMENT, "num_groups*A exceeds RELAY_MAX_RANKS");
  relay_status_t st = check_scale(coll, dtype, scale);
  if (st != RELAY_OK) return st;
  if (send == nullptr || recv == nullptr || scratch == nullptr)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "pointer arrays must not be NULL");
  std::vector<relay_plan_t> plans(num_groups);
  std::vector<std::vector<int>> gmap(num_groups);
  std::vector<std::vector<void*>> ls(num_groups), lr(num_groups), lw(num_groups);
  std::vector<Range> ranges;
  std::string why;
  for (int g = 0; g < num_groups; ++g) {
    if (counts[g] > (size_t)INT64_MAX) return fail(RELAY_ERR_INVALID_ARGUMENT, "count too large");
    st = make_plan(coll, (int64_t)counts[g], dtype, A, R, opts, &plans[g], &why);
    if (st != RELAY_OK) return fail(st, "group " + std::to_string(g) + ": " + why);
    gmap[g] = group_ranks(g, A, R);
    ls[g].assign(R, nullptr);
    lr[g].assign(R, nullptr);
    lw[g].assign(R, nullptr);
    for (int l = 0; l < R; ++l) {
      const int r = gmap[g][l];
      if (l < A) {
        ls[g][l] = send[r];
        lr[g][l] = recv[r];
      }
      lw[g][l] = scratch[(size_t)g * R + r];
    }
    if (plans[g].count == 0) continue;
    st = validate_group(plans[g], ls[g].data(), lr[g].data(), lw[g].data(), gmap[g].data(),
                        &ranges);
    if (st != RELAY_OK) return fail(st, "group " + std::to_string(g) + ": " + relay_last_error());
  }
  if ((st = check_disjoint(ranges)) != RELAY_OK) return st;
  std::vector<Buffers> bufs(num_groups);
  for (int g = 0; g < num_groups; ++g) bufs[g] = Buffers{ls[g].data(), lr[g].data(), lw[g].data()};
  std::vector<Pass> passes;
  build_multi_program(plans, bufs, gmap, &passes);
  return execute(passes, ranges, dtype, scale, opts, stream);
}

}  // namespace

relay_status_t report_error(relay_status_t st, const std::string& msg) { return fail(st, msg); }

}  // namespace relay

using namespace relay;

extern "C" {

void relay_opts_init(relay_opts_t* o) {
  if (!o) return;
  memset(o, 0, sizeof *o);
  o->offload_permille = -1;
  o->schedule = RELAY_SCHEDULE_AUTO;
  o->relay_threshold_bytes = -1;
}

int relay_abi_version(void) { return RELAY_ABI_VERSION; }

const char* relay_last_error(void) { return g_last_error.c_str(); }

const char* relay_last_launch(void) { return g_last_launch.c_str(); }

relay_status_t relay_plan(relay_coll_t coll, size_t count, relay_dtype_t dtype, int A, int R,
                          const relay_opts_t* opts, relay_plan_t* out) {
  if (count > (size_t)INT64_MAX) return fail(RELAY_ERR_INVALID_ARGUMENT, "count too large");
  std::string why;
  const relay_status_t st = make_plan(coll, (int64_t)count, dtype, A, R, opts, out, &why);
  if (st != RELAY_OK) return fail(st, why);
  return RELAY_OK;
}

relay_status_t relay_plan_link_bytes(const relay_plan_t* plan, uint64_t* out, size_t cap) {
  if (!plan || !out) return fail(RELAY_ERR_INVALID_ARGUMENT, "NULL argument");
  const int R = plan->R, G = plan->num_groups;
  if (R <= 0 || R > RELAY_MAX_RANKS || G < 0 || G > 3)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "not a plan");
  const size_t need = (size_t)G * R * R;
  if (cap < need) return fail(RELAY_ERR_INVALID_ARGUMENT, "link table too small");
  std::fill(out, out + need, 0);
  FakeBuffers fb(*plan, false);
  std::vector<Pass> passes;
  build_program(*plan, fb.view(), false, &passes);
  for (const Pass& ps : passes)
    for (size_t i = 0; i < ps.segs.size(); ++i) {
      const SegMeta& m = ps.meta[i];
      if (m.group < 0) continue;
      if (m.group >= G) return fail(RELAY_ERR_INVALID_ARGUMENT, "internal: group out of range");
      for (int d = 0; d < ps.segs[i].ndst; ++d)
        if (m.dst_rank[d] != m.exec_rank)
          out[((size_t)m.group * R + m.exec_rank) * R + m.dst_rank[d]] +=
              (uint64_t)seg_dst_bytes(ps.segs[i], plan->esize);
    }
  return RELAY_OK;
}

uint64_t relay_plan_cost_bytes(const relay_plan_t* plan) {
  if (!plan || plan->R <= 0 || plan->R > RELAY_MAX_RANKS || plan->num_groups > 3) return 0;
  std::vector<uint64_t> t((size_t)std::max(plan->num_groups, 1) * plan->R * plan->R);
  if (relay_plan_link_bytes(plan, t.data(), t.size()) != RELAY_OK) return 0;
  uint64_t total = 0;
  const size_t per = (size_t)plan->R * plan->R;
  for (int g = 0; g < plan->num_groups; ++g)
    total += *std::max_element(t.begin() + g * per, t.begin() + (g + 1) * per);
  return total;
}

int relay_plan_passes(const relay_plan_t* plan, int in_place, relay_pass_info_t* out, int cap) {
  if (!plan || plan->R <= 0 || plan->R > RELAY_MAX_RANKS) return -1;
  FakeBuffers fb(*plan, in_place != 0);
  std::vector<Pass> passes;
  build_program(*plan, fb.view(), in_place != 0, &passes);
  for (size_t i = 0; i < passes.size() && (int)i < cap && out; ++i) {
    relay_pass_info_t& q = out[i];
    q.kind = passes[i].kind;
    q.num_segments = (int32_t)passes[i].segs.size();
    q.bytes_read = q.bytes_written = 0;
    for (const Seg& s : passes[i].segs) {
      for (int k = 0; k < s.nsrc; ++k) q.bytes_read += seg_src_bytes(s, k, plan->esize);
      q.bytes_written += seg_dst_bytes(s, plan->esize) * s.ndst;
    }
  }
  return (int)passes.size();
}

const char* relay_pass_name(int kind) {
  switch (kind) {
    case RELAY_PASS_G1: return "group1";
    case RELAY_PASS_G2: return "group2";
    case RELAY_PASS_G3: return "group3";
    case RELAY_PASS_ACTIVE_REDUCE: return "active_reduce";
    case RELAY_PASS_PACK: return "pack";
    case RELAY_PASS_HELPER_FORWARD: return "helper_forward";
    case RELAY_PASS_UNPACK: return "unpack";
    default: return "unknown";
  }
}

int64_t relay_helper_size(const relay_plan_t* plan) { return plan ? plan->helper_elems : -1; }

int64_t relay_active_scratch_size(const relay_plan_t* plan) {
  return plan ? plan->active_scratch_elems : -1;
}

int64_t relay_helper_contract_size(relay_coll_t coll, int64_t count, int A, int R) {
  if (count < 0 || (A != 2 && A != 4) || R <= A || coll < RELAY_ALLREDUCE || coll > RELAY_ALL_TO_ALL)
    return -1;
  if (A == 2) return relay_passthrough_helper_size(count, A, (R - A) + 1);
  switch (coll) {
    case RELAY_ALLREDUCE:
    case RELAY_REDUCE_SCATTER: return 2 * count;
    case RELAY_ALL_GATHER: return (int64_t)A * count;
    default: return 1;
  }
}

// D115998394, D115998388, D115998370: A slots, each a whole number of 128-element
// chunks, never more than the group count itself
int64_t relay_passthrough_helper_size(int64_t count_g, int A, int num_chunks) {
  if (count_g < 0 || A <= 0 || num_chunks <= 0) return -1;
  const int64_t chunk = (count_g / num_chunks) / RELAY_ALIGN_ELEMS * RELAY_ALIGN_ELEMS;
  if (chunk == 0) return count_g;
  return std::min<int64_t>(count_g, (int64_t)A * chunk);
}

relay_status_t relay_allreduce(void* const* send, void* const* recv, void* const* scratch,
                               size_t count, relay_dtype_t dtype, int A, int R, float scale,
                               const relay_opts_t* opts, cudaStream_t stream) {
  return run_collective(RELAY_ALLREDUCE, send, recv, scratch, count, dtype, A, R, scale, opts,
                        stream);
}

relay_status_t relay_reduce_scatter(void* const* send, void* const* recv, void* const* scratch,
                                    size_t recv_count, relay_dtype_t dtype, int A, int R,
                                    float scale, const relay_opts_t* opts, cudaStream_t stream) {
  return run_collective(RELAY_REDUCE_SCATTER, send, recv, scratch, recv_count, dtype, A, R, scale,
                        opts, stream);
}

relay_status_t relay_all_gather(void* const* send, void* const* recv, void* const* scratch,
                                size_t send_count, relay_dtype_t dtype, int A, int R,
                                const relay_opts_t* opts, cudaStream_t stream) {
  return run_collective(RELAY_ALL_GATHER, send, recv, scratch, send_count, dtype, A, R, 1.0f, opts,
                        stream);
}

relay_status_t relay_all_to_all(void* const* send, void* const* recv, void* const* scratch,
                                size_t segment_count, relay_dtype_t dtype, int A, int R,
                                const relay_opts_t* opts, cudaStream_t stream) {
  return run_collective(RELAY_ALL_TO_ALL, send, recv, scratch, segment_count, dtype, A, R, 1.0f,
                        opts, stream);
}

relay_status_t relay_multi_group(relay_coll_t coll, int num_groups, const size_t* counts,
                                 void* const* send, void* const* recv, void* const* scratch,
                                 relay_dtype_t dtype, int A, float scale,
                                 const relay_opts_t* opts, cudaStream_t stream) {
  if (coll < RELAY_ALLREDUCE || coll > RELAY_ALL_TO_ALL)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "unknown collective");
  if (coll == RELAY_ALL_GATHER || coll == RELAY_ALL_TO_ALL) scale = 1.0f;
  return run_multi(coll, num_groups, counts, send, recv, scratch, dtype, A, scale, opts, stream);
}

// D115998366: the distributed layer packs the caller's tensors into the active flat
// buffer with one launch and unpacks the result with one launch; here both are a single
// pass of copy segments (split only past 384 tensors).
static relay_status_t flat_copy(const void* const* parts, const size_t* counts, int n,
                                void* flat, relay_dtype_t dtype, bool pack, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (parts == nullptr || counts == nullptr)))
    return fail(RELAY_ERR_INVALID_ARGUMENT, "bad tensor list");
  if (dtype < RELAY_F32 || dtype > RELAY_I32) return fail(RELAY_ERR_INVALID_ARGUMENT, "unknown dtype");
  const int E = esize_of(dtype);
  Pass ps{pack ? RELAY_PASS_PACK : RELAY_PASS_UNPACK, {}, {}};
  std::vector<Range> ranges;
  int64_t off = 0;
  for (int i = 0; i < n; ++i) {
    if (counts[i] > (size_t)INT64_MAX / 16) return fail(RELAY_ERR_INVALID_ARGUMENT, "count too large");
    const int64_t c = (int64_t)counts[i];
    if (c == 0) continue;
    if (parts[i] == nullptr || flat == nullptr)
      return fail(RELAY_ERR_INVALID_ARGUMENT, "tensor " + std::to_string(i) + " is NULL");
    if ((reinterpret_cast<uintptr_t>(parts[i]) | reinterpret_cast<uintptr_t>(flat)) % E)
      return fail(RELAY_ERR_INVALID_ARGUMENT, "tensor " + std::to_string(i) + " not element-aligned");
    const uintptr_t lo = reinterpret_cast<uintptr_t>(parts[i]);
    ranges.push_back(Range{lo, lo + (uintptr_t)(c * E), "tensor " + std::to_string(i)});
    Seg sg{};
    char* f = static_cast<char*>(flat) + off * E;
    sg.src[0] = pack ? parts[i] : f;
    sg.dst[0] = pack ? (void*)f : const_cast<void*>(parts[i]);
    sg.n = c;
    sg.op = kOpCopy;
    sg.nsrc = sg.ndst = 1;
    ps.segs.push_back(sg);
    ps.meta.push_back(SegMeta{-1, 0, {0, -1, -1, -1}});
    off += c;
  }
  if (off == 0) return RELAY_OK;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(flat);
  ranges.push_back(Range{lo, lo + (uintptr_t)(off * E), "flat"});
  relay_status_t st = check_disjoint(ranges);
  if (st != RELAY_OK) return st;
  const cudaError_t e = launch_pass(dtype, ps, 1.0f, stream);
  if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
  return RELAY_OK;
}

relay_status_t relay_pack_flat(const void* const* srcs, const size_t* counts, int n, void* flat,
                               relay_dtype_t dtype, cudaStream_t stream) {
  return flat_copy(srcs, counts, n, flat, dtype, true, stream);
}

relay_status_t relay_unpack_flat(const void* flat, void* const* dsts, const size_t* counts, int n,
                                 relay_dtype_t dtype, cudaStream_t stream) {
  return flat_copy(const_cast<const void* const*>(dsts), counts, n, const_cast<void*>(flat), dtype,
                   false, stream);
}

// Where the device can reach `p`: device or managed memory and pinned/registered host
// memory through their device address, pageable host memory only on devices that read
// the host's page tables. *dev receives the address the kernel uses.
static relay_status_t device_view(const void* p, const char* what, const void** dev) {
  cudaPointerAttributes at{};
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(RELAY_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  }
  if (at.type == cudaMemoryTypeUnregistered) {
    int d = 0, pageable = 0;
    if (cudaGetDevice(&d) != cudaSuccess ||
        cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, d) != cudaSuccess) {
      cudaGetLastError();
      return fail(RELAY_ERR_CUDA, std::string(what) + ": device query failed");
    }
    if (!pageable)
      return fail(RELAY_ERR_UNSUPPORTED,
                  std::string(what) + " is pageable host memory this device cannot address");
    *dev = p;
    return RELAY_OK;
  }
  if (at.type == cudaMemoryTypeHost && at.devicePointer != nullptr) {
    // the device address of this byte: the allocation's device base + the same offset
    *dev = static_cast<const char*>(at.devicePointer) +
           (static_cast<const char*>(p) - static_cast<const char*>(at.hostPointer));
    return RELAY_OK;
  }
  *dev = p;
  return RELAY_OK;
}

relay_status_t relay_copy(void* dst, const void* src, size_t count, relay_dtype_t dtype,
                          int max_ctas, cudaStream_t stream) {
  if (dtype < RELAY_F32 || dtype > RELAY_I32) return fail(RELAY_ERR_INVALID_ARGUMENT, "unknown dtype");
  if (max_ctas < 0) return fail(RELAY_ERR_INVALID_ARGUMENT, "max_ctas < 0");
  if (count == 0) return RELAY_OK;
  if (count > (size_t)INT64_MAX / 16) return fail(RELAY_ERR_INVALID_ARGUMENT, "count too large");
  if (dst == nullptr || src == nullptr) return fail(RELAY_ERR_INVALID_ARGUMENT, "NULL pointer");
  const int E = esize_of(dtype);
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % E)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "pointer not element-aligned");
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t bytes = (uintptr_t)count * E;
  relay_status_t st = check_disjoint({Range{s0, s0 + bytes, "src"}, Range{d0, d0 + bytes, "dst"}});
  if (st != RELAY_OK) return st;
  const void *sv = nullptr, *dv = nullptr;
  if ((st = device_view(src, "src", &sv)) != RELAY_OK) return st;
  if ((st = device_view(dst, "dst", &dv)) != RELAY_OK) return st;
  Pass ps{RELAY_PASS_PACK, {}, {}};
  Seg sg{};
  sg.src[0] = sv;
  sg.dst[0] = const_cast<void*>(dv);
  sg.n = (int64_t)count;
  sg.op = kOpCopy;
  sg.nsrc = sg.ndst = 1;
  ps.segs.push_back(sg);
  ps.meta.push_back(SegMeta{-1, 0, {0, -1, -1, -1}});
  // either side may be host memory: keep to the register path (no bulk copies)
  const cudaError_t e = launch_pass(dtype, ps, 1.0f, stream, max_ctas, false);
  if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
  return RELAY_OK;
}

relay_status_t relay_device_status(void) {
  unsigned fault = 0;
  const cudaError_t e = read_device_fault(&fault);
  if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
  if (fault)
    return fail(RELAY_ERR_CUDA,
                "a bounded wait in a relay kernel gave up (a bulk copy into shared memory did "
                "not land in time); the affected tiles were not written");
  return RELAY_OK;
}

relay_status_t relay_test_staged_wait(void* dst, const void* src, size_t count,
                                      relay_dtype_t dtype, int extra_bytes, cudaStream_t stream) {
  if (dtype < RELAY_F32 || dtype > RELAY_I32) return fail(RELAY_ERR_INVALID_ARGUMENT, "unknown dtype");
  if (dst == nullptr || src == nullptr || count == 0 || count > (size_t)(tile_elems(esize_of(dtype))) ||
      extra_bytes < 0 || extra_bytes > (1 << 20))
    return fail(RELAY_ERR_INVALID_ARGUMENT, "one tile of device memory, 0 <= extra_bytes <= 1 MiB");
  const int E = esize_of(dtype);
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) || reinterpret_cast<uintptr_t>(src) % E)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "dst must be 16-byte aligned, src element-aligned");
  const cudaError_t e = launch_staged_wait_test(dst, src, (int64_t)count, dtype, extra_bytes, stream);
  if (e != cudaSuccess) return fail(RELAY_ERR_CUDA, cudaGetErrorString(e));
  return RELAY_OK;
}

relay_status_t relay_multi_group_link_bytes(relay_coll_t coll, int num_groups,
                                            const size_t* counts, relay_dtype_t dtype, int A,
                                            const relay_opts_t* opts, uint64_t* out, size_t cap,
                                            int* num_phases) {
  if (!counts || !out || num_groups < 2 || (A != 2 && A != 4) || num_groups * A > RELAY_MAX_RANKS)
    return fail(RELAY_ERR_INVALID_ARGUMENT, "bad fused-call description");
  const int R = num_groups * A;
  std::vector<relay_plan_t> plans(num_groups);
  std::vector<std::vector<int>> gmap(num_groups);
  std::vector<FakeBuffers> fakes;
  fakes.reserve(num_groups);
  std::string why;
  int G = 0;
  for (int g = 0; g < num_groups; ++g) {
    const relay_status_t st =
        make_plan(coll, (int64_t)counts[g], dtype, A, R, opts, &plans[g], &why);
    if (st != RELAY_OK) return fail(st, why);
    G = std::max(G, plans[g].num_groups);
    gmap[g] = group_ranks(g, A, R);
    fakes.emplace_back(plans[g], false, g);
  }
  const size_t need = (size_t)G * R * R;
  if (num_phases) *num_phases = G;
  if (cap < need) return fail(RELAY_ERR_INVALID_ARGUMENT, "link table too small");
  std::fill(out, out + need, 0);
  std::vector<Buffers> bufs;
  for (auto& f : fakes) bufs.push_back(f.view());
  std::vector<Pass> passes;
  build_multi_program(plans, bufs, gmap, &passes);
  for (const Pass& ps : passes)
    for (size_t i = 0; i < ps.segs.size(); ++i) {
      const SegMeta& m = ps.meta[i];
      if (m.group < 0) continue;
      for (int d = 0; d < ps.segs[i].ndst; ++d)
        if (m.dst_rank[d] != m.exec_rank)
          out[((size_t)m.group * R + m.exec_rank) * R + m.dst_rank[d]] +=
              (uint64_t)ps.segs[i].n * esize_of(dtype);
    }
  return RELAY_OK;
}

}  // extern "C"
