// program.cpp -- the relay schedules as kernel passes over segment tables (host).
//
// Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)" (torchrec pull
// request #4570): "item k" of its summary, "Dnnnnnnnnn" a commit of its stack.
//
// Conventions. Ranks 0..A-1 are the actives, rank A+h is helper h (D115998382). A
// transfer of schedule group g is a segment executed for its sending rank whose
// stores land in the receiving rank's memory (a push). Reductions read only the
// executing rank's own memory; where the page fuses a reduction with the hop that
// follows it (a helper returning its reduced chunk, item 2; an owner all-gathering
// its reduced slice, item 4), the reduction stores straight into the receivers.
// Sources of a reduction are listed in ascending source rank.
#include <algorithm>
#include <initializer_list>
#include <utility>

#include "program.h"

namespace relay {
namespace {

struct Dst {
  int rank;
  void* ptr;
};

class Builder {
 public:
  Builder(const relay_plan_t& p, const Buffers& b, std::vector<Pass>* out)
      : p_(p), b_(b), out_(out), E_(p.esize) {}

  void begin(relay_pass_kind_t kind) {
    out_->push_back(Pass{kind, {}, {}});
    cur_ = &out_->back();
    phase_ = -1;
  }
  // earliest one-launch phase of the segments emitted from here on (-1: their own pass)
  void phase(int ph) { phase_ = ph; }

  // group: schedule group of the transfer (0-based), or -1 for work local to `exec`
  void copy(int group, int exec, const void* src, std::initializer_list<Dst> dsts, int64_t n) {
    std::vector<Dst> d(dsts);
    emit(group, exec, kOpCopy, &src, 1, d, n, false);
  }
  void copy(int group, int exec, const void* src, const std::vector<Dst>& dsts, int64_t n) {
    emit(group, exec, kOpCopy, &src, 1, dsts, n, false);
  }
  void reduce(int group, int exec, const std::vector<const void*>& srcs,
              const std::vector<Dst>& dsts, int64_t n, bool scale, uint8_t extra_flags = 0) {
    emit(group, exec, kOpReduce, srcs.data(), (int)srcs.size(), dsts, n, scale);
    if (n > 0) cur_->segs.back().flags |= extra_flags;
  }

  // element-offset pointers into the rank buffers
  char* X(int a, int64_t off) const { return (char*)b_.send[a] + off * E_; }
  char* Y(int a, int64_t off) const { return (char*)b_.recv[a] + off * E_; }
  char* W(int a, int64_t off) const { return (char*)b_.scratch[a] + off * E_; }
  char* Hh(int h, int64_t off) const { return (char*)b_.scratch[p_.A + h] + off * E_; }

 private:
  void emit(int group, int exec, SegOp op, const void* const* srcs, int nsrc,
            const std::vector<Dst>& dsts, int64_t n, bool scale) {
    if (n <= 0) return;
    Seg s{};
    SegMeta m{};
    s.n = n;
    s.op = op;
    s.nsrc = (uint8_t)nsrc;
    s.ndst = (uint8_t)dsts.size();
    s.flags = scale ? kFlagScale : 0;
    for (int i = 0; i < nsrc; ++i) s.src[i] = srcs[i];
    m.group = (int8_t)group;
    m.exec_rank = (int8_t)exec;
    m.phase = (int8_t)phase_;
    for (int i = 0; i < kMaxDst; ++i) m.dst_rank[i] = -1;
    for (size_t i = 0; i < dsts.size(); ++i) {
      s.dst[i] = dsts[i].ptr;
      m.dst_rank[i] = (int8_t)dsts[i].rank;
    }
    cur_->segs.push_back(s);
    cur_->meta.push_back(m);
  }

  const relay_plan_t& p_;
  const Buffers& b_;
  std::vector<Pass>* out_;
  Pass* cur_ = nullptr;
  int E_;
  int phase_ = -1;
};

// index of `s` among the A-1 ranks other than `o`, ascending
inline int other_index(int s, int o) { return s < o ? s : s - 1; }

// ---------------------------------------------------------------------------------
// A = 2. The two actives exchange one region each: `src(a)` is where active a's
// outgoing region starts, `dst(a)` where it lands in the other active's memory
// (position-aligned). Helpers are passthrough (item 2, reduce-scatter; D115998370).
// ---------------------------------------------------------------------------------
template <class SrcF, class DstF>
void a2_exchange(Builder& B, const relay_plan_t& p, SrcF src, DstF dst,
                 const std::vector<std::pair<int, std::pair<const void*, void*>>>& self) {
  const int H = p.H;
  const int64_t n = p.count, c = p.chunk;
  auto add_self = [&]() {
    for (auto& s : self)
      if (s.second.first != s.second.second)
        B.copy(-1, s.first, s.second.first, {Dst{s.first, s.second.second}}, n);
  };
  switch (p.kind) {
    case RELAY_KIND_DIRECT:
      // item 3: one full exchange
      B.begin(RELAY_PASS_G1);
      for (int a = 0; a < 2; ++a) B.copy(0, a, src(a, 0), {Dst{1 - a, dst(a, 0)}}, n);
      add_self();
      break;
    case RELAY_KIND_ZERO_CHUNK:
      // D115998367: dirA (half) in group 1, dirB (the rest) in group 2
      B.begin(RELAY_PASS_G1);
      for (int a = 0; a < 2; ++a) B.copy(0, a, src(a, 0), {Dst{1 - a, dst(a, 0)}}, p.dirA_size);
      add_self();
      B.begin(RELAY_PASS_G2);
      for (int a = 0; a < 2; ++a)
        B.copy(1, a, src(a, p.dirA_size), {Dst{1 - a, dst(a, p.dirA_size)}}, p.dirB_size);
      break;
    case RELAY_KIND_RELAY:
      // item 1: group 1 scatters chunk h to helper h (slot a) and carries dirA;
      // group 2 forwards each slot to the other active and carries dirB
      B.begin(RELAY_PASS_G1);
      for (int a = 0; a < 2; ++a) {
        for (int h = 0; h < H; ++h) B.copy(0, a, src(a, h * c), {Dst{2 + h, B.Hh(h, a * c)}}, c);
        B.copy(0, a, src(a, p.dirA_offset), {Dst{1 - a, dst(a, p.dirA_offset)}}, p.dirA_size);
      }
      add_self();
      B.begin(RELAY_PASS_G2);
      for (int h = 0; h < H; ++h)
        for (int a = 0; a < 2; ++a) B.copy(1, 2 + h, B.Hh(h, a * c), {Dst{1 - a, dst(a, h * c)}}, c);
      for (int a = 0; a < 2; ++a) {
        const int64_t off = p.dirA_offset + p.dirA_size;
        B.copy(1, a, src(a, off), {Dst{1 - a, dst(a, off)}}, p.dirB_size);
      }
      break;
    case RELAY_KIND_LEGACY:
      // item 1, before: scatter, forward, then a separate direct exchange
      B.begin(RELAY_PASS_G1);
      for (int a = 0; a < 2; ++a)
        for (int h = 0; h < H; ++h) B.copy(0, a, src(a, h * c), {Dst{2 + h, B.Hh(h, a * c)}}, c);
      add_self();
      B.begin(RELAY_PASS_G2);
      for (int h = 0; h < H; ++h)
        for (int a = 0; a < 2; ++a) B.copy(1, 2 + h, B.Hh(h, a * c), {Dst{1 - a, dst(a, h * c)}}, c);
      B.begin(RELAY_PASS_G3);
      for (int a = 0; a < 2; ++a)
        B.copy(2, a, src(a, p.dirA_offset), {Dst{1 - a, dst(a, p.dirA_offset)}}, p.dirA_size);
      break;
  }
}

// The actives' closing reduction: out = Q(scale * (own + received)), sources ascending
// by rank (D115998376 phases 3 and 5 fused into one pass).
void a2_active_reduce(Builder& B, int64_t n, const void* own0, const void* recv0, void* out0,
                      const void* own1, const void* recv1, void* out1, int phase = -1) {
  B.begin(RELAY_PASS_ACTIVE_REDUCE);
  B.phase(phase);
  B.reduce(-1, 0, {own0, recv0}, {Dst{0, out0}}, n, true);
  B.reduce(-1, 1, {recv1, own1}, {Dst{1, out1}}, n, true);
}

void build_a2(Builder& B, const relay_plan_t& p) {
  const int64_t n = p.count;
  using SelfList = std::vector<std::pair<int, std::pair<const void*, void*>>>;
  switch (p.coll) {
    case RELAY_ALLREDUCE: {
      if (p.kind == RELAY_KIND_RELAY) {
        // item 1 geometry + item 2: the helper sums its two slots, scales, casts and
        // returns the one reduced chunk to both actives. The actives' scratch holds
        // only the direct region: [dirA | dirB].
        const int H = p.H;
        const int64_t c = p.chunk, d0 = p.dirA_offset;
        B.begin(RELAY_PASS_G1);
        for (int a = 0; a < 2; ++a) {
          for (int h = 0; h < H; ++h) B.copy(0, a, B.X(a, h * c), {Dst{2 + h, B.Hh(h, a * c)}}, c);
          B.copy(0, a, B.X(a, d0), {Dst{1 - a, B.W(1 - a, 0)}}, p.dirA_size);
        }
        B.begin(RELAY_PASS_G2);
        for (int h = 0; h < H; ++h)
          B.reduce(1, 2 + h, {B.Hh(h, 0), B.Hh(h, c)},
                   {Dst{0, B.Y(0, h * c)}, Dst{1, B.Y(1, h * c)}}, c, true);
        // In the one-launch kernel the dirB copies read only inputs, so they run with
        // group 1, and the closing reduction needs only dirA and dirB, so it runs with the
        // helper reductions: two phases and one grid barrier instead of three and two.
        B.phase(0);
        for (int a = 0; a < 2; ++a)
          B.copy(1, a, B.X(a, d0 + p.dirA_size), {Dst{1 - a, B.W(1 - a, p.dirA_size)}},
                 p.dirB_size);
        a2_active_reduce(B, n - d0, B.X(0, d0), B.W(0, 0), B.Y(0, d0), B.X(1, d0), B.W(1, 0),
                         B.Y(1, d0), 1);
      } else {
        // item 3 full exchange, D115998367 halves, or the legacy three groups: the
        // received region is staged position-aligned in the scratch
        a2_exchange(
            B, p, [&](int a, int64_t o) { return B.X(a, o); },
            [&](int a, int64_t o) { return B.W(1 - a, o); }, SelfList{});
        a2_active_reduce(B, n, B.X(0, 0), B.W(0, 0), B.Y(0, 0), B.X(1, 0), B.W(1, 0), B.Y(1, 0));
      }
      break;
    }
    case RELAY_REDUCE_SCATTER: {
      // D115998376: input = 2 blocks of recvCount, block k destined for active k; each
      // active relays block[other] (helpers passthrough, item 2) into the other's
      // scratch, then adds its own block
      const int64_t m = n;
      a2_exchange(
          B, p, [&](int a, int64_t o) { return B.X(a, (1 - a) * m + o); },
          [&](int a, int64_t o) { return B.W(1 - a, o); }, SelfList{});
      a2_active_reduce(B, m, B.X(0, 0), B.W(0, 0), B.Y(0, 0), B.X(1, m), B.W(1, 0), B.Y(1, 0));
      break;
    }
    case RELAY_ALL_GATHER: {
      // D115998385: out_b[k*S + i] = x_k[i]; the relayed region lands in the other
      // active's output slot directly
      const int64_t S = n;
      SelfList self{{0, {B.X(0, 0), B.Y(0, 0)}}, {1, {B.X(1, 0), B.Y(1, S)}}};
      a2_exchange(
          B, p, [&](int a, int64_t o) { return B.X(a, o); },
          [&](int a, int64_t o) { return B.Y(1 - a, a * S + o); }, self);
      break;
    }
    default: {
      // D115998370: out_d[s*seg + i] = x_s[d*seg + i]
      const int64_t seg = n;
      SelfList self{{0, {B.X(0, 0), B.Y(0, 0)}}, {1, {B.X(1, seg), B.Y(1, seg)}}};
      a2_exchange(
          B, p, [&](int a, int64_t o) { return B.X(a, (1 - a) * seg + o); },
          [&](int a, int64_t o) { return B.Y(1 - a, a * seg + o); }, self);
      break;
    }
  }
}

// ---------------------------------------------------------------------------------
// A = 4 (and any power-of-two A > 2 the plan allows)
// ---------------------------------------------------------------------------------
void build_a4_allreduce(Builder& B, const relay_plan_t& p) {
  // item 4 + D115998382: offload region [0, H*oc) in H helper slices, reduced at the
  // helpers and broadcast; direct region [H*oc, n) in A owner slices, reduce-scattered
  // to the owners (group 1) and all-gathered back from them (group 2)
  const int A = p.A, H = p.H;
  const int64_t oc = p.chunk;
  auto off = [&](int o) { return H * oc + o * p.owner_slice; };
  auto len = [&](int o) { return o == A - 1 ? p.owner_slice_last : p.owner_slice; };
  B.begin(RELAY_PASS_G1);
  for (int a = 0; a < A; ++a)
    for (int h = 0; h < H; ++h) B.copy(0, a, B.X(a, h * oc), {Dst{A + h, B.Hh(h, a * oc)}}, oc);
  for (int o = 0; o < A; ++o)
    for (int s = 0; s < A; ++s)
      if (s != o)
        B.copy(0, s, B.X(s, off(o)), {Dst{o, B.W(o, other_index(s, o) * len(o))}}, len(o));
  B.begin(RELAY_PASS_G2);
  for (int h = 0; h < H; ++h) {
    std::vector<const void*> srcs;
    std::vector<Dst> dsts;
    for (int a = 0; a < A; ++a) {
      srcs.push_back(B.Hh(h, a * oc));
      dsts.push_back(Dst{a, B.Y(a, h * oc)});
    }
    B.reduce(1, A + h, srcs, dsts, oc, true);
  }
  for (int o = 0; o < A; ++o) {
    std::vector<const void*> srcs;
    std::vector<Dst> dsts;
    for (int s = 0; s < A; ++s)
      srcs.push_back(s == o ? (const void*)B.X(o, off(o))
                            : (const void*)B.W(o, other_index(s, o) * len(o)));
    for (int b = 0; b < A; ++b) dsts.push_back(Dst{b, B.Y(b, off(o))});
    B.reduce(1, o, srcs, dsts, len(o), true);
  }
}

void build_a4_reduce_scatter(Builder& B, const relay_plan_t& p) {
  // item 6: flat reduce-at-helper. Helper h owns position slice h of every block; the
  // A-1 non-owner sources send it their slice (group 1), the helper sums them into one
  // partial and returns that single chunk to the owner (group 2). The direct positions
  // go source -> owner in two parts (group 1, group 2). The owner scratch:
  //   [partials: H*oc positions, payload-typed | A-1 direct slots of pD], or, with fp32
  //   partials, [H*oc fp32 partials, starting at the first 16-byte boundary, with
  //   kWideSlackElems elements of slack in all | A-1 direct slots of pD].
  const int A = p.A, H = p.H;
  const int64_t m = p.count, oc = p.chunk, pD = p.direct_total;
  const int64_t P = H * oc;                      // offload positions per block
  const int64_t pw = p.wide_partial ? 2 : 1;     // payload elements per partial element
  const int64_t slack = p.wide_partial ? kWideSlackElems : 0;
  // element offset of owner o's partial region: 16-byte aligned for fp32 partials
  auto pofs = [&](int o) -> int64_t {
    if (!p.wide_partial) return 0;
    const unsigned mis = (unsigned)(reinterpret_cast<uintptr_t>(B.W(o, 0)) & 15u);
    return (int64_t)((16u - mis) & 15u) / p.esize;
  };
  auto slot = [&](int o, int s) { return (o * (A - 1) + other_index(s, o)) * oc; };
  auto dslot = [&](int o, int s) { return pw * P + slack + other_index(s, o) * pD; };
  B.begin(RELAY_PASS_G1);
  for (int s = 0; s < A; ++s)
    for (int h = 0; h < H; ++h)
      for (int o = 0; o < A; ++o)
        if (o != s) B.copy(0, s, B.X(s, o * m + h * oc), {Dst{A + h, B.Hh(h, slot(o, s))}}, oc);
  for (int s = 0; s < A; ++s)
    for (int o = 0; o < A; ++o)
      if (o != s) B.copy(0, s, B.X(s, o * m + P), {Dst{o, B.W(o, dslot(o, s))}}, p.direct_g1);
  if (p.num_groups > 1) {
    B.begin(RELAY_PASS_G2);
    for (int h = 0; h < H; ++h)
      for (int o = 0; o < A; ++o) {
        std::vector<const void*> srcs;
        for (int s = 0; s < A; ++s)
          if (s != o) srcs.push_back(B.Hh(h, slot(o, s)));
        B.reduce(1, A + h, srcs, {Dst{o, B.W(o, pofs(o) + pw * h * oc)}}, oc, false,
                 p.wide_partial ? kFlagOutF32 : 0);
      }
    for (int s = 0; s < A; ++s)
      for (int o = 0; o < A; ++o)
        if (o != s)
          B.copy(1, s, B.X(s, o * m + P + p.direct_g1), {Dst{o, B.W(o, dslot(o, s) + p.direct_g1)}},
                 p.direct_g2);
  }
  B.begin(RELAY_PASS_ACTIVE_REDUCE);
  for (int o = 0; o < A; ++o) {
    // offload positions: the owner's own value first, then the returned partial
    B.reduce(-1, o, {B.X(o, o * m), B.W(o, pofs(o))}, {Dst{o, B.Y(o, 0)}}, P, true,
             p.wide_partial ? kFlagSrc1F32 : 0);
    std::vector<const void*> srcs;
    for (int s = 0; s < A; ++s)
      srcs.push_back(s == o ? (const void*)B.X(o, o * m + P) : (const void*)B.W(o, dslot(o, s)));
    B.reduce(-1, o, srcs, {Dst{o, B.Y(o, P)}}, pD, true);
  }
}

void build_a4_all_gather(Builder& B, const relay_plan_t& p) {
  // item 5: group 1 scatters slice h to helper h and sends the first direct part to
  // every other active; group 2 has each helper broadcast every source's slice h to
  // the A-1 actives that lack it and carries the rest of the direct region
  const int A = p.A, H = p.H;
  const int64_t S = p.count, oc = p.chunk, P = H * oc;
  auto others = [&](int a, int64_t off) {
    std::vector<Dst> d;
    for (int b = 0; b < A; ++b)
      if (b != a) d.push_back(Dst{b, B.Y(b, a * S + off)});
    return d;
  };
  B.begin(RELAY_PASS_G1);
  for (int a = 0; a < A; ++a)
    if (B.X(a, 0) != B.Y(a, a * S)) B.copy(-1, a, B.X(a, 0), {Dst{a, B.Y(a, a * S)}}, S);
  for (int a = 0; a < A; ++a)
    for (int h = 0; h < H; ++h) B.copy(0, a, B.X(a, h * oc), {Dst{A + h, B.Hh(h, a * oc)}}, oc);
  for (int a = 0; a < A; ++a) B.copy(0, a, B.X(a, P), others(a, P), p.direct_g1);
  if (p.num_groups > 1) {
    B.begin(RELAY_PASS_G2);
    for (int h = 0; h < H; ++h)
      for (int k = 0; k < A; ++k) B.copy(1, A + h, B.Hh(h, k * oc), others(k, h * oc), oc);
    // The second direct part reads only inputs and writes output blocks nothing else
    // touches, so the one-launch forms may run it with group 1 (where it shares its loads
    // with the actives' own copies of the same input).
    B.phase(0);
    for (int a = 0; a < A; ++a)
      B.copy(1, a, B.X(a, P + p.direct_g1), others(a, P + p.direct_g1), p.direct_g2);
  }
}

void build_a4_all_to_all(Builder& B, const relay_plan_t& p) {
  // item 7's open lead, coalesced: source s packs, for helper h, slice h of every
  // segment d != s (a gather strided by segmentCount) into one contiguous message; the
  // helper re-packs per destination (one contiguous message of A-1 chunks to each d);
  // d unpacks it (a scatter strided by segmentCount). Direct parts go s -> d in two
  // parts, straight into the output.
  const int A = p.A, H = p.H;
  const int64_t seg = p.count, oc = p.chunk, P = H * oc;
  const bool relay = oc > 0;
  B.begin(relay ? RELAY_PASS_PACK : RELAY_PASS_G1);
  for (int a = 0; a < A; ++a) B.copy(-1, a, B.X(a, a * seg), {Dst{a, B.Y(a, a * seg)}}, seg);
  for (int s = 0; s < A && relay; ++s)
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < A; ++d)
        if (d != s)
          B.copy(0, s, B.X(s, d * seg + h * oc),
                 {Dst{A + h, B.Hh(h, (s * (A - 1) + other_index(d, s)) * oc)}}, oc);
  for (int s = 0; s < A; ++s)
    for (int d = 0; d < A; ++d)
      if (d != s) B.copy(0, s, B.X(s, d * seg + P), {Dst{d, B.Y(d, s * seg + P)}}, p.direct_g1);
  if (!relay) return;
  B.begin(RELAY_PASS_HELPER_FORWARD);
  for (int h = 0; h < H; ++h)
    for (int d = 0; d < A; ++d)
      for (int s = 0; s < A; ++s)
        if (s != d)
          B.copy(1, A + h, B.Hh(h, (s * (A - 1) + other_index(d, s)) * oc),
                 {Dst{d, B.W(d, (h * (A - 1) + other_index(s, d)) * oc)}}, oc);
  for (int s = 0; s < A; ++s)
    for (int d = 0; d < A; ++d)
      if (d != s)
        B.copy(1, s, B.X(s, d * seg + P + p.direct_g1), {Dst{d, B.Y(d, s * seg + P + p.direct_g1)}},
               p.direct_g2);
  B.begin(RELAY_PASS_UNPACK);
  for (int d = 0; d < A; ++d)
    for (int h = 0; h < H; ++h)
      for (int s = 0; s < A; ++s)
        if (s != d)
          B.copy(-1, d, B.W(d, (h * (A - 1) + other_index(s, d)) * oc),
                 {Dst{d, B.Y(d, s * seg + h * oc)}}, oc);
}

}  // namespace

void build_program(const relay_plan_t& p, const Buffers& b, bool in_place,
                   std::vector<Pass>* out) {
  (void)in_place;  // self copies are skipped wherever source and destination coincide
  out->clear();
  if (p.count == 0) return;
  Builder B(p, b, out);
  if (p.A == 2) {
    build_a2(B, p);
  } else {
    switch (p.coll) {
      case RELAY_ALLREDUCE: build_a4_allreduce(B, p); break;
      case RELAY_REDUCE_SCATTER: build_a4_reduce_scatter(B, p); break;
      case RELAY_ALL_GATHER: build_a4_all_gather(B, p); break;
      default: build_a4_all_to_all(B, p); break;
    }
  }
  // drop passes that ended up empty (e.g. a pure-direct group with nothing to move)
  out->erase(std::remove_if(out->begin(), out->end(), [](const Pass& ps) { return ps.segs.empty(); }),
             out->end());
}

std::vector<int> group_ranks(int g, int A, int R) {
  std::vector<int> m;
  m.reserve(R);
  for (int a = 0; a < A; ++a) m.push_back(g * A + a);
  for (int r = 0; r < R; ++r)
    if (r / A != g) m.push_back(r);
  return m;
}

namespace {
// Order of a pass within a phase-synchronized fused call.
int phase_of(relay_pass_kind_t k) {
  switch (k) {
    case RELAY_PASS_G1:
    case RELAY_PASS_PACK: return 0;
    case RELAY_PASS_G2:
    case RELAY_PASS_HELPER_FORWARD: return 1;
    case RELAY_PASS_G3: return 2;
    default: return 3;
  }
}
}  // namespace

void build_multi_program(const std::vector<relay_plan_t>& plans, const std::vector<Buffers>& bufs,
                         const std::vector<std::vector<int>>& global_rank, std::vector<Pass>* out) {
  out->clear();
  std::vector<Pass> merged(4);
  for (int ph = 0; ph < 4; ++ph) merged[ph].kind = RELAY_PASS_G1;
  std::vector<bool> used(4, false);
  for (size_t g = 0; g < plans.size(); ++g) {
    std::vector<Pass> one;
    build_program(plans[g], bufs[g], false, &one);
    for (Pass& ps : one) {
      const int ph = phase_of(ps.kind);
      if (!used[ph]) merged[ph].kind = ps.kind;
      used[ph] = true;
      for (size_t i = 0; i < ps.segs.size(); ++i) {
        SegMeta m = ps.meta[i];
        m.exec_rank = (int8_t)global_rank[g][m.exec_rank];
        for (int d = 0; d < kMaxDst; ++d)
          if (m.dst_rank[d] >= 0) m.dst_rank[d] = (int8_t)global_rank[g][m.dst_rank[d]];
        merged[ph].segs.push_back(ps.segs[i]);
        merged[ph].meta.push_back(m);
      }
    }
  }
  for (int ph = 0; ph < 4; ++ph)
    if (used[ph] && !merged[ph].segs.empty()) out->push_back(std::move(merged[ph]));
}

void fused_phases(const std::vector<Pass>& passes, std::vector<Pass>* out) {
  out->clear();
  std::vector<Pass> ph(passes.size());
  for (size_t p = 0; p < passes.size(); ++p) ph[p].kind = passes[p].kind;
  for (size_t p = 0; p < passes.size(); ++p)
    for (size_t i = 0; i < passes[p].segs.size(); ++i) {
      const SegMeta& m = passes[p].meta[i];
      const size_t q = (m.phase >= 0 && (size_t)m.phase < p) ? (size_t)m.phase : p;
      ph[q].segs.push_back(passes[p].segs[i]);
      ph[q].meta.push_back(m);
    }
  for (Pass& q : ph)
    if (!q.segs.empty()) out->push_back(std::move(q));
}

}  // namespace relay
