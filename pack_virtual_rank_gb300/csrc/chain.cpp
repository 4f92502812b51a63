// chain.cpp -- host side of the chained launch: a whole call in one ordinary launch, with
// no grid-wide barrier and no wait of one CTA on another.
//
// A call's passes run in order because pass p+1 reads what pass p wrote (a relay chunk
// landing in a helper's slot, then the helper's reduction of that slot), or writes what an
// earlier pass read (in-place forms). Every such dependency here is elementwise: element i
// of a consumer touches exactly element i of its producer. So the segments of all passes
// can be cut into pieces whose dependent ranges coincide, the pieces that touch the same
// bytes (one of them writing) joined into a group, and each group tiled: one CTA runs tile
// t of every piece of a group, in pass order, with a block barrier between passes. Nothing
// one CTA reads or writes is touched by another CTA, so no CTA ever waits for another,
// and the schedule's transfers and reductions all still run, each in its pass or in the
// earlier one-launch phase its data allow (the cooperative launch's phases).
//
// Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)", items 3 and 5:
// in the latency-bound regime a group boundary costs a round trip; here it costs a block
// barrier inside the CTA that holds both sides of it.
#include <algorithm>
#include <numeric>
#include <string>
#include <vector>

#include "program.h"

namespace relay {
namespace {

struct Piece {
  Seg s;
  int pass;
  int order;  // position among all pieces in build order (keeps groups deterministic)
};

struct Operand {
  uintptr_t lo, hi;  // bytes [lo, hi)
  int piece;
  bool write;
  int width;         // bytes per element of this operand (an fp32 partial next to bf16: 4)
};

// Bytes per element of a segment's source k / destinations (program.h: mixed-width
// segments carry an fp32 partial next to the payload type).
int src_width(const Seg& s, int k, int E) { return (k == 1 && (s.flags & kFlagSrc1F32)) ? 4 : E; }
int dst_width(const Seg& s, int E) { return (s.flags & kFlagOutF32) ? 4 : E; }

void operands(const std::vector<Piece>& ps, int E, std::vector<Operand>* out) {
  out->clear();
  for (int i = 0; i < (int)ps.size(); ++i) {
    const Seg& s = ps[i].s;
    for (int k = 0; k < s.nsrc; ++k) {
      const int w = src_width(s, k, E);
      const uintptr_t lo = reinterpret_cast<uintptr_t>(s.src[k]);
      out->push_back(Operand{lo, lo + (uintptr_t)s.n * (uintptr_t)w, i, false, w});
    }
    const int w = dst_width(s, E);
    for (int d = 0; d < s.ndst; ++d) {
      const uintptr_t lo = reinterpret_cast<uintptr_t>(s.dst[d]);
      out->push_back(Operand{lo, lo + (uintptr_t)s.n * (uintptr_t)w, i, true, w});
    }
  }
  std::sort(out->begin(), out->end(), [](const Operand& a, const Operand& b) {
    return a.lo != b.lo ? a.lo < b.lo : a.hi < b.hi;
  });
}

// Every pair of operands of different pieces that overlap, at least one of them written:
// fn(a, b). Operands are sorted by start, so the partners of operand i are the ones after
// it that start before it ends.
template <class Fn>
void for_each_conflict(const std::vector<Operand>& ops, Fn fn) {
  for (size_t i = 0; i < ops.size(); ++i)
    for (size_t j = i + 1; j < ops.size() && ops[j].lo < ops[i].hi; ++j)
      if (ops[i].piece != ops[j].piece && (ops[i].write || ops[j].write)) fn(ops[i], ops[j]);
}

// Every pair of copies of one pass whose sources overlap element for element (same width,
// offsets on the element grid): fn(a, b) with their source operands. Such copies can share
// one load once their source ranges coincide.
template <class Fn>
void for_each_shared_read(const std::vector<Operand>& ops, const std::vector<Piece>& ps, Fn fn) {
  for (size_t i = 0; i < ops.size(); ++i)
    for (size_t j = i + 1; j < ops.size() && ops[j].lo < ops[i].hi; ++j) {
      const Operand &a = ops[i], &b = ops[j];
      if (a.write || b.write || a.piece == b.piece || a.width != b.width) continue;
      const Piece &pa = ps[a.piece], &pb = ps[b.piece];
      if (pa.pass != pb.pass || pa.s.op != kOpCopy || pb.s.op != kOpCopy) continue;
      if ((b.lo - a.lo) % (uintptr_t)a.width) continue;  // sorted: b.lo >= a.lo
      fn(a, b);
    }
}

int find(std::vector<int>& parent, int x) {
  while (parent[x] != x) {
    parent[x] = parent[parent[x]];
    x = parent[x];
  }
  return x;
}

ByteRange src_range(const Seg& s, int k, int E) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(s.src[k]);
  return ByteRange{lo, lo + (uintptr_t)s.n * (uintptr_t)src_width(s, k, E)};
}
ByteRange dst_range(const Seg& s, int d, int E) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(s.dst[d]);
  return ByteRange{lo, lo + (uintptr_t)s.n * (uintptr_t)dst_width(s, E)};
}
bool overlap(const ByteRange& a, const ByteRange& b) { return a.lo < b.hi && b.lo < a.hi; }
bool same(const ByteRange& a, const ByteRange& b) { return a.lo == b.lo && a.hi == b.hi; }
bool inside_any(const ByteRange& r, const std::vector<ByteRange>& v) {
  for (const ByteRange& b : v)
    if (r.lo >= b.lo && r.hi <= b.hi) return true;
  return false;
}
// Sources a segment's kernel reads: a copy reads source 0 only.
int sources_read(const Seg& s) { return s.op == kOpCopy ? 1 : s.nsrc; }

// A piece whose operands all sit on 16-byte boundaries: the kernel runs it with thread t on
// 16-byte payload vectors t, t + 256, ... (elements 8v .. 8v + 7 of a bf16 piece, and the
// same elements of an fp32 partial beside it) and the scalar tail elements t, t + 256, ...
// of every tile, whichever path it takes.
bool thread_local_piece(const Seg& s) {
  for (int k = 0; k < sources_read(s); ++k)
    if (reinterpret_cast<uintptr_t>(s.src[k]) % 16) return false;
  for (int d = 0; d < s.ndst; ++d)
    if (reinterpret_cast<uintptr_t>(s.dst[d]) % 16) return false;
  return true;
}

// Bit k of drop[i]: source k of piece i lies in scratch, an earlier pass of the piece's
// group wrote exactly those bytes, and nothing of the group touches them after this read
// (nothing of another group touches them at all: a writer and its readers share a group).
void mark_drops(ChainPlan* c, int E, const std::vector<ByteRange>& scratch) {
  c->drop.assign(c->segs.size(), 0);
  if (scratch.empty()) return;
  for (size_t g = 0; g + 1 < c->gfirst.size(); ++g) {
    const int f = c->gfirst[g], l = c->gfirst[g + 1];
    for (int i = f; i < l; ++i) {
      const Seg& s = c->segs[i];
      for (int k = 0; k < sources_read(s); ++k) {
        const ByteRange r = src_range(s, k, E);
        if (!inside_any(r, scratch)) continue;
        bool produced = false, live = false;
        for (int j = f; j < l && !live; ++j) {
          const Seg& t = c->segs[j];
          for (int d = 0; d < t.ndst; ++d) {
            const ByteRange w = dst_range(t, d, E);
            if (c->level[j] < c->level[i]) produced |= same(w, r);
            else live |= overlap(w, r);  // rewritten by this pass or a later one
          }
          if (c->level[j] > c->level[i])
            for (int q = 0; q < sources_read(t); ++q) live |= overlap(src_range(t, q, E), r);
        }
        if (produced && !live) c->drop[i] |= (uint8_t)(1u << k);
      }
    }
  }
}

Seg advance(const Seg& s, int64_t e, int64_t n, int E) {
  Seg t = s;
  for (int k = 0; k < t.nsrc; ++k) t.src[k] = static_cast<const char*>(t.src[k]) + e * src_width(s, k, E);
  for (int d = 0; d < t.ndst; ++d) t.dst[d] = static_cast<char*>(t.dst[d]) + e * dst_width(s, E);
  t.n = n;
  return t;
}

}  // namespace

namespace {

// merge_reads: also cut copies of one pass at each other's source boundaries and merge the
// ones that then read the same bytes (see build_chain).
bool build_chain_with(const std::vector<Pass>& passes, int E, const std::vector<ByteRange>& scratch,
                      bool merge_reads, ChainPlan* out, std::string* why) {
  auto fail = [&](const std::string& m) {
    if (why) *why = m;
    return false;
  };
  if (passes.size() > 200) return fail("too many passes");
  // A piece runs in its segment's one-launch phase: its own pass, or an earlier one where
  // the program builder found that its data allow it (program.h, SegMeta::phase); the
  // host's hazard checks verify those phases for the cooperative launch as well.
  std::vector<Piece> ps;
  for (size_t p = 0; p < passes.size(); ++p)
    for (size_t i = 0; i < passes[p].segs.size(); ++i) {
      const Seg& s = passes[p].segs[i];
      if (s.n <= 0) continue;
      // only bf16 payloads widen, and every fp32 operand must be 4-byte aligned
      if (seg_mixed(s) && (E != 2 || !seg_operands_aligned(s, E)))
        return fail("mixed-width segment on a payload other than bf16, or misaligned");
      const int ph = i < passes[p].meta.size() ? passes[p].meta[i].phase : -1;
      ps.push_back(Piece{s, (ph >= 0 && (size_t)ph < p) ? ph : (int)p, (int)ps.size()});
    }
  if (ps.empty()) return fail("nothing to run");

  // 1. Refine: cut pieces until every conflicting pair of operands covers the same bytes.
  std::vector<Operand> ops;
  for (int round = 0;; ++round) {
    if (round > 64 || ps.size() > (size_t)kChainMaxPieces) return fail("does not refine");
    operands(ps, E, &ops);
    std::vector<std::vector<int64_t>> cuts(ps.size());
    bool bad = false;
    for_each_conflict(ops, [&](const Operand& a, const Operand& b) {
      if (ps[a.piece].pass == ps[b.piece].pass) bad = true;  // a race inside one pass
      if (a.width != b.width) bad = true;                    // not element for element
      if (a.lo == b.lo && a.hi == b.hi) return;
      const uintptr_t lo = std::max(a.lo, b.lo), hi = std::min(a.hi, b.hi);
      for (const Operand* x : {&a, &b}) {
        const uintptr_t w = (uintptr_t)x->width;
        if ((lo - x->lo) % w || (hi - x->lo) % w) bad = true;
        if (x->lo < lo) cuts[x->piece].push_back((int64_t)((lo - x->lo) / w));
        if (x->hi > hi) cuts[x->piece].push_back((int64_t)((hi - x->lo) / w));
      }
    });
    if (bad) return fail("overlap that is not elementwise");
    if (merge_reads)
      for_each_shared_read(ops, ps, [&](const Operand& a, const Operand& b) {
        if (a.lo == b.lo && a.hi == b.hi) return;
        const uintptr_t lo = std::max(a.lo, b.lo), hi = std::min(a.hi, b.hi);
        for (const Operand* x : {&a, &b}) {
          const uintptr_t w = (uintptr_t)x->width;
          if (x->lo < lo) cuts[x->piece].push_back((int64_t)((lo - x->lo) / w));
          if (x->hi > hi) cuts[x->piece].push_back((int64_t)((hi - x->lo) / w));
        }
      });
    bool any = false;
    std::vector<Piece> next;
    next.reserve(ps.size());
    for (size_t i = 0; i < ps.size(); ++i) {
      std::vector<int64_t>& c = cuts[i];
      c.push_back(0);
      c.push_back(ps[i].s.n);
      std::sort(c.begin(), c.end());
      c.erase(std::unique(c.begin(), c.end()), c.end());
      any |= c.size() > 2;
      for (size_t k = 0; k + 1 < c.size(); ++k)
        next.push_back(Piece{advance(ps[i].s, c[k], c[k + 1] - c[k], E), ps[i].pass, 0});
    }
    for (size_t i = 0; i < next.size(); ++i) next[i].order = (int)i;
    ps.swap(next);
    if (!any) break;
  }

  // 1b. Copies of one pass that read exactly the same bytes become one copy with all their
  // destinations (at most kMaxDst): one load per element instead of one per copy. Every
  // store of the schedule still happens. (An all-gather's self copy and its scatter of the
  // same input to helpers and peers are such copies.)
  if (merge_reads) {
    std::vector<Piece> next;
    next.reserve(ps.size());
    std::vector<int> open;  // indices into next of copies that may still absorb another
    for (const Piece& p : ps) {
      bool merged = false;
      if (p.s.op == kOpCopy)
        for (int j : open) {
          Seg& t = next[j].s;
          if (next[j].pass != p.pass || t.src[0] != p.s.src[0] || t.n != p.s.n ||
              t.flags != p.s.flags || t.ndst + p.s.ndst > kMaxDst)
            continue;
          for (int d = 0; d < p.s.ndst; ++d) t.dst[t.ndst + d] = p.s.dst[d];
          t.ndst = (uint8_t)(t.ndst + p.s.ndst);
          merged = true;
          break;
        }
      if (merged) continue;
      if (p.s.op == kOpCopy) open.push_back((int)next.size());
      next.push_back(p);
    }
    for (size_t i = 0; i < next.size(); ++i) next[i].order = (int)i;
    ps.swap(next);
    operands(ps, E, &ops);
  }

  // 2. Join conflicting pieces into groups. A piece whose output a later pass reads keeps
  // its stores in L2 (no streaming hint): its own CTA reads them back right away.
  std::vector<int> parent(ps.size());
  std::iota(parent.begin(), parent.end(), 0);
  for (Piece& p : ps) p.s.flags &= (uint8_t)~kFlagKeep;
  for_each_conflict(ops, [&](const Operand& a, const Operand& b) {
    const int ra = find(parent, a.piece), rb = find(parent, b.piece);
    if (ra != rb) parent[std::max(ra, rb)] = std::min(ra, rb);
    if (a.write && !b.write && ps[a.piece].pass < ps[b.piece].pass) ps[a.piece].s.flags |= kFlagKeep;
    if (b.write && !a.write && ps[b.piece].pass < ps[a.piece].pass) ps[b.piece].s.flags |= kFlagKeep;
  });
  std::vector<std::vector<int>> members(ps.size());
  for (int i = 0; i < (int)ps.size(); ++i) members[find(parent, i)].push_back(i);

  // 3. Lay the groups out, each in pass order (build order within a pass).
  out->segs.clear();
  out->level.clear();
  out->gfirst.clear();
  out->gn.clear();
  for (auto& m : members) {
    if (m.empty()) continue;
    std::stable_sort(m.begin(), m.end(), [&](int a, int b) { return ps[a].pass < ps[b].pass; });
    const int64_t n = ps[m[0]].s.n;
    out->gfirst.push_back((int32_t)out->segs.size());
    out->gn.push_back(n);
    for (int i : m) {
      if (ps[i].s.n != n) return fail("a group's pieces differ in length");
      out->segs.push_back(ps[i].s);
      out->level.push_back((uint8_t)ps[i].pass);
    }
  }
  out->gfirst.push_back((int32_t)out->segs.size());
  mark_drops(out, E, scratch);
  out->local.assign(out->gn.size(), 0);
  for (size_t g = 0; g < out->gn.size(); ++g) {
    bool local = true;
    for (int i = out->gfirst[g]; i < out->gfirst[g + 1]; ++i) local &= thread_local_piece(out->segs[i]);
    out->local[g] = local ? 1 : 0;
  }
  return true;
}

}  // namespace

// Copies of one pass that read the same bytes share their loads where the program still
// fits one launch that way; otherwise the program is built without that merge.
bool build_chain(const std::vector<Pass>& passes, int E, const std::vector<ByteRange>& scratch,
                 ChainPlan* out, std::string* why) {
  return build_chain_with(passes, E, scratch, true, out, why) ||
         build_chain_with(passes, E, scratch, false, out, why);
}

// An independent re-check of a chained program (host hazard checks): no two pieces of
// different groups touch the same bytes with either writing, and no two pieces of one
// group's pass do. Quadratic in the pieces, so only run when the caller asks for checks.
bool check_chain(const ChainPlan& c, int E, const std::vector<ByteRange>& scratch,
                 std::string* why) {
  const int G = (int)c.gn.size();
  if (c.drop.size() != c.segs.size() || c.local.size() != c.gn.size()) {
    *why = "chained program without a drop mask per piece or a flag per group";
    return false;
  }
  for (int g = 0; g < G; ++g)
    for (int i = c.gfirst[g]; c.local[g] && i < c.gfirst[g + 1]; ++i) {
      const Seg& s = c.segs[i];
      bool ok = true;
      for (int k = 0; k < sources_read(s); ++k) ok &= reinterpret_cast<uintptr_t>(s.src[k]) % 16 == 0;
      for (int d = 0; d < s.ndst; ++d) ok &= reinterpret_cast<uintptr_t>(s.dst[d]) % 16 == 0;
      if (!ok) {
        *why = "chained group " + std::to_string(g) + " runs without block barriers but piece " +
               std::to_string(i) + " is off the 16-byte grid";
        return false;
      }
    }
  std::vector<int> group(c.segs.size());
  for (int g = 0; g < G; ++g)
    for (int i = c.gfirst[g]; i < c.gfirst[g + 1]; ++i) {
      group[i] = g;
      if (c.segs[i].n != c.gn[g]) {
        *why = "chained group " + std::to_string(g) + " has pieces of different lengths";
        return false;
      }
      if (i > c.gfirst[g] && c.level[i] < c.level[i - 1]) {
        *why = "chained group " + std::to_string(g) + " is not in pass order";
        return false;
      }
    }
  auto rng = [&](const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return std::make_pair(lo, lo + (uintptr_t)bytes);
  };
  auto ov = [](std::pair<uintptr_t, uintptr_t> a, std::pair<uintptr_t, uintptr_t> b) {
    return a.first < b.second && b.first < a.second;
  };
  for (size_t i = 0; i < c.segs.size(); ++i)
    for (size_t j = 0; j < c.segs.size(); ++j) {
      if (i == j) continue;
      const bool same_group = group[i] == group[j];
      if (same_group && c.level[i] != c.level[j]) continue;  // ordered by the block barrier
      const Seg &a = c.segs[i], &b = c.segs[j];
      for (int d = 0; d < a.ndst; ++d) {
        const auto w = rng(a.dst[d], seg_dst_bytes(a, E));
        bool hit = false;
        for (int k = 0; k < b.nsrc; ++k) hit |= ov(w, rng(b.src[k], seg_src_bytes(b, k, E)));
        for (int k = 0; k < b.ndst; ++k) hit |= ov(w, rng(b.dst[k], seg_dst_bytes(b, E)));
        if (hit) {
          *why = "chained pieces " + std::to_string(i) + " and " + std::to_string(j) +
                 (same_group ? " of one pass of a group" : " of different groups") +
                 " touch the same bytes, one of them writing";
          return false;
        }
      }
    }
  // A dropped source: scratch, written exactly by an earlier pass of its group, and touched
  // by nothing after the read (no piece of another group, no later pass of its own group,
  // no write in its own pass).
  for (size_t i = 0; i < c.segs.size(); ++i)
    for (int k = 0; k < 8; ++k) {
      if (!((c.drop[i] >> k) & 1)) continue;
      const Seg& a = c.segs[i];
      auto bad = [&](const std::string& m) {
        *why = "chained piece " + std::to_string(i) + " drops source " + std::to_string(k) + ": " + m;
        return false;
      };
      if (k >= sources_read(a)) return bad("a source the piece does not read");
      const auto r = rng(a.src[k], seg_src_bytes(a, k, E));
      const ByteRange br{r.first, r.second};
      if (!inside_any(br, scratch)) return bad("not inside a scratch buffer");
      bool produced = false;
      for (size_t j = 0; j < c.segs.size(); ++j) {
        const Seg& b = c.segs[j];
        const bool other = group[j] != group[i];
        const bool later = !other && c.level[j] > c.level[i];
        const bool earlier = !other && c.level[j] < c.level[i];
        for (int d = 0; d < b.ndst; ++d) {
          const auto w = rng(b.dst[d], seg_dst_bytes(b, E));
          if (earlier) produced |= w == r;
          else if (ov(w, r)) return bad("written again, or by another group");
        }
        if (other || later)
          for (int q = 0; q < sources_read(b); ++q)
            if (ov(rng(b.src[q], seg_src_bytes(b, q, E)), r))
              return bad("read after the drop, or by another group");
      }
      if (!produced) return bad("no earlier pass of its group wrote exactly these bytes");
    }
  return true;
}

}  // namespace relay
