// program.h -- internal: the relay schedule as a list of kernel passes.
//
// A pass is one batched launch over a table of segments. A segment is a contiguous
// run of n elements that is either copied from one source to up to four
// destinations, or reduced from up to four sources (summed in ascending order,
// optionally scaled, rounded to the payload type) and stored to up to four
// destinations. Every transfer of a schedule group is a segment whose destination
// belongs to another virtual rank; the host metadata beside each segment records who
// executes it and where its stores land, which is what the link-byte accountant sums.
#pragma once

#include <stdint.h>

#include <string>
#include <vector>

#include "relay.h"

#ifdef __CUDACC__
#define RELAY_HD __host__ __device__
#else
#define RELAY_HD
#endif

namespace relay {

// Per-process caches of device properties hold this many device ordinals; a device past
// them is queried on every call instead.
constexpr int kMaxDevices = 64;

constexpr int kMaxSrc = 4;
constexpr int kMaxDst = 4;

enum SegOp : uint8_t { kOpCopy = 0, kOpReduce = 1 };
enum SegFlag : uint8_t {
  kFlagScale = 1,
  kFlagVector = 2,    // every pointer 16-byte aligned (set at launch)
  kFlagRealign = 4,   // destinations aligned, sources realigned in registers (set at launch)
  kFlagOutF32 = 8,    // bf16 sources, result stored as fp32 (a wide helper partial)
  kFlagSrc1F32 = 16,  // source 1 is fp32, the rest bf16 (an owner adding a wide partial)
  kFlagKeep = 32      // chained launch: a later pass of the same CTA reads what this stores
};

// Device-visible segment descriptor (kernel parameter space).
struct Seg {
  const void* src[kMaxSrc];
  void* dst[kMaxDst];
  int64_t n;      // elements
  int32_t tile0;  // first tile of this segment within its launch
  uint8_t op, nsrc, ndst, flags;
};
static_assert(sizeof(Seg) == 80, "Seg layout");

// Host-only bookkeeping for one segment.
struct SegMeta {
  int8_t group;           // schedule group whose transfer this is; -1: local work only
  int8_t exec_rank;       // rank whose kernel work this is (owner of the sources)
  int8_t dst_rank[kMaxDst];
  // Earliest phase of the one-launch kernel this segment may run in, where its data
  // dependencies allow running it before its own pass; -1: its own pass. Phases stand in
  // for group boundaries only inside that kernel: the per-pass launches keep one launch
  // per schedule group.
  int8_t phase = -1;
};

// Bytes one source / one destination of a segment spans (mixed-width segments carry
// fp32 next to the payload type).
inline int64_t seg_src_bytes(const Seg& s, int k, int E) {
  return s.n * ((k == 1 && (s.flags & kFlagSrc1F32)) ? 4 : E);
}
inline int64_t seg_dst_bytes(const Seg& s, int E) {
  return s.n * ((s.flags & kFlagOutF32) ? 4 : E);
}
RELAY_HD inline bool seg_mixed(const Seg& s) { return (s.flags & (kFlagOutF32 | kFlagSrc1F32)) != 0; }

// bf16 elements of slack in an owner's scratch with fp32 partials. The partials start on
// the first 16-byte boundary within the slack whatever the scratch pointer's alignment
// (bf16 pointers are only 2-byte aligned; fp32 accesses need 4, the vector path 16), and
// the direct slots after the slack keep the 256-byte offset they would have had: a
// misalignment of the direct slots to the 128-byte lines cost ~6% on GB300.
constexpr int64_t kWideSlackElems = 128;

// Every operand of a segment sits at an address its element width divides: payload
// operands at multiples of E, fp32 partials at multiples of 4.
inline bool seg_operands_aligned(const Seg& s, int E) {
  for (int k = 0; k < s.nsrc; ++k) {
    const uintptr_t w = (k == 1 && (s.flags & kFlagSrc1F32)) ? 4 : (uintptr_t)E;
    if (reinterpret_cast<uintptr_t>(s.src[k]) % w) return false;
  }
  const uintptr_t w = (s.flags & kFlagOutF32) ? 4 : (uintptr_t)E;
  for (int d = 0; d < s.ndst; ++d)
    if (reinterpret_cast<uintptr_t>(s.dst[d]) % w) return false;
  return true;
}

struct Pass {
  relay_pass_kind_t kind;
  std::vector<Seg> segs;
  std::vector<SegMeta> meta;
};

// The one-launch kernel's phases: segment i of pass p runs in phase meta.phase if that is
// set, else in phase p; empty phases are dropped. Each phase keeps the kind of the
// earliest pass that lands in it -- program.cpp.
void fused_phases(const std::vector<Pass>& passes, std::vector<Pass>* out);

// Plan (relay_plan_t is the public POD) -- plan.cpp.
relay_status_t make_plan(relay_coll_t coll, int64_t count, relay_dtype_t dtype, int A, int R,
                         const relay_opts_t* opts, relay_plan_t* out, std::string* why);

// Buffers of one call: R entries each (helpers' send/recv unused).
struct Buffers {
  void* const* send;
  void* const* recv;
  void* const* scratch;
};

// Build the passes of a planned collective -- program.cpp. in_place tells the builder
// which in-place form the buffers use (it only removes redundant self copies).
void build_program(const relay_plan_t& p, const Buffers& b, bool in_place,
                   std::vector<Pass>* out);

// Global ranks of group g's local ranks in a fused multi-group call: its A actives
// (ranks g*A .. g*A+A-1, D115998382) first, then every other rank ascending as its
// helpers.
std::vector<int> group_ranks(int g, int A, int R);

// Programs of several groups merged phase by phase (every group's group-1 transfers in
// one launch, then group 2, ...), local ranks renamed to global ones -- program.cpp.
void build_multi_program(const std::vector<relay_plan_t>& plans, const std::vector<Buffers>& bufs,
                         const std::vector<std::vector<int>>& global_rank, std::vector<Pass>* out);

// Launch one pass on `stream` -- passes.cu. Splits into several launches when the
// segment table exceeds one launch's parameter capacity.
// max_ctas > 0 caps each launch's grid (its CTAs then walk the tiles); 0 is one CTA per tile.
// staged: realigned segments may take the TMA-staged kernel (bulk copies into shared
// memory); false keeps them on the register path (buffers that may be host memory).
cudaError_t launch_pass(int dtype, const Pass& pass, float scale, cudaStream_t stream,
                        int max_ctas = 0, bool staged = true);

// One TMA-staged copy of `count` elements whose barrier expects `extra_bytes` more than
// its copies bring, so that every wait runs out (a test of the bounded wait) -- passes.cu.
cudaError_t launch_staged_wait_test(void* dst, const void* src, int64_t count, int dtype,
                                    int extra_bytes, cudaStream_t stream);
// Read and clear the device's fault word (bit 0: a bounded wait in a kernel gave up) --
// passes.cu. Synchronous.
cudaError_t read_device_fault(unsigned* fault);

// Launch every pass of a small call as one cooperative kernel with grid barriers between
// the passes -- passes.cu. Returns false (and launches nothing) when the call does not
// qualify: more than 4 passes, more than 384 segments after alignment splitting, a
// mixed-width segment, or no cooperative launch on this device. Unless `forced`, it also
// declines calls of more than 128 segments that the per-pass launches run faster.
bool launch_fused(int dtype, const std::vector<Pass>& passes, float scale, cudaStream_t stream,
                  cudaError_t* err, bool forced = false);

// The chained launch: a whole call in one ordinary launch whose CTAs never wait for one
// another. The passes' segments are cut into pieces so that every dependency between
// passes links identical element ranges, pieces that touch the same bytes (one writing)
// form a group, and one CTA runs tile t of every piece of a group in pass order, with a
// block barrier between passes -- chain.cpp (analysis), chain_kernel.cu (kernel).
constexpr int kChainMaxPieces = 384;
struct ChainPlan {
  std::vector<Seg> segs;        // every group's pieces contiguous, in pass order
  std::vector<uint8_t> level;   // pass of each piece
  // Per piece, bit k: source k is scratch that an earlier pass of the group wrote and that
  // nothing touches after this read. Its CTA drops those bytes' whole 128-byte lines from
  // L2 without a write-back once the tile's last pass is done.
  std::vector<uint8_t> drop;
  std::vector<int32_t> gfirst;  // first piece of each group, then one past the last
  std::vector<int64_t> gn;      // elements of each piece of the group
  // Per group, 1: every operand is 16-byte aligned at the group's first element. Every
  // executor path (the mixed-width one included) then gives thread t the same elements of
  // every piece, so each dependency between passes stays inside one thread and needs no
  // block barrier.
  std::vector<uint8_t> local;
};
struct ByteRange {
  uintptr_t lo, hi;  // [lo, hi)
};
// scratch: the call's scratch buffers whose dead lines may be dropped (device memory).
bool build_chain(const std::vector<Pass>& passes, int E, const std::vector<ByteRange>& scratch,
                 ChainPlan* out, std::string* why);
bool check_chain(const ChainPlan& c, int E, const std::vector<ByteRange>& scratch,
                 std::string* why);
// Launches the chained kernel; false (nothing launched) when the program does not fit one
// launch's parameters.
bool launch_chain(int dtype, const ChainPlan& c, float scale, cudaStream_t stream,
                  cudaError_t* err);

// SMs of the current device (cached per device) -- passes.cu.
int sm_count();

// Record `msg` as this thread's last error and return `st` -- abi.cpp.
relay_status_t report_error(relay_status_t st, const std::string& msg);

// Tile size in elements for a payload of esize bytes (shared by host tiling and the
// kernel).
constexpr int kThreads = 256;
constexpr int kVecBytes = 16;
constexpr int kUnroll = 4;
constexpr int64_t kTileBytes = (int64_t)kThreads * kUnroll * kVecBytes;  // 16 KiB
inline int64_t tile_elems(int esize) { return kTileBytes / esize; }

inline int esize_of(int dtype) { return dtype == RELAY_BF16 ? 2 : 4; }

}  // namespace relay
