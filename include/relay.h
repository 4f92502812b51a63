/*
 * relay.h -- C ABI of the GB300 sharded relay collectives.
 *
 * A relay collective runs among A "active" ranks (0..A-1) of an R-rank node and
 * recruits the H = R - A idle ranks (A..R-1, helper h = rank A+h) as relay helpers.
 * Here every virtual rank is a set of buffers in ONE GPU's HBM: a transfer over a
 * (src, dst) "link" is a store from a kernel executed for rank src into memory owned
 * by rank dst, and each serialized group of the schedule is one batched kernel launch
 * on the caller's stream.
 *
 * Sources (page "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)",
 * torchrec pull request #4570, and the commits of its stack, cited by their
 * Differential Revision number):
 *   cost model       -- the paragraph before summary item 1
 *   items 1..7       -- the numbered items of that page's summary
 *   D115998367       -- zero-chunk per-group direct fallback
 *   D115998376       -- reduce-scatter semantics, in-place convention, SUM/AVG only
 *   D115998385       -- all-gather semantics and in-place convention
 *   D115998370       -- all-to-all semantics (out-of-place only), helper sizing
 *   D115998382       -- actives are consecutive local ranks; A in {2, 4}; R > A
 *   D115998394, D115998388 -- helper-buffer size contract and its literals
 *
 * Ownership: the caller allocates and owns every buffer and the stream. The library
 * allocates no device memory and keeps no state between calls. Calls are asynchronous
 * on `stream`; a status reports only validation and launch errors.
 *
 * Element counts are in ELEMENTS of the payload type; byte figures say so.
 */
#ifndef RELAY_H
#define RELAY_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RELAY_ABI_VERSION 1
#define RELAY_MAX_RANKS 64
#define RELAY_ALIGN_ELEMS 128 /* chunks are aligned down to 128 elements (D115998394) */

typedef enum {
  RELAY_OK = 0,
  RELAY_ERR_INVALID_ARGUMENT = 1, /* bad A/R/dtype/scale/pointer/alias/size */
  RELAY_ERR_UNSUPPORTED = 2,      /* valid request this library does not execute */
  RELAY_ERR_CUDA = 3              /* a CUDA launch or event call failed */
} relay_status_t;

typedef enum { RELAY_F32 = 0, RELAY_BF16 = 1, RELAY_I32 = 2 } relay_dtype_t;

typedef enum {
  RELAY_ALLREDUCE = 0,
  RELAY_REDUCE_SCATTER = 1,
  RELAY_ALL_GATHER = 2,
  RELAY_ALL_TO_ALL = 3
} relay_coll_t;

/* Schedule the planner picked. */
typedef enum {
  RELAY_KIND_RELAY = 0,      /* helpers carry the relay chunks (items 1, 2, 4, 5, 6) */
  RELAY_KIND_ZERO_CHUNK = 1, /* A=2 chunk aligned down to 0: direct halves (D115998367) */
  RELAY_KIND_DIRECT = 2,     /* pure-direct below the crossover (items 3, 4, 7) */
  RELAY_KIND_LEGACY = 3      /* A=2 numChunks = H+1, three groups (item 1, "before") */
} relay_kind_t;

/* Schedule request. */
typedef enum {
  RELAY_SCHEDULE_AUTO = 0,   /* relay iff the per-active-rank input passes the crossover */
  RELAY_SCHEDULE_RELAY = 1,  /* relay whenever the geometry allows it */
  RELAY_SCHEDULE_DIRECT = 2, /* pure-direct */
  RELAY_SCHEDULE_LEGACY = 3  /* A=2 only: the three-group numChunks = H+1 schedule */
} relay_schedule_t;

/* relay_opts_t.flags */
#define RELAY_FLAG_CHECK_HAZARDS 1 /* host checks before launching: every segment lies
                                      inside a declared buffer, and no launch writes what
                                      another segment of it reads or writes (O(segs^2)) */
#define RELAY_FLAG_DRY_RUN 2       /* validate, plan, build and check; launch nothing */
#define RELAY_FLAG_SEPARATE_PASSES 4 /* one launch per pass even for small calls */
#define RELAY_FLAG_FUSED_PASSES 8  /* one cooperative launch for the whole call whenever it
                                      qualifies, whatever its size */
#define RELAY_FLAG_CHAINED 32      /* one chained launch for the whole call whenever its
                                      program allows it (the default does the same; the flag
                                      documents the intent) */
#define RELAY_FLAG_KEEP_SCRATCH 64 /* chained launch: write every scratch line back to
                                      memory. By default a CTA drops from L2, without a
                                      write-back, the whole 128-byte lines of device-memory
                                      scratch that an earlier pass of its chain wrote and that
                                      nothing reads again in the call */
/* Launch policy. A call that records pass events, or sets RELAY_FLAG_SEPARATE_PASSES,
 * launches each pass separately. Any other call runs as ONE chained launch where its
 * program allows: the segments of all passes are cut into pieces so that each dependency
 * between passes links identical element ranges; pieces that touch the same bytes, one of
 * them writing, form a group; one CTA runs tile t of every piece of a group in pass order
 * with a block barrier between passes. No CTA waits for another, and a consumer reads
 * from L2 what its own CTA just wrote. It takes programs whose pieces number at most 384
 * after cutting (fp32 partials of a bf16 payload included). Else a call of at most
 * RELAY_FUSED_MAX_BYTES runs as one cooperative launch (at most 4 passes
 * and 384 segments after alignment splitting, no mixed-width segments; passes separated
 * by grid-wide barriers), and anything else pass by pass.
 * relay_last_launch() names the form the calling thread's last call took. */
#define RELAY_FUSED_MAX_BYTES (256ll << 20)
#define RELAY_FLAG_PAYLOAD_PARTIAL 16 /* 4-active reduce-scatter, bf16 payload. By default
                                      (flag clear) each helper's partial crosses to its owner
                                      in fp32: twice the bytes of that hop and H*chunk + 128
                                      more elements of owner scratch; the owner adds its own
                                      value and the partial, scales once and rounds once, so
                                      results are within one bf16 ulp of the fp32-accumulated
                                      sum (and of the exact sum unless a tiny term needs more
                                      than 24 bits next to large ones). With the flag set the
                                      partial crosses in the payload type, one payload-sized
                                      chunk per return hop as in the link model (item 6): it
                                      is rounded to bf16 at the helper before the owner adds,
                                      a second rounding that can move a result several ulps
                                      off the exact sum on cancelling inputs. fp32 and int32
                                      payloads are unaffected. */

typedef struct relay_opts {
  int32_t offload_permille;      /* A=4 allreduce / reduce-scatter / all-gather offload share;
                                    <0: 500 (item 4) */
  int32_t schedule;              /* relay_schedule_t */
  int64_t relay_threshold_bytes; /* <0: per-collective default crossover (items 3, 4, 7) */
  void* pass_events;             /* NULL, or cudaEvent_t[n_pass_events]: event i is recorded on
                                    the stream before pass i and event n_passes after the last;
                                    needs n_pass_events >= n_passes + 1 */
  int32_t n_pass_events;
  int32_t flags;                 /* RELAY_FLAG_* */
} relay_opts_t;

/* Fill `opts` with the defaults (every field "use the default"). */
void relay_opts_init(relay_opts_t* opts);

/*
 * Schedule geometry (plan). Integer only; identical on every machine.
 *
 * count is the per-group count the collective is called with:
 *   allreduce: elements per rank (input = output = count);
 *   reduce-scatter: recvCount (input = A*count, output = count) (D115998376);
 *   all-gather: sendCount (input = count, output = A*count) (D115998385);
 *   all-to-all: segmentCount (input = output = A*count) (D115998370).
 *
 * A = 2 (item 1): numChunks = H+2, chunk = align_down(count / numChunks, 128); relay
 *   chunk h (offset h*chunk) goes to helper h; the direct region follows the relay
 *   region: dirA = [H*chunk, (H+1)*chunk) rides group 1, dirB = the rest rides group 2.
 *   chunk == 0 -> zero-chunk fallback: dirA = count/2 at offset 0, dirB = the rest.
 *   Legacy (item 1, before): numChunks = H+1, three groups, direct = count - H*chunk.
 *   Below the crossover: one full direct exchange (item 3).
 * A = 4: chunk ("oc") is the offload slice each helper carries; direct_total = pD =
 *   count - H*oc. allreduce, reduce-scatter and all-gather take
 *   oc = align_down(permille*count/(1000*H)) (item 4; 500 permille = equal direct and
 *   offload regions). allreduce: owner slice = align_down(pD/A), the last owner takes
 *   the remainder. reduce-scatter (item 6): direct part split direct_g1 =
 *   align_down((A-1)*pD/A) in group 1 and the rest in group 2. all-gather (item 5):
 *   direct split 1:(A-1), direct_g1 = align_down(pD/A). all-to-all (item 7, coalesced
 *   helper offload): oc = align_down(count/(2(A-1)+H)); group 1 carries (A-1)*oc of
 *   direct, group 2 the rest. Pure-direct (oc = 0): allreduce keeps two groups (direct
 *   reduce-scatter + all-gather); the others take one.
 */
typedef struct relay_plan {
  int32_t coll, dtype, A, R, H, esize;
  int32_t kind;            /* relay_kind_t */
  int32_t num_groups;      /* serialized groups of the schedule (cost model) */
  int32_t offload_permille;
  int32_t wide_partial;    /* 1: 4-active reduce-scatter partials cross in fp32 (bf16
                              payload without RELAY_FLAG_PAYLOAD_PARTIAL) */
  int64_t count;
  int64_t chunk;           /* A=2: relay chunk; A=4: offload slice per helper */
  int64_t relay_total;     /* H * chunk */
  int64_t dirA_offset, dirA_size, dirB_size; /* A=2 direct regions */
  int64_t direct_total;    /* A=4: pD */
  int64_t direct_g1, direct_g2;              /* A=4 RS/AG/A2A direct split */
  int64_t owner_slice, owner_slice_last;     /* A=4 allreduce owner slices */
  int64_t helper_elems;    /* scratch each helper needs (elements) */
  int64_t active_scratch_elems; /* scratch each active needs (elements) */
  int64_t input_elems, output_elems; /* per active rank */
} relay_plan_t;

/* Plan a collective. opts may be NULL. INVALID_ARGUMENT on A not in {2,4}, R <= A,
 * R > RELAY_MAX_RANKS, bad dtype/coll, permille outside [0,1000], byte-size overflow,
 * or LEGACY at A=4 / LEGACY whose chunk aligns down to 0. */
relay_status_t relay_plan(relay_coll_t coll, size_t count, relay_dtype_t dtype, int A, int R,
                          const relay_opts_t* opts, relay_plan_t* out);

/* Link-byte accountant (cost model): out[(g*R + src)*R + dst] = payload BYTES the
 * executed schedule moves from rank src to rank dst in serialized group g, counted
 * from the very segments the kernels execute. cap is the length of `out` in entries
 * and must be >= num_groups*R*R. Returns INVALID_ARGUMENT if it is not. */
relay_status_t relay_plan_link_bytes(const relay_plan_t* plan, uint64_t* out, size_t cap);

/* Cost model: sum over groups of the largest (src, dst) entry, in BYTES. */
uint64_t relay_plan_cost_bytes(const relay_plan_t* plan);

/* Pass descriptions: one entry per kernel pass the executed schedule launches, in
 * launch order. Returns the number of passes (even when cap is smaller), or -1 on a
 * bad plan. in_place selects the in-place variant where it changes the passes. */
typedef enum {
  RELAY_PASS_G1 = 0,            /* group 1: transfers (scatter to helpers + direct) */
  RELAY_PASS_G2 = 1,            /* group 2: helper reduce/forward + direct transfers */
  RELAY_PASS_G3 = 2,            /* legacy group 3: direct exchange */
  RELAY_PASS_ACTIVE_REDUCE = 3, /* actives' own + received, scale, cast */
  RELAY_PASS_PACK = 4,          /* all-to-all: gather strided by segmentCount */
  RELAY_PASS_HELPER_FORWARD = 5,/* all-to-all: helper per-destination coalesced forward */
  RELAY_PASS_UNPACK = 6         /* all-to-all: scatter strided by segmentCount */
} relay_pass_kind_t;

typedef struct relay_pass_info {
  int32_t kind;     /* relay_pass_kind_t */
  int32_t num_segments;
  int64_t bytes_read, bytes_written; /* algorithmic bytes of the pass */
} relay_pass_info_t;

int relay_plan_passes(const relay_plan_t* plan, int in_place, relay_pass_info_t* out, int cap);
const char* relay_pass_name(int kind);

/* Scratch sizes of a plan, in elements (the plan's helper_elems / active_scratch_elems):
 * what each helper and each active must be given for this schedule. */
int64_t relay_helper_size(const relay_plan_t* plan);
int64_t relay_active_scratch_size(const relay_plan_t* plan);

/* The page's helper-buffer contract for one group (what its distributed layer
 * allocates per helper), in elements: the passthrough size with num_chunks = (R-A)+1 at
 * A=2 (D115998370); 2*count for the 4-active allreduce (D115998382) and reduce-scatter
 * (item 6); A*count for the 4-active all-gather (D115998397); 1 for the 4-active
 * all-to-all, which the page runs pure-direct (D115998358). -1 on bad arguments. This
 * library's schedules never need more than the contract, except the coalesced 4-active
 * all-to-all, which the page does not have. */
int64_t relay_helper_contract_size(relay_coll_t coll, int64_t count, int A, int R);

/* Helper-buffer size contract of the page's distributed layer (D115998394, D115998388,
 * D115998370): min(count_g, A * align_down(count_g / num_chunks, 128)); count_g when the
 * aligned chunk is 0 (the page only says the fallback can over-allocate). */
int64_t relay_passthrough_helper_size(int64_t count_g, int A, int num_chunks);

/*
 * The collectives. Pointer arrays hold R entries, entry r for virtual rank r:
 *   send[a], recv[a] (a < A): the actives' input and output buffers;
 *   scratch[a] (a < A):       >= plan.active_scratch_elems elements (may be NULL if 0);
 *   scratch[A+h]:             helper h, >= plan.helper_elems elements (NULL if 0).
 *   send/recv entries of helpers are ignored (may be NULL).
 * All device pointers; element-aligned; any further alignment is optional (16-byte
 * aligned buffers take the vectorized path).
 * Scratch is workspace: every scratch byte a call reads it wrote earlier in the same call,
 * and its contents after the call are unspecified (see RELAY_FLAG_KEEP_SCRATCH).
 * Aliasing: every buffer must be disjoint from every other except the in-place forms:
 *   allreduce      recv[a] == send[a]                          (D115998369)
 *   reduce-scatter recv[a] == send[a] + a*count elements       (D115998376)
 *   all-gather     send[a] == recv[a] + a*count elements       (D115998385)
 *   all-to-all     out-of-place only                           (D115998370)
 * scale multiplies the fp32 sum once before the cast: 1 for SUM, 1/A for AVG
 * (D115998376); int32 accepts only scale == 1 (integer AVG is undefined).
 * Arithmetic: fp32 and bf16 sum in fp32 in ascending source rank, multiply by scale
 * once, round to nearest-even into the payload type; int32 sums wrap modulo 2^32. The
 * one partial sum that crosses a link, the 4-active relay reduce-scatter's helper partial
 * (item 6), is summed over the A-1 non-owner sources in ascending rank; the owner then
 * adds its own value first and the partial second. For a bf16 payload the partial
 * crosses in fp32 unless RELAY_FLAG_PAYLOAD_PARTIAL asks for the payload type (see that
 * flag for the rounding each choice gives).
 * count == 0 returns RELAY_OK without a launch.
 */
relay_status_t relay_allreduce(void* const* send, void* const* recv, void* const* scratch,
                               size_t count, relay_dtype_t dtype, int A, int R, float scale,
                               const relay_opts_t* opts, cudaStream_t stream);
relay_status_t relay_reduce_scatter(void* const* send, void* const* recv, void* const* scratch,
                                    size_t recv_count, relay_dtype_t dtype, int A, int R,
                                    float scale, const relay_opts_t* opts, cudaStream_t stream);
relay_status_t relay_all_gather(void* const* send, void* const* recv, void* const* scratch,
                                size_t send_count, relay_dtype_t dtype, int A, int R,
                                const relay_opts_t* opts, cudaStream_t stream);
relay_status_t relay_all_to_all(void* const* send, void* const* recv, void* const* scratch,
                                size_t segment_count, relay_dtype_t dtype, int A, int R,
                                const relay_opts_t* opts, cudaStream_t stream);

/*
 * Fused multi-group call (D115998367, D115998376, D115998378): the R = num_groups*A
 * ranks form num_groups sparse groups of A consecutive ranks (group g = ranks g*A ..
 * g*A+A-1, D115998382). Every rank is active in its own group and a relay helper in
 * every other group; each group plans its own schedule from counts[g] (a group whose
 * chunk aligns down to zero takes the direct fallback while the others relay). The
 * groups run phase-synchronized: one launch carries every group's group-1 transfers,
 * the next every group's group-2 transfers, and so on, then every group's closing
 * reductions.
 *   send[r], recv[r]   (r < R): rank r's input and output for its own group;
 *   scratch[g*R + r]   rank r's scratch for group g: its active scratch when r is in
 *                      group g (plan.active_scratch_elems), its helper scratch otherwise
 *                      (plan.helper_elems); NULL where the size is 0.
 * Sizes, dtypes, in-place forms and scale are as for the single-group calls; scale is
 * ignored for all-gather and all-to-all. Every buffer must be disjoint from every other
 * except the in-place forms.
 */
relay_status_t relay_multi_group(relay_coll_t coll, int num_groups, const size_t* counts,
                                 void* const* send, void* const* recv, void* const* scratch,
                                 relay_dtype_t dtype, int A, float scale,
                                 const relay_opts_t* opts, cudaStream_t stream);

/* Link-byte accountant of a fused call: out[(p*R + src)*R + dst] = payload BYTES moved
 * from rank src to rank dst in phase p (the groups' serialized group p, summed over
 * groups). *num_phases receives the number of phases; cap >= num_phases*R*R. */
relay_status_t relay_multi_group_link_bytes(relay_coll_t coll, int num_groups,
                                            const size_t* counts, relay_dtype_t dtype, int A,
                                            const relay_opts_t* opts, uint64_t* out, size_t cap,
                                            int* num_phases);

/*
 * Flat packing of a caller's tensor list (D115998366: the distributed layer packs the
 * tensors into the active flat buffer and unpacks the result, one launch each).
 * relay_pack_flat copies tensors srcs[0..n-1] (counts[i] elements each) end to end
 * into `flat`; relay_unpack_flat copies them back out into dsts. One launch for up to
 * 384 non-empty tensors. `flat` must hold sum(counts) elements and overlap no tensor.
 */
relay_status_t relay_pack_flat(const void* const* srcs, const size_t* counts, int n, void* flat,
                               relay_dtype_t dtype, cudaStream_t stream);
relay_status_t relay_unpack_flat(const void* flat, void* const* dsts, const size_t* counts, int n,
                                 relay_dtype_t dtype, cudaStream_t stream);

/*
 * relay_copy -- copies `count` elements of `dtype` from `src` to `dst` with the library's
 * streaming kernel, asynchronously on `stream`. It is how callers stage a collective's
 * inputs into HBM and its results back out when those live in host memory. The page has
 * no counterpart: its buffers always sit in device memory.
 *   - Either pointer may be device memory, pinned or registered host memory, or (only
 *     where the device reports cudaDevAttrPageableMemoryAccess) ordinary pageable host
 *     memory. The SMs load and store across the host link themselves. On GB300 this
 *     reaches the link's rate whether or not the copy engines do.
 *   - max_ctas caps the CTAs of the launch. Each CTA then walks 16 KiB tiles. 0 means
 *     one CTA per tile, the fastest form for device-to-device copies. A copy over the host
 *     link reaches the link's rate with about one CTA per SM, which leaves the other CTA
 *     slots to kernels running at the same time on other streams.
 *   - Pointers must be element-aligned, and the two ranges must not overlap.
 *   - count == 0 returns RELAY_OK without a launch.
 *   - Errors: RELAY_ERR_INVALID_ARGUMENT (NULL, misaligned, overlapping, max_ctas < 0);
 *     RELAY_ERR_UNSUPPORTED (pageable host memory on a device that cannot address it);
 *     RELAY_ERR_CUDA (pointer query or launch failure).
 */
relay_status_t relay_copy(void* dst, const void* src, size_t count, relay_dtype_t dtype,
                          int max_ctas, cudaStream_t stream);

/*
 * relay_allreduce_noalloc -- an allreduce for callers that cannot allocate device
 * memory when they call it (an allocator or memory-pool hook that would recurse into
 * itself, a process that reserved all of HBM at start-up, a path that cannot take the
 * synchronisation an allocation may cause). The page has no counterpart to this entry
 * point.
 *
 * Arguments and results are those of relay_allreduce, without `scratch`: the helpers'
 * relay slots and the actives' receive staging come from one file-scope device array of
 * RELAY_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds until exit.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - Limit: A*round256(active_scratch_elems*esize) + H*round256(helper_elems*esize)
 *     bytes (relay_plan gives both sizes) must fit the array; larger calls return
 *     RELAY_ERR_INVALID_ARGUMENT with a message. For the 2-active relay that is about
 *     2*count*esize, i.e. up to 32 MiB per rank.
 *   - Set-up: the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before any
 *     stream capture.
 *   - Sharing: every call on a device uses the same array and leaves its contents
 *     there. Nothing in it needs clearing (each call writes every element before it
 *     reads it), but calls whose execution overlaps on the GPU (other streams, other
 *     host threads) race on it: order them.
 */
#define RELAY_NOALLOC_SCRATCH_BYTES (64u << 20)
relay_status_t relay_allreduce_noalloc(void* const* send, void* const* recv, size_t count,
                                       relay_dtype_t dtype, int A, int R, float scale,
                                       const relay_opts_t* opts, cudaStream_t stream);

/*
 * relay_device_status -- reads and clears the device's fault word. Passes whose sources
 * sit off the 16-byte grid stage each tile's source bytes in shared memory with a bulk
 * copy and wait for it on an mbarrier (the schedule's strided pack/unpack, item 7). That
 * wait is bounded (200 ms of the global timer); if it ever runs out, the kernel records a
 * fault, leaves that tile unwritten and returns instead of hanging. Call this after
 * synchronizing the streams that ran collectives: RELAY_ERR_CUDA if a wait gave up since
 * the last call (or a CUDA call failed), RELAY_OK otherwise. Synchronous.
 */
relay_status_t relay_device_status(void);

/*
 * relay_test_staged_wait -- a test of that bounded wait: one staged copy of `count`
 * elements (at most one 16 KiB tile) from `src` to `dst` (device memory, dst 16-byte
 * aligned) whose barrier expects `extra_bytes` more than its copy brings. With
 * extra_bytes > 0 the wait runs out, the copy's destination is left unwritten, and the
 * next relay_device_status() reports RELAY_ERR_CUDA; the context stays usable. With 0 it
 * is an ordinary copy. The page has no counterpart.
 */
relay_status_t relay_test_staged_wait(void* dst, const void* src, size_t count,
                                      relay_dtype_t dtype, int extra_bytes, cudaStream_t stream);

/* Human-readable text of the last error this thread's calls produced. */
const char* relay_last_error(void);
/* How the calling thread's last collective call was launched: "chained: G groups, P
 * pieces, D dropped" (D: scratch sources whose dead lines the launch drops from L2),
 * "cooperative" or "passes" (see the launch policy above); "dry run" for a
 * RELAY_FLAG_DRY_RUN call that would not run chained, "none" before the first call. */
const char* relay_last_launch(void);
int relay_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RELAY_H */
