/*
 * oracle.h -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU statement of what the sharded relay collectives compute and of
 * the relay planner's geometry and link-byte cost model.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code, header,
 * table or helper with the CUDA library in pack_virtual_rank_gb300/, and the library
 * never calls it.
 *
 * Parity unpinned (readings the page does not fix; the tests hold them to the stated
 * reading only): the crossover values the page gives no figure for (A=2 allreduce full
 * exchange, A=2 all-gather and all-to-all, A=4 all-to-all), the A=2 chunk-to-helper
 * mapping and direct-region placement, the A=4 owner-slice alignment, and the value of
 * orc_passthrough_helper_size when the aligned chunk is zero.  Everything else here is
 * pinned by tests/test_oracle_pins.py.
 *
 * Citations name the page "Link-balance the sharded relay schedules (up to 3.2x vs
 * NCCL)" (torchrec pull request #4570).  "Sk" is item k of that page's summary;
 * "cost model" is the paragraph before item 1; "Dnnnnnnnnn" is the commit of the
 * page's commit stack with that Differential Revision number.
 */
#ifndef RELAY_ORACLE_H
#define RELAY_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* payload types (same numbering as the public ABI, restated here on purpose) */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_I32 = 2 };
/* collectives */
enum { ORC_AR = 0, ORC_RS = 1, ORC_AG = 2, ORC_A2A = 3 };
/* schedule kinds */
enum { ORC_KIND_RELAY = 0, ORC_KIND_ZERO_CHUNK = 1, ORC_KIND_DIRECT = 2, ORC_KIND_LEGACY = 3 };
/* forced schedule requests */
enum { ORC_FORCE_AUTO = 0, ORC_FORCE_RELAY = 1, ORC_FORCE_DIRECT = 2, ORC_FORCE_LEGACY = 3 };

/* ---- bfloat16 ---------------------------------------------------------- */
uint16_t orc_bf16_rne(float f);
float orc_bf16_to_f32(uint16_t h);
void orc_bf16_rne_array(const float* in, uint16_t* out, int64_t n);

/* ---- collective semantics ---------------------------------------------- */
/* Any of ref64 / ref32 / refq may be NULL.  Windows are [i0, i1) of one output. */
void orc_allreduce(int dtype, int A, const void* const* x, int64_t i0, int64_t i1,
                   float scale, double* ref64, float* ref32, void* refq);
void orc_reduce_scatter(int dtype, int A, const void* const* x, int64_t m, int owner,
                        int64_t i0, int64_t i1, float scale, int64_t helper_span,
                        double* ref64, float* ref32, void* refq);
void orc_reduce_scatter_wide(int dtype, int A, const void* const* x, int64_t m, int owner,
                             int64_t i0, int64_t i1, float scale, int64_t helper_span,
                             double* ref64, float* ref32, void* refq);
void orc_all_gather(int esize, int A, const void* const* x, int64_t S, void* out);
void orc_all_to_all(int esize, int A, const void* const* x, int64_t seg, int dst, void* out);

/* ---- planner restatement ----------------------------------------------- */
enum {
  ORC_G_COLL = 0, ORC_G_A, ORC_G_R, ORC_G_H, ORC_G_ESIZE, ORC_G_COUNT, ORC_G_KIND,
  ORC_G_GROUPS, ORC_G_CHUNK, ORC_G_DIRA, ORC_G_DIRA_OFF, ORC_G_DIRB, ORC_G_PD,
  ORC_G_D1, ORC_G_D2, ORC_G_OWNER_SLICE, ORC_G_OWNER_LAST, ORC_G_NFIELDS
};
int64_t orc_align_down(int64_t x);
int orc_plan(int coll, int A, int R, int64_t count, int esize, int permille, int force,
             int64_t* g /* ORC_G_NFIELDS */);
/* table[(grp * R + src) * R + dst] in ELEMENTS; returns the number of groups or -1 */
int orc_link_elems(const int64_t* g, uint64_t* table, int64_t cap);
uint64_t orc_cost_elems(const int64_t* g);

/* ---- helper-buffer contracts ------------------------------------------- */
int64_t orc_passthrough_helper_size(int64_t count_g, int A, int num_chunks);
int64_t orc_relay_helper_contract(int coll, int A, int R, int64_t count);

#ifdef __cplusplus
}
#endif
#endif
