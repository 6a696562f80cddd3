/*
 * bsa.h -- C ABI of libbsa: dynamic block-sparse attention (BSA) forward for
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes ("Decoupling Logical Masks from GPU Execution for
 * Dynamic Block-Sparse Attention" (Tessera), abstract): attention computed
 * only over the (query-block, key-block) pairs that a logical block mask
 * selects, with every selected interaction preserved.  For batch b, query head
 * h (KV head h / g) and query row i, with J the keys whose block the mask
 * selects for i's block:
 *     O[i]   = sum_{j in J} exp(s_j - m) V[j] / sum_{j in J} exp(s_j - m),
 *     s_j    = scale * <Q[i], K[j]>,  scale = 1/sqrt(d) unless overridden,
 *     LSE[i] = m + ln(sum_{j in J} exp(s_j - m))  (natural log),
 * and O[i] = 0, LSE[i] = -inf when J is empty.
 *
 * Two stages, both stream-ordered and free of host synchronisation:
 *   bsa_plan_create  -- the physical mapping and task organisation layers of
 *                       the Tessera abstract: logical blocks are retained,
 *                       combined or subdivided into 128-row physical tiles,
 *                       and each (batch, head, 128-row q-tile) gets a CSR list
 *                       of the K/V tiles it needs, plus a schedule (rows that
 *                       share a K/V head together, heaviest group first,
 *                       longest row first) and (for GQA) a per-group union table
 *                       ("CompactAttention", summary: Q-block union plus
 *                       intra-group union).
 *   bsa_forward      -- runs attention over exactly the tiles of a plan.
 * Variants: bsa_plan_create_affine (rows given by affine descriptors instead
 * of mask bytes), BSA_PLAN_REMAP (per-plane q-unit regrouping),
 * bsa_forward_ex (paged K/V, key lengths, intra-block causality),
 * bsa_forward_stage (the forward's passes one by one), bsa_attention_host
 * (from host buffers with overlapped copies), bsa_attention_static (no
 * allocation at all).
 *
 * Conventions
 *   - Every pointer argument named "device" is a CUDA device pointer owned by
 *     the caller; the library never allocates, frees or retains device
 *     memory.  The only host allocation is the small bsa_plan handle
 *     (bsa_attention_host also creates two streams and a few events for the
 *     duration of the call).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls enqueue work on it and return without synchronising,
 *     except bsa_sync_status and bsa_plan_check, which synchronise it.
 *   - Layouts are row-major and contiguous: mask u8 [B][H][NQB][NKB];
 *     Q and O bf16 [B][Hq][Nq][d]; K and V bf16 [B][Hkv][Nk][d];
 *     LSE fp32 [B][Hq][Nq].  Nq = NQB*bq, Nk = NKB*bk, Hkv = Hq/gqa_group.
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned as a negative bsa_status.  Errors the kernels detect
 *     (watchdog expiry, an out-of-range plan entry) are recorded in a status
 *     word in the plan workspace and reported by bsa_sync_status.
 */
#ifndef BSA_H_
#define BSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BSA_VERSION 1

typedef enum bsa_status {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size or shape */
  BSA_ERR_UNSUPPORTED = -2,   /* block size, head dim or size outside the supported set */
  BSA_ERR_ARCH = -3,          /* current device is not compute capability 10.3 */
  BSA_ERR_CUDA = -4,          /* a CUDA runtime/driver call failed */
  BSA_ERR_WORKSPACE = -5,     /* workspace too small */
  BSA_ERR_TIMEOUT = -6,       /* a kernel wait exceeded its limit (device watchdog) */
  BSA_ERR_PLAN_MISMATCH = -7  /* plan inconsistent with itself or with the inputs */
} bsa_status;

/* Opaque host handle of a plan.  It holds sizes and a pointer into the
 * caller's workspace; it stays valid until bsa_plan_destroy or until the
 * workspace is freed, whichever comes first. */
typedef struct bsa_plan bsa_plan;

/* Plan geometry and the placement of every plan array inside the workspace
 * (byte offsets from the workspace base, each 256-byte aligned).  Pure host
 * arithmetic on sizes. */
typedef struct bsa_plan_layout {
  int32_t B, H, Hkv, NQB, NKB, bq, bk, gqa_group;
  /* mapping: qu = rows per q-unit, rq = q-units per 128-row q-tile,
   * sq = q-units per logical q-block; ku, rk, sk likewise for keys */
  int32_t qu, rq, sq, ku, rk, sk;
  int32_t NQT;          /* q-tiles per head  = Nq / (qu * rq): 128-row tiles, or 64 with BSA_PLAN_Q64 */
  int32_t NKU;          /* k-units per head  = Nk / ku */
  int32_t rows;         /* plan rows R = B*H*NQT */
  int32_t urows;        /* union rows = B*Hkv*NQT when gqa_group > 1, else 0 */
  int32_t max_row_slots;/* ceil(NKU / rk): most slots one row can need */
  int32_t groups;       /* K/V-head groups of the schedule = B*Hkv */
  int64_t slot_capacity;  /* rows * max_row_slots */
  int64_t union_capacity; /* urows * NKU */
  uint64_t off_row_ptr;   /* int32 [rows+1]   CSR row pointer into slots */
  uint64_t off_slot_ku;   /* int32 [slot_capacity*rk] k-unit of each slot position, -1 = padding */
  uint64_t off_slot_mask; /* uint32 [slot_capacity] bit i*rk+j: q-unit i attends slot position j */
  uint64_t off_urow_ptr;  /* int32 [urows+1]  GQA union CSR row pointer */
  uint64_t off_ukb;       /* int32 [union_capacity] union k-units, ascending */
  uint64_t off_order;     /* int32 [rows]     schedule: K/V-head groups heaviest first, rows longest first */
  uint64_t off_totals;    /* int64 [4]: slots, selected logical blocks, union entries, 0 */
  uint64_t off_control;   /* int32 [16]: [0] work counter, [1] status, [2] status detail */
  uint64_t off_scratch;   /* plan-construction scratch */
  uint64_t workspace_bytes; /* total bytes the caller must provide */
  uint64_t off_sigma;     /* int32 [B*H] q-unit grouping stride of each (b, h) plane:
                           * q-tile t = run*s + r of a plane with stride s holds
                           * q-units run*s*rq + r + i*s, i < rq (s = 1: t*rq + i) */
} bsa_plan_layout;

/* Plan flags */
#define BSA_PLAN_NO_UNION 0x1   /* skip the GQA union table even when gqa_group > 1 */
/* Choose each (b, h) plane's q-unit grouping stride among 1, 2, 4, 8, 16
 * (those dividing the plane's q-tiles) by the slots its tiles need, fewest
 * first, ties to the smaller stride -- the physical mapping of combined
 * blocks ("Decoupling Logical Masks from GPU Execution for Dynamic
 * Block-Sparse Attention" (Tessera), abstract: logical blocks are combined
 * into physical tiles).  Only when tiles combine several q-units (bq < 128),
 * gqa_group == 1 and the plane has at most 8192 q-tiles; otherwise (and
 * without the flag) every stride is 1.  One extra kernel launch. */
#define BSA_PLAN_REMAP 0x2
/* 64-row q-tiles, for query blocks of at most 64 rows (bq in {32, 64};
 * BSA_ERR_UNSUPPORTED otherwise): a 64-row query block is a q-tile of its own
 * and two 32-row blocks share one, instead of two (four) blocks sharing a
 * 128-row tile and the union of their selections -- a second physical mapping
 * of small blocks ("Decoupling Logical Masks from GPU Execution for Dynamic
 * Block-Sparse Attention" (Tessera), abstract: logical blocks are combined
 * into physical tiles).  Nq must then be a multiple of 64.  bsa_forward runs
 * such plans with a kernel that puts the 128 keys of a slot on the MMA's M
 * dimension and the tile's 64 queries on N (contiguous K/V, no element mask:
 * bsa_forward_ex returns BSA_ERR_UNSUPPORTED for pages, key lengths or
 * causality on these plans). */
#define BSA_PLAN_Q64 0x4

/*
 * bsa_plan_select_flags -- plan flags for a problem shape, chosen from a
 * table of measured forward times compiled into the library (the
 * profile-guided selection of a runtime configuration from offline
 * profiles, "Decoupling Logical Masks from GPU Execution for Dynamic
 * Block-Sparse Attention" (Tessera), abstract).  The table gives, per
 * (bq, bk, d), the physical q-tile height (BSA_PLAN_Q64 or not) that was
 * faster over a sweep of mask densities; BSA_PLAN_REMAP is added wherever
 * tiles combine several q-units and gqa_group == 1 (its stride is chosen on
 * the device from exact slot counts).  Depends on shapes only, never on the
 * mask, so it needs no device access.  Nq = NQB * bq.  Returns the flags,
 * or a negative bsa_status for shapes bsa_plan_layout_query rejects.
 */
int bsa_plan_select_flags(int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group, int d);

/*
 * bsa_plan_layout_query -- sizes and workspace layout for a plan.
 * Arguments: mask geometry B, H (query heads), NQB, NKB; logical block sizes
 * bq, bk in {32, 64, 128, 256}; gqa_group g >= 1 dividing H; flags as for
 * bsa_plan_create.  Requires Nq = NQB*bq to be a multiple of 128.
 * Writes *out; returns BSA_ERR_INVALID_ARG / BSA_ERR_UNSUPPORTED otherwise.
 * Touches no device.
 */
bsa_status bsa_plan_layout_query(int B, int H, int NQB, int NKB, int bq, int bk,
                                 int gqa_group, int flags, bsa_plan_layout* out);

/*
 * bsa_plan_workspace_bytes -- device workspace bytes a plan of this geometry
 * needs (bsa_plan_layout_query(..., flags = 0, ...).workspace_bytes: plan
 * arrays, plan-construction scratch and the forward's scratch).  The same
 * for BSA_PLAN_REMAP and BSA_PLAN_NO_UNION plans (an upper bound for the
 * latter); plans with 64-row q-tiles (BSA_PLAN_Q64) have twice the rows:
 * query bsa_plan_layout_query with that flag.  Returns 0 for arguments
 * bsa_plan_layout_query rejects.  Touches no device.
 */
size_t bsa_plan_workspace_bytes(int B, int H, int NQB, int NKB, int bq, int bk, int gqa_group);

/*
 * bsa_plan_create -- build the plan of one logical mask on the GPU: the
 * physical mapping layer (logical blocks retained, combined or subdivided
 * into physical tiles) and the task organisation layer (tiles grouped per
 * q-tile and scheduled) of "Decoupling Logical Masks from GPU Execution for
 * Dynamic Block-Sparse Attention" (Tessera), abstract, plus the per-group
 * union table of "CompactAttention: Accelerating Chunked Prefill with
 * Block-Union KV Selection", summary.
 * mask: device, u8 [B][H][NQB][NKB]; any non-zero byte selects the block.
 * workspace: device, >= layout.workspace_bytes bytes, 256-byte aligned, owned
 * by the caller and reused by every bsa_forward on this plan (it also holds
 * the work counter and status word those launches use, so two launches on
 * one plan must not overlap in time).
 * Enqueues three kernels on `stream` (no host sync): per-row counts,
 * prefix sums, then compaction + schedule.  *out receives a new handle.
 * Errors: BSA_ERR_INVALID_ARG (null/misaligned pointers, bad shapes),
 * BSA_ERR_UNSUPPORTED, BSA_ERR_WORKSPACE, BSA_ERR_ARCH, BSA_ERR_CUDA.
 */
bsa_status bsa_plan_create(const uint8_t* mask, int B, int H, int NQB, int NKB, int bq,
                           int bk, int gqa_group, void* workspace, size_t workspace_bytes,
                           int flags, void* stream, bsa_plan** out);

/*
 * bsa_plan_create_affine -- bsa_plan_create for a logical mask given (wholly
 * or partly) by affine row descriptors ("SPLAT: A framework for optimised GPU
 * code-generation for SParse reguLar ATtention", abstract: the
 * affine-compressed-sparse-row format captures the regular geometry of
 * sparse attention patterns, analysed just in time).  Each query head h owns
 * segments seg_ptr[h] .. seg_ptr[h+1]-1 of `segments`; segment
 * {a, b, stride, count} selects, for logical query block qb, the key blocks
 *     a*qb + b + stride*t,  t = 0 .. count-1,  kept when in [0, NKB)
 * (a = 1: relative to the query block -- sliding windows, strided and
 * dilated patterns; a = 0: fixed key blocks -- global columns; stride may be
 * negative, stride 0 repeats one block).  A head with segments selects their
 * union, the same for every batch entry, generated by the plan kernels
 * without reading mask bytes; a head without segments takes its rows of
 * `mask` (irregular heads, e.g. random blocks).
 * mask: device u8 [B][H][NQB][NKB] (only the rows of heads without segments
 *   are read), or NULL when every head has segments (a head without
 *   segments then selects nothing).
 * segments: device int32 [nseg][4], 16-byte aligned (may be NULL if nseg = 0).
 * seg_ptr: device int32 [H+1], non-decreasing; entries are clamped to
 *   [0, nseg] on the device.  Both caller-owned; they are read by the plan
 *   kernels of this call only.
 * The plan and its arrays are exactly those bsa_plan_create builds from the
 * expanded mask.  Other arguments and errors as bsa_plan_create.
 */
bsa_status bsa_plan_create_affine(const uint8_t* mask, const int32_t* segments,
                                  const int32_t* seg_ptr, int nseg, int B, int H, int NQB,
                                  int NKB, int bq, int bk, int gqa_group, void* workspace,
                                  size_t workspace_bytes, int flags, void* stream,
                                  bsa_plan** out);

/* Copy the layout of an existing plan into *out. */
bsa_status bsa_plan_get_layout(const bsa_plan* plan, bsa_plan_layout* out);

/* Device base pointer of the plan's workspace (NULL for a NULL plan). */
void* bsa_plan_workspace(const bsa_plan* plan);

/* Free the host handle (not the workspace).  NULL is a no-op. */
void bsa_plan_destroy(bsa_plan* plan);

/*
 * Host copies of a plan's arrays for bsa_plan_export.  Each pointer is a
 * caller-owned HOST buffer of the given capacity in elements, or NULL to
 * skip that array.  Lengths needed (element counts, see bsa_plan_layout):
 *   row_ptr rows+1, slot_ku totals[0]*rk, slot_mask totals[0],
 *   urow_ptr urows+1 (1 when there is no union table), ukb totals[2],
 *   order rows, plane_sigma B*H.
 */
typedef struct bsa_plan_arrays {
  int32_t* row_ptr;     size_t row_ptr_cap;
  int32_t* slot_ku;     size_t slot_ku_cap;
  uint32_t* slot_mask;  size_t slot_mask_cap;
  int32_t* urow_ptr;    size_t urow_ptr_cap;
  int32_t* ukb;         size_t ukb_cap;
  int32_t* order;       size_t order_cap;
  int32_t* plane_sigma; size_t plane_sigma_cap;
  int64_t totals[4];    /* written: slots, selected logical blocks, union entries, 0 */
} bsa_plan_arrays;

/*
 * bsa_plan_export -- synchronise `stream` (the plan's kernels must have been
 * enqueued on it or before it), then copy the plan's totals and every
 * requested array into the caller's host buffers.  For tests, inspection
 * and handing a plan to other tools; the forward reads the plan on the
 * device and never needs this.  Errors: BSA_ERR_INVALID_ARG (NULL/foreign
 * plan or `out`), BSA_ERR_WORKSPACE (a buffer smaller than its array; the
 * totals are written first, so the caller can size the buffers from them),
 * BSA_ERR_CUDA.
 */
bsa_status bsa_plan_export(const bsa_plan* plan, void* stream, bsa_plan_arrays* out);

/*
 * bsa_forward -- block-sparse attention forward over a plan: attention over
 * exactly the (query-block, key-block) pairs the plan's mask selects, every
 * selected interaction preserved ("Decoupling Logical Masks from GPU
 * Execution for Dynamic Block-Sparse Attention" (Tessera), abstract), with
 * the online-softmax fusion of FlashAttention-style kernels ("Sol-Attn"
 * summary) and the TMA + warp-specialised tile-skipping structure the
 * "Veda" summary describes for Hopper, here on tcgen05 tensor cores.
 * Q: device bf16 [B][Hq][Nq][d]; K, V: device bf16 [B][Hkv][Nk][d];
 * O: device bf16 [B][Hq][Nq][d] (written); LSE: device fp32 [B][Hq][Nq]
 * (written; natural log, -inf for rows with no selected key).  All 16-byte
 * aligned (an O that is also 32-byte aligned is written with 32-byte stores,
 * a little faster; the values are the same); Q/K/V/O must not alias.
 * d in {64, 128}.  scale <= 0 selects 1/sqrt(d).  Nq, Nk, Hkv and the block
 * sizes come from the plan.
 * Enqueues one memset of the plan's control words and four kernels on
 * `stream`: the key-norm and row-bound passes, the forward pass over every
 * plan row, and an exact second pass over the rows the first one queued (it
 * exits at once when none was).  Errors: BSA_ERR_INVALID_ARG,
 * BSA_ERR_UNSUPPORTED, BSA_ERR_PLAN_MISMATCH (NULL/foreign plan),
 * BSA_ERR_ARCH, BSA_ERR_CUDA.  Same as bsa_forward_ex with no pages, no key
 * lengths and no flags.
 */
bsa_status bsa_forward(const bsa_plan* plan, const void* Q, const void* K, const void* V,
                       void* O, float* LSE, int d, float scale, void* stream);

/*
 * Paged K/V for bsa_forward_ex ("CompactAttention: Accelerating Chunked
 * Prefill with Block-Union KV Selection", summary: zero-copy paged attention
 * execution; the PagedAttention entry of the related-papers list on the
 * "TiledAttention" page: on-demand page allocation of the KV cache).
 * The K and V pools are device bf16 [num_pages][Hkv][page_size][d]; key
 * position j of sequence b lives in physical page
 * block_table[b * max_pages + j / page_size], row j % page_size.
 * page_size must be a positive multiple of the plan's K unit min(bk, 128)
 * (so a unit never straddles two pages); max_pages * page_size >= Nk.
 */
typedef struct bsa_kv_pages {
  const int32_t* block_table;  /* device int32 [B][max_pages], caller-owned */
  int max_pages;               /* logical pages per sequence */
  int page_size;               /* keys per page */
  int num_pages;               /* pages in each pool */
} bsa_kv_pages;

/* Intra-block causal masking: key position j is visible to query position i
 * only when j <= i + (Nk - Nq) (queries are the last Nq positions). */
#define BSA_FWD_CAUSAL 0x1
/* Apply every row's softmax weights as two bf16 terms, hi = bf16(p) and
 * lo = bf16(p - hi), with a second P V product for lo (weights exact to about
 * 2^-16 instead of 2^-8).  Without the flag this is done only for rows whose
 * selected K/V units hold a V element of magnitude above 8, where bf16
 * weights would move O by more than a few thousandths; the tensor work of
 * such rows grows by half. */
#define BSA_FWD_SPLIT_P 0x2

/*
 * bsa_forward_ex -- bsa_forward with paged K/V, per-sequence key lengths and
 * intra-block causal masking.  Within every block the mask selects, element
 * (i, j) is dropped when BSA_FWD_CAUSAL is set and j > i + Nk - Nq, or when
 * kv_lens is given and j >= kv_lens[b]; a row left with no key gets O = 0
 * and LSE = -inf, as a row with no selected block does.
 * pages: NULL for contiguous K, V [B][Hkv][Nk][d]; else K and V are the
 *   pools described above.
 * kv_lens: NULL, or device int32 [B] (each in [0, Nk]), caller-owned.
 * flags: 0 or an OR of BSA_FWD_CAUSAL and BSA_FWD_SPLIT_P.
 * Other arguments and errors as bsa_forward; additionally
 * BSA_ERR_UNSUPPORTED for a page size that is not a multiple of the K unit
 * and BSA_ERR_INVALID_ARG for a NULL block table, non-positive sizes or
 * unknown flags.  Keys at or past kv_lens[b] are masked out, so the entry
 * of a page holding none below it may be anything (-1 for an unallocated
 * page; the kernel then reads page 0 in its place and discards it); an entry
 * outside [0, num_pages) for a page that holds a key below kv_lens[b] (every
 * key when kv_lens is NULL) is skipped and reported by bsa_sync_status as
 * BSA_ERR_PLAN_MISMATCH.
 */
bsa_status bsa_forward_ex(const bsa_plan* plan, const void* Q, const void* K, const void* V,
                          const bsa_kv_pages* pages, const int32_t* kv_lens, int flags,
                          void* O, float* LSE, int d, float scale, void* stream);

/*
 * bsa_forward_stage -- bsa_forward_ex in stages, so that a caller can time
 * or interleave them: BSA_STAGE_PREPARE (reset the pass counters, the
 * key-norm pass and the row-bound pass), BSA_STAGE_BOUNDED (the bounded
 * pass over every plan row), BSA_STAGE_EXACT (the exact pass over the rows
 * the bounded pass queued).  `stages` is a non-empty OR of them; the stages
 * of one forward must run in that order, with the same arguments, and no
 * other forward on the same plan in between (BSA_STAGE_KNORM may run on
 * another stream, see below; the caller orders the streams).  Calling all
 * three at once (BSA_STAGE_ALL) is bsa_forward_ex.  Errors as bsa_forward_ex,
 * plus BSA_ERR_INVALID_ARG for an empty or unknown stage set.
 */
#define BSA_STAGE_PREPARE 0x1
#define BSA_STAGE_BOUNDED 0x2
#define BSA_STAGE_EXACT 0x4
#define BSA_STAGE_ALL 0x7
/* The two halves of BSA_STAGE_PREPARE: the key-norm pass (reads only K, so
 * it may be enqueued on another stream before or while the plan is built,
 * e.g. beside bsa_plan_create, as long as it completes before the row-bound
 * pass starts) and the row-bound pass (needs the plan and the key norms). */
#define BSA_STAGE_KNORM 0x8
#define BSA_STAGE_ROWBOUND 0x10
bsa_status bsa_forward_stage(const bsa_plan* plan, const void* Q, const void* K, const void* V,
                             const bsa_kv_pages* pages, const int32_t* kv_lens, int flags,
                             void* O, float* LSE, int d, float scale, int stages, void* stream);

/*
 * bsa_sync_status -- synchronise `stream`, then report the status word the
 * last bsa_forward on this plan left: BSA_OK, BSA_ERR_TIMEOUT (a wait in the
 * kernel ran past the watchdog limit; the kernel stopped cleanly) or
 * BSA_ERR_PLAN_MISMATCH (an out-of-range plan entry was skipped).  *detail
 * (may be NULL) receives (block << 8) | wait-site of the first failure.
 */
bsa_status bsa_sync_status(const bsa_plan* plan, void* stream, int32_t* detail);

/*
 * bsa_plan_check -- synchronise `stream`, copy the plan arrays to the host
 * and verify them (row pointers monotone and within capacity, k-units in
 * range and ascending, padding only at the end of a row, schedule a
 * permutation).  Returns BSA_OK or BSA_ERR_PLAN_MISMATCH.  For tests and
 * debugging; allocates host memory.
 */
bsa_status bsa_plan_check(const bsa_plan* plan, void* stream);

/*
 * bsa_watchdog_selftest -- launch a one-block kernel that waits on a barrier
 * nothing ever completes, with a limit of `limit_us` microseconds, using the
 * same bounded wait as the forward kernel; synchronise `stream` and return
 * the status the kernel recorded (BSA_ERR_TIMEOUT when the watchdog works).
 * `status` is device int32[4] scratch owned by the caller.
 */
bsa_status bsa_watchdog_selftest(int32_t* status, int limit_us, void* stream);

/*
 * bsa_attention_static -- plan + forward in one call, allocating nothing.
 * The method's pages have no counterpart of this call; it exists for callers
 * that cannot allocate device memory (for example an inference-engine plugin
 * whose execute step must not call cudaMalloc, or a component that only ever
 * receives device pointers).  Instead of a caller workspace it uses a scratch
 * area compiled into the library: a file-scope __device__ array of
 * BSA_STATIC_WORKSPACE_BYTES that every GPU loading the library holds until
 * the process exits.
 * Arguments: as bsa_plan_create (mask, geometry, block sizes, gqa_group)
 * followed by bsa_forward's (Q, K, V, O, LSE, d, scale) and the stream; the
 * GQA union table is not built.  All pointers are device pointers owned by
 * the caller.
 * Limits and behaviour:
 *   - Returns BSA_ERR_WORKSPACE, before anything is enqueued, when the
 *     problem's plan needs more than BSA_STATIC_WORKSPACE_BYTES.
 *   - Calls no cudaMalloc/cudaFree or other allocating routine.  The first
 *     call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  With lazy module loading (the CUDA default)
 *     that first call is also where the driver loads the library's device
 *     code and commits the scratch array on the device, so a caller that
 *     must not allocate during execution makes one call (any small problem)
 *     at set-up time.  The looked-up address is kept for the life of the
 *     process: after cudaDeviceReset, or anything else that destroys the
 *     device's primary context, this call is not supported.
 *   - Every call on a device shares the one scratch area and leaves its
 *     contents behind; the call clears what must start at zero (work counter
 *     and status words) itself.  Calls whose GPU work overlaps in time (for
 *     example on two streams) race on the scratch area and must be avoided.
 *   - Enqueues a memset, the three plan kernels and the forward passes on
 *     `stream` without synchronising.  Errors detected by the kernels
 *     (watchdog expiry, out-of-range plan data) are recorded in the scratch
 *     area, not returned by this call (it returns host-detected argument
 *     errors and launch failures only); bsa_attention_static_status reads
 *     them back.
 */
#define BSA_STATIC_WORKSPACE_BYTES (16u << 20)
bsa_status bsa_attention_static(const uint8_t* mask, int B, int H, int NQB, int NKB, int bq,
                                int bk, int gqa_group, const void* Q, const void* K, const void* V,
                                void* O, float* LSE, int d, float scale, void* stream);

/*
 * bsa_attention_static_status -- synchronise `stream` and report the status
 * the kernels of the last bsa_attention_static call on the current device
 * left in the scratch area, with the same codes and *detail encoding as
 * bsa_sync_status (BSA_OK when no call has run on the device yet).  The
 * status words are read with one cudaMemcpyAsync on `stream` into a local
 * host array.  Meaningful only while no other bsa_attention_static call on
 * the device is in flight.
 */
bsa_status bsa_attention_static_status(void* stream, int32_t* detail);

/*
 * bsa_attention_host -- plan + forward from HOST buffers, with the transfers
 * overlapped with the computation.  The pages describe the attention and its
 * GPU execution, not host transfers; this is plumbing around the same plan
 * and forward (each row's result is bit-identical to bsa_plan_create +
 * bsa_forward on device copies of the same inputs).
 * The B*Hkv (batch, K/V head) units are cut into `chunks` contiguous chunks
 * (clamped to [1, B*Hkv]); chunk i is copied in on one stream, planned and
 * run on `stream`, and copied out on another, so that the copy-in of chunk
 * i+1 and the copy-out of chunk i-1 overlap the computation of chunk i.
 * mask, Q, K, V: host, layouts as for bsa_plan_create / bsa_forward (pinned
 * memory lets the copies run asynchronously; pageable memory works but
 * serialises them).  O, LSE: host outputs, same layouts.
 * buffer: device scratch of at least bsa_attention_host_buffer_bytes(...)
 * bytes, 256-byte aligned, owned by the caller (two chunk slots: inputs,
 * outputs, plan workspace; and one status word per chunk).
 * Plans are built without the GQA union table (the forward does not read
 * it) and without regrouping.
 * Synchronous: returns once O and LSE are in host memory (it synchronises
 * `stream`).  Errors: BSA_ERR_INVALID_ARG, BSA_ERR_UNSUPPORTED,
 * BSA_ERR_WORKSPACE (buffer too small), BSA_ERR_ARCH, BSA_ERR_CUDA, and the
 * first device status a chunk's forward recorded (BSA_ERR_TIMEOUT,
 * BSA_ERR_PLAN_MISMATCH).
 */
bsa_status bsa_attention_host_buffer_bytes(int B, int H, int NQB, int NKB, int bq, int bk,
                                           int gqa_group, int d, int chunks, size_t* bytes);
bsa_status bsa_attention_host(const uint8_t* mask, int B, int H, int NQB, int NKB, int bq, int bk,
                              int gqa_group, const void* Q, const void* K, const void* V, void* O,
                              float* LSE, int d, float scale, int chunks, void* buffer,
                              size_t buffer_bytes, void* stream);

/* Human-readable name of a status code (static string). */
const char* bsa_status_string(int status);

/* BSA_VERSION of the compiled library. */
int bsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSA_H_ */
