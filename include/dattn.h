/*
 * dattn.h - C ABI of libdattn, split-KV decode attention for GB300 (sm_103a).
 *
 * One or a few query rows per request attend over a long K/V history held in
 * a contiguous or paged cache, with grouped-query (GQA) heads.  The K/V
 * sequence axis is cut into chunks; each chunk produces an exact partial
 * softmax state (m, l, u) and an LSE merge folds the states into the global
 * softmax ("M4.5 Decode Attention Kernels, Mask Programs, and Backend
 * Boundaries", §0x01-§0x03).  Retention mask programs ("M5.4 Long-Context KV
 * Policies", §0x04-§0x06) and quantized K/V formats ("M8.6 Live-Data
 * Quantization", §0x05-§0x06) run through the same kernels.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  The library never allocates
 *    device memory; a plan owns only host memory.  Pointers marked "device"
 *    must be device (or managed) memory, "host" ones host memory.
 *  - Errors: every call returns a dattn_status.  Nothing aborts, nothing
 *    throws across the ABI and nothing falls back to another path.  All
 *    validation runs before any launch or any write to a cache
 *    (M4.5 §0x07A semantic pre-checks, §0x08C append transaction).
 *    dattn_last_error() returns a text with every failed check of the last
 *    failing call on the calling thread (the rejection vector of M4.5 §0x07B).
 *  - Streams: "stream" is a cudaStream_t passed as void*.  Device work is
 *    enqueued on it and the library never synchronises the device, except in
 *    dattn_device_status / dattn_step_host_status, which read back one word,
 *    and dattn_step_host, which returns its results in host memory.
 *  - Numbers: scores, maxima, sums and partial states are fp32; O is bf16
 *    rounded to nearest even; LSE is fp32 in natural-log units.  A query row
 *    with no visible key gets O = 0 and LSE = -inf (M4.5 §0x02C).
 */
#ifndef DATTN_H
#define DATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DATTN_OK = 0,
  DATTN_EINVAL = 1,          /* malformed call: a semantic pre-check failed             */
  DATTN_EUNSUPPORTED = 2,    /* well formed, but outside what this library implements   */
  DATTN_EWORKSPACE = 3,      /* workspace NULL, too small or not 256-byte aligned        */
  DATTN_ESTALE_PLAN = 4,     /* run-time problem differs from the plan's key (§0x07F)    */
  DATTN_ECUDA = 5,           /* a CUDA runtime call or launch failed                     */
  DATTN_EDEVICE_CHECK = 6    /* a device-side bounds check fired (dattn_device_status)   */
} dattn_status;

/* K/V storage (M4.5 §0x04B, §0x04D; M5.4 §0x04C).
 *  DATTN_KV_CONTIG_NHD: K, V bf16 [B_cache, T_cap, H_kv, d]; request b uses
 *      cache row cache_batch_idx[b] (b when the pointer is NULL).
 *  DATTN_KV_PAGED_HND:  pools [num_pages, H_kv, P, d] (format-dependent element,
 *      see dattn_format); request b's logical block j = t / P lives in page
 *      page_indices[page_indptr[b] + j] at page row t mod P (CSR page list).
 *  DATTN_KV_PACKED_ROWS: the ragged packed view of retained rows (M5.4 §0x04C):
 *      K, V bf16 [R_total, d].  Slice s = b * H_kv + h_kv holds rows
 *      index_indptr[s] .. index_indptr[s+1]-1, row r being the (b, h_kv) source
 *      row at original position index_list[r] (the position map: strictly
 *      increasing within a slice, each < T_b).  Requires DATTN_MASK_INDEX_LIST,
 *      whose visibility applies to the original positions; the packed row is a
 *      storage coordinate only.  bf16 only; kv_append does not write it. */
typedef enum { DATTN_KV_CONTIG_NHD = 0, DATTN_KV_PAGED_HND = 1, DATTN_KV_PACKED_ROWS = 2 } dattn_layout;

/* K/V element formats (M8.6 §0x05B, §0x06A-B, §0x09C, §0x0A-0x0AA).  Paged layout only for
 * the quantized formats.
 *  DATTN_FMT_BF16:       K, V bf16.
 *  DATTN_FMT_INT8_TOKEN: K, V uint8 codes [num_pages, H_kv, P, d];
 *      k_qparams, v_qparams fp16 pairs (s, z) [num_pages, H_kv, P, 2], one per
 *      (token, kv head); x_hat = code * s + z.
 *  DATTN_FMT_INT4_KIVI:  K, V uint8 [num_pages, H_kv, P, d/2], two 4-bit codes
 *      per byte, the even channel in the low nibble.
 *      k_qparams fp16 (s, z) [num_pages, H_kv, max(1, P/G), d, 2]: one pair per
 *      (G-token group, channel), stored on the page of the group's first token
 *      at slot (first_token mod P) / G (slot 0 when P < G).
 *      v_qparams fp16 (s, z) [num_pages, H_kv, P, d/Gv, 2]: per (token, Gv channels).
 *      k_residual, v_residual bf16 [B, R, H_kv, d]: token t >= n_q(T_b) of
 *      request b sits in slot t mod R, where n_q(T) = G * ceil(max(0, T - R) / G)
 *      (the residual holds at most R rows; its oldest G rows close into a
 *      group while it holds more than R, M8.6 §0x06B).
 *  DATTN_FMT_FP8_E4M3:   K, V uint8 E4M3 codes [num_pages, H_kv, P, d] (sign,
 *      4 exponent bits with bias 7, 3 mantissa bits; no infinities, 0x7F / 0xFF
 *      NaN, largest magnitude 448).  k_qparams, v_qparams fp32 [H_kv]: one scale
 *      per kv head, NULL for 1 (no calibration); x_hat = value(code) * s_h.
 *  DATTN_FMT_FP8_E5M2:   the same with E5M2 codes (5 exponent bits with bias 15,
 *      2 mantissa bits, the upper byte of the IEEE half of the same value;
 *      largest finite magnitude 57344).
 *  DATTN_FMT_INT4_HEAD:  per-head asymmetric KV4 (M8.6 §0x09C): K, V uint8
 *      [num_pages, H_kv, P, d/2], two 4-bit codes per byte, the even channel in
 *      the low nibble; k_qparams, v_qparams fp16 pairs (s, o) [num_pages, H_kv, P, 2],
 *      one per (token, kv head), with the floating offset o not clamped to the
 *      code range; x_hat = (code - o) * s.  kv_append writes s = fp16((max - min) / 15),
 *      o = fp16(-min / ((max - min) / 15)) (fp32 arithmetic, fp16 saturated to
 *      +-65504; a constant head stores s = 1, o = fp16(-min); a scale below 2^-14
 *      is raised to 2^-14 and the offset computed with it) and codes
 *      clip(rint(x / s + o), 0, 15) with the stored s, o.  K/V rows must be finite. */
typedef enum {
  DATTN_FMT_BF16 = 0,
  DATTN_FMT_INT8_TOKEN = 1,
  DATTN_FMT_INT4_KIVI = 2,
  DATTN_FMT_FP8_E4M3 = 3,
  DATTN_FMT_FP8_E5M2 = 4,
  DATTN_FMT_INT4_HEAD = 5
} dattn_format;

/* Visibility programs.  Query row i of request b sits at position
 * p_i = T_b - S_q + i and has frontier F_i = max(0, min(T_b, p_i + 1))
 * (bottom-right alignment, M4.5 §0x08B).
 *  DATTN_MASK_CAUSAL:      keys [0, F_i).
 *  DATTN_MASK_SINK_WINDOW: keys [0, min(n_sink, F_i)) U [max(0, F_i - window), F_i)
 *                          (M5.4 §0x05 union, never double counted).
 *  DATTN_MASK_INDEX_LIST:  keys of the sorted list of (b, h_kv) that are < F_i
 *                          (per-kv-head retained sets, M5.4 §0x06E shape).
 *  DATTN_MASK_FLASHMASK:   two masked query-row intervals per key column (M4.5
 *                          §0x06A): key j in [0, T_b) is hidden from query row i of
 *                          the call (0 <= i < S_q) when UTS_j <= i < UTE_j or
 *                          LTS_j <= i < LTE_j, with (UTS, UTE, LTS, LTE)_j =
 *                          fm_intervals[off_b + j], off_b = T_0 + ... + T_{b-1}
 *                          (device int32 [sum T_b, 4], one set per request, shared
 *                          by its heads).  No causal limit applies.  Every format;
 *                          INT4 KIVI with a power-of-two page_size (else
 *                          EUNSUPPORTED). */
typedef enum {
  DATTN_MASK_CAUSAL = 0,
  DATTN_MASK_SINK_WINDOW = 1,
  DATTN_MASK_INDEX_LIST = 2,
  DATTN_MASK_FLASHMASK = 3
} dattn_mask_kind;

/* Tile classes of M4.5 §0x05C. */
typedef enum { DATTN_TILE_SKIP = 0, DATTN_TILE_FULL = 1, DATTN_TILE_PARTIAL = 2 } dattn_tile_class;

/* The static problem: the dispatch/plan key of M4.5 §0x07A and §0x07F. */
typedef struct {
  int32_t B;              /* requests (>= 1)                                        */
  int32_t S_q;            /* query rows per request (>= 1)                          */
  int32_t H_q, H_kv;      /* heads; H_q % H_kv == 0, g = H_q / H_kv, g * S_q <= 32  */
  int32_t d_h;            /* head width, 64 or 128 (d_v = d_h)                      */
  int32_t layout;         /* dattn_layout                                           */
  int32_t fmt;            /* dattn_format                                           */
  int32_t page_size;      /* P >= 1 (paged); ignored for contiguous                  */
  int32_t num_pages;      /* pool pages (paged): every page id must be < num_pages  */
  int32_t T_cap;          /* token capacity per contiguous cache row                */
  int32_t B_cache;        /* contiguous cache rows                                  */
  int32_t kivi_group;     /* G  (INT4 KIVI, K tokens per group), e.g. 32            */
  int32_t kivi_v_group;   /* Gv (INT4 KIVI, V channels per group), e.g. 32          */
  int32_t kivi_residual;  /* R  (INT4 KIVI, residual rows), multiple of G           */
  int32_t mask;           /* dattn_mask_kind                                        */
  int32_t n_sink;         /* SINK_WINDOW: sink rows (>= 0)                          */
  int32_t window;         /* SINK_WINDOW: recent rows (>= 1)                        */
  float   sm_scale;       /* softmax scale; 0 selects 1 / sqrt(d_h)                 */
  int32_t fixed_splits;   /* > 0: that many balanced splits per (request, kv head)
                             (M4.5 §0x03B); 0: the planner chooses chunks          */
} dattn_problem;

/* Host-side inputs of the planner. */
typedef struct {
  const int32_t* kv_len;        /* host [B]: stored rows T_b (>= 0)                       */
  const int32_t* page_indptr;   /* host [B+1] or NULL: checked against ceil(T_b / P); when
                                   given, runs take the page-list bounds from the plan, so
                                   the device page_indptr must hold the same contents    */
  const int32_t* index_indptr;  /* host [B*H_kv+1], INDEX_LIST only: list of (b, h_kv) is
                                   index_list[index_indptr[b*H_kv+h] : ...[b*H_kv+h+1]]  */
  const int32_t* index_list;    /* host or NULL; when given, every list is checked to be
                                   strictly increasing and inside [0, T_b)               */
  int32_t num_sms;              /* SMs to plan for (>= 1)                                 */
  int32_t ctas_per_sm;          /* resident CTAs per SM to plan for; 0 = library default  */
  int32_t chunk_tokens;         /* chunk width in keys; 0 = planner default               */
  int32_t fused_merge;          /* 1: bf16 groups of several chunks are merged inside the
                                   partial kernel by the last CTA to finish them (one
                                   launch); 0: by the LSE-merge kernel.  Off by default: on
                                   GB300 the merge then sits on the partial kernel's tail,
                                   and the step is slower (see the design notes)          */
  const int32_t* qo_indptr;     /* host [B+1] or NULL: a mixed batch (M4.5 §0x08F).  Request
                                   b has C_b = qo_indptr[b+1] - qo_indptr[b] query rows
                                   (0 <= C_b <= S_q), packed rows qo_indptr[b] .. of q, o
                                   and lse ([qo_indptr[B], H_q, d] and [qo_indptr[B], H_q]),
                                   at positions T_b - C_b + i (bottom-right).  NULL: C_b =
                                   S_q for every request.  Non-uniform C_b: every format;
                                   INT4 KIVI with a power-of-two page_size (else
                                   EUNSUPPORTED) */
  int32_t item_cost_keys;       /* default (equal-segment) mode: the fixed cost of a work
                                   item, in keys, charged when the concatenated streams are
                                   cut into one segment per CTA, so that a CTA holding many
                                   short items (tiny requests) gets fewer keys.  0 = library
                                   default (about 48 KB of K/V per item); < 0 = none     */
  int32_t merge_tags;           /* bf16 plans with an LSE-merge kernel: 1 = every partial
                                   warp tags its state rows with the run's number once
                                   written (after one gpu-scope fence), and the merge folds
                                   each group as soon as its states carry the tag, while the
                                   rest of the partial grid still runs; -1 = the merge waits
                                   for the whole partial grid; 0 = library default (tags
                                   when the merge folds at least 64 group rows).
                                   Ignored for the other formats (their merge waits for
                                   the grid) and for fused_merge plans                    */
} dattn_plan_inputs;

typedef struct dattn_plan_s dattn_plan_t;

/* Device buffers of one call.  Unused pointers may be NULL. */
typedef struct {
  const void* q;                 /* device bf16 [B, S_q, H_q, d]                          */
  const void* k;                 /* device K cache (layout / format above)                */
  const void* v;                 /* device V cache                                        */
  const void* k_qparams;         /* device, INT8 / INT4 KIVI / FP8 (scales, may be NULL)  */
  const void* v_qparams;
  const void* k_residual;        /* device, INT4 KIVI                                     */
  const void* v_residual;
  const int32_t* page_indptr;    /* device [B+1], paged                                   */
  const int32_t* page_indices;   /* device, paged                                         */
  const int32_t* cache_batch_idx;/* device [B] or NULL, contiguous                        */
  const int32_t* index_indptr;   /* device [B*H_kv+1], INDEX_LIST                          */
  const int32_t* index_list;     /* device, INDEX_LIST                                     */
  void* o;                       /* device bf16 [B, S_q, H_q, d] (output)                  */
  float* lse;                    /* device fp32 [B, S_q, H_q] (output) or NULL             */
  const int32_t* fm_intervals;   /* device int32 [sum T_b, 4], FLASHMASK, 16-byte aligned  */
} dattn_tensors;

/* Summary of a plan, for reporting (split counts of M4.5 §0x0AC). */
typedef struct {
  int64_t workspace_bytes;  /* bytes dattn_run needs                                   */
  int64_t blob_bytes;       /* of which: work list copied host->device on every run    */
  int32_t n_items;          /* work items (request, kv head, key chunk)                */
  int32_t n_ctas;           /* CTAs of the partial kernel                              */
  int32_t n_slots;          /* partial-state slots (items that do not write O directly) */
  int32_t n_merge_groups;   /* (request, kv head) groups with more than one item       */
  int32_t max_splits;       /* largest number of items of one group                    */
  int32_t rows;             /* query rows per group, g * S_q                           */
  int64_t stream_keys;      /* keys read by all groups (sum of visible streams)        */
  int64_t max_cta_keys;     /* keys of the most loaded CTA                             */
  int32_t fused_merge;      /* 1: the last CTA to finish a group's chunks merges it     */
                            /*    inside the partial kernel (no merge launch)          */
  int32_t merge_tags;       /* 1: the merge waits for state-row tags (see merge_tags)  */
} dattn_plan_info;

/* One work item as planned: keys [a, e) of the visible stream of (b, h_kv).
 * slot < 0: the item writes O/LSE directly; else it writes partial slot "slot". */
typedef struct {
  int32_t b, h_kv, a, e, slot, cta;
} dattn_work_item;

/* ---- planning (host only; usable without a GPU) ------------------------------------ */

/* Validates the call, builds the visible key stream of every (request, kv
 * head), cuts it into chunks (balanced quotient/remainder bounds when
 * fixed_splits > 0, M4.5 §0x03B; otherwise chunks of equal width assigned
 * longest-first to the least-loaded CTA, the planner of M4.5 §0x09E), and
 * sizes the workspace (M4.5 §0x03D-§0x03E).  *out receives a plan owned by the
 * caller (free it with dattn_plan_destroy); *workspace_bytes the bytes that
 * dattn_run needs.  Returns EINVAL / EUNSUPPORTED with every failed check in
 * dattn_last_error(). */
dattn_status dattn_plan(const dattn_problem* prob, const dattn_plan_inputs* in,
                        dattn_plan_t** out, size_t* workspace_bytes);

void dattn_plan_destroy(dattn_plan_t* plan);

/* Copies the plan summary into *info. */
dattn_status dattn_plan_get_info(const dattn_plan_t* plan, dattn_plan_info* info);

/* Copies up to "capacity" planned items into "items" (host) in item order and
 * stores the item count in *count. */
dattn_status dattn_plan_get_items(const dattn_plan_t* plan, dattn_work_item* items,
                                  int32_t capacity, int32_t* count);

/* ---- execution ---------------------------------------------------------------------- */

/* Runs one decode step: copies the plan's work list into the head of
 * "workspace" (device, >= info.workspace_bytes, 256-byte aligned), launches
 * the partial kernel (producer warps streaming K/V rows through a shared
 * memory ring, consumer warps updating exact (m, l, u) states) and, when some
 * group has several chunks, merges their states (M4.5 §0x03I) with a second,
 * LSE-merge kernel, or, for a bf16 plan made with fused_merge, inside the
 * partial kernel (the last CTA to finish a group's chunks merges it;
 * info.fused_merge = 1).  A fused run that ended with a device error leaves
 * the merge counters undefined: upload the plan again (a run without
 * DATTN_RUN_REUSE_UPLOAD) afterwards.  "prob" must equal the planned problem
 * (else ESTALE_PLAN).  Device-side bounds checks (page id < num_pages, block
 * inside the request's page list, list entry inside [0, T_b), cache row <
 * B_cache) raise a flag that dattn_device_status reports; the offending rows
 * are never read (they are skipped, or taken as zero rows), so the outputs of
 * the groups they belong to are undefined.  Device list bounds that disagree
 * with the plan drop the group's keys: its rows come out all-masked. */
dattn_status dattn_run(const dattn_plan_t* plan, const dattn_problem* prob,
                       const dattn_tensors* t, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Options of dattn_run_ex. */
#define DATTN_RUN_REUSE_UPLOAD 1u  /* the workspace already holds this plan's work list
                                      (dattn_plan_upload or an earlier run with this plan and
                                      workspace); skip the host->device copy. The caller
                                      guarantees that nothing overwrote the workspace since. */
#define DATTN_RUN_SHARED_SHIFT 2u  /* shared-shift partials (M4.5 §0x09C, bf16 K/V only): the
                                      partial states accumulate e^(s - phi) v and e^(s - phi)
                                      in the common frame "shift_phi" (natural-log score
                                      units, s = q.k * sm_scale) with no running maximum, as
                                      long as every visible score of a consumer warp's keys
                                      satisfies shift_lo < s - phi < shift_hi (the range
                                      guard); a warp whose guard fails continues in the
                                      synchronized running-max frame from that point (the
                                      fallback), so the result is the softmax either way.
                                      Requires -80 <= shift_lo < shift_hi <= 40 and a finite
                                      shift_phi.  dattn_shift_fallbacks counts the fallbacks */
#define DATTN_RUN_TEST_SKIP_ARRIVAL 4u  /* test hook of the fail-closed path (M4.5 §0x07B),
                                      bf16 K/V only: the producers of CTA 0 withhold the
                                      completion of its first ring stage, so its consumers'
                                      bounded wait runs out after wait_limit_us (required,
                                      1 .. 100000).  Nothing faults or hangs: the CTA stops,
                                      the status word gets the timeout bit (16) and no output
                                      row is written from the states it left unwritten (the
                                      rows of the groups it worked on stay as they were) */
typedef struct {
  uint32_t flags;     /* DATTN_RUN_* bits                                                  */
  void* events[3];    /* cudaEvent_t (as void*) recorded on "stream" before the partial
                         kernel, after it and after the merge kernel; NULL entries skipped */
  float shift_phi, shift_lo, shift_hi;   /* DATTN_RUN_SHARED_SHIFT frame and guard      */
  uint32_t wait_limit_us;   /* limit of each bounded wait on a ring stage in microseconds
                               (0: 2 s).  A wait that runs out stops its CTA, sets the
                               timeout bit (16) of the device status word, and its warps
                               mark their partial states unwritten, so that no output row
                               depending on them is written (fail closed, row by row)      */
  void* trace;        /* NULL, or (bf16 K/V) a device uint64 array of at least
                         16 n_ctas + 2 n_merge_groups rows words (zeroed by the caller):
                         %globaltimer stamps in ns.  Partial CTA c writes words
                         16 c + {0: entry, 1: records read, 2: producer warp 0 past
                         the wait for the preceding grid, 3: its first stage's copies
                         issued, 4: the first stage landed for consumer warp 0,
                         5: the SM it ran on (%smid), 8 + w: consumer warp w done};
                         merge block j then writes
                         16 n_ctas + 2 j (past its wait) and + 2 j + 1 (done)        */
} dattn_run_options;

/* Number of consumer warps that left the shared-shift frame (guard failed) since the work
 * list was last uploaded to "workspace" (synchronises "stream"). */
dattn_status dattn_shift_fallbacks(const void* workspace, int32_t* count, void* stream);

/* Copies the plan's work list into the head of "workspace" (stream-ordered).
 * A plan is typically built once per decode step and then run by every layer
 * of the model with DATTN_RUN_REUSE_UPLOAD (the FlashInfer plan/run split,
 * M4.5 §0x0AD), so the copy happens once per step. */
dattn_status dattn_plan_upload(const dattn_plan_t* plan, void* workspace, size_t workspace_bytes,
                               void* stream);

/* dattn_run with options (NULL = dattn_run). */
dattn_status dattn_run_ex(const dattn_plan_t* plan, const dattn_problem* prob,
                          const dattn_tensors* t, void* workspace, size_t workspace_bytes,
                          void* stream, const dattn_run_options* options);

/* ---- one step from host memory (the end-to-end path) --------------------------------
 *
 * The plan/run lifecycle of M4.5 §0x07F and §0x0AD in one call for a caller
 * whose query and page table live in host memory: plan from the host lengths,
 * one host->device transfer of the query, the page table and the work list,
 * the partial and merge kernels, one device->host transfer of O and LSE, then
 * the results are copied into the caller's host arrays.  Returns after the
 * step has completed on "stream" (it synchronises the stream).  The cache
 * (K, V and their qparams / residual) stays on the device: "cache" supplies
 * only those pointers; its q, o, lse, page_indptr, page_indices fields are
 * ignored.  Visibility programs that read device-side lists (INDEX_LIST,
 * FLASHMASK) and mixed batches go through dattn_plan / dattn_run instead
 * (EUNSUPPORTED here).  The step's device bounds-check word is read with
 * dattn_step_host_status.
 *
 * Layouts (offsets from the start of each buffer, 256-byte aligned pieces):
 *   workspace: [q | page_indptr | page_indices | plan workspace | O | LSE]
 *   staging:   [q | page_indptr | page_indices | work list | ... | O | LSE] in
 *              pinned host memory; the first four are sent in one transfer, O
 *              and LSE come back in one transfer into the buffer's last
 *              round_up(O, 256) + round_up(LSE, 256) bytes (16-byte aligned).
 * The staging buffer should be page-locked (cudaHostAlloc / pinned) so that
 * both transfers are asynchronous DMA; the library never allocates it. */
typedef struct {
  const void* q;                 /* host bf16 [B, S_q, H_q, d]                             */
  const int32_t* kv_len;         /* host [B]: stored rows T_b                              */
  const int32_t* page_indptr;    /* host [B+1] (paged layout; NULL for contiguous)         */
  const int32_t* page_indices;   /* host [page_indptr[B]] (paged layout)                   */
  void* o;                       /* host bf16 [B, S_q, H_q, d] (output)                    */
  float* lse;                    /* host fp32 [B, S_q, H_q] (output) or NULL               */
  int32_t num_sms;               /* SMs to plan for (>= 1)                                 */
} dattn_host_step;

/* Bytes of the device workspace and of the pinned staging buffer that
 * dattn_step_host needs for this call (it plans once to find out). */
dattn_status dattn_step_host_sizes(const dattn_problem* prob, const dattn_host_step* io,
                                   size_t* workspace_bytes, size_t* staging_bytes);

/* One decode step through host memory (see above).  The transfer of q and the
 * page table is issued before the host plans, so that it overlaps planning;
 * it writes only the workspace's input region.  Every other check (the plan's
 * validation, the full workspace and staging sizes) runs before any kernel is
 * launched; a failure returns its status (EWORKSPACE names the sizes needed)
 * after the stream has at most received that one transfer. */
dattn_status dattn_step_host(const dattn_problem* prob, const dattn_host_step* io, const dattn_tensors* cache,
                             void* staging, size_t staging_bytes, void* workspace, size_t workspace_bytes,
                             void* stream);

/* The same step split in two, so that the host work of the next step (its
 * staging copies and planning) overlaps this step on the device.
 * dattn_step_host_submit does everything dattn_step_host does up to the
 * enqueue of the output transfer, records "done_event" (a cudaEvent_t as
 * void*, required) on "stream" after it and returns without waiting.
 * dattn_step_host_finish waits for "done_event" and copies O and LSE from the
 * staging buffer into io->o / io->lse.  Between the two calls the staging
 * buffer belongs to the step: a pipelined caller alternates two staging
 * buffers (and two events); steps on one stream may share a workspace.
 * Errors as for dattn_step_host; a failed submit records no event. */
dattn_status dattn_step_host_submit(const dattn_problem* prob, const dattn_host_step* io,
                                    const dattn_tensors* cache, void* staging, size_t staging_bytes,
                                    void* workspace, size_t workspace_bytes, void* stream, void* done_event);
dattn_status dattn_step_host_finish(const dattn_problem* prob, const dattn_host_step* io, const void* staging,
                                    size_t staging_bytes, void* done_event);

/* The step's transfers on streams of their own (dattn_step_host_submit_ex).
 * Every field is required (cudaStream_t / cudaEvent_t as void*, caller-owned).
 * The two directions take two streams: on one stream, step k+1's inputs would
 * queue behind step k's outputs, which wait for step k's kernels. */
typedef struct {
  void* h2d_stream;     /* carries the host->device transfers                       */
  void* d2h_stream;     /* carries the device->host transfer                        */
  void* inputs_event;   /* recorded on h2d_stream once the step's inputs are sent;
                           "stream" waits for it before the kernels                  */
  void* kernels_event;  /* recorded on "stream" after the kernels; d2h_stream waits
                           for it before the output transfer                         */
} dattn_step_copies;

/* dattn_step_host_submit with the transfers on the streams of "copies" (NULL
 * copies: dattn_step_host_submit).  The host->device stream first waits for
 * done_event's previous record, the last step that used this staging buffer
 * and workspace, then sends the inputs; the kernels run on "stream" after
 * them; the outputs come back on the device->host stream, after which
 * done_event is recorded there.  A caller that alternates two (staging,
 * workspace, event set) slots thus sends step k+1's inputs and receives step
 * k-1's outputs while step k's kernels run.  Steps that share a workspace
 * must not be in flight together.  EINVAL when done_event, or a field of a
 * non-NULL copies, is NULL; otherwise errors as for dattn_step_host. */
dattn_status dattn_step_host_submit_ex(const dattn_problem* prob, const dattn_host_step* io,
                                       const dattn_tensors* cache, void* staging, size_t staging_bytes,
                                       void* workspace, size_t workspace_bytes, void* stream, void* done_event,
                                       const dattn_step_copies* copies);

/* Device bounds-check word of the last dattn_step_host on this workspace (like
 * dattn_device_status; synchronises "stream"). */
dattn_status dattn_step_host_status(const dattn_problem* prob, const dattn_host_step* io, const void* workspace,
                                    int32_t* flags, void* stream);

/* Size of the library-owned scratch array that dattn_run_noalloc uses on each device. */
#define DATTN_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)  /* 16 MiB */

/* dattn_run without a caller workspace; the pages have no counterpart of this
 * call.  It serves callers that cannot allocate device memory or hand over a
 * buffer at step time.  Examples: an engine that reserved all of HBM for its
 * K/V page pool at start-up, and a latency-bound decode loop that cannot take
 * the device synchronisation of cudaMalloc / cudaFree.
 *
 * Scratch array:
 *  - The workspace is a file-scope device array of DATTN_NOALLOC_SCRATCH_BYTES
 *    (256-byte aligned).
 *  - Every GPU on which the library's device code is loaded holds that array
 *    until the process exits.
 *  - The call itself allocates nothing: no cudaMalloc, no cudaFree, no
 *    allocating library routine.
 *
 * First call on a device:
 *  - It looks up the array's address with cudaGetSymbolAddress on the current
 *    device and keeps it, per device ordinal, for later calls.
 *  - Make that call before any stream capture on that device.
 *  - The kept address belongs to the device's primary context as it was at
 *    that call: after cudaDeviceReset, or from a thread bound to another
 *    driver context of the same device, it no longer names the array, so
 *    neither case is supported once a call has been made.
 *
 * Copies:
 *  - Each call copies the plan's work list from the plan's host memory into
 *    the array, on "stream".  That host memory is ordinary (pageable), so
 *    CUDA may complete this copy synchronously with respect to the host
 *    before the call returns; a caller that needs the call to return at once
 *    uses dattn_plan_upload / dattn_run_ex with its own workspace instead.
 *
 * Sharing and races:
 *  - All calls on a device share the one array, which keeps the last call's
 *    contents.
 *  - The only part that must start at zero is the device status word. It is
 *    cleared by the work-list copy that each call enqueues.
 *  - Calls whose work overlaps on the GPU (different streams, or other host
 *    threads) race on the array. Serialise them on one stream.
 *
 * Errors:
 *  - A plan whose info.workspace_bytes exceeds DATTN_NOALLOC_SCRATCH_BYTES
 *    gets DATTN_EWORKSPACE and a message; use dattn_run for it.
 *  - Any other argument error is reported as dattn_run reports it.
 *
 * The device bounds checks of this call (page id outside the pool, block
 * outside the request's page list, ...) and a bounded wait that gave up are
 * reported in the array's status word: read it with dattn_noalloc_status. */
dattn_status dattn_run_noalloc(const dattn_plan_t* plan, const dattn_problem* prob,
                               const dattn_tensors* t, void* stream);

/* Device status word of the last dattn_run_noalloc on the current device, read
 * from the library's scratch array (like dattn_device_status: synchronises
 * "stream", *flags = 0 when no device check fired, DATTN_EDEVICE_CHECK when
 * one did).  Allocates nothing; the pages have no counterpart. */
dattn_status dattn_noalloc_status(int32_t* flags, void* stream);

/* Reads the device status word of the last run that used "workspace"
 * (synchronises "stream").  *flags = 0 when no device check fired. */
dattn_status dattn_device_status(const void* workspace, int32_t* flags, void* stream);

/* ---- cache writer ---------------------------------------------------------------------- */

typedef struct {
  const int32_t* kv_len_old;   /* host [B]: committed rows before the append            */
  const int32_t* new_indptr;   /* host [B+1]: request b appends rows
                                  new_indptr[b] .. new_indptr[b+1]-1 of k_new / v_new    */
  const int32_t* page_indptr;  /* host [B+1]: same contents as the device page_indptr   */
} dattn_append_inputs;

/* Bytes of scratch kv_append needs for B requests. */
size_t kv_append_workspace_bytes(const dattn_problem* prob);

/* Appends bf16 rows k_new, v_new (device, packed [sum n_b, H_kv, d]) at
 * positions kv_len_old[b] .. kv_len_old[b] + n_b - 1 of each request, writing
 * codes and qparams together (M8.6 §0x05B, §0x06B):
 *  - BF16: rows copied into their pages.
 *  - INT8: per (token, kv head) s = fp16((max - min) / 255) (fp32 divide),
 *    z = fp16(min), s = 1 when max == min, s raised to 2^-14 when smaller;
 *    code = clip(rint_even((x - z) / s), 0, 255) with the re-read stored s, z.
 *  - INT4 KIVI: every K group of G tokens that closes gets per-channel (s, z)
 *    with 15 levels, its V rows per-token (s, z) per Gv channels; rows that
 *    stay inside the residual are written to the residual ring.  The ring must
 *    hold the request's previous residual rows (as this function leaves them).
 *  - FP8 E4M3: code = nearest E4M3 value to x / s_h (the quotient rounded in
 *    fp32), ties to the even code, saturated to +-448; the scales are inputs.
 *  - FP8 E5M2: the same, saturated to +-57344.
 * Capacity (page list long enough for the new length) and arguments are
 * checked on the host before any write.  The caller advances its lengths
 * after the stream reaches this point.  "workspace" (device,
 * kv_append_workspace_bytes) holds the per-request descriptors. */
dattn_status kv_append(const dattn_problem* prob, const dattn_append_inputs* in,
                       const dattn_tensors* cache, const void* k_new, const void* v_new,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ---- bit-exact debug hooks (same device functions as the kernels) -------------------- */

/* For n coordinates (b, t, h_q, x) (device int32 [n, 4]) writes the element
 * offset of K[b, t, h_kv(h_q), x] in the K cache (device int64 [n]), or -1 when
 * the coordinate is outside the request's stored rows or its page list
 * (M4.5 §0x04A-§0x04F, the four invariants of §0x04H). */
dattn_status dattn_debug_translate(const dattn_problem* prob, const dattn_tensors* t,
                                   const int32_t* kv_len, const int32_t* coords, int32_t n,
                                   int64_t* out, void* stream);

/* For n tiles (b, h_kv, j) (device int32 [n, 3]) writes the exact class
 * (dattn_tile_class, device int32 [n]) of the tile "every query row of the
 * group x keys [j P, (j + 1) P)", using the visibility program of "prob"
 * (M4.5 §0x05C; keys >= T_b are masked).  kv_len is device int32 [B]. */
dattn_status dattn_debug_classify(const dattn_problem* prob, const dattn_tensors* t,
                                  const int32_t* kv_len, const int32_t* tiles, int32_t n,
                                  int32_t* out, void* stream);

/* Writes, for group (b, h_kv), the logical key positions that the planned
 * items read, in stream order (device int32, capacity entries), and the
 * number of positions in *count (host).  Uses the plan's work list, which it
 * copies into "workspace" like dattn_run. */
dattn_status dattn_debug_gather(const dattn_plan_t* plan, const dattn_problem* prob,
                                const dattn_tensors* t, void* workspace, size_t workspace_bytes,
                                int32_t b, int32_t h_kv, int32_t* out, int32_t capacity,
                                int32_t* count, void* stream);

/* ---- misc ---------------------------------------------------------------------------- */

/* Text listing every failed check of the last failing call on this thread. */
const char* dattn_last_error(void);

/* Library ABI version (major * 100 + minor). */
int32_t dattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DATTN_H */
