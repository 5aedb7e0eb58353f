// Internal definitions shared by the host planner and the CUDA kernels of libdattn.
#pragma once

#include <cstddef>
#include <cstdint>

#include <vector_types.h>

#include "dattn.h"

namespace dattn {

// ---- kernel geometry ---------------------------------------------------------------
constexpr int kTK = 64;              // keys per pipeline stage
constexpr int kConsumerWarps = 8;    // two warpgroups that compute
constexpr int kProducerWarps = 4;    // one warpgroup that fills the ring, a stage per warp in turn
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kProducerRegs = 56;    // setmaxnreg split of the launch's register file:
constexpr int kConsumerRegs = 224;   // 128 * 56 + 256 * 224 = 64512 = 384 threads * 168
constexpr int kMaxRows = 32;         // g * S_q rows per (request, kv head) group
constexpr int kDefaultCtasPerSm = 1;
constexpr int kWsAlign = 256;
constexpr uint32_t kBlobMagic = 0x64617474u;  // "datt"

// Device status bits (workspace header word).
enum StatusBits : int32_t {
  kStPageRange = 1,     // page id outside [0, num_pages)
  kStBlockRange = 2,    // logical block outside the request's page list
  kStListRange = 4,     // index-list entry outside [0, T_b) or list length mismatch
  kStRowRange = 8,      // contiguous cache row / token outside its capacity
  kStTimeout = 16,      // a bounded barrier wait gave up
  kStAppend = 32,       // kv_append met an inconsistent descriptor
  kStPipeline = 64,     // a consumer found a ring stage stamped with another stage number
};

// KIVI INT4 problems with d = 128 (Gv = 16 or 32) or d = 64 (Gv = 16), at most
// 32 rows, an interval visibility program and a power-of-two page size P run
// on the tensor-core kernel (partial_q4.cu); other KIVI problems on the
// byte-format kernel (partial.cu).  The residual length R is any positive
// multiple of G on both.
inline bool kivi_on_tensor_cores(int d, int rows, int Gv, int mask, int P, int R) {
  return ((d == 128 && (Gv == 16 || Gv == 32)) || (d == 64 && Gv == 16)) && rows <= 32 &&
         mask != DATTN_MASK_INDEX_LIST && P > 0 && (P & (P - 1)) == 0 && R > 0;
}

// Partial states an item leaves per query row.  Consumer warps are arranged
// in row blocks (16 rows, one mma tile, in the bf16 and INT8 tensor-core
// kernels, 8 rows in the KIVI and per-head INT4 ones; 4 rows in the
// byte-format kernel); every
// warp leaves the state of its block's rows over its own share of the item's
// keys.
inline int states_per_item(int rows, int fmt, bool kivi_tc) {
  if (fmt == DATTN_FMT_INT4_HEAD || (fmt == DATTN_FMT_INT4_KIVI && kivi_tc))
    return kConsumerWarps / (rows <= 8 ? 1 : rows <= 16 ? 2 : 4);
  if (fmt != DATTN_FMT_INT4_KIVI) return kConsumerWarps / (rows <= 16 ? 1 : 2);
  return kConsumerWarps / (rows <= 4 ? 1 : rows <= 8 ? 2 : rows <= 16 ? 4 : 8);
}

// One unit of producer work: keys [a, e) of the visible stream of group (b, h).
// Interval programs: stream index j maps to position j < x0 ? j : x1 + (j - x0).
// Index lists: x0 is the list offset of the group, position = index_list[x0 + j].
// FlashMask: position = j (x0 = T), x1 = the request's row offset in fm_intervals.
struct WorkItem {
  int32_t b, h, a, e, slot, T, x0, x1;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

struct MergeGroup {
  int32_t b, h, slot0, n;
  int32_t qo, nq;      // request b's first packed query row and its query rows C_b
  int32_t pad0, pad1;
};
static_assert(sizeof(MergeGroup) == 32, "MergeGroup layout");

// A work item with its request's page-list bounds, stored in CTA order so a
// CTA reads its items with one dependent load.
struct ItemRec {
  WorkItem it;
  int32_t lo, hi;      // paged layout: page list entries [lo, hi) of request it.b
  int32_t crow;        // contiguous layout: cache row, resolved by the kernel
  int32_t merge;       // index of the item's merge group, -1 when it writes O directly
  int32_t qo, nq;      // request it.b's first packed query row and its query rows C_b
  int32_t ring_off;    // INT4 KIVI: residual key t sits in ring slot t + ring_off, less R once >= R
  int32_t pad1;
};
static_assert(sizeof(ItemRec) == 64, "ItemRec layout");

// Head of the plan blob, copied to the start of the workspace by every run.
struct BlobHeader {
  uint32_t magic;
  int32_t status;        // device status word, zeroed by the copy
  int32_t n_items, n_ctas, n_merge, rows, n_slots;
  int32_t fused;         // merge groups merged inside the partial kernel
  int32_t shift_fallbacks;   // warps that left the shared-shift frame, zeroed by the upload
  int32_t tags;          // the separate merge waits for state-row tags, not for the whole grid
  int64_t off_items, off_cta_indptr, off_cta_items, off_merge, off_ml, off_u, off_cta_recs;
  int64_t off_count;     // int32 [n_merge]: finished items per merge group (fused merge)
  int64_t off_seq;       // int32 [rows][n_slots]: run tag of every state row (when tags), zeroed
};
static_assert(sizeof(BlobHeader) == 112, "BlobHeader layout");

// Arguments of the partial kernel (passed by value as a grid constant).
struct PartialParams {
  const void* q;
  const void* k;
  const void* v;
  const void* kqp;
  const void* vqp;
  const void* kres;
  const void* vres;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const int32_t* cache_batch_idx;
  const int32_t* index_indptr;
  const int32_t* index_list;
  const int32_t* fm_intervals;   // FLASHMASK: [sum T_b, 4]
  void* o;
  float* lse;
  const WorkItem* items;
  const int32_t* cta_indptr;   // [n_ctas + 1]: item range of every CTA
  const int32_t* cta_items;
  const ItemRec* cta_recs;   // the items of cta_items as records, same order
  float2* ml;            // [n_slots * rows] (m in log2 units, l)
  float* u;              // [n_slots * rows * d]
  int32_t* status;
  const MergeGroup* groups;   // [n_merge]
  int32_t* group_count;       // [n_merge], fused merge: zero between runs
  int32_t fused;              // 1: the last CTA to finish a group merges it
  int32_t B, S_q, H_q, H_kv, g, rows;
  int32_t layout, fmt, mask, P, num_pages, T_cap, B_cache;
  int32_t n_sink, window, kivi_G, kivi_Gv, kivi_R;
  int32_t P_shift;       // log2(P) when P is a power of two, else -1
  float scale_log2;      // sm_scale * log2(e)
  int32_t shift_on;       // shared-shift partials (bf16 kernel)
  float shift_phi2, shift_lo2, shift_hi2;   // frame and guard, log2 units
  int32_t* shift_fallbacks;
  uint64_t wait_ns;       // limit of every bounded mbarrier wait
  int32_t skip_arrival;   // test hook (bf16 kernel): CTA 0 never completes its first stage
  uint64_t* trace;        // timeline trace (bf16 kernel): kTraceSlots %globaltimer stamps per CTA, or null
  // Separate merge: the tag of each state row, [rows][n_slots] (a row's tags of
  // consecutive states are adjacent, as the merge polls them), stored once the
  // row's (m, l, u) is written; null when no merge kernel follows.
  int32_t* state_seq;
  int32_t run_seq;        // this run's tag (never 0)
  int32_t n_slots;
};

// Timeline trace of the bf16 partial kernel: per CTA, kTraceSlots words of
// %globaltimer (ns): entry, records read, producer warp 0 past the wait for the
// preceding grid, its first stage's copies issued, the first stage landed for
// consumer warp 0, the SM the CTA runs on (slot 5, %smid, not a time), the
// first stage's page ids checked by producer warp 0 (slot 6, page-run
// producer), and the end of each consumer warp (slots 8 + warp).  The merge
// kernel follows with two words per block: past its wait (or, with state tags,
// its states ready), and done.
enum TraceSlot : int { kTrEntry = 0, kTrRecords = 1, kTrWaitDone = 2, kTrFirstCopy = 3, kTrFirstStage = 4,
                       kTrSm = 5, kTrFirstPage = 6, kTrConsumerEnd = 8 };
constexpr int kTraceSlots = 16;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s

struct MergeParams {
  const MergeGroup* groups;
  const float2* ml;
  const float* u;
  void* o;
  float* lse;
  int32_t* status;
  int32_t n_groups, rows, g, S_q, H_q;
  int32_t mean_states;   // partial states per merge group, on average (chooses the warps per row)
  uint64_t* trace;       // two stamps per block (its states ready, done), or null
  const int32_t* state_seq;   // the partial kernel's state-row tags ([rows][n_slots]), or null (then wait
                              // for the whole grid)
  int32_t run_seq, n_slots;
  int32_t end_wait;      // with tags: wait for the partial grid before completing (some item
                         // writes O directly, which only the grid's completion makes visible)
  uint64_t wait_ns;      // limit of a warp's wait for its states' tags
};

// Kernel launchers (partial*.cu, merge.cu); return cudaError_t as int.
int launch_partial(const PartialParams& p, int d, int n_ctas, void* stream);
int launch_partial_bf16(const PartialParams& p, int d, int n_ctas, void* stream);
int launch_partial_q8(const PartialParams& p, int d, int n_ctas, void* stream);
int launch_partial_q4(const PartialParams& p, int d, int n_ctas, void* stream);
int launch_partial_q4h(const PartialParams& p, int d, int n_ctas, void* stream);
int launch_merge(const MergeParams& p, int d, void* stream);

}  // namespace dattn
