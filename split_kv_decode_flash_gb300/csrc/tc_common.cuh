// Pieces shared by the tensor-core partial kernels (bf16 and INT8 K/V): the
// CTA's item records, the producer's stage cursor and three-step slot
// description (logical key, page id, checked K/V row), L2 cache policies and
// the PTX wrappers (cp.async, ldmatrix, mma.sync).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "stream.cuh"

namespace dattn {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kItemCache = 256;       // work items of a CTA kept in shared memory
constexpr uint32_t kNoRow = 0xFFFFFFFFu;

// Completes item record r with what only the device knows: the page-list
// bounds when the plan was made without the host page list, the cache row
// (contiguous layout), and the index-list consistency check (keys dropped,
// e = a, when the list offsets disagree with the plan).  Reads device inputs,
// so only after griddepcontrol.wait.  Paged index-list records are complete as
// planned (rec_complete_as_planned): slot_keys makes the same check where the
// list is read, so that no CTA-wide wait precedes the first list load.
__device__ __forceinline__ ItemRec complete_rec(const PartialParams& p, ItemRec r, bool report) {
  if (p.mask == DATTN_MASK_INDEX_LIST) {
    const int g = r.it.b * p.H_kv + r.it.h;
    const int lo = p.index_indptr[g], n = p.index_indptr[g + 1] - lo;
    if (lo != r.it.x0 || r.it.e > n) {
      if (report) atomicOr(p.status, kStListRange);
      r.it.e = r.it.a;
    }
  }
  if (p.layout == DATTN_KV_PAGED_HND) {
    if (r.lo < 0) {
      r.lo = p.page_indptr[r.it.b];
      r.hi = p.page_indptr[r.it.b + 1];
    }
  } else {
    r.crow = cache_row(p.cache_batch_idx, r.it.b, p.B_cache, report ? p.status : nullptr);
  }
  return r;
}

// True when complete_rec changes nothing for this problem (paged layout with
// the page-list bounds in the plan).
__device__ __forceinline__ bool rec_complete_as_planned(const PartialParams& p, const ItemRec& r) {
  return p.layout == DATTN_KV_PAGED_HND && r.lo >= 0;
}

__device__ __forceinline__ ItemRec load_rec(const PartialParams& p, int ii, bool report) {
  return complete_rec(p, p.cta_recs[ii], report);
}

// Out of line: reached only by CTAs with more than kItemCache items, and
// inlining it at every record read would multiply the kernels' code size.
__device__ __noinline__ ItemRec load_rec_uncached(const PartialParams& p, int ii) { return load_rec(p, ii, false); }

// The CTA's item list: the first kItemCache records come from shared memory
// (filled once at kernel start), later ones from global memory.
struct Walk {
  const PartialParams& p;
  const ItemRec* cache;
  int begin, end;
  uint64_t keep;      // L2 evict-last policy for the page-table reads
  __device__ __forceinline__ ItemRec rec(int ii) const {
    return ii - begin < kItemCache ? cache[ii - begin] : load_rec_uncached(p, ii);
  }
};

// The end of a consumer warp (separate merge): tags of every state row it
// wrote, after one fence (see state_tags_fence).  rows_of(rec, state, ra, rb)
// gives, for an item, the warp's state index and the lane's two rows (-1:
// none), and whether this lane wrote their (m, l).
template <typename RowsOf>
__device__ __forceinline__ void publish_warp_states(const Walk& w, RowsOf rows_of) {
  const PartialParams& p = w.p;
  if (!p.state_seq) return;
  __syncwarp();
  state_tags_fence();
  for (int ii = w.begin; ii < w.end; ++ii) {
    const ItemRec rec = w.rec(ii);
    if (rec.it.slot < 0) continue;
    int st, ra, rb;
    if (!rows_of(rec, st, ra, rb)) continue;
    tag_state_row(p, rec.it.slot + st, ra, rec.nq);
    tag_state_row(p, rec.it.slot + st, rb, rec.nq);
  }
}

// ---- PTX wrappers -----------------------------------------------------------------------

// L2 eviction policies: K/V rows are streamed once (evict first); the page
// table and the plan's records are read by every launch and stay resident
// (evict last) while the K/V stream passes through L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ int ld_keep(const int* p, uint64_t pol) {
  int v;
  asm volatile("ld.global.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ ItemRec ld_rec_keep(const ItemRec* p, uint64_t pol) {
  ItemRec r;
  int4* d = reinterpret_cast<int4*>(&r);
  const int4* s = reinterpret_cast<const int4*>(p);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(ItemRec) / 16); ++i)
    asm volatile("ld.global.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(d[i].x), "=r"(d[i].y), "=r"(d[i].z), "=r"(d[i].w)
                 : "l"(s + i), "l"(pol));
  return r;
}

// 16-byte global -> shared copy; src_bytes = 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes), "l"(pol)
               : "memory");
}

// Arrive on "bar" once every earlier cp.async of this thread has landed (the
// pending count is raised first, so the barrier's expected count is unchanged).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

// c += a (16x16, row-major bf16) * b (16x8, column-major bf16), fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// c += a (16x16, row-major f16) * b (16x8, column-major f16), fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 4-byte global -> shared copy (cache-all path); src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// Byte offset of 16-byte chunk c of key slot s inside a stage tile whose rows
// hold ROWB bytes; chunks are XOR-swizzled by the slot's low bits so the
// rows read together by a warp fall in distinct bank groups.
template <int ROWB>
__device__ __forceinline__ uint32_t tile_off(int s, int c) {
  constexpr int kMask = ROWB / 16 >= 8 ? 7 : ROWB / 16 - 1;
  return static_cast<uint32_t>(s * ROWB + ((c ^ (s & kMask)) << 4));
}

// ---- timeline trace ----------------------------------------------------------------------

__device__ __forceinline__ void trace_stamp(const PartialParams& p, int slot) {
  if (p.trace) p.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + slot] = global_ns();
}

// ---- kernel prologue ----------------------------------------------------------------------
//
// The kernels are launched as programmatic dependents: the plan's records may
// be read while the preceding kernel of the stream still runs, device inputs
// (Q, K/V, page tables, lists) and the workspace only after griddepcontrol.wait.

// Copies the CTA's records into shared memory; nonzero when some record
// needs device inputs to complete (index lists, cache rows, page bounds the
// plan lacks) or the CTA has more records than the cache holds.
__device__ __forceinline__ int fill_item_cache(const PartialParams& p, ItemRec* cache, int it_begin, int it_end) {
  int incomplete = it_end - it_begin > kItemCache;
  for (int i = threadIdx.x; i < min(it_end - it_begin, kItemCache); i += blockDim.x) {
    cache[i] = ld_rec_keep(p.cta_recs + it_begin + i, policy_evict_last());
    incomplete |= !rec_complete_as_planned(p, cache[i]);
  }
  return incomplete;
}

// The whole CTA waits for the preceding grid and completes the records.
__device__ __forceinline__ void complete_item_cache(const PartialParams& p, ItemRec* cache, int it_begin,
                                                    int it_end) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < min(it_end - it_begin, kItemCache); i += blockDim.x)
    if (!rec_complete_as_planned(p, cache[i])) cache[i] = complete_rec(p, cache[i], true);
  __syncthreads();
}

// A warp's own wait, just before its first device read, when the CTA did not
// wait as a whole.
__device__ __forceinline__ void dependency_wait(bool needed) {
  if (needed) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- producer ---------------------------------------------------------------------------

// A producer warp's position: stream keys [j0, j1) of item ii (ii == end:
// none), in stages of KS keys.
struct PCur {
  int ii, j0, j1;
};

template <int KS>
__device__ __forceinline__ void pc_seek(const Walk& w, PCur& c) {
  for (; c.ii < w.end; ++c.ii) {
    const WorkItem it = w.rec(c.ii).it;
    if (it.e > it.a) {
      c.j0 = it.a;
      c.j1 = min(it.a + KS, it.e);
      return;
    }
  }
}

template <int KS>
__device__ __forceinline__ void pc_advance(const Walk& w, PCur& c, int n) {
  for (int i = 0; i < n && c.ii < w.end; ++i) {
    const int e = w.rec(c.ii).it.e;
    if (c.j1 < e) {
      c.j0 = c.j1;
      c.j1 = min(c.j0 + KS, e);
    } else {
      ++c.ii;
      pc_seek<KS>(w, c);
    }
  }
}

// The description of a stage of 32 S slots is built in three steps, each
// issued one stage of the warp ahead of the next, so no load result is
// awaited right after it was issued: logical keys (index-list entries are
// loads), page ids of the keys' blocks (page-list loads, M4.5 §0x04D), and
// finally the checked K/V row of every slot.  Lane l describes slots
// l, l + 32, ..., l + 32 (S - 1).
template <int S>
struct SlotKeys {
  int t[S];      // logical key (-1: none)
  bool bad;      // index lists: the group's device list bounds disagree with the plan
};
template <int S, bool FM = false>
struct SlotPages {
  int pi[S];     // page id of the key's block (-2: block outside the page list)
  int4 iv[S];    // FlashMask: the key column's (UTS, UTE, LTS, LTE), used a stage later
};
template <int S>
struct SlotPages<S, false> {
  int pi[S];
};
template <int S, bool FM = false>
struct SlotRows {
  int t[S];           // logical key, -1 when the slot is empty or invalid
  uint32_t row[S];    // K/V row in the cache in rows of d elements (kNoRow: none)
  uint32_t vis[S];    // FlashMask: bit i set when query row i sees the key
  bool full;          // FULL stage class
};
template <int S>
struct SlotRows<S, false> {
  int t[S];
  uint32_t row[S];
  bool full;
};

// Bits [a, b) of a 32-bit row mask (clipped to [0, 32)).
__device__ __forceinline__ uint32_t row_bits(int a, int b) {
  auto below = [](int x) { return x <= 0 ? 0u : x >= 32 ? 0xFFFFFFFFu : (1u << x) - 1u; };
  return b > a ? below(b) & ~below(a) : 0u;
}

// Index lists: the entries are read at the planned offsets, and the group's
// device list bounds beside them, without waiting for either (so the next
// stages' loads are issued at once); when the bounds disagree with the plan,
// slot_rows drops every key of the stage and the status word says why, so the
// consumers see only masked slots.  LIST = false: the caller never runs an
// index-list program (FlashMask producers), and none of this is compiled.
template <int S, bool LIST = true>
__device__ __forceinline__ SlotKeys<S> slot_keys(const Walk& w, const PCur& c, int lane) {
  SlotKeys<S> k;
  k.bad = false;
#pragma unroll
  for (int h = 0; h < S; ++h) k.t[h] = -1;
  if (c.ii >= w.end) return k;
  const WorkItem it = w.rec(c.ii).it;
#pragma unroll
  for (int h = 0; h < S; ++h) {
    const int j = c.j0 + lane + 32 * h;
    if (j < c.j1) k.t[h] = stream_key(it, w.p.mask, w.p.index_list, j);
  }
  if (LIST && w.p.mask == DATTN_MASK_INDEX_LIST) {
    const int g = it.b * w.p.H_kv + it.h;
    const int lo = w.p.index_indptr[g], n = w.p.index_indptr[g + 1] - lo;
    k.bad = lo != it.x0 || it.e > n;
  }
  return k;
}

// ---- L2 prefetch before the wait for the preceding grid ----------------------------------
// A producer warp, before that wait, puts the K/V rows of its first stages into
// L2, so that DRAM works while that grid ends and the stages' copies after the
// wait hit L2: page-run stages (two per warp, a bulk prefetch per page and
// operand) and the first stage of an index list (line hints per lone row).
// Stages of arithmetic keys described slot by slot (FlashMask, contiguous
// caches) are not prefetched: their page-id loads before the wait delayed the
// wait by more than the prefetch won.  Device inputs (page ids, list entries)
// are read here without ordering against that grid and past L1: a stale value
// only prefetches another row of the cache (values outside it are skipped),
// and the stages' own values are loaded after the wait.  Nothing read here
// decides a result.

__device__ __forceinline__ int ld_hint(const int* p) {
  int v;
  asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void prefetch_l2(const char* a, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(bytes) : "memory");
}

// A key's prefetch in two steps, so that all of a warp's page-id loads are in
// flight before its first prefetch needs one: hint_key issues the load,
// hint_row turns the value into the key's K/V row (kNoRow: none; the
// packed-row layout is not prefetched).
struct HintKey {
  int t, pid;
  bool ok;
};

__device__ __forceinline__ HintKey hint_key(const PartialParams& p, const ItemRec& r, int t) {
  HintKey h{t, 0, false};
  if (t < 0 || t >= r.it.T) return h;
  if (p.layout == DATTN_KV_PAGED_HND) {
    const int blk = blk_of(p, t);
    if (blk >= r.hi - r.lo) return h;
    h.pid = ld_hint(p.page_indices + r.lo + blk);
    h.ok = true;
  } else if (p.layout == DATTN_KV_CONTIG_NHD && r.crow >= 0 && t < p.T_cap) {
    h.ok = true;
  }
  return h;
}

__device__ __forceinline__ uint32_t hint_row(const PartialParams& p, const ItemRec& r, const HintKey& h) {
  if (!h.ok) return kNoRow;
  if (p.layout == DATTN_KV_PAGED_HND) {
    if (h.pid < 0 || h.pid >= p.num_pages) return kNoRow;
    return (static_cast<uint32_t>(h.pid) * p.H_kv + r.it.h) * p.P + row_of(p, h.t);
  }
  return (static_cast<uint32_t>(r.crow) * p.T_cap + h.t) * p.H_kv + r.it.h;
}

// One key row: a line hint per 128 bytes (a bulk prefetch per lone row costs
// more issue than the rows are worth).
__device__ __forceinline__ void prefetch_row(const char* kbase, const char* vbase, uint32_t row, uint32_t row_bytes) {
  if (row == kNoRow) return;
  const char* k = kbase + static_cast<size_t>(row) * row_bytes;
  const char* v = vbase + static_cast<size_t>(row) * row_bytes;
  for (uint32_t o = 0; o < row_bytes; o += 128) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(k + o) : "memory");
    asm volatile("prefetch.global.L2 [%0];" ::"l"(v + o) : "memory");
  }
}

// Index lists: a producer warp's first keys are list entries, device inputs.
// Their lines, the group's list bounds and the request's page-table lines are
// prefetched into L2 (plan addresses only), then the warp waits for the
// preceding grid before slot_keys reads them.  With row_bytes > 0 the K/V rows
// of the first stage's keys (S per lane) are prefetched too, from list entries
// and page ids read as hints.  No-op for the other programs, whose keys are
// arithmetic.
template <int S = 2>
__device__ __forceinline__ void index_list_prologue(const Walk& w, const PCur& c0, int lane, bool dep_wait,
                                                    const char* kbase = nullptr, const char* vbase = nullptr,
                                                    uint32_t row_bytes = 0) {
  const PartialParams& p = w.p;
  if (p.mask != DATTN_MASK_INDEX_LIST) return;
  if (c0.ii < w.end) {
    const ItemRec r = w.rec(c0.ii);
    if (dep_wait && row_bytes) {   // entries, then page ids, then rows: each step's loads together
      int t[S];
      HintKey hk[S];
#pragma unroll
      for (int h = 0; h < S; ++h) {
        const int j = c0.j0 + lane + 32 * h;
        t[h] = j < c0.j1 ? ld_hint(p.index_list + r.it.x0 + j) : -1;
      }
#pragma unroll
      for (int h = 0; h < S; ++h) hk[h] = hint_key(p, r, t[h]);
#pragma unroll
      for (int h = 0; h < S; ++h) prefetch_row(kbase, vbase, hint_row(p, r, hk[h]), row_bytes);
    }
    const int j = c0.j0 + 32 * lane;                         // 32 entries (one line) per lane
    if (j < r.it.e) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.index_list + r.it.x0 + j));
    if (lane == 0)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p.index_indptr + r.it.b * p.H_kv + r.it.h));
    if (p.layout == DATTN_KV_PAGED_HND && r.lo >= 0) {
      for (int e = r.lo + 32 * lane; e < r.hi && e < r.lo + 2048; e += 32 * 32)
        asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p.page_indices + e));
    }
  }
  dependency_wait(dep_wait);
}

template <int S, bool FM = false>
__device__ __forceinline__ SlotPages<S, FM> slot_pages(const Walk& w, const PCur& c, const SlotKeys<S>& k) {
  SlotPages<S, FM> g;
#pragma unroll
  for (int h = 0; h < S; ++h) g.pi[h] = -2;
  if constexpr (FM) {
#pragma unroll
    for (int h = 0; h < S; ++h) g.iv[h] = make_int4(0, 0, 0, 0);
  }
  if (c.ii >= w.end) return g;
  const ItemRec r = w.rec(c.ii);
  if constexpr (FM) {   // the column intervals travel with the page ids (not awaited here)
#pragma unroll
    for (int h = 0; h < S; ++h) {
      const int t = k.t[h];
      if (t >= 0 && t < r.it.T) g.iv[h] = *reinterpret_cast<const int4*>(w.p.fm_intervals + 4ll * (r.it.x1 + t));
    }
  }
  if (w.p.layout != DATTN_KV_PAGED_HND) return g;
#pragma unroll
  for (int h = 0; h < S; ++h) {
    const int t = k.t[h];
    if (t >= 0 && t < r.it.T) {
      const int blk = blk_of(w.p, t);
      if (blk < r.hi - r.lo) g.pi[h] = ld_keep(w.p.page_indices + r.lo + blk, w.keep);
    }
  }
  return g;
}

// PACKED: the kernel may see the packed-row layout (bf16 only; the planner
// rejects it for the other formats, whose producers are compiled without it).
template <int S, bool FM = false, bool PACKED = false>
__device__ __forceinline__ SlotRows<S, FM> slot_rows(const Walk& w, const PCur& c, const SlotKeys<S>& k,
                                                     const SlotPages<S, FM>& g, int lane) {
  const PartialParams& p = w.p;
  SlotRows<S, FM> d;
#pragma unroll
  for (int h = 0; h < S; ++h) {
    d.t[h] = -1;
    d.row[h] = kNoRow;
    if constexpr (FM) d.vis[h] = 0u;
  }
  d.full = false;
  if (c.ii >= w.end) return d;
  const ItemRec r = w.rec(c.ii);
  if (k.bad && lane == 0) atomicOr(p.status, kStListRange);
  int tmax = -1;
#pragma unroll
  for (int h = 0; h < S; ++h) {
    int t = k.bad ? -1 : k.t[h];
    uint32_t row = kNoRow;
    if (p.mask == DATTN_MASK_INDEX_LIST && c.j0 + lane + 32 * h < c.j1 && (t < 0 || t >= r.it.T)) {
      atomicOr(p.status, kStListRange);
      t = -1;
    }
    if constexpr (FM) {   // a column hidden from every query row is never loaded
      const uint32_t rows = row_bits(0, r.nq);
      d.vis[h] = t >= 0 ? rows & ~(row_bits(g.iv[h].x, g.iv[h].y) | row_bits(g.iv[h].z, g.iv[h].w)) : 0u;
      if (d.vis[h] == 0u) t = -1;
    }
    if (t >= 0) {
      if (p.layout == DATTN_KV_PAGED_HND) {
        const int pi = g.pi[h];
        if (pi == -2) atomicOr(p.status, kStBlockRange);
        else if (pi < 0 || pi >= p.num_pages) atomicOr(p.status, kStPageRange);
        else row = (static_cast<uint32_t>(pi) * p.H_kv + r.it.h) * p.P + row_of(p, t);
      } else if (PACKED && p.layout == DATTN_KV_PACKED_ROWS) {
        // packed view: list entry x0 + j is packed row x0 + j (its position t only masks)
        row = static_cast<uint32_t>(r.it.x0 + c.j0 + lane + 32 * h);
      } else if (r.crow >= 0 && t < p.T_cap) {
        row = (static_cast<uint32_t>(r.crow) * p.T_cap + t) * p.H_kv + r.it.h;
      } else {
        atomicOr(p.status, kStRowRange);
      }
      if (row == kNoRow) t = -1;
    }
    d.t[h] = t;
    d.row[h] = row;
    tmax = max(tmax, t);
  }
  if constexpr (FM) {   // FULL: every slot of the stage holds a key that every row sees
    bool all = true;
#pragma unroll
    for (int h = 0; h < S; ++h)
      if (c.j0 + lane + 32 * h < c.j1) all = all && d.vis[h] == row_bits(0, r.nq);
    d.full = __all_sync(kAll, all);
  } else {
    // list bounds that disagree with the plan drop every key of the stage, which must
    // then stay masked: only the consumers' per-key path does that
    d.full = stage_is_full(p, r.it, r.nq, c.j0, c.j1, tmax, -1) && !k.bad;
  }
  return d;
}

// Page-run stage description (interval visibility programs on a paged cache
// whose P is a power of two with KS / P + 4 <= 32, see runs_apply).  A stage's
// positions are at most two runs of consecutive keys, so instead of describing
// its KS keys one by one (key, page id, row per slot) a producer loads one
// page id per lane (the pages the runs touch) a stage ahead and derives each
// slot's key and row from its position and a shuffle of its page's id.
struct RunStage {
  int ii;              // item of the stage (w.end: none)
  int p0, n1, q0, n2;  // slots [0, n1) hold keys p0 + s; slots [n1, n1 + n2) keys q0 + s - n1
  int b1, np1, b2;     // first logical block of each run; run 1's pages are lanes [0, np1)
  bool full;
};

__device__ __forceinline__ RunStage run_stage(const Walk& w, const PCur& c) {
  RunStage r{};
  r.ii = c.ii;
  if (c.ii >= w.end) return r;
  const ItemRec rec = w.rec(c.ii);
  Run a, b;
  const int n = item_runs(rec.it, c.j0, c.j1, a, b);
  const int ps = w.p.P_shift;
  r.p0 = a.p0;
  r.n1 = n > 0 ? a.p1 - a.p0 : 0;
  r.q0 = b.p0;
  r.n2 = n > 1 ? b.p1 - b.p0 : 0;
  r.b1 = r.p0 >> ps;
  r.np1 = r.n1 ? ((r.p0 + r.n1 - 1) >> ps) - r.b1 + 1 : 0;
  r.b2 = r.q0 >> ps;
  r.full = stage_is_full(w.p, rec.it, rec.nq, c.j0, c.j1, -1, -1);
  return r;
}

// The lane's page id for stage r, its load issued without waiting for it: the
// value is checked (check_stage_page) when the stage is described, a stage
// later, so that the load's latency overlaps the previous stage.  state: 0
// loaded, 1 the lane holds none, 2 the block lies outside the request's page
// list (reported).
struct StagePage {
  int pid, state;
};

__device__ __forceinline__ StagePage run_stage_page(const Walk& w, const RunStage& r, int lane) {
  if (r.ii >= w.end) return {0, 1};
  const PartialParams& p = w.p;
  const ItemRec rec = w.rec(r.ii);
  const int np2 = r.n2 ? ((r.q0 + r.n2 - 1) >> p.P_shift) - r.b2 + 1 : 0;
  int blk;
  if (lane < r.np1) blk = r.b1 + lane;
  else if (lane < r.np1 + np2) blk = r.b2 + (lane - r.np1);
  else return {0, 1};
  if (blk >= rec.hi - rec.lo) {
    atomicOr(p.status, kStBlockRange);
    return {0, 2};
  }
  return {ld_keep(p.page_indices + rec.lo + blk, w.keep), 0};
}

// The K/V rows of a page-run stage, one range per page and operand, in two
// steps like hint_key / hint_row: run_hint loads the lane's page id, and
// prefetch_run issues its ranges.
struct RunHint {
  int pid, row0, n;   // the page, its first row in the stage's keys and their count (n = 0: none)
  int h;
};

__device__ __forceinline__ RunHint run_hint(const Walk& w, const RunStage& r, int lane) {
  RunHint g{0, 0, 0, 0};
  if (r.ii >= w.end) return g;
  const PartialParams& p = w.p;
  const ItemRec rec = w.rec(r.ii);
  const int np2 = r.n2 ? ((r.q0 + r.n2 - 1) >> p.P_shift) - r.b2 + 1 : 0;
  int blk, t0, t1;   // the lane's page and the stage's keys [t0, t1) in its run
  if (lane < r.np1) {
    blk = r.b1 + lane;
    t0 = r.p0;
    t1 = r.p0 + r.n1;
  } else if (lane < r.np1 + np2) {
    blk = r.b2 + (lane - r.np1);
    t0 = r.q0;
    t1 = r.q0 + r.n2;
  } else {
    return g;
  }
  if (blk >= rec.hi - rec.lo) return g;
  t0 = max(t0, blk << p.P_shift);
  t1 = min(min(t1, (blk + 1) << p.P_shift), rec.it.T);
  if (t1 <= t0) return g;
  g.pid = ld_hint(p.page_indices + rec.lo + blk);
  g.row0 = t0 & (p.P - 1);
  g.n = t1 - t0;
  g.h = rec.it.h;
  return g;
}

__device__ __forceinline__ void prefetch_run(const PartialParams& p, const RunHint& g, const char* kbase,
                                             const char* vbase, uint32_t row_bytes) {
  if (g.n == 0 || g.pid < 0 || g.pid >= p.num_pages) return;
  const size_t off = ((static_cast<size_t>(g.pid) * p.H_kv + g.h) * p.P + g.row0) * row_bytes;
  const uint32_t bytes = static_cast<uint32_t>(g.n) * row_bytes;
  prefetch_l2(kbase + off, bytes);
  prefetch_l2(vbase + off, bytes);
}

// The page id as run_slot takes it: -1 the lane holds none, -2 invalid (reported).
__device__ __forceinline__ int check_stage_page(const PartialParams& p, const StagePage& g) {
  if (g.state == 1) return -1;
  if (g.state == 2) return -2;
  if (g.pid < 0 || g.pid >= p.num_pages) {
    atomicOr(p.status, kStPageRange);
    return -2;
  }
  return g.pid;
}

// Key (-1: none) and K/V row (kNoRow: none) of slot s of stage r; every lane
// of the warp calls it (the page id comes by shuffle from its lane).
__device__ __forceinline__ void run_slot(const PartialParams& p, const RunStage& r, int T, int h, int pid_lane,
                                         int s, int& t, uint32_t& row) {
  int pl = 0;
  t = -1;
  if (s < r.n1) {
    t = r.p0 + s;
    pl = (t >> p.P_shift) - r.b1;
  } else if (s < r.n1 + r.n2) {
    t = r.q0 + (s - r.n1);
    pl = r.np1 + (t >> p.P_shift) - r.b2;
  }
  const int pid = __shfl_sync(kAll, pid_lane, pl & 31);
  if (t < 0 || t >= T || pid < 0) {
    t = -1;
    row = kNoRow;
    return;
  }
  row = (static_cast<uint32_t>(pid) * p.H_kv + h) * p.P + (t & (p.P - 1));
}

// Whether stages of KS keys can use the page-run description.
template <int KS>
__device__ __forceinline__ bool runs_apply(const PartialParams& p) {
  return p.layout == DATTN_KV_PAGED_HND && p.P_shift >= 0 && (KS >> p.P_shift) + 4 <= 32 &&
         (p.mask == DATTN_MASK_CAUSAL || p.mask == DATTN_MASK_SINK_WINDOW);
}

}  // namespace

}  // namespace dattn
