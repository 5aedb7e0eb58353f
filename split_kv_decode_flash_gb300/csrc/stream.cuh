// Walking a CTA's work items stage by stage: the cursor over (item, stage),
// the mapping of stream positions to logical keys and the FULL / PARTIAL
// class of a stage.  Shared by the partial kernels of every K/V format.
#pragma once

#include <climits>

#include "device.cuh"

namespace dattn {

constexpr int kFlagFull = 1, kFlagResidual = 2;

__host__ __device__ constexpr int align16(int x) { return (x + 15) / 16 * 16; }

__device__ __forceinline__ int kivi_prefix(int T, int G, int R) { return T > R ? (T - R + G - 1) / G * G : 0; }

// Stream index where KIVI residual keys begin (INT_MAX for other formats).
__device__ __forceinline__ int residual_start(const PartialParams& p, const WorkItem& it) {
  if (p.fmt != DATTN_FMT_INT4_KIVI) return INT_MAX;
  const int nq = kivi_prefix(it.T, p.kivi_G, p.kivi_R);
  return nq <= it.x0 ? nq : it.x0 + max(0, nq - it.x1);
}

// End of the stage that starts at stream index j0 (a stage never straddles
// the start of the residual keys).
__device__ __forceinline__ int stage_end(const WorkItem& it, int j0, int jq) {
  int j1 = min(j0 + kTK, it.e);
  if (j0 < jq) j1 = min(j1, jq);
  return j1;
}

struct Run {
  int p0, p1;
};

// Position runs of stream [j0, j1) of an interval item (at most two).
__device__ __forceinline__ int item_runs(const WorkItem& it, int j0, int j1, Run& r0, Run& r1) {
  int n = 0;
  Run a{0, 0}, b{0, 0};
  if (j0 < it.x0) a = Run{j0, min(j1, it.x0)}, n = 1;
  if (j1 > it.x0) {
    const int s = max(j0, it.x0);
    const Run x{it.x1 + (s - it.x0), it.x1 + (j1 - it.x0)};
    if (n == 0) a = x; else b = x;
    ++n;
  }
  r0 = a;
  r1 = b;
  return n;
}

// Logical block and page row of key t (shifts when P is a power of two).
__device__ __forceinline__ int blk_of(const PartialParams& p, int t) { return p.P_shift >= 0 ? t >> p.P_shift : t / p.P; }
__device__ __forceinline__ int row_of(const PartialParams& p, int t) {
  return p.P_shift >= 0 ? t & (p.P - 1) : t % p.P;
}

// Reads work item "idx" and, for index lists, drops its keys when the list
// offsets disagree with the plan (the producer and the consumers both apply it).
__device__ __forceinline__ WorkItem read_item(const PartialParams& p, int idx, bool report) {
  WorkItem it = p.items[idx];
  if (p.mask == DATTN_MASK_INDEX_LIST) {
    const int g = it.b * p.H_kv + it.h;
    const int lo = p.index_indptr[g], n = p.index_indptr[g + 1] - lo;
    if (lo != it.x0 || it.e > n) {
      if (report) atomicOr(p.status, kStListRange);
      it.e = it.a;
    }
  }
  return it;
}

// ---- producer cursor over (item, stage) ---------------------------------------------

struct Cursor {
  int ii;           // position in the CTA's item list
  WorkItem it;
  int jq, lo, hi, crow;
  int j0, j1;
  bool valid;
};

__device__ __forceinline__ void load_item(const PartialParams& p, Cursor& c, int lane) {
  c.it = read_item(p, p.cta_items[c.ii], lane == 0);
  c.jq = residual_start(p, c.it);
  c.lo = c.hi = c.crow = 0;
  if (p.layout == DATTN_KV_PAGED_HND) {
    c.lo = p.page_indptr[c.it.b];
    c.hi = p.page_indptr[c.it.b + 1];
  } else {
    c.crow = cache_row(p.cache_batch_idx, c.it.b, p.B_cache, lane == 0 ? p.status : nullptr);
  }
}

// First stage at or after item position ii whose item has keys.
__device__ __forceinline__ void seek(const PartialParams& p, Cursor& c, int it_end, int lane) {
  c.valid = false;
  for (; c.ii < it_end; ++c.ii) {
    load_item(p, c, lane);
    if (c.it.e > c.it.a) {
      c.j0 = c.it.a;
      c.j1 = stage_end(c.it, c.j0, c.jq);
      c.valid = true;
      return;
    }
  }
}

__device__ __forceinline__ void advance(const PartialParams& p, Cursor& c, int it_end, int lane) {
  if (!c.valid) return;
  if (c.j1 < c.it.e) {
    c.j0 = c.j1;
    c.j1 = stage_end(c.it, c.j0, c.jq);
    return;
  }
  ++c.ii;
  seek(p, c, it_end, lane);
}

// FULL when every one of the request's S_q query rows sees every key of stream
// [j0, j1) of item "it" (M4.5 §0x05C); the consumers then skip the per-element
// predicate.  For index lists the keys are the lane's two slot keys t0, t1 (-1
// when empty): the stage is FULL when the largest listed key is visible to the
// first (most restricted) row.  Called by all 32 lanes of a warp.
__device__ __forceinline__ bool stage_is_full(const PartialParams& p, const WorkItem& it, int S_q, int j0, int j1,
                                              int t0, int t1) {
  const MaskCtx mc{p.mask, S_q, it.T, p.n_sink, p.window};
  if (p.mask == DATTN_MASK_INDEX_LIST) {
    int mx = max(t0, t1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    return mx < frontier(mc, 0);
  }
  Run r0, r1;
  const int nr = item_runs(it, j0, j1, r0, r1);
  bool full = true;
  for (int i = 0; i < S_q && full; ++i) {
    if (nr > 0 && visible_in_run(mc, i, r0.p0, r0.p1) != r0.p1 - r0.p0) full = false;
    if (nr > 1 && visible_in_run(mc, i, r1.p0, r1.p1) != r1.p1 - r1.p0) full = false;
  }
  return full;
}

}  // namespace dattn
