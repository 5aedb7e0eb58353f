// Device layer of libdattn: mbarrier / bulk-copy primitives, the K/V address
// translator and the visibility predicates.  Every kernel and every debug hook
// uses these same functions, so the debug hooks observe exactly what the
// kernels do.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "internal.h"

namespace dattn {

// ---- shared-memory barriers and bulk copies (TMA engine) ---------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait.  The thread sleeps inside try_wait (hardware suspend, woken
// by the phase completing) instead of spinning, so waiting warps leave the
// issue slots to working ones.  After the CTA's wait limit of wall time (2 s
// unless the caller set another; a uint64 of ns kept 8 bytes after the abort
// flag, read only on this slow path) it raises the abort flag and the timeout
// status bit, so that every warp of the CTA stops.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((it & 7u) == 7u) {
      if (*abort_flag) return false;
      const uint64_t limit_ns =
          *reinterpret_cast<const volatile unsigned long long*>(reinterpret_cast<const volatile char*>(abort_flag) + 8);
      if (global_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStTimeout);
        return false;
      }
    }
  }
}

// One bulk global->shared copy; completion is counted in bytes on "bar".
// src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- visibility programs (M4.5 §0x05A, §0x08B; M5.4 §0x04-§0x05) --------------------

// 2^x with the hardware's approximate exponential (PTX ex2.approx.ftz.f32:
// relative error about 2^-22, -inf gives +0, results below 2^-126 flush to
// zero).  The softmax weights it produces are summed in fp32 and cast to
// f16 / bf16 for the P.V product, far coarser than its error.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct MaskCtx {
  int mask, S_q, T, n_sink, window;
};

// Frontier of query row i: F_i = max(0, min(T, T - S_q + i + 1)).
__device__ __forceinline__ int frontier(const MaskCtx& m, int i) {
  return max(0, min(m.T, m.T - m.S_q + i + 1));
}

__device__ __forceinline__ int overlap(int a0, int a1, int b0, int b1) {
  return max(0, min(a1, b1) - max(a0, b0));
}

// Is key t visible to query row i?  For index lists, t is a listed key and
// only the causal frontier applies.
__device__ __forceinline__ bool key_visible(const MaskCtx& m, int i, int t) {
  const int F = frontier(m, i);
  if (t < 0 || t >= F) return false;
  if (m.mask == DATTN_MASK_SINK_WINDOW) return t < min(m.n_sink, F) || t >= F - m.window;
  return true;
}

// Number of keys of [x0, x1) visible to row i under an interval program.
__device__ __forceinline__ int visible_in_run(const MaskCtx& m, int i, int x0, int x1) {
  const int F = frontier(m, i);
  if (m.mask == DATTN_MASK_SINK_WINDOW) {
    const int s = min(m.n_sink, F), w = max(0, F - m.window);
    return overlap(x0, x1, 0, s) + overlap(x0, x1, w, F) - overlap(x0, x1, w, s);
  }
  return overlap(x0, x1, 0, F);
}

// Number of entries of the sorted list L[0, n) inside [x0, x1).
__device__ __forceinline__ int count_in_sorted(const int32_t* L, int n, int x0, int x1) {
  auto lower = [&](int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (L[mid] < x) lo = mid + 1; else hi = mid;
    }
    return lo;
  };
  return x1 > x0 ? lower(x1) - lower(x0) : 0;
}

// Exact class of "every query row x keys [x0, x1)" (M4.5 §0x05C).
// list/list_n: the group's sorted index list (INDEX_LIST), else unused.
__device__ __forceinline__ int classify_keys(const MaskCtx& m, int x0, int x1, const int32_t* list,
                                             int list_n) {
  long visible = 0;
  for (int i = 0; i < m.S_q; ++i) {
    if (m.mask == DATTN_MASK_INDEX_LIST)
      visible += count_in_sorted(list, list_n, x0, min(x1, frontier(m, i)));
    else
      visible += visible_in_run(m, i, x0, x1);
  }
  const long cells = static_cast<long>(m.S_q) * (x1 - x0);
  if (visible == 0) return DATTN_TILE_SKIP;
  return visible == cells ? DATTN_TILE_FULL : DATTN_TILE_PARTIAL;
}

// ---- visible stream -> logical key (see WorkItem) ----------------------------------

__device__ __forceinline__ int stream_key(const WorkItem& it, int mask, const int32_t* index_list, int j) {
  if (mask == DATTN_MASK_INDEX_LIST) return index_list[it.x0 + j];
  return j < it.x0 ? j : it.x1 + (j - it.x0);
}

// ---- address translation (M4.5 §0x04B-§0x04F) ----------------------------------------

// Physical page of request b's logical block j, or -1 (with a status bit) when
// the block is outside the request's page list or the page outside the pool.
__device__ __forceinline__ int page_of(const int32_t* page_indptr, const int32_t* page_indices, int b,
                                       int j, int num_pages, int32_t* status) {
  const int lo = page_indptr[b], hi = page_indptr[b + 1];
  if (j < 0 || lo + j >= hi) {
    if (status) atomicOr(status, kStBlockRange);
    return -1;
  }
  const int pi = page_indices[lo + j];
  if (pi < 0 || pi >= num_pages) {
    if (status) atomicOr(status, kStPageRange);
    return -1;
  }
  return pi;
}

// Element offset of paged HND (pi, r, h, x): ((pi H + h) P + r) d + x.
__device__ __forceinline__ long long paged_hnd_offset(int pi, int r, int h, int x, int P, int H, int d) {
  return ((static_cast<long long>(pi) * H + h) * P + r) * d + x;
}

// Element offset of contiguous NHD (c, t, h, x): ((c T_cap + t) H + h) d + x.
__device__ __forceinline__ long long contig_nhd_offset(int c, int t, int h, int x, int T_cap, int H, int d) {
  return ((static_cast<long long>(c) * T_cap + t) * H + h) * d + x;
}

// Cache row of request b (cache_batch_idx remap, M4.5 §0x04A), or -1.
__device__ __forceinline__ int cache_row(const int32_t* cache_batch_idx, int b, int B_cache, int32_t* status) {
  const int c = cache_batch_idx ? cache_batch_idx[b] : b;
  if (c < 0 || c >= B_cache) {
    if (status) atomicOr(status, kStRowRange);
    return -1;
  }
  return c;
}

// Marks partial-state row "srow" as never written (m = l = NaN): a consumer
// warp whose bounded wait gave up leaves this instead of a state, and the
// merge writes none of the rows that depend on it (fail closed, row by row).
__device__ __forceinline__ void mark_state_unwritten(float2* ml, long long srow) {
  ml[srow] = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
}

// State-row tags (a partial kernel followed by a separate merge kernel): once a
// consumer warp has written (or marked unwritten) every state of its items, a
// __syncwarp and one gpu-scope fence order those writes before the tags, which
// the lanes that wrote the rows' (m, l) then store (relaxed, gpu scope).  The
// merge reads a tag with acquire semantics and folds the state once it carries
// the run's number, so a finished group is merged while the rest of the grid
// still runs.  (A fence per item end instead stalled the consumers: the INT8
// and KIVI steps took 6-9 % longer.)
__device__ __forceinline__ void state_tags_fence() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void store_relaxed_gpu(int32_t* addr, int32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Tags state row "row" of slot "slot" when the row is one of the request's g C_b.
__device__ __forceinline__ void tag_state_row(const PartialParams& p, int slot, int row, int nq) {
  if (row >= 0 && row < p.g * nq) store_relaxed_gpu(p.state_seq + static_cast<long long>(row) * p.n_slots + slot, p.run_seq);
}

__device__ __forceinline__ int32_t load_acquire_gpu(const int32_t* addr) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

// ---- small numeric helpers ------------------------------------------------------------

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace dattn
