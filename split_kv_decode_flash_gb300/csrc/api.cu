// C entry points of libdattn that touch the device: dattn_run,
// dattn_device_status and the bit-exact debug hooks.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <string>

#include "device.cuh"
#include "plan.h"

namespace dattn {

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Pointer checks of one call (the tensor part of the admission vector, M4.5 §0x07B).
void check_tensors(const dattn_problem& p, const dattn_tensors* t, bool need_q_o, Checker& c) {
  if (!t) {
    c.fail(DATTN_EINVAL, "tensors are NULL");
    return;
  }
  if (need_q_o) {
    if (!t->q || !aligned16(t->q)) c.fail(DATTN_EINVAL, "q must be a 16-byte aligned device pointer");
    if (!t->o || !aligned16(t->o)) c.fail(DATTN_EINVAL, "o must be a 16-byte aligned device pointer");
  }
  if (!t->k || !aligned16(t->k)) c.fail(DATTN_EINVAL, "k must be a 16-byte aligned device pointer");
  if (!t->v || !aligned16(t->v)) c.fail(DATTN_EINVAL, "v must be a 16-byte aligned device pointer");
  if (p.layout == DATTN_KV_PAGED_HND && (!t->page_indptr || !t->page_indices))
    c.fail(DATTN_EINVAL, "paged layout needs page_indptr and page_indices");
  if (p.mask == DATTN_MASK_INDEX_LIST && (!t->index_indptr || !t->index_list))
    c.fail(DATTN_EINVAL, "index_list mask needs index_indptr and index_list");
  if (p.mask == DATTN_MASK_FLASHMASK && (!t->fm_intervals || !aligned16(t->fm_intervals)))
    c.fail(DATTN_EINVAL, "flashmask needs 16-byte aligned fm_intervals");
  if (p.fmt == DATTN_FMT_INT8_TOKEN || p.fmt == DATTN_FMT_INT4_KIVI || p.fmt == DATTN_FMT_INT4_HEAD) {
    if (!t->k_qparams || !t->v_qparams || !aligned16(t->k_qparams) || !aligned16(t->v_qparams))
      c.fail(DATTN_EINVAL, "INT8 and INT4 formats need 16-byte aligned k_qparams and v_qparams");
  }
  if ((p.fmt == DATTN_FMT_FP8_E4M3 || p.fmt == DATTN_FMT_FP8_E5M2) &&
      ((reinterpret_cast<uintptr_t>(t->k_qparams) % 4) || (reinterpret_cast<uintptr_t>(t->v_qparams) % 4)))
    c.fail(DATTN_EINVAL, "FP8 scales (k_qparams, v_qparams) must be 4-byte aligned fp32 arrays or NULL");
  if (p.fmt == DATTN_FMT_INT4_KIVI) {
    if (!t->k_residual || !t->v_residual || !aligned16(t->k_residual) || !aligned16(t->v_residual))
      c.fail(DATTN_EINVAL, "INT4 KIVI needs 16-byte aligned k_residual and v_residual");
  }
}

void fill_common(const dattn_problem& p, const dattn_tensors& t, PartialParams& k) {
  std::memset(&k, 0, sizeof(k));
  k.q = t.q;
  k.k = t.k;
  k.v = t.v;
  k.kqp = t.k_qparams;
  k.vqp = t.v_qparams;
  k.kres = t.k_residual;
  k.vres = t.v_residual;
  k.page_indptr = t.page_indptr;
  k.page_indices = t.page_indices;
  k.cache_batch_idx = t.cache_batch_idx;
  k.index_indptr = t.index_indptr;
  k.index_list = t.index_list;
  k.fm_intervals = t.fm_intervals;
  k.o = t.o;
  k.lse = t.lse;
  k.B = p.B;
  k.S_q = p.S_q;
  k.H_q = p.H_q;
  k.H_kv = p.H_kv;
  k.g = p.H_q / p.H_kv;
  k.rows = group_rows(p);
  k.layout = p.layout;
  k.fmt = p.fmt;
  k.mask = p.mask;
  k.P = p.page_size;
  k.P_shift = -1;
  if (p.page_size > 0 && (p.page_size & (p.page_size - 1)) == 0) {
    k.P_shift = 0;
    while ((1 << k.P_shift) < p.page_size) ++k.P_shift;
  }
  k.num_pages = p.num_pages;
  k.T_cap = p.T_cap;
  // the packed-row layout has no cache rows: the kernels' row lookup (identity
  // over the B requests) then passes and is not used
  k.B_cache = p.layout == DATTN_KV_PACKED_ROWS ? p.B : p.B_cache;
  if (p.layout == DATTN_KV_PACKED_ROWS) k.cache_batch_idx = nullptr;
  k.n_sink = p.n_sink;
  k.window = p.window;
  k.kivi_G = p.kivi_group;
  k.kivi_Gv = p.kivi_v_group;
  k.kivi_R = p.kivi_residual;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.f / std::sqrt(static_cast<float>(p.d_h));
  k.scale_log2 = scale * 1.4426950408889634f;
  k.wait_ns = kDefaultWaitNs;
}

dattn_status cuda_fail(const char* where, int err) {
  set_error(std::string(where) + ": CUDA error " + cudaGetErrorString(static_cast<cudaError_t>(err)));
  return DATTN_ECUDA;
}

// ---- debug kernels (same device functions as the partial kernel) ---------------------

__global__ void translate_kernel(PartialParams p, int d, const int32_t* kv_len, const int32_t* coords, int n,
                                 int64_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int b = coords[4 * i], t = coords[4 * i + 1], hq = coords[4 * i + 2], x = coords[4 * i + 3];
  long long off = -1;
  if (b >= 0 && b < p.B && hq >= 0 && hq < p.H_q && x >= 0 && x < d && t >= 0 && t < kv_len[b]) {
    const int h = hq / p.g;
    if (p.layout == DATTN_KV_PAGED_HND) {
      const int pi = page_of(p.page_indptr, p.page_indices, b, t / p.P, p.num_pages, nullptr);
      if (pi >= 0) off = paged_hnd_offset(pi, t % p.P, h, x, p.P, p.H_kv, d);
    } else if (p.layout == DATTN_KV_PACKED_ROWS) {
      // the packed row that holds original position t of slice (b, h), if retained
      const int s = b * p.H_kv + h;
      int lo = p.index_indptr[s], hi = p.index_indptr[s + 1];
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (p.index_list[mid] < t) lo = mid + 1; else hi = mid;
      }
      if (lo < p.index_indptr[s + 1] && p.index_list[lo] == t) off = static_cast<long long>(lo) * d + x;
    } else {
      const int c = cache_row(p.cache_batch_idx, b, p.B_cache, nullptr);
      if (c >= 0 && t < p.T_cap) off = contig_nhd_offset(c, t, h, x, p.T_cap, p.H_kv, d);
    }
  }
  out[i] = off;
}

__global__ void classify_kernel(PartialParams p, const int32_t* kv_len, const int32_t* tiles, int n, int width,
                                int32_t* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int b = tiles[3 * i], h = tiles[3 * i + 1], j = tiles[3 * i + 2];
  if (b < 0 || b >= p.B || h < 0 || h >= p.H_kv || j < 0) {
    out[i] = -1;
    return;
  }
  const MaskCtx mc{p.mask, p.S_q, kv_len[b], p.n_sink, p.window};
  const int32_t* list = nullptr;
  int list_n = 0;
  if (p.mask == DATTN_MASK_INDEX_LIST) {
    const int g = b * p.H_kv + h;
    list = p.index_list + p.index_indptr[g];
    list_n = p.index_indptr[g + 1] - p.index_indptr[g];
  }
  out[i] = classify_keys(mc, j * width, (j + 1) * width, list, list_n);
}

__global__ void gather_kernel(PartialParams p, int item, int out_off, int32_t* out, int capacity) {
  const WorkItem it = p.items[item];
  for (int j = it.a + threadIdx.x; j < it.e; j += blockDim.x) {
    const int o = out_off + (j - it.a);
    if (o < capacity) out[o] = stream_key(it, p.mask, p.index_list, j);
  }
}

// Device pointers of the plan's arrays inside "ws".
void bind_blob(const dattn_plan_t* plan, void* ws, PartialParams& k) {
  const BlobHeader* h = reinterpret_cast<const BlobHeader*>(plan->blob.data());
  uint8_t* base = static_cast<uint8_t*>(ws);
  k.items = reinterpret_cast<const WorkItem*>(base + h->off_items);
  k.cta_indptr = reinterpret_cast<const int32_t*>(base + h->off_cta_indptr);
  k.cta_items = reinterpret_cast<const int32_t*>(base + h->off_cta_items);
  k.cta_recs = reinterpret_cast<const ItemRec*>(base + h->off_cta_recs);
  k.ml = reinterpret_cast<float2*>(base + h->off_ml);
  k.u = reinterpret_cast<float*>(base + h->off_u);
  k.status = reinterpret_cast<int32_t*>(base + offsetof(BlobHeader, status));
  k.groups = reinterpret_cast<const MergeGroup*>(base + h->off_merge);
  k.group_count = reinterpret_cast<int32_t*>(base + h->off_count);
  k.fused = h->fused;
  k.state_seq = h->tags ? reinterpret_cast<int32_t*>(base + h->off_seq) : nullptr;
}

// A tag no earlier run of this process carried (never 0, the uploaded value).
int32_t next_run_seq() {
  static std::atomic<uint32_t> seq{0};
  uint32_t s = seq.fetch_add(1, std::memory_order_relaxed) + 1;
  if (s == 0) s = seq.fetch_add(1, std::memory_order_relaxed) + 1;
  return static_cast<int32_t>(s);
}

dattn_status upload_blob(const dattn_plan_t* plan, void* ws, cudaStream_t s, PartialParams& k) {
  cudaError_t err = cudaMemcpyAsync(ws, plan->blob.data(), plan->blob.size(), cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return cuda_fail("copy of the work list", err);
  bind_blob(plan, ws, k);
  return DATTN_OK;
}

dattn_status check_run_args(const dattn_plan_t* plan, const dattn_problem* prob, const dattn_tensors* t,
                            void* ws, size_t ws_bytes, bool need_q_o, const char* where) {
  Checker c;
  if (!plan) c.fail(DATTN_EINVAL, "plan is NULL");
  check_problem(prob, c);
  if (c.status != DATTN_OK) return c.finish(where);
  if (!same_problem(plan->prob, *prob)) {
    c.fail(DATTN_ESTALE_PLAN, "problem differs from the planned problem");
    c.status = DATTN_ESTALE_PLAN;
    return c.finish(where);
  }
  check_tensors(*prob, t, need_q_o, c);
  if (c.status != DATTN_OK) return c.finish(where);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kWsAlign) ||
      ws_bytes < static_cast<size_t>(plan->info.workspace_bytes)) {
    c.fail(DATTN_EWORKSPACE, "workspace must be 256-byte aligned and hold " +
                                 std::to_string(plan->info.workspace_bytes) + " bytes");
    c.status = DATTN_EWORKSPACE;
    return c.finish(where);
  }
  return DATTN_OK;
}

}  // namespace
}  // namespace dattn

using namespace dattn;

namespace {

dattn_status record(void* const* events, int i, cudaStream_t s) {
  if (!events || !events[i]) return DATTN_OK;
  const cudaError_t err = cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
  return err == cudaSuccess ? DATTN_OK : cuda_fail("dattn_run_with_events", err);
}

dattn_status run_impl(const dattn_plan_t* plan, const dattn_problem* prob, const dattn_tensors* t, void* workspace,
                      size_t workspace_bytes, void* stream, const dattn_run_options* opt, const char* where) {
  const bool shift = opt && (opt->flags & DATTN_RUN_SHARED_SHIFT);
  const bool skip_arrival = opt && (opt->flags & DATTN_RUN_TEST_SKIP_ARRIVAL);
  if (shift) {
    Checker c;
    if (prob && prob->fmt != DATTN_FMT_BF16) c.fail(DATTN_EUNSUPPORTED, "shared-shift partials run on bf16 K/V");
    if (!std::isfinite(opt->shift_phi)) c.fail(DATTN_EINVAL, "shift_phi must be finite");
    if (!(opt->shift_lo >= -80.f && opt->shift_lo < opt->shift_hi && opt->shift_hi <= 40.f))
      c.fail(DATTN_EINVAL, "the guard needs -80 <= shift_lo < shift_hi <= 40");
    if (c.status != DATTN_OK) return c.finish(where);
  }
  if (skip_arrival) {
    Checker c;
    if (prob && prob->fmt != DATTN_FMT_BF16) c.fail(DATTN_EUNSUPPORTED, "the skipped-arrival hook runs on bf16 K/V");
    if (opt->wait_limit_us == 0 || opt->wait_limit_us > 100000u)
      c.fail(DATTN_EINVAL, "the skipped-arrival hook needs a wait limit of 1 .. 100000 us");
    if (c.status != DATTN_OK) return c.finish(where);
  }
  dattn_status st = check_run_args(plan, prob, t, workspace, workspace_bytes, true, where);
  if (st != DATTN_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* const* events = opt ? opt->events : nullptr;
  PartialParams k;
  fill_common(*prob, *t, k);
  if (shift) {
    constexpr float kLog2e = 1.4426950408889634f;
    k.shift_on = 1;
    k.shift_phi2 = opt->shift_phi * kLog2e;
    k.shift_lo2 = opt->shift_lo * kLog2e;
    k.shift_hi2 = opt->shift_hi * kLog2e;
    k.shift_fallbacks = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                                   offsetof(BlobHeader, shift_fallbacks));
  }
  if (opt && opt->wait_limit_us) k.wait_ns = static_cast<uint64_t>(opt->wait_limit_us) * 1000ull;
  k.skip_arrival = skip_arrival ? 1 : 0;
  uint64_t* trace = opt && prob->fmt == DATTN_FMT_BF16 ? static_cast<uint64_t*>(opt->trace) : nullptr;
  k.trace = trace;
  if (opt && (opt->flags & DATTN_RUN_REUSE_UPLOAD)) {
    bind_blob(plan, workspace, k);
  } else {
    st = upload_blob(plan, workspace, s, k);
    if (st != DATTN_OK) return st;
  }
  k.run_seq = next_run_seq();
  k.n_slots = plan->info.n_slots;
  if ((st = record(events, 0, s)) != DATTN_OK) return st;
  if (plan->info.n_ctas > 0) {
    const int err = launch_partial(k, prob->d_h, plan->info.n_ctas, stream);
    if (err != cudaSuccess) return cuda_fail("dattn_run partial kernel", err);
  }
  if ((st = record(events, 1, s)) != DATTN_OK) return st;
  if (plan->info.n_merge_groups > 0 && !plan->info.fused_merge) {
    const BlobHeader* h = reinterpret_cast<const BlobHeader*>(plan->blob.data());
    MergeParams m{};
    m.groups = reinterpret_cast<const MergeGroup*>(static_cast<uint8_t*>(workspace) + h->off_merge);
    m.ml = k.ml;
    m.u = k.u;
    m.o = t->o;
    m.lse = t->lse;
    m.status = k.status;
    m.n_groups = plan->info.n_merge_groups;
    m.rows = k.rows;
    m.g = k.g;
    m.S_q = k.S_q;
    m.H_q = k.H_q;
    m.mean_states = plan->info.n_slots / plan->info.n_merge_groups;
    m.trace = trace ? trace + static_cast<size_t>(plan->info.n_ctas) * kTraceSlots : nullptr;
    // the merge warps wait for their states' tags; the limit only bounds a failure, as a
    // group's states may take the whole partial kernel to complete
    m.state_seq = k.state_seq;
    m.run_seq = k.run_seq;
    m.n_slots = k.n_slots;
    m.end_wait = plan->direct_items > 0 ? 1 : 0;
    m.wait_ns = std::max<uint64_t>(2 * k.wait_ns, 4000000000ull);
    const int err = launch_merge(m, prob->d_h, stream);
    if (err != cudaSuccess) return cuda_fail("dattn_run merge kernel", err);
  }
  return record(events, 2, s);
}

}  // namespace

extern "C" dattn_status dattn_run(const dattn_plan_t* plan, const dattn_problem* prob, const dattn_tensors* t,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return run_impl(plan, prob, t, workspace, workspace_bytes, stream, nullptr, "dattn_run");
}

extern "C" dattn_status dattn_run_ex(const dattn_plan_t* plan, const dattn_problem* prob, const dattn_tensors* t,
                                     void* workspace, size_t workspace_bytes, void* stream,
                                     const dattn_run_options* options) {
  return run_impl(plan, prob, t, workspace, workspace_bytes, stream, options, "dattn_run_ex");
}

extern "C" dattn_status dattn_plan_upload(const dattn_plan_t* plan, void* workspace, size_t workspace_bytes,
                                          void* stream) {
  if (!plan || !workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) ||
      workspace_bytes < static_cast<size_t>(plan->info.workspace_bytes)) {
    set_error("dattn_plan_upload: plan missing or workspace too small / misaligned");
    return plan ? DATTN_EWORKSPACE : DATTN_EINVAL;
  }
  PartialParams k;
  std::memset(&k, 0, sizeof(k));
  return upload_blob(plan, workspace, static_cast<cudaStream_t>(stream), k);
}

extern "C" dattn_status dattn_shift_fallbacks(const void* workspace, int32_t* count, void* stream) {
  if (!workspace || !count) {
    set_error("dattn_shift_fallbacks: NULL argument");
    return DATTN_EINVAL;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(count, static_cast<const uint8_t*>(workspace) + offsetof(BlobHeader, shift_fallbacks),
                                    sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  return err == cudaSuccess ? DATTN_OK : cuda_fail("dattn_shift_fallbacks", err);
}

extern "C" dattn_status dattn_device_status(const void* workspace, int32_t* flags, void* stream) {
  if (!workspace || !flags) {
    set_error("dattn_device_status: NULL argument");
    return DATTN_EINVAL;
  }
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(flags, static_cast<const uint8_t*>(workspace) + offsetof(BlobHeader, status),
                                    sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail("dattn_device_status", err);
  return *flags ? DATTN_EDEVICE_CHECK : DATTN_OK;
}

extern "C" dattn_status dattn_debug_translate(const dattn_problem* prob, const dattn_tensors* t,
                                              const int32_t* kv_len, const int32_t* coords, int32_t n,
                                              int64_t* out, void* stream) {
  Checker c;
  check_problem(prob, c);
  if (c.status == DATTN_OK) check_tensors(*prob, t, false, c);
  if (!kv_len || (n > 0 && (!coords || !out))) c.fail(DATTN_EINVAL, "kv_len, coords and out are required");
  if (n < 0) c.fail(DATTN_EINVAL, "n must be >= 0");
  if (c.status != DATTN_OK) return c.finish("dattn_debug_translate");
  if (n == 0) return DATTN_OK;
  PartialParams k;
  fill_common(*prob, *t, k);
  translate_kernel<<<(n + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(k, prob->d_h, kv_len, coords,
                                                                                   n, out);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? DATTN_OK : cuda_fail("dattn_debug_translate", err);
}

extern "C" dattn_status dattn_debug_classify(const dattn_problem* prob, const dattn_tensors* t,
                                             const int32_t* kv_len, const int32_t* tiles, int32_t n, int32_t* out,
                                             void* stream) {
  Checker c;
  check_problem(prob, c);
  if (c.status == DATTN_OK && prob->page_size < 1) c.fail(DATTN_EINVAL, "classification tiles are page_size keys wide");
  if (!kv_len || (n > 0 && (!tiles || !out))) c.fail(DATTN_EINVAL, "kv_len, tiles and out are required");
  if (c.status == DATTN_OK && prob->mask == DATTN_MASK_INDEX_LIST && (!t || !t->index_indptr || !t->index_list))
    c.fail(DATTN_EINVAL, "index_list mask needs index_indptr and index_list");
  if (c.status == DATTN_OK && prob->mask == DATTN_MASK_FLASHMASK)
    c.fail(DATTN_EUNSUPPORTED, "the tile classifier covers interval programs and index lists");
  if (n < 0) c.fail(DATTN_EINVAL, "n must be >= 0");
  if (c.status != DATTN_OK) return c.finish("dattn_debug_classify");
  if (n == 0) return DATTN_OK;
  PartialParams k;
  dattn_tensors empty{};
  fill_common(*prob, t ? *t : empty, k);
  classify_kernel<<<(n + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(k, kv_len, tiles, n,
                                                                                  prob->page_size, out);
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? DATTN_OK : cuda_fail("dattn_debug_classify", err);
}

extern "C" dattn_status dattn_debug_gather(const dattn_plan_t* plan, const dattn_problem* prob,
                                           const dattn_tensors* t, void* workspace, size_t workspace_bytes,
                                           int32_t b, int32_t h_kv, int32_t* out, int32_t capacity, int32_t* count,
                                           void* stream) {
  Checker c;
  if (!plan) c.fail(DATTN_EINVAL, "plan is NULL");
  check_problem(prob, c);
  if (c.status != DATTN_OK) return c.finish("dattn_debug_gather");
  if (!same_problem(plan->prob, *prob)) {
    c.fail(DATTN_ESTALE_PLAN, "problem differs from the planned problem");
    c.status = DATTN_ESTALE_PLAN;
    return c.finish("dattn_debug_gather");
  }
  if (!count || (capacity > 0 && !out) || b < 0 || b >= prob->B || h_kv < 0 || h_kv >= prob->H_kv)
    c.fail(DATTN_EINVAL, "bad group or output");
  if (prob->mask == DATTN_MASK_INDEX_LIST && (!t || !t->index_list)) c.fail(DATTN_EINVAL, "index_list is required");
  if (prob->mask == DATTN_MASK_FLASHMASK) c.fail(DATTN_EUNSUPPORTED, "the gather covers interval programs and index lists");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) ||
      workspace_bytes < static_cast<size_t>(plan->info.workspace_bytes)) {
    c.fail(DATTN_EWORKSPACE, "workspace too small or misaligned");
  }
  if (c.status != DATTN_OK) return c.finish("dattn_debug_gather");
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  PartialParams k;
  dattn_tensors empty{};
  fill_common(*prob, t ? *t : empty, k);
  dattn_status st = upload_blob(plan, workspace, s, k);
  if (st != DATTN_OK) return st;
  int total = 0;
  for (size_t i = 0; i < plan->items.size(); ++i) {
    const WorkItem& w = plan->items[i];
    if (w.b != b || w.h != h_kv) continue;
    if (w.e > w.a) gather_kernel<<<1, 256, 0, s>>>(k, static_cast<int>(i), total, out, capacity);
    total += w.e - w.a;
  }
  *count = total;
  const cudaError_t err = cudaGetLastError();
  return err == cudaSuccess ? DATTN_OK : cuda_fail("dattn_debug_gather", err);
}

// ---- one step from host memory ---------------------------------------------------------

namespace {

struct StepLayout {
  size_t q_bytes, pi_bytes, px_bytes, o_bytes, lse_bytes;
  size_t pi_off, px_off, plan_off;      // device and staging (inputs, then the work list)
  size_t o_off, lse_off, ws_total;      // device
  size_t o_off_s, staging_total;        // staging: the work list's end, and the size with the outputs
};

size_t align_ws(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

StepLayout step_layout(const dattn_problem& p, long long n_pidx, size_t plan_ws, size_t blob_bytes) {
  StepLayout L{};
  const bool paged = p.layout == DATTN_KV_PAGED_HND;
  const size_t rows = static_cast<size_t>(p.B) * p.S_q * p.H_q;
  L.q_bytes = rows * p.d_h * 2;
  L.pi_bytes = paged ? static_cast<size_t>(p.B + 1) * 4 : 0;
  L.px_bytes = paged ? static_cast<size_t>(n_pidx) * 4 : 0;
  L.o_bytes = rows * p.d_h * 2;
  L.lse_bytes = rows * 4;
  L.pi_off = align_ws(L.q_bytes);
  L.px_off = L.pi_off + align_ws(L.pi_bytes);
  L.plan_off = L.px_off + align_ws(L.px_bytes);
  L.o_off = L.plan_off + align_ws(plan_ws);
  L.lse_off = L.o_off + align_ws(L.o_bytes);
  L.ws_total = L.lse_off + align_ws(L.lse_bytes);
  L.o_off_s = L.plan_off + align_ws(blob_bytes);
  L.staging_total = L.o_off_s + align_ws(L.o_bytes) + align_ws(L.lse_bytes);
  return L;
}

dattn_status check_step(const dattn_problem* prob, const dattn_host_step* io, bool need_io_arrays,
                        const char* where) {
  Checker c;
  check_problem(prob, c);
  if (!io) c.fail(DATTN_EINVAL, "io is NULL");
  if (c.status != DATTN_OK) return c.finish(where);
  if (prob->mask != DATTN_MASK_CAUSAL && prob->mask != DATTN_MASK_SINK_WINDOW)
    c.fail(DATTN_EUNSUPPORTED, "index-list and flashmask programs read device lists: use dattn_run");
  if (!io->kv_len) c.fail(DATTN_EINVAL, "kv_len is required");
  if (io->num_sms < 1) c.fail(DATTN_EINVAL, "num_sms must be >= 1");
  if (prob->layout == DATTN_KV_PAGED_HND && (!io->page_indptr || !io->page_indices))
    c.fail(DATTN_EINVAL, "paged layout needs host page_indptr and page_indices");
  if (need_io_arrays && (!io->q || !io->o)) c.fail(DATTN_EINVAL, "host q and o are required");
  return c.finish(where);
}

// Plans the step; on success *plan is owned by the caller.
dattn_status plan_step(const dattn_problem* prob, const dattn_host_step* io, dattn_plan_t** plan, size_t* plan_ws) {
  dattn_plan_inputs in{};
  in.kv_len = io->kv_len;
  in.page_indptr = prob->layout == DATTN_KV_PAGED_HND ? io->page_indptr : nullptr;
  in.num_sms = io->num_sms;
  return dattn_plan(prob, &in, plan, plan_ws);
}

long long page_entries(const dattn_problem* prob, const dattn_host_step* io) {
  return prob->layout == DATTN_KV_PAGED_HND ? io->page_indptr[prob->B] : 0;
}

}  // namespace

extern "C" dattn_status dattn_step_host_sizes(const dattn_problem* prob, const dattn_host_step* io,
                                              size_t* workspace_bytes, size_t* staging_bytes) {
  dattn_status st = check_step(prob, io, false, "dattn_step_host_sizes");
  if (st != DATTN_OK) return st;
  if (!workspace_bytes || !staging_bytes) {
    set_error("dattn_step_host_sizes: NULL output");
    return DATTN_EINVAL;
  }
  dattn_plan_t* plan = nullptr;
  size_t plan_ws = 0;
  if ((st = plan_step(prob, io, &plan, &plan_ws)) != DATTN_OK) return st;
  const StepLayout L = step_layout(*prob, page_entries(prob, io), plan_ws, plan->blob.size());
  dattn_plan_destroy(plan);
  *workspace_bytes = L.ws_total;
  *staging_bytes = L.staging_total;
  return DATTN_OK;
}

namespace {

// Where O and LSE come back in the staging buffer: its last
// align_ws(o) + align_ws(lse) bytes (a fixed place, so that the step's finish
// finds them without the plan).
size_t staging_out_off(const StepLayout& L, size_t staging_bytes) {
  const size_t out = align_ws(L.o_bytes) + align_ws(L.lse_bytes);
  return staging_bytes >= out ? (staging_bytes - out) / 16 * 16 : 0;
}

// cp (optional): the transfers go on cp's two streams, ordered against the kernels
// on "stream" by events, so that they overlap the kernels of the neighbouring steps.
dattn_status step_submit(const dattn_problem* prob, const dattn_host_step* io, const dattn_tensors* cache,
                         void* staging, size_t staging_bytes, void* workspace, size_t workspace_bytes,
                         void* stream, void* done_event, const char* where,
                         const dattn_step_copies* cp = nullptr) {
  dattn_status st = check_step(prob, io, true, where);
  if (st != DATTN_OK) return st;
  if (!cache || !staging) {
    set_error(std::string(where) + ": cache and staging are required");
    return DATTN_EINVAL;
  }
  // The input region (q, page table) does not depend on the plan: its transfer
  // is issued first and runs while the host plans.  Only the workspace's input
  // region is written before the plan's checks.
  const StepLayout L0 = step_layout(*prob, page_entries(prob, io), 0, 0);
  const size_t out0 = staging_out_off(L0, staging_bytes);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) || workspace_bytes < L0.plan_off ||
      (reinterpret_cast<uintptr_t>(staging) % 16) || staging_bytes < L0.plan_off || out0 < L0.plan_off) {
    set_error(std::string(where) + ": workspace (256-byte aligned) and staging (16-byte aligned) must hold at "
              "least " + std::to_string(L0.plan_off) + " bytes of inputs; dattn_step_host_sizes gives the full "
              "sizes");
    return DATTN_EWORKSPACE;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* sg = static_cast<uint8_t*>(staging);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the streams of the transfers: with cp, the inputs' stream first waits for the
  // last use of this workspace and staging buffer (done_event's previous record)
  const cudaStream_t cs = cp ? static_cast<cudaStream_t>(cp->h2d_stream) : s;
  const cudaStream_t os = cp ? static_cast<cudaStream_t>(cp->d2h_stream) : s;
  cudaError_t err = cudaSuccess;
  if (cp) err = cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(done_event), 0);
  if (err != cudaSuccess) return cuda_fail("host step copy-stream order", err);
  std::memcpy(sg, io->q, L0.q_bytes);
  if (L0.pi_bytes) std::memcpy(sg + L0.pi_off, io->page_indptr, L0.pi_bytes);
  if (L0.px_bytes) std::memcpy(sg + L0.px_off, io->page_indices, L0.px_bytes);
  err = cudaMemcpyAsync(ws, sg, L0.plan_off, cudaMemcpyHostToDevice, cs);
  if (err != cudaSuccess) return cuda_fail("host step input transfer", err);

  dattn_plan_t* plan = nullptr;
  size_t plan_ws = 0;
  if ((st = plan_step(prob, io, &plan, &plan_ws)) != DATTN_OK) return st;
  const StepLayout L = step_layout(*prob, page_entries(prob, io), plan_ws, plan->blob.size());
  if (workspace_bytes < L.ws_total || staging_bytes < L.staging_total) {
    set_error(std::string(where) + ": workspace needs " + std::to_string(L.ws_total) + " bytes and staging " +
              std::to_string(L.staging_total) + " bytes");
    dattn_plan_destroy(plan);
    return DATTN_EWORKSPACE;
  }
  // the cache pointers from "cache"; the step's inputs and outputs in the workspace
  dattn_tensors t = *cache;
  t.q = ws;
  t.o = ws + L.o_off;
  t.lse = reinterpret_cast<float*>(ws + L.lse_off);
  if (prob->layout == DATTN_KV_PAGED_HND) {
    t.page_indptr = reinterpret_cast<const int32_t*>(ws + L.pi_off);
    t.page_indices = reinterpret_cast<const int32_t*>(ws + L.px_off);
  }
  if ((st = check_run_args(plan, prob, &t, ws + L.plan_off, plan_ws, true, where)) != DATTN_OK) {
    dattn_plan_destroy(plan);
    return st;
  }
  // the work list (the staging copy of the inputs may still be in flight: that
  // part of the staging buffer is not touched again before the step is done)
  std::memcpy(sg + L.plan_off, plan->blob.data(), plan->blob.size());
  err = cudaMemcpyAsync(ws + L.plan_off, sg + L.plan_off, plan->blob.size(), cudaMemcpyHostToDevice, cs);
  if (err == cudaSuccess && cp) {   // the kernels wait for the step's inputs
    err = cudaEventRecord(static_cast<cudaEvent_t>(cp->inputs_event), cs);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(cp->inputs_event), 0);
  }
  if (err != cudaSuccess) {
    dattn_plan_destroy(plan);
    return cuda_fail("host step work-list transfer", err);
  }
  dattn_run_options opt{};
  opt.flags = DATTN_RUN_REUSE_UPLOAD;
  st = run_impl(plan, prob, &t, ws + L.plan_off, plan_ws, stream, &opt, where);
  dattn_plan_destroy(plan);
  if (st != DATTN_OK) return st;
  // outputs: one device->host transfer into the end of the staging buffer (with cp,
  // on the device->host stream once the kernels are done)
  if (cp) {
    err = cudaEventRecord(static_cast<cudaEvent_t>(cp->kernels_event), s);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(os, static_cast<cudaEvent_t>(cp->kernels_event), 0);
    if (err != cudaSuccess) return cuda_fail("host step output order", err);
  }
  err = cudaMemcpyAsync(sg + staging_out_off(L, staging_bytes), ws + L.o_off, align_ws(L.o_bytes) + L.lse_bytes,
                        cudaMemcpyDeviceToHost, os);
  if (err == cudaSuccess && done_event) err = cudaEventRecord(static_cast<cudaEvent_t>(done_event), os);
  if (err != cudaSuccess) return cuda_fail("host step output transfer", err);
  return DATTN_OK;
}

// Copies a finished step's O and LSE from the staging buffer into the caller's arrays.
void step_copy_out(const dattn_problem* prob, const dattn_host_step* io, const void* staging, size_t staging_bytes) {
  const StepLayout L = step_layout(*prob, page_entries(prob, io), 0, 0);
  const uint8_t* out = static_cast<const uint8_t*>(staging) + staging_out_off(L, staging_bytes);
  std::memcpy(io->o, out, L.o_bytes);
  if (io->lse) std::memcpy(io->lse, out + align_ws(L.o_bytes), L.lse_bytes);
}

}  // namespace

extern "C" dattn_status dattn_step_host(const dattn_problem* prob, const dattn_host_step* io,
                                        const dattn_tensors* cache, void* staging, size_t staging_bytes,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  dattn_status st = step_submit(prob, io, cache, staging, staging_bytes, workspace, workspace_bytes, stream,
                                nullptr, "dattn_step_host");
  if (st != DATTN_OK) return st;
  const cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail("dattn_step_host", err);
  step_copy_out(prob, io, staging, staging_bytes);
  return DATTN_OK;
}

extern "C" dattn_status dattn_step_host_submit(const dattn_problem* prob, const dattn_host_step* io,
                                               const dattn_tensors* cache, void* staging, size_t staging_bytes,
                                               void* workspace, size_t workspace_bytes, void* stream,
                                               void* done_event) {
  if (!done_event) {
    set_error("dattn_step_host_submit: done_event is required");
    return DATTN_EINVAL;
  }
  return step_submit(prob, io, cache, staging, staging_bytes, workspace, workspace_bytes, stream, done_event,
                     "dattn_step_host_submit");
}

extern "C" dattn_status dattn_step_host_submit_ex(const dattn_problem* prob, const dattn_host_step* io,
                                                  const dattn_tensors* cache, void* staging, size_t staging_bytes,
                                                  void* workspace, size_t workspace_bytes, void* stream,
                                                  void* done_event, const dattn_step_copies* copies) {
  if (!done_event || (copies && (!copies->h2d_stream || !copies->d2h_stream || !copies->inputs_event ||
                                 !copies->kernels_event))) {
    set_error("dattn_step_host_submit_ex: done_event and, when copies is given, its streams and events are required");
    return DATTN_EINVAL;
  }
  return step_submit(prob, io, cache, staging, staging_bytes, workspace, workspace_bytes, stream, done_event,
                     "dattn_step_host_submit_ex", copies);
}

extern "C" dattn_status dattn_step_host_finish(const dattn_problem* prob, const dattn_host_step* io,
                                               const void* staging, size_t staging_bytes, void* done_event) {
  Checker c;
  check_problem(prob, c);
  if (!io || !io->o || !staging || !done_event) c.fail(DATTN_EINVAL, "io, io->o, staging and done_event are required");
  if (c.status != DATTN_OK) return c.finish("dattn_step_host_finish");
  const cudaError_t err = cudaEventSynchronize(static_cast<cudaEvent_t>(done_event));
  if (err != cudaSuccess) return cuda_fail("dattn_step_host_finish", err);
  step_copy_out(prob, io, staging, staging_bytes);
  return DATTN_OK;
}

extern "C" dattn_status dattn_step_host_status(const dattn_problem* prob, const dattn_host_step* io,
                                               const void* workspace, int32_t* flags, void* stream) {
  dattn_status st = check_step(prob, io, false, "dattn_step_host_status");
  if (st != DATTN_OK) return st;
  const StepLayout L = step_layout(*prob, page_entries(prob, io), 0, 0);
  return dattn_device_status(static_cast<const uint8_t*>(workspace) + L.plan_off, flags, stream);
}
