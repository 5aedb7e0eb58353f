// Host planner of libdattn: call validation, visible key streams, chunking,
// CTA assignment and workspace sizing.  Plain C++, no CUDA calls, so it runs
// (and is tested) on a machine without a GPU.
//
// "M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries":
//  - §0x07A semantic pre-checks and §0x07B the full rejection vector;
//  - §0x03B balanced quotient/remainder split bounds (fixed split counts) and
//    fixed-width chunks (planner mode);
//  - §0x09E / §0x09G the paper planner: chunks no wider than a bound, sorted
//    longest first and each given to the least-loaded CTA, deterministically;
//  - §0x0AD request_indices / kv_tile_indices / o_indptr: here the work items
//    and the merge groups;
//  - §0x03D-§0x03E workspace: (m, l, u) fp32 per (slot, row), validity
//    encoded as l = 0 with m = -inf.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <queue>
#include <string>
#include <vector>

#include "plan.h"

namespace {
thread_local std::string g_last_error;
}

namespace dattn {

void set_error(const std::string& s) { g_last_error = s; }

void Checker::fail(dattn_status st, const std::string& why) {
  if (status == DATTN_OK || (status == DATTN_EUNSUPPORTED && st == DATTN_EINVAL)) status = st;
  if (!reasons.empty()) reasons += "; ";
  reasons += why;
}

dattn_status Checker::finish(const char* where) {
  if (status != DATTN_OK) set_error(std::string(where) + ": " + reasons);
  return status;
}

int group_rows(const dattn_problem& p) { return (p.H_q / std::max(1, p.H_kv)) * p.S_q; }

void check_problem(const dattn_problem* p, Checker& c) {
  if (!p) {
    c.fail(DATTN_EINVAL, "problem is NULL");
    return;
  }
  if (p->B < 1) c.fail(DATTN_EINVAL, "B must be >= 1");
  if (p->S_q < 1) c.fail(DATTN_EINVAL, "S_q must be >= 1 (q_len > 0)");
  if (p->H_q < 1 || p->H_kv < 1) c.fail(DATTN_EINVAL, "H_q and H_kv must be >= 1");
  else if (p->H_q % p->H_kv) c.fail(DATTN_EINVAL, "H_q must be a multiple of H_kv (GQA group)");
  else if (p->S_q >= 1 && group_rows(*p) > kMaxRows)
    c.fail(DATTN_EUNSUPPORTED, "g * S_q query rows per kv head must be <= 32");
  if (p->d_h != 64 && p->d_h != 128) c.fail(DATTN_EUNSUPPORTED, "d_h must be 64 or 128");
  if (p->layout != DATTN_KV_CONTIG_NHD && p->layout != DATTN_KV_PAGED_HND && p->layout != DATTN_KV_PACKED_ROWS)
    c.fail(DATTN_EINVAL, "unknown layout");
  if (p->layout == DATTN_KV_PACKED_ROWS) {
    if (p->fmt != DATTN_FMT_BF16) c.fail(DATTN_EUNSUPPORTED, "the packed-row layout holds bf16 rows");
    if (p->mask != DATTN_MASK_INDEX_LIST)
      c.fail(DATTN_EINVAL, "the packed-row layout needs the index-list program (its position map)");
  }
  if (p->fmt < DATTN_FMT_BF16 || p->fmt > DATTN_FMT_INT4_HEAD) c.fail(DATTN_EINVAL, "unknown format");
  if (p->mask < DATTN_MASK_CAUSAL || p->mask > DATTN_MASK_FLASHMASK) c.fail(DATTN_EINVAL, "unknown mask");
  // K/V rows (one kv head, one token) are addressed with 32-bit row indices
  const long long kMaxPoolRows = 0xFFFFFFFFll;
  if (p->layout == DATTN_KV_PAGED_HND) {
    if (p->page_size < 1) c.fail(DATTN_EINVAL, "paged layout needs page_size >= 1");
    if (p->num_pages < 1) c.fail(DATTN_EINVAL, "paged layout needs num_pages >= 1");
    if (p->page_size >= 1 && p->num_pages >= 1 && p->H_kv >= 1 &&
        static_cast<long long>(p->num_pages) * p->H_kv * p->page_size >= kMaxPoolRows)
      c.fail(DATTN_EUNSUPPORTED, "num_pages * H_kv * page_size must be below 2^32 - 1 rows");
  } else if (p->layout == DATTN_KV_CONTIG_NHD) {
    if (p->fmt != DATTN_FMT_BF16) c.fail(DATTN_EUNSUPPORTED, "quantized formats need the paged layout");
    if (p->T_cap < 1) c.fail(DATTN_EINVAL, "contiguous layout needs T_cap >= 1");
    if (p->B_cache < 1) c.fail(DATTN_EINVAL, "contiguous layout needs B_cache >= 1");
    if (p->T_cap >= 1 && p->B_cache >= 1 && p->H_kv >= 1 &&
        static_cast<long long>(p->B_cache) * p->T_cap * p->H_kv >= kMaxPoolRows)
      c.fail(DATTN_EUNSUPPORTED, "B_cache * T_cap * H_kv must be below 2^32 - 1 rows");
  }
  if (p->fmt == DATTN_FMT_INT8_TOKEN && p->page_size >= 1 && (p->page_size % 4 || p->page_size > 256))
    c.fail(DATTN_EUNSUPPORTED, "INT8 pages must hold a multiple of 4 rows, at most 256");
  if (p->fmt == DATTN_FMT_INT4_KIVI) {
    const int G = p->kivi_group, Gv = p->kivi_v_group, R = p->kivi_residual;
    if (G != 32 && G != 64) c.fail(DATTN_EUNSUPPORTED, "kivi_group must be 32 or 64");
    if (Gv != 16 && Gv != 32 && Gv != 64) c.fail(DATTN_EUNSUPPORTED, "kivi_v_group must be 16, 32 or 64");
    else if (4 * Gv > p->d_h) c.fail(DATTN_EUNSUPPORTED, "kivi_v_group must be at most d_h / 4");
    if (p->mask == DATTN_MASK_INDEX_LIST)
      c.fail(DATTN_EUNSUPPORTED, "INT4 KIVI reads causal, sink+window or flashmask streams");
    if (p->mask == DATTN_MASK_FLASHMASK && p->page_size >= 1 && (p->page_size & (p->page_size - 1)) != 0)
      c.fail(DATTN_EUNSUPPORTED, "flashmask on INT4 KIVI needs a power-of-two page_size");
    if (G >= 1 && (R < G || R % G)) c.fail(DATTN_EINVAL, "kivi_residual must be a positive multiple of kivi_group");
    if (G >= 1 && p->page_size >= 1 && p->page_size % G && G % p->page_size)
      c.fail(DATTN_EUNSUPPORTED, "page_size and kivi_group must divide one another");
  }
  if (p->mask == DATTN_MASK_SINK_WINDOW) {
    if (p->n_sink < 0) c.fail(DATTN_EINVAL, "n_sink must be >= 0");
    if (p->window < 1) c.fail(DATTN_EINVAL, "window must be >= 1");
  }
  if (!(p->sm_scale >= 0.f) || !std::isfinite(p->sm_scale)) c.fail(DATTN_EINVAL, "sm_scale must be finite and >= 0");
  if (p->fixed_splits < 0) c.fail(DATTN_EINVAL, "fixed_splits must be >= 0");
}

// Default cost of a work item in the equal-segment partition, in keys of the
// format: about 48 KB of K/V of fixed pipeline time (a stage and a half of the
// bf16 kernel) plus the partial states the item writes (rows x states per row
// x (d + 2) fp32 values), which the merge reads back.
static long long default_item_cost_keys(const dattn_problem& p, int item_rows, int states_per_row) {
  const long long d = p.d_h;
  long long kb;   // K and V bytes of one key
  switch (p.fmt) {
    case DATTN_FMT_INT8_TOKEN: kb = 2 * d + 8; break;
    case DATTN_FMT_FP8_E4M3:
    case DATTN_FMT_FP8_E5M2: kb = 2 * d; break;
    case DATTN_FMT_INT4_HEAD:
    case DATTN_FMT_INT4_KIVI: kb = d + 8; break;
    default: kb = 4 * d;
  }
  const long long bytes = 49152 + static_cast<long long>(item_rows) * states_per_row * (d + 2) * 4;
  return (bytes / kb + 15) / 16 * 16;
}

bool same_problem(const dattn_problem& a, const dattn_problem& b) {
  return std::memcmp(&a, &b, sizeof(dattn_problem)) == 0;
}

// Visible key stream of one group: length and the two-interval map.
static void stream_of(const dattn_problem& p, int T, int C, int list_len, int list_off, int& n, int& x0,
                      int& x1) {
  if (C == 0) {   // a request without query rows reads nothing
    n = x0 = x1 = 0;
    return;
  }
  if (p.mask == DATTN_MASK_INDEX_LIST) {
    n = list_len;
    x0 = list_off;
    x1 = 0;
    return;
  }
  if (p.mask == DATTN_MASK_SINK_WINDOW) {
    // Union over rows of [0, min(n_sink, F_i)) U [max(0, F_i - W), F_i)
    // with F_i = max(0, min(T, T - C + i + 1)); F_i grows with i.
    const int f_max = std::max(0, T);
    const int f_min = std::max(0, std::min(T, T - C + 1));
    const int sink_end = std::min(p.n_sink, f_max);
    const int win_start = std::max(0, f_min - p.window);
    if (win_start <= sink_end) {
      n = f_max;
      x0 = f_max;
      x1 = 0;
    } else {
      n = sink_end + (f_max - win_start);
      x0 = sink_end;
      x1 = win_start;
    }
    return;
  }
  n = std::max(0, T);  // causal: union over rows is every stored key
  x0 = n;
  x1 = 0;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace dattn

using namespace dattn;

extern "C" dattn_status dattn_plan(const dattn_problem* prob, const dattn_plan_inputs* in,
                                   dattn_plan_t** out, size_t* workspace_bytes) {
  Checker c;
  check_problem(prob, c);
  if (!in) c.fail(DATTN_EINVAL, "plan inputs are NULL");
  if (!out) c.fail(DATTN_EINVAL, "out is NULL");
  if (c.status != DATTN_OK) return c.finish("dattn_plan");
  const dattn_problem& p = *prob;
  if (!in->kv_len) c.fail(DATTN_EINVAL, "kv_len is NULL");
  if (in->num_sms < 1) c.fail(DATTN_EINVAL, "num_sms must be >= 1");
  if (in->ctas_per_sm < 0) c.fail(DATTN_EINVAL, "ctas_per_sm must be >= 0");
  if (in->chunk_tokens < 0) c.fail(DATTN_EINVAL, "chunk_tokens must be >= 0");
  if (p.mask == DATTN_MASK_INDEX_LIST && !in->index_indptr)
    c.fail(DATTN_EINVAL, "index_list mask needs index_indptr");
  if (c.status != DATTN_OK) return c.finish("dattn_plan");

  const int B = p.B, H = p.H_kv;
  for (int b = 0; b < B; ++b) {
    const int T = in->kv_len[b];
    if (T < 0) c.fail(DATTN_EINVAL, "kv_len[" + std::to_string(b) + "] < 0");
    if (p.layout == DATTN_KV_CONTIG_NHD && T > p.T_cap)
      c.fail(DATTN_EINVAL, "kv_len[" + std::to_string(b) + "] > T_cap");
    if (p.layout == DATTN_KV_PAGED_HND && in->page_indptr && T >= 0 && p.page_size >= 1) {
      const int have = in->page_indptr[b + 1] - in->page_indptr[b];
      const long need = (static_cast<long>(T) + p.page_size - 1) / p.page_size;
      if (have < 0) c.fail(DATTN_EINVAL, "page_indptr must be non-decreasing");
      else if (have < need)
        c.fail(DATTN_EINVAL, "request " + std::to_string(b) + " has " + std::to_string(have) +
                                 " pages but needs " + std::to_string(need));
    }
    if (p.mask == DATTN_MASK_INDEX_LIST) {
      for (int h = 0; h < H; ++h) {
        const int k = b * H + h;
        const int n = in->index_indptr[k + 1] - in->index_indptr[k];
        if (n < 0) {
          c.fail(DATTN_EINVAL, "index_indptr must be non-decreasing");
          continue;
        }
        if (n > std::max(0, T)) c.fail(DATTN_EINVAL, "index list of (" + std::to_string(b) + "," +
                                                         std::to_string(h) + ") longer than T_b");
        if (in->index_list) {
          const int32_t* L = in->index_list + in->index_indptr[k];
          for (int i = 0; i < n; ++i) {
            if (L[i] < 0 || L[i] >= T) {
              c.fail(DATTN_EINVAL, "index list of (" + std::to_string(b) + "," + std::to_string(h) +
                                       ") has an entry outside [0, T_b)");
              break;
            }
            if (i && L[i] <= L[i - 1]) {
              c.fail(DATTN_EINVAL, "index list of (" + std::to_string(b) + "," + std::to_string(h) +
                                       ") is not strictly increasing");
              break;
            }
          }
        }
      }
    }
  }
  if (p.mask == DATTN_MASK_INDEX_LIST && in->index_indptr[0] != 0)
    c.fail(DATTN_EINVAL, "index_indptr[0] must be 0");
  if (in->qo_indptr) {
    if (in->qo_indptr[0] != 0) c.fail(DATTN_EINVAL, "qo_indptr[0] must be 0");
    bool mixed = false;
    for (int b = 0; b < B; ++b) {
      const int cb = in->qo_indptr[b + 1] - in->qo_indptr[b];
      if (cb < 0 || cb > p.S_q)
        c.fail(DATTN_EINVAL, "request " + std::to_string(b) + " has " + std::to_string(cb) +
                                 " query rows; 0 <= C_b <= S_q");
      mixed = mixed || cb != p.S_q;
    }
    // the KIVI byte-format kernel (page sizes that are not a power of two) reads uniform batches
    if (mixed && p.fmt == DATTN_FMT_INT4_KIVI && (p.page_size & (p.page_size - 1)) != 0)
      c.fail(DATTN_EUNSUPPORTED, "mixed query-row counts on INT4 KIVI need a power-of-two page_size");
  }
  if (p.mask == DATTN_MASK_FLASHMASK) {
    long long keys = 0;
    for (int b = 0; b < B; ++b) keys += std::max(0, in->kv_len[b]);
    if (keys > INT32_MAX / 4) c.fail(DATTN_EUNSUPPORTED, "flashmask intervals of more than 2^29 keys");
  }
  if (c.status != DATTN_OK) return c.finish("dattn_plan");

  auto* plan = new dattn_plan_s();
  plan->prob = p;
  plan->kv_len.assign(in->kv_len, in->kv_len + B);
  const int rows = group_rows(p);
  const int n_groups = B * H;

  // 1. visible key stream of every group
  // request b's packed query rows: qo_indptr[b] .. + C_b (uniform S_q without qo_indptr)
  auto query_start = [&](int b) { return in->qo_indptr ? in->qo_indptr[b] : b * p.S_q; };
  auto query_rows = [&](int b) { return in->qo_indptr ? in->qo_indptr[b + 1] - in->qo_indptr[b] : p.S_q; };
  std::vector<int> gn(n_groups), gx0(n_groups), gx1(n_groups);
  long long W = 0, fm_off = 0;
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h) {
      const int k = b * H + h;
      int len = 0, off = 0;
      if (p.mask == DATTN_MASK_INDEX_LIST) {
        off = in->index_indptr[k];
        len = in->index_indptr[k + 1] - off;
      }
      stream_of(p, in->kv_len[b], query_rows(b), len, off, gn[k], gx0[k], gx1[k]);
      // FlashMask: every stored key is in the stream; x1 locates the request's intervals
      if (p.mask == DATTN_MASK_FLASHMASK) gx1[k] = static_cast<int>(fm_off);
      W += gn[k];
    }
    fm_off += in->kv_len[b];
  }


  // 2. chunks.  Three modes:
  //  - fixed_splits > 0: balanced quotient/remainder bounds per group (§0x03B);
  //  - chunk_tokens > 0: chunks of that width, assigned in step 4 longest-first
  //    to the least-loaded CTA (the FlashInfer paper planner, §0x09E);
  //  - default: the concatenation of all groups' visible streams is cut into
  //    equal key segments, one per CTA, and a group is chunked where segment
  //    boundaries fall into it (every CTA streams the same number of keys).
  const int cps = in->ctas_per_sm > 0 ? in->ctas_per_sm : kDefaultCtasPerSm;
  const long long cta_target = static_cast<long long>(in->num_sms) * cps;
  const long long L = in->chunk_tokens;
  const bool segmented = p.fixed_splits <= 0 && L <= 0;
  // Every item also costs a fixed amount of pipeline time (its first stage's
  // fill, its states), which the segments account for as "pad" keys charged
  // at the start of each non-empty group: without it, a CTA that receives
  // many tiny groups streams as many keys as the others plus their overheads,
  // and finishes last.
  const bool kivi_tc = kivi_on_tensor_cores(p.d_h, rows, p.kivi_v_group, p.mask, p.page_size, p.kivi_residual);
  const int spi = states_per_item(rows, p.fmt, kivi_tc);
  // states per row of request b's items: bf16 requests of at most 16 rows run
  // the one-tile layout (8) even when the call's widest request has more
  auto spi_of = [&](int b) {
    return p.fmt == DATTN_FMT_BF16 && rows > 16 && (p.H_q / p.H_kv) * query_rows(b) <= 16
               ? states_per_item(16, p.fmt, kivi_tc) : spi;
  };
  // The segments are cut on an axis of sixteenths of a key: a group's keys
  // weigh kKeyUnit each, those of a bf16 request with more than 16 rows (the
  // 32-row tile, about a quarter slower per key on GB300 than one 16-row tile)
  // kWideKeyUnit, and each non-empty group starts with its pad.
  constexpr long long kKeyUnit = 16, kWideKeyUnit = 20;
  auto weight_of = [&](int b) {
    return p.fmt == DATTN_FMT_BF16 && (p.H_q / p.H_kv) * query_rows(b) > 16 ? kWideKeyUnit : kKeyUnit;
  };
  std::vector<long long> pad(n_groups, 0);
  long long Wp = 0;                                  // padded, weighted length of the concatenation
  for (int k = 0; k < n_groups; ++k) {
    const int b = k / H;
    Wp += static_cast<long long>(gn[k]) * weight_of(b);
    if (!segmented || gn[k] == 0 || in->item_cost_keys < 0) continue;
    pad[k] = kKeyUnit * (in->item_cost_keys > 0 ? in->item_cost_keys
                                                : default_item_cost_keys(p, (p.H_q / p.H_kv) * query_rows(b), spi_of(b)));
    Wp += pad[k];
  }
  long long seg = 1;
  int n_seg = 1;
  if (segmented && Wp > 0) {
    const long long keys = (Wp + kKeyUnit - 1) / kKeyUnit;
    const long long want = std::max<long long>(1, std::min<long long>(cta_target, (keys + kTK - 1) / kTK));
    seg = (Wp + want - 1) / want;
    seg = (seg + 16 * kKeyUnit - 1) / (16 * kKeyUnit) * (16 * kKeyUnit);   // whole 16-key tiles
    n_seg = static_cast<int>((Wp + seg - 1) / seg);
  }
  std::vector<int> group_first(n_groups + 1, 0);
  std::vector<int> seg_cta;                          // segmented mode: the CTA of every item
  auto& items = plan->items;
  items.reserve(static_cast<size_t>(n_groups) + (segmented ? n_seg : 0) +
                (p.fixed_splits > 0 ? static_cast<size_t>(n_groups) * p.fixed_splits : 0));
  seg_cta.reserve(items.capacity());
  long long g_off = 0;                               // offset of the group in the concatenation
  for (int k = 0; k < n_groups; ++k) {
    group_first[k] = static_cast<int>(items.size());
    const int b = k / H, h = k % H, n = gn[k];
    auto add = [&](int a, int e) {
      items.push_back(WorkItem{b, h, a, e, -1, plan->kv_len[b], gx0[k], gx1[k]});
    };
    if (p.fixed_splits > 0) {
      const int S = p.fixed_splits, q = n / S, r = n % S;
      for (int s = 0; s < S; ++s) {
        const int a = s * q + std::min(s, r);
        add(a, a + q + (s < r ? 1 : 0));
      }
    } else if (segmented) {
      if (n == 0) {
        add(0, 0);
        seg_cta.push_back(static_cast<int>(std::min<long long>(n_seg - 1, g_off / seg)));
      }
      // KIVI: cuts rounded up onto the 32-key grid, so that the consumers' 32-key
      // steps never straddle a K group (a CTA streams at most 31 keys more)
      const long long grid = p.fmt == DATTN_FMT_INT4_KIVI ? 32 : 1;
      const long long k0 = g_off + pad[k];   // padded position of the group's first key
      const long long wk = weight_of(b);
      for (long long a = 0; a < n;) {
        const long long c = std::min<long long>(n_seg - 1, (k0 + a * wk) / seg);
        const long long cut = ((c + 1) * seg - k0 + wk - 1) / wk;    // first key of the next segment
        const long long e = std::min<long long>(n, std::max<long long>(a + 1, (cut + grid - 1) / grid * grid));
        add(static_cast<int>(a), static_cast<int>(e));
        seg_cta.push_back(static_cast<int>(c));
        a = e;
      }
    } else if (n == 0) {
      add(0, 0);
    } else {
      for (long long a = 0; a < n; a += L) add(static_cast<int>(a), static_cast<int>(std::min<long long>(n, a + L)));
    }
    g_off += static_cast<long long>(n) * (segmented ? weight_of(b) : 1) + pad[k];
  }
  group_first[n_groups] = static_cast<int>(items.size());

  // 3. partial-state slots and merge groups (o_indptr): every consumer warp of
  //    an item leaves its own state, so an item owns states_per_item slots; a
  //    group that is one item with one state per row writes O directly.
  std::vector<MergeGroup> merges;
  std::vector<int> merge_of_group(n_groups, -1);
  int n_slots = 0, max_splits = 0;
  for (int k = 0; k < n_groups; ++k) {
    const int n = group_first[k + 1] - group_first[k];
    max_splits = std::max(max_splits, n);
    const int spi_k = spi_of(k / H);
    if (n * spi_k > 1) {
      merge_of_group[k] = static_cast<int>(merges.size());
      merges.push_back(MergeGroup{k / H, k % H, n_slots, n * spi_k, query_start(k / H), query_rows(k / H), 0, 0});
      for (int i = 0; i < n; ++i) items[group_first[k] + i].slot = n_slots + i * spi_k;
      n_slots += n * spi_k;
    }
  }

  // 4. CTA assignment: the segment owner (default mode; items are generated
  //    in segment order already), else longest-first to the least-loaded CTA
  //    (deterministic ties).  cta_start / cta_order: counting-sort layout of
  //    the per-CTA item lists.
  const int n_items = static_cast<int>(items.size());
  const int n_ctas = segmented ? n_seg : static_cast<int>(std::min<long long>(cta_target, n_items));
  auto cost = [&](int i) { return static_cast<long long>(items[i].e - items[i].a) + 16; };
  std::vector<long long> keys_of(n_ctas, 0);
  std::vector<int> cta_start(n_ctas + 1, 0), cta_order(n_items);
  plan->item_cta.assign(n_items, 0);
  std::vector<int> order(n_items);          // order in which items are listed per CTA
  for (int i = 0; i < n_items; ++i) order[i] = i;
  if (segmented) {
    for (int i = 0; i < n_items; ++i) plan->item_cta[i] = seg_cta[i];
  } else {
    using Slot = std::pair<long long, int>;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost(x) > cost(y); });
    std::vector<Slot> heap_store;
    heap_store.reserve(n_ctas);
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap(std::greater<Slot>(), std::move(heap_store));
    for (int cta = 0; cta < n_ctas; ++cta) heap.push({0, cta});
    for (int i : order) {
      auto [load, cta] = heap.top();
      heap.pop();
      plan->item_cta[i] = cta;
      heap.push({load + cost(i), cta});
    }
  }
  for (int i = 0; i < n_items; ++i) {
    ++cta_start[plan->item_cta[i] + 1];
    keys_of[plan->item_cta[i]] += items[i].e - items[i].a;
  }
  for (int c = 0; c < n_ctas; ++c) cta_start[c + 1] += cta_start[c];
  {
    std::vector<int> fill(cta_start.begin(), cta_start.end() - 1);
    for (int i : order) cta_order[fill[plan->item_cta[i]]++] = i;
  }

  // 5. blob and workspace
  BlobHeader hdr{};
  hdr.magic = kBlobMagic;
  hdr.n_items = n_items;
  hdr.n_ctas = n_ctas;
  hdr.n_merge = static_cast<int>(merges.size());
  hdr.rows = rows;
  hdr.n_slots = n_slots;
  // on request, bf16 groups are merged inside the partial kernel by the last CTA to finish them
  hdr.fused = in->fused_merge != 0 && p.fmt == DATTN_FMT_BF16 && !merges.empty();
  size_t off = align_up(sizeof(BlobHeader), 16);
  hdr.off_items = off;
  off = align_up(off + sizeof(WorkItem) * n_items, 16);
  hdr.off_cta_indptr = off;
  off = align_up(off + sizeof(int32_t) * (n_ctas + 1), 16);
  hdr.off_cta_items = off;
  off = align_up(off + sizeof(int32_t) * n_items, 16);
  hdr.off_merge = off;
  off = align_up(off + sizeof(MergeGroup) * merges.size(), 16);
  hdr.off_cta_recs = off;
  off = align_up(off + sizeof(ItemRec) * n_items, 16);
  hdr.off_count = off;
  off = align_up(off + sizeof(int32_t) * merges.size(), 16);
  // State-row tags of the separate merge (bf16), zero (no run's tag) in every upload:
  // the merge starts on each group as soon as its states are tagged.  Measured on GB300
  // against the merge waiting for the whole grid: mixed batch -3.0 us, long context
  // S_q = 1 -1.3 us, tree verify -1.0 us, sink + window -0.4 us, index lists -0.2 us,
  // the headline unchanged, long context S_q = 4 +0.2 us; a merge of fewer than 64 group
  // rows (the 8 of the tiny decode) gains nothing to make up for the fence, +0.2 us.
  hdr.tags = !merges.empty() && !hdr.fused && p.fmt == DATTN_FMT_BF16 &&
             (in->merge_tags > 0 || (in->merge_tags == 0 && static_cast<long long>(merges.size()) * rows >= 64));
  hdr.off_seq = off;
  if (hdr.tags) off += sizeof(int32_t) * static_cast<size_t>(n_slots) * rows;
  off = align_up(off, kWsAlign);
  const size_t blob_bytes = off;
  hdr.off_ml = off;
  off = align_up(off + sizeof(float) * 2 * static_cast<size_t>(n_slots) * rows, kWsAlign);
  hdr.off_u = off;
  off = align_up(off + sizeof(float) * static_cast<size_t>(n_slots) * rows * p.d_h, kWsAlign);
  const size_t ws_bytes = off;

  plan->blob.assign(blob_bytes, 0);
  uint8_t* base = plan->blob.data();
  std::memcpy(base, &hdr, sizeof(hdr));
  std::memcpy(base + hdr.off_items, items.data(), sizeof(WorkItem) * n_items);
  auto* cta_indptr = reinterpret_cast<int32_t*>(base + hdr.off_cta_indptr);
  auto* cta_items = reinterpret_cast<int32_t*>(base + hdr.off_cta_items);
  auto* cta_recs = reinterpret_cast<ItemRec*>(base + hdr.off_cta_recs);
  int pos = 0;
  for (int cta = 0; cta < n_ctas; ++cta) {
    cta_indptr[cta] = pos;
    for (int k = cta_start[cta]; k < cta_start[cta + 1]; ++k) {
      const int i = cta_order[k];
      ItemRec r{};
      r.it = items[i];
      r.merge = merge_of_group[static_cast<size_t>(items[i].b) * H + items[i].h];
      r.qo = query_start(items[i].b);
      r.nq = query_rows(items[i].b);
      if (p.fmt == DATTN_FMT_INT4_KIVI) {   // residual keys lie in [n_q, T) with T - n_q <= R
        const int T = items[i].T, G = p.kivi_group, R = p.kivi_residual;
        const int nq = T > R ? (T - R + G - 1) / G * G : 0;
        r.ring_off = nq % R - nq;
      }
      r.lo = r.hi = -1;      // resolved by the kernel when the host page list is unknown
      if (p.layout == DATTN_KV_PAGED_HND && in->page_indptr) {
        r.lo = in->page_indptr[items[i].b];
        r.hi = in->page_indptr[items[i].b + 1];
      }
      cta_recs[pos] = r;
      cta_items[pos++] = i;
    }
  }
  cta_indptr[n_ctas] = pos;
  if (!merges.empty()) std::memcpy(base + hdr.off_merge, merges.data(), sizeof(MergeGroup) * merges.size());

  dattn_plan_info& info = plan->info;
  info.workspace_bytes = static_cast<int64_t>(ws_bytes);
  info.blob_bytes = static_cast<int64_t>(blob_bytes);
  info.n_items = n_items;
  info.n_ctas = n_ctas;
  info.n_slots = n_slots;
  plan->direct_items = 0;
  for (const WorkItem& w : items) plan->direct_items += w.slot < 0 ? 1 : 0;
  info.n_merge_groups = static_cast<int>(merges.size());
  info.fused_merge = hdr.fused;
  info.merge_tags = hdr.tags;
  info.max_splits = max_splits;
  info.rows = rows;
  info.stream_keys = W;
  info.max_cta_keys = keys_of.empty() ? 0 : *std::max_element(keys_of.begin(), keys_of.end());

  *out = plan;
  if (workspace_bytes) *workspace_bytes = ws_bytes;
  return DATTN_OK;
}

extern "C" void dattn_plan_destroy(dattn_plan_t* plan) { delete plan; }

extern "C" dattn_status dattn_plan_get_info(const dattn_plan_t* plan, dattn_plan_info* info) {
  if (!plan || !info) {
    set_error("dattn_plan_get_info: NULL argument");
    return DATTN_EINVAL;
  }
  *info = plan->info;
  return DATTN_OK;
}

extern "C" dattn_status dattn_plan_get_items(const dattn_plan_t* plan, dattn_work_item* items,
                                             int32_t capacity, int32_t* count) {
  if (!plan || !count || (capacity > 0 && !items)) {
    set_error("dattn_plan_get_items: NULL argument");
    return DATTN_EINVAL;
  }
  const int n = static_cast<int>(plan->items.size());
  *count = n;
  for (int i = 0; i < std::min(n, capacity); ++i) {
    const WorkItem& w = plan->items[i];
    items[i] = dattn_work_item{w.b, w.h, w.a, w.e, w.slot, plan->item_cta[i]};
  }
  return DATTN_OK;
}

extern "C" const char* dattn_last_error(void) { return g_last_error.c_str(); }

extern "C" int32_t dattn_version(void) { return 100; }
