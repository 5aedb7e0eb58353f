// Partial kernel of split-KV decode attention (bf16 K/V).
//
// One persistent CTA per SM walks its list of work items (request b, kv head
// h, keys [a, e) of the group's visible stream).  A producer warp turns every
// 64-key stage of an item into page segments (M4.5 §0x04E), translates each
// logical block through the CSR page list (§0x04D), and issues one bulk
// (TMA-engine) copy per segment and per K/V into a 4-deep shared-memory ring
// guarded by mbarriers.  It also classifies the stage (FULL / PARTIAL,
// §0x05C) so that FULL stages skip the per-element predicate; keys outside the
// visible stream (SKIP tiles) are never loaded at all (§0x05D).
//
// Eight consumer warps share every K/V tile across the GQA group (§0x03A):
// each warp owns 4 query rows (a row block) and a slice of the stage's keys.
// Lanes form 4 key groups x 8 lanes; a lane holds 16 (d=128) or 8 (d=64)
// channels of its key and of the 4 query rows, so q.k is 16 packed-fp32 FMAs
// plus a 3-step shuffle reduction.  The online softmax (§0x02B) is updated
// every 8 keys with exp2 in log2 units; masked scores become -inf before the
// maximum and the sums (§0x05C).  At the end of an item the warps of a row
// block merge their states through shared memory with the same (m, l, u)
// rule and write either O / LSE directly (single-chunk groups, as in
// FlashInfer's unpartitioned path, §0x0AD) or an fp32 partial state.
#include <cuda_runtime.h>

#include "device.cuh"

namespace dattn {

namespace {

constexpr unsigned kFull = 0xffffffffu;

template <int D>
struct Layout {
  static constexpr int kTileBytes = kTK * D * 2;            // one K (or V) tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kPos = kStages * kStageBytes;         // int32 [kStages][kTK]
  static constexpr int kCls = kPos + kStages * kTK * 4;      // int32 [kStages]
  static constexpr int kFullBar = (kCls + kStages * 4 + 15) / 16 * 16;
  static constexpr int kEmptyBar = kFullBar + kStages * 8;
  static constexpr int kAbort = kEmptyBar + kStages * 8;
  static constexpr int kScratch = (kAbort + 16 + 15) / 16 * 16;
  // per consumer warp: 4 rows x D values of u, then 4 x (m, l)
  static constexpr int kScratchWarp = 4 * D * 4 + 4 * 8;
  static constexpr int kTotal = kScratch + kConsumerWarps * kScratchWarp;
};

struct Run {
  int p0, p1, s0;  // positions [p0, p1) land in slots s0 ...
};

// Runs of consecutive positions covered by stream [j0, j1) of an interval item
// (at most two: the sink interval and the window / causal interval).
__device__ __forceinline__ int item_runs(const WorkItem& it, int j0, int j1, Run& r0, Run& r1) {
  int n = 0;
  Run a{0, 0, 0}, b{0, 0, 0};
  if (j0 < it.x0) a = Run{j0, min(j1, it.x0), 0}, n = 1;
  if (j1 > it.x0) {
    const int s = max(j0, it.x0);
    const Run x{it.x1 + (s - it.x0), it.x1 + (j1 - it.x0), s - j0};
    if (n == 0) a = x; else b = x;
    ++n;
  }
  r0 = a;
  r1 = b;
  return n;
}

__device__ __forceinline__ int run_segments(const Run& r, int P) {
  return r.p1 > r.p0 ? (r.p1 - 1) / P - r.p0 / P + 1 : 0;
}

// Segment "sg" of the runs: page block jb and positions [sp0, sp1) landing in slot "slot".
__device__ __forceinline__ void segment(const Run& r0, const Run& r1, int ns0, int sg, int P, int& jb, int& sp0,
                                        int& sp1, int& slot) {
  const bool first = sg < ns0;
  const int p0 = first ? r0.p0 : r1.p0, p1 = first ? r0.p1 : r1.p1, s0 = first ? r0.s0 : r1.s0;
  jb = p0 / P + (first ? sg : sg - ns0);
  sp0 = max(p0, jb * P);
  sp1 = min(p1, (jb + 1) * P);
  slot = s0 + (sp0 - p0);
}

// ---- producer ---------------------------------------------------------------------

template <int D>
__device__ void produce(const PartialParams& p, uint8_t* smem, int it_begin, int it_end, int lane) {
  using L = Layout<D>;
  int* pos_all = reinterpret_cast<int*>(smem + L::kPos);
  int* cls_all = reinterpret_cast<int*>(smem + L::kCls);
  const uint32_t full0 = smem_u32(smem + L::kFullBar);
  const uint32_t empty0 = smem_u32(smem + L::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(p.v);
  const bool paged = p.layout == DATTN_KV_PAGED_HND;
  const bool listed = p.mask == DATTN_MASK_INDEX_LIST;
  constexpr uint32_t kRowBytes = D * 2;

  uint32_t k = 0;
  for (int ii = it_begin; ii < it_end; ++ii) {
    const WorkItem it = p.items[p.cta_items[ii]];
    const MaskCtx mc{p.mask, p.S_q, it.T, p.n_sink, p.window};
    int list_n = 0;
    bool list_ok = true;
    if (listed) {
      const int g = it.b * p.H_kv + it.h;
      list_n = p.index_indptr[g + 1] - p.index_indptr[g];
      list_ok = p.index_indptr[g] == it.x0 && it.e <= list_n;
      if (!list_ok && lane == 0) atomicOr(p.status, kStListRange);
    }
    int c_row = 0;
    if (!paged) c_row = cache_row(p.cache_batch_idx, it.b, p.B_cache, lane == 0 ? p.status : nullptr);
    for (int j0 = it.a; j0 < it.e; j0 += kTK, ++k) {
      const int st = k % kStages;
      const uint32_t use = k / kStages;
      if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) return;
      const int j1 = min(j0 + kTK, it.e);
      const int n = j1 - j0;
      int* pos = pos_all + st * kTK;
      uint8_t* kt = smem + st * L::kStageBytes;
      uint8_t* vt = kt + L::kTileBytes;

      // pass 1: positions, validity and byte count
      for (int s = lane; s < kTK; s += 32) {
        int t = -1;
        if (s < n && list_ok) {
          t = stream_key(it, p.mask, p.index_list, j0 + s);
          if (listed && (t < 0 || t >= it.T)) {
            atomicOr(p.status, kStListRange);
            t = -1;
          }
        }
        pos[s] = t;
      }
      __syncwarp();
      uint32_t bytes = 0;
      if (paged && !listed) {
        Run r0, r1;
        const int nr = item_runs(it, j0, j1, r0, r1);
        const int ns0 = nr > 0 ? run_segments(r0, p.P) : 0;
        const int ns1 = nr > 1 ? run_segments(r1, p.P) : 0;
        for (int sg = lane; sg < ns0 + ns1; sg += 32) {
          int jb, sp0, sp1, slot;
          segment(r0, r1, ns0, sg, p.P, jb, sp0, sp1, slot);
          const int pi = page_of(p.page_indptr, p.page_indices, it.b, jb, p.num_pages, p.status);
          if (pi < 0) {
            for (int s = slot; s < slot + (sp1 - sp0); ++s) pos[s] = -1;
          } else {
            bytes += 2u * (sp1 - sp0) * kRowBytes;
          }
        }
      } else {
        for (int s = lane; s < n; s += 32) {
          const int t = pos[s];
          if (t < 0) continue;
          bool ok;
          if (paged) {
            ok = page_of(p.page_indptr, p.page_indices, it.b, t / p.P, p.num_pages, p.status) >= 0;
          } else {
            ok = c_row >= 0 && t < p.T_cap;
            if (!ok && c_row >= 0) atomicOr(p.status, kStRowRange);
          }
          if (ok) bytes += 2u * kRowBytes;
          else pos[s] = -1;
        }
      }
      bytes = __reduce_add_sync(kFull, bytes);

      // stage class: FULL when every query row sees every key of the stage
      if (lane == 0) {
        bool full = true;
        if (listed) {
          full = n == 0 || pos[n - 1] < frontier(mc, 0);
        } else {
          Run r0, r1;
          const int nr = item_runs(it, j0, j1, r0, r1);
          for (int i = 0; i < p.S_q && full; ++i) {
            if (nr > 0 && visible_in_run(mc, i, r0.p0, r0.p1) != r0.p1 - r0.p0) full = false;
            if (nr > 1 && visible_in_run(mc, i, r1.p0, r1.p1) != r1.p1 - r1.p0) full = false;
          }
        }
        cls_all[st] = full ? DATTN_TILE_FULL : DATTN_TILE_PARTIAL;
      }
      __syncwarp();
      const uint32_t fb = full0 + 8 * st;
      if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
      __syncwarp();

      // pass 2: issue the copies
      if (paged && !listed) {
        Run r0, r1;
        const int nr = item_runs(it, j0, j1, r0, r1);
        const int ns0 = nr > 0 ? run_segments(r0, p.P) : 0;
        const int ns1 = nr > 1 ? run_segments(r1, p.P) : 0;
        for (int sg = lane; sg < ns0 + ns1; sg += 32) {
          int jb, sp0, sp1, slot;
          segment(r0, r1, ns0, sg, p.P, jb, sp0, sp1, slot);
          const int pi = page_of(p.page_indptr, p.page_indices, it.b, jb, p.num_pages, nullptr);
          if (pi < 0) continue;
          const long long off = paged_hnd_offset(pi, sp0 - jb * p.P, it.h, 0, p.P, p.H_kv, D);
          const uint32_t nb = (sp1 - sp0) * kRowBytes;
          bulk_g2s(smem_u32(kt + slot * kRowBytes), kbase + off, nb, fb);
          bulk_g2s(smem_u32(vt + slot * kRowBytes), vbase + off, nb, fb);
        }
      } else {
        for (int s = lane; s < n; s += 32) {
          const int t = pos[s];
          if (t < 0) continue;
          long long off;
          if (paged) {
            const int pi = page_of(p.page_indptr, p.page_indices, it.b, t / p.P, p.num_pages, nullptr);
            off = paged_hnd_offset(pi, t % p.P, it.h, 0, p.P, p.H_kv, D);
          } else {
            off = contig_nhd_offset(c_row, t, it.h, 0, p.T_cap, p.H_kv, D);
          }
          bulk_g2s(smem_u32(kt + s * kRowBytes), kbase + off, kRowBytes, fb);
          bulk_g2s(smem_u32(vt + s * kRowBytes), vbase + off, kRowBytes, fb);
        }
      }
    }
  }
}

// ---- consumers ---------------------------------------------------------------------

template <int D>
__device__ void consume(const PartialParams& p, uint8_t* smem, int it_begin, int it_end, int cw, int lane) {
  using L = Layout<D>;
  constexpr int NCH = D / 64;          // 8-channel chunks per lane
  constexpr int NV = NCH * 4;          // float2 per row per lane
  const int* pos_all = reinterpret_cast<const int*>(smem + L::kPos);
  const int* cls_all = reinterpret_cast<const int*>(smem + L::kCls);
  const uint32_t full0 = smem_u32(smem + L::kFullBar);
  const uint32_t empty0 = smem_u32(smem + L::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  float* scratch = reinterpret_cast<float*>(smem + L::kScratch);

  const int nrb = p.rows <= 4 ? 1 : p.rows <= 8 ? 2 : p.rows <= 16 ? 4 : 8;  // row blocks
  const int nts = kConsumerWarps / nrb;                                        // key slices
  const int rb = cw % nrb, ts = cw / nrb;
  const int keys_per_warp = kTK / nts;                                         // 8 * nrb
  const int tg = lane >> 3, j = lane & 7;
  const int rr = j >> 1;                         // row (within block) this lane reduces to
  const int my_row = rb * 4 + rr;
  const int my_qi = my_row / p.g;                // query index of that row
  const bool my_row_ok = my_row < p.rows;

  uint32_t k = 0;
  bool dead = false;   // a bounded wait gave up: skip work but keep every named barrier
  for (int ii = it_begin; ii < it_end; ++ii) {
    const WorkItem it = p.items[p.cta_items[ii]];
    const MaskCtx mc{p.mask, p.S_q, it.T, p.n_sink, p.window};

    // query rows of this block, pre-scaled by sm_scale * log2(e)
    float2 q[4][NV], o[4][NV];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = rb * 4 + r;
#pragma unroll
      for (int x = 0; x < NV; ++x) o[r][x] = make_float2(0.f, 0.f);
      if (row < p.rows) {
        const int i = row / p.g, hq = it.h * p.g + row % p.g;
        const uint4* qp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) +
                                                         ((static_cast<long long>(it.b) * p.S_q + i) * p.H_q + hq) * D);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          const uint4 w = qp[c * 8 + j];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const float2 f = bf16x2_to_float2(ws[x]);
            q[r][c * 4 + x] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
          }
        }
      } else {
#pragma unroll
        for (int x = 0; x < NV; ++x) q[r][x] = make_float2(0.f, 0.f);
      }
    }
    float m_run = -INFINITY, l_run = 0.f;

    for (int j0 = it.a; j0 < it.e; j0 += kTK, ++k) {
      const int st = k % kStages;
      const uint32_t use = k / kStages;
      if (dead || !mbar_wait(full0 + 8 * st, use & 1, abort_flag, p.status)) {
        dead = true;
        break;
      }
      const int* pos = pos_all + st * kTK;
      const bool stage_full = cls_all[st] == DATTN_TILE_FULL;
      const uint8_t* kt = smem + st * L::kStageBytes;
      const uint8_t* vt = kt + L::kTileBytes;

      for (int sub = 0; sub < nrb; ++sub) {
        float sv[2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int slot = ts * keys_per_warp + sub * 8 + pp * 4 + tg;
          const int t = pos[slot];
          const uint4* krow = reinterpret_cast<const uint4*>(kt + slot * D * 2);
          float2 acc[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 w = krow[c * 8 + j];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float2 kf = bf16x2_to_float2(ws[x]);
#pragma unroll
              for (int r = 0; r < 4; ++r) acc[r] = __ffma2_rn(q[r][c * 4 + x], kf, acc[r]);
            }
          }
          float s[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) s[r] = acc[r].x + acc[r].y;
          // 8-lane reduction: lane j ends with the full score of row j >> 1
          const bool b2 = j & 4, b1 = j & 2;
          float k0 = b2 ? s[2] : s[0], k1 = b2 ? s[3] : s[1];
          const float x0 = b2 ? s[0] : s[2], x1 = b2 ? s[1] : s[3];
          k0 += __shfl_xor_sync(kFull, x0, 4);
          k1 += __shfl_xor_sync(kFull, x1, 4);
          float kk = b1 ? k1 : k0;
          const float xx = b1 ? k0 : k1;
          kk += __shfl_xor_sync(kFull, xx, 2);
          kk += __shfl_xor_sync(kFull, kk, 1);
          bool vis = t >= 0 && my_row_ok;
          if (vis && !stage_full) vis = key_visible(mc, my_qi, t);
          sv[pp] = vis ? kk : -INFINITY;
        }
        // online softmax update for this lane's row over 8 keys of the warp
        float mx = fmaxf(sv[0], sv[1]);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run - m_new);
        const float p0 = sv[0] == -INFINITY ? 0.f : exp2f(sv[0] - m_new);
        const float p1 = sv[1] == -INFINITY ? 0.f : exp2f(sv[1] - m_new);
        l_run = l_run * alpha + p0 + p1;
        m_run = m_new;
        if (__any_sync(kFull, alpha != 1.f)) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = __shfl_sync(kFull, alpha, 2 * r);
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int x = 0; x < NV; ++x) o[r][x] = __fmul2_rn(o[r][x], a2);
          }
        }
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const int slot = ts * keys_per_warp + sub * 8 + pp * 4 + tg;
          const float pv = pp ? p1 : p0;
          float2 pr[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = __shfl_sync(kFull, pv, tg * 8 + 2 * r);
            pr[r] = make_float2(a, a);
          }
          const uint4* vrow = reinterpret_cast<const uint4*>(vt + slot * D * 2);
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const uint4 w = vrow[c * 8 + j];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int x = 0; x < 4; ++x) {
              const float2 vf = bf16x2_to_float2(ws[x]);
#pragma unroll
              for (int r = 0; r < 4; ++r) o[r][c * 4 + x] = __ffma2_rn(pr[r], vf, o[r][c * 4 + x]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }

    // ---- end of item: reduce over the 4 key groups, then across warps ----
    l_run += __shfl_xor_sync(kFull, l_run, 8);
    l_run += __shfl_xor_sync(kFull, l_run, 16);
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int x = 0; x < NV; ++x) {
        o[r][x].x += __shfl_xor_sync(kFull, o[r][x].x, 8);
        o[r][x].y += __shfl_xor_sync(kFull, o[r][x].y, 8);
        o[r][x].x += __shfl_xor_sync(kFull, o[r][x].x, 16);
        o[r][x].y += __shfl_xor_sync(kFull, o[r][x].y, 16);
      }
    float* mine = scratch + cw * (L::kScratchWarp / 4);
    if (tg == 0) {
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int dim = c * 64 + j * 8 + 2 * x;
            mine[r * D + dim] = o[r][c * 4 + x].x;
            mine[r * D + dim + 1] = o[r][c * 4 + x].y;
          }
      if ((j & 1) == 0) {
        mine[4 * D + 2 * rr] = m_run;
        mine[4 * D + 2 * rr + 1] = l_run;
      }
    }
    named_barrier(1, kConsumerWarps * 32);
    const int tid = cw * 32 + lane;
    const int n_out = nrb * 4 * D;
    for (int e = tid; e < n_out; e += kConsumerWarps * 32) {
      const int row_in = e / D, dim = e % D;
      const int b_of = row_in >> 2, r_of = row_in & 3;
      const int row = b_of * 4 + r_of;
      if (row >= p.rows) continue;
      float M = -INFINITY;
      for (int s2 = 0; s2 < nts; ++s2) {
        const float* w = scratch + (b_of + nrb * s2) * (L::kScratchWarp / 4);
        M = fmaxf(M, w[4 * D + 2 * r_of]);
      }
      float Lsum = 0.f, U = 0.f;
      if (M != -INFINITY) {
        for (int s2 = 0; s2 < nts; ++s2) {
          const float* w = scratch + (b_of + nrb * s2) * (L::kScratchWarp / 4);
          const float mw = w[4 * D + 2 * r_of];
          if (mw == -INFINITY) continue;
          const float a = exp2f(mw - M);
          Lsum += a * w[4 * D + 2 * r_of + 1];
          U += a * w[r_of * D + dim];
        }
      }
      const int i = row / p.g, hq = it.h * p.g + row % p.g;
      const long long orow = (static_cast<long long>(it.b) * p.S_q + i) * p.H_q + hq;
      if (it.slot < 0) {
        const float val = Lsum > 0.f ? U / Lsum : 0.f;
        static_cast<__nv_bfloat16*>(p.o)[orow * D + dim] = __float2bfloat16_rn(val);
        if (dim == 0 && p.lse)
          p.lse[orow] = Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
      } else {
        const long long srow = static_cast<long long>(it.slot) * p.rows + row;
        p.u[srow * D + dim] = U;
        if (dim == 0) p.ml[srow] = make_float2(Lsum > 0.f ? M : -INFINITY, Lsum);
      }
    }
    named_barrier(1, kConsumerWarps * 32);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) partial_bf16_kernel(const __grid_constant__ PartialParams p) {
  using L = Layout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // zero the K/V ring so that slots never written hold finite values
  for (int i = threadIdx.x; i < kStages * L::kStageBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(smem + L::kFullBar + 8 * s), 1);
      mbar_init(smem_u32(smem + L::kEmptyBar + 8 * s), kConsumerWarps);
    }
    *reinterpret_cast<int*>(smem + L::kAbort) = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  const int it_begin = p.cta_indptr[blockIdx.x], it_end = p.cta_indptr[blockIdx.x + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kConsumerWarps) {
    produce<D>(p, smem, it_begin, it_end, lane);
  } else {
    consume<D>(p, smem, it_begin, it_end, warp, lane);
  }
}

}  // namespace

size_t partial_smem_bytes(int d, int fmt) {
  (void)fmt;
  return d == 64 ? Layout<64>::kTotal : Layout<128>::kTotal;
}

int launch_partial(const PartialParams& p, int d, int n_ctas, void* stream) {
  const size_t smem = partial_smem_bytes(d, p.fmt);
  cudaError_t err;
  if (d == 64) {
    err = cudaFuncSetAttribute(partial_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    partial_bf16_kernel<64><<<n_ctas, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  } else {
    err = cudaFuncSetAttribute(partial_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    partial_bf16_kernel<128><<<n_ctas, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace dattn
