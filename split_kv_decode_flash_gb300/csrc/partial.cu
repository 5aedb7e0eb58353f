// Partial kernel of split-KV decode attention for the byte formats: INT8
// per-token and KIVI INT4 K/V (bf16 K/V has a tensor-core kernel of its own).
//
// One persistent CTA per SM walks its list of work items (request b, kv head
// h, keys [a, e) of the group's visible stream).
//
// Producer warps.  Every 64-key stage is described per key slot (logical key
// t, physical page pi) one stage ahead, so the dependent loads of the page
// walk (list entry -> page id, M4.5 §0x04D) overlap the wait for a free ring
// slot.  Slots whose keys are consecutive inside one page are merged into one
// run with two warp ballots (the page segments of §0x04E); each run becomes
// one bulk (TMA-engine) copy per tensor into a shared-memory ring guarded by
// mbarriers.  Keys outside the visible stream (SKIP tiles) are never loaded;
// each stage is classified FULL or PARTIAL (§0x05C) so FULL stages skip the
// per-element predicate.  The qparams are staged with the codes: INT8
// per-token (s, z) as 16-byte aligned chunks packed by a warp scan; KIVI the
// per-channel K group qparams and per-token V qparams (M8.6 §0x06A); KIVI
// residual keys come from the bf16 ring in stages of their own.
//
// Eight consumer warps share every K/V tile across the GQA group (§0x03A):
// each warp owns 4 query rows (a row block) and a slice of the stage's keys.
// Lanes form 4 key groups x 8 lanes; a lane holds 16 (d=128) or 8 (d=64)
// channels of its key and of the 4 query rows, so q.k is a handful of packed
// fp32 FMAs plus a 3-step shuffle reduction.  Scales stay where M8.6 §0x03A-C
// puts them: a per-token K scale multiplies the finished dot product, a
// per-channel K scale is applied while dequantising, a per-token V scale is
// folded into the probability and its offset into a per-row sum.  The online
// softmax (§0x02B) runs every 16 keys in log2 units; masked scores are -inf
// before the maximum and the sums.  At the end of an item every warp leaves
// its own fp32 partial state (or O / LSE when it is the group's only state).
#include <cuda_runtime.h>

#include "launch.cuh"
#include "stream.cuh"

namespace dattn {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kMaxKGroups = 6;      // KIVI K groups per stage (G >= 32, at most two runs)
constexpr int kQpEntries = 512;     // INT8 qparam entries per stage and tensor

template <int D, int FMT>
struct Cfg {
  static constexpr bool kI8 = FMT == DATTN_FMT_INT8_TOKEN;
  static constexpr bool kI4 = FMT == DATTN_FMT_INT4_KIVI;
  // Even depth: with two consumer stage groups taking alternate stages, every
  // ring slot then always belongs to the same group, so no group can wait for
  // a slot two phases ahead (mbarrier parity would alias).
  static constexpr int kStagesN = 6;
  static_assert(kStagesN % 2 == 0, "ring depth must be even");
  static constexpr int kTile = kTK * D * 2;                                  // bf16-sized tile
  static constexpr int kKQ = kI8 ? kQpEntries * 4 : kI4 ? kMaxKGroups * D * 4 : 0;
  static constexpr int kVQ = kI8 ? kQpEntries * 4 : kI4 ? kTK * (D / 16) * 4 : 0;
  static constexpr int kStage = 2 * kTile + kKQ + kVQ;
  static constexpr int kPos = kStagesN * kStage;                             // int32 [stages][kTK]
  static constexpr int kQsel = kPos + kStagesN * kTK * 4;                    // int32 [stages][kTK] (quantized)
  static constexpr int kFlags = kQsel + kStagesN * kTK * 4;                  // int32 [stages]
  static constexpr int kSeq = kFlags + kStagesN * 4;                          // int32 [stages]: stage number
  static constexpr int kFullBar = align16(kSeq + kStagesN * 4);
  static constexpr int kEmptyBar = kFullBar + kStagesN * 8;
  static constexpr int kAbort = kEmptyBar + kStagesN * 8;
  static constexpr int kTotal = align16(kAbort + 16);
  static_assert(kTotal <= 232448, "shared memory of one CTA");
  // a lane's channels of a row are contiguous
  static __device__ __forceinline__ int chan(int j, int v) { return (D / 8) * j + 2 * v; }
  static_assert(FMT != DATTN_FMT_BF16, "bf16 K/V use the tensor-core kernel");
};

// Consumer stage groups: with one 4-row block, two groups of four warps take
// alternate stages (16 keys per warp and stage); otherwise all warps share a stage.
__host__ __device__ __forceinline__ int stage_groups(int rows) { return rows <= 4 ? 2 : 1; }

__device__ __forceinline__ float2 u8_pair(uint32_t w, int pair) {
  const uint32_t a = __byte_perm(w, 0x4B000000u, 0x7540u | (2 * pair));
  const uint32_t b = __byte_perm(w, 0x4B000000u, 0x7540u | (2 * pair + 1));
  return __fadd2_rn(make_float2(__uint_as_float(a), __uint_as_float(b)), make_float2(-8388608.f, -8388608.f));
}

__device__ __forceinline__ float2 u4_pair(uint32_t w, int pair) {   // nibbles 2*pair, 2*pair+1
  const uint32_t a = ((w >> (8 * pair)) & 0xFu) | 0x4B000000u;
  const uint32_t b = ((w >> (8 * pair + 4)) & 0xFu) | 0x4B000000u;
  return __fadd2_rn(make_float2(__uint_as_float(a), __uint_as_float(b)), make_float2(-8388608.f, -8388608.f));
}

__device__ __forceinline__ float2 half2_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// ---- producer ---------------------------------------------------------------------

struct Desc {
  int t[2];     // logical key of slots lane, lane + 32 (-1: none)
  int pg[2];    // physical page (paged), cache row (contiguous), 0 (residual)
  int gpg[2];   // KIVI: page holding the key's K-group qparams
  bool whole;   // page-aligned stage of consecutive keys: pg[0] is the page of lane's block
};

// A stage of consecutive keys that starts on a page boundary is described per
// page (one lane per page) instead of per key.
template <int FMT>
__device__ __forceinline__ bool whole_pages(const PartialParams& p, const Cursor& c) {
  return FMT != DATTN_FMT_INT4_KIVI && c.valid && p.layout == DATTN_KV_PAGED_HND &&
         p.mask != DATTN_MASK_INDEX_LIST && p.P_shift >= 1 && p.P <= kTK && c.j1 <= c.it.x0 &&
         (c.j0 & (p.P - 1)) == 0;
}

template <int FMT>
__device__ __forceinline__ Desc describe(const PartialParams& p, const Cursor& c, int lane) {
  Desc d;
  d.whole = whole_pages<FMT>(p, c);
  if (d.whole) {
    const int np = (c.j1 - c.j0 + p.P - 1) >> p.P_shift;
    const int blk = (c.j0 >> p.P_shift) + lane;
    int pg = -1;
    if (lane < np) {
      const int pi = blk < c.hi - c.lo ? p.page_indices[c.lo + blk] : -1;
      pg = (pi >= 0 && pi < p.num_pages) ? pi : -1;
    }
    d.pg[0] = pg;
    d.t[0] = d.t[1] = d.pg[1] = d.gpg[0] = d.gpg[1] = -1;
    return d;
  }
  const bool resid = c.j0 >= c.jq;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    const int j = c.j0 + s;
    int t = -1, pg = -1, gpg = -1;
    if (c.valid && j < c.j1) {
      t = stream_key(c.it, p.mask, p.index_list, j);
      if (p.mask == DATTN_MASK_INDEX_LIST && (t < 0 || t >= c.it.T)) {
        atomicOr(p.status, kStListRange);
        t = -1;
      }
      if (t >= 0) {
        if (resid) {
          pg = 0;
        } else if (p.layout == DATTN_KV_PAGED_HND) {
          const int blk = blk_of(p, t);
          if (blk < c.hi - c.lo) {
            const int pi = p.page_indices[c.lo + blk];
            if (pi >= 0 && pi < p.num_pages) pg = pi;
            else atomicOr(p.status, kStPageRange);
          } else {
            atomicOr(p.status, kStBlockRange);
          }
          if (FMT == DATTN_FMT_INT4_KIVI && pg >= 0) {
            const int gblk = blk_of(p, (t / p.kivi_G) * p.kivi_G);
            const int pi = p.page_indices[c.lo + gblk];
            if (pi >= 0 && pi < p.num_pages) {
              gpg = pi;
            } else {
              atomicOr(p.status, kStPageRange);
              pg = -1;
            }
          }
        } else {
          if (c.crow >= 0 && t < p.T_cap) pg = c.crow;
          else atomicOr(p.status, kStRowRange);
        }
        if (pg < 0) t = -1;
      }
    }
    d.t[h] = t;
    d.pg[h] = pg;
    d.gpg[h] = gpg;
  }
  return d;
}

__device__ __forceinline__ int next_breaker_len(unsigned long long brk, int s) {
  const unsigned long long rest = s < 63 ? brk >> (s + 1) : 0ull;
  return rest ? __ffsll(static_cast<long long>(rest)) : 64 - s;
}

__device__ __forceinline__ unsigned long long ballot64(bool lo, bool hi) {
  return static_cast<unsigned long long>(__ballot_sync(kAll, lo)) |
         (static_cast<unsigned long long>(__ballot_sync(kAll, hi)) << 32);
}

__device__ __forceinline__ int rank_at(unsigned long long mask, int s) {   // set bits at or below s, minus one
  return __popcll(static_cast<long long>(mask & ((2ull << s) - 1ull))) - 1;
}

template <int D, int FMT>
__device__ void produce(const PartialParams& p, uint8_t* smem, int it_begin, int it_end, int lane, int pw) {
  using C = Cfg<D, FMT>;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const uint8_t* kbase = static_cast<const uint8_t*>(p.k);
  const uint8_t* vbase = static_cast<const uint8_t*>(p.v);
  const bool paged = p.layout == DATTN_KV_PAGED_HND;
  constexpr int kRowB = FMT == DATTN_FMT_INT8_TOKEN ? D : D / 2;  // code row bytes

  // producer warp pw fills stages pw, pw + kProducerWarps, ... of the CTA's stage sequence
  Cursor cur;
  cur.ii = it_begin;
  seek(p, cur, it_end, lane);
  for (int i = 0; i < pw; ++i) advance(p, cur, it_end, lane);
  Desc dcur = describe<FMT>(p, cur, lane);
  for (uint32_t k = pw; cur.valid; k += kProducerWarps) {
    Cursor nxt = cur;
    for (int i = 0; i < kProducerWarps; ++i) advance(p, nxt, it_end, lane);
    const Desc dnxt = describe<FMT>(p, nxt, lane);      // loads in flight while we wait

    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) return;
    uint8_t* stage = smem + st * C::kStage;
    uint8_t* kt = stage;
    uint8_t* vt = stage + C::kTile;
    uint8_t* kq = stage + 2 * C::kTile;
    uint8_t* vq = kq + C::kKQ;
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kTK;
    int* qsel = reinterpret_cast<int*>(smem + C::kQsel) + st * kTK;
    const bool resid = cur.j0 >= cur.jq;
    const WorkItem& it = cur.it;

    if (dcur.whole) {
      // whole pages: lane l owns page l of the stage
      const int n = cur.j1 - cur.j0;
      const int np = (n + p.P - 1) >> p.P_shift;
      const int pg = dcur.pg[0];
      const int rows = lane < np ? min(p.P, n - (lane << p.P_shift)) : 0;
      const bool bad = lane < np && pg < 0;
      if (__any_sync(kAll, bad) && lane == 0) atomicOr(p.status, kStPageRange);
      const unsigned badmask = __ballot_sync(kAll, bad);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int s = lane + 32 * h;
        const bool ok = s < n && !((badmask >> (s >> p.P_shift)) & 1u);
        pos[s] = ok ? cur.j0 + s : -1;
        if (FMT == DATTN_FMT_INT8_TOKEN) qsel[s] = s;
      }
      const uint32_t good_rows = __reduce_add_sync(kAll, bad ? 0u : static_cast<uint32_t>(rows));
      uint32_t bytes = good_rows * 2u * kRowB;
      if (FMT == DATTN_FMT_INT8_TOKEN) bytes += 2u * 4u * p.P * __popc(__ballot_sync(kAll, lane < np && !bad));
      int flags = kFlagFull;
      const MaskCtx mc{p.mask, p.S_q, it.T, p.n_sink, p.window};
      for (int i = 0; i < p.S_q; ++i)
        if (visible_in_run(mc, i, cur.j0, cur.j1) != n) flags = 0;
      if (lane == 0) {
        reinterpret_cast<int*>(smem + C::kFlags)[st] = flags;
        reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
      }
      __syncwarp();
      const uint32_t fb = full0 + 8 * st;
      if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
      __syncwarp();
      // Bulk copies issued by one thread complete one after another, so every
      // page slab is cut into row pieces spread over the warp's 32 lanes: lane
      // (page l, tensor z, piece q) copies rows [q rp, (q + 1) rp) of one slab.
      const int per_page = 32 / np;                 // lanes per page (>= 1)
      const bool both = per_page < 2;               // one lane copies both tensors of its page
      const int pieces = both ? 1 : per_page >> 1;  // pieces per tensor slab
      const int l = lane / per_page;
      const int z = both ? 0 : (lane % per_page) / pieces, q = both ? 0 : (lane % per_page) % pieces;
      const int pg_l = __shfl_sync(kAll, pg, min(l, 31));
      const bool bad_l = l < np && ((badmask >> l) & 1u);
      if (l < np && z < 2 && !bad_l) {
        const int rows_l = min(p.P, n - (l << p.P_shift));
        const int rp = (rows_l + pieces - 1) / pieces;
        const int r0 = q * rp, r1 = min(rows_l, r0 + rp);
        const long long prow = (static_cast<long long>(pg_l) * p.H_kv + it.h) << p.P_shift;
        for (int zz = 0; zz < 2; ++zz) {
          if (!both && zz != z) continue;
          if (r1 > r0) {
            const int s = (l << p.P_shift) + r0;
            bulk_g2s(smem_u32((zz ? vt : kt) + s * kRowB), (zz ? vbase : kbase) + (prow + r0) * kRowB,
                     (r1 - r0) * kRowB, fb);
          }
          if (FMT == DATTN_FMT_INT8_TOKEN && q == 0) {
            const uint8_t* qb = static_cast<const uint8_t*>(zz ? p.vqp : p.kqp);
            bulk_g2s(smem_u32((zz ? vq : kq) + (l << p.P_shift) * 4), qb + prow * 4, p.P * 4, fb);
          }
        }
      }
      cur = nxt;
      dcur = dnxt;
      continue;
    }

    // runs of consecutive keys in one page
    const int t0 = dcur.t[0], t1 = dcur.t[1];
    const int up0 = __shfl_up_sync(kAll, t0, 1), up1 = __shfl_up_sync(kAll, t1, 1);
    const int last0 = __shfl_sync(kAll, t0, 31);
    const int prev0 = lane ? up0 : -1, prev1 = lane ? up1 : last0;
    const bool mergeable = paged && !resid;
    const bool cont0 = mergeable && t0 >= 0 && prev0 >= 0 && t0 == prev0 + 1 && row_of(p, t0) != 0;
    const bool cont1 = mergeable && t1 >= 0 && prev1 >= 0 && t1 == prev1 + 1 && row_of(p, t1) != 0;
    const bool st0 = t0 >= 0 && !cont0, st1 = t1 >= 0 && !cont1;
    const unsigned long long brk = ballot64(st0 || t0 < 0, st1 || t1 < 0);
    const unsigned long long starts = ballot64(st0, st1);
    const int nvalid = __popcll(static_cast<long long>(ballot64(t0 >= 0, t1 >= 0)));
    const int len0 = st0 ? next_breaker_len(brk, lane) : 0;
    const int len1 = st1 ? next_breaker_len(brk, lane + 32) : 0;
    pos[lane] = t0;
    pos[lane + 32] = t1;

    uint32_t bytes = 0;
    int qd0 = 0, qd1 = 0, qlo0 = 0, qlo1 = 0;
    if (resid) {
      bytes = static_cast<uint32_t>(nvalid) * 2u * D * 2u;
    } else if (FMT == DATTN_FMT_INT8_TOKEN) {
      // qparam chunks [floor4(r0), ceil4(r0 + len)) packed by an exclusive scan in slot order
      qlo0 = st0 ? row_of(p, t0) & ~3 : 0;
      qlo1 = st1 ? row_of(p, t1) & ~3 : 0;
      const int c0 = st0 ? ((row_of(p, t0) + len0 + 3) & ~3) - qlo0 : 0;
      const int c1 = st1 ? ((row_of(p, t1) + len1 + 3) & ~3) - qlo1 : 0;
      int inc0 = c0, inc1 = c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(kAll, inc0, o), b = __shfl_up_sync(kAll, inc1, o);
        if (lane >= o) inc0 += a, inc1 += b;
      }
      const int tot0 = __shfl_sync(kAll, inc0, 31), tot1 = __shfl_sync(kAll, inc1, 31);
      qd0 = inc0 - c0;
      qd1 = tot0 + inc1 - c1;
      bytes = static_cast<uint32_t>(nvalid) * 2u * kRowB + 2u * 4u * (tot0 + tot1);
      // every valid slot: entry of its row inside its run's chunk
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int s = lane + 32 * h, t = h ? t1 : t0;
        const unsigned long long upto = starts & ((2ull << s) - 1ull);
        const int ss = upto ? 63 - __clzll(static_cast<long long>(upto)) : 0;
        const int dA = __shfl_sync(kAll, qd0, ss & 31), dB = __shfl_sync(kAll, qd1, ss & 31);
        const int lA = __shfl_sync(kAll, qlo0, ss & 31), lB = __shfl_sync(kAll, qlo1, ss & 31);
        if (t >= 0) qsel[s] = ((ss >> 5) ? dB : dA) + row_of(p, t) - ((ss >> 5) ? lB : lA);
      }
    } else {  // KIVI quantized stage: one K-group qparam row per distinct group
      const int g0 = t0 >= 0 ? t0 / p.kivi_G : -1, g1 = t1 >= 0 ? t1 / p.kivi_G : -1;
      const int gu0 = __shfl_up_sync(kAll, g0, 1), gu1 = __shfl_up_sync(kAll, g1, 1);
      const int gl0 = __shfl_sync(kAll, g0, 31);
      const int gp0 = lane ? gu0 : -1, gp1 = lane ? gu1 : gl0;
      const bool gs0 = g0 >= 0 && g0 != gp0, gs1 = g1 >= 0 && g1 != gp1;
      const unsigned long long gst = ballot64(gs0, gs1);
      const int ng = min(kMaxKGroups, __popcll(static_cast<long long>(gst)));
      if (__popcll(static_cast<long long>(gst)) > kMaxKGroups && lane == 0) atomicOr(p.status, kStRowRange);
      if (t0 >= 0) qsel[lane] = min(kMaxKGroups - 1, rank_at(gst, lane));
      if (t1 >= 0) qsel[lane + 32] = min(kMaxKGroups - 1, rank_at(gst, lane + 32));
      bytes = static_cast<uint32_t>(nvalid) * (2u * kRowB + (D / p.kivi_Gv) * 4u) + static_cast<uint32_t>(ng) * D * 4u;
      qd0 = gs0 ? rank_at(gst, lane) : -1;
      qd1 = gs1 ? rank_at(gst, lane + 32) : -1;
    }

    // stage class
    int flags = resid ? kFlagResidual : 0;
    const bool full = stage_is_full(p, cur.it, p.S_q, cur.j0, cur.j1, t0, t1);
    if (full) flags |= kFlagFull;
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = flags;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    __syncwarp();
    const uint32_t fb = full0 + 8 * st;
    if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
    __syncwarp();

    // copies, one per run and tensor
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const bool is_start = h ? st1 : st0;
      if (!is_start) continue;
      const int s = lane + 32 * h;
      const int t = h ? t1 : t0, pg = h ? dcur.pg[1] : dcur.pg[0];
      const int len = h ? len1 : len0;
      if (resid) {
        const long long off = ((static_cast<long long>(it.b) * p.kivi_R + t % p.kivi_R) * p.H_kv + it.h) * D;
        bulk_g2s(smem_u32(kt + s * D * 2), static_cast<const __nv_bfloat16*>(p.kres) + off, D * 2, fb);
        bulk_g2s(smem_u32(vt + s * D * 2), static_cast<const __nv_bfloat16*>(p.vres) + off, D * 2, fb);
        continue;
      }
      const long long row = paged ? (static_cast<long long>(pg) * p.H_kv + it.h) * p.P + row_of(p, t)
                                  : (static_cast<long long>(pg) * p.T_cap + t) * p.H_kv + it.h;
      const uint32_t nb = static_cast<uint32_t>(len) * kRowB;
      bulk_g2s(smem_u32(kt + s * kRowB), kbase + row * kRowB, nb, fb);
      bulk_g2s(smem_u32(vt + s * kRowB), vbase + row * kRowB, nb, fb);
      if (FMT == DATTN_FMT_INT8_TOKEN) {
        const int qlo = h ? qlo1 : qlo0, qd = h ? qd1 : qd0;
        const int cn = ((row_of(p, t) + len + 3) & ~3) - qlo;
        const long long qrow = (static_cast<long long>(pg) * p.H_kv + it.h) * p.P + qlo;
        bulk_g2s(smem_u32(kq + qd * 4), static_cast<const uint8_t*>(p.kqp) + qrow * 4, cn * 4, fb);
        bulk_g2s(smem_u32(vq + qd * 4), static_cast<const uint8_t*>(p.vqp) + qrow * 4, cn * 4, fb);
      }
      if (FMT == DATTN_FMT_INT4_KIVI) {
        const int vqb = (D / p.kivi_Gv) * 4;
        bulk_g2s(smem_u32(vq + s * vqb), static_cast<const uint8_t*>(p.vqp) + row * vqb, len * vqb, fb);
      }
    }
    if (FMT == DATTN_FMT_INT4_KIVI && !resid) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int gi = h ? qd1 : qd0;
        if (gi < 0 || gi >= kMaxKGroups) continue;
        const int t = h ? t1 : t0, gpg = h ? dcur.gpg[1] : dcur.gpg[0];
        const int g0 = (t / p.kivi_G) * p.kivi_G;
        const int slots = p.P >= p.kivi_G ? p.P / p.kivi_G : 1;
        const int slot = p.P >= p.kivi_G ? (g0 % p.P) / p.kivi_G : 0;
        const long long qrow = (static_cast<long long>(gpg) * p.H_kv + it.h) * slots + slot;
        bulk_g2s(smem_u32(kq + gi * D * 4), static_cast<const uint8_t*>(p.kqp) + qrow * D * 4, D * 4, fb);
      }
    }
    cur = nxt;
    dcur = dnxt;
  }
}

// ---- consumers ---------------------------------------------------------------------

template <int D, int FMT>
__device__ void consume(const PartialParams& p, uint8_t* smem, int it_begin, int it_end, int cw, int lane) {
  using C = Cfg<D, FMT>;
  constexpr int NV = D / 16;             // float2 per row per lane
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);

  // Warps are split into stage groups that take turns on the ring's stages, row
  // blocks of 4 query rows, and key slices of at least 16 keys per stage.
  const int nrb = p.rows <= 4 ? 1 : p.rows <= 8 ? 2 : p.rows <= 16 ? 4 : 8;  // row blocks
  const int ng = stage_groups(p.rows);                                         // stage groups
  const int wps = kConsumerWarps / ng;                                         // warps per stage
  const int sgrp = cw / wps, wi = cw % wps;
  const int rb = wi % nrb, ts = wi / nrb;
  const int nts = wps / nrb;                                                   // key slices
  const int keys_per_warp = kTK / nts;                                         // 16, 32 or 64
  const int tg = lane >> 3, j = lane & 7;
  const int rr = j >> 1;
  const int my_row = rb * 4 + rr;
  const int my_qi = my_row / p.g;
  const bool my_row_ok = my_row < p.rows;
  const int vgroup = C::kI4 ? (D / 8) * j / p.kivi_Gv : 0;     // lane's V channel group (KIVI)
  const int my_state = (cw - rb) / nrb;                         // this warp's state among them

  uint32_t k = 0;
  bool dead = false;   // a bounded wait gave up: skip work but keep every named barrier
  for (int ii = it_begin; ii < it_end; ++ii) {
    const WorkItem it = read_item(p, p.cta_items[ii], false);
    const int jq = residual_start(p, it);
    const MaskCtx mc{p.mask, p.S_q, it.T, p.n_sink, p.window};

    float2 q[4][NV], o[4][NV];
    float zacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = rb * 4 + r;
#pragma unroll
      for (int x = 0; x < NV; ++x) o[r][x] = make_float2(0.f, 0.f);
      if (row < p.rows) {
        const int i = row / p.g, hq = it.h * p.g + row % p.g;
        const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(p.q) +
                                  ((static_cast<long long>(it.b) * p.S_q + i) * p.H_q + hq) * D;
#pragma unroll
        for (int x = 0; x < NV; x += 4) {
          const uint4 w = *reinterpret_cast<const uint4*>(qp + C::chan(j, x));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const float2 f = bf16x2_to_float2(ws[y]);
            q[r][x + y] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
          }
        }
      } else {
#pragma unroll
        for (int x = 0; x < NV; ++x) q[r][x] = make_float2(0.f, 0.f);
      }
    }
    float qsum_my = 0.f;      // INT8: sum of the row's scaled query channels
    if (C::kI8) {
      float qs[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float a = 0.f;
#pragma unroll
        for (int x = 0; x < NV; ++x) a += q[r][x].x + q[r][x].y;
        a += __shfl_xor_sync(kAll, a, 1);
        a += __shfl_xor_sync(kAll, a, 2);
        a += __shfl_xor_sync(kAll, a, 4);
        qs[r] = a;
      }
      qsum_my = rr == 0 ? qs[0] : rr == 1 ? qs[1] : rr == 2 ? qs[2] : qs[3];
    }
    float2 ks[NV], kz[NV];    // KIVI: per-channel K scale / offset of the current group
    int cur_gid = -1;
#pragma unroll
    for (int x = 0; x < NV; ++x) ks[x] = kz[x] = make_float2(0.f, 0.f);

    float m_run = -INFINITY, l_run = 0.f;
    for (int j0 = it.a; j0 < it.e; ++k) {
      const int j1 = stage_end(it, j0, jq);
      if (static_cast<int>(k % ng) != sgrp) {     // the other stage group's turn
        j0 = j1;
        continue;
      }
      const int st = k % C::kStagesN;
      const uint32_t use = k / C::kStagesN;
      if (dead || !mbar_wait(full0 + 8 * st, use & 1, abort_flag, p.status)) {
        dead = true;
        break;
      }
      if (reinterpret_cast<const volatile int*>(smem + C::kSeq)[st] != static_cast<int>(k)) {
        if (lane == 0) atomicOr(p.status, kStPipeline);   // wrong phase: stop, never consume stale data
        *abort_flag = 1;
        dead = true;
        break;
      }
      const uint8_t* stage = smem + st * C::kStage;
      const uint8_t* kt = stage;
      const uint8_t* vt = stage + C::kTile;
      const uint8_t* kqs = stage + 2 * C::kTile;
      const uint8_t* vqs = kqs + C::kKQ;
      const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kTK;
      const int* qsel = reinterpret_cast<const int*>(smem + C::kQsel) + st * kTK;
      const int flags = reinterpret_cast<const int*>(smem + C::kFlags)[st];
      const bool stage_full = flags & kFlagFull;
      const bool resid = flags & kFlagResidual;

      for (int sub = 0; sub < keys_per_warp / 16; ++sub) {
        float sv[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int slot = ts * keys_per_warp + sub * 16 + pp * 4 + tg;
          const int t = pos[slot];
          float2 acc[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[r] = make_float2(0.f, 0.f);
          if (resid) {
            const __nv_bfloat16* krow = reinterpret_cast<const __nv_bfloat16*>(kt) + slot * D;
#pragma unroll
            for (int x = 0; x < NV; x += 4) {
              const uint4 w = *reinterpret_cast<const uint4*>(krow + C::chan(j, x));
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                const float2 kf = bf16x2_to_float2(ws[y]);
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = __ffma2_rn(q[r][x + y], kf, acc[r]);
              }
            }
          } else if (C::kI8) {
            const uint8_t* krow = kt + slot * D + (D / 8) * j;
#pragma unroll
            for (int x = 0; x < NV; x += 2) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(krow + 2 * x);
#pragma unroll
              for (int y = 0; y < 2; ++y) {
                const float2 kf = u8_pair(w, y);
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = __ffma2_rn(q[r][x + y], kf, acc[r]);
              }
            }
          } else {  // KIVI quantized key: per-channel dequantisation inside the dot
            if (t >= 0 && t / p.kivi_G != cur_gid) {
              cur_gid = t / p.kivi_G;
              const uint32_t* g = reinterpret_cast<const uint32_t*>(kqs + qsel[slot] * D * 4) + (D / 8) * j;
#pragma unroll
              for (int x = 0; x < NV; ++x) {
                const float2 a = half2_to_float2(g[2 * x]), b = half2_to_float2(g[2 * x + 1]);
                ks[x] = make_float2(a.x, b.x);
                kz[x] = make_float2(a.y, b.y);
              }
            }
            const uint8_t* krow = kt + slot * (D / 2) + (D / 16) * j;
#pragma unroll
            for (int x = 0; x < NV; x += 4) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(krow + x);   // 8 nibbles
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                const float2 kf = __ffma2_rn(u4_pair(w, y), ks[x + y], kz[x + y]);
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = __ffma2_rn(q[r][x + y], kf, acc[r]);
              }
            }
          }
          float s[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) s[r] = acc[r].x + acc[r].y;
          // 8-lane reduction: lane j ends with the full dot product of row j >> 1
          const bool b2 = j & 4, b1 = j & 2;
          float k0 = b2 ? s[2] : s[0], k1 = b2 ? s[3] : s[1];
          const float x0 = b2 ? s[0] : s[2], x1 = b2 ? s[1] : s[3];
          k0 += __shfl_xor_sync(kAll, x0, 4);
          k1 += __shfl_xor_sync(kAll, x1, 4);
          float kk = b1 ? k1 : k0;
          const float xx = b1 ? k0 : k1;
          kk += __shfl_xor_sync(kAll, xx, 2);
          kk += __shfl_xor_sync(kAll, kk, 1);
          if (C::kI8 && !resid && t >= 0) {         // per-token K scale outside the dot
            const float2 sz = half2_to_float2(reinterpret_cast<const uint32_t*>(kqs)[qsel[slot]]);
            kk = fmaf(sz.x, kk, sz.y * qsum_my);
          }
          bool vis = t >= 0 && my_row_ok;
          if (vis && !stage_full) vis = key_visible(mc, my_qi, t);
          sv[pp] = vis ? kk : -INFINITY;
        }
        // online softmax update for this lane's row over 16 keys of the warp
        float mx = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
        mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = m_new == -INFINITY ? 1.f : ex2_approx(m_run - m_new);
        float pk[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) pk[pp] = sv[pp] == -INFINITY ? 0.f : ex2_approx(sv[pp] - m_new);
        l_run = l_run * alpha + ((pk[0] + pk[1]) + (pk[2] + pk[3]));
        m_run = m_new;
        if (__any_sync(kAll, alpha != 1.f)) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float a = __shfl_sync(kAll, alpha, 2 * r);
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int x = 0; x < NV; ++x) o[r][x] = __fmul2_rn(o[r][x], a2);
            zacc[r] *= a;
          }
        }
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int slot = ts * keys_per_warp + sub * 16 + pp * 4 + tg;
          const float pv = pk[pp];
          float pr[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) pr[r] = __shfl_sync(kAll, pv, tg * 8 + 2 * r);
          if (resid) {
            // a KIVI residual stage may hold stale code bytes (not bf16) in its unused slots
            if (C::kI4 && pos[slot] < 0) continue;
            const __nv_bfloat16* vrow = reinterpret_cast<const __nv_bfloat16*>(vt) + slot * D;
#pragma unroll
            for (int x = 0; x < NV; x += 4) {
              const uint4 w = *reinterpret_cast<const uint4*>(vrow + C::chan(j, x));
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                const float2 vf = bf16x2_to_float2(ws[y]);
#pragma unroll
                for (int r = 0; r < 4; ++r) o[r][x + y] = __ffma2_rn(make_float2(pr[r], pr[r]), vf, o[r][x + y]);
              }
            }
          } else {
            // per-token V scale folded into the probability, offset into a per-row sum
            float2 sz = make_float2(0.f, 0.f);
            if (pos[slot] >= 0) {
              if (C::kI8) sz = half2_to_float2(reinterpret_cast<const uint32_t*>(vqs)[qsel[slot]]);
              else sz = half2_to_float2(reinterpret_cast<const uint32_t*>(vqs)[slot * (D / p.kivi_Gv) + vgroup]);
            }
            float2 ps[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              ps[r] = make_float2(pr[r] * sz.x, pr[r] * sz.x);
              zacc[r] = fmaf(pr[r], sz.y, zacc[r]);
            }
            if (C::kI8) {
              const uint8_t* vrow = vt + slot * D + (D / 8) * j;
#pragma unroll
              for (int x = 0; x < NV; x += 2) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow + 2 * x);
#pragma unroll
                for (int y = 0; y < 2; ++y) {
                  const float2 vf = u8_pair(w, y);
#pragma unroll
                  for (int r = 0; r < 4; ++r) o[r][x + y] = __ffma2_rn(ps[r], vf, o[r][x + y]);
                }
              }
            } else {
              const uint8_t* vrow = vt + slot * (D / 2) + (D / 16) * j;
#pragma unroll
              for (int x = 0; x < NV; x += 4) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow + x);
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                  const float2 vf = u4_pair(w, y);
#pragma unroll
                  for (int r = 0; r < 4; ++r) o[r][x + y] = __ffma2_rn(ps[r], vf, o[r][x + y]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      j0 = j1;
    }

    // ---- end of item: reduce over the 4 key groups and leave this warp's state ----
    l_run += __shfl_xor_sync(kAll, l_run, 8);
    l_run += __shfl_xor_sync(kAll, l_run, 16);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      zacc[r] += __shfl_xor_sync(kAll, zacc[r], 8);
      zacc[r] += __shfl_xor_sync(kAll, zacc[r], 16);
#pragma unroll
      for (int x = 0; x < NV; ++x) {
        o[r][x].x += __shfl_xor_sync(kAll, o[r][x].x, 8);
        o[r][x].y += __shfl_xor_sync(kAll, o[r][x].y, 8);
        o[r][x].x += __shfl_xor_sync(kAll, o[r][x].x, 16);
        o[r][x].y += __shfl_xor_sync(kAll, o[r][x].y, 16);
      }
    }
    // every key group now holds the totals; key group tg writes row tg of the block
    const float m_mine = __shfl_sync(kAll, m_run, 2 * tg);      // row tg's (m, l) live in lane 2 tg
    const float l_mine = __shfl_sync(kAll, l_run, 2 * tg);
    const int row = rb * 4 + tg;
    float2 ov[NV];
#pragma unroll
    for (int x = 0; x < NV; ++x) {
      const float2 v = tg == 0 ? o[0][x] : tg == 1 ? o[1][x] : tg == 2 ? o[2][x] : o[3][x];
      const float z = tg == 0 ? zacc[0] : tg == 1 ? zacc[1] : tg == 2 ? zacc[2] : zacc[3];
      ov[x] = make_float2(v.x + z, v.y + z);
    }
    if (row < p.rows && !dead) {
      const int i = row / p.g, hq = it.h * p.g + row % p.g;
      const long long orow = (static_cast<long long>(it.b) * p.S_q + i) * p.H_q + hq;
      if (it.slot < 0) {        // single state for the row: final output
        const float inv = l_mine > 0.f ? 1.f / l_mine : 0.f;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
        for (int x = 0; x < NV; ++x)
          *reinterpret_cast<__nv_bfloat162*>(out + C::chan(j, x)) = __floats2bfloat162_rn(ov[x].x * inv, ov[x].y * inv);
        if (j == 0 && p.lse)
          p.lse[orow] = l_mine > 0.f ? (m_mine + __log2f(l_mine)) * 0.69314718055994531f : -INFINITY;
      } else {
        const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
        float* u = p.u + srow * D;
#pragma unroll
        for (int x = 0; x < NV; x += 2)
          *reinterpret_cast<float4*>(u + C::chan(j, x)) = make_float4(ov[x].x, ov[x].y, ov[x + 1].x, ov[x + 1].y);
        if (j == 0) p.ml[srow] = make_float2(l_mine > 0.f ? m_mine : -INFINITY, l_mine);
      }
    } else if (row < p.rows && dead && it.slot >= 0 && j == 0) {   // the warp gave up: its state is marked
      mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + row);
    }
  }
}

template <int D, int FMT>
__global__ void __launch_bounds__(kThreads, 1) partial_kernel(const __grid_constant__ PartialParams p) {
  using C = Cfg<D, FMT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // zero the ring so that slots never written hold finite values
  for (int i = threadIdx.x; i < C::kStagesN * C::kStage / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesN; ++s) {
      mbar_init(smem_u32(smem + C::kFullBar + 8 * s), 1);
      mbar_init(smem_u32(smem + C::kEmptyBar + 8 * s), kConsumerWarps / stage_groups(p.rows));
    }
    *reinterpret_cast<int*>(smem + C::kAbort) = 0;
    *reinterpret_cast<uint64_t*>(smem + C::kAbort + 8) = p.wait_ns;   // read by the bounded waits
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  __syncthreads();
  const int it_begin = p.cta_indptr[blockIdx.x], it_end = p.cta_indptr[blockIdx.x + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kConsumerWarps) {
    // the producer warpgroup hands registers to the consumers; one warp produces
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    produce<D, FMT>(p, smem, it_begin, it_end, lane, warp - kConsumerWarps);
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
  consume<D, FMT>(p, smem, it_begin, it_end, warp, lane);
}

template <int D, int FMT>
int launch_one(const PartialParams& p, int n_ctas, void* stream) {
  const size_t smem = Cfg<D, FMT>::kTotal;
  // the register budget check and the shared-memory opt-in, once per device
  static std::atomic<unsigned long long> ready{0};
  cudaError_t err = prepare_kernel_once(partial_kernel<D, FMT>, smem, 128 * kProducerRegs + 32 * kConsumerWarps * kConsumerRegs, ready);
  if (err != cudaSuccess) return err;
  partial_kernel<D, FMT><<<n_ctas, kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError();
}

}  // namespace

int launch_partial(const PartialParams& p, int d, int n_ctas, void* stream) {
  if (p.fmt == DATTN_FMT_BF16) return launch_partial_bf16(p, d, n_ctas, stream);
  if (p.fmt == DATTN_FMT_INT8_TOKEN || p.fmt == DATTN_FMT_FP8_E4M3 || p.fmt == DATTN_FMT_FP8_E5M2)
    return launch_partial_q8(p, d, n_ctas, stream);
  if (p.fmt == DATTN_FMT_INT4_HEAD) return launch_partial_q4h(p, d, n_ctas, stream);
  if (kivi_on_tensor_cores(d, p.rows, p.kivi_Gv, p.mask, p.P, p.kivi_R)) return launch_partial_q4(p, d, n_ctas, stream);
  return d == 64 ? launch_one<64, DATTN_FMT_INT4_KIVI>(p, n_ctas, stream)
                 : launch_one<128, DATTN_FMT_INT4_KIVI>(p, n_ctas, stream);
}

}  // namespace dattn
