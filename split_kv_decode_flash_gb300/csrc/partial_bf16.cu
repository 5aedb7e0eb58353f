// Partial kernel of split-KV decode attention for bf16 K/V, on the tensor
// cores.
//
// One persistent CTA per SM walks its list of work items (request b, kv head
// h, keys [a, e) of the group's visible stream), as in the byte-format
// kernel; only the data movement and the arithmetic differ.
//
// Producer warps (4).  Warp w fills stages w, w + 4, ... of the CTA's stage
// sequence.  A stage holds 64 key slots; each slot is described one stage
// ahead by the logical key and its K/V row in the cache (the page walk of
// M4.5 §0x04D, or the contiguous row with cache_batch_idx, §0x04A).  Every
// key row is then copied with 16-byte cp.async operations (one warp
// instruction moves two 256-byte rows) into a shared-memory ring whose
// 16-byte chunks are XOR-swizzled by the slot's low three bits, so the
// ldmatrix reads of the consumers never meet a bank conflict.  Empty slots
// (stage tail, a key outside the cache) are zero-filled by the same copy
// with a zero source size, so masked keys hold finite values.  Completion is
// tracked by cp.async.mbarrier.arrive on the stage's full barrier; the ring
// is guarded by full / empty mbarriers with bounded waits.
//
// Consumer warps (8).  The query rows of the group (g * S_q <= 32, the GQA
// rows that share each K/V row, M4.5 §0x03A) form the M side of
// mma.sync.m16n8k16 bf16 tiles (one tile of 16 rows, two for 32 rows).  A
// warp takes 16 keys of a stage:
//   S (16 rows x 16 keys) = Q K^T: K fragments by ldmatrix, fp32 accumulate;
//   masked cells -> -inf, online softmax in log2 units (§0x02B) on the
//   accumulator fragments, row maxima over the lane quad;
//   O (16 rows x d) += P V: the S accumulators re-packed as the bf16 A
//   operand, V fragments by ldmatrix.trans.
// With one row tile, two groups of four warps take alternate stages.  At the
// end of an item every warp leaves its own fp32 state (m, l, u) per row, or
// O / LSE when it is the group's only state.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "merge.cuh"
#include "tc_common.cuh"

namespace dattn {

namespace {

// setmaxnreg split of the launch's 384 x 168 registers: the producer
// warpgroup's description pipeline needs more than the byte-format kernel's.
constexpr int kBfProducerRegs = 96;
constexpr int kBfConsumerRegs = 200;
static_assert(128 * kBfProducerRegs + 32 * kConsumerWarps * kBfConsumerRegs <= kThreads * 168, "register split");

template <int D>
struct Bf {
  // Even depth: with two consumer stage groups taking alternate stages, every
  // ring slot then always belongs to the same group (no mbarrier parity alias).
  static constexpr int kStagesN = 6;
  static_assert(kStagesN % 2 == 0, "ring depth must be even");
  static constexpr int kRowB = D * 2;              // bytes of one key row
  static constexpr int kChunks = kRowB / 16;       // 16-byte chunks per row
  static constexpr int kTile = kTK * kRowB;        // one tensor's stage tile
  static constexpr int kStage = 2 * kTile;
  static constexpr int kPos = kStagesN * kStage;   // int32 [stages][kTK]: logical key or -1
  static constexpr int kVis = kPos + kStagesN * kTK * 4;   // uint32 [stages][kTK]: FlashMask row bits
  static constexpr int kFlags = kVis + kStagesN * kTK * 4;
  static constexpr int kSeq = kFlags + kStagesN * 4;   // int32 [stages]: stage number
  static constexpr int kFullBar = align16(kSeq + kStagesN * 4);
  static constexpr int kEmptyBar = kFullBar + kStagesN * 8;
  static constexpr int kAbort = kEmptyBar + kStagesN * 8;
  static constexpr int kItems = align16(kAbort + 16);   // ItemRec [kItemCache]
  static constexpr int kTotal = kItems + kItemCache * static_cast<int>(sizeof(ItemRec));
  static_assert(kTotal <= 232448, "shared memory of one CTA");
};


// HK: the instance with the timeline stamps and the skipped-arrival test hook
// (launched only when a run asks for either; the plain instance has neither).
template <int D, bool FM, bool HK>
__device__ void produce_bf16(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Bf<D>;
  const PartialParams& p = w.p;
  constexpr int kSlotsPerPass = 32 / C::kChunks;   // key rows per warp instruction
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const int sub = lane / C::kChunks, ch = lane % C::kChunks;
  const uint64_t stream_pol = policy_evict_first();

  // this warp's stages: pw, pw + 4, pw + 8, ... of the CTA's stage sequence
  PCur c0{w.begin, 0, 0};
  pc_seek<kTK>(w, c0);
  pc_advance<kTK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kTK>(w, c1, kProducerWarps);
  PCur c2 = c1;
  pc_advance<kTK>(w, c2, kProducerWarps);
  if constexpr (!FM)   // index lists: list entries are device inputs
    index_list_prologue<2>(w, c0, lane, dep_wait, kbase, vbase, C::kRowB);
  const SlotKeys<2> k0 = slot_keys<2, !FM>(w, c0, lane);
  SlotKeys<2> k1 = slot_keys<2, !FM>(w, c1, lane);
  SlotKeys<2> k2 = slot_keys<2, !FM>(w, c2, lane);
  // Up to here only the plan was read; the page table is a device input.
  dependency_wait(dep_wait);
  if constexpr (HK) {
    if (pw == 0 && lane == 0) trace_stamp(p, kTrWaitDone);
  }
  const SlotPages<2, FM> g0 = slot_pages<2, FM>(w, c0, k0);     // both stages' page lookups in flight together
  SlotPages<2, FM> g1 = slot_pages<2, FM>(w, c1, k1);
  SlotRows<2, FM> r0 = slot_rows<2, FM, true>(w, c0, k0, g0, lane);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kTK;
    pos[lane] = r0.t[0];
    pos[lane + 32] = r0.t[1];
    if constexpr (FM) {
      uint32_t* vis = reinterpret_cast<uint32_t*>(smem + C::kVis) + st * kTK;
      vis[lane] = r0.vis[0];
      vis[lane + 32] = r0.vis[1];
    }
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = r0.full ? kFlagFull : 0;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
#pragma unroll
    for (int s0 = 0; s0 < kTK; s0 += kSlotsPerPass) {
      const int s = s0 + sub;
      const uint32_t row = __shfl_sync(kAll, s0 < 32 ? r0.row[0] : r0.row[1], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = tile_off<2 * D>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
    const uint32_t fb = full0 + 8 * st;
    if (!(HK && p.skip_arrival && blockIdx.x == 0 && k == 0)) {   // the test hook withholds stage 0 of CTA 0
      cp_async_mbar_arrive(fb);
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);   // publishes pos / flags / stamp; the copies complete the phase
    }
    if constexpr (HK) {
      if (k == 0 && lane == 0) trace_stamp(p, kTrFirstCopy);
    }

    // move the description pipeline one stage of this warp forward
    r0 = slot_rows<2, FM, true>(w, c1, k1, g1, lane);
    c0 = c1;
    g1 = slot_pages<2, FM>(w, c2, k2);
    k1 = k2;
    c1 = c2;
    pc_advance<kTK>(w, c2, kProducerWarps);
    k2 = slot_keys<2, !FM>(w, c2, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

// The same producer for interval programs on power-of-two pages (not
// FlashMask): one page id per lane and stage instead of a key, a page-table
// load and a row per slot (RunStage in tc_common.cuh).
template <int D, bool HK>
__device__ void produce_bf16_runs(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Bf<D>;
  const PartialParams& p = w.p;
  constexpr int kSlotsPerPass = 32 / C::kChunks;   // key rows per warp instruction
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const int sub = lane / C::kChunks, ch = lane % C::kChunks;
  const uint64_t stream_pol = policy_evict_first();

  PCur c0{w.begin, 0, 0};
  pc_seek<kTK>(w, c0);
  pc_advance<kTK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kTK>(w, c1, kProducerWarps);
  RunStage s0 = run_stage(w, c0);
  RunStage s1 = run_stage(w, c1);
  if (dep_wait) {   // this warp's first two stages go into L2
    const RunHint h0 = run_hint(w, s0, lane), h1 = run_hint(w, s1, lane);
    prefetch_run(p, h0, kbase, vbase, C::kRowB);
    prefetch_run(p, h1, kbase, vbase, C::kRowB);
  }
  dependency_wait(dep_wait);   // the page table is a device input
  if constexpr (HK) {
    if (pw == 0 && lane == 0) trace_stamp(p, kTrWaitDone);
  }
  StagePage g0 = run_stage_page(w, s0, lane);
  StagePage g1 = run_stage_page(w, s1, lane);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    const ItemRec rec = w.rec(c0.ii);
    const int pid0 = check_stage_page(p, g0);   // loaded a stage ago
    if constexpr (HK) {
      if (k == 0 && lane == 0) trace_stamp(p, kTrFirstPage);
    }
    uint32_t rows[2];
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kTK;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int t;
      run_slot(p, s0, rec.it.T, rec.it.h, pid0, lane + 32 * h, t, rows[h]);
      pos[lane + 32 * h] = t;
    }
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = s0.full ? kFlagFull : 0;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
#pragma unroll
    for (int s0i = 0; s0i < kTK; s0i += kSlotsPerPass) {
      const int s = s0i + sub;
      const uint32_t row = __shfl_sync(kAll, s0i < 32 ? rows[0] : rows[1], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = tile_off<2 * D>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
    const uint32_t fb = full0 + 8 * st;
    if (!(HK && p.skip_arrival && blockIdx.x == 0 && k == 0)) {   // the test hook withholds stage 0 of CTA 0
      cp_async_mbar_arrive(fb);
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);   // publishes pos / flags / stamp; the copies complete the phase
    }
    if constexpr (HK) {
      if (k == 0 && lane == 0) trace_stamp(p, kTrFirstCopy);
    }

    c0 = c1;
    s0 = s1;
    g0 = g1;
    pc_advance<kTK>(w, c1, kProducerWarps);
    s1 = run_stage(w, c1);
    g1 = run_stage_page(w, s1, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

// ---- consumers --------------------------------------------------------------------------

// Writes one query row of a warp's result: O / LSE when the item is its
// group's only state, else the row's partial state (m in log2 units, l, u).
// qo: the request's first packed query row.
template <int D>
__device__ __forceinline__ void emit_row(const PartialParams& p, const WorkItem& it, int qo, int my_state, int row,
                                         float m, float l, const float (&o)[D / 8][4], int half, int t4) {
  const int i = row / p.g, hq = it.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(qo) + i) * p.H_q + hq;
  if (it.slot < 0) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<__nv_bfloat162*>(out + 8 * n + 2 * t4) =
          __floats2bfloat162_rn(o[n][2 * half] * inv, o[n][2 * half + 1] * inv);
    if (t4 == 0 && p.lse) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
  } else {
    const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
    float* u = p.u + srow * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
      *reinterpret_cast<float2*>(u + 8 * n + 2 * t4) = make_float2(o[n][2 * half], o[n][2 * half + 1]);
    if (t4 == 0) p.ml[srow] = make_float2(l > 0.f ? m : -INFINITY, l);
  }
}

// The two accumulator rows r0, r1 of a lane, for item record "r", as mma A
// fragments (rows past the request's g C_b rows are zero).
template <int D>
__device__ __forceinline__ void load_q(const PartialParams& p, const ItemRec& r, int r0, int r1, int t4,
                                       uint32_t (&qa)[D / 16][4]) {
  const bool ok0 = r0 < p.g * r.nq, ok1 = r1 < p.g * r.nq;
  const uint32_t* q0 = static_cast<const uint32_t*>(p.q) +
                       ((static_cast<long long>(r.qo) + r0 / p.g) * p.H_q + r.it.h * p.g + r0 % p.g) * (D / 2);
  const uint32_t* q1 = static_cast<const uint32_t*>(p.q) +
                       ((static_cast<long long>(r.qo) + r1 / p.g) * p.H_q + r.it.h * p.g + r1 % p.g) * (D / 2);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    qa[kk][0] = ok0 ? q0[8 * kk + t4] : 0u;
    qa[kk][1] = ok1 ? q1[8 * kk + t4] : 0u;
    qa[kk][2] = ok0 ? q0[8 * kk + 4 + t4] : 0u;
    qa[kk][3] = ok1 ? q1[8 * kk + 4 + t4] : 0u;
  }
}

// A consumer warp's part of an item.  Two stage groups of four warps take
// alternate stages.  KW = 16: one row block of 16 query rows, each warp owns
// 16 keys of its stages (8 states per row).  KW = 32: two row blocks (17 to
// 32 rows) times two key halves, each warp owns 32 keys, so that its S
// accumulation runs as four independent mma chains and one softmax update
// covers 32 keys (4 states per row).
template <int KW>
struct WarpRole {
  static_assert(KW == 16 || KW == 32, "keys per warp");
  static constexpr int nrb = KW == 16 ? 1 : 2;
  int sgrp, rb, ts, my_state, r0, r1;
  __device__ __forceinline__ WarpRole(int cw, int lane) {
    constexpr int wps = kConsumerWarps / 2;
    sgrp = cw / wps;
    const int wi = cw % wps;
    rb = wi % nrb;
    ts = wi / nrb;
    my_state = (cw - rb) / nrb;
    r0 = rb * 16 + (lane >> 2);   // the lane's two accumulator rows
    r1 = r0 + 8;
  }
};

// One item: its stages (k counts the CTA's stages across items), then its rows.
template <int D, int KW, bool SHIFT, bool HK>
__device__ __forceinline__ void consume_item(const Walk& w, uint8_t* smem, const ItemRec& rec,
                                             const uint32_t (&qa)[D / 16][4], int cw, int lane, uint32_t& k,
                                             bool& dead) {
  using C = Bf<D>;
  const PartialParams& p = w.p;
  constexpr int KS = D / 16;   // k-steps of q.k
  constexpr int NT = D / 8;    // 8-channel tiles of the output
  constexpr int NTK = KW / 8;  // 8-key tiles of a warp's keys
  constexpr int ng = 2;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const WarpRole<KW> role(cw, lane);
  const int sgrp = role.sgrp, ts = role.ts, my_state = role.my_state, r0 = role.r0, r1 = role.r1;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int qi0 = r0 / p.g, qi1 = r1 / p.g;
  const int lrow = lane & 7, lmat = lane >> 3;   // ldmatrix address roles
  const float sc = p.scale_log2;
  const bool fm = p.mask == DATTN_MASK_FLASHMASK;
  const WorkItem it = rec.it;
  const MaskCtx mc{p.mask, rec.nq, it.T, p.n_sink, p.window};
  const bool ok0 = r0 < p.g * rec.nq, ok1 = r1 < p.g * rec.nq;   // rows of the request
  (void)g4;
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // Shared-shift partials (M4.5 §0x09C): the states live in the common frame phi
  // (log2 units) with no running maximum while the warp's guard holds.  A failed
  // guard moves the accumulated keys to their own maximum (tracked per lane,
  // reduced only then) and continues with the running-max softmax, so the
  // result is that of the synchronized states.
  bool shared = SHIFT;
  float m0 = shared ? p.shift_phi2 : -INFINITY, m1 = m0, l0 = 0.f, l1 = 0.f;
  float sx0 = -INFINITY, sx1 = -INFINITY;   // this lane's largest accepted score per row

  for (int j0 = it.a; j0 < it.e; ++k) {
    const int j1 = min(j0 + kTK, it.e);
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
    if constexpr (HK) {
      if (k == 0 && cw == 0 && lane == 0) trace_stamp(p, kTrFirstStage);
    }
    const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kTK;
    const uint32_t* vis = reinterpret_cast<const uint32_t*>(smem + C::kVis) + st * kTK;
    const bool full = reinterpret_cast<const int*>(smem + C::kFlags)[st] & kFlagFull;
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
    const int base = ts * KW;

    // S = Q K^T over the warp's KW keys (8-key tiles)
    float s[NTK][4];
#pragma unroll
    for (int nt = 0; nt < NTK; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int m = 0; m < KS / 2; ++m) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kt + tile_off<2 * D>(base + nt * 8 + lrow, 4 * m + lmat), b0, b1, b2, b3);
        mma_bf16(s[nt], qa[2 * m], b0, b1);
        mma_bf16(s[nt], qa[2 * m + 1], b2, b3);
      }
    }
    // scale to log2 units, -inf where the key is absent or masked for the row.  32-row
    // tiles: a FULL stage whose slots of this warp all hold keys masks only the rows the
    // request does not have (16-row tiles keep the per-key path: with a fast path the
    // headline and long context S_q = 1 ran 0.2-0.7 us slower, long context S_q = 4 2 us
    // faster)
    if (KW == 32 && full && base + KW <= j1 - j0) {
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          s[nt][e] = ok0 ? s[nt][e] * sc : -INFINITY;
          s[nt][2 + e] = ok1 ? s[nt][2 + e] * sc : -INFINITY;
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int slot = base + nt * 8 + 2 * t4 + e;
          const int t = pos[slot];
          bool v0, v1;
          if (fm) {   // FlashMask: the producer's row bits of the column
            const uint32_t bits = vis[slot];
            v0 = t >= 0 && ok0 && (full || ((bits >> qi0) & 1u));
            v1 = t >= 0 && ok1 && (full || ((bits >> qi1) & 1u));
          } else {
            v0 = t >= 0 && ok0 && (full || key_visible(mc, qi0, t));
            v1 = t >= 0 && ok1 && (full || key_visible(mc, qi1, t));
          }
          s[nt][e] = v0 ? s[nt][e] * sc : -INFINITY;
          s[nt][2 + e] = v1 ? s[nt][2 + e] * sc : -INFINITY;
        }
      }
    }
    if (shared) {   // the range guard of the common frame
      bool bad = false;
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float dl = s[nt][e] - p.shift_phi2;
          bad = bad || (s[nt][e] != -INFINITY && !(dl > p.shift_lo2 && dl < p.shift_hi2));
        }
      if (__any_sync(kAll, bad)) {
        shared = false;
        if (lane == 0) atomicAdd(p.shift_fallbacks, 1);
        sx0 = fmaxf(sx0, __shfl_xor_sync(kAll, sx0, 1));
        sx1 = fmaxf(sx1, __shfl_xor_sync(kAll, sx1, 1));
        sx0 = fmaxf(sx0, __shfl_xor_sync(kAll, sx0, 2));
        sx1 = fmaxf(sx1, __shfl_xor_sync(kAll, sx1, 2));
        // accepted scores lie in (phi + lo, phi + hi): the factor stays inside fp32
        const float a0 = sx0 == -INFINITY ? 0.f : ex2_approx(m0 - sx0);
        const float a1 = sx1 == -INFINITY ? 0.f : ex2_approx(m1 - sx1);
        m0 = sx0;
        m1 = sx1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= a0;
          o[n][1] *= a0;
          o[n][2] *= a1;
          o[n][3] *= a1;
        }
      }
    }
    float (&pr)[NTK][4] = s;   // the probabilities replace the scores
    if (shared) {   // e^(s - phi): no maximum, no rescale
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[nt][e] = ex2_approx(s[nt][e] - p.shift_phi2);
        sx0 = fmaxf(sx0, fmaxf(s[nt][0], s[nt][1]));
        sx1 = fmaxf(sx1, fmaxf(s[nt][2], s[nt][3]));
        ps0 += pr[nt][0] + pr[nt][1];
        ps1 += pr[nt][2] + pr[nt][3];
      }
      l0 += ps0;
      l1 += ps1;
    } else {
      // online softmax: row maxima over the lane quad
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
#pragma unroll
      for (int nt = 2; nt < NTK; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(kAll, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kAll, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(kAll, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(kAll, mx1, 2));
      const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
      const float a0 = n0 == -INFINITY ? 1.f : ex2_approx(m0 - n0);
      const float a1 = n1 == -INFINITY ? 1.f : ex2_approx(m1 - n1);
      const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NTK; ++nt) {
        pr[nt][0] = ex2_approx(s[nt][0] - u0);
        pr[nt][1] = ex2_approx(s[nt][1] - u0);
        pr[nt][2] = ex2_approx(s[nt][2] - u1);
        pr[nt][3] = ex2_approx(s[nt][3] - u1);
        ps0 += pr[nt][0] + pr[nt][1];
        ps1 += pr[nt][2] + pr[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
      m0 = n0;
      m1 = n1;
      if (__any_sync(kAll, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= a0;
          o[n][1] *= a0;
          o[n][2] *= a1;
          o[n][3] *= a1;
        }
      }
    }
    // O += P V: the S fragments re-packed as the A operand (keys are the k index),
    // one k-step per 16 keys
#pragma unroll
    for (int kb = 0; kb < KW / 16; ++kb) {
      const uint32_t pa[4] = {pack_bf16(pr[2 * kb][0], pr[2 * kb][1]), pack_bf16(pr[2 * kb][2], pr[2 * kb][3]),
                              pack_bf16(pr[2 * kb + 1][0], pr[2 * kb + 1][1]),
                              pack_bf16(pr[2 * kb + 1][2], pr[2 * kb + 1][3])};
#pragma unroll
      for (int n2 = 0; n2 < NT / 2; ++n2) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vt + tile_off<2 * D>(base + 16 * kb + (lmat & 1) * 8 + lrow, 2 * n2 + (lmat >> 1)), v0, v1,
                      v2, v3);
        mma_bf16(o[2 * n2], pa, v0, v1);
        mma_bf16(o[2 * n2 + 1], pa, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    j0 = j1;
  }

  // end of item: complete the row sums over the quad and leave the rows
  l0 += __shfl_xor_sync(kAll, l0, 1);
  l1 += __shfl_xor_sync(kAll, l1, 1);
  l0 += __shfl_xor_sync(kAll, l0, 2);
  l1 += __shfl_xor_sync(kAll, l1, 2);
  if (!dead) {
    if (ok0) emit_row<D>(p, it, rec.qo, my_state, r0, m0, l0, o, 0, t4);
    if (ok1) emit_row<D>(p, it, rec.qo, my_state, r1, m1, l1, o, 1, t4);
  } else if (it.slot >= 0 && t4 == 0) {   // the warp gave up: its states are marked, never guessed
    if (ok0) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + r0);
    if (ok1) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + r1);
  }
}

// Items of a call with at most 16 rows run the one-tile layout, each loading
// its query fragments at its start (loading the next item's during the current
// one was no faster: headline 52.10 against 51.94 us).  In a call with more
// rows (a mixed batch's widest request, or a uniform batch of 17 to 32 rows)
// each item takes the layout of its own request's g C_b rows.
// SHIFT: shared-shift partials; the synchronized path is compiled without them.
template <int D, bool SHIFT, bool HK>
__device__ void consume_bf16(const Walk& w, uint8_t* smem, int cw, int lane, bool dep_wait) {
  dependency_wait(dep_wait);   // before Q and the state writes
  const PartialParams& p = w.p;
  constexpr int KS = D / 16;
  const int t4 = lane & 3;
  uint32_t k = 0;
  bool dead = false;   // a bounded wait gave up: stop consuming, write nothing
  if (p.rows <= 16) {
    const WarpRole<16> role(cw, lane);
    for (int ii = w.begin; ii < w.end; ++ii) {
      uint32_t qa[KS][4];
      load_q<D>(p, w.rec(ii), role.r0, role.r1, t4, qa);
      consume_item<D, 16, SHIFT, HK>(w, smem, w.rec(ii), qa, cw, lane, k, dead);
    }
  } else {
    for (int ii = w.begin; ii < w.end; ++ii) {
      const ItemRec rec = w.rec(ii);
      uint32_t qa[KS][4];
      if (p.g * rec.nq <= 16) {
        const WarpRole<16> role(cw, lane);
        load_q<D>(p, rec, role.r0, role.r1, t4, qa);
        consume_item<D, 16, SHIFT, HK>(w, smem, rec, qa, cw, lane, k, dead);
      } else {
        const WarpRole<32> role(cw, lane);
        load_q<D>(p, rec, role.r0, role.r1, t4, qa);
        consume_item<D, 32, SHIFT, HK>(w, smem, rec, qa, cw, lane, k, dead);
      }
    }
  }
}

// A consumer warp's states are written (or marked): tag them for the merge.
// Its rows of an item follow the item's layout, as in consume_bf16.
__device__ __forceinline__ void publish_bf16_states(const Walk& w, int cw, int lane) {
  const PartialParams& p = w.p;
  publish_warp_states(w, [&](const ItemRec& rec, int& st, int& ra, int& rb) {
    if (p.rows > 16 && p.g * rec.nq > 16) {
      const WarpRole<32> role(cw, lane);
      st = role.my_state, ra = role.r0, rb = role.r1;
    } else {
      const WarpRole<16> role(cw, lane);
      st = role.my_state, ra = role.r0, rb = role.r1;
    }
    return (lane & 3) == 0;
  });
}

// Fused LSE merge (M4.5 §0x02B-§0x02C, as in the merge kernel): after the
// consumers have written their states, the CTA counts its finished items per
// merge group; the CTA that completes a group's count merges that group.  The
// states were written before a gpu-scope fence and the count (release); the
// merging CTA fences after reading the final count (acquire) and reads the
// states through L2.  Warps take (row, share of the states) tasks and combine
// a row's shares in shared memory (the drained ring).  The merging CTA resets
// the group's count for the next run.
template <int D>
__device__ void fused_merge(const Walk& w, uint8_t* smem, int cw, int lane) {
  constexpr int C = D / 32;
  const PartialParams& p = w.p;
  constexpr int kCW = kConsumerWarps;
  int* list = reinterpret_cast<int*>(smem);                       // [0]: n, then merge group ids
  float* sm_u = reinterpret_cast<float*>(smem + 1024);            // [kCW][D]
  float* sm_ml = sm_u + kCW * D;                                  // [kCW][2]
  __threadfence();                                                // this thread's state writes
  named_barrier(1, 32 * kCW);
  // A CTA whose wait gave up left some states unwritten: it counts none of its
  // items, so their groups are never merged (no row from stale states).
  if (*reinterpret_cast<volatile int*>(smem + Bf<D>::kAbort)) return;
  if (cw == 0 && lane == 0) {
    int n = 0;
    for (int ii = w.begin; ii < w.end; ++ii) {
      const int g = w.rec(ii).merge;
      if (g < 0) continue;
      // states per item: 8 for requests of at most 16 rows, else 4
      const int spi = p.rows <= 16 || p.g * p.groups[g].nq <= 16 ? kConsumerWarps : kConsumerWarps / 2;
      const int total = p.groups[g].n / spi;
      if (atomicAdd(p.group_count + g, 1) + 1 == total) list[1 + n++] = g;
    }
    list[0] = n;
    __threadfence();
  }
  named_barrier(1, 32 * kCW);
  const int n = list[0];
  if (n == 0) return;
  __threadfence();
  const int R = p.rows;
  const int W = R >= kCW ? 1 : kCW / R;      // warps per row
  for (int k = 0; k < n; ++k) {
    const int gi = list[1 + k];
    const MergeGroup grp = p.groups[gi];
    for (int r0 = 0; r0 < R; r0 += kCW / W) {
      const int row = r0 + cw / W, share = cw % W;
      const bool active = cw / W < kCW / W && row < p.g * grp.nq;
      RowFold<D> f;
      fold_init(f);
      if (active) {
        const int n_mine = grp.n > share ? (grp.n - share + W - 1) / W : 0;
        fold_states<D>(p.ml, p.u, R, row, grp.slot0 + share, n_mine, W, lane, f);
      }
      if (W > 1) {
#pragma unroll
        for (int c = 0; c < C; ++c) sm_u[cw * D + lane * C + c] = f.U[c];
        if (lane == 0) {
          sm_ml[2 * cw] = f.M;
          sm_ml[2 * cw + 1] = f.bad ? __int_as_float(0x7fc00000) : f.L;   // NaN carries the unwritten mark
        }
        named_barrier(1, 32 * kCW);
        if (active && share == 0) {
          RowFold<D> t;
          fold_init(t);
          for (int j = cw; j < cw + W; ++j) {
            t.M = fmaxf(t.M, sm_ml[2 * j + 1] > 0.f ? sm_ml[2 * j] : -INFINITY);
            t.bad = t.bad || sm_ml[2 * j + 1] != sm_ml[2 * j + 1];
          }
          if (t.M != -INFINITY) {
            for (int j = cw; j < cw + W; ++j) {
              if (!(sm_ml[2 * j + 1] > 0.f)) continue;
              const float a = exp2f(sm_ml[2 * j] - t.M);
              t.L += a * sm_ml[2 * j + 1];
#pragma unroll
              for (int c = 0; c < C; ++c) t.U[c] = fmaf(a, sm_u[j * D + lane * C + c], t.U[c]);
            }
          }
          f = t;
        }
        named_barrier(1, 32 * kCW);
      }
      if (active && share == 0) {
        const int i = row / p.g, hq = grp.h * p.g + row % p.g;
        if (!f.bad) write_folded_row<D>(p.o, p.lse, (static_cast<long long>(grp.qo) + i) * p.H_q + hq, f, lane);
      }
    }
    if (cw == 0 && lane == 0) p.group_count[gi] = 0;    // ready for the next run
  }
}

// TAGS: the instance for plans whose merge waits for state-row tags (see
// state_tags_fence); the other instances compile none of it.
template <int D, bool HK, bool TAGS>
__global__ void __launch_bounds__(kThreads, 1) partial_bf16_kernel(const __grid_constant__ PartialParams p) {
  using C = Bf<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (HK && threadIdx.x == 0) {
    trace_stamp(p, kTrEntry);
    if (p.trace) {
      uint32_t sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      p.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + kTrSm] = sm;
    }
  }
  const int it_begin = p.cta_indptr[blockIdx.x], it_end = p.cta_indptr[blockIdx.x + 1];
  ItemRec* cache = reinterpret_cast<ItemRec*>(smem + C::kItems);
  const int incomplete = fill_item_cache(p, cache, it_begin, it_end);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesN; ++s) {   // four consumer warps take each stage
      mbar_init(smem_u32(smem + C::kFullBar + 8 * s), 1);
      mbar_init(smem_u32(smem + C::kEmptyBar + 8 * s), kConsumerWarps / 2);
    }
    *reinterpret_cast<int*>(smem + C::kAbort) = 0;
    *reinterpret_cast<uint64_t*>(smem + C::kAbort + 8) = p.wait_ns;   // read by the bounded waits
    fence_barrier_init();
  }
  // Records that need device inputs are completed by the whole CTA after the
  // wait.  Otherwise each warp waits on its own, just before its first device
  // read, and the producers set up their first stages' keys in the meantime.
  const bool complete_now = __syncthreads_or(incomplete);
  if (HK && threadIdx.x == 0) trace_stamp(p, kTrRecords);
  if (complete_now) complete_item_cache(p, cache, it_begin, it_end);
  const Walk w{p, cache, it_begin, it_end, policy_evict_last()};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kConsumerWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBfProducerRegs));
    if (p.mask == DATTN_MASK_FLASHMASK) produce_bf16<D, true, HK>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else if (runs_apply<kTK>(p)) produce_bf16_runs<D, HK>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else produce_bf16<D, false, HK>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBfConsumerRegs));
  if (p.shift_on) consume_bf16<D, true, HK>(w, smem, warp, lane, !complete_now);
  else consume_bf16<D, false, HK>(w, smem, warp, lane, !complete_now);
  if constexpr (TAGS) publish_bf16_states(w, warp, lane);
  if (HK && lane == 0) trace_stamp(p, kTrConsumerEnd + warp);
  if (p.fused) fused_merge<D>(w, smem, warp, lane);
}

template <int D, bool HK, bool TAGS>
int launch_bf16_inst(const PartialParams& p, int n_ctas, void* stream) {
  const size_t smem = Bf<D>::kTotal;
  // the register budget check and the shared-memory opt-in, once per device
  static std::atomic<unsigned long long> ready{0};
  cudaError_t err = prepare_kernel_once(partial_bf16_kernel<D, HK, TAGS>, smem, 128 * kBfProducerRegs + 32 * kConsumerWarps * kBfConsumerRegs, ready);
  if (err != cudaSuccess) return err;
  // programmatic launch: the prologue overlaps the tail of the preceding kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, partial_bf16_kernel<D, HK, TAGS>, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int D>
int launch_bf16(const PartialParams& p, int n_ctas, void* stream) {
  const bool hk = p.trace || p.skip_arrival;
  if (p.state_seq)
    return hk ? launch_bf16_inst<D, true, true>(p, n_ctas, stream) : launch_bf16_inst<D, false, true>(p, n_ctas, stream);
  return hk ? launch_bf16_inst<D, true, false>(p, n_ctas, stream) : launch_bf16_inst<D, false, false>(p, n_ctas, stream);
}

}  // namespace

int launch_partial_bf16(const PartialParams& p, int d, int n_ctas, void* stream) {
  return d == 64 ? launch_bf16<64>(p, n_ctas, stream) : launch_bf16<128>(p, n_ctas, stream);
}

}  // namespace dattn
