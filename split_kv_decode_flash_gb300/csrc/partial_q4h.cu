// Partial kernel of split-KV decode attention for per-head asymmetric INT4
// K/V ("M8.6 Live-Data Quantization", §0x09C: one fp16 scale and one floating
// fp16 offset per token and kv head, x_hat = (code - o) * s) on the tensor
// cores.
//
// Same persistent producer / consumer structure as the bf16 and INT8
// kernels (item records in shared memory, four producer warps with a
// three-step slot description, per-warp partial states).  Stages hold 256
// keys, so a stage carries as many code bytes as a bf16 stage of 64 keys.
//
// Producer.  Every key row's codes (d/2 bytes, two per byte, the even
// channel in the low nibble) move with 16-byte cp.async into XOR-swizzled
// rows, its (s, o) pairs with 4-byte copies; empty slots are zero-filled.
//
// Consumers (two stage groups of four warps; keys on the M side of the mma,
// query rows on N in blocks of 8).  Codes enter the mma as f16 subnormals: a
// nibble masked in place into the mantissa of an f16 is exactly code * 2^-24
// (bits 0-3) or 16 code * 2^-24 (bits 4-7), so a word of eight codes becomes
// four f16 pairs with one shift and four ands, and nothing needs cancelling.
// The per-token scale stays outside the dot (§0x03A):
//   K: q . k_hat = s_t (q . code_t) - o_t s_t (q . 1).  S'^T = codes . Q^T
//      with Q in f16 (exact for bf16 values in f16's range; the channels of
//      high nibbles carry q / 16; rows whose largest |q| is beyond 2^14 are
//      divided by a power of two first).
//   V: sum_t p_t (code_t - o_t) s_t = sum_t P'_t code_t - sum_t P'_t o_t with
//      P' = p s_t, packed to f16 and transposed with movmatrix into the B
//      operand of O^T = V^T codes . P'^T (V codes from ldmatrix.trans).
//      Output tile 4 c + j holds channels 64 c + 4 g4 + j (accumulator rows
//      g4) and 64 c + 32 + 4 g4 + j (rows g4 + 8); odd j carry the factor 16.
// The online softmax is the bf16 kernel's (log2 units, -inf for masked
// cells, row maxima over the 8 lanes that share a query-row pair).
#include <cuda_runtime.h>

#include "launch.cuh"
#include "tc_common.cuh"

namespace dattn {

namespace {

constexpr int kHK = 256;              // keys per stage
constexpr int kHS = kHK / 32;         // slots per producer lane
constexpr int kHProducerRegs = 104;
constexpr int kHConsumerRegs = 200;
static_assert(128 * kHProducerRegs + 32 * kConsumerWarps * kHConsumerRegs <= kThreads * 168, "register split");
// The FlashMask instance's producers carry four interval ends for each of
// their 8 slots a stage ahead: it keeps the launch's even split (168 each).
template <bool FM>
constexpr int q4h_producer_regs() { return FM ? 168 : kHProducerRegs; }
template <bool FM>
constexpr int q4h_consumer_regs() { return FM ? 168 : kHConsumerRegs; }

// FM: the FlashMask instance, whose ring also carries each key column's row
// bits (two stages fewer, to make room for them).
template <int D, bool FM = false>
struct Q4H {
  // Even depth: with two consumer stage groups taking alternate stages, every
  // ring slot always belongs to the same group (no mbarrier parity alias).
  static constexpr int kStagesN = D == 128 ? (FM ? 4 : 6) : (FM ? 8 : 10);
  static_assert(kStagesN % 2 == 0, "ring depth must be even");
  static constexpr int kRowB = D / 2;              // code bytes of one key row
  static constexpr int kChunks = kRowB / 16;
  static constexpr int kTile = kHK * kRowB;        // one tensor's codes
  static constexpr int kQp = kHK * 4;              // one tensor's (s, o) pairs
  static constexpr int kStage = 2 * kTile + 2 * kQp;
  static constexpr int kPos = kStagesN * kStage;   // int32 [stages][kHK]
  static constexpr int kVis = kPos + kStagesN * kHK * 4;   // FM: uint32 [stages][kHK] row bits
  static constexpr int kFlags = kVis + (FM ? kStagesN * kHK * 4 : 0);
  static constexpr int kSeq = kFlags + kStagesN * 4;
  static constexpr int kFullBar = align16(kSeq + kStagesN * 4);
  static constexpr int kEmptyBar = kFullBar + kStagesN * 8;
  static constexpr int kAbort = kEmptyBar + kStagesN * 8;
  static constexpr int kItems = align16(kAbort + 16);
  static constexpr int kTotal = kItems + kItemCache * static_cast<int>(sizeof(ItemRec));
  static_assert(kTotal <= 232448, "shared memory of one CTA");
};

// 16-byte chunk c of key slot s in a tile of ROWB-byte rows (64 or 32), XOR-
// swizzled so that the eight rows an ldmatrix reads fall in distinct bank groups.
template <int ROWB>
__device__ __forceinline__ uint32_t code_off(int s, int c) {
  if constexpr (ROWB == 64) return static_cast<uint32_t>(s * 64 + ((c ^ ((s >> 1) & 3)) << 4));
  else return static_cast<uint32_t>(s * 32 + ((c ^ ((s >> 2) & 1)) << 4));
}

// Masks of the low and the high nibble of bytes 0 and 2 of a code word; the
// masked word is an f16 pair of subnormals, code * 2^-24 (low) or 16 code *
// 2^-24 (high).
constexpr uint32_t kNibLo = 0x000F000Fu, kNibHi = 0x00F000F0u;
constexpr float kCodeUnit = 16777216.f;   // 2^24

__device__ __forceinline__ uint32_t movmatrix_tr(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t w) { return __half22float2(*reinterpret_cast<const __half2*>(&w)); }

// ---- producer ---------------------------------------------------------------------------

template <int D, bool FM>
__device__ void produce_q4h(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Q4H<D, FM>;
  const PartialParams& p = w.p;
  constexpr int kSlotsPerPass = 32 / C::kChunks;   // key rows per warp instruction
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const char* kqbase = static_cast<const char*>(p.kqp);
  const char* vqbase = static_cast<const char*>(p.vqp);
  const int sub = lane / C::kChunks, ch = lane % C::kChunks;
  const uint64_t stream_pol = policy_evict_first();

  PCur c0{w.begin, 0, 0};
  pc_seek<kHK>(w, c0);
  pc_advance<kHK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kHK>(w, c1, kProducerWarps);
  PCur c2 = c1;
  pc_advance<kHK>(w, c2, kProducerWarps);
  if constexpr (!FM) index_list_prologue(w, c0, lane, dep_wait);   // index lists: list entries are device inputs
  const SlotKeys<kHS> k0 = slot_keys<kHS, !FM>(w, c0, lane);
  SlotKeys<kHS> k1 = slot_keys<kHS, !FM>(w, c1, lane);
  dependency_wait(dep_wait);   // the page table is a device input
  const SlotPages<kHS, FM> g0 = slot_pages<kHS, FM>(w, c0, k0);
  SlotPages<kHS, FM> g1 = slot_pages<kHS, FM>(w, c1, k1);
  SlotKeys<kHS> k2 = slot_keys<kHS, !FM>(w, c2, lane);
  SlotRows<kHS, FM> r0 = slot_rows<kHS, FM>(w, c0, k0, g0, lane);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kHK;
#pragma unroll
    for (int h = 0; h < kHS; ++h) pos[lane + 32 * h] = r0.t[h];
    if constexpr (FM) {
      uint32_t* vis = reinterpret_cast<uint32_t*>(smem + C::kVis) + st * kHK;
#pragma unroll
      for (int h = 0; h < kHS; ++h) vis[lane + 32 * h] = r0.vis[h];
    }
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = r0.full ? kFlagFull : 0;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
    const uint32_t kq = vt + C::kTile, vq = kq + C::kQp;
#pragma unroll
    for (int s0 = 0; s0 < kHK; s0 += kSlotsPerPass) {
      const int s = s0 + sub;
      const uint32_t row = __shfl_sync(kAll, r0.row[s0 / 32], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = code_off<C::kRowB>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
#pragma unroll
    for (int h = 0; h < kHS; ++h) {
      const uint32_t row = r0.row[h];
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * 4;
      cp_async4(kq + 4 * (lane + 32 * h), kqbase + off, ok ? 4u : 0u);
      cp_async4(vq + 4 * (lane + 32 * h), vqbase + off, ok ? 4u : 0u);
    }
    const uint32_t fb = full0 + 8 * st;
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) mbar_arrive(fb);     // publishes pos / flags / stamp; the copies complete the phase

    r0 = slot_rows<kHS, FM>(w, c1, k1, g1, lane);
    c0 = c1;
    g1 = slot_pages<kHS, FM>(w, c2, k2);
    k1 = k2;
    c1 = c2;
    pc_advance<kHK>(w, c2, kProducerWarps);
    k2 = slot_keys<kHS, !FM>(w, c2, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

template <int D>
__device__ void produce_q4h_runs(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Q4H<D, false>;
  const PartialParams& p = w.p;
  constexpr int kSlotsPerPass = 32 / C::kChunks;   // key rows per warp instruction
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const char* kqbase = static_cast<const char*>(p.kqp);
  const char* vqbase = static_cast<const char*>(p.vqp);
  const int sub = lane / C::kChunks, ch = lane % C::kChunks;
  const uint64_t stream_pol = policy_evict_first();

  PCur c0{w.begin, 0, 0};
  pc_seek<kHK>(w, c0);
  pc_advance<kHK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kHK>(w, c1, kProducerWarps);
  RunStage s0 = run_stage(w, c0);
  RunStage s1 = run_stage(w, c1);
  dependency_wait(dep_wait);   // the page table is a device input
  StagePage g0 = run_stage_page(w, s0, lane);
  StagePage g1 = run_stage_page(w, s1, lane);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    const ItemRec rec = w.rec(c0.ii);
    const int pid0 = check_stage_page(p, g0);   // loaded a stage ago
    uint32_t rows[kHS];
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kHK;
#pragma unroll
    for (int h = 0; h < kHS; ++h) {
      int t;
      run_slot(p, s0, rec.it.T, rec.it.h, pid0, lane + 32 * h, t, rows[h]);
      pos[lane + 32 * h] = t;
    }
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = s0.full ? kFlagFull : 0;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
    const uint32_t kq = vt + C::kTile, vq = kq + C::kQp;
#pragma unroll
    for (int s0i = 0; s0i < kHK; s0i += kSlotsPerPass) {
      const int s = s0i + sub;
      const uint32_t row = __shfl_sync(kAll, rows[s0i / 32], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = code_off<C::kRowB>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
#pragma unroll
    for (int h = 0; h < kHS; ++h) {
      const uint32_t row = rows[h];
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * 4;
      cp_async4(kq + 4 * (lane + 32 * h), kqbase + off, ok ? 4u : 0u);
      cp_async4(vq + 4 * (lane + 32 * h), vqbase + off, ok ? 4u : 0u);
    }
    const uint32_t fb = full0 + 8 * st;
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) mbar_arrive(fb);     // publishes pos / flags / stamp; the copies complete the phase

    c0 = c1;
    s0 = s1;
    g0 = g1;
    pc_advance<kHK>(w, c1, kProducerWarps);
    s1 = run_stage(w, c1);
    g1 = run_stage_page(w, s1, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

// ---- consumers --------------------------------------------------------------------------

// Query row "row" (the lane's B-fragment column g4 of its row block) as f16
// B fragments: for 32-channel chunk c and nibble pair m, b[c][m][0] holds
// channels 32 c + 8 t4 + 2 m and + 4 (low nibbles of the lane's code word),
// b[c][m][1] channels 32 c + 8 t4 + 2 m + 1 and + 5 divided by 16 (high
// nibbles).  The row's channel sum and the factor 2^24 / f (f: the power of
// two the row was divided by to fit f16) go to the lanes that own
// accumulator rows 2 t4 and 2 t4 + 1.
template <int D>
struct QH {
  uint32_t b[D / 32][2][2];
  float qsum0, qsum1, unit0, unit1;
};

// rec: the item's record; its request's query rows are packed rows rec.qo ..
// rec.qo + rec.nq - 1 (a mixed batch, M4.5 §0x08F), and rows past g rec.nq are zero.
template <int D>
__device__ __forceinline__ void load_q4h(const PartialParams& p, const ItemRec& rec, int row, int t4, QH<D>& q) {
  constexpr int NCH = D / 32;
  const bool ok = row < p.g * rec.nq;
  const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(p.q) +
                            ((static_cast<long long>(rec.qo) + row / p.g) * p.H_q + rec.it.h * p.g + row % p.g) * D;
  float v[NCH][8];
  float mx = 0.f, sum = 0.f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (ok) w = *reinterpret_cast<const uint4*>(qr + 32 * c + 8 * t4);
    const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
    const float2 e = bf16x2_to_float2(w.z), f = bf16x2_to_float2(w.w);
    v[c][0] = a.x; v[c][1] = a.y; v[c][2] = b.x; v[c][3] = b.y;
    v[c][4] = e.x; v[c][5] = e.y; v[c][6] = f.x; v[c][7] = f.y;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mx = fmaxf(mx, fabsf(v[c][i]));
      sum += v[c][i];
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, o));
    sum += __shfl_xor_sync(kAll, sum, o);
  }
  // power-of-two divisor that brings the row below 2^14 (exact in f16)
  const float fac = mx > 16384.f ? exp2f(ceilf(log2f(mx / 16384.f))) : 1.f;
  const float inv = 1.f / fac, inv16 = inv * 0.0625f;
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      q.b[c][m][0] = pack_f16(v[c][2 * m] * inv, v[c][2 * m + 4] * inv);
      q.b[c][m][1] = pack_f16(v[c][2 * m + 1] * inv16, v[c][2 * m + 5] * inv16);
    }
  }
  // query row r of the block lives in the quad g4 = r (lanes 4 r .. 4 r + 3)
  const float unit = fac * kCodeUnit;
  q.qsum0 = __shfl_sync(kAll, sum, 8 * t4);
  q.qsum1 = __shfl_sync(kAll, sum, 8 * t4 + 4);
  q.unit0 = __shfl_sync(kAll, unit, 8 * t4);
  q.unit1 = __shfl_sync(kAll, unit, 8 * t4 + 4);
}

// S'^T (16 keys x 8 rows) = codes (A, keys x d) . Q^T (B): two mma per
// 32-channel chunk for 16 keys.  A lane's accumulators hold keys g4, g4 + 8
// for the block's rows 2 t4, 2 t4 + 1; row maxima and sums reduce over the 8
// lanes that share t4.  A warp steps over 32 keys, two 16-key blocks that
// share the row maxima and the rescale.  Row blocks of 8 split a stage's keys
// among the four warps of a stage group: 1 block, 64 keys a warp; 2 blocks,
// 128; 4 blocks, 256, so that an item leaves 8, 4 or 2 states per row.
template <int D, bool FM>
__device__ void consume_q4h(const Walk& w, uint8_t* smem, int cw, int lane) {
  using C = Q4H<D, FM>;
  constexpr int NCH = D / 32;   // 32-channel chunks
  constexpr int NT = D / 16;    // output tiles (16 channels x 8 rows)
  const PartialParams& p = w.p;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);

  constexpr int wps = kConsumerWarps / 2;       // warps of a stage group
  const int nrb = p.rows <= 8 ? 1 : p.rows <= 16 ? 2 : 4;
  const int sgrp = cw / wps, wi = cw % wps;
  const int rb = wi % nrb, ts = wi / nrb;
  const int splits = wps / nrb;
  const int my_state = sgrp * splits + ts;
  const int keys_per_warp = kHK / splits;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int ra = 8 * rb + 2 * t4, rb1 = ra + 1;  // the lane's accumulator rows
  const int qia = ra / p.g, qib = rb1 / p.g;
  const int lrow = lane & 7, lmat = lane >> 3;
  const float sc = p.scale_log2;

  uint32_t k = 0;
  bool dead = false;

  for (int ii = w.begin; ii < w.end; ++ii) {
    const WorkItem it = w.rec(ii).it;
    const int nq = w.rec(ii).nq;                  // the request's query rows
    const MaskCtx mc{p.mask, nq, it.T, p.n_sink, p.window};
    const bool oka = ra < p.g * nq, okb = rb1 < p.g * nq;
    // the item's query (loading the next item's during this one held its registers
    // through the whole item: 0.6 us slower per step, 1 us on a mixed batch)
    QH<D> q;
    load_q4h<D>(p, w.rec(ii), 8 * rb + g4, t4, q);
    // log2-unit score = s_t (sc 2^24 / f) S' + z_t (sc sum q), per row
    const float ku0 = sc * q.unit0, ku1 = sc * q.unit1, kz0 = sc * q.qsum0, kz1 = sc * q.qsum1;
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    // per lane, rows ra / rb1: running max, and partial sums over the lane's
    // keys of p and of P' o_v (the f16 P' the mma used)
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f, za = 0.f, zb = 0.f;

    for (int j0 = it.a; j0 < it.e; ++k) {
      const int j1 = min(j0 + kHK, it.e);
      if (static_cast<int>(k & 1u) != sgrp) {
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
        if (lane == 0) atomicOr(p.status, kStPipeline);
        *abort_flag = 1;
        dead = true;
        break;
      }
      const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kHK;
      const bool full = reinterpret_cast<const int*>(smem + C::kFlags)[st] & kFlagFull;
      const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
      const uint32_t* kqp = reinterpret_cast<const uint32_t*>(smem + st * C::kStage + 2 * C::kTile);
      const uint32_t* vqp = kqp + kHK;

      // steps of 32 keys: two 16-key blocks share the row maxima and the rescale
      for (int stp = 0; stp < keys_per_warp / 32; ++stp) {
        const int base = ts * keys_per_warp + stp * 32;
        if (base >= j1 - j0) break;     // the rest of the warp's slots are empty
        float s[2][4];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          s[bb][0] = s[bb][1] = s[bb][2] = s[bb][3] = 0.f;
#pragma unroll
          for (int c2 = 0; c2 < NCH / 2; ++c2) {
            uint32_t v[4];
            ldsm_x4(kt + code_off<C::kRowB>(base + 16 * bb + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1],
                    v[2], v[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t x = v[2 * h], y = v[2 * h + 1];     // keys g4, g4 + 8
              const uint32_t x8 = x >> 8, y8 = y >> 8;
              const uint32_t a0[4] = {x & kNibLo, y & kNibLo, x & kNibHi, y & kNibHi};
              mma_f16(s[bb], a0, q.b[2 * c2 + h][0][0], q.b[2 * c2 + h][0][1]);
              const uint32_t a1[4] = {x8 & kNibLo, y8 & kNibLo, x8 & kNibHi, y8 & kNibHi};
              mma_f16(s[bb], a1, q.b[2 * c2 + h][1][0], q.b[2 * c2 + h][1][1]);
            }
          }
        }
        // block bb: keys base + 16 bb + g4 (s0, s1) and + 8 (s2, s3); rows ra (s0, s2), rb1 (s1, s3).
        // q . k_hat = s_t 2^24 S' - o_t s_t sum(q), in log2 units; -inf where masked.  A
        // step of a FULL stage whose 32 slots all hold keys needs no visibility (rows past
        // the request's have a zero query, stay finite and are never written).
        const bool all_seen = full && base + 32 <= j1 - j0;
        float vsx[2], vsy[2], vox[2], voy[2];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int kx = base + 16 * bb + g4, ky = kx + 8;
          const float2 ksx = h2_to_f2(kqp[kx]), ksy = h2_to_f2(kqp[ky]);
          const float2 vqx = h2_to_f2(vqp[kx]), vqy = h2_to_f2(vqp[ky]);
          vsx[bb] = vqx.x;
          vox[bb] = vqx.y;
          vsy[bb] = vqy.x;
          voy[bb] = vqy.y;
          const float zx = -ksx.y * ksx.x, zy = -ksy.y * ksy.x;   // exact: fp16 x fp16
          if (all_seen) {
            s[bb][0] = fmaf(ksx.x * ku0, s[bb][0], zx * kz0);
            s[bb][1] = fmaf(ksx.x * ku1, s[bb][1], zx * kz1);
            s[bb][2] = fmaf(ksy.x * ku0, s[bb][2], zy * kz0);
            s[bb][3] = fmaf(ksy.x * ku1, s[bb][3], zy * kz1);
            continue;
          }
          const int tx = pos[kx], ty = pos[ky];
          bool vxa, vxb, vya, vyb;
          if constexpr (FM) {   // FlashMask: the producer's row bits of the columns
            const uint32_t* vis = reinterpret_cast<const uint32_t*>(smem + C::kVis) + st * kHK;
            const uint32_t bx = vis[kx], by = vis[ky];
            vxa = tx >= 0 && oka && (full || ((bx >> qia) & 1u));
            vxb = tx >= 0 && okb && (full || ((bx >> qib) & 1u));
            vya = ty >= 0 && oka && (full || ((by >> qia) & 1u));
            vyb = ty >= 0 && okb && (full || ((by >> qib) & 1u));
          } else {
            vxa = tx >= 0 && oka && (full || key_visible(mc, qia, tx));
            vxb = tx >= 0 && okb && (full || key_visible(mc, qib, tx));
            vya = ty >= 0 && oka && (full || key_visible(mc, qia, ty));
            vyb = ty >= 0 && okb && (full || key_visible(mc, qib, ty));
          }
          s[bb][0] = vxa ? fmaf(ksx.x * ku0, s[bb][0], zx * kz0) : -INFINITY;
          s[bb][1] = vxb ? fmaf(ksx.x * ku1, s[bb][1], zx * kz1) : -INFINITY;
          s[bb][2] = vya ? fmaf(ksy.x * ku0, s[bb][2], zy * kz0) : -INFINITY;
          s[bb][3] = vyb ? fmaf(ksy.x * ku1, s[bb][3], zy * kz1) : -INFINITY;
        }
        float mxa = fmaxf(fmaxf(s[0][0], s[0][2]), fmaxf(s[1][0], s[1][2]));
        float mxb = fmaxf(fmaxf(s[0][1], s[0][3]), fmaxf(s[1][1], s[1][3]));
#pragma unroll
        for (int x = 4; x <= 16; x <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(kAll, mxa, x));
          mxb = fmaxf(mxb, __shfl_xor_sync(kAll, mxb, x));
        }
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        const float aa = na == -INFINITY ? 1.f : ex2_approx(ma - na);
        const float ab = nb == -INFINITY ? 1.f : ex2_approx(mb - nb);
        const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
        // P'^T (keys x rows) = p s_v in f16, transposed into B fragments
        uint32_t pb[2][2];
        float sla = 0.f, slb = 0.f, sza = 0.f, szb = 0.f;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const float p0 = ex2_approx(s[bb][0] - ua), p1 = ex2_approx(s[bb][1] - ub);
          const float p2 = ex2_approx(s[bb][2] - ua), p3 = ex2_approx(s[bb][3] - ub);
          const uint32_t px = pack_f16(p0 * vsx[bb], p1 * vsx[bb]), py = pack_f16(p2 * vsy[bb], p3 * vsy[bb]);
          const float2 fx = h2_to_f2(px), fy = h2_to_f2(py);
          sla += p0 + p2;
          slb += p1 + p3;
          sza += fx.x * vox[bb] + fy.x * voy[bb];
          szb += fx.y * vox[bb] + fy.y * voy[bb];
          pb[bb][0] = movmatrix_tr(px);
          pb[bb][1] = movmatrix_tr(py);
        }
        la = la * aa + sla;
        lb = lb * ab + slb;
        za = za * aa + sza;
        zb = zb * ab + szb;
        ma = na;
        mb = nb;
        // the rescale of the accumulators runs every step: a vote and a branch around
        // it cost more here (106.6 against 105.5 us per step) than the multiplies
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= aa;
          o[n][1] *= ab;
          o[n][2] *= aa;
          o[n][3] *= ab;
        }
        // O'^T += V^T codes . P'^T: ldmatrix.trans gives a lane keys (2 t4,
        // 2 t4 + 1) of keys 0-7 / 8-15 at channels 4 g4 .. 4 g4 + 3 of two chunks
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
#pragma unroll
          for (int c2 = 0; c2 < NCH / 2; ++c2) {
            uint32_t v[4];
            ldsm_x4_trans(vt + code_off<C::kRowB>(base + 16 * bb + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0],
                          v[1], v[2], v[3]);
            // v[0] keys 0-7 / chunk 2 c2, v[1] keys 8-15 / chunk 2 c2, v[2], v[3] chunk 2 c2 + 1
            const uint32_t w0 = v[0] >> 8, w1 = v[1] >> 8, w2 = v[2] >> 8, w3 = v[3] >> 8;
            const uint32_t a0[4] = {v[0] & kNibLo, v[2] & kNibLo, v[1] & kNibLo, v[3] & kNibLo};
            mma_f16(o[4 * c2 + 0], a0, pb[bb][0], pb[bb][1]);
            const uint32_t a1[4] = {v[0] & kNibHi, v[2] & kNibHi, v[1] & kNibHi, v[3] & kNibHi};
            mma_f16(o[4 * c2 + 1], a1, pb[bb][0], pb[bb][1]);
            const uint32_t a2[4] = {w0 & kNibLo, w2 & kNibLo, w1 & kNibLo, w3 & kNibLo};
            mma_f16(o[4 * c2 + 2], a2, pb[bb][0], pb[bb][1]);
            const uint32_t a3[4] = {w0 & kNibHi, w2 & kNibHi, w1 & kNibHi, w3 & kNibHi};
            mma_f16(o[4 * c2 + 3], a3, pb[bb][0], pb[bb][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      j0 = j1;
    }

    // end of item: complete the sums over the 8 lanes sharing t4
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      la += __shfl_xor_sync(kAll, la, x);
      lb += __shfl_xor_sync(kAll, lb, x);
      za += __shfl_xor_sync(kAll, za, x);
      zb += __shfl_xor_sync(kAll, zb, x);
    }
    if (!dead) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? rb1 : ra;
        if (!(rr ? okb : oka)) continue;
        const float m = rr ? mb : ma, l = rr ? lb : la, z = rr ? zb : za;
        const int i = row / p.g, hq = it.h * p.g + row % p.g;
        const long long orow = (static_cast<long long>(w.rec(ii).qo) + i) * p.H_q + hq;
        if (it.slot < 0) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
          for (int c2 = 0; c2 < D / 64; ++c2) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {   // channels 64 c2 + 32 hh + 4 g4 + j
              const float* t0 = o[4 * c2], *t1 = o[4 * c2 + 1], *t2 = o[4 * c2 + 2], *t3 = o[4 * c2 + 3];
              const int e = 2 * hh + rr;
              uint2 pk;
              pk.x = pack_bf16((t0[e] * kCodeUnit - z) * inv, (t1[e] * (kCodeUnit / 16.f) - z) * inv);
              pk.y = pack_bf16((t2[e] * kCodeUnit - z) * inv, (t3[e] * (kCodeUnit / 16.f) - z) * inv);
              *reinterpret_cast<uint2*>(out + 64 * c2 + 32 * hh + 4 * g4) = pk;
            }
          }
          if (g4 == 0 && p.lse) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
          const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
          float* u = p.u + srow * D;
#pragma unroll
          for (int c2 = 0; c2 < D / 64; ++c2) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int e = 2 * hh + rr;
              *reinterpret_cast<float4*>(u + 64 * c2 + 32 * hh + 4 * g4) =
                  make_float4(o[4 * c2][e] * kCodeUnit - z, o[4 * c2 + 1][e] * (kCodeUnit / 16.f) - z,
                              o[4 * c2 + 2][e] * kCodeUnit - z, o[4 * c2 + 3][e] * (kCodeUnit / 16.f) - z);
            }
          }
          if (g4 == 0) p.ml[srow] = make_float2(l > 0.f ? m : -INFINITY, l);
        }
      }
    } else if (it.slot >= 0 && g4 == 0) {   // the warp gave up: its states are marked, never guessed
      if (oka) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + ra);
      if (okb) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + rb1);
    }
  }
}

template <int D, bool FM>
__global__ void __launch_bounds__(kThreads, 1) partial_q4h_kernel(const __grid_constant__ PartialParams p) {
  using C = Q4H<D, FM>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int it_begin = p.cta_indptr[blockIdx.x], it_end = p.cta_indptr[blockIdx.x + 1];
  ItemRec* cache = reinterpret_cast<ItemRec*>(smem + C::kItems);
  const int incomplete = fill_item_cache(p, cache, it_begin, it_end);
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStagesN; ++s) {
      mbar_init(smem_u32(smem + C::kFullBar + 8 * s), 1);
      mbar_init(smem_u32(smem + C::kEmptyBar + 8 * s), kConsumerWarps / 2);
    }
    *reinterpret_cast<int*>(smem + C::kAbort) = 0;
    *reinterpret_cast<uint64_t*>(smem + C::kAbort + 8) = p.wait_ns;   // read by the bounded waits
    fence_barrier_init();
  }
  // without records to complete, each warp waits just before its first device read
  const bool complete_now = __syncthreads_or(incomplete);
  if (complete_now) complete_item_cache(p, cache, it_begin, it_end);
  const Walk w{p, cache, it_begin, it_end, policy_evict_last()};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp >= kConsumerWarps) {
    if constexpr (!FM) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(q4h_producer_regs<FM>()));
    if constexpr (FM) produce_q4h<D, true>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else if (runs_apply<kHK>(p)) produce_q4h_runs<D>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else produce_q4h<D, false>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    return;
  }
  if constexpr (!FM) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(q4h_consumer_regs<FM>()));
  dependency_wait(!complete_now);   // before Q and the state writes
  consume_q4h<D, FM>(w, smem, warp, lane);
}

template <int D, bool FM>
int launch_q4h(const PartialParams& p, int n_ctas, void* stream) {
  const size_t smem = Q4H<D, FM>::kTotal;
  // the register budget check and the shared-memory opt-in, once per device
  static std::atomic<unsigned long long> ready{0};
  cudaError_t err = prepare_kernel_once(partial_q4h_kernel<D, FM>, smem,
                                        128 * q4h_producer_regs<FM>() + 32 * kConsumerWarps * q4h_consumer_regs<FM>(), ready);
  if (err != cudaSuccess) return err;
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
  err = cudaLaunchKernelEx(&cfg, partial_q4h_kernel<D, FM>, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

int launch_partial_q4h(const PartialParams& p, int d, int n_ctas, void* stream) {
  if (p.mask == DATTN_MASK_FLASHMASK)
    return d == 64 ? launch_q4h<64, true>(p, n_ctas, stream) : launch_q4h<128, true>(p, n_ctas, stream);
  return d == 64 ? launch_q4h<64, false>(p, n_ctas, stream) : launch_q4h<128, false>(p, n_ctas, stream);
}

}  // namespace dattn
