// Partial kernel of split-KV decode attention for KIVI INT4 K/V ("M8.6 Live-
// Data Quantization", §0x06A-B format) on the tensor cores, for d_h = 64 and
// 128, at most 32 query rows per kv head and V channel groups Gv = 32 (other KIVI
// shapes, and index-list visibility programs, run on the byte-format kernel).
//
// Same persistent producer / consumer structure as the bf16 and INT8
// kernels.  Quantized keys move in stages of 256 (32 KB of codes at d = 128); the
// residual keys (bf16 rows of the per-request ring) in stages of 64.
//
// Producer.  Per quantized stage: the codes of every key row (16-byte
// cp.async into XOR-swizzled 64-byte rows), the key's V qparams (per token,
// per Gv channels) and a table of the K-group qparams (per channel) of every
// group the stage touches.  The groups of a stage follow from its two runs
// of stream positions (at most 256 / G + 2 of them), so a key's table slot is
// arithmetic, not stored.  The page of a group's first token is looked up
// alongside the keys' pages.
//
// Consumers (two stage groups of four warps; keys on the M side of the mma,
// as in the INT8 kernel; a warp scores one block of 8 query rows, and 2 or 4
// blocks share a stage's keys between fewer warps each):
//   Codes enter the mma as f16 subnormals: a nibble masked in place into the
//   mantissa of an f16 is the exact value code * 2^-24 (bits 0-3) or
//   code * 2^-20 (bits 4-7), so a word of eight codes becomes four f16 pairs
//   with one shift and four ands, and no offset needs cancelling afterwards.
//   The factor 16 of the high nibbles is matched on the other operand (K) or
//   undone on the output rows it lands in (V).
//   K: q.k_hat = sum_c (q_c s_gc) code_tc + sum_c q_c z_gc.  For each group
//      the query rows are scaled per channel, Q' = q s_g, and split into f16
//      hi + lo parts (two mma per k-step keep Q' to about 22 bits); the
//      offset term sum_c q_c z_gc is added per row.  A 16-key block that
//      straddles group boundaries is scored with each group's Q' and every
//      key keeps its own group's score.
//   V: sum_t p_t (s_t,cg code_tc + z_t,cg): per channel group cg the
//      probabilities are scaled, P'_cg = p s_t,cg, packed to f16 and
//      transposed with movmatrix into the B operand of O^T = V^T codes . P'^T
//      (ldmatrix.trans); sum_t p_t z_t,cg is kept per (row, channel group).
//      Output tile 2 c + e holds channels 32 c + 4 g4 + 2 e (+1).
//   Residual keys (bf16) use the bf16 mma with the plain query and the
//   probabilities times 2^-24, so they share the accumulators' units.
#include <cuda_runtime.h>

#include "launch.cuh"
#include "tc_common.cuh"

namespace dattn {

namespace {

constexpr int kQKeys = 256;           // keys of a quantized stage
constexpr int kRKeys = 64;            // keys of a residual stage
constexpr int kQSlots = kQKeys / 32;  // slots per producer lane
constexpr int kMaxGroups = 11;        // K groups a stage of two runs may touch (G >= 32)
constexpr int kQ4ProducerRegs = 104;
constexpr int kQ4ConsumerRegs = 200;
static_assert(128 * kQ4ProducerRegs + 32 * kConsumerWarps * kQ4ConsumerRegs <= kThreads * 168, "register split");
// The FlashMask instance's producers also load and reduce each slot's column
// intervals: they get more of the register file.
constexpr int kQ4FmProducerRegs = 120;
constexpr int kQ4FmConsumerRegs = 192;
static_assert(128 * kQ4FmProducerRegs + 32 * kConsumerWarps * kQ4FmConsumerRegs <= kThreads * 168, "register split");
template <bool FM>
constexpr int q4_producer_regs() { return FM ? kQ4FmProducerRegs : kQ4ProducerRegs; }
template <bool FM>
constexpr int q4_consumer_regs() { return FM ? kQ4FmConsumerRegs : kQ4ConsumerRegs; }

// FM: the FlashMask instance, whose ring also carries each key column's row bits.
template <int D, int GV, bool FM>
struct Q4 {
  static constexpr int kStagesN = 4;               // even: stage groups alternate
  static constexpr int kCodeRow = D / 2;           // bytes of a key's codes
  static constexpr int kTile = kQKeys * kCodeRow;  // 16 KB (d = 128) of codes per tensor
  static constexpr int kGT = kMaxGroups * D * 4;   // K-group (s, z) table
  static constexpr int kVQB = D / GV * 4;          // bytes of a key's V (s, z) pairs: 16 or 32
  static_assert(kVQB == 16 || kVQB == 32, "V qparams of a key: one or two 16-byte chunks");
  static constexpr int kVQ = kQKeys * kVQB;
  static constexpr int kOffGT = 2 * kTile;
  static constexpr int kOffVQ = kOffGT + kGT;
  static constexpr int kStage = (kOffVQ + kVQ + 127) / 128 * 128;
  static_assert(kStage >= 2 * kRKeys * D * 2, "a residual stage fits in a stage slot");
  static constexpr int kPos = kStagesN * kStage;   // int32 [stages][kQKeys]: logical key per slot
  static constexpr int kRows = kPos + kStagesN * kQKeys * 4;   // uint32 [stages][kQKeys]: source row per slot
  static constexpr int kVis = kRows + kStagesN * kQKeys * 4;    // FM: uint32 [stages][kQKeys] row bits
  static constexpr int kFlags = kVis + (FM ? kStagesN * kQKeys * 4 : 0);
  static constexpr int kSeq = kFlags + kStagesN * 4;
  static constexpr int kFullBar = align16(kSeq + kStagesN * 4);
  static constexpr int kEmptyBar = kFullBar + kStagesN * 8;
  static constexpr int kAbort = kEmptyBar + kStagesN * 8;
  static constexpr int kItems = align16(kAbort + 16);
  static constexpr int kTotal = kItems + kItemCache * static_cast<int>(sizeof(ItemRec));
  static_assert(kTotal <= 232448, "shared memory of one CTA");
};

// Code rows of ROWB = 64 (d = 128) or 32 (d = 64) bytes: 16-byte chunk c of
// slot s, swizzled so that the eight rows an ldmatrix reads fall in distinct
// bank groups.
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

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t times16_bf16x2(uint32_t w) {
  __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w);
  v = __hmul2(v, __floats2bfloat162_rn(16.f, 16.f));
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 h2f2(uint32_t w) { return __half22float2(*reinterpret_cast<const __half2*>(&w)); }

// A key's V (s, z) pairs, one word per channel group (4 or 8 groups).
template <int NG>
__device__ __forceinline__ void load_vq(const uint8_t* src, uint32_t (&w)[NG]) {
#pragma unroll
  for (int i = 0; i < NG / 4; ++i) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
  }
}

// ---- stages -------------------------------------------------------------------------

// Stream keys [j0, j1) of item ii (ii == end: none); jq: start of the residual keys.
struct QCur {
  int ii, j0, j1, jq;
};

__device__ __forceinline__ int q4_stage_end(const WorkItem& it, int j0, int jq) {
  return j0 < jq ? min(min(j0 + kQKeys, it.e), jq) : min(j0 + kRKeys, it.e);
}

__device__ __forceinline__ void qc_seek(const Walk& w, QCur& c) {
  for (; c.ii < w.end; ++c.ii) {
    const WorkItem it = w.rec(c.ii).it;
    if (it.e > it.a) {
      c.jq = residual_start(w.p, it);
      c.j0 = it.a;
      c.j1 = q4_stage_end(it, c.j0, c.jq);
      return;
    }
  }
}

__device__ __forceinline__ void qc_advance(const Walk& w, QCur& c, int n) {
  for (int i = 0; i < n && c.ii < w.end; ++i) {
    const WorkItem it = w.rec(c.ii).it;
    if (c.j1 < it.e) {
      c.j0 = c.j1;
      c.j1 = q4_stage_end(it, c.j0, c.jq);
    } else {
      ++c.ii;
      qc_seek(w, c);
    }
  }
}

// The K groups of quantized stage [j0, j1) of item it: n groups; group k has
// id gid(k); stream position j lies in group slot qsel(j).  Run 1 holds
// positions j < x0 (token j), run 2 the rest (token x1 + j - x0).
struct StageGroups {
  int n1, n, g1a, g2a;   // groups of run 1, all groups, first group id of each run
  __device__ __forceinline__ int gid(int k) const { return k < n1 ? g1a + k : g2a + (k - n1); }
};

// (gsh = log2 G.)
__device__ __forceinline__ StageGroups stage_groups_of(const WorkItem& it, int j0, int j1, int gsh) {
  StageGroups s;
  const int r1e = min(j1, it.x0);
  s.g1a = j0 >> gsh;
  s.n1 = j0 < r1e ? ((r1e - 1) >> gsh) - s.g1a + 1 : 0;
  const int r2s = max(j0, it.x0);
  s.g2a = (it.x1 + r2s - it.x0) >> gsh;
  const int n2 = r2s < j1 ? ((it.x1 + j1 - 1 - it.x0) >> gsh) - s.g2a + 1 : 0;
  s.n = s.n1 + n2;
  return s;
}

__device__ __forceinline__ int qsel_of(const StageGroups& sg, const WorkItem& it, int j, int gsh) {
  return j < it.x0 ? (j >> gsh) - sg.g1a : sg.n1 + ((it.x1 + j - it.x0) >> gsh) - sg.g2a;
}

// ---- producer ---------------------------------------------------------------------------

struct Q4Desc {
  int t[kQSlots];          // logical key (-1: none)
  uint32_t row[kQSlots];   // codes row (quantized) or ring row (residual); kNoRow: none
  uint32_t vis[kQSlots];   // FlashMask: bit i set when query row i sees the key
  int gpg;                 // lane k < groups: page of group k's first token (-2: none)
  uint32_t grow;           // lane k < groups: row of group k's qparams (kNoRow: none)
  bool full, resid;
};

// The producer's index arithmetic: P and G are powers of two on this kernel
// (shifts psh, gsh); R, the residual ring's length, is any multiple of G.
struct Q4Shapes {
  int psh, gsh, R;
};

__device__ __forceinline__ void q4_keys(const Walk& w, const QCur& c, int lane, int (&t)[kQSlots]) {
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) t[h] = -1;
  if (c.ii >= w.end) return;
  const WorkItem it = w.rec(c.ii).it;
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) {
    const int j = c.j0 + lane + 32 * h;   // interval program: two runs of positions
    if (j < c.j1) t[h] = j < it.x0 ? j : it.x1 + (j - it.x0);
  }
}

// Page ids of the keys' blocks and of the lane's group's first token.
__device__ __forceinline__ void q4_pages(const Walk& w, const QCur& c, const int (&t)[kQSlots], int lane,
                                         const Q4Shapes& sh, int (&pi)[kQSlots], int& gpi) {
  const PartialParams& p = w.p;
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) pi[h] = -2;
  gpi = -2;
  if (c.ii >= w.end || c.j0 >= c.jq) return;     // residual stages read the ring
  const ItemRec r = w.rec(c.ii);
  const int nblk = r.hi - r.lo;
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) {
    const int blk = t[h] >> sh.psh;
    if (t[h] >= 0 && blk < nblk) pi[h] = ld_keep(p.page_indices + r.lo + blk, w.keep);
  }
  const StageGroups sg = stage_groups_of(r.it, c.j0, c.j1, sh.gsh);
  if (lane < sg.n) {
    const int blk = (sg.gid(lane) << sh.gsh) >> sh.psh;
    if (blk < nblk) gpi = ld_keep(p.page_indices + r.lo + blk, w.keep);
  }
}

template <bool FM>
__device__ __forceinline__ Q4Desc q4_rows(const Walk& w, const QCur& c, const int (&t)[kQSlots],
                                          const int (&pi)[kQSlots], int gpi, int lane, const Q4Shapes& sh) {
  const PartialParams& p = w.p;
  Q4Desc d;
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) {
    d.t[h] = -1;
    d.row[h] = kNoRow;
    d.vis[h] = 0u;
  }
  d.gpg = gpi;
  d.grow = kNoRow;
  d.full = false;
  d.resid = false;
  if (c.ii >= w.end) return d;
  const ItemRec r = w.rec(c.ii);
  d.resid = c.j0 >= c.jq;
  int tmax = -1, err = 0;
  // residual ring row of token t: (b R + (t mod R)) H + h; page row: (pi H + h) P + (t mod P).
  // Residual keys lie in [n_q, T) with T - n_q <= R, so t mod R = (n_q mod R) + (t - n_q),
  // less R once it reaches R; the planner stores (n_q mod R) - n_q in the item's record.
  const uint32_t ring0 = static_cast<uint32_t>(r.it.b) * sh.R;
  const int roff = r.ring_off;   // ring slot of residual key t: t + roff, less R once it reaches R
#pragma unroll
  for (int h = 0; h < kQSlots; ++h) {
    const int tk = t[h];
    uint32_t row = kNoRow;
    if (tk >= 0) {
      if (d.resid) {
        int sl = tk + roff;
        if (sl >= sh.R) sl -= sh.R;
        row = (ring0 + static_cast<uint32_t>(sl)) * p.H_kv + r.it.h;
      } else if (pi[h] == -2) {
        err |= kStBlockRange;
      } else if (pi[h] < 0 || pi[h] >= p.num_pages) {
        err |= kStPageRange;
      } else {
        row = ((static_cast<uint32_t>(pi[h]) * p.H_kv + r.it.h) << sh.psh) + (tk & ((1 << sh.psh) - 1));
      }
    }
    d.t[h] = row == kNoRow ? -1 : tk;
    d.row[h] = row;
    tmax = max(tmax, d.t[h]);
  }
  if (!d.resid) {
    const StageGroups sg = stage_groups_of(r.it, c.j0, c.j1, sh.gsh);
    if (lane < sg.n) {
      if (gpi == -2) {
        err |= kStBlockRange;
      } else if (gpi < 0 || gpi >= p.num_pages) {
        err |= kStPageRange;
      } else {
        // group qparams sit on the page of the group's first token, slot (first mod P) / G
        const int g0 = sg.gid(lane) << sh.gsh;
        const int per_page_sh = max(0, sh.psh - sh.gsh);
        const int slot = (g0 & ((1 << sh.psh) - 1)) >> sh.gsh;
        d.grow = ((static_cast<uint32_t>(gpi) * p.H_kv + r.it.h) << per_page_sh) + slot;
      }
    }
  }
  if (err) atomicOr(p.status, err);
  if constexpr (FM) {
    // FlashMask: the column's two hidden row intervals; a column hidden from
    // every query row is not loaded.  FULL: every slot holds a key every row sees.
    const uint32_t all_rows = row_bits(0, r.nq);
    bool all = true;
#pragma unroll
    for (int h = 0; h < kQSlots; ++h) {
      uint32_t v = 0u;
      if (d.t[h] >= 0) {
        const int4 iv = *reinterpret_cast<const int4*>(p.fm_intervals + 4ll * (r.it.x1 + d.t[h]));
        v = all_rows & ~(row_bits(iv.x, iv.y) | row_bits(iv.z, iv.w));
      }
      if (v == 0u) {
        d.t[h] = -1;
        d.row[h] = kNoRow;
      }
      d.vis[h] = v;
      if (c.j0 + lane + 32 * h < c.j1) all = all && v == all_rows;
    }
    d.full = __all_sync(kAll, all);
    return d;
  }
  d.full = stage_is_full(p, r.it, r.nq, c.j0, c.j1, tmax, -1);
  return d;
}

template <int D, int GV, bool FM>
__device__ void produce_q4(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Q4<D, GV, FM>;
  const PartialParams& p = w.p;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);
  const char* kbase = static_cast<const char*>(p.k);
  const char* vbase = static_cast<const char*>(p.v);
  const char* kres = static_cast<const char*>(p.kres);
  const char* vres = static_cast<const char*>(p.vres);
  const char* kqbase = static_cast<const char*>(p.kqp);
  const char* vqbase = static_cast<const char*>(p.vqp);
  const uint64_t stream_pol = policy_evict_first();
  const Q4Shapes sh{p.P_shift, p.kivi_G == 32 ? 5 : 6, p.kivi_R};

  // Stages are described in three steps a stage apart (keys two stages ahead,
  // page ids one stage ahead, rows for the stage at hand), so the page-table
  // loads have a whole stage to land; each step has one call site.
  QCur c0{w.begin, 0, 0, 0};
  qc_seek(w, c0);
  qc_advance(w, c0, pw);
  QCur c1 = c0;
  qc_advance(w, c1, kProducerWarps);
  int t0[kQSlots], t1[kQSlots], pi0[kQSlots], g0i;
  q4_keys(w, c0, lane, t0);
  q4_keys(w, c1, lane, t1);
  dependency_wait(dep_wait);   // the page table is a device input
  q4_pages(w, c0, t0, lane, sh, pi0, g0i);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const Q4Desc r0 = q4_rows<FM>(w, c0, t0, pi0, g0i, lane, sh);
    q4_pages(w, c1, t1, lane, sh, pi0, g0i);   // next stage's page ids, in flight until then
    QCur c2 = c1;
    qc_advance(w, c2, kProducerWarps);
#pragma unroll
    for (int h = 0; h < kQSlots; ++h) t0[h] = t1[h];
    q4_keys(w, c2, lane, t1);
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kQKeys;
    uint32_t* rows = reinterpret_cast<uint32_t*>(smem + C::kRows) + st * kQKeys;
#pragma unroll
    for (int h = 0; h < kQSlots; ++h) {
      pos[lane + 32 * h] = r0.t[h];
      rows[lane + 32 * h] = r0.row[h];
    }
    if constexpr (FM) {
      uint32_t* vis = reinterpret_cast<uint32_t*>(smem + C::kVis) + st * kQKeys;
#pragma unroll
      for (int h = 0; h < kQSlots; ++h) vis[lane + 32 * h] = r0.vis[h];
    }
    __syncwarp();
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = (r0.full ? kFlagFull : 0) | (r0.resid ? kFlagResidual : 0);
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
    if (r0.resid) {
      // bf16 rows of the residual ring: 64 slots, RC chunks per row, 32 / RC rows per instruction
      constexpr int RC = D * 2 / 16;
      const uint32_t rkt = kt, rvt = kt + kRKeys * D * 2;
      const int sub = lane / RC, ch = lane % RC;
#pragma unroll 1
      for (int s0 = 0; s0 < kRKeys; s0 += 32 / RC) {
        const int s = s0 + sub;
        const uint32_t row = rows[s];
        const bool ok = row != kNoRow;
        const size_t off = static_cast<size_t>(ok ? row : 0u) * (D * 2) + ch * 16;
        const uint32_t dst = tile_off<D * 2>(s, ch);
        cp_async16(rkt + dst, kres + off, ok ? 16u : 0u, stream_pol);
        cp_async16(rvt + dst, vres + off, ok ? 16u : 0u, stream_pol);
      }
    } else {
      // codes: 256 slots, CC chunks per row, 32 / CC rows per instruction (the
      // swizzle of slot s0 + sub only depends on sub, as s0 steps by a multiple of 8)
      constexpr int CC = C::kCodeRow / 16;
      const int sub = lane / CC, ch = lane % CC;
      const uint32_t dst0 = code_off<C::kCodeRow>(sub, ch);
      const char* kb = kbase + ch * 16;
      const char* vb = vbase + ch * 16;
#pragma unroll 4
      for (int s0 = 0; s0 < kQKeys; s0 += 32 / CC) {
        const uint32_t row = rows[s0 + sub];
        const bool ok = row != kNoRow;
        const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kCodeRow;
        const uint32_t dst = dst0 + s0 * C::kCodeRow;
        cp_async16(kt + dst, kb + off, ok ? 16u : 0u, stream_pol);
        cp_async16(vt + dst, vb + off, ok ? 16u : 0u, stream_pol);
      }
      // per-key V qparams (one or two 16-byte chunks)
      const uint32_t vq = kt + C::kOffVQ;
#pragma unroll 1
      for (int s = lane; s < kQKeys; s += 32) {
        const uint32_t row = rows[s];
        const bool ok = row != kNoRow;
        const char* src = vqbase + static_cast<size_t>(ok ? row : 0u) * C::kVQB;
#pragma unroll
        for (int i = 0; i < C::kVQB / 16; ++i)
          cp_async16(vq + C::kVQB * s + 16 * i, src + 16 * i, ok ? 16u : 0u, stream_pol);
      }
      // K-group qparams table: group k (lane k's description) -> D / 4 chunks of 16 bytes
      const uint32_t gt = kt + C::kOffGT;
      const WorkItem it = w.rec(c0.ii).it;
      const int n_g = stage_groups_of(it, c0.j0, c0.j1, sh.gsh).n;
      for (int g = 0; g < n_g && g < kMaxGroups; ++g) {
        const uint32_t grow = __shfl_sync(kAll, r0.grow, g);
        const bool ok = grow != kNoRow;
        if (lane < D / 4)
          cp_async16(gt + g * D * 4 + lane * 16, kqbase + static_cast<size_t>(ok ? grow : 0u) * D * 4 + lane * 16,
                     ok ? 16u : 0u, stream_pol);
      }
    }
    const uint32_t fb = full0 + 8 * st;
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) mbar_arrive(fb);

    c0 = c1;
    c1 = c2;
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// ---- consumers --------------------------------------------------------------------------

__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// a * (low half of b, in both halves), rounded to nearest.
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2_rn(*reinterpret_cast<const __half2*>(&a), __low2half2(*reinterpret_cast<const __half2*>(&b)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// a * b - c with one rounding: the exact low part of a split f16 product.
__device__ __forceinline__ uint32_t hfma2_rn_sub(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("{ .reg .b32 nc; neg.f16x2 nc, %3; fma.rn.f16x2 %0, %1, %2, nc; }" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hmax2_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("{ .reg .b32 x, y; abs.f16x2 x, %1; abs.f16x2 y, %2; max.f16x2 %0, x, y; }" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// c + (half "H" of q) * (high half of zw), the product exact, one rounding in f32.
template <int H>
__device__ __forceinline__ float fma_q_zhi(uint32_t q, uint32_t zw, float c) {
  float d;
  if constexpr (H == 0)
    asm("{ .reg .b16 q0, q1, z0, z1; mov.b32 {q0, q1}, %1; mov.b32 {z0, z1}, %2; fma.rn.f32.f16 %0, q0, z1, %3; }"
        : "=f"(d) : "r"(q), "r"(zw), "f"(c));
  else
    asm("{ .reg .b16 q0, q1, z0, z1; mov.b32 {q0, q1}, %1; mov.b32 {z0, z1}, %2; fma.rn.f32.f16 %0, q1, z1, %3; }"
        : "=f"(d) : "r"(q), "r"(zw), "f"(c));
  return d;
}

// A lane's query row for the K side as f16 pairs: qh[c][k] holds channels
// (32 c' + 8 t4 + k, 32 c' + 8 t4 + k + 4) of true chunk c' = c ^ cswap (cswap
// = d / 64 on the lo lanes of the PACKED layout, else 0); the pairs k = 0, 2
// (which meet low-nibble codes) carry 16 q.  A row whose largest |q| exceeds
// 2^10 is scaled by a power of two wq (qinv = 1 / wq) so that 16 q stays in range.
template <int D>
struct QRow {
  uint32_t qh[D / 32][4];
  float qinv;
};

template <int D>
__device__ __forceinline__ void load_qrow(const __nv_bfloat16* qrow, bool ok, QRow<D>& r, int t4, int cswap) {
  float qf[D / 4];
  float mx = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint4 wq = make_uint4(0u, 0u, 0u, 0u);
    if (ok) wq = *reinterpret_cast<const uint4*>(qrow + 32 * (c ^ cswap) + 8 * t4);   // stored chunk c: true c ^ cswap
    const uint32_t ws[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = bf16x2_to_float2(ws[e]);
      qf[8 * c + 2 * e] = f.x;
      qf[8 * c + 2 * e + 1] = f.y;
      mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
  const float wq = mx > 1024.f ? exp2f(10.f - ceilf(__log2f(mx))) : 1.f;
  r.qinv = 1.f / wq;
#pragma unroll
  for (int c = 0; c < D / 32; ++c)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float f = (k & 1) ? wq : 16.f * wq;
      r.qh[c][k] = pack_f16(qf[8 * c + k] * f, qf[8 * c + k + 4] * f);
    }
}

// Q' = q s_g of one K group as f16 B fragments, split hi + lo so that the
// pair carries Q' to about 22 bits: k-step 2c holds the pairs k = 0 (b0)
// and k = 1 (b1) of chunk c, k-step 2c + 1 the pairs k = 2 and k = 3.
// PACKED (at most 4 rows): B column n is row n & 3, its hi part for n < 4
// and its lo part for n >= 4, so one mma covers both.  Otherwise b holds
// the hi parts and lo the lo parts of rows 0-7.  Per-row terms for rows ra,
// rb: off = sum_c q_c z_gc and inv = 2^20 / (wq w), w a power of two that
// keeps a row's hi parts finite (1 unless a product nears the f16 limit).
template <int D, bool PACKED>
struct QPrime {
  uint32_t b[D / 16][2];
  uint32_t lo[PACKED ? 1 : D / 16][2];
  float offa, offb, inva, invb;
};

// Packs the hi / lo f16 parts of chunk c into the B fragments (see QPrime).
template <int D, bool PACKED>
__device__ __forceinline__ void pack_qprime(const uint32_t (&hi)[D / 32][4], const uint32_t (&lo)[D / 32][4],
                                            bool lo_lane, QPrime<D, PACKED>& out) {
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int ks = 2 * c + (k >> 1), r = k & 1;
      if constexpr (PACKED) {
        out.b[ks][r] = lo_lane ? lo[c][k] : hi[c][k];
      } else {
        out.b[ks][r] = hi[c][k];
        out.lo[ks][r] = lo[c][k];
      }
    }
  }
}

// Q' of one K group without a branch: the f16 split of q s_g, the offsets and
// the factors for w = 1.  Returns whether the lane's row kept every hi part
// below 2^15; when some row did not, qprime_rescaled must redo the split.
// PACKED: lane L and lane L ^ 16 hold the same row (hi and lo columns); each
// splits the products of its own half of the chunks (its stored chunks 0 ..
// d / 64 - 1, see QRow) and the two trade the parts the other one keeps.
template <int D, bool PACKED>
__device__ __forceinline__ bool qprime_fast(const QRow<D>& q, const uint8_t* gt_row, int t4, bool lo_lane, int ra,
                                            QPrime<D, PACKED>& out) {
  constexpr int NCH = PACKED ? D / 64 : D / 32;   // chunks this lane splits
  uint32_t hi[NCH][4], lo[NCH][4];
  float offe = 0.f, offo = 0.f;   // sum q z over the pairs carrying 16 q, and over the others
  uint32_t mx2 = 0u;
  const int cofs = PACKED && lo_lane ? D / 64 : 0;   // true chunk of stored chunk 0
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    // (s, z) of channels 32 c' + 8 t4 + 0..7 of true chunk c' = c + cofs
    const uint8_t* g = gt_row + (32 * (c + cofs) + 8 * t4) * 4;
    const uint4 w0 = *reinterpret_cast<const uint4*>(g);
    const uint4 w1 = *reinterpret_cast<const uint4*>(g + 16);
    const uint32_t sz[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t s2 = __byte_perm(sz[k], sz[k + 4], 0x5410u);
      hi[c][k] = hmul2_rn(q.qh[c][k], s2);
      lo[c][k] = hfma2_rn_sub(q.qh[c][k], s2, hi[c][k]);
      mx2 = hmax2_abs(mx2, hi[c][k]);
      float& off = (k & 1) ? offo : offe;
      off = fma_q_zhi<0>(q.qh[c][k], sz[k], off);
      off = fma_q_zhi<1>(q.qh[c][k], sz[k + 4], off);
    }
  }
  const float2 m2 = h2f2(mx2);
  float mx = fmaxf(m2.x, m2.y);
  float off = fmaf(offe, 1.f / 16.f, offo);
  if constexpr (PACKED) {
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 16));
    off += __shfl_xor_sync(kAll, off, 16);
    // the hi lane keeps hi parts, the lo lane lo parts: each sends the other kind
#pragma unroll
    for (int c = 0; c < NCH; ++c)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t mine = lo_lane ? lo[c][k] : hi[c][k];
        const uint32_t theirs = __shfl_xor_sync(kAll, lo_lane ? hi[c][k] : lo[c][k], 16);
        // true chunks c (the hi lane's own) and c + NCH (the lo lane's own)
        out.b[2 * c + (k >> 1)][k & 1] = lo_lane ? theirs : mine;
        out.b[2 * (c + NCH) + (k >> 1)][k & 1] = lo_lane ? mine : theirs;
      }
  } else {
    pack_qprime<D, PACKED>(hi, lo, lo_lane, out);
  }
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, 2));
  off += __shfl_xor_sync(kAll, off, 1);
  off += __shfl_xor_sync(kAll, off, 2);
  off *= q.qinv;
  const float inv = kCodeUnit / 16.f * q.qinv;
  // row r lives in the quad r (and, PACKED, in the quad r + 4 too)
  out.offa = __shfl_sync(kAll, off, 4 * ra);
  out.offb = __shfl_sync(kAll, off, 4 * ra + 4);
  out.inva = __shfl_sync(kAll, inv, 4 * ra);
  out.invb = __shfl_sync(kAll, inv, 4 * ra + 4);
  return mx < 32768.f;
}

// Rare: a product reached the f16 limit; redo the split in f32 at a power-of-
// two scale w per row and fold 1 / w into the factors (the offsets stand).
// (With this path and the fast one in a single function the KIVI step took
// 5 % longer: the split leaves the fast part without a branch.)
template <int D, bool PACKED>
__device__ void qprime_rescaled(const QRow<D>& qs, const uint8_t* gt_row, int t4, bool lo_lane, int ra,
                                QPrime<D, PACKED>& out) {
  QRow<D> q;   // the query in true chunk order (PACKED lo lanes store their halves swapped)
  q.qinv = qs.qinv;
#pragma unroll
  for (int c = 0; c < D / 32; ++c)
#pragma unroll
    for (int k = 0; k < 4; ++k) q.qh[c][k] = PACKED && lo_lane ? qs.qh[c ^ (D / 64)][k] : qs.qh[c][k];
  uint32_t hi[D / 32][4], lo[D / 32][4];
  float pm = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(gt_row + (32 * c + 8 * t4) * 4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(gt_row + (32 * c + 8 * t4) * 4 + 16);
    const uint32_t sz[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 qq = h2f2(q.qh[c][k]);
      pm = fmaxf(pm, fmaxf(fabsf(qq.x * h2f2(sz[k]).x), fabsf(qq.y * h2f2(sz[k + 4]).x)));
    }
  }
  pm = fmaxf(pm, __shfl_xor_sync(kAll, pm, 1));
  pm = fmaxf(pm, __shfl_xor_sync(kAll, pm, 2));
  const float w = pm > 16384.f ? exp2f(14.f - ceilf(__log2f(pm))) : 1.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    const uint4 w0 = *reinterpret_cast<const uint4*>(gt_row + (32 * c + 8 * t4) * 4);
    const uint4 w1 = *reinterpret_cast<const uint4*>(gt_row + (32 * c + 8 * t4) * 4 + 16);
    const uint32_t sz[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 qq = h2f2(q.qh[c][k]);
      const float a = qq.x * h2f2(sz[k]).x * w, b = qq.y * h2f2(sz[k + 4]).x * w;
      hi[c][k] = pack_f16(a, b);
      const float2 hf = h2f2(hi[c][k]);
      lo[c][k] = pack_f16(a - hf.x, b - hf.y);
    }
  }
  pack_qprime<D, PACKED>(hi, lo, lo_lane, out);
  const float inv = kCodeUnit / 16.f * q.qinv / w;
  out.inva = __shfl_sync(kAll, inv, 4 * ra);
  out.invb = __shfl_sync(kAll, inv, 4 * ra + 4);
}

template <int D, bool PACKED>
__device__ __forceinline__ void make_qprime(const QRow<D>& q, const uint8_t* gt_row, int t4, bool lo_lane, int ra,
                                            QPrime<D, PACKED>& out) {
  if (!__all_sync(kAll, qprime_fast<D, PACKED>(q, gt_row, t4, lo_lane, ra, out)))
    qprime_rescaled<D, PACKED>(q, gt_row, t4, lo_lane, ra, out);
}

// Raw S'^T (16 keys x 8 columns) = codes . B for the 16 keys at slot "base",
// in 2^-20 units; separate accumulators keep the mma chains short.
template <int D, bool PACKED>
__device__ __forceinline__ void k_mma(uint32_t kt, int base, int lrow, int lmat, const QPrime<D, PACKED>& q,
                                      float (&s)[4]) {
  constexpr int NA = PACKED ? 2 : 4;
  float acc[NA][4];
#pragma unroll
  for (int x = 0; x < NA; ++x) acc[x][0] = acc[x][1] = acc[x][2] = acc[x][3] = 0.f;
#pragma unroll
  for (int c2 = 0; c2 < D / 64; ++c2) {
    uint32_t v[4];
    ldsm_x4(kt + code_off<D / 2>(base + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1], v[2], v[3]);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int c = 2 * c2 + hh;
      const uint32_t lo_keys = v[2 * hh], hi_keys = v[2 * hh + 1];   // keys 0-7, 8-15
      const uint32_t lo8 = lo_keys >> 8, hi8 = hi_keys >> 8;
      const uint32_t a0[4] = {lo_keys & kNibLo, hi_keys & kNibLo, lo_keys & kNibHi, hi_keys & kNibHi};
      const uint32_t a1[4] = {lo8 & kNibLo, hi8 & kNibLo, lo8 & kNibHi, hi8 & kNibHi};
      mma_f16(acc[0], a0, q.b[2 * c][0], q.b[2 * c][1]);
      mma_f16(acc[1], a1, q.b[2 * c + 1][0], q.b[2 * c + 1][1]);
      if constexpr (!PACKED) {
        mma_f16(acc[2], a0, q.lo[2 * c][0], q.lo[2 * c][1]);
        mma_f16(acc[3], a1, q.lo[2 * c + 1][0], q.lo[2 * c + 1][1]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float t = acc[0][e] + acc[1][e];
    if constexpr (!PACKED) t += acc[2][e] + acc[3][e];
    s[e] = t;
  }
  if constexpr (PACKED) {   // columns 2 t4 (+1) and 2 t4 + 4 (+1): the hi and lo parts of one row
#pragma unroll
    for (int e = 0; e < 4; ++e) s[e] += __shfl_xor_sync(kAll, s[e], 2);
  }
}

template <int D, int GV, bool FM, bool PACKED>
__device__ void consume_q4(const Walk& w, uint8_t* smem, int cw, int lane) {
  using C = Q4<D, GV, FM>;
  constexpr int NT = D / 16;                  // output tiles
  constexpr int kCg = D / GV;                 // V channel groups
  constexpr int NS = PACKED ? 2 : 1;          // 16-key sub-blocks per step
  const PartialParams& p = w.p;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);

  constexpr int ng = 2;
  constexpr int wps = kConsumerWarps / ng;
  // row blocks of 8 rows (PACKED: one block of at most 4) split a stage's keys
  // among the four warps of a stage group: 1 block, a quarter of the keys a
  // warp; 2 blocks, a half; 4 blocks, all of them
  const int nrb = PACKED || p.rows <= 8 ? 1 : p.rows <= 16 ? 2 : 4;
  const int sgrp = cw / wps, wi = cw % wps;
  const int rbk = wi % nrb, ts = wi / nrb;
  const int splits = wps / nrb;
  const int my_state = sgrp * splits + ts;
  const int g4 = lane >> 2, t4 = lane & 3;
  // rows of the lane's score, probability and output fragments (PACKED: lanes
  // t4 = 2, 3 repeat the rows of lanes t4 = 0, 1 and write nothing); lra is
  // the row within the block
  const int lra = PACKED ? 2 * (t4 & 1) : 2 * t4;
  const int ra = 8 * rbk + lra, rb = ra + 1;
  const bool writer = !PACKED || t4 < 2;
  const int qia = ra / p.g, qib = rb / p.g;
  // query row of the lane's B fragments
  const int rq = PACKED ? (g4 & 3) : 8 * rbk + g4;
  const bool lo_lane = PACKED && g4 >= 4;
  // PACKED: a lane and its partner lane ^ 16 hold the same row; each splits the
  // Q' products of half of the chunks, the lo lane's query stored with its
  // halves swapped (stored chunk c is true chunk c ^ cswap)
  const int cswap = lo_lane ? D / 64 : 0;
  const int lrow = lane & 7, lmat = lane >> 3;
  const float sc = p.scale_log2;
  const int gsh = p.kivi_G == 32 ? 5 : 6;   // log2 G
  // Gv = 16: the lane's V code rows belong to channel group 2 c (g4 < 4) or 2 c + 1
  const uint32_t gmask_lo = g4 < 4 ? kNibLo : 0u, gmask_hi = g4 < 4 ? kNibHi : 0u;

  uint32_t k = 0;
  bool dead = false;
  for (int ii = w.begin; ii < w.end; ++ii) {
    const WorkItem it = w.rec(ii).it;
    // the request's query rows are packed rows qo .. qo + nq - 1 (a mixed batch,
    // M4.5 §0x08F); rows past g nq have a zero query and are never written
    const int qo = w.rec(ii).qo, nq = w.rec(ii).nq;
    const MaskCtx mc{p.mask, nq, it.T, p.n_sink, p.window};
    const bool oka = ra < p.g * nq, okb = rb < p.g * nq, okq = rq < p.g * nq;
    const int jq = residual_start(p, it);
    const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(p.q) +
                                ((static_cast<long long>(qo) + rq / p.g) * p.H_q + it.h * p.g + rq % p.g) * D;
    QRow<D> qr;
    load_qrow(qrow, okq, qr, t4, cswap);
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    float za[kCg], zb[kCg];   // per V channel group and row: sum_t p_t z_t
#pragma unroll
    for (int x = 0; x < kCg; ++x) za[x] = zb[x] = 0.f;
    QPrime<D, PACKED> qp;
    int cur_gid = -1;         // K group whose Q' is in qp

    for (int j0 = it.a; j0 < it.e; ++k) {
      const int j1 = q4_stage_end(it, j0, jq);
      if (static_cast<int>(k % ng) != sgrp) {
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
      const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kQKeys;
      const int flags = reinterpret_cast<const int*>(smem + C::kFlags)[st];
      const bool full = flags & kFlagFull;
      const bool resid = flags & kFlagResidual;
      const uint8_t* stage = smem + st * C::kStage;
      const uint32_t kt = smem_u32(stage), vt = kt + C::kTile;
      const StageGroups sg = stage_groups_of(it, j0, j1, gsh);
      const uint8_t* gt = stage + C::kOffGT;
      const uint8_t* vq = stage + C::kOffVQ;
      const int slice = resid ? kRKeys / splits : kQKeys / splits;

      for (int b0 = 0; b0 < slice; b0 += 16 * NS) {
        const int base0 = ts * slice + b0;
        if (j0 + base0 >= j1) break;
        // NS sub-blocks of 16 keys at slots base0 + 16 u; in sub-block u the lane
        // scores keys g4 (s[u][0], s[u][1]) and g4 + 8 (s[u][2], s[u][3]) for rows
        // ra (s[u][0], s[u][2]) and rb (s[u][1], s[u][3])
        float s[NS][4];
#pragma unroll
        for (int u = 0; u < NS; ++u) s[u][0] = s[u][1] = s[u][2] = s[u][3] = 0.f;
        if (!resid) {
          // the step's keys lie in table slots [sel0, sel1] (one slot unless they
          // straddle a group boundary); each key keeps its own slot's score.
          // Slots past j1 hold zero codes and are masked below.
          const int sel0 = qsel_of(sg, it, j0 + base0, gsh);
          const int sel1 = qsel_of(sg, it, min(j0 + base0 + 16 * NS - 1, j1 - 1), gsh);
          int selx[NS], sely[NS];
#pragma unroll
          for (int u = 0; u < NS; ++u) selx[u] = sely[u] = sel0;
          if (sel1 != sel0) {
#pragma unroll
            for (int u = 0; u < NS; ++u) {
              selx[u] = qsel_of(sg, it, min(j0 + base0 + 16 * u + g4, j1 - 1), gsh);
              sely[u] = qsel_of(sg, it, min(j0 + base0 + 16 * u + g4 + 8, j1 - 1), gsh);
            }
          }
          for (int sel = sel0; sel <= sel1; ++sel) {
            if (sg.gid(sel) != cur_gid) {
              make_qprime<D, PACKED>(qr, gt + sel * D * 4, t4, lo_lane, lra, qp);
              cur_gid = sg.gid(sel);
            }
            float t[NS][4];
#pragma unroll
            for (int u = 0; u < NS; ++u) k_mma<D, PACKED>(kt, base0 + 16 * u, lrow, lmat, qp, t[u]);
#pragma unroll
            for (int u = 0; u < NS; ++u) {
              if (selx[u] == sel) {
                s[u][0] = fmaf(t[u][0], qp.inva, qp.offa);
                s[u][1] = fmaf(t[u][1], qp.invb, qp.offb);
              }
              if (sely[u] == sel) {
                s[u][2] = fmaf(t[u][2], qp.inva, qp.offa);
                s[u][3] = fmaf(t[u][3], qp.invb, qp.offb);
              }
            }
          }
        } else {
          // residual keys (bf16 rows, 16 per warp: sub-block 0 only): the plain
          // query on the bf16 mma
          const uint32_t* qw = reinterpret_cast<const uint32_t*>(qrow);
          const bool okb16 = okq && !lo_lane;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(kt + tile_off<D * 2>(base0 + (lmat & 1) * 8 + lrow, 2 * kk + (lmat >> 1)), a[0], a[1], a[2], a[3]);
            mma_bf16(s[0], a, okb16 ? qw[8 * kk + t4] : 0u, okb16 ? qw[8 * kk + 4 + t4] : 0u);
          }
          if constexpr (PACKED) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[0][e] += __shfl_xor_sync(kAll, s[0][e], 2);
          }
        }
        // visibility: the slot's key, the row, the mask program.  A step of a
        // FULL stage whose slots all hold keys needs none of it (rows past
        // p.rows have a zero query, stay finite and are never written).
        float mxa = -INFINITY, mxb = -INFINITY;
        if (full && !resid && j0 + base0 + 16 * NS <= j1) {
#pragma unroll
          for (int u = 0; u < NS; ++u) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[u][e] *= sc;
            mxa = fmaxf(mxa, fmaxf(s[u][0], s[u][2]));
            mxb = fmaxf(mxb, fmaxf(s[u][1], s[u][3]));
          }
        } else {
#pragma unroll
          for (int u = 0; u < NS; ++u) {
            const bool live = !resid || u == 0;
            const int kx = base0 + 16 * u + g4, ky = kx + 8;
            const int tx = live ? pos[kx] : -1, ty = live ? pos[ky] : -1;
            bool vxa, vxb, vya, vyb;
            if constexpr (FM) {   // FlashMask: the producer's row bits of the columns
              const uint32_t* vis = reinterpret_cast<const uint32_t*>(smem + C::kVis) + st * kQKeys;
              const uint32_t bx = live ? vis[kx] : 0u, by = live ? vis[ky] : 0u;
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
            s[u][0] = vxa ? s[u][0] * sc : -INFINITY;
            s[u][1] = vxb ? s[u][1] * sc : -INFINITY;
            s[u][2] = vya ? s[u][2] * sc : -INFINITY;
            s[u][3] = vyb ? s[u][3] * sc : -INFINITY;
            mxa = fmaxf(mxa, fmaxf(s[u][0], s[u][2]));
            mxb = fmaxf(mxb, fmaxf(s[u][1], s[u][3]));
          }
        }
#pragma unroll
        for (int x = 4; x <= 16; x <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(kAll, mxa, x));
          mxb = fmaxf(mxb, __shfl_xor_sync(kAll, mxb, x));
        }
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        const float aa = na == -INFINITY ? 1.f : ex2_approx(ma - na);
        const float ab = nb == -INFINITY ? 1.f : ex2_approx(mb - nb);
        const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
        float pr[NS][4];
#pragma unroll
        for (int u = 0; u < NS; ++u) {
          pr[u][0] = ex2_approx(s[u][0] - ua);
          pr[u][1] = ex2_approx(s[u][1] - ub);
          pr[u][2] = ex2_approx(s[u][2] - ua);
          pr[u][3] = ex2_approx(s[u][3] - ub);
        }
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int u = 0; u < NS; ++u) {
          sa += pr[u][0] + pr[u][2];
          sb += pr[u][1] + pr[u][3];
        }
        la = la * aa + sa;
        lb = lb * ab + sb;
        ma = na;
        mb = nb;
        if (__any_sync(kAll, aa != 1.f || ab != 1.f)) {
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            o[n][0] *= aa;
            o[n][1] *= ab;
            o[n][2] *= aa;
            o[n][3] *= ab;
          }
#pragma unroll
          for (int x = 0; x < kCg; ++x) {
            za[x] *= aa;
            zb[x] *= ab;
          }
        }
        if (!resid) {
#pragma unroll
          for (int u = 0; u < NS; ++u) {
            const int kx = base0 + 16 * u + g4, ky = kx + 8;
            // per channel group: P' = p s_v (f16 pairs) as the B operand, sum p z_v aside
            uint32_t sx[kCg], sy[kCg];
            load_vq<kCg>(vq + C::kVQB * kx, sx);
            load_vq<kCg>(vq + C::kVQB * ky, sy);
            // rows (ra, rb) of keys g4 and g4 + 8
            const uint32_t px = pack_f16(pr[u][0], pr[u][1]), py = pack_f16(pr[u][2], pr[u][3]);
            uint32_t pb[kCg][2];
#pragma unroll
            for (int x = 0; x < kCg; ++x) {
              pb[x][0] = movmatrix_t(hmul2_lo(px, sx[x]));
              pb[x][1] = movmatrix_t(hmul2_lo(py, sy[x]));
              za[x] = fma_q_zhi<0>(px, sx[x], fma_q_zhi<0>(py, sy[x], za[x]));
              zb[x] = fma_q_zhi<1>(px, sx[x], fma_q_zhi<1>(py, sy[x], zb[x]));
            }
            // O'^T += V^T codes . P'^T
#pragma unroll
            for (int c2 = 0; c2 < D / 64; ++c2) {
              uint32_t v[4];
              ldsm_x4_trans(vt + code_off<D / 2>(base0 + 16 * u + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1],
                            v[2], v[3]);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int c = 2 * c2 + hh;   // code chunk c: channels 32 c .. 32 c + 31
                const uint32_t lo_keys = v[2 * hh], hi_keys = v[2 * hh + 1];
                const uint32_t lo8 = lo_keys >> 8, hi8 = hi_keys >> 8;
                // M rows g4 (even channel, low nibble) and g4 + 8 (odd channel, high nibble: 16 x)
                if constexpr (GV == 32) {   // chunk c is channel group c
                  const uint32_t a0[4] = {lo_keys & kNibLo, lo_keys & kNibHi, hi_keys & kNibLo, hi_keys & kNibHi};
                  mma_f16(o[2 * c], a0, pb[c][0], pb[c][1]);
                  const uint32_t a1[4] = {lo8 & kNibLo, lo8 & kNibHi, hi8 & kNibLo, hi8 & kNibHi};
                  mma_f16(o[2 * c + 1], a1, pb[c][0], pb[c][1]);
                } else {
                  // Gv = 16: the M rows of lanes g4 < 4 (channels 32 c + 0..15) are group
                  // 2 c, those of lanes g4 >= 4 group 2 c + 1; each group's mma sees the
                  // other group's rows as zero codes
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const uint32_t ml = e ? kNibLo ^ gmask_lo : gmask_lo, mh = e ? kNibHi ^ gmask_hi : gmask_hi;
                    const uint32_t a0[4] = {lo_keys & ml, lo_keys & mh, hi_keys & ml, hi_keys & mh};
                    mma_f16(o[2 * c], a0, pb[2 * c + e][0], pb[2 * c + e][1]);
                    const uint32_t a1[4] = {lo8 & ml, lo8 & mh, hi8 & ml, hi8 & mh};
                    mma_f16(o[2 * c + 1], a1, pb[2 * c + e][0], pb[2 * c + e][1]);
                  }
                }
              }
            }
          }
        } else {
          // bf16 V rows with the probabilities times 2^-24 (the accumulators' units)
          constexpr float kU = 1.f / kCodeUnit;
          const uint32_t pb0 = movmatrix_t(pack_bf16(pr[0][0] * kU, pr[0][1] * kU));
          const uint32_t pb1 = movmatrix_t(pack_bf16(pr[0][2] * kU, pr[0][3] * kU));
          // V^T in the quantized tiles' channel order: keys 2 t4, 2 t4 + 1 (and + 8)
          // at channels 32 c + 4 g4 + 0..3 (8 bytes of a bf16 row)
          const int ka = base0 + 2 * t4, kb2 = base0 + 8 + 2 * t4;
          const uint8_t* rv = stage + kRKeys * D * 2;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            const int chunk = 4 * c + (g4 >> 1), boff = 8 * (g4 & 1);
            const uint2 wa = *reinterpret_cast<const uint2*>(rv + tile_off<D * 2>(ka, chunk) + boff);
            const uint2 wb = *reinterpret_cast<const uint2*>(rv + tile_off<D * 2>(ka + 1, chunk) + boff);
            const uint2 wc = *reinterpret_cast<const uint2*>(rv + tile_off<D * 2>(kb2, chunk) + boff);
            const uint2 wd = *reinterpret_cast<const uint2*>(rv + tile_off<D * 2>(kb2 + 1, chunk) + boff);
            // M rows g4 + 8 carry the factor 16 of the quantized tiles' high nibbles
            const uint32_t a0[4] = {__byte_perm(wa.x, wb.x, 0x5410u), times16_bf16x2(__byte_perm(wa.x, wb.x, 0x7632u)),
                                    __byte_perm(wc.x, wd.x, 0x5410u), times16_bf16x2(__byte_perm(wc.x, wd.x, 0x7632u))};
            mma_bf16(o[2 * c], a0, pb0, pb1);
            const uint32_t a1[4] = {__byte_perm(wa.y, wb.y, 0x5410u), times16_bf16x2(__byte_perm(wa.y, wb.y, 0x7632u)),
                                    __byte_perm(wc.y, wd.y, 0x5410u), times16_bf16x2(__byte_perm(wc.y, wd.y, 0x7632u))};
            mma_bf16(o[2 * c + 1], a1, pb0, pb1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      j0 = j1;
    }

    // end of item: sums over the 8 lanes sharing t4; leave rows ra, rb
#pragma unroll
    for (int x = 4; x <= 16; x <<= 1) {
      la += __shfl_xor_sync(kAll, la, x);
      lb += __shfl_xor_sync(kAll, lb, x);
#pragma unroll
      for (int y = 0; y < kCg; ++y) {
        za[y] += __shfl_xor_sync(kAll, za[y], x);
        zb[y] += __shfl_xor_sync(kAll, zb[y], x);
      }
    }
    if (!dead && writer) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? rb : ra;
        if (!(rr ? okb : oka)) continue;
        const float m = rr ? mb : ma, l = rr ? lb : la;
        const int i = row / p.g, hq = it.h * p.g + row % p.g;
        const long long orow = (static_cast<long long>(qo) + i) * p.H_q + hq;
        float val[D / 32][4];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          // accumulator rows g4 in 2^-24 units, rows g4 + 8 in 2^-20 units; the lane's
          // channels 32 c + 4 g4 + 0..3 lie in V channel group c (Gv = 32) or
          // 2 c + (g4 >= 4) (Gv = 16)
          float add;
          if constexpr (GV == 32) add = rr ? zb[c] : za[c];
          else add = g4 < 4 ? (rr ? zb[2 * c] : za[2 * c]) : (rr ? zb[2 * c + 1] : za[2 * c + 1]);
          val[c][0] = fmaf(o[2 * c][rr], kCodeUnit, add);
          val[c][1] = fmaf(o[2 * c][2 + rr], kCodeUnit / 16.f, add);
          val[c][2] = fmaf(o[2 * c + 1][rr], kCodeUnit, add);
          val[c][3] = fmaf(o[2 * c + 1][2 + rr], kCodeUnit / 16.f, add);
        }
        if (it.slot < 0) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + 32 * c + 4 * g4);
            dst[0] = __floats2bfloat162_rn(val[c][0] * inv, val[c][1] * inv);
            dst[1] = __floats2bfloat162_rn(val[c][2] * inv, val[c][3] * inv);
          }
          if (g4 == 0 && p.lse) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
          const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
          float* u = p.u + srow * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            *reinterpret_cast<float4*>(u + 32 * c + 4 * g4) = make_float4(val[c][0], val[c][1], val[c][2], val[c][3]);
          if (g4 == 0) p.ml[srow] = make_float2(l > 0.f ? m : -INFINITY, l);
        }
      }
    } else if (dead && writer && it.slot >= 0 && g4 == 0) {   // the warp gave up: its states are marked
      if (oka) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + ra);
      if (okb) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + rb);
    }
  }
}

template <int D, int GV, bool FM>
__global__ void __launch_bounds__(kThreads, 1) partial_q4_kernel(const __grid_constant__ PartialParams p) {
  using C = Q4<D, GV, FM>;
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(q4_producer_regs<FM>()));
    produce_q4<D, GV, FM>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(q4_consumer_regs<FM>()));
  dependency_wait(!complete_now);   // before Q and the state writes
  if (p.rows <= 4) consume_q4<D, GV, FM, true>(w, smem, warp, lane);
  else consume_q4<D, GV, FM, false>(w, smem, warp, lane);
}

template <int D, int GV, bool FM>
int launch_d(const PartialParams& p, int n_ctas, void* stream) {
  const size_t smem = Q4<D, GV, FM>::kTotal;
  // the register budget check and the shared-memory opt-in, once per device
  static std::atomic<unsigned long long> ready{0};
  cudaError_t err = prepare_kernel_once(partial_q4_kernel<D, GV, FM>, smem,
                                        128 * q4_producer_regs<FM>() + 32 * kConsumerWarps * q4_consumer_regs<FM>(), ready);
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
  err = cudaLaunchKernelEx(&cfg, partial_q4_kernel<D, GV, FM>, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace

int launch_partial_q4(const PartialParams& p, int d, int n_ctas, void* stream) {
  if (p.mask == DATTN_MASK_FLASHMASK) {
    if (d == 64) return launch_d<64, 16, true>(p, n_ctas, stream);
    return p.kivi_Gv == 16 ? launch_d<128, 16, true>(p, n_ctas, stream) : launch_d<128, 32, true>(p, n_ctas, stream);
  }
  if (d == 64) return launch_d<64, 16, false>(p, n_ctas, stream);
  return p.kivi_Gv == 16 ? launch_d<128, 16, false>(p, n_ctas, stream) : launch_d<128, 32, false>(p, n_ctas, stream);
}

}  // namespace dattn
