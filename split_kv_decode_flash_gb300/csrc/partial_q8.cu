// Partial kernel of split-KV decode attention for byte-code K/V on the tensor
// cores: INT8 per-token ("M8.6 Live-Data Quantization", §0x05B format) and
// FP8 E4M3 / E5M2 with a per-head scale (§0x0A-0x0AA).  FP8 codes become exact
// f16 values (one cvt per E4M3 pair; an E5M2 byte is the upper byte of its f16)
// and have no offset, so their (s, z) are the head's scale and zero, and the
// 1024 bias below is zero.
//
// Same persistent producer / consumer structure as the bf16 kernel (item
// records in shared memory, four producer warps with a three-step slot
// description, per-warp partial states); stages hold 128 keys so that a
// stage carries as many bytes as a bf16 one.
//
// Producer.  Every key row's codes are copied with 16-byte cp.async into
// XOR-swizzled tiles, and its (s, z) fp16 pairs with 4-byte copies; empty
// slots are zero-filled.
//
// Consumers (two stage groups of four warps, 32 keys per warp and stage,
// in blocks of 16).  Scales stay where M8.6 §0x03 puts them:
//   K: q.k_hat = s_t (q . code_t) + z_t (q . 1).  K codes are read with
//      ldmatrix (byte pairs as 16-bit elements) and turned into f16 by one
//      prmt per pair (1024 + code, exact); q . (1024 + code) comes from
//      mma.sync.m16n8k16 f16 with the query rows converted to f16 (exact for
//      bf16 values in f16's range; rows whose largest |q| is beyond 2^14 are
//      scaled by a power of two first), fp32 accumulate, and the 1024 bias is
//      folded into the offset: s = s_t S' + (z_t - 1024 s_t) (q . 1).
//   V: sum_t p_t (s_t code_t + z_t) = sum_t (p_t s_t) code_t + sum_t p_t z_t.
//      P' = p s_t is the f16 A operand of the P V mma; V codes come from
//      ldmatrix.trans, so a lane holds the codes of two keys at two channels
//      and one prmt makes each B register.  The bias adds 1024 sum_t P'_t to
//      every channel, removed at the end together with adding
//      sum_t p_t z_t.  Output tile 2 C + e holds channels 16 C + 2 n + e.
// The online softmax is the same as in the bf16 kernel (log2 units, -inf
// for masked cells, row maxima over the lane quad).
#include <cuda_runtime.h>

#include "launch.cuh"
#include "tc_common.cuh"

namespace dattn {

namespace {

constexpr int kQK = 128;              // keys per stage
constexpr int kQS = kQK / 32;         // slots per producer lane
constexpr int kQ8ProducerRegs = 88;
constexpr int kQ8ConsumerRegs = 208;
static_assert(128 * kQ8ProducerRegs + 32 * kConsumerWarps * kQ8ConsumerRegs <= kThreads * 168, "register split");
// The FlashMask instance's producers carry four interval ends per slot a stage
// ahead: they get more of the register file.
constexpr int kQ8FmProducerRegs = 104;
constexpr int kQ8FmConsumerRegs = 200;
static_assert(128 * kQ8FmProducerRegs + 32 * kConsumerWarps * kQ8FmConsumerRegs <= kThreads * 168, "register split");
template <bool FM>
constexpr int q8_producer_regs() { return FM ? kQ8FmProducerRegs : kQ8ProducerRegs; }
template <bool FM>
constexpr int q8_consumer_regs() { return FM ? kQ8FmConsumerRegs : kQ8ConsumerRegs; }

template <int D>
struct Q8 {
  // Even depth: with two consumer stage groups taking alternate stages, every
  // ring slot always belongs to the same group (no mbarrier parity alias).
  static constexpr int kStagesN = D == 128 ? 6 : 10;
  static_assert(kStagesN % 2 == 0, "ring depth must be even");
  static constexpr int kRowB = D;                  // code bytes of one key row
  static constexpr int kChunks = kRowB / 16;
  static constexpr int kTile = kQK * kRowB;        // one tensor's codes
  static constexpr int kQp = kQK * 4;              // one tensor's (s, z) pairs
  static constexpr int kStage = 2 * kTile + 2 * kQp;
  static constexpr int kPos = kStagesN * kStage;   // int32 [stages][kQK]
  static constexpr int kVis = kPos + kStagesN * kQK * 4;   // uint32 [stages][kQK]: FlashMask row bits
  static constexpr int kFlags = kVis + kStagesN * kQK * 4;
  static constexpr int kSeq = kFlags + kStagesN * 4;
  static constexpr int kFullBar = align16(kSeq + kStagesN * 4);
  static constexpr int kEmptyBar = kFullBar + kStagesN * 8;
  static constexpr int kAbort = kEmptyBar + kStagesN * 8;
  static constexpr int kItems = align16(kAbort + 16);
  static constexpr int kTotal = kItems + kItemCache * static_cast<int>(sizeof(ItemRec));
  static_assert(kTotal <= 232448, "shared memory of one CTA");
};

// Two code bytes of w as an f16 pair; sel names them like a prmt selector:
// 0x4140 bytes 0 and 1, 0x4342 bytes 2 and 3, 0x4240 bytes 0 and 2, 0x4341
// bytes 1 and 3.  INT8: 1024 + byte each (exact), with kBias = 1024 to
// remove.  FP8 E4M3: the byte's value, exact in f16 (cvt.rn.f16x2.e4m3x2).
template <int FMT>
struct Codes;

template <>
struct Codes<DATTN_FMT_INT8_TOKEN> {
  static constexpr float kBias = 1024.f;
  static __device__ __forceinline__ uint32_t pair(uint32_t w, uint32_t sel) {
    return __byte_perm(w, 0x64646464u, sel);
  }
};

template <>
struct Codes<DATTN_FMT_FP8_E5M2> {
  static constexpr float kBias = 0.f;
  static __device__ __forceinline__ uint32_t pair(uint32_t w, uint32_t sel) {
    // byte A (sel nibble 0) to byte 1, byte B (nibble 2) to byte 3, zero low bytes
    return __byte_perm(w, 0u, 0x0404u | ((sel & 0xFu) << 4) | (((sel >> 8) & 0xFu) << 12));
  }
};

template <>
struct Codes<DATTN_FMT_FP8_E4M3> {
  static constexpr float kBias = 0.f;
  static __device__ __forceinline__ uint32_t pair(uint32_t w, uint32_t sel) {
    // the two bytes as the low half of a word: byte A (sel nibble 0) low, byte B (nibble 2) high
    const uint32_t b = sel == 0x4140u ? w : sel == 0x4342u ? w >> 16 : __byte_perm(w, 0u, (sel & 0xFu) | ((sel >> 4) & 0xF0u));
    uint32_t d;
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %1; cvt.rn.f16x2.e4m3x2 %0, lo; }" : "=r"(d) : "r"(b));
    return d;
  }
};

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// ---- producer ---------------------------------------------------------------------------

template <int D, int FMT, bool FM>
__device__ void produce_q8(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Q8<D>;
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
  pc_seek<kQK>(w, c0);
  pc_advance<kQK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kQK>(w, c1, kProducerWarps);
  PCur c2 = c1;
  pc_advance<kQK>(w, c2, kProducerWarps);
  if constexpr (!FM) index_list_prologue(w, c0, lane, dep_wait);   // index lists: list entries are device inputs
  const SlotKeys<kQS> k0 = slot_keys<kQS, !FM>(w, c0, lane);
  SlotKeys<kQS> k1 = slot_keys<kQS, !FM>(w, c1, lane);
  dependency_wait(dep_wait);   // the page table is a device input
  const SlotPages<kQS, FM> g0 = slot_pages<kQS, FM>(w, c0, k0);
  SlotPages<kQS, FM> g1 = slot_pages<kQS, FM>(w, c1, k1);
  SlotKeys<kQS> k2 = slot_keys<kQS, !FM>(w, c2, lane);
  SlotRows<kQS, FM> r0 = slot_rows<kQS, FM>(w, c0, k0, g0, lane);

  for (uint32_t k = pw; c0.ii < w.end; k += kProducerWarps) {
    const int st = k % C::kStagesN;
    const uint32_t use = k / C::kStagesN;
    if (use > 0 && !mbar_wait(empty0 + 8 * st, (use - 1) & 1, abort_flag, p.status)) break;
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kQK;
#pragma unroll
    for (int h = 0; h < kQS; ++h) pos[lane + 32 * h] = r0.t[h];
    if constexpr (FM) {
      uint32_t* vis = reinterpret_cast<uint32_t*>(smem + C::kVis) + st * kQK;
#pragma unroll
      for (int h = 0; h < kQS; ++h) vis[lane + 32 * h] = r0.vis[h];
    }
    if (lane == 0) {
      reinterpret_cast<int*>(smem + C::kFlags)[st] = r0.full ? kFlagFull : 0;
      reinterpret_cast<int*>(smem + C::kSeq)[st] = static_cast<int>(k);
    }
    const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
    const uint32_t kq = vt + C::kTile, vq = kq + C::kQp;
#pragma unroll
    for (int s0 = 0; s0 < kQK; s0 += kSlotsPerPass) {
      const int s = s0 + sub;
      const uint32_t row = __shfl_sync(kAll, r0.row[s0 / 32], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = tile_off<D>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
    if constexpr (FMT == DATTN_FMT_INT8_TOKEN) {   // per-token (s, z); FP8 has per-head scales
#pragma unroll
      for (int h = 0; h < kQS; ++h) {
        const uint32_t row = r0.row[h];
        const bool ok = row != kNoRow;
        const size_t off = static_cast<size_t>(ok ? row : 0u) * 4;
        cp_async4(kq + 4 * (lane + 32 * h), kqbase + off, ok ? 4u : 0u);
        cp_async4(vq + 4 * (lane + 32 * h), vqbase + off, ok ? 4u : 0u);
      }
    }
    const uint32_t fb = full0 + 8 * st;
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) mbar_arrive(fb);     // publishes pos / flags / stamp; the copies complete the phase

    r0 = slot_rows<kQS, FM>(w, c1, k1, g1, lane);
    c0 = c1;
    g1 = slot_pages<kQS, FM>(w, c2, k2);
    k1 = k2;
    c1 = c2;
    pc_advance<kQK>(w, c2, kProducerWarps);
    k2 = slot_keys<kQS, !FM>(w, c2, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

// The same producer for interval programs on power-of-two pages: one page id
// per lane and stage instead of a key, a page-table load and a row per slot
// (RunStage in tc_common.cuh).
template <int D, int FMT>
__device__ void produce_q8_runs(const Walk& w, uint8_t* smem, int lane, int pw, bool dep_wait) {
  using C = Q8<D>;
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
  pc_seek<kQK>(w, c0);
  pc_advance<kQK>(w, c0, pw);
  PCur c1 = c0;
  pc_advance<kQK>(w, c1, kProducerWarps);
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
    uint32_t rows[kQS];
    int* pos = reinterpret_cast<int*>(smem + C::kPos) + st * kQK;
#pragma unroll
    for (int h = 0; h < kQS; ++h) {
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
    for (int s0i = 0; s0i < kQK; s0i += kSlotsPerPass) {
      const int s = s0i + sub;
      const uint32_t row = __shfl_sync(kAll, rows[s0i / 32], s & 31);
      const bool ok = row != kNoRow;
      const size_t off = static_cast<size_t>(ok ? row : 0u) * C::kRowB + ch * 16;
      const uint32_t dst = tile_off<D>(s, ch);
      cp_async16(kt + dst, kbase + off, ok ? 16u : 0u, stream_pol);
      cp_async16(vt + dst, vbase + off, ok ? 16u : 0u, stream_pol);
    }
    if constexpr (FMT == DATTN_FMT_INT8_TOKEN) {   // per-token (s, z); FP8 has per-head scales
#pragma unroll
      for (int h = 0; h < kQS; ++h) {
        const uint32_t row = rows[h];
        const bool ok = row != kNoRow;
        const size_t off = static_cast<size_t>(ok ? row : 0u) * 4;
        cp_async4(kq + 4 * (lane + 32 * h), kqbase + off, ok ? 4u : 0u);
        cp_async4(vq + 4 * (lane + 32 * h), vqbase + off, ok ? 4u : 0u);
      }
    }
    const uint32_t fb = full0 + 8 * st;
    cp_async_mbar_arrive(fb);
    __syncwarp();
    if (lane == 0) mbar_arrive(fb);     // publishes pos / flags / stamp; the copies complete the phase

    c0 = c1;
    s0 = s1;
    g0 = g1;
    pc_advance<kQK>(w, c1, kProducerWarps);
    s1 = run_stage(w, c1);
    g1 = run_stage_page(w, s1, lane);
  }
  asm volatile("cp.async.wait_all;\n" ::: "memory");   // no copy of this thread outlives it
}

// ---- consumers --------------------------------------------------------------------------

// Query rows r0, r1 of item "it" as f16 A fragments in the channel order the
// K fragments use (k-step kk, lane quad t4: channels 16 kk + 4 t4 + 0..3),
// their channel sums, and the power-of-two factor each row was divided by to
// fit f16 (1 unless its largest |q| exceeds 2^14).
template <int D>
struct QRows {
  uint32_t a[D / 16][4];
  float qsum0, qsum1, fac0, fac1;
};

// rec: the item's record; its request's query rows are packed rows rec.qo ..
// rec.qo + rec.nq - 1 (a mixed batch, M4.5 §0x08F), and rows past g rec.nq are zero.
template <int D>
__device__ __forceinline__ void load_q8(const PartialParams& p, const ItemRec& rec, int r0, int r1, int t4,
                                        QRows<D>& q) {
  constexpr int KS = D / 16;
  const WorkItem& it = rec.it;
  const bool ok0 = r0 < p.g * rec.nq, ok1 = r1 < p.g * rec.nq;
  const __nv_bfloat16* q0 = static_cast<const __nv_bfloat16*>(p.q) +
                            ((static_cast<long long>(rec.qo) + r0 / p.g) * p.H_q + it.h * p.g + r0 % p.g) * D;
  const __nv_bfloat16* q1 = static_cast<const __nv_bfloat16*>(p.q) +
                            ((static_cast<long long>(rec.qo) + r1 / p.g) * p.H_q + it.h * p.g + r1 % p.g) * D;
  float v0[KS][4], v1[KS][4];
  float mx0 = 0.f, mx1 = 0.f, s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    uint2 w0 = make_uint2(0u, 0u), w1 = make_uint2(0u, 0u);
    if (ok0) w0 = *reinterpret_cast<const uint2*>(q0 + 16 * kk + 4 * t4);
    if (ok1) w1 = *reinterpret_cast<const uint2*>(q1 + 16 * kk + 4 * t4);
    const float2 a = bf16x2_to_float2(w0.x), b = bf16x2_to_float2(w0.y);
    const float2 c = bf16x2_to_float2(w1.x), d = bf16x2_to_float2(w1.y);
    v0[kk][0] = a.x; v0[kk][1] = a.y; v0[kk][2] = b.x; v0[kk][3] = b.y;
    v1[kk][0] = c.x; v1[kk][1] = c.y; v1[kk][2] = d.x; v1[kk][3] = d.y;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx0 = fmaxf(mx0, fabsf(v0[kk][e]));
      mx1 = fmaxf(mx1, fabsf(v1[kk][e]));
      s0 += v0[kk][e];
      s1 += v1[kk][e];
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(kAll, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kAll, mx1, o));
    s0 += __shfl_xor_sync(kAll, s0, o);
    s1 += __shfl_xor_sync(kAll, s1, o);
  }
  // power-of-two scale that brings the row below 2^14 (exact in f16)
  q.fac0 = mx0 > 16384.f ? exp2f(ceilf(log2f(mx0 / 16384.f))) : 1.f;
  q.fac1 = mx1 > 16384.f ? exp2f(ceilf(log2f(mx1 / 16384.f))) : 1.f;
  const float i0 = 1.f / q.fac0, i1 = 1.f / q.fac1;
  q.qsum0 = s0;
  q.qsum1 = s1;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    q.a[kk][0] = pack_f16(v0[kk][0] * i0, v0[kk][1] * i0);
    q.a[kk][1] = pack_f16(v1[kk][0] * i1, v1[kk][1] * i1);
    q.a[kk][2] = pack_f16(v0[kk][2] * i0, v0[kk][3] * i0);
    q.a[kk][3] = pack_f16(v1[kk][2] * i1, v1[kk][3] * i1);
  }
}

// Writes one accumulator row: O / LSE when the item is its group's only
// chunk, else the row's partial state.  Output tile 2 C + e holds, in
// columns 2 t4 and 2 t4 + 1, channels 16 C + 4 t4 + e and 16 C + 4 t4 + 2 + e;
// "bias" (1024 sum P') is removed and z (sum p z) added on every channel, and
// the result multiplied by vsc (FP8: the head's V scale, kept out of the f16
// probabilities so that they stay in f16's normal range).
template <int D>
__device__ __forceinline__ void emit_row_q8(const PartialParams& p, const WorkItem& it, int qo, int my_state, int row,
                                            float m, float l, float z, float bias, float vsc,
                                            const float (&o)[D / 8][4], int half, int t4) {
  const int i = row / p.g, hq = it.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(qo) + i) * p.H_q + hq;
  const float add = z - bias;
  if (it.slot < 0) {
    const float inv = l > 0.f ? vsc / l : 0.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const float* a0 = o[2 * c], *a1 = o[2 * c + 1];
      __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + 16 * c + 4 * t4);
      dst[0] = __floats2bfloat162_rn((a0[2 * half] + add) * inv, (a1[2 * half] + add) * inv);
      dst[1] = __floats2bfloat162_rn((a0[2 * half + 1] + add) * inv, (a1[2 * half + 1] + add) * inv);
    }
    if (t4 == 0 && p.lse) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
  } else {
    const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
    float* u = p.u + srow * D;
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      const float* a0 = o[2 * c], *a1 = o[2 * c + 1];
      *reinterpret_cast<float4*>(u + 16 * c + 4 * t4) =
          make_float4((a0[2 * half] + add) * vsc, (a1[2 * half] + add) * vsc, (a0[2 * half + 1] + add) * vsc,
                      (a1[2 * half + 1] + add) * vsc);
    }
    if (t4 == 0) p.ml[srow] = make_float2(l > 0.f ? m : -INFINITY, l);
  }
}

// FM: FlashMask columns (the row bits of each key column from the producer);
// the other programs are compiled without them.
template <int D, int FMT, bool FM>
__device__ void consume_q8(const Walk& w, uint8_t* smem, int cw, int lane) {
  using C = Q8<D>;
  constexpr int KS = D / 16;   // k-steps of q.k
  constexpr int NT = D / 8;    // 8-channel output tiles
  const PartialParams& p = w.p;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);

  const int nrb = p.rows <= 16 ? 1 : 2;
  const int ng = nrb == 1 ? 2 : 1;
  const int wps = kConsumerWarps / ng;
  const int sgrp = cw / wps, wi = cw % wps;
  const int rb = wi % nrb, ts = wi / nrb;
  const int my_state = (cw - rb) / nrb;
  const int keys_per_warp = kQK / (wps / nrb);     // 32
  const int g4 = lane >> 2, t4 = lane & 3;
  const int r0 = rb * 16 + g4, r1 = r0 + 8;
  const int qi0 = r0 / p.g, qi1 = r1 / p.g;
  const int lrow = lane & 7, lmat = lane >> 3;   // ldmatrix address roles
  const float sc = p.scale_log2;

  uint32_t k = 0;
  bool dead = false;

  for (int ii = w.begin; ii < w.end; ++ii) {
    const WorkItem it = w.rec(ii).it;
    const int nq = w.rec(ii).nq;                  // the request's query rows
    const MaskCtx mc{p.mask, nq, it.T, p.n_sink, p.window};
    const bool ok0 = r0 < p.g * nq, ok1 = r1 < p.g * nq;
    // the item's query rows (loading the next item's during this one held their
    // registers through the item: tree verify 65.2 -> 66.2 us, a mixed batch 67.3 -> 70.0)
    QRows<D> q;
    load_q8<D>(p, w.rec(ii), r0, r1, t4, q);
    float hk = 1.f, hv = 1.f;   // FP8: the kv head's scales (1 when not given); INT8: 1
    if constexpr (FMT != DATTN_FMT_INT8_TOKEN) {
      if (p.kqp) hk = static_cast<const float*>(p.kqp)[it.h];
      if (p.vqp) hv = static_cast<const float*>(p.vqp)[it.h];
    }
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f, z0 = 0.f, z1 = 0.f, b0 = 0.f, b1 = 0.f;

    for (int j0 = it.a; j0 < it.e; ++k) {
      const int j1 = min(j0 + kQK, it.e);
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
      const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kQK;
      const uint32_t* vis = reinterpret_cast<const uint32_t*>(smem + C::kVis) + st * kQK;
      const bool full = reinterpret_cast<const int*>(smem + C::kFlags)[st] & kFlagFull;
      const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
      const uint32_t* kqp = reinterpret_cast<const uint32_t*>(smem + st * C::kStage + 2 * C::kTile);
      const uint32_t* vqp = kqp + kQK;

      for (int blk = 0; blk < keys_per_warp / 16; ++blk) {
        const int base = ts * keys_per_warp + blk * 16;
        // q . (1024 + code) over 16 keys (two 8-key tiles); one ldmatrix.x4
        // gives a lane 4 codes of its key for each of 4 k-steps
        float s[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
          for (int m = 0; m < KS / 4; ++m) {
            uint32_t r[4];
            ldsm_x4(kt + tile_off<D>(base + nt * 8 + lrow, 4 * m + lmat), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              mma_f16(s[nt], q.a[4 * m + i], Codes<FMT>::pair(r[i], 0x4140u), Codes<FMT>::pair(r[i], 0x4342u));
          }
        }
        // per-token K scale outside the dot, log2 units, -inf where masked
        float vs[2][2], vz[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int slot = base + nt * 8 + 2 * t4 + e;
            const int t = pos[slot];
            const float2 ks = FMT == DATTN_FMT_INT8_TOKEN ? half2_bits_to_float2(kqp[slot]) : make_float2(hk, 0.f);
            const float2 vq = FMT == DATTN_FMT_INT8_TOKEN ? half2_bits_to_float2(vqp[slot]) : make_float2(1.f, 0.f);
            vs[nt][e] = vq.x;
            vz[nt][e] = vq.y;
            const float off = fmaf(-Codes<FMT>::kBias, ks.x, ks.y);
            bool v0, v1;
            if constexpr (FM) {   // FlashMask: the producer's row bits of the column
              const uint32_t bits = vis[slot];
              v0 = t >= 0 && ok0 && (full || ((bits >> qi0) & 1u));
              v1 = t >= 0 && ok1 && (full || ((bits >> qi1) & 1u));
            } else {
              v0 = t >= 0 && ok0 && (full || key_visible(mc, qi0, t));
              v1 = t >= 0 && ok1 && (full || key_visible(mc, qi1, t));
            }
            s[nt][e] = v0 ? sc * fmaf(ks.x * q.fac0, s[nt][e], off * q.qsum0) : -INFINITY;
            s[nt][2 + e] = v1 ? sc * fmaf(ks.x * q.fac1, s[nt][2 + e], off * q.qsum1) : -INFINITY;
          }
        }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kAll, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kAll, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(kAll, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kAll, mx1, 2));
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float a0 = n0 == -INFINITY ? 1.f : ex2_approx(m0 - n0);
        const float a1 = n1 == -INFINITY ? 1.f : ex2_approx(m1 - n1);
        const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = ex2_approx(s[nt][0] - u0);
          pr[nt][1] = ex2_approx(s[nt][1] - u0);
          pr[nt][2] = ex2_approx(s[nt][2] - u1);
          pr[nt][3] = ex2_approx(s[nt][3] - u1);
        }
        // per-token V scale folded into the probabilities (the f16 A operand)
        const uint32_t pa[4] = {pack_f16(pr[0][0] * vs[0][0], pr[0][1] * vs[0][1]),
                                pack_f16(pr[0][2] * vs[0][0], pr[0][3] * vs[0][1]),
                                pack_f16(pr[1][0] * vs[1][0], pr[1][1] * vs[1][1]),
                                pack_f16(pr[1][2] * vs[1][0], pr[1][3] * vs[1][1])};
        // sums of the f16 P' values the mma uses (rows r0: pa 0, 2; r1: pa 1, 3)
        const float2 q0a = half2_bits_to_float2(pa[0]), q0b = half2_bits_to_float2(pa[2]);
        const float2 q1a = half2_bits_to_float2(pa[1]), q1b = half2_bits_to_float2(pa[3]);
        l0 = l0 * a0 + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
        l1 = l1 * a1 + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
        z0 = z0 * a0 + ((pr[0][0] * vz[0][0] + pr[0][1] * vz[0][1]) + (pr[1][0] * vz[1][0] + pr[1][1] * vz[1][1]));
        z1 = z1 * a1 + ((pr[0][2] * vz[0][0] + pr[0][3] * vz[0][1]) + (pr[1][2] * vz[1][0] + pr[1][3] * vz[1][1]));
        b0 = b0 * a0 + ((q0a.x + q0a.y) + (q0b.x + q0b.y));
        b1 = b1 * a1 + ((q1a.x + q1a.y) + (q1b.x + q1b.y));
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
        // V codes by ldmatrix.trans: matrices (keys 0-7 | 8-15) x chunks (2 c2, 2 c2 + 1);
        // a lane gets keys (2 t4, 2 t4 + 1) at channels 16 C + 2 g4 + {0, 1}
#pragma unroll
        for (int c2 = 0; c2 < D / 32; ++c2) {
          uint32_t v[4];
          ldsm_x4_trans(vt + tile_off<D>(base + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1], v[2], v[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {          // chunk 2 c2 + h: v[2 h] keys 0-7, v[2 h + 1] keys 8-15
            const int C = 2 * c2 + h;
            mma_f16(o[2 * C], pa, Codes<FMT>::pair(v[2 * h], 0x4240u), Codes<FMT>::pair(v[2 * h + 1], 0x4240u));
            mma_f16(o[2 * C + 1], pa, Codes<FMT>::pair(v[2 * h], 0x4341u), Codes<FMT>::pair(v[2 * h + 1], 0x4341u));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      j0 = j1;
    }

    // end of item: row sums and value offsets over the quad; leave the rows
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      l0 += __shfl_xor_sync(kAll, l0, x);
      l1 += __shfl_xor_sync(kAll, l1, x);
      z0 += __shfl_xor_sync(kAll, z0, x);
      z1 += __shfl_xor_sync(kAll, z1, x);
      b0 += __shfl_xor_sync(kAll, b0, x);
      b1 += __shfl_xor_sync(kAll, b1, x);
    }
    if (!dead) {
      const int qo = w.rec(ii).qo;
      if (ok0) emit_row_q8<D>(p, it, qo, my_state, r0, m0, l0, z0, Codes<FMT>::kBias * b0, hv, o, 0, t4);
      if (ok1) emit_row_q8<D>(p, it, qo, my_state, r1, m1, l1, z1, Codes<FMT>::kBias * b1, hv, o, 1, t4);
    } else if (it.slot >= 0 && t4 == 0) {   // the warp gave up: its states are marked, never guessed
      if (ok0) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + r0);
      if (ok1) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + r1);
    }
  }
}

// ---- consumers, at most 8 query rows: keys on the M side of the mma ----------------
//
// S^T (16 keys x 8 rows) = codes (A, keys x d) . Q^T (B): one mma per k-step
// for 16 keys.  A lane's accumulators hold keys g4, g4 + 8 for rows 2 t4,
// 2 t4 + 1; row maxima and sums reduce over the 8 lanes that share t4.  The
// probabilities (times the V scale) are packed to f16 and transposed with
// movmatrix into the B operand of O^T (16 channels x 8 rows) = V^T codes (A,
// from ldmatrix.trans) . P'^T: one mma per 16 channels for 16 keys.  Output
// tile C holds channels 16 C + 2 g4 (rows: columns) and 16 C + 2 g4 + 1.

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Query row g4 as f16 B fragments (k-step kk: channels 16 kk + 4 t4 + 0..3),
// with the row's channel sum and power-of-two f16 scale, both handed to the
// lanes that own rows 2 t4 and 2 t4 + 1 of the accumulators.
template <int D>
struct QCols {
  uint32_t b[D / 16][2];
  float qsum0, qsum1, fac0, fac1;   // rows 2 t4, 2 t4 + 1
};

template <int D>
__device__ __forceinline__ void load_q8_cols(const PartialParams& p, const ItemRec& rec, int g4, int t4,
                                             QCols<D>& q) {
  constexpr int KS = D / 16;
  const WorkItem& it = rec.it;
  const bool ok = g4 < p.g * rec.nq;
  const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(p.q) +
                            ((static_cast<long long>(rec.qo) + g4 / p.g) * p.H_q + it.h * p.g + g4 % p.g) * D;
  float v[KS][4];
  float mx = 0.f, sum = 0.f;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    uint2 w = make_uint2(0u, 0u);
    if (ok) w = *reinterpret_cast<const uint2*>(qr + 16 * kk + 4 * t4);
    const float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
    v[kk][0] = a.x; v[kk][1] = a.y; v[kk][2] = b.x; v[kk][3] = b.y;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      mx = fmaxf(mx, fabsf(v[kk][e]));
      sum += v[kk][e];
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, o));
    sum += __shfl_xor_sync(kAll, sum, o);
  }
  const float fac = mx > 16384.f ? exp2f(ceilf(log2f(mx / 16384.f))) : 1.f;
  const float inv = 1.f / fac;
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    q.b[kk][0] = pack_f16(v[kk][0] * inv, v[kk][1] * inv);
    q.b[kk][1] = pack_f16(v[kk][2] * inv, v[kk][3] * inv);
  }
  // row r's values live in the quad g4 = r (lanes 4 r .. 4 r + 3)
  q.qsum0 = __shfl_sync(kAll, sum, 8 * t4);
  q.qsum1 = __shfl_sync(kAll, sum, 8 * t4 + 4);
  q.fac0 = __shfl_sync(kAll, fac, 8 * t4);
  q.fac1 = __shfl_sync(kAll, fac, 8 * t4 + 4);
}

template <int D, int FMT, bool FM>
__device__ void consume_q8_swap(const Walk& w, uint8_t* smem, int cw, int lane) {
  using C = Q8<D>;
  constexpr int KS = D / 16;   // k-steps of q.k
  constexpr int NC = D / 16;   // 16-channel output tiles
  const PartialParams& p = w.p;
  const uint32_t full0 = smem_u32(smem + C::kFullBar);
  const uint32_t empty0 = smem_u32(smem + C::kEmptyBar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kAbort);

  constexpr int ng = 2;                         // stage groups of four warps
  const int wps = kConsumerWarps / ng;
  const int sgrp = cw / wps, ts = cw % wps;
  const int my_state = cw;
  const int keys_per_warp = kQK / wps;          // 32
  const int g4 = lane >> 2, t4 = lane & 3;
  const int ra = 2 * t4, rb = 2 * t4 + 1;       // the lane's accumulator rows
  const int qia = ra / p.g, qib = rb / p.g;
  const int lrow = lane & 7, lmat = lane >> 3;
  const float sc = p.scale_log2;

  uint32_t k = 0;
  bool dead = false;
  QCols<D> qn;
  if (w.begin < w.end) load_q8_cols<D>(p, w.rec(w.begin), g4, t4, qn);
  for (int ii = w.begin; ii < w.end; ++ii) {
    const WorkItem it = w.rec(ii).it;
    const int nq = w.rec(ii).nq;                  // the request's query rows
    const MaskCtx mc{p.mask, nq, it.T, p.n_sink, p.window};
    const bool oka = ra < p.g * nq, okb = rb < p.g * nq;
    const QCols<D> q = qn;
    if (ii + 1 < w.end) load_q8_cols<D>(p, w.rec(ii + 1), g4, t4, qn);
    float hk = 1.f, hv = 1.f;   // FP8: the kv head's scales (1 when not given); INT8: 1
    if constexpr (FMT != DATTN_FMT_INT8_TOKEN) {
      if (p.kqp) hk = static_cast<const float*>(p.kqp)[it.h];
      if (p.vqp) hv = static_cast<const float*>(p.vqp)[it.h];
    }
    float o[NC][4];
#pragma unroll
    for (int n = 0; n < NC; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    // per lane, rows ra / rb: running max, and partial sums over the lane's keys of
    // p, p z_v and the f16 P' the mma used
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f, za = 0.f, zb = 0.f, ba = 0.f, bb = 0.f;

    for (int j0 = it.a; j0 < it.e; ++k) {
      const int j1 = min(j0 + kQK, it.e);
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
      const int* pos = reinterpret_cast<const int*>(smem + C::kPos) + st * kQK;
      const uint32_t* vis = reinterpret_cast<const uint32_t*>(smem + C::kVis) + st * kQK;
      const bool full = reinterpret_cast<const int*>(smem + C::kFlags)[st] & kFlagFull;
      const uint32_t kt = smem_u32(smem + st * C::kStage), vt = kt + C::kTile;
      const uint32_t* kqp = reinterpret_cast<const uint32_t*>(smem + st * C::kStage + 2 * C::kTile);
      const uint32_t* vqp = kqp + kQK;

      for (int blk = 0; blk < keys_per_warp / 16; ++blk) {
        const int base = ts * keys_per_warp + blk * 16;
        // S'^T = (1024 + codes) . Q^T: ldmatrix.x4 gives keys g4 and g4 + 8 at
        // two k-steps; one prmt per f16 pair
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c2 = 0; c2 < KS / 2; ++c2) {
          uint32_t v[4];
          ldsm_x4(kt + tile_off<D>(base + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1], v[2], v[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a[4] = {Codes<FMT>::pair(v[2 * h], 0x4140u), Codes<FMT>::pair(v[2 * h + 1], 0x4140u),
                                   Codes<FMT>::pair(v[2 * h], 0x4342u), Codes<FMT>::pair(v[2 * h + 1], 0x4342u)};
            mma_f16(s, a, q.b[2 * c2 + h][0], q.b[2 * c2 + h][1]);
          }
        }
        // keys g4 (s0, s1) and g4 + 8 (s2, s3); rows ra (s0, s2), rb (s1, s3)
        const int kx = base + g4, ky = base + g4 + 8;
        const int tx = pos[kx], ty = pos[ky];
        constexpr bool kI8 = FMT == DATTN_FMT_INT8_TOKEN;
        const float2 ksx = kI8 ? half2_bits_to_float2(kqp[kx]) : make_float2(hk, 0.f);
        const float2 ksy = kI8 ? half2_bits_to_float2(kqp[ky]) : make_float2(hk, 0.f);
        const float2 vqx = kI8 ? half2_bits_to_float2(vqp[kx]) : make_float2(1.f, 0.f);
        const float2 vqy = kI8 ? half2_bits_to_float2(vqp[ky]) : make_float2(1.f, 0.f);
        const float offx = fmaf(-Codes<FMT>::kBias, ksx.x, ksx.y), offy = fmaf(-Codes<FMT>::kBias, ksy.x, ksy.y);
        bool vxa, vxb, vya, vyb;
        if constexpr (FM) {   // FlashMask: the producer's row bits of the columns
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
        s[0] = vxa ? sc * fmaf(ksx.x * q.fac0, s[0], offx * q.qsum0) : -INFINITY;
        s[1] = vxb ? sc * fmaf(ksx.x * q.fac1, s[1], offx * q.qsum1) : -INFINITY;
        s[2] = vya ? sc * fmaf(ksy.x * q.fac0, s[2], offy * q.qsum0) : -INFINITY;
        s[3] = vyb ? sc * fmaf(ksy.x * q.fac1, s[3], offy * q.qsum1) : -INFINITY;
        // row maxima over the 8 lanes sharing t4
        float mxa = fmaxf(s[0], s[2]), mxb = fmaxf(s[1], s[3]);
#pragma unroll
        for (int x = 4; x <= 16; x <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(kAll, mxa, x));
          mxb = fmaxf(mxb, __shfl_xor_sync(kAll, mxb, x));
        }
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        const float aa = na == -INFINITY ? 1.f : ex2_approx(ma - na);
        const float ab = nb == -INFINITY ? 1.f : ex2_approx(mb - nb);
        const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
        const float p0 = ex2_approx(s[0] - ua), p1 = ex2_approx(s[1] - ub), p2 = ex2_approx(s[2] - ua), p3 = ex2_approx(s[3] - ub);
        // P'^T (keys x rows), V scale folded in, f16; transposed into B fragments
        const uint32_t px = pack_f16(p0 * vqx.x, p1 * vqx.x), py = pack_f16(p2 * vqy.x, p3 * vqy.x);
        const float2 fx = half2_bits_to_float2(px), fy = half2_bits_to_float2(py);
        la = la * aa + (p0 + p2);
        lb = lb * ab + (p1 + p3);
        za = za * aa + (p0 * vqx.y + p2 * vqy.y);
        zb = zb * ab + (p1 * vqx.y + p3 * vqy.y);
        ba = ba * aa + (fx.x + fy.x);
        bb = bb * ab + (fx.y + fy.y);
        ma = na;
        mb = nb;
        if (__any_sync(kAll, aa != 1.f || ab != 1.f)) {
#pragma unroll
          for (int n = 0; n < NC; ++n) {
            o[n][0] *= aa;
            o[n][1] *= ab;
            o[n][2] *= aa;
            o[n][3] *= ab;
          }
        }
        const uint32_t pb0 = movmatrix_trans(px), pb1 = movmatrix_trans(py);
        // O'^T += V^T codes . P'^T: ldmatrix.trans gives keys (2 t4, 2 t4 + 1) of
        // keys 0-7 / 8-15 at channel pair g4 of two chunks
#pragma unroll
        for (int c2 = 0; c2 < NC / 2; ++c2) {
          uint32_t v[4];
          ldsm_x4_trans(vt + tile_off<D>(base + (lmat & 1) * 8 + lrow, 2 * c2 + (lmat >> 1)), v[0], v[1], v[2], v[3]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t a[4] = {Codes<FMT>::pair(v[2 * h], 0x4240u), Codes<FMT>::pair(v[2 * h], 0x4341u),
                                   Codes<FMT>::pair(v[2 * h + 1], 0x4240u), Codes<FMT>::pair(v[2 * h + 1], 0x4341u)};
            mma_f16(o[2 * c2 + h], a, pb0, pb1);
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
      ba += __shfl_xor_sync(kAll, ba, x);
      bb += __shfl_xor_sync(kAll, bb, x);
    }
    if (!dead) {
      const int qo = w.rec(ii).qo;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int row = rr ? rb : ra;
        if (!(rr ? okb : oka)) continue;
        const float m = rr ? mb : ma, l = rr ? lb : la;
        const float add = (rr ? zb : za) - Codes<FMT>::kBias * (rr ? bb : ba);
        const int i = row / p.g, hq = it.h * p.g + row % p.g;
        const long long orow = (static_cast<long long>(qo) + i) * p.H_q + hq;
        if (it.slot < 0) {
          const float inv = l > 0.f ? hv / l : 0.f;
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + orow * D;
#pragma unroll
          for (int c = 0; c < NC; ++c)
            *reinterpret_cast<__nv_bfloat162*>(out + 16 * c + 2 * g4) =
                __floats2bfloat162_rn((o[c][rr] + add) * inv, (o[c][2 + rr] + add) * inv);
          if (g4 == 0 && p.lse) p.lse[orow] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
        } else {
          const long long srow = static_cast<long long>(it.slot + my_state) * p.rows + row;
          float* u = p.u + srow * D;
#pragma unroll
          for (int c = 0; c < NC; ++c)
            *reinterpret_cast<float2*>(u + 16 * c + 2 * g4) = make_float2((o[c][rr] + add) * hv, (o[c][2 + rr] + add) * hv);
          if (g4 == 0) p.ml[srow] = make_float2(l > 0.f ? m : -INFINITY, l);
        }
      }
    } else if (it.slot >= 0 && g4 == 0) {   // the warp gave up: its states are marked, never guessed
      if (oka) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + ra);
      if (okb) mark_state_unwritten(p.ml, static_cast<long long>(it.slot + my_state) * p.rows + rb);
    }
  }
}

// FM: the FlashMask instance (producers carry each column's row bits), launched
// only for that program; the other programs run the instance compiled without it.
template <int D, int FMT, bool FM>
__global__ void __launch_bounds__(kThreads, 1) partial_q8_kernel(const __grid_constant__ PartialParams p) {
  using C = Q8<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  // the merge kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int it_begin = p.cta_indptr[blockIdx.x], it_end = p.cta_indptr[blockIdx.x + 1];
  ItemRec* cache = reinterpret_cast<ItemRec*>(smem + C::kItems);
  const int incomplete = fill_item_cache(p, cache, it_begin, it_end);
  if (threadIdx.x == 0) {
    const int warps_per_stage = p.rows <= 16 ? kConsumerWarps / 2 : kConsumerWarps;
    for (int s = 0; s < C::kStagesN; ++s) {
      mbar_init(smem_u32(smem + C::kFullBar + 8 * s), 1);
      mbar_init(smem_u32(smem + C::kEmptyBar + 8 * s), warps_per_stage);
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
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(q8_producer_regs<FM>()));
    if constexpr (FM) produce_q8<D, FMT, true>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else if (runs_apply<kQK>(p)) produce_q8_runs<D, FMT>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    else produce_q8<D, FMT, false>(w, smem, lane, warp - kConsumerWarps, !complete_now);
    return;
  }
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(q8_consumer_regs<FM>()));
  dependency_wait(!complete_now);   // before Q and the state writes
  if (p.rows <= 8) consume_q8_swap<D, FMT, FM>(w, smem, warp, lane);
  else consume_q8<D, FMT, FM>(w, smem, warp, lane);
}

template <int D, int FMT, bool FM>
int launch_q8_inst(const PartialParams& p, int n_ctas, void* stream) {
  const size_t smem = Q8<D>::kTotal;
  // the register budget check and the shared-memory opt-in, once per device
  static std::atomic<unsigned long long> ready{0};
  cudaError_t err = prepare_kernel_once(partial_q8_kernel<D, FMT, FM>, smem, 128 * q8_producer_regs<FM>() + 32 * kConsumerWarps * q8_consumer_regs<FM>(), ready);
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
  err = cudaLaunchKernelEx(&cfg, partial_q8_kernel<D, FMT, FM>, p);
  return err != cudaSuccess ? err : cudaGetLastError();
}

template <int D, int FMT>
int launch_q8(const PartialParams& p, int n_ctas, void* stream) {
  return p.mask == DATTN_MASK_FLASHMASK ? launch_q8_inst<D, FMT, true>(p, n_ctas, stream)
                                        : launch_q8_inst<D, FMT, false>(p, n_ctas, stream);
}

}  // namespace

int launch_partial_q8(const PartialParams& p, int d, int n_ctas, void* stream) {
  if (p.fmt == DATTN_FMT_FP8_E4M3)
    return d == 64 ? launch_q8<64, DATTN_FMT_FP8_E4M3>(p, n_ctas, stream)
                   : launch_q8<128, DATTN_FMT_FP8_E4M3>(p, n_ctas, stream);
  if (p.fmt == DATTN_FMT_FP8_E5M2)
    return d == 64 ? launch_q8<64, DATTN_FMT_FP8_E5M2>(p, n_ctas, stream)
                   : launch_q8<128, DATTN_FMT_FP8_E5M2>(p, n_ctas, stream);
  return d == 64 ? launch_q8<64, DATTN_FMT_INT8_TOKEN>(p, n_ctas, stream)
                 : launch_q8<128, DATTN_FMT_INT8_TOKEN>(p, n_ctas, stream);
}

}  // namespace dattn
