// LSE merge of partial (m, l, u) states, one query row by one warp (the
// merge kernel's building block).
//
// "M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries":
// §0x02B binary merge through the common frame m = max(m_A, m_B), applied as
// a fold; §0x02C validity branch before any exponential (a state is empty iff
// l = 0, stored with m = -inf); O = u / l rounded to bf16, LSE = m + ln l, an
// all-masked row giving O = 0 and LSE = -inf.  m is in log2 units.
#pragma once

#include <cuda_bf16.h>

#include "device.cuh"

namespace dattn {

// A warp's running fold of one row: frame M (log2 units), sum L, the lane's
// D / 32 channels of u, and whether some state was marked unwritten (l = NaN:
// its partial-kernel warp gave up, see mark_state_unwritten) so that the row
// must not be written.
template <int D>
struct RowFold {
  float M, L, U[D / 32];
  bool bad;
};

template <int D>
__device__ __forceinline__ void fold_init(RowFold<D>& f) {
  f.bad = false;
  f.M = -INFINITY;
  f.L = 0.f;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) f.U[c] = 0.f;
}

// The state-row tags a merge warp waits for (see store_release_gpu): null
// when the whole partial grid is complete before the merge reads (then every
// state is).  A warp that sees no tag of this run for "limit_ns" gives up:
// status kStTimeout, and the row is not written.
struct StateTags {
  const int32_t* seq;   // [rows][n_slots]
  int32_t run_seq, n_slots;
  uint64_t limit_ns;
  int32_t* status;
};

__device__ __forceinline__ unsigned long long merge_now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits until the lane's state (lane < n) carries this run's tag in its row
// (the row's tags of consecutive states are adjacent: a warp's poll reads a
// few sectors); false when the wait gave up.  The acquire loads and the
// __syncwarp order every lane's later reads of the states after their tags.
__device__ __forceinline__ bool wait_state_tags(const StateTags& tg, long long tag, bool mine, int lane) {
  constexpr unsigned kAll = 0xffffffffu;
  bool ready = !mine || load_acquire_gpu(tg.seq + tag) == tg.run_seq;
  if (!__all_sync(kAll, ready)) {
    const unsigned long long t0 = merge_now_ns();
    for (;;) {
      __nanosleep(128);
      if (!ready) ready = load_acquire_gpu(tg.seq + tag) == tg.run_seq;
      if (__all_sync(kAll, ready)) break;
      if (merge_now_ns() - t0 > tg.limit_ns) {
        if (lane == 0) atomicOr(tg.status, kStTimeout);
        return false;
      }
    }
  }
  __syncwarp();
  return true;
}

// Folds states s_first + s_stride * i, i in [0, n), of row "row" into f.
// Lanes fetch (m, l) of 32 states at a time (TAGS: first waiting for their
// tags); the u vectors of the live ones are then read kBatch at a time with
// all loads in flight (a batch is unrolled: its unused slots still cost their
// predicated instructions).
template <int D, int kBatch = 8, bool TAGS = false>
__device__ __forceinline__ void fold_states(const float2* ml, const float* u, int rows, int row, int s_first,
                                            int n_states, int s_stride, int lane, RowFold<D>& f,
                                            const StateTags& tg = StateTags{}) {
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int C = D / 32;
  const long long stride = static_cast<long long>(s_stride) * rows * D;   // between consecutive states
  for (int i0 = 0; i0 < n_states; i0 += 32) {
    const int n = min(32, n_states - i0);
    const int s0 = s_first + s_stride * i0;
    if constexpr (TAGS) {
      if (!wait_state_tags(tg, static_cast<long long>(row) * tg.n_slots + s0 + s_stride * lane, lane < n, lane)) {
        f.bad = true;
        return;
      }
    }
    float2 v = make_float2(-INFINITY, 0.f);
    if (lane < n) v = __ldcg(ml + static_cast<long long>(s0 + s_stride * lane) * rows + row);
    if (__any_sync(kAll, v.y != v.y)) f.bad = true;    // a state marked unwritten
    const bool valid = v.y > 0.f;
    float mc = valid ? v.x : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kAll, mc, o));
    if (mc == -INFINITY) continue;
    const float m_new = fmaxf(f.M, mc);
    const float scale_old = f.M == -INFINITY ? 0.f : exp2f(f.M - m_new);
    const float wt = valid ? exp2f(v.x - m_new) : 0.f;
    float lw = wt * v.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(kAll, lw, o);
    f.L = f.L * scale_old + lw;
#pragma unroll
    for (int c = 0; c < C; ++c) f.U[c] *= scale_old;
    f.M = m_new;
    const unsigned live = __ballot_sync(kAll, valid);
    const float* u0 = u + (static_cast<long long>(s0) * rows + row) * D + lane * C;
    for (int q0 = 0; q0 < n; q0 += kBatch) {
      float x[kBatch][C];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const bool use = q0 + q < n && ((live >> (q0 + q)) & 1u);
        const float* src = u0 + (q0 + q) * stride;
        if constexpr (C == 4) {
          const float4 t = use ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          x[q][0] = t.x; x[q][1] = t.y; x[q][2] = t.z; x[q][3] = t.w;
        } else {
          const float2 t = use ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
          x[q][0] = t.x; x[q][1] = t.y;
        }
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const float wq = __shfl_sync(kAll, wt, (q0 + q) & 31);
#pragma unroll
        for (int c = 0; c < C; ++c) f.U[c] = fmaf(wq, x[q][c], f.U[c]);
      }
    }
  }
}

// Writes O (bf16, the lane's D / 32 channels) and LSE (natural log, lane 0)
// of output row "orow" from a finished fold.
template <int D>
__device__ __forceinline__ void write_folded_row(void* o, float* lse, long long orow, const RowFold<D>& f, int lane) {
  constexpr int C = D / 32;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(o) + orow * D + lane * C;
  const float inv = f.L > 0.f ? 1.f / f.L : 0.f;
#pragma unroll
  for (int c = 0; c < C; c += 2)
    *reinterpret_cast<__nv_bfloat162*>(out + c) = __floats2bfloat162_rn(f.U[c] * inv, f.U[c + 1] * inv);
  if (lane == 0 && lse) lse[orow] = f.L > 0.f ? (f.M + __log2f(f.L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace dattn
