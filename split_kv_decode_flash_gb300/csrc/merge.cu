// LSE-merge kernel: folds the partial (m, l, u) states of every (request, kv
// head) group that the planner cut into several chunks.
//
// "M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries":
// §0x02B binary merge through the common frame m = max(m_A, m_B), applied as
// a running fold; §0x02C validity branch before any exponential (a state is
// empty iff l = 0, stored with m = -inf); O = u / l rounded to bf16 and
// LSE = m + ln l, all-masked rows giving O = 0 and LSE = -inf.  One warp
// owns one query row; each lane owns d / 32 channels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace dattn {

namespace {

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int C = D / 32;
  constexpr unsigned kAll = 0xffffffffu;
  __shared__ float sm_u[4][D];
  __shared__ float sm_ml[4][2];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = blockIdx.x / p.rows, row = blockIdx.x % p.rows;
  const MergeGroup grp = p.groups[gi];

  // Warp w folds chunks w, w + 4, ... of 32 states: every lane fetches one
  // state's (m, l), the warp agrees on the frame, then the u vectors are read
  // back to back with the weights broadcast.
  float M = -INFINITY, Lsum = 0.f, U[C];
#pragma unroll
  for (int c = 0; c < C; ++c) U[c] = 0.f;
  for (int base = 32 * w; base < grp.n; base += 128) {
    const int n = min(32, grp.n - base);
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = p.ml[static_cast<long long>(grp.slot0 + base + lane) * p.rows + row];
    const bool valid = ml.y > 0.f;                         // empty state: identity
    float mc = valid ? ml.x : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kAll, mc, o));
    if (mc == -INFINITY) continue;
    const float m_new = fmaxf(M, mc);
    const float scale_old = M == -INFINITY ? 0.f : exp2f(M - m_new);
    const float wt = valid ? exp2f(ml.x - m_new) : 0.f;
    float lw = wt * ml.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(kAll, lw, o);
    Lsum = Lsum * scale_old + lw;
#pragma unroll
    for (int c = 0; c < C; ++c) U[c] *= scale_old;
    M = m_new;
    const unsigned live = __ballot_sync(kAll, valid);
    const float* u0 = p.u + (static_cast<long long>(grp.slot0 + base) * p.rows + row) * D + lane * C;
    const long long stride = static_cast<long long>(p.rows) * D;
    for (int s0 = 0; s0 < n; s0 += 8) {
      float v[8][C];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const bool use = s0 + q < n && ((live >> (s0 + q)) & 1u);
        if constexpr (C == 4) {
          const float4 x = use ? *reinterpret_cast<const float4*>(u0 + (s0 + q) * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y; v[q][2] = x.z; v[q][3] = x.w;
        } else {
          const float2 x = use ? *reinterpret_cast<const float2*>(u0 + (s0 + q) * stride) : make_float2(0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y;
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float wq = __shfl_sync(kAll, wt, (s0 + q) & 31);
#pragma unroll
        for (int c = 0; c < C; ++c) U[c] = fmaf(wq, v[q][c], U[c]);
      }
    }
  }
  // combine the four warps' states
#pragma unroll
  for (int c = 0; c < C; ++c) sm_u[w][lane * C + c] = U[c];
  if (lane == 0) {
    sm_ml[w][0] = M;
    sm_ml[w][1] = Lsum;
  }
  __syncthreads();
  if (w != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int k = 0; k < 4; ++k) Mt = fmaxf(Mt, sm_ml[k][1] > 0.f ? sm_ml[k][0] : -INFINITY);
  float Lt = 0.f, Ut[C];
#pragma unroll
  for (int c = 0; c < C; ++c) Ut[c] = 0.f;
  if (Mt != -INFINITY) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (!(sm_ml[k][1] > 0.f)) continue;
      const float a = exp2f(sm_ml[k][0] - Mt);
      Lt += a * sm_ml[k][1];
#pragma unroll
      for (int c = 0; c < C; ++c) Ut[c] = fmaf(a, sm_u[k][lane * C + c], Ut[c]);
    }
  }
  const int i = row / p.g, hq = grp.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(grp.b) * p.S_q + i) * p.H_q + hq;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + orow * D + lane * C;
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
#pragma unroll
  for (int c = 0; c < C; c += 2)
    *reinterpret_cast<__nv_bfloat162*>(o + c) = __floats2bfloat162_rn(Ut[c] * inv, Ut[c + 1] * inv);
  if (lane == 0 && p.lse) p.lse[orow] = Lt > 0.f ? (Mt + __log2f(Lt)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int launch_merge(const MergeParams& p, int d, void* stream) {
  const int blocks = p.n_groups * p.rows;       // one block of 4 warps per (group, row)
  if (blocks == 0) return cudaSuccess;
  if (d == 64)
    merge_kernel<64><<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
  else
    merge_kernel<128><<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError();
}

}  // namespace dattn
