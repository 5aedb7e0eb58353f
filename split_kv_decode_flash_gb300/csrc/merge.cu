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
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.n_groups * p.rows) return;
  const int gi = warp_global / p.rows, row = warp_global % p.rows;
  const MergeGroup grp = p.groups[gi];

  float M = -INFINITY, Lsum = 0.f, U[C];
#pragma unroll
  for (int c = 0; c < C; ++c) U[c] = 0.f;
  for (int s = 0; s < grp.n; ++s) {
    const long long srow = static_cast<long long>(grp.slot0 + s) * p.rows + row;
    const float2 ml = p.ml[srow];
    if (!(ml.y > 0.f)) continue;                      // empty state: identity
    const float m_new = fmaxf(M, ml.x);
    const float a = exp2f(M - m_new);                 // M = -inf -> 0 (U, Lsum are 0)
    const float b = exp2f(ml.x - m_new);
    const float* us = p.u + srow * D;
    Lsum = a * Lsum + b * ml.y;
    if constexpr (C == 4) {
      const float4 v = reinterpret_cast<const float4*>(us)[lane];
      U[0] = a * U[0] + b * v.x;
      U[1] = a * U[1] + b * v.y;
      U[2] = a * U[2] + b * v.z;
      U[3] = a * U[3] + b * v.w;
    } else {
      const float2 v = reinterpret_cast<const float2*>(us)[lane];
      U[0] = a * U[0] + b * v.x;
      U[1] = a * U[1] + b * v.y;
    }
    M = m_new;
  }
  const int i = row / p.g, hq = grp.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(grp.b) * p.S_q + i) * p.H_q + hq;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + orow * D + lane * C;
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
  for (int c = 0; c < C; c += 2) {
    const float x0 = Lsum > 0.f ? U[c] * inv : 0.f;
    const float x1 = Lsum > 0.f ? U[c + 1] * inv : 0.f;
    *reinterpret_cast<__nv_bfloat162*>(o + c) = __floats2bfloat162_rn(x0, x1);
  }
  if (lane == 0 && p.lse) p.lse[orow] = Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int launch_merge(const MergeParams& p, int d, void* stream) {
  const int warps = p.n_groups * p.rows;
  if (warps == 0) return cudaSuccess;
  const int blocks = (warps + 3) / 4;
  if (d == 64)
    merge_kernel<64><<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
  else
    merge_kernel<128><<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError();
}

}  // namespace dattn
