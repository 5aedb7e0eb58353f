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
  const int warp_global = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp_global >= p.n_groups * p.rows) return;
  const int gi = warp_global / p.rows, row = warp_global % p.rows;
  const MergeGroup grp = p.groups[gi];

  float M = -INFINITY, Lsum = 0.f, U[C];
#pragma unroll
  for (int c = 0; c < C; ++c) U[c] = 0.f;
  // 32 slots at a time: every lane fetches one state's (m, l), the warp agrees on
  // the frame, then the u vectors are read back to back with the weights broadcast.
  for (int base = 0; base < grp.n; base += 32) {
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
    const float w = valid ? exp2f(ml.x - m_new) : 0.f;
    float lw = w * ml.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(kAll, lw, o);
    Lsum = Lsum * scale_old + lw;
#pragma unroll
    for (int c = 0; c < C; ++c) U[c] *= scale_old;
    M = m_new;
    const float* u0 = p.u + (static_cast<long long>(grp.slot0 + base) * p.rows + row) * D + lane * C;
    const long long stride = static_cast<long long>(p.rows) * D;
    int s = 0;
    for (; s + 4 <= n; s += 4) {
      float v[4][C];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (C == 4) {
          const float4 x = *reinterpret_cast<const float4*>(u0 + (s + q) * stride);
          v[q][0] = x.x; v[q][1] = x.y; v[q][2] = x.z; v[q][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(u0 + (s + q) * stride);
          v[q][0] = x.x; v[q][1] = x.y;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float wq = __shfl_sync(kAll, w, s + q);
#pragma unroll
        for (int c = 0; c < C; ++c) U[c] = fmaf(wq, v[q][c], U[c]);
      }
    }
    for (; s < n; ++s) {
      const float wq = __shfl_sync(kAll, w, s);
      if constexpr (C == 4) {
        const float4 x = *reinterpret_cast<const float4*>(u0 + s * stride);
        U[0] = fmaf(wq, x.x, U[0]); U[1] = fmaf(wq, x.y, U[1]);
        U[2] = fmaf(wq, x.z, U[2]); U[3] = fmaf(wq, x.w, U[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(u0 + s * stride);
        U[0] = fmaf(wq, x.x, U[0]); U[1] = fmaf(wq, x.y, U[1]);
      }
    }
  }
  const int i = row / p.g, hq = grp.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(grp.b) * p.S_q + i) * p.H_q + hq;
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.o) + orow * D + lane * C;
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
  for (int c = 0; c < C; c += 2)
    *reinterpret_cast<__nv_bfloat162*>(o + c) = __floats2bfloat162_rn(U[c] * inv, U[c + 1] * inv);
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
