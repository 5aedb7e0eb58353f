// LSE-merge kernel: folds the partial (m, l, u) states of every (request, kv
// head) group that the planner cut into several chunks.
//
// "M4.5 Decode Attention Kernels, Mask Programs, and Backend Boundaries":
// §0x02B binary merge through the common frame m = max(m_A, m_B), applied as
// a fold over the group's states; §0x02C validity branch before any
// exponential (a state is empty iff l = 0, stored with m = -inf); O = u / l
// rounded to bf16 and LSE = m + ln l, all-masked rows giving O = 0 and
// LSE = -inf.
//
// One block of four warps per (group, query row).  Warp w takes states
// w, w + 4, ...: its lanes fetch (m, l) of up to 32 states at once, the warp
// agrees on the frame, and the u vectors of all of them are then read with
// every load in flight (each lane owns d / 32 channels).  The four warps'
// folds combine in shared memory.  The kernel is launched as a programmatic
// dependent of the partial kernel: it is resident before the partial kernel
// ends and waits (griddepcontrol.wait) for its states to be complete.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace dattn {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kMergeWarps = 4;
constexpr int kBatch = 16;     // u loads in flight per lane

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int C = D / 32;
  __shared__ float sm_u[kMergeWarps][D];
  __shared__ float sm_ml[kMergeWarps][2];
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the partial kernel's states are complete
  // a programmatically launched successor may be scheduled; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = blockIdx.x / p.rows, row = blockIdx.x % p.rows;
  const MergeGroup grp = p.groups[gi];
  const long long stride = static_cast<long long>(kMergeWarps) * p.rows * D;   // between a warp's states

  float M = -INFINITY, Lsum = 0.f, U[C];
#pragma unroll
  for (int c = 0; c < C; ++c) U[c] = 0.f;
  // this warp's states: w + kMergeWarps * i, i = 0, 1, ...; 32 at a time
  const int n_mine = grp.n > w ? (grp.n - w + kMergeWarps - 1) / kMergeWarps : 0;
  for (int i0 = 0; i0 < n_mine; i0 += 32) {
    const int n = min(32, n_mine - i0);
    const int s_first = grp.slot0 + w + kMergeWarps * i0;
    float2 ml = make_float2(-INFINITY, 0.f);
    if (lane < n) ml = __ldcg(p.ml + static_cast<long long>(s_first + kMergeWarps * lane) * p.rows + row);
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
    const float* u0 = p.u + (static_cast<long long>(s_first) * p.rows + row) * D + lane * C;
    for (int q0 = 0; q0 < n; q0 += kBatch) {
      float v[kBatch][C];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const bool use = q0 + q < n && ((live >> (q0 + q)) & 1u);
        const float* src = u0 + (q0 + q) * stride;
        if constexpr (C == 4) {
          const float4 x = use ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y; v[q][2] = x.z; v[q][3] = x.w;
        } else {
          const float2 x = use ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y;
        }
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const float wq = __shfl_sync(kAll, wt, (q0 + q) & 31);
#pragma unroll
        for (int c = 0; c < C; ++c) U[c] = fmaf(wq, v[q][c], U[c]);
      }
    }
  }
  // combine the warps' folds
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
  for (int k = 0; k < kMergeWarps; ++k) Mt = fmaxf(Mt, sm_ml[k][1] > 0.f ? sm_ml[k][0] : -INFINITY);
  float Lt = 0.f, Ut[C];
#pragma unroll
  for (int c = 0; c < C; ++c) Ut[c] = 0.f;
  if (Mt != -INFINITY) {
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) {
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

template <int D>
cudaError_t launch_d(const MergeParams& p, int blocks, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D>, p);
}

}  // namespace

int launch_merge(const MergeParams& p, int d, void* stream) {
  const int blocks = p.n_groups * p.rows;       // one block per (group, row)
  if (blocks == 0) return cudaSuccess;
  const cudaError_t err = d == 64 ? launch_d<64>(p, blocks, stream) : launch_d<128>(p, blocks, stream);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace dattn
