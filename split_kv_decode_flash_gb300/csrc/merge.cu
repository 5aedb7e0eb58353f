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
// Groups of fewer than 8 rows (or many states): one block of four warps per
// (group, query row); warp w takes states w, w + 4, ..., and the four warps'
// folds combine in shared memory.  Groups of 8 rows or more: one warp per
// (group, row).  A warp's lanes fetch (m, l) of up to 32 states at once, the
// warp agrees on the frame, and the u vectors of the live states are then
// read a batch at a time with the loads in flight (each lane owns d / 32
// channels).  The kernel is launched as a programmatic dependent of the
// partial kernel, whose warps tag each state row with the run's number once
// it is written (release); a merge warp waits (acquire) for the tags of its
// own states only, so the groups that finish early are merged while the
// partial grid's last CTAs still run.  Each block ends with griddepcontrol.wait,
// so that the merge grid completes after the partial grid.  Without tags the
// whole grid is awaited first.
#include <cuda_runtime.h>

#include "merge.cuh"

namespace dattn {

namespace {

constexpr int kMergeWarps = 4;

__device__ __forceinline__ unsigned long long merge_clock_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Timeline trace (TAGS): the time the block's (first warp's) states were
// ready and folded.
__device__ __forceinline__ void merge_trace_ready(const MergeParams& p, int lane) {
  if (p.trace && lane == 0) atomicCAS(reinterpret_cast<unsigned long long*>(p.trace) + 2 * blockIdx.x, 0ull, merge_clock_ns());
}

// A warp's last step: its trace stamp (latest warp: done), then (TAGS, when
// some item of the plan writes O directly) the wait for the partial grid, so
// that this grid's completion implies those writes too.  When every item
// leaves partial states, the merge has read every one of them, all written and
// fenced before their tags: nothing of the partial grid remains to wait for.
template <bool TAGS>
__device__ __forceinline__ void merge_end(const MergeParams& p, int lane) {
  if (p.trace && lane == 0)
    atomicMax(reinterpret_cast<unsigned long long*>(p.trace) + 2 * blockIdx.x + 1, merge_clock_ns());
  if constexpr (TAGS) {
    if (p.end_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  }
}

// WPR = 4: one block of four warps per (group, row); warp w folds states w,
// w + 4, ... and the four folds combine in shared memory (few rows, many
// states).  WPR = 1: one warp per (group, row), four rows per block, each
// warp folding all of its row's states (many rows, few states each: the
// combine and its barrier would cost more than the fold).
// KB: u vectors read per batch.  TAGS: the warps wait for their states' tags
// instead of the whole partial grid.
template <int D, int WPR, int KB, bool TAGS>
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const __grid_constant__ MergeParams p) {
  constexpr int C = D / 32;
  constexpr int kRowsPerBlock = kMergeWarps / WPR;
  __shared__ float sm_u[WPR > 1 ? kMergeWarps : 1][D];
  __shared__ float sm_ml[WPR > 1 ? kMergeWarps : 1][2];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blocks_per_group = (p.rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int gi = blockIdx.x / blocks_per_group;
  const int row = (blockIdx.x % blocks_per_group) * kRowsPerBlock + (WPR > 1 ? 0 : w);
  // the merge groups are part of the plan, copied before the partial kernel started:
  // they may be read before the wait
  const MergeGroup grp = p.groups[gi];
  const StateTags tg{p.state_seq, p.run_seq, p.n_slots, p.wait_ns, p.status};
  if constexpr (!TAGS) asm volatile("griddepcontrol.wait;" ::: "memory");   // the partial kernel's states are complete
  // a programmatically launched successor may be scheduled; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!TAGS && p.trace && threadIdx.x == 0) p.trace[2 * blockIdx.x] = merge_clock_ns();
  const int i = row / p.g, hq = grp.h * p.g + row % p.g;
  const long long orow = (static_cast<long long>(grp.qo) + i) * p.H_q + hq;
  if constexpr (WPR == 1) {
    if (row >= p.g * grp.nq) {   // the request has fewer query rows than the widest one
      merge_end<TAGS>(p, lane);
      return;
    }
    RowFold<D> f;
    fold_init(f);
    fold_states<D, KB, TAGS>(p.ml, p.u, p.rows, row, grp.slot0, grp.n, 1, lane, f, tg);
    if (TAGS) merge_trace_ready(p, lane);
    if (!f.bad) write_folded_row<D>(p.o, p.lse, orow, f, lane);   // rows with an unwritten state stay unwritten
    merge_end<TAGS>(p, lane);
    return;
  } else {
    if (row >= p.g * grp.nq) {
      merge_end<TAGS>(p, lane);
      return;
    }
    // warp w folds states w, w + kMergeWarps, ...
    RowFold<D> f;
    fold_init(f);
    const int n_mine = grp.n > w ? (grp.n - w + kMergeWarps - 1) / kMergeWarps : 0;
    fold_states<D, KB, TAGS>(p.ml, p.u, p.rows, row, grp.slot0 + w, n_mine, kMergeWarps, lane, f, tg);
    // combine the warps' folds
#pragma unroll
    for (int c = 0; c < C; ++c) sm_u[w][lane * C + c] = f.U[c];
    if (lane == 0) {
      sm_ml[w][0] = f.M;
      sm_ml[w][1] = f.bad ? __int_as_float(0x7fc00000) : f.L;   // NaN carries the unwritten mark
    }
    __syncthreads();
    if (w != 0) {
      merge_end<TAGS>(p, lane);
      return;
    }
    if (TAGS) merge_trace_ready(p, lane);
    RowFold<D> t;
    fold_init(t);
#pragma unroll
    for (int k = 0; k < kMergeWarps; ++k) {
      t.M = fmaxf(t.M, sm_ml[k][1] > 0.f ? sm_ml[k][0] : -INFINITY);
      t.bad = t.bad || sm_ml[k][1] != sm_ml[k][1];
    }
    if (t.M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < kMergeWarps; ++k) {
        if (!(sm_ml[k][1] > 0.f)) continue;
        const float a = exp2f(sm_ml[k][0] - t.M);
        t.L += a * sm_ml[k][1];
#pragma unroll
        for (int c = 0; c < C; ++c) t.U[c] = fmaf(a, sm_u[k][lane * C + c], t.U[c]);
      }
    }
    if (!t.bad) write_folded_row<D>(p.o, p.lse, orow, t, lane);
    merge_end<TAGS>(p, lane);
  }
}

// One warp merges a row alone when the groups have at least 8 rows and at
// most 20 states on average (then the four-warp blocks, one per row, and
// their shared-memory combine cost more than they save; with more states one
// warp's sequential batches lengthen the merge's critical path).  A row's
// whole fold in one round (every state's u read at once) was slower: the
// unrolled batch of 32 predicated loads costs more than the round trips it
// saves.
constexpr int kOneWarpRows = 8, kOneWarpStates = 20;

template <int D, int WPR, int KB>
cudaError_t launch_d(const MergeParams& p, void* stream) {
  constexpr int kRowsPerBlock = kMergeWarps / WPR;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_groups * ((p.rows + kRowsPerBlock - 1) / kRowsPerBlock));
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.state_seq ? cudaLaunchKernelEx(&cfg, merge_kernel<D, WPR, KB, true>, p)
                     : cudaLaunchKernelEx(&cfg, merge_kernel<D, WPR, KB, false>, p);
}

}  // namespace

int launch_merge(const MergeParams& p, int d, void* stream) {
  if (p.n_groups * p.rows == 0) return cudaSuccess;
  cudaError_t err;
  if (p.rows >= kOneWarpRows && p.mean_states <= kOneWarpStates)
    err = d == 64 ? launch_d<64, 1, 8>(p, stream) : launch_d<128, 1, 8>(p, stream);
  else
    err = d == 64 ? launch_d<64, 4, 8>(p, stream) : launch_d<128, 4, 8>(p, stream);
  return err != cudaSuccess ? err : cudaGetLastError();
}

}  // namespace dattn
