// kv_append: writes new K/V rows into the cache, codes and qparams together.
//
// "M8.6 Live-Data Quantization: Activations and KV Cache":
//  - §0x02A stored-scale conventions: fp32 range, fp16 stored scale and
//    offset, encoding with the re-read stored values, ties to even, a
//    sentinel scale of one when the range is zero and no subnormal scale;
//  - §0x05B per-token scales are append-local (INT8: one (s, z) per token and
//    kv head, written in the same call as the codes);
//  - §0x06A-B KIVI: K per channel over closed groups of G tokens, V per token
//    per Gv channels; rows stay bf16 in a residual ring until their group
//    closes (the oldest G rows close while the residual holds more than R).
//  - §0x09C the zero point is a floating value offset stored as fp16
//    (x_hat = code * s + z), not an integer clamped to the code range; the
//    per-head asymmetric INT4 format stores one (s, o) per token and kv head
//    and encodes rint(x / s + o) with x_hat = (code - o) * s.
// All arguments, and the page capacity of every request, are validated on the
// host before any launch (the append transaction of M4.5 §0x08C).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>
#include <vector>

#include "device.cuh"
#include "plan.h"

namespace dattn {

namespace {

constexpr unsigned kAll = 0xffffffffu;

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  void* k;
  void* v;
  void* kqp;
  void* vqp;
  __nv_bfloat16* kres;
  __nv_bfloat16* vres;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  const int32_t* cache_batch_idx;
  const int32_t* new_indptr;   // [B+1] rows of k_new per request
  const int32_t* t_old;        // [B]
  const int32_t* work_indptr;  // [B+1] per-request work units (rows, or closing groups)
  const int32_t* res_indptr;   // [B+1] KIVI residual rows written by this call
  int32_t* status;
  int B, H, P, num_pages, T_cap, B_cache, layout, G, Gv, R;
};

__device__ __forceinline__ int find_request(const int32_t* indptr, int B, int unit) {
  int lo = 0, hi = B;  // largest b with indptr[b] <= unit
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (indptr[mid] <= unit) lo = mid; else hi = mid;
  }
  return lo;
}

// Stored (s, z) of a group with range [mn, mx] and qmax levels.
__device__ __forceinline__ void qparams(float mn, float mx, float qmax, __half& s, __half& z) {
  if (mx == mn) {
    s = __float2half_rn(1.f);
  } else {
    s = __float2half_rn(__fdiv_rn(mx - mn, qmax));
    if (__half2float(s) < 6.103515625e-05f) s = __float2half_rn(6.103515625e-05f);
  }
  z = __float2half_rn(mn);
}

__device__ __forceinline__ uint32_t encode(float x, float s, float z, float qmax) {
  const float r = rintf(__fdiv_rn(x - z, s));
  return static_cast<uint32_t>(fminf(fmaxf(r, 0.f), qmax));
}

// Per-head asymmetric INT4 (§0x09C): s = fp16((mx - mn) / 15), floating offset
// o = fp16(-mn / ((mx - mn) / 15)), both saturated to the finite fp16 range; a
// constant head stores s = 1, o = fp16(-mn); a scale below 2^-14 is raised to
// 2^-14 and the offset taken with it.
__device__ __forceinline__ __half f16_sat(float x) { return __float2half_rn(fminf(fmaxf(x, -65504.f), 65504.f)); }

__device__ __forceinline__ void head_qparams(float mn, float mx, __half& s, __half& o) {
  const float width = mx - mn;
  float base = width == 0.f ? 1.f : __fdiv_rn(width, 15.f);
  s = f16_sat(base);
  if (width != 0.f && __half2float(s) < 6.103515625e-05f) {
    s = __float2half_rn(6.103515625e-05f);
    base = 6.103515625e-05f;
  }
  o = f16_sat(__fdiv_rn(-mn, base));
}

// code = clip(rint(x / s + o), 0, 15): the offset is added before rounding.
__device__ __forceinline__ uint32_t encode_offset(float x, float s, float o) {
  const float r = rintf(__fadd_rn(__fdiv_rn(x, s), o));
  return static_cast<uint32_t>(fminf(fmaxf(r, 0.f), 15.f));
}

__device__ __forceinline__ float warp_min(float x, int width) {
  for (int o = width / 2; o > 0; o >>= 1) x = fminf(x, __shfl_xor_sync(kAll, x, o));
  return x;
}
__device__ __forceinline__ float warp_max(float x, int width) {
  for (int o = width / 2; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kAll, x, o));
  return x;
}

// Loads C consecutive bf16 channels of a row as floats.
template <int C>
__device__ __forceinline__ void load_channels(const __nv_bfloat16* row, int lane, float* x) {
  if constexpr (C == 4) {
    const uint2 w = reinterpret_cast<const uint2*>(row)[lane];
    float2 a = bf16x2_to_float2(w.x), b = bf16x2_to_float2(w.y);
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    const uint32_t w = reinterpret_cast<const uint32_t*>(row)[lane];
    float2 a = bf16x2_to_float2(w);
    x[0] = a.x; x[1] = a.y;
  }
}

// One warp per (new row, kv head): bf16 copy, INT8 per-token quantisation, or
// FP8 E4M3 / E5M2 codes of x / s_h (correctly rounded fp32 quotient, then the
// hardware's round-to-nearest-even conversion with saturation to the largest
// finite value).
template <int D, int FMT>
__global__ void append_rows_kernel(AppendParams p, int total_rows) {
  constexpr int C = D / 32;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total_rows * p.H) return;
  const int row = w / p.H, h = w % p.H;
  const int b = find_request(p.new_indptr, p.B, row);
  const int t = p.t_old[b] + (row - p.new_indptr[b]);
  long long dst_row;  // element offset of (row t, head h, channel 0)
  if (p.layout == DATTN_KV_PAGED_HND) {
    const int pi = page_of(p.page_indptr, p.page_indices, b, t / p.P, p.num_pages, lane == 0 ? p.status : nullptr);
    if (pi < 0) return;
    dst_row = paged_hnd_offset(pi, t % p.P, h, 0, p.P, p.H, D);
  } else {
    const int c = cache_row(p.cache_batch_idx, b, p.B_cache, lane == 0 ? p.status : nullptr);
    if (c < 0 || t >= p.T_cap) return;
    dst_row = contig_nhd_offset(c, t, h, 0, p.T_cap, p.H, D);
  }
  const long long src = (static_cast<long long>(row) * p.H + h) * D;
#pragma unroll
  for (int kv = 0; kv < 2; ++kv) {
    const __nv_bfloat16* in = (kv ? p.v_new : p.k_new) + src;
    if constexpr (FMT == DATTN_FMT_BF16) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(kv ? p.v : p.k) + dst_row;
      if constexpr (C == 4) reinterpret_cast<uint2*>(out)[lane] = reinterpret_cast<const uint2*>(in)[lane];
      else reinterpret_cast<uint32_t*>(out)[lane] = reinterpret_cast<const uint32_t*>(in)[lane];
    } else if constexpr (FMT == DATTN_FMT_FP8_E4M3 || FMT == DATTN_FMT_FP8_E5M2) {
      float x[C];
      load_channels<C>(in, lane, x);
      const float* scales = static_cast<const float*>(kv ? p.vqp : p.kqp);
      const float sh = scales ? scales[h] : 1.f;
      uint32_t packed = 0;
#pragma unroll
      for (int c = 0; c < C; c += 2) {
        const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(
            make_float2(__fdiv_rn(x[c], sh), __fdiv_rn(x[c + 1], sh)), __NV_SATFINITE,
            FMT == DATTN_FMT_FP8_E4M3 ? __NV_E4M3 : __NV_E5M2);
        packed |= static_cast<uint32_t>(two) << (8 * c);
      }
      uint8_t* codes = static_cast<uint8_t*>(kv ? p.v : p.k) + dst_row;
      if constexpr (C == 4) reinterpret_cast<uint32_t*>(codes)[lane] = packed;
      else reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
    } else if constexpr (FMT == DATTN_FMT_INT4_HEAD) {
      float x[C];
      load_channels<C>(in, lane, x);
      float mn = x[0], mx = x[0];
#pragma unroll
      for (int c = 1; c < C; ++c) { mn = fminf(mn, x[c]); mx = fmaxf(mx, x[c]); }
      mn = warp_min(mn, 32);
      mx = warp_max(mx, 32);
      __half s, o;
      head_qparams(mn, mx, s, o);
      const float sf = __half2float(s), of = __half2float(o);
      uint32_t packed = 0;
#pragma unroll
      for (int c = 0; c < C; ++c) packed |= encode_offset(x[c], sf, of) << (4 * c);
      uint8_t* codes = static_cast<uint8_t*>(kv ? p.v : p.k) + dst_row / 2;
      if constexpr (C == 4) reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
      else codes[lane] = static_cast<uint8_t>(packed);
      if (lane == 0) {
        __half2* qp = static_cast<__half2*>(kv ? p.vqp : p.kqp);
        qp[dst_row / D] = __halves2half2(s, o);   // [page][h][row] matches the code row
      }
    } else {
      float x[C];
      load_channels<C>(in, lane, x);
      float mn = x[0], mx = x[0];
#pragma unroll
      for (int c = 1; c < C; ++c) { mn = fminf(mn, x[c]); mx = fmaxf(mx, x[c]); }
      mn = warp_min(mn, 32);
      mx = warp_max(mx, 32);
      __half s, z;
      qparams(mn, mx, 255.f, s, z);
      const float sf = __half2float(s), zf = __half2float(z);
      uint32_t packed = 0;
#pragma unroll
      for (int c = 0; c < C; ++c) packed |= encode(x[c], sf, zf, 255.f) << (8 * c);
      uint8_t* codes = static_cast<uint8_t*>(kv ? p.v : p.k) + dst_row;
      if constexpr (C == 4) reinterpret_cast<uint32_t*>(codes)[lane] = packed;
      else reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
      if (lane == 0) {
        __half2* qp = static_cast<__half2*>(kv ? p.vqp : p.kqp);
        qp[dst_row / D] = __halves2half2(s, z);   // [page][h][row] matches the code row
      }
    }
  }
}

// KIVI: one warp per (request, closing group, kv head).
template <int D>
__global__ void kivi_close_kernel(AppendParams p, int total_groups) {
  constexpr int C = D / 32;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total_groups * p.H) return;
  const int unit = w / p.H, h = w % p.H;
  const int b = find_request(p.work_indptr, p.B, unit);
  const int T_old = p.t_old[b];
  const int nq_old = T_old > p.R ? (T_old - p.R + p.G - 1) / p.G * p.G : 0;
  const int t0 = nq_old + (unit - p.work_indptr[b]) * p.G;

  auto src_row = [&](int t, int kv) -> const __nv_bfloat16* {
    if (t < T_old) {
      const __nv_bfloat16* ring = kv ? p.vres : p.kres;
      return ring + ((static_cast<long long>(b) * p.R + t % p.R) * p.H + h) * D;
    }
    const int row = p.new_indptr[b] + (t - T_old);
    return (kv ? p.v_new : p.k_new) + (static_cast<long long>(row) * p.H + h) * D;
  };

  // K: per-channel range over the G tokens
  float mn[C], mx[C];
#pragma unroll
  for (int c = 0; c < C; ++c) { mn[c] = INFINITY; mx[c] = -INFINITY; }
  for (int t = t0; t < t0 + p.G; ++t) {
    float x[C];
    load_channels<C>(src_row(t, 0), lane, x);
#pragma unroll
    for (int c = 0; c < C; ++c) { mn[c] = fminf(mn[c], x[c]); mx[c] = fmaxf(mx[c], x[c]); }
  }
  __half s[C], z[C];
  float sf[C], zf[C];
#pragma unroll
  for (int c = 0; c < C; ++c) {
    qparams(mn[c], mx[c], 15.f, s[c], z[c]);
    sf[c] = __half2float(s[c]);
    zf[c] = __half2float(z[c]);
  }
  const int qpage = page_of(p.page_indptr, p.page_indices, b, t0 / p.P, p.num_pages, lane == 0 ? p.status : nullptr);
  if (qpage < 0) return;
  const int qslot = p.P >= p.G ? (t0 % p.P) / p.G : 0;
  const int slots = p.P >= p.G ? p.P / p.G : 1;
  __half2* kq = static_cast<__half2*>(p.kqp) + ((static_cast<long long>(qpage) * p.H + h) * slots + qslot) * D;
#pragma unroll
  for (int c = 0; c < C; ++c) kq[lane * C + c] = __halves2half2(s[c], z[c]);

  const int lanes_per_vgroup = p.Gv / C;
  for (int t = t0; t < t0 + p.G; ++t) {
    const int pi = page_of(p.page_indptr, p.page_indices, b, t / p.P, p.num_pages, lane == 0 ? p.status : nullptr);
    if (pi < 0) continue;
    const long long code_row = (static_cast<long long>(pi) * p.H + h) * p.P + t % p.P;  // row index
    // K codes of this token
    {
      float x[C];
      load_channels<C>(src_row(t, 0), lane, x);
      uint32_t packed = 0;
#pragma unroll
      for (int c = 0; c < C; ++c) packed |= encode(x[c], sf[c], zf[c], 15.f) << (4 * c);
      uint8_t* codes = static_cast<uint8_t*>(p.k) + code_row * (D / 2);
      if constexpr (C == 4) reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
      else codes[lane] = static_cast<uint8_t>(packed);
    }
    // V: per token, per Gv channels
    {
      float x[C];
      load_channels<C>(src_row(t, 1), lane, x);
      float vmn = x[0], vmx = x[0];
#pragma unroll
      for (int c = 1; c < C; ++c) { vmn = fminf(vmn, x[c]); vmx = fmaxf(vmx, x[c]); }
      vmn = warp_min(vmn, lanes_per_vgroup);
      vmx = warp_max(vmx, lanes_per_vgroup);
      __half vs, vz;
      qparams(vmn, vmx, 15.f, vs, vz);
      const float vsf = __half2float(vs), vzf = __half2float(vz);
      uint32_t packed = 0;
#pragma unroll
      for (int c = 0; c < C; ++c) packed |= encode(x[c], vsf, vzf, 15.f) << (4 * c);
      uint8_t* codes = static_cast<uint8_t*>(p.v) + code_row * (D / 2);
      if constexpr (C == 4) reinterpret_cast<uint16_t*>(codes)[lane] = static_cast<uint16_t>(packed);
      else codes[lane] = static_cast<uint8_t>(packed);
      if (lane % lanes_per_vgroup == 0) {
        __half2* vq = static_cast<__half2*>(p.vqp) + code_row * (D / p.Gv);
        vq[lane / lanes_per_vgroup] = __halves2half2(vs, vz);
      }
    }
  }
}

// KIVI: one warp per (request, residual row written by this call, kv head).
template <int D>
__global__ void kivi_residual_kernel(AppendParams p, int total_rows) {
  constexpr int C = D / 32;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total_rows * p.H) return;
  const int unit = w / p.H, h = w % p.H;
  const int b = find_request(p.res_indptr, p.B, unit);
  const int T_old = p.t_old[b];
  const int T_new = T_old + (p.new_indptr[b + 1] - p.new_indptr[b]);
  const int nq_new = T_new > p.R ? (T_new - p.R + p.G - 1) / p.G * p.G : 0;
  const int t = max(T_old, nq_new) + (unit - p.res_indptr[b]);
  const int row = p.new_indptr[b] + (t - T_old);
  const long long src = (static_cast<long long>(row) * p.H + h) * D;
  const long long dst = ((static_cast<long long>(b) * p.R + t % p.R) * p.H + h) * D;
  if constexpr (C == 4) {
    reinterpret_cast<uint2*>(p.kres + dst)[lane] = reinterpret_cast<const uint2*>(p.k_new + src)[lane];
    reinterpret_cast<uint2*>(p.vres + dst)[lane] = reinterpret_cast<const uint2*>(p.v_new + src)[lane];
  } else {
    reinterpret_cast<uint32_t*>(p.kres + dst)[lane] = reinterpret_cast<const uint32_t*>(p.k_new + src)[lane];
    reinterpret_cast<uint32_t*>(p.vres + dst)[lane] = reinterpret_cast<const uint32_t*>(p.v_new + src)[lane];
  }
}

int kivi_prefix(int T, int G, int R) { return T > R ? (T - R + G - 1) / G * G : 0; }

template <typename K, typename... A>
cudaError_t launch_warps(K kernel, long long warps, cudaStream_t s, A... args) {
  if (warps <= 0) return cudaSuccess;
  const long long blocks = (warps + 7) / 8;
  kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(args...);
  return cudaGetLastError();
}

}  // namespace
}  // namespace dattn

using namespace dattn;

extern "C" size_t kv_append_workspace_bytes(const dattn_problem* prob) {
  if (!prob || prob->B < 1) return 0;
  return (static_cast<size_t>(4) * (prob->B + 1) * sizeof(int32_t) + 256 + kWsAlign - 1) / kWsAlign * kWsAlign;
}

extern "C" dattn_status kv_append(const dattn_problem* prob, const dattn_append_inputs* in,
                                  const dattn_tensors* cache, const void* k_new, const void* v_new, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  Checker c;
  check_problem(prob, c);
  if (!in || !in->kv_len_old || !in->new_indptr) c.fail(DATTN_EINVAL, "kv_len_old and new_indptr are required");
  if (!cache || !cache->k || !cache->v) c.fail(DATTN_EINVAL, "cache k and v are required");
  if (prob->layout == DATTN_KV_PACKED_ROWS)
    c.fail(DATTN_EUNSUPPORTED, "kv_append writes paged or contiguous caches, not a packed view");
  if (c.status != DATTN_OK) return c.finish("kv_append");
  const dattn_problem& p = *prob;
  const bool paged = p.layout == DATTN_KV_PAGED_HND;
  if (paged && (!in->page_indptr || !cache->page_indptr || !cache->page_indices))
    c.fail(DATTN_EINVAL, "paged cache needs host and device page_indptr and device page_indices");
  if ((p.fmt == DATTN_FMT_INT8_TOKEN || p.fmt == DATTN_FMT_INT4_KIVI || p.fmt == DATTN_FMT_INT4_HEAD) &&
      (!cache->k_qparams || !cache->v_qparams))
    c.fail(DATTN_EINVAL, "INT8 and INT4 formats need k_qparams and v_qparams");
  if (p.fmt == DATTN_FMT_INT4_KIVI && (!cache->k_residual || !cache->v_residual))
    c.fail(DATTN_EINVAL, "INT4 KIVI needs k_residual and v_residual");
  const size_t need = kv_append_workspace_bytes(prob);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign) || workspace_bytes < need)
    c.fail(DATTN_EWORKSPACE, "workspace must be 256-byte aligned and hold " + std::to_string(need) + " bytes");
  if (c.status != DATTN_OK) return c.finish("kv_append");

  const int B = p.B;
  std::vector<int32_t> host(4 * (B + 1), 0);
  int32_t* new_indptr = host.data();
  int32_t* t_old = host.data() + (B + 1);
  int32_t* work_indptr = host.data() + 2 * (B + 1);
  int32_t* res_indptr = host.data() + 3 * (B + 1);
  if (in->new_indptr[0] != 0) c.fail(DATTN_EINVAL, "new_indptr[0] must be 0");
  for (int b = 0; b < B; ++b) {
    const int T = in->kv_len_old[b], n = in->new_indptr[b + 1] - in->new_indptr[b];
    if (T < 0 || n < 0) {
      c.fail(DATTN_EINVAL, "request " + std::to_string(b) + ": negative length or non-monotone new_indptr");
      continue;
    }
    const long long T_new = static_cast<long long>(T) + n;
    if (paged) {
      const long long cap = static_cast<long long>(in->page_indptr[b + 1] - in->page_indptr[b]) * p.page_size;
      if (T_new > cap)
        c.fail(DATTN_EINVAL, "request " + std::to_string(b) + ": page list holds " + std::to_string(cap) +
                                 " rows, append needs " + std::to_string(T_new));
    } else if (T_new > p.T_cap) {
      c.fail(DATTN_EINVAL, "request " + std::to_string(b) + ": append exceeds T_cap");
    }
    new_indptr[b + 1] = in->new_indptr[b + 1];
    t_old[b] = T;
    if (p.fmt == DATTN_FMT_INT4_KIVI) {
      const int nq_old = kivi_prefix(T, p.kivi_group, p.kivi_residual);
      const int nq_new = kivi_prefix(static_cast<int>(T_new), p.kivi_group, p.kivi_residual);
      work_indptr[b + 1] = work_indptr[b] + (nq_new - nq_old) / p.kivi_group;
      res_indptr[b + 1] = res_indptr[b] + static_cast<int>(T_new - std::max<long long>(T, nq_new));
    } else {
      work_indptr[b + 1] = work_indptr[b] + n;
    }
  }
  if (c.status != DATTN_OK) return c.finish("kv_append");
  if (new_indptr[B] > 0 && (!k_new || !v_new)) {
    c.fail(DATTN_EINVAL, "k_new and v_new are required");
    return c.finish("kv_append");
  }

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t err = cudaMemcpyAsync(ws + 256, host.data(), host.size() * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(ws, 0, 256, s);
  if (err != cudaSuccess) {
    set_error(std::string("kv_append: CUDA error ") + cudaGetErrorString(err));
    return DATTN_ECUDA;
  }
  AppendParams a{};
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.k = const_cast<void*>(cache->k);
  a.v = const_cast<void*>(cache->v);
  a.kqp = const_cast<void*>(cache->k_qparams);
  a.vqp = const_cast<void*>(cache->v_qparams);
  a.kres = static_cast<__nv_bfloat16*>(const_cast<void*>(cache->k_residual));
  a.vres = static_cast<__nv_bfloat16*>(const_cast<void*>(cache->v_residual));
  a.page_indptr = cache->page_indptr;
  a.page_indices = cache->page_indices;
  a.cache_batch_idx = cache->cache_batch_idx;
  const int32_t* dev = reinterpret_cast<const int32_t*>(ws + 256);
  a.new_indptr = dev;
  a.t_old = dev + (B + 1);
  a.work_indptr = dev + 2 * (B + 1);
  a.res_indptr = dev + 3 * (B + 1);
  a.status = reinterpret_cast<int32_t*>(ws);
  a.B = B;
  a.H = p.H_kv;
  a.P = p.page_size;
  a.num_pages = p.num_pages;
  a.T_cap = p.T_cap;
  a.B_cache = p.B_cache;
  a.layout = p.layout;
  a.G = p.kivi_group;
  a.Gv = p.kivi_v_group;
  a.R = p.kivi_residual;
  const long long H = p.H_kv;
  const bool d128 = p.d_h == 128;
  if (p.fmt == DATTN_FMT_BF16) {
    err = d128 ? launch_warps(append_rows_kernel<128, DATTN_FMT_BF16>, new_indptr[B] * H, s, a, new_indptr[B])
               : launch_warps(append_rows_kernel<64, DATTN_FMT_BF16>, new_indptr[B] * H, s, a, new_indptr[B]);
  } else if (p.fmt == DATTN_FMT_INT8_TOKEN) {
    err = d128 ? launch_warps(append_rows_kernel<128, DATTN_FMT_INT8_TOKEN>, new_indptr[B] * H, s, a, new_indptr[B])
               : launch_warps(append_rows_kernel<64, DATTN_FMT_INT8_TOKEN>, new_indptr[B] * H, s, a, new_indptr[B]);
  } else if (p.fmt == DATTN_FMT_INT4_HEAD) {
    err = d128 ? launch_warps(append_rows_kernel<128, DATTN_FMT_INT4_HEAD>, new_indptr[B] * H, s, a, new_indptr[B])
               : launch_warps(append_rows_kernel<64, DATTN_FMT_INT4_HEAD>, new_indptr[B] * H, s, a, new_indptr[B]);
  } else if (p.fmt == DATTN_FMT_FP8_E4M3) {
    err = d128 ? launch_warps(append_rows_kernel<128, DATTN_FMT_FP8_E4M3>, new_indptr[B] * H, s, a, new_indptr[B])
               : launch_warps(append_rows_kernel<64, DATTN_FMT_FP8_E4M3>, new_indptr[B] * H, s, a, new_indptr[B]);
  } else if (p.fmt == DATTN_FMT_FP8_E5M2) {
    err = d128 ? launch_warps(append_rows_kernel<128, DATTN_FMT_FP8_E5M2>, new_indptr[B] * H, s, a, new_indptr[B])
               : launch_warps(append_rows_kernel<64, DATTN_FMT_FP8_E5M2>, new_indptr[B] * H, s, a, new_indptr[B]);
  } else {
    const int groups = work_indptr[B], rows = res_indptr[B];
    err = d128 ? launch_warps(kivi_close_kernel<128>, groups * H, s, a, groups)
               : launch_warps(kivi_close_kernel<64>, groups * H, s, a, groups);
    if (err == cudaSuccess)
      err = d128 ? launch_warps(kivi_residual_kernel<128>, rows * H, s, a, rows)
                 : launch_warps(kivi_residual_kernel<64>, rows * H, s, a, rows);
  }
  if (err != cudaSuccess) {
    set_error(std::string("kv_append: CUDA error ") + cudaGetErrorString(err));
    return DATTN_ECUDA;
  }
  return DATTN_OK;
}
