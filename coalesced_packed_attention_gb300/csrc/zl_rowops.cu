// Row-parallel, HBM-bound kernels of the engine: the LSE-weighted merge of k-split
// partials, the backward row sums D = rowsum(dO * O) (plus zeroing of the dQ
// accumulator), and the dQ finalisation.  One warp per (row, head); each lane owns
// d/32 consecutive elements, so a warp moves whole 256/512-byte rows per access and
// consecutive warps walk consecutive rows of a [rows, heads, d] block.  The dQ
// accumulator is tiled by query block (acc_index); the finalisation walks it row by
// row within a head, so neighbouring warps read neighbouring 16-byte pieces.
//
// The merge is the combine that a k split of theta=(q,h,k) implies ("Zellige",
// pith.science review, "What carries the argument"; ring attention [19] combines
// per-chunk partials the same way): with M = max_c LSE_c,
//   LSE = M + ln sum_c exp(LSE_c - M),   O = sum_c exp(LSE_c - LSE) O_c.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zl_internal.h"
#include "zl_kernels.h"
#include "zl_ptx.cuh"

namespace zl {

namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2f = 0.69314718055994530942f;
constexpr float kNegInfF = -__builtin_huge_valf();

template <typename T>
__device__ __forceinline__ int find_segment(const T* segs, int n, int64_t idx) {
  int lo = 0, hi = n - 1;  // last segment with rowhead_begin <= idx
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].rowhead_begin <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D>
struct Vec;  // d/32 fp32 values per lane
template <>
struct Vec<128> {
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  }
  __device__ __forceinline__ void store(float* p) const {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ __forceinline__ void load_bf16(const __nv_bfloat16* p) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&x.y);
    v[0] = __low2float(a); v[1] = __high2float(a); v[2] = __low2float(b); v[3] = __high2float(b);
  }
  __device__ __forceinline__ void store_bf16(__nv_bfloat16* p) const {
    uint2 x;
    x.x = pack_bf16(v[0], v[1]);
    x.y = pack_bf16(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = x;
  }
};
template <>
struct Vec<64> {
  float v[2];
  __device__ __forceinline__ void load(const float* p) {
    const float2 x = __ldg(reinterpret_cast<const float2*>(p));
    v[0] = x.x; v[1] = x.y;
  }
  __device__ __forceinline__ void store(float* p) const {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
  __device__ __forceinline__ void load_bf16(const __nv_bfloat16* p) {
    const uint32_t x = __ldg(reinterpret_cast<const unsigned int*>(p));
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&x);
    v[0] = __low2float(a); v[1] = __high2float(a);
  }
  __device__ __forceinline__ void store_bf16(__nv_bfloat16* p) const {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16(v[0], v[1]);
  }
};

template <int D>
__global__ void __launch_bounds__(256) zl_merge_kernel(const DevGroup* __restrict__ groups, int32_t n_groups,
                                                       const DevMember* __restrict__ members, int64_t total,
                                                       const float* __restrict__ o_partial,
                                                       const float* __restrict__ lse_partial,
                                                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse_out) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += nwarps) {
    const DevGroup G = groups[find_segment(groups, n_groups, w)];
    const int64_t local = w - G.rowhead_begin;
    const int64_t row = local / G.nh;
    const int hl = (int)(local - row * G.nh);
    const int64_t vec_off = (row * G.nh + hl) * D + lane * E;
    const int64_t lse_idx = (int64_t)hl * G.nq + row;
    // pass 1: the members' LSE values (one per lane, lanes stride over members)
    float m = kNegInfF;
    for (int c = lane; c < G.n_members; c += 32) m = fmaxf(m, __ldg(lse_partial + members[G.member_begin + c].lse_offset + lse_idx));
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
    Vec<D> acc;
#pragma unroll
    for (int e = 0; e < E; ++e) acc.v[e] = 0.f;
    float lse = kNegInfF;
    if (m != kNegInfF) {
      float tot = 0.f;
      for (int c = lane; c < G.n_members; c += 32)
        tot += ex2((__ldg(lse_partial + members[G.member_begin + c].lse_offset + lse_idx) - m) * kLog2e);
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
      lse = m + lg2(tot) * kLn2f;
      // pass 2: weighted sum of the partial outputs, in member order; up to four
      // members' rows are loaded before their products are added
      for (int c0 = 0; c0 < G.n_members; c0 += 4) {
        Vec<D> x[4];
        float wgt[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (c0 + u < G.n_members) {
            const DevMember mb = members[G.member_begin + c0 + u];
            wgt[u] = ex2((__ldg(lse_partial + mb.lse_offset + lse_idx) - lse) * kLog2e);
            x[u].load(o_partial + mb.o_offset + vec_off);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (c0 + u < G.n_members) {
#pragma unroll
            for (int e = 0; e < E; ++e) acc.v[e] = fmaf(wgt[u], x[u].v[e], acc.v[e]);
          }
        }
      }
    }
    acc.store_bf16(o + G.out_offset + vec_off);
    if (lane == 0) lse_out[G.lse_offset + lse_idx] = lse;
  }
}

template <int D>
__global__ void __launch_bounds__(256) zl_bwd_pre_kernel(const DevItem* __restrict__ items, int32_t n_items,
                                                         int64_t total, const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ d_o,
                                                         float* __restrict__ ws_d, float* __restrict__ ws_dq,
                                                         int64_t acc_total) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  // zero the whole accumulator and any turn counters after it (a multiple of 4
  // words, 16-byte aligned)
  {
    float4* z4 = reinterpret_cast<float4*>(ws_dq);
    const int64_t n4 = acc_total / 4, nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += nthreads)
      z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += nwarps) {
    const DevItem& it = items[find_segment(items, n_items, w)];
    const int nh = it.h_hi - it.h_lo, nq = it.q_hi - it.q_lo;
    const int64_t local = w - it.rowhead_begin;
    const int64_t row = local / nh;
    const int hl = (int)(local - row * nh);
    const int64_t vec_off = (row * nh + hl) * D + lane * E;
    Vec<D> a, g;
    a.load_bf16(o + it.fin_out_offset + vec_off);
    g.load_bf16(d_o + it.fin_out_offset + vec_off);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) s = fmaf(a.v[e], g.v[e], s);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
    if (lane == 0) ws_d[it.ws_d_offset + (int64_t)hl * nq + row] = s;
  }
}

template <int D>
__global__ void __launch_bounds__(256) zl_dq_finalize_kernel(const DevItem* __restrict__ items, int32_t n_items,
                                                             int64_t total, const float* __restrict__ ws_dq,
                                                             float* __restrict__ dq, float scale) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += nwarps) {
    const DevItem& it = items[find_segment(items, n_items, w)];
    const int nh = it.h_hi - it.h_lo, nq = it.q_hi - it.q_lo;
    const int64_t local = w - it.rowhead_begin;
    const int hl = (int)(local / nq);
    const int64_t row = local - (int64_t)hl * nq;
    const int64_t vec_off = (row * nh + hl) * D + lane * E;
    Vec<D> a;
    a.load(ws_dq + it.ws_dq_offset + acc_index(row, hl, lane * E, nq, D));
#pragma unroll
    for (int e = 0; e < E; ++e) a.v[e] *= scale;
    a.store(dq + it.dq_offset + vec_off);
  }
}

int row_grid(int64_t total, int num_sms) {
  const int64_t warps_per_block = 8;
  int64_t blocks = (total + warps_per_block - 1) / warps_per_block;
  const int64_t cap = (int64_t)num_sms * 8;  // 8 resident 256-thread blocks per SM
  return (int)(blocks < cap ? blocks : cap);
}

}  // namespace

cudaError_t launch_merge(int head_dim, const DevGroup* groups, int32_t n_groups, const DevMember* members,
                         int64_t total, const float* o_partial, const float* lse_partial, __nv_bfloat16* o,
                         float* lse_out, int num_sms, cudaStream_t stream) {
  if (total == 0 || n_groups == 0) return cudaSuccess;
  const int grid = row_grid(total, num_sms);
  if (head_dim == 128)
    zl_merge_kernel<128><<<grid, 256, 0, stream>>>(groups, n_groups, members, total, o_partial, lse_partial, o, lse_out);
  else
    zl_merge_kernel<64><<<grid, 256, 0, stream>>>(groups, n_groups, members, total, o_partial, lse_partial, o, lse_out);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(int head_dim, const DevItem* items, int32_t n_items, int64_t total,
                           const __nv_bfloat16* o, const __nv_bfloat16* d_o, float* ws_d, float* ws_dq,
                           int64_t acc_total, int num_sms, cudaStream_t stream) {
  if (total == 0) return cudaSuccess;
  const int grid = row_grid(total > acc_total / 128 ? total : acc_total / 128, num_sms);
  if (head_dim == 128)
    zl_bwd_pre_kernel<128><<<grid, 256, 0, stream>>>(items, n_items, total, o, d_o, ws_d, ws_dq, acc_total);
  else
    zl_bwd_pre_kernel<64><<<grid, 256, 0, stream>>>(items, n_items, total, o, d_o, ws_d, ws_dq, acc_total);
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(int head_dim, const DevItem* items, int32_t n_items, int64_t total,
                               const float* ws_dq, float* dq, float scale, int num_sms, cudaStream_t stream) {
  if (total == 0) return cudaSuccess;
  const int grid = row_grid(total, num_sms);
  if (head_dim == 128)
    zl_dq_finalize_kernel<128><<<grid, 256, 0, stream>>>(items, n_items, total, ws_dq, dq, scale);
  else
    zl_dq_finalize_kernel<64><<<grid, 256, 0, stream>>>(items, n_items, total, ws_dq, dq, scale);
  return cudaGetLastError();
}

}  // namespace zl
