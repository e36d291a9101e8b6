// Row-parallel, HBM-bound kernels of the engine: the LSE-weighted merge of k-split
// partials, the backward row sums D = rowsum(dO * O) (plus zeroing of the dQ
// accumulator), and the dQ finalisation.  Each is a single pass over its bytes, so the
// design goal is enough independent 16-byte loads in flight per SM to cover DRAM
// latency: every load of a (row, head) pair is issued before any of its arithmetic
// (the merge issues its members' partial rows together with their LSE values instead of
// after the weights), consecutive pairs go to neighbouring lanes or warps, and the
// segment (item or group) of a pair is found by moving forward from the previous one.
// The dQ accumulator is tiled by query block (acc_index); the finalisation reads it in
// storage order (fully coalesced) and transposes it through shared memory, so that its
// writes to dq are whole 256-byte row pieces too.
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

// Segment holding index idx: the last segment whose start (key(seg)) is <= idx, found
// from `cur` (a segment at or before it): a short forward walk over the next few
// segments, a binary search beyond them.  Empty segments share their start with the next
// one, so the last match is the non-empty one.
template <typename T, typename Key>
__device__ __forceinline__ int seek(const T* segs, int n, int cur, int64_t idx, Key key) {
#pragma unroll 1
  for (int step = 0; step < 4; ++step) {
    if (cur + 1 >= n || key(segs[cur + 1]) > idx) return cur;
    ++cur;
  }
  int lo = cur, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (key(segs[mid]) <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// by row-head index (items and merge groups)
template <typename T>
__device__ __forceinline__ int seek_segment(const T* segs, int n, int cur, int64_t idx) {
  return seek(segs, n, cur, idx, [](const T& x) { return x.rowhead_begin; });
}

__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint2 ldg8(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

// sum of the products of two packed bf16 pairs
__device__ __forceinline__ float dot_bf16x2(uint32_t a, uint32_t b, float acc) {
  acc = fmaf(__uint_as_float(a << 16), __uint_as_float(b << 16), acc);
  return fmaf(__uint_as_float(a & 0xffff0000u), __uint_as_float(b & 0xffff0000u), acc);
}

// d/32 fp32 values per lane: one member's piece of a partial row
template <int D>
struct Piece;
template <>
struct Piece<128> {
  float v[4];
  __device__ __forceinline__ void load(const float* p) {
    const uint4 x = ldg16(p);
    v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y); v[2] = __uint_as_float(x.z); v[3] = __uint_as_float(x.w);
  }
  __device__ __forceinline__ void store_bf16(__nv_bfloat16* p) const {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
  }
};
template <>
struct Piece<64> {
  float v[2];
  __device__ __forceinline__ void load(const float* p) {
    const uint2 x = ldg8(p);
    v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y);
  }
  __device__ __forceinline__ void store_bf16(__nv_bfloat16* p) const {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16(v[0], v[1]);
  }
};

// One (row, head) of a merge group, in two phases so that a warp can have the loads of
// two pairs in flight: load() issues every member's LSE (one per lane) and every member's
// piece of the partial row (groups of up to kMem members); finish() forms the weights
// and the weighted sum in member order and stores.  Larger groups are merged entirely in
// finish(), kMem members' pieces at a time.
template <int D, int kMem>
struct MergePair {
  static constexpr int E = D / 32;
  bool valid = false;
  int n = 0;
  const DevMember* mem = nullptr;
  int64_t vec_off = 0, lse_idx = 0, out_off = 0, lse_out_off = 0;
  float l = -__builtin_huge_valf();
  Piece<D> x[kMem];

  __device__ __forceinline__ void load(const DevGroup* groups, int n_groups, const DevMember* members, int& g,
                                       int64_t w, int64_t total, const float* o_partial, const float* lse_partial,
                                       int lane) {
    valid = w < total;
    if (!valid) return;
    g = seek_segment(groups, n_groups, g, w);
    const DevGroup G = groups[g];
    const int64_t local = w - G.rowhead_begin;
    const int64_t row = local / G.nh;
    const int hl = (int)(local - row * G.nh);
    vec_off = (row * G.nh + hl) * D + lane * E;
    lse_idx = (int64_t)hl * G.nq + row;
    out_off = G.out_offset + vec_off;
    lse_out_off = G.lse_offset + lse_idx;
    mem = members + G.member_begin;
    n = G.n_members;
    if (n > kMem) return;
    if (lane < n) l = __ldg(lse_partial + mem[lane].lse_offset + lse_idx);
#pragma unroll
    for (int c = 0; c < kMem; ++c)
      if (c < n) x[c].load(o_partial + mem[c].o_offset + vec_off);
  }

  __device__ __forceinline__ void finish(const float* o_partial, const float* lse_partial, __nv_bfloat16* o,
                                         float* lse_out, int lane) {
    if (!valid) return;  // warp-uniform
    Piece<D> acc;
#pragma unroll
    for (int e = 0; e < E; ++e) acc.v[e] = 0.f;
    float lse = kNegInfF;
    if (n <= kMem) {
      float m = l;
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
      float wgt = 0.f;
      if (m != kNegInfF) {
        float tot = ex2((l - m) * kLog2e);  // 0 for lanes without a member (l = -inf)
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
        lse = m + lg2(tot) * kLn2f;
        wgt = ex2((l - lse) * kLog2e);
      }
#pragma unroll
      for (int c = 0; c < kMem; ++c) {
        const float wc = __shfl_sync(0xffffffffu, wgt, c);
        if (c < n) {
#pragma unroll
          for (int e = 0; e < E; ++e) acc.v[e] = fmaf(wc, x[c].v[e], acc.v[e]);
        }
      }
    } else {
      // pass 1: the members' LSE values (lanes stride over members)
      float m = kNegInfF;
      for (int c = lane; c < n; c += 32) m = fmaxf(m, __ldg(lse_partial + mem[c].lse_offset + lse_idx));
#pragma unroll
      for (int s = 16; s > 0; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
      if (m != kNegInfF) {
        float tot = 0.f;
        for (int c = lane; c < n; c += 32) tot += ex2((__ldg(lse_partial + mem[c].lse_offset + lse_idx) - m) * kLog2e);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, s);
        lse = m + lg2(tot) * kLn2f;
        // pass 2: kMem members' pieces in flight at a time, added in member order
        for (int c0 = 0; c0 < n; c0 += kMem) {
          float wc[kMem];
#pragma unroll
          for (int u = 0; u < kMem; ++u) {
            if (c0 + u < n) {
              const DevMember mb = mem[c0 + u];
              wc[u] = ex2((__ldg(lse_partial + mb.lse_offset + lse_idx) - lse) * kLog2e);
              x[u].load(o_partial + mb.o_offset + vec_off);
            }
          }
#pragma unroll
          for (int u = 0; u < kMem; ++u) {
            if (c0 + u < n) {
#pragma unroll
              for (int e = 0; e < E; ++e) acc.v[e] = fmaf(wc[u], x[u].v[e], acc.v[e]);
            }
          }
        }
      }
    }
    acc.store_bf16(o + out_off);
    if (lane == 0) lse_out[lse_out_off] = lse;
  }
};

// One warp per (row, head) of a group; kPairs pairs (grid-stride neighbours) per warp and
// iteration with all their loads in flight before any arithmetic.  kMem is chosen at
// launch from the largest group (registers grow with it; occupancy falls).
template <int D, int kMem, int kPairs>
__global__ void __launch_bounds__(256) zl_merge_kernel(const DevGroup* __restrict__ groups, int32_t n_groups,
                                                       const DevMember* __restrict__ members, int64_t total,
                                                       const float* __restrict__ o_partial,
                                                       const float* __restrict__ lse_partial,
                                                       __nv_bfloat16* __restrict__ o, float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  int g[kPairs];
#pragma unroll
  for (int u = 0; u < kPairs; ++u) g[u] = 0;
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < total; w += kPairs * nwarps) {
    MergePair<D, kMem> pr[kPairs];
#pragma unroll
    for (int u = 0; u < kPairs; ++u)
      pr[u].load(groups, n_groups, members, g[u], w + u * nwarps, total, o_partial, lse_partial, lane);
#pragma unroll
    for (int u = 0; u < kPairs; ++u) pr[u].finish(o_partial, lse_partial, o, lse_out, lane);
  }
}

// Row sums D: kPieces lanes per (row, head) (one 16-byte piece of its O and dO row each),
// 32 / kPieces pairs per warp and step, kUnroll steps' loads in flight together.  The
// block first zeroes its share of the dQ accumulator (and of any turn counters after it).
template <int D>
__global__ void __launch_bounds__(256) zl_bwd_pre_kernel(const DevItem* __restrict__ items, int32_t n_items,
                                                         int64_t total, const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ d_o,
                                                         float* __restrict__ ws_d, float* __restrict__ ws_dq,
                                                         int64_t acc_total) {
  constexpr int kPieces = D * 2 / 16;  // 16 (d = 128) or 8 (d = 64)
  constexpr int kRows = 32 / kPieces;
  constexpr int kUnroll = 4;
  constexpr int kPerWarp = kRows * kUnroll;
  const int lane = threadIdx.x & 31, sub = lane / kPieces, piece = lane % kPieces;
  {
    // zero the whole accumulator and any turn counters after it (a multiple of 4 words,
    // 16-byte aligned)
    float4* z4 = reinterpret_cast<float4*>(ws_dq);
    const int64_t n4 = acc_total / 4, nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += nthreads)
      z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  int seg = 0;
  for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kPerWarp; base < total;
       base += nwarps * kPerWarp) {
    uint4 a[kUnroll], b[kUnroll];
    int64_t dst[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t w = base + u * kRows + sub;
      dst[u] = -1;
      a[u] = b[u] = make_uint4(0u, 0u, 0u, 0u);
      if (w < total) {
        seg = seek_segment(items, n_items, seg, w);
        const DevItem& it = items[seg];
        const int nh = it.h_hi - it.h_lo, nq = it.q_hi - it.q_lo;
        const int64_t local = w - it.rowhead_begin;
        const int64_t row = local / nh;
        const int hl = (int)(local - row * nh);
        const int64_t off = it.fin_out_offset + (row * nh + hl) * D + piece * 8;
        a[u] = ldg16(o + off);
        b[u] = ldg16(d_o + off);
        dst[u] = it.ws_d_offset + (int64_t)hl * nq + row;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float s = dot_bf16x2(a[u].x, b[u].x, 0.f);
      s = dot_bf16x2(a[u].y, b[u].y, s);
      s = dot_bf16x2(a[u].z, b[u].z, s);
      s = dot_bf16x2(a[u].w, b[u].w, s);
#pragma unroll
      for (int k = kPieces / 2; k > 0; k >>= 1) s += __shfl_xor_sync(0xffffffffu, s, k);
      if (piece == 0 && dst[u] >= 0) ws_d[dst[u]] = s;
    }
  }
}

// dQ finalisation: one block per slab of the tiled accumulator, the 128 rows x 64 columns
// of one (item, head, query block, 64-column half): the block reads the slab in storage
// order (32 KB contiguous), stages it in shared memory and writes each row's 64 columns
// (256 contiguous bytes of dq), scaled.  Every item's accumulator is a whole number of
// slabs laid out in item order, so slab s starts at 16-byte piece 2048 s.
template <int D>
__global__ void __launch_bounds__(256) zl_dq_finalize_kernel(const DevItem* __restrict__ items, int32_t n_items,
                                                             int64_t n_slabs, const float* __restrict__ ws_dq,
                                                             float* __restrict__ dq, float scale) {
  constexpr int kHalves = D / 64;
  __shared__ float4 tile[kBlockM][17];  // 16 pieces per row + 1: both walks free of bank conflicts
  const float4* acc4 = reinterpret_cast<const float4*>(ws_dq);
  int seg = 0;
  for (int64_t sl = blockIdx.x; sl < n_slabs; sl += gridDim.x) {
    const int64_t k0 = sl * (kBlockM * 16);
    seg = seek(items, n_items, seg, k0, [](const DevItem& x) { return x.ws_dq_offset / 4; });
    const DevItem& it = items[seg];
    const int nh = it.h_hi - it.h_lo, nq = it.q_hi - it.q_lo;
    const int nqb = (nq + kBlockM - 1) / kBlockM;
    // piece j of the item: ((hl * nqb + qb) * (d / 4) + c4) * 128 + r
    const int64_t j0 = k0 - it.ws_dq_offset / 4;
    const int64_t hq = j0 / (kBlockM * (D / 4));
    const int half = (int)((j0 / (kBlockM * 16)) % kHalves);
    const int qb = (int)(hq % nqb), hl = (int)(hq / nqb);
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = __ldg(acc4 + k0 + u * 256 + threadIdx.x);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = u * 256 + threadIdx.x;  // piece (c4 = k / 128, r = k % 128) of the slab
      tile[k & (kBlockM - 1)][k >> 7] = x[u];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = u * 256 + threadIdx.x;  // row r = k / 16, piece c = k % 16 of the output
      const int r = k >> 4, c = k & 15;
      const int row = qb * kBlockM + r;
      if (row < nq) {
        const float4 v = tile[r][c];
        *reinterpret_cast<float4*>(dq + it.dq_offset + ((int64_t)row * nh + hl) * D + half * 64 + 4 * c) =
            make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
      }
    }
    __syncthreads();
  }
}

// Grid of a grid-stride row kernel: enough 256-thread blocks for `units` (one unit per
// warp), at most as many as can be resident at once (one wave).
template <typename K>
int row_grid(K kernel, int64_t units, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int64_t blocks = (units + 7) / 8;
  const int64_t cap = (int64_t)num_sms * per_sm;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_merge(int head_dim, const DevGroup* groups, int32_t n_groups, const DevMember* members,
                         int64_t total, int32_t max_members, const float* o_partial, const float* lse_partial,
                         __nv_bfloat16* o, float* lse_out, int num_sms, cudaStream_t stream) {
  if (total == 0 || n_groups == 0) return cudaSuccess;
  using K = void (*)(const DevGroup*, int32_t, const DevMember*, int64_t, const float*, const float*, __nv_bfloat16*,
                     float*);
  // members loaded together: 2 or 4 with two pairs per warp in flight, else 8 with one
  K k;
  int pairs;
  if (max_members <= 2) {
    k = head_dim == 128 ? zl_merge_kernel<128, 2, 2> : zl_merge_kernel<64, 2, 2>; pairs = 2;
  } else if (max_members <= 4) {
    k = head_dim == 128 ? zl_merge_kernel<128, 4, 2> : zl_merge_kernel<64, 4, 2>; pairs = 2;
  } else {
    k = head_dim == 128 ? zl_merge_kernel<128, 8, 1> : zl_merge_kernel<64, 8, 1>; pairs = 1;
  }
  const int grid = row_grid(k, (total + pairs - 1) / pairs, num_sms);
  k<<<grid, 256, 0, stream>>>(groups, n_groups, members, total, o_partial, lse_partial, o, lse_out);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(int head_dim, const DevItem* items, int32_t n_items, int64_t total,
                           const __nv_bfloat16* o, const __nv_bfloat16* d_o, float* ws_d, float* ws_dq,
                           int64_t acc_total, int num_sms, cudaStream_t stream) {
  if (total == 0) return cudaSuccess;
  const int per_warp = (head_dim == 128 ? 2 : 4) * 4;  // pairs per warp and iteration
  auto k = head_dim == 128 ? zl_bwd_pre_kernel<128> : zl_bwd_pre_kernel<64>;
  const int grid = row_grid(k, (total + per_warp - 1) / per_warp, num_sms);
  k<<<grid, 256, 0, stream>>>(items, n_items, total, o, d_o, ws_d, ws_dq, acc_total);
  return cudaGetLastError();
}

cudaError_t launch_dq_finalize(int head_dim, const DevItem* items, int32_t n_items, int64_t acc_floats_total,
                               const float* ws_dq, float* dq, float scale, int num_sms, cudaStream_t stream) {
  const int64_t n_slabs = acc_floats_total / (kBlockM * 64);
  if (n_slabs == 0) return cudaSuccess;
  auto k = head_dim == 128 ? zl_dq_finalize_kernel<128> : zl_dq_finalize_kernel<64>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)num_sms * per_sm;
  const int grid = (int)(n_slabs < cap ? n_slabs : cap);
  k<<<grid, 256, 0, stream>>>(items, n_items, n_slabs, ws_dq, dq, scale);
  return cudaGetLastError();
}

}  // namespace zl
