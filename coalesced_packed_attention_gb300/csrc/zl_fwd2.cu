// Forward kernel of the coalesced attention engine, two query sub-tiles per CTA (sm_103a).
//
// Computes exactly what the single-tile forward computes — exact softmax attention of
// every work item over its own KV chunk, O and LSE ("Zellige", pith.science review,
// "What carries the argument": whole sequences and theta=(q,h,k) shards share one
// launch; FlashAttention [7] for the exact-attention cost model) — but a tile is 256
// query rows of one (item, head), split into two 128-row sub-tiles that share every K/V
// block loaded into shared memory.  Two softmax warpgroups, one per sub-tile, ping-pong
// against the tensor core:
//
//   tensor pipe:  ... PV0_{j-1}  S0_j  PV1_{j-1}  S1_j  PV0_j  S0_{j+1} ...
//   warpgroup 0:        softmax(S0_j) while PV1_{j-1} and S1_j run
//   warpgroup 1:        softmax(S1_j) while PV0_j and S0_{j+1} run
//
// so each softmax has two MMA slots of slack, and K/V traffic per FLOP is halved.
// Because S_w,j is issued after PV_w,{j-1}, the commit that signals S_w,j also proves
// PV_w,{j-1} complete: a warpgroup may rescale its O row right after it sees S.
//
// Roles (320 threads, one CTA per SM):
//   warps 0-3  softmax warpgroup 0 (query rows 0..127 of the tile; thread = TMEM lane)
//   warps 4-7  softmax warpgroup 1 (query rows 128..255)
//   warp 8     TMA producer (tile claims, Q0/Q1 once per tile, K/V ring)
//   warp 9     MMA issuer (single thread)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [384,384+d).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zl_internal.h"
#include "zl_kernels.h"
#include "zl_ptx.cuh"

namespace zl {

namespace {

template <int D>
struct Fwd2Layout {
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr int kBox = 128 * 128;           // one 128-row x 128-byte TMA box
  static constexpr int kTile = 128 * D * 2;        // one bf16 [128, D] tile
  static constexpr int kQ = 0;                     // Q0, Q1
  static constexpr int kK = kQ + 2 * kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  static constexpr int kNumBars = 2 + 1 + 4 * kStages + 2 + 2 + 2 + 2 + 2 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;     // room to align the base to 1024 B
};

constexpr float kThr = 8.0f;  // rescale O only when the row max grows by > 2^8 (log2 units)
constexpr float kLn2v = 0.69314718055994530942f;
constexpr float kNegInfv = -__builtin_huge_valf();

__device__ __forceinline__ bool wait2(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long limit,
                                      int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(status, 0, ZL_ERR_TIMEOUT);
      return false;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    zl_fwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Fwd2Layout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* q_full = bar;              // [2] one per sub-tile
  uint64_t* q_empty = bar + 2;
  uint64_t* k_full = bar + 3;          // [S]
  uint64_t* k_empty = k_full + S;
  uint64_t* v_full = k_empty + S;
  uint64_t* v_empty = v_full + S;
  uint64_t* s_full = v_empty + S;      // [2] per sub-tile
  uint64_t* p_full = s_full + 2;       // [2]
  uint64_t* o_bar = p_full + 2;        // [2] last PV of a tile done
  uint64_t* tile_full = o_bar + 2;     // [2]
  uint64_t* tile_empty = tile_full + 2;
  uint64_t* drain = tile_empty + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* tmem_slot = misc;
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(misc + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(o_bar + i, 1);
      mbar_init(tile_full + i, 1);
      mbar_init(tile_empty + i, 1 + 8);
    }
    mbar_init(q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(v_full + s, 1);
      mbar_init(v_empty + s, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const long long lim = p.wait_limit;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t tile_it = 0, kv_it = 0, q_it = 0;
      bool ok = true;
      while (ok) {
        const int t = atomicAdd(p.counter, 1);
        const int tid = t < p.n_tiles ? t : -1;
        const uint32_t slot = tile_it & 1;
        if (!wait2(tile_empty + slot, ((tile_it >> 1) & 1) ^ 1, abort_flag, lim, p.status)) break;
        ring[slot] = tid;
        mbar_arrive(tile_full + slot);
        ++tile_it;
        if (tid < 0) break;
        const DevTile tl = p.tiles[tid];
        const DevItem& it = p.items[tl.item];
        const int nblk = (it.kv_hi - it.kv_lo + kBlockN - 1) / kBlockN;
        if (nblk == 0) continue;
        const int rows = it.q_hi - it.q_lo - tl.block * kFwdBlockM;
        const int nsub = rows > 128 ? 2 : 1;
        if (!wait2(q_empty, (q_it & 1) ^ 1, abort_flag, lim, p.status)) break;
        ++q_it;
        const int row0 = (int)it.seq_offset + it.q_lo + tl.block * kFwdBlockM;
        for (int w = 0; w < nsub; ++w) {
          mbar_arrive_expect_tx(q_full + w, L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sQ + w * L::kTile + c * L::kBox, &tm_q, q_full + w, 64 * c, tl.head, row0 + 128 * w);
        }
        const int kv0 = (int)it.seq_offset + it.kv_lo;
        for (int j = 0; j < nblk; ++j) {
          const uint32_t s = kv_it % S, ph = (kv_it / S) & 1;
          if (!wait2(k_empty + s, ph ^ 1, abort_flag, lim, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(k_full + s, L::kTile);
          if (p.withhold_load && kv_it == 0) {
            // test hook: the announced bytes never arrive; a bounded wait runs out
          } else {
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sK + s * L::kTile + c * L::kBox, &tm_k, k_full + s, 64 * c, tl.head, kv0 + j * kBlockN);
          }
          if (!wait2(v_empty + s, ph ^ 1, abort_flag, lim, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(v_full + s, L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sV + s * L::kTile + c * L::kBox, &tm_v, v_full + s, 64 * c, tl.head, kv0 + j * kBlockN);
          ++kv_it;
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (control flow, waits and descriptors are
    // warp-uniform); one elected lane executes each product and commit.
    {
      constexpr uint32_t kIdS = idesc_bf16(128, kBlockN, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      uint32_t tile_it = 0, kv_it = 0;
      uint32_t qcount[2] = {0, 0};  // Q sub-tile loads consumed
      uint32_t pcount[2] = {0, 0};  // P handoffs consumed per sub-tile
      bool ok = true;
      auto wait_w = [&](uint64_t* b, uint32_t parity) {
        return __all_sync(0xffffffffu, wait2(b, parity, abort_flag, lim, p.status));
      };
      // operand descriptors built once; a K step only advances the start address
      const uint64_t dQ0 = sdesc_sw128(aQ, 16, 1024), dK0 = sdesc_sw128(aK, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(aV, L::kBox, 1024);
      auto issue_s = [&](int w, uint32_t stage) {
        const uint64_t dq = sdesc_add(dQ0, w * L::kTile), dk = sdesc_add(dK0, stage * L::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * L::kBox + (kk & 3) * 32;
          mma_ss_w(tmem + 128 * w, sdesc_add(dq, koff), sdesc_add(dk, koff), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit_w(s_full + w);
      };
      auto issue_pv = [&](int w, uint32_t stage, bool first) -> bool {
        if (!wait_w(p_full + w, pcount[w] & 1)) return false;
        ++pcount[w];
        tc_fence_after();
        const uint64_t dv = sdesc_add(dV0, stage * L::kTile);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_w(tmem + 256 + 128 * w, tmem + 128 * w + kk * 8, sdesc_add(dv, kk * 2048), kIdPV,
                   (first && kk == 0) ? 0u : 1u);
        return true;
      };
      while (ok) {
        const uint32_t slot = tile_it & 1;
        if (!wait_w(tile_full + slot, (tile_it >> 1) & 1)) break;
        const int tid = ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(tile_empty + slot);
        ++tile_it;
        if (tid < 0) break;
        const DevTile tl = p.tiles[tid];
        const DevItem& it = p.items[tl.item];
        const int nblk = (it.kv_hi - it.kv_lo + kBlockN - 1) / kBlockN;
        if (nblk == 0) continue;
        const int nsub = (it.q_hi - it.q_lo - tl.block * kFwdBlockM) > 128 ? 2 : 1;
        uint32_t pstage = 0, pph = 0;
        for (int j = 0; j < nblk && ok; ++j) {
          const uint32_t s = kv_it % S, ph = (kv_it / S) & 1;
          if (!wait_w(k_full + s, ph)) { ok = false; break; }
          if (j > 0 && !wait_w(v_full + pstage, pph)) { ok = false; break; }
          if (j == 0 && !wait_w(q_full + 0, (qcount[0]++) & 1)) { ok = false; break; }
          tc_fence_after();
          if (j > 0 && !issue_pv(0, pstage, j == 1)) { ok = false; break; }
          issue_s(0, s);
          if (nsub == 2) {
            if (j == 0 && !wait_w(q_full + 1, (qcount[1]++) & 1)) { ok = false; break; }
            tc_fence_after();
            if (j > 0 && !issue_pv(1, pstage, j == 1)) { ok = false; break; }
            issue_s(1, s);
          }
          if (j > 0) mma_commit_w(v_empty + pstage);
          mma_commit_w(k_empty + s);
          if (j == nblk - 1) mma_commit_w(q_empty);
          pstage = s; pph = ph;
          ++kv_it;
        }
        if (!ok) break;
        if (!wait_w(v_full + pstage, pph)) break;
        // the last block's V rows past the item's KV range are other tokens: their
        // weights are zero, but 0 x NaN is not, so they are zeroed before PV reads them
        const int vrows = (it.kv_hi - it.kv_lo) - (nblk - 1) * kBlockN;
        if (vrows < kBlockN) {
          zero_tile_rows<D>(aV + pstage * L::kTile, vrows, lane);
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (!issue_pv(0, pstage, nblk == 1)) break;
        mma_commit_w(o_bar + 0);
        if (nsub == 2) {
          if (!issue_pv(1, pstage, nblk == 1)) break;
          mma_commit_w(o_bar + 1);
        }
        mma_commit_w(v_empty + pstage);
      }
      mma_commit_w(drain);
      wait_w(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int w = warp >> 2;                   // sub-tile of this warpgroup
    const int r = threadIdx.x & 127;           // row of the sub-tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + 128 * w;
    const uint32_t tO = tmem + lane_base + 256 + 128 * w;
    const float sl2 = p.scale_log2;
    uint32_t tile_it = 0, sc = 0, tiles_done = 0;
    for (;;) {
      const uint32_t slot = tile_it & 1;
      if (!__all_sync(0xffffffffu, wait2(tile_full + slot, (tile_it >> 1) & 1, abort_flag, lim, p.status))) break;
      const int tid = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(tile_empty + slot);
      ++tile_it;
      if (tid < 0) break;
      const DevTile tl = p.tiles[tid];
      const DevItem it = p.items[tl.item];
      const int nkv = it.kv_hi - it.kv_lo;
      const int nblk = (nkv + kBlockN - 1) / kBlockN;
      const int nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo;
      const int sub_rows = nq - tl.block * kFwdBlockM - 128 * w;  // rows of this sub-tile (<= 0: none)
      if (sub_rows <= 0) continue;
      const int q_local = tl.block * kFwdBlockM + 128 * w + r;
      const bool row_ok = r < sub_rows;
      const int hl = tl.head - it.h_lo;

      float m_used = kNegInfv, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk; ++j) {
        if (!__all_sync(0xffffffffu, wait2(s_full + w, sc & 1, abort_flag, lim, p.status))) { ok = false; break; }
        ++sc;
        tc_fence_after();
        float s[128];
        {
          uint32_t u[4][32];  // all four loads in flight, one wait
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, u[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) s[32 * c + e] = __uint_as_float(u[c][e]);
        }
        const int valid = nkv - j * kBlockN;
        if (valid < kBlockN) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= valid) s[c] = kNegInfv;
        }
        // row max as 8 independent chains of three-input maxima (one warp per
        // sub-partition per warpgroup leaves little room to hide a long dependent chain);
        // chain e takes s[e + 8k], k = 0..15
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float m = max3(s[e], s[e + 8], s[e + 16]);
#pragma unroll
          for (int k = 3; k < 15; k += 2) m = max3(m, s[e + 8 * k], s[e + 8 * k + 8]);
          mx8[e] = fmaxf(m, s[e + 120]);
        }
        const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_blk = mx * sl2;
        const bool need = m_blk > m_used + kThr;
        const bool rescale = j > 0 && __any_sync(0xffffffffu, need);
        const float f = need ? ex2(m_used - m_blk) : 1.f;  // exp2(-inf) = 0 on the first block
        if (need) { l *= f; m_used = m_blk; }
        // exponent arguments and the row sum two columns per instruction; sum chain k
        // (lane x / y) collects the columns = 2k / 2k+1 mod 8, in column order
        float2 sum4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        const float2 sl2v = make_float2(sl2, sl2), nm = make_float2(-m_used, -m_used);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = fma2(make_float2(s[32 * c + 2 * e], s[32 * c + 2 * e + 1]), sl2v, nm);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            sum4[e & 3] = add2(sum4[e & 3], pp);
            pk[e] = pack_bf16(pp.x, pp.y);
          }
          tmem_st16(tS + 16 * c, pk);
        }
        l += ((sum4[0].x + sum4[0].y) + (sum4[1].x + sum4[1].y)) + ((sum4[2].x + sum4[2].y) + (sum4[3].x + sum4[3].y));
        if (rescale) {
          // S_w,j was issued after PV_w,{j-1}: its commit proves O_w stable here, and
          // PV_w,j waits for this warpgroup's P handoff below
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tO + 32 * c, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * f);
            tmem_st32(tO + 32 * c, u);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + w);
      }
      if (!ok) break;
      if (nblk > 0) {
        if (!__all_sync(0xffffffffu, wait2(o_bar + w, tiles_done & 1, abort_flag, lim, p.status))) break;
        ++tiles_done;
        tc_fence_after();
      }
      // ---- epilogue: O / l and LSE
      const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
      const float lse_v = nblk > 0 ? (m_used + lg2(l)) * kLn2v : kNegInfv;
      const int64_t row_off = (int64_t)q_local * nh * D + (int64_t)hl * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (nblk > 0) {
          tmem_ld32(tO + 32 * c, u);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = 0u;
        }
        if (row_ok) {
          if (!it.emit_lse) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + it.out_offset + row_off + 32 * c);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4) {
              uint4 q4;
              q4.x = pack_bf16(__uint_as_float(u[8 * v4 + 0]) * inv_l, __uint_as_float(u[8 * v4 + 1]) * inv_l);
              q4.y = pack_bf16(__uint_as_float(u[8 * v4 + 2]) * inv_l, __uint_as_float(u[8 * v4 + 3]) * inv_l);
              q4.z = pack_bf16(__uint_as_float(u[8 * v4 + 4]) * inv_l, __uint_as_float(u[8 * v4 + 5]) * inv_l);
              q4.w = pack_bf16(__uint_as_float(u[8 * v4 + 6]) * inv_l, __uint_as_float(u[8 * v4 + 7]) * inv_l);
              dst[v4] = q4;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.o_partial + it.out_offset + row_off + 32 * c);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst[v4] = make_float4(__uint_as_float(u[4 * v4 + 0]) * inv_l, __uint_as_float(u[4 * v4 + 1]) * inv_l,
                                    __uint_as_float(u[4 * v4 + 2]) * inv_l, __uint_as_float(u[4 * v4 + 3]) * inv_l);
          }
        }
      }
      if (row_ok) p.lse[it.lse_offset + (int64_t)hl * nq + q_local] = lse_v;
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
cudaError_t launch_fwd2_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int num_sms, cudaStream_t stream) {
  using L = Fwd2Layout<D>;
  const int smem = L::kAlloc > 120 * 1024 ? L::kAlloc : 120 * 1024;  // one CTA per SM (TMEM 512 cols)
  static PerDeviceOnce configured;
  cudaError_t e = configured.run(
      [&] { return cudaFuncSetAttribute(zl_fwd2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (e != cudaSuccess) return e;
  const int grid = p.n_tiles < num_sms ? p.n_tiles : num_sms;
  if (grid == 0) return cudaSuccess;
  e = cudaMemsetAsync(p.counter, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  zl_fwd2_kernel<D><<<grid, 320, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd2(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const FwdParams& p, int num_sms, cudaStream_t stream) {
  return head_dim == 128 ? launch_fwd2_impl<128>(tq, tk, tv, p, num_sms, stream)
                         : launch_fwd2_impl<64>(tq, tk, tv, p, num_sms, stream);
}

}  // namespace zl
