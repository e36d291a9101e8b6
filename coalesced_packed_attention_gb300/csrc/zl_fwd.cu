// Forward kernel of the coalesced attention engine (sm_103a).
//
// One persistent launch runs every forward tile of a plan: a tile is 128 query rows
// of one head of one work item (a whole sequence or a theta=(q,h,k) shard; "Zellige",
// pith.science review, "What carries the argument").  The result is exact softmax
// attention over the item's own KV chunk (FlashAttention [7], cited there for the
// quadratic-compute / linear-memory assumption): S = scale Q K^T, an online softmax
// with row maxima and sums, O = P V, and LSE = ln sum exp(S).
//
// Roles (192 threads, one CTA per SM):
//   warps 0-3  softmax warpgroup: thread t owns query row t of the tile.  It reads its
//              S row from TMEM, keeps the running max / sum, writes P (bf16) back into
//              TMEM over S, rescales its O row when the max grows by more than 2^8,
//              and runs the epilogue (O / l, LSE) with 16-byte stores.
//   warp 4     TMA producer: claims tiles from the plan's atomic counter (longest
//              first), publishes them through a 2-slot ring, loads Q once per tile and
//              K/V blocks through a kStages-deep ring.
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T (SMEM x SMEM -> TMEM) and
//              O += P_{j-1} V_{j-1} (TMEM x SMEM -> TMEM), software-pipelined so the
//              softmax of block j overlaps the PV product of block j-1.
// TMEM (512 columns): S double buffer at columns [0,128) and [128,256), O at [256,256+d).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zl_internal.h"
#include "zl_kernels.h"
#include "zl_ptx.cuh"

namespace zl {


template <int D>
struct FwdLayout {
  static constexpr int kStages = D == 128 ? 2 : 3;
  static constexpr int kBox = 128 * 128;           // one 128-row x 128-byte TMA box
  static constexpr int kTile = 128 * D * 2;        // one bf16 [128, D] tile
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kBar = kV + kStages * kTile;
  static constexpr int kNumBars = 2 + 4 * kStages + 2 + 2 + 1 + 2 + 2 + 1;
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;     // room to align the base to 1024 B
};

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays <= 256 between rescales
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kNegInf = -__builtin_huge_valf();

struct FwdBars {
  uint64_t *q_full, *q_empty, *k_full, *k_empty, *v_full, *v_empty, *s_full, *p_full, *o_bar,
      *tile_full, *tile_empty, *drain;
};

__device__ __forceinline__ void record_error(int32_t* status, volatile int* abort_flag, int code) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long limit,
                                              int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      record_error(status, abort_flag, ZL_ERR_TIMEOUT);
      return false;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(192, 1)
    zl_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  FwdBars b;
  b.q_full = bar;
  b.q_empty = bar + 1;
  b.k_full = bar + 2;
  b.k_empty = b.k_full + S;
  b.v_full = b.k_empty + S;
  b.v_empty = b.v_full + S;
  b.s_full = b.v_empty + S;
  b.p_full = b.s_full + 2;
  b.o_bar = b.p_full + 2;
  b.tile_full = b.o_bar + 1;
  b.tile_empty = b.tile_full + 2;
  b.drain = b.tile_empty + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* tmem_slot = misc;
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(misc + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(b.q_full, 1);
    mbar_init(b.q_empty, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(b.k_full + s, 1);
      mbar_init(b.k_empty + s, 1);
      mbar_init(b.v_full + s, 1);
      mbar_init(b.v_empty + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b.s_full + i, 1);
      mbar_init(b.p_full + i, 128);
      mbar_init(b.tile_full + i, 1);
      mbar_init(b.tile_empty + i, 1 + 4);
    }
    mbar_init(b.o_bar, 1);
    mbar_init(b.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t tile_it = 0, kv_it = 0, q_it = 0;
      for (;;) {
        const int t = atomicAdd(p.counter, 1);
        const int tid = t < p.n_tiles ? t : -1;
        const uint32_t slot = tile_it & 1;
        if (!wait_or_abort(b.tile_empty + slot, ((tile_it >> 1) & 1) ^ 1, abort_flag, p.wait_limit, p.status)) break;
        ring[slot] = tid;
        mbar_arrive(b.tile_full + slot);
        ++tile_it;
        if (tid < 0) break;
        const DevTile tl = p.tiles[tid];
        const DevItem& it = p.items[tl.item];
        const int nkv = it.kv_hi - it.kv_lo;
        const int nblk = (nkv + kBlockN - 1) / kBlockN;
        if (nblk == 0) continue;
        if (!wait_or_abort(b.q_empty, (q_it & 1) ^ 1, abort_flag, p.wait_limit, p.status)) break;
        ++q_it;
        const int row0 = (int)it.seq_offset + it.q_lo + tl.block * kBlockM;
        mbar_arrive_expect_tx(b.q_full, L::kTile);
        for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * L::kBox, &tm_q, b.q_full, 64 * c, tl.head, row0);
        const int kv0 = (int)it.seq_offset + it.kv_lo;
        bool ok = true;
        for (int j = 0; j < nblk && ok; ++j) {
          const uint32_t s = kv_it % S, ph = (kv_it / S) & 1;
          ok = wait_or_abort(b.k_empty + s, ph ^ 1, abort_flag, p.wait_limit, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(b.k_full + s, L::kTile);
          if (p.withhold_load && kv_it == 0) {
            // test hook: the bytes announced above never arrive, so the MMA warp's
            // bounded wait runs out and the kernel reports ZL_ERR_TIMEOUT
          } else {
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(sK + s * L::kTile + c * L::kBox, &tm_k, b.k_full + s, 64 * c, tl.head, kv0 + j * kBlockN);
          }
          ok = wait_or_abort(b.v_empty + s, ph ^ 1, abort_flag, p.wait_limit, p.status);
          if (!ok) break;
          mbar_arrive_expect_tx(b.v_full + s, L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sV + s * L::kTile + c * L::kBox, &tm_v, b.v_full + s, 64 * c, tl.head, kv0 + j * kBlockN);
          ++kv_it;
        }
        if (!ok) break;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(128, kBlockN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      const uint32_t tO = tmem + 256;
      uint32_t tile_it = 0, kv_it = 0, q_it = 0, sc = 0;
      bool ok = true;
      // O += P_jj V_jj, P read from the S buffer the softmax overwrote with bf16.
      // operand descriptors built once; a K step or a ring slot only advances the start
      const uint64_t dQ = sdesc_sw128(aQ, 16, 1024), dK0 = sdesc_sw128(aK, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(aV, L::kBox, 1024);
      auto issue_pv = [&](uint32_t stage, uint32_t kvph, uint32_t scc, bool first) -> bool {
        if (!wait_or_abort(b.p_full + (scc & 1), (scc >> 1) & 1, abort_flag, p.wait_limit, p.status)) return false;
        if (!wait_or_abort(b.v_full + stage, kvph, abort_flag, p.wait_limit, p.status)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + (scc & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts(tO, tP + kk * 8, sdesc_add(dV0, stage * L::kTile + kk * 2048), kIdescPV, (first && kk == 0) ? 0u : 1u);
        mma_commit(b.v_empty + stage);
        mma_commit(b.o_bar);
        return true;
      };
      while (ok) {
        const uint32_t slot = tile_it & 1;
        if (!wait_or_abort(b.tile_full + slot, (tile_it >> 1) & 1, abort_flag, p.wait_limit, p.status)) break;
        const int tid = ring[slot];
        mbar_arrive(b.tile_empty + slot);
        ++tile_it;
        if (tid < 0) break;
        const DevTile tl = p.tiles[tid];
        const DevItem& it = p.items[tl.item];
        const int nblk = (it.kv_hi - it.kv_lo + kBlockN - 1) / kBlockN;
        if (nblk == 0) continue;
        if (!wait_or_abort(b.q_full, q_it & 1, abort_flag, p.wait_limit, p.status)) break;
        ++q_it;
        tc_fence_after();
        uint32_t pstage = 0, pph = 0, psc = 0;
        for (int j = 0; j < nblk; ++j) {
          const uint32_t s = kv_it % S, ph = (kv_it / S) & 1;
          if (!wait_or_abort(b.k_full + s, ph, abort_flag, p.wait_limit, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tS = tmem + (sc & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * L::kBox + (kk & 3) * 32;
            mma_ss(tS, sdesc_add(dQ, koff), sdesc_add(dK0, s * L::kTile + koff), kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(b.k_empty + s);
          mma_commit(b.s_full + (sc & 1));
          if (j == nblk - 1) mma_commit(b.q_empty);
          if (j > 0 && !issue_pv(pstage, pph, psc, j == 1)) { ok = false; break; }
          pstage = s; pph = ph; psc = sc;
          ++kv_it;
          ++sc;
        }
        if (!ok) break;
        if (!issue_pv(pstage, pph, psc, nblk == 1)) break;
      }
      // make sure no MMA is still writing TMEM before it is released
      mma_commit(b.drain);
      wait_or_abort(b.drain, 0, abort_flag, p.wait_limit, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int r = threadIdx.x;                 // row of the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    uint32_t tile_it = 0, sc = 0, pv_seen = 0;
    for (;;) {
      const uint32_t slot = tile_it & 1;
      if (!__all_sync(0xffffffffu, wait_or_abort(b.tile_full + slot, (tile_it >> 1) & 1, abort_flag, p.wait_limit, p.status))) break;
      const int tid = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(b.tile_empty + slot);
      ++tile_it;
      if (tid < 0) break;
      const DevTile tl = p.tiles[tid];
      const DevItem it = p.items[tl.item];
      const int nkv = it.kv_hi - it.kv_lo;
      const int nblk = (nkv + kBlockN - 1) / kBlockN;
      const int nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo;
      const int q_local = tl.block * kBlockM + r;
      const bool row_ok = q_local < nq;
      const int hl = tl.head - it.h_lo;

      float m_used = kNegInf, l = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk; ++j) {
        const uint32_t buf = sc & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(b.s_full + buf, (sc >> 1) & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem + lane_base + buf * 128;
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
        const int valid = nkv - j * kBlockN;  // columns >= valid are past the chunk
        if (valid < kBlockN) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= valid) s[c] = kNegInf;
        }
        // row max as 8 chains of three-input maxima; chain e takes s[e + 8k], k = 0..15
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
        const bool need = m_blk > m_used + kRescaleThreshold;
        bool waited = false;
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          // O holds P_{<j} V; wait for the last PV product before rescaling it
          if (!__all_sync(0xffffffffu, wait_or_abort(b.o_bar, pv_seen & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
          ++pv_seen;
          waited = true;
          tc_fence_after();
          const float f = need ? ex2(m_used - m_blk) : 1.f;
          if (need) { l *= f; m_used = m_blk; }
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_base + 256 + 32 * c, u);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * f);
            tmem_st32(tmem + lane_base + 256 + 32 * c, u);
          }
        } else if (need) {
          m_used = m_blk;  // first block: O is overwritten by the first PV product
        }
        // exponent arguments and the row sum two columns per instruction (four chains)
        float2 sum4[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        const float2 sl2v = make_float2(sl2, sl2), nm = make_float2(-m_used, -m_used);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = fma2(make_float2(s[64 * c + 2 * e], s[64 * c + 2 * e + 1]), sl2v, nm);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            sum4[e & 3] = add2(sum4[e & 3], pp);
            pk[e] = pack_bf16(pp.x, pp.y);
          }
          tmem_st32(tS + 32 * c, pk);
        }
        l += ((sum4[0].x + sum4[0].y) + (sum4[1].x + sum4[1].y)) + ((sum4[2].x + sum4[2].y) + (sum4[3].x + sum4[3].y));
        tmem_st_wait();
        if (j > 0 && !waited) {
          if (!__all_sync(0xffffffffu, wait_or_abort(b.o_bar, pv_seen & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
          ++pv_seen;
        }
        tc_fence_before();
        mbar_arrive(b.p_full + buf);
        ++sc;
      }
      if (!ok) break;
      if (nblk > 0) {
        if (!__all_sync(0xffffffffu, wait_or_abort(b.o_bar, pv_seen & 1, abort_flag, p.wait_limit, p.status))) break;
        ++pv_seen;
        tc_fence_after();
      }
      // ---- epilogue: O / l and LSE
      const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
      const float lse_v = nblk > 0 ? (m_used + lg2(l)) * kLn2 : kNegInf;
      const int64_t row_off = (int64_t)q_local * nh * D + (int64_t)hl * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t u[32];
        if (nblk > 0) {
          tmem_ld32(tmem + lane_base + 256 + 32 * c, u);
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
              uint4 w;
              w.x = pack_bf16(__uint_as_float(u[8 * v4 + 0]) * inv_l, __uint_as_float(u[8 * v4 + 1]) * inv_l);
              w.y = pack_bf16(__uint_as_float(u[8 * v4 + 2]) * inv_l, __uint_as_float(u[8 * v4 + 3]) * inv_l);
              w.z = pack_bf16(__uint_as_float(u[8 * v4 + 4]) * inv_l, __uint_as_float(u[8 * v4 + 5]) * inv_l);
              w.w = pack_bf16(__uint_as_float(u[8 * v4 + 6]) * inv_l, __uint_as_float(u[8 * v4 + 7]) * inv_l);
              dst[v4] = w;
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
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch_fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, int num_sms, cudaStream_t stream) {
  using L = FwdLayout<D>;
  const int smem = L::kAlloc > 120 * 1024 ? L::kAlloc : 120 * 1024;  // one CTA per SM (TMEM 512 cols)
  static PerDeviceOnce configured;
  cudaError_t e = configured.run(
      [&] { return cudaFuncSetAttribute(zl_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (e != cudaSuccess) return e;
  const int grid = p.n_tiles < num_sms ? p.n_tiles : num_sms;
  if (grid == 0) return cudaSuccess;
  e = cudaMemsetAsync(p.counter, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  zl_fwd_kernel<D><<<grid, 192, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int num_sms, cudaStream_t stream) {
  return head_dim == 128 ? launch_fwd_impl<128>(tq, tk, tv, p, num_sms, stream)
                         : launch_fwd_impl<64>(tq, tk, tv, p, num_sms, stream);
}

}  // namespace zl
