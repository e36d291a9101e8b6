// Backward kernel of the coalesced attention engine (sm_103a).
//
// Gradient of exact softmax attention for every work item, with each item's FINAL
// output O and global LSE (a k-split shard of theta=(q,h,k) uses its merged group's
// values, so its dQ is that chunk's contribution and its dK/dV are final; "Zellige",
// pith.science review, "What carries the argument").  With D_i = rowsum(dO_i * O_i):
//   P_ij = exp(s_ij - LSE_i),  dS_ij = P_ij (dO_i . V_j - D_i),
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij Q_i,  dQ_i = scale sum_j dS_ij K_j.
//
// A tile is 128 KV rows of one head of one item; the CTA keeps K_j, V_j in shared
// memory and dK_j, dV_j in TMEM while it walks the item's query blocks.  Per block:
//   S^T  = K Q_i^T      (SMEM x SMEM -> TMEM R0)   lanes = KV rows, columns = queries
//   dP^T = V dO_i^T     (SMEM x SMEM -> TMEM R1)
//   softmax warpgroups (thread = KV row; each takes 64 query columns): P^T and dS^T in
//   registers; P^T (bf16) goes to TMEM in place of S^T (R0 columns [0,32) and [64,96))
//   and dS^T (bf16) to shared memory
//   dV  += P^T dO_i     (TMEM x SMEM, dO read MN-major)
//   dQ_i = dS K         (SMEM x SMEM -> TMEM R1; both operands MN-major)
//   dK  += dS^T Q_i     (SMEM x SMEM; dS^T read K-major, Q MN-major)
//   the dQ warpgroup (thread = query row) reads dQ_i out of TMEM, stages it through shared
//   memory 16 KB at a time and hands each chunk to the bulk-copy engine as one reduce-add
//   into the fp32 accumulator; the scale is applied once when dQ is finalised.
// The tensor pipe runs dP^T_i, dV_i, S^T_{i+1}, dQ_i, dK_i: R0 is free once dV_i has
// read P^T and R1 once the warpgroups have read dP^T_i, so the softmax warpgroups form
// P_{i+1} while dQ_i and dK_i run and dQ_i drains.  The drain has warps of its own
// because an SM hands reductions to L2 at only some 30-45 GB/s, whichever unit issues
// them: the 64 KB of one block's dQ take about as long as the block's five products, so
// they must overlap everything else.  Bulk reduce-adds from shared memory keep them out
// of the sub-partitions' memory-instruction queues, where vector `red` instructions
// (paced or not) held up the TMEM loads, MMA issues and TMA issues of the warps beside
// them.  On long items the kernel runs against the board's power cap: the bytes it moves
// per FLOP (64 KB of reduce-adds and 64 KB of Q/dO per block pair) cost clock rate
// more than any one stage stalls the block period.
// Ordered dQ (plan flag ZL_PLAN_DETERMINISTIC_DQ; a separate instantiation, so the
// default kernel carries none of it): the order in which CTAs reach a query block
// decides the order of the fp32 additions, so by default dQ may change in its last bits
// between runs.  With the flag, the drain adds with vector reductions from registers,
// and each drain warp waits before adding its 32 rows of a
// block until that slice's turn counter (workspace) equals its KV-block index, and
// passes the turn on (index + 1, after a fence) when it reaches its next block, by
// which time most of those reductions have landed (handing it over right after the
// reductions made the fence wait for all of them: 1.4x slower); every element then
// sums KV tiles 0, 1, 2, ... in order.  Every tile walks the query blocks from block 0, and the
// planner lists the tiles of each cost block-major, so the KV tiles of one (item, head)
// are claimed in ascending order and far apart: waits are rare and only ever on tiles
// claimed earlier (held by running CTAs), which rules out a cycle of waits.
// TMEM (512 columns): R0 [0,128) S^T / P^T, R1 [128,256) dP^T / dQ, dV [256,256+d),
// dK [384,384+d).  Shared memory: K, V, Q (2 stages), dO (1 stage: free once dV has read
// it), dS^T, and two 16 KB dQ staging buffers; with ordered dQ adds, which stage nothing,
// their 32 KB hold a second dO stage.
// Warps: 0-7 softmax (two warpgroups), 8-11 dQ drain, 12 TMA producer, 13 MMA issuer,
// 14-15 idle.  The block is launched with 128 registers per thread (16 warps: four per
// SM sub-partition, 16K registers each) and the warpgroups then trade registers with
// setmaxnreg: per sub-partition 2 x 136 (softmax) + 152 (dQ) + 88 (producer / MMA) =
// 512 = 4 x 128, exactly the launch allocation, so no increase can wait for registers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zl_internal.h"
#include "zl_kernels.h"
#include "zl_ptx.cuh"

namespace zl {

namespace {

template <int D>
struct BwdLayout {
  static constexpr int kBox = 128 * 128;
  static constexpr int kTile = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;             // 2 stages
  static constexpr int kDO = kQ + 2 * kTile;        // 1 stage (free once dV has read it); ordered dQ
                                                    // adds use the staging region as a 2nd stage
  static constexpr int kDS = kDO + kTile;           // [128 kv][128 q] bf16, two 128-byte-swizzled boxes
  static constexpr int kStageBytes = 128 * 32 * 4;  // one 32-column chunk of a block's dQ, fp32
  static constexpr int kStage = kDS + 2 * kBox;     // 2 staging buffers of the dQ drain
  static constexpr int kLD = kStage + 2 * kStageBytes;  // [2 block parities] LSE*log2(e) and D of a block's 128 queries
  static constexpr int kBar = kLD + 2 * 2 * 128 * 4;
  static constexpr int kNumBars = 27;
  static_assert(2 * kStageBytes >= kTile && kStage % 1024 == 0, "second dO stage does not fit the staging region");
  static constexpr int kMisc = kBar + kNumBars * 8;
  static constexpr int kBytes = kMisc + 64;
};

constexpr float kLog2eB = 1.44269504088896340736f;
constexpr float kInfB = __builtin_huge_valf();

__device__ __forceinline__ void rec_err(int32_t* status, volatile int* abort_flag, int code) {
  *abort_flag = 1;
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long limit, int32_t* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      rec_err(status, abort_flag, ZL_ERR_TIMEOUT);
      return false;
    }
  }
}

// The per-item dO maps are rewritten in global memory by every backward call.
__device__ __forceinline__ void tensormap_acquire(const void* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}
// Fire-and-forget fp32 add of four consecutive floats (16-byte aligned) in global memory.
__device__ __forceinline__ void red_add_v4(float* addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(__uint_as_float(a)),
               "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
               : "memory");
}

// Bulk (1-D) reduce-add of `bytes` bytes of fp32 from shared memory into global memory
// by the bulk-copy engine, tracked by this thread's bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most one of this thread's bulk groups still has to read its source
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// wait until all of this thread's bulk groups are complete (their writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiles of one (item, head) walk the query blocks starting at different blocks, so
// CTAs running side by side add into different dQ rows instead of contending on one.
// With ordered dQ adds every tile walks from block 0: a tile then reaches each block no
// earlier than the tile before it in the add order.
template <bool kOrdered>
__device__ __forceinline__ int block_start(int kv_block, int nqb) {
  if constexpr (kOrdered) return 0;
  return nqb > 0 ? kv_block % nqb : 0;
}
__device__ __forceinline__ int first_block(int step, int start, int n) {
  const int b = start + step;
  return b >= n ? b - n : b;
}

// Ordered dQ adds (turn counters in global memory, written by other CTAs).
__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* a) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t* a, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// Orders this thread's earlier memory operations (the dQ reductions) before its later
// ones at GPU scope; acquire-release strength is all a turn hand-over needs (a
// sequentially consistent fence, as __threadfence() issues, costs far more).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Bounded wait until *turn == mine.  The tiles that advance the counter to `mine` were
// claimed before this one, so they are held by running CTAs; the limit only ends the
// wait when one of them has given up.
__device__ __forceinline__ bool wait_turn(const int32_t* turn, int32_t mine, volatile int* abort_flag, long long limit,
                                          int32_t* status) {
  if (ld_acquire_gpu(turn) == mine) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(32);
    if (ld_acquire_gpu(turn) == mine) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      rec_err(status, abort_flag, ZL_ERR_TIMEOUT);
      return false;
    }
  }
}

// TMEM column of the packed bf16 P^T in R0 for MMA K-step kk (16 queries): queries 0-63
// are packed by warpgroup 0 into columns [0,32), queries 64-127 by warpgroup 1 into
// [64,96), each over S^T columns it has already read.
__device__ __forceinline__ uint32_t pcol(int kk) { return (uint32_t)((kk >> 2) * 64 + (kk & 3) * 8); }

// Registers per thread of a warpgroup after the split.  setmaxnreg.inc only raises and
// setmaxnreg.dec only lowers the current count (the launch count before the first), so
// the form is chosen from the target; the launcher checks the launch count.
constexpr uint32_t kRegsLaunch = 128;
constexpr uint32_t kRegsSoftmax = 136, kRegsDrain = 152, kRegsMisc = 88;
static_assert(2 * kRegsSoftmax + kRegsDrain + kRegsMisc == 4 * kRegsLaunch,
              "register split must equal the launch allocation");
template <uint32_t N>
__device__ __forceinline__ void regs_to() {
  static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg takes a multiple of 8 in [24, 256]");
  if constexpr (N > kRegsLaunch)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
  else if constexpr (N < kRegsLaunch)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int D, bool kOrdered>
__global__ void __launch_bounds__(512, 1) zl_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                        const __grid_constant__ CUtensorMap tm_k,
                                                        const __grid_constant__ CUtensorMap tm_v,
                                                        const BwdParams p) {
  using L = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint64_t* kv_full = bar + 0;
  uint64_t* kv_empty = bar + 1;
  uint64_t* q_full = bar + 2;     // [2]
  uint64_t* do_full = bar + 4;    // dO of the block in shared memory
  uint64_t* do_empty = bar + 5;   // dV (the last reader of dO) complete
  uint64_t* q_empty = bar + 6;    // [2]
  uint64_t* s_full = bar + 8;     // S^T of the block in TMEM R0
  uint64_t* ds_ready = bar + 9;   // dS^T in shared memory, dP^T read out of R1 (256 arrivals)
  uint64_t* dq_full = bar + 10;
  uint64_t* dq_empty = bar + 11;
  uint64_t* kv_done = bar + 12;
  uint64_t* tile_full = bar + 13;   // [2]
  uint64_t* tile_empty = bar + 15;  // [2]
  uint64_t* drain = bar + 17;
  uint64_t* ld_full = bar + 18;   // LSE / D of a query block staged in shared memory
  uint64_t* p_ready = bar + 19;   // P^T in TMEM R0 (256 arrivals): the dV product may start
  uint64_t* dp_full = bar + 20;   // dP^T of the block in TMEM R1
  uint64_t* stage_full = bar + 21;  // [2] a dQ chunk written to staging buffer b (128 arrivals)
  uint64_t* stage_free = bar + 23;  // [2] the bulk reduce-add of buffer b has read it
  // dO stages: one (default), or two with ordered dQ adds, whose drain needs no staging
  // buffers (the second stage takes their place): block qit's dO is in stage dst_of(qit)
  constexpr uint32_t kDOStages = kOrdered ? 2 : 1;
  auto do_stage = [](uint32_t qit) { return kDOStages == 2 ? (qit & 1) : 0u; };
  auto do_phase = [](uint32_t qit) { return kDOStages == 2 ? ((qit >> 1) & 1) : (qit & 1); };
  auto do_full_s = [&](uint32_t st) { return st ? bar + 25 : do_full; };
  auto do_empty_s = [&](uint32_t st) { return st ? bar + 26 : do_empty; };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  uint32_t* tmem_slot = misc;
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(misc + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  float* sLD = reinterpret_cast<float*>(smem + L::kLD);  // block parity b: LSE at 256 b, D at 256 b + 128

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.status, 0, ZL_ERR_UNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1);
      mbar_init(q_empty + i, 1);
      mbar_init(stage_full + i, 128);
      mbar_init(stage_free + i, 1);
      mbar_init(tile_full + i, 1);
      mbar_init(tile_empty + i, 1 + 8 + 4);
    }
    for (uint32_t i = 0; i < 2; ++i) {
      mbar_init(do_full_s(i), 1);
      mbar_init(do_empty_s(i), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(kv_done, 1);
    mbar_init(drain, 1);
    mbar_init(ld_full, 256);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t* sK = smem + L::kK;
  uint8_t* sV = smem + L::kV;
  uint8_t* sQ = smem + L::kQ;
  uint8_t* sDO = smem + L::kDO;
  auto sDO_s = [&](uint32_t st) { return st ? smem + L::kStage : sDO; };
  uint8_t* sDS = smem + L::kDS;

  if (warp >= 12) {
   regs_to<kRegsMisc>();
   if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t tile_it = 0, kt = 0, qit = 0;
      bool ok = true;
      while (ok) {
        const int t = atomicAdd(p.counter, 1);
        const int tid = t < p.n_tiles ? t : -1;
        const uint32_t slot = tile_it & 1;
        if (!bwait(tile_empty + slot, ((tile_it >> 1) & 1) ^ 1, abort_flag, p.wait_limit, p.status)) break;
        ring[slot] = tid;
        mbar_arrive(tile_full + slot);
        ++tile_it;
        if (tid < 0) break;
        const DevTile tl = p.tiles[tid];
        const DevItem& it = p.items[tl.item];
        const int nq = it.q_hi - it.q_lo;
        const int nqb = (nq + kBlockM - 1) / kBlockM;
        if (nqb == 0) continue;
        const CUtensorMap* tm_do = p.do_maps + tl.item;
        tensormap_acquire(tm_do);
        if (!bwait(kv_empty, (kt & 1) ^ 1, abort_flag, p.wait_limit, p.status)) break;
        ++kt;
        const int kvrow = (int)it.seq_offset + it.kv_lo + tl.block * kBlockN;
        mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
        if (p.withhold_load && kt == 1) {
          // test hook: the announced bytes never arrive; a bounded wait runs out
        } else {
          for (int c = 0; c < D / 64; ++c) {
            tma_load_3d(sK + c * L::kBox, &tm_k, kv_full, 64 * c, tl.head, kvrow);
            tma_load_3d(sV + c * L::kBox, &tm_v, kv_full, 64 * c, tl.head, kvrow);
          }
        }
        const int hl = tl.head - it.h_lo;
        const int start = block_start<kOrdered>(tl.block, nqb);
        for (int is = 0; is < nqb; ++is) {
          const int ib = first_block(is, start, nqb);
          const uint32_t st = qit & 1, ph = (qit >> 1) & 1;
          if (!bwait(q_empty + st, ph ^ 1, abort_flag, p.wait_limit, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(q_full + st, L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sQ + st * L::kTile + c * L::kBox, &tm_q, q_full + st, 64 * c, tl.head,
                        (int)it.seq_offset + it.q_lo + ib * kBlockM);
          // block qit's dO waits until dV of the block that last used its stage has read it
          const uint32_t dst = do_stage(qit), dph = do_phase(qit);
          if (!bwait(do_empty_s(dst), dph ^ 1, abort_flag, p.wait_limit, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(do_full_s(dst), L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sDO_s(dst) + c * L::kBox, tm_do, do_full_s(dst), 64 * c, hl, ib * kBlockM);
          ++qit;
        }
      }
    }
   } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop (control flow, waits and descriptors are
    // warp-uniform); one elected lane executes each product and commit.
    {
      constexpr uint32_t kIdSq = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdKV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kIdDQ = idesc_bf16(128, D, true, true);
      const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aDO = smem_u32(sDO),
                     aDS = smem_u32(sDS);
      const uint32_t tR0 = tmem, tR1 = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
      auto wait_w = [&](uint64_t* b, uint32_t parity) {
        return __all_sync(0xffffffffu, bwait(b, parity, abort_flag, p.wait_limit, p.status));
      };
      // operand descriptors built once (K-major: LBO 16 B; MN-major: LBO one 16 KB box);
      // a K step or a ring slot only advances the start address
      // (low words only: all share the high word, see sdesc_join)
      const uint32_t kK = sdesc_lo(aK, 16), kV = sdesc_lo(aV, 16), kQ = sdesc_lo(aQ, 16), kDO = sdesc_lo(aDO, 16);
      const uint32_t kDS = sdesc_lo(aDS, 16);
      const uint32_t mK = sdesc_lo(aK, L::kBox), mQ = sdesc_lo(aQ, L::kBox), mDO = sdesc_lo(aDO, L::kBox);
      const uint32_t aDO1 = smem_u32(sDO_s(1));
      const uint32_t kDO1 = sdesc_lo(aDO1, 16), mDO1 = sdesc_lo(aDO1, L::kBox);
      const uint32_t mDS = sdesc_lo(aDS, L::kBox);
      auto dsc = [](uint32_t lo, uint32_t bytes) { return sdesc_join(lo + (bytes >> 4)); };
      uint32_t tile_it = 0, kt = 0, qit = 0, nblocks = 0;
      bool ok = true;
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
        const int nq = it.q_hi - it.q_lo;
        const int nqb = (nq + kBlockM - 1) / kBlockM;
        if (nqb == 0) continue;
        if (!wait_w(kv_full, kt & 1)) break;
        ++kt;
        // rows of a ragged tile past the item's KV or query range are other tokens of the
        // packed tensors: their weights are zero, but 0 x NaN is not, so they are zeroed
        // in shared memory before any product reads them (dO needs nothing: its per-item
        // maps end at the item, and TMA fills past the end with zeros)
        const int kvrows = (it.kv_hi - it.kv_lo) - tl.block * kBlockN;
        if (kvrows < kBlockN) {
          zero_tile_rows<D>(aK, kvrows, lane);
          zero_tile_rows<D>(aV, kvrows, lane);
          fence_proxy_async_smem();
          __syncwarp();
        }
        const int qstart = block_start<kOrdered>(tl.block, nqb);
        auto fix_q = [&](int is, uint32_t st) {
          const int qrows = nq - first_block(is, qstart, nqb) * kBlockM;
          if (qrows < kBlockM) {
            zero_tile_rows<D>(aQ + st * L::kTile, qrows, lane);
            fence_proxy_async_smem();
            __syncwarp();
          }
        };
        tc_fence_after();
        // S^T = K Q^T of the query block in slot st (TMEM R0)
        auto issue_s = [&](uint32_t st) {
          const uint32_t dq = kQ + ((st * L::kTile) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * L::kBox + (kk & 3) * 32;
            mma_ss_w(tR0, dsc(kK, off), dsc(dq, off), kIdSq, kk > 0);
          }
          mma_commit_w(s_full);
        };
        if (!wait_w(q_full + (qit & 1), (qit >> 1) & 1)) break;
        fix_q(0, qit & 1);
        tc_fence_after();
        issue_s(qit & 1);
        for (int is = 0; is < nqb; ++is) {
          const uint32_t st = qit & 1;
          const uint32_t dst = do_stage(qit);
          if (!wait_w(do_full_s(dst), do_phase(qit))) { ok = false; break; }
          const uint32_t kDOb = dst ? kDO1 : kDO, mDOb = dst ? mDO1 : mDO;
          if (nblocks > 0 && !wait_w(dq_empty, (nblocks - 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {  // dP^T = V dO^T
            const uint32_t off = (kk >> 2) * L::kBox + (kk & 3) * 32;
            mma_ss_w(tR1, dsc(kV, off), dsc(kDOb, off), kIdSq, kk > 0);
          }
          mma_commit_w(dp_full);
          // dV += P^T dO as soon as P^T is in TMEM (the warpgroup then forms dS^T)
          if (!wait_w(p_ready, nblocks & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // K = 128 queries
            mma_ts_w(tdV, tR0 + pcol(kk), dsc(mDOb, kk * 2048), kIdKV, (is > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(do_empty_s(dst));  // the producer may load a later block's dO into the stage
          if (is + 1 < nqb) {
            // S^T of the next block as soon as dV has read P^T out of R0 (one thread's
            // products run in issue order): the softmax warpgroups start on it while
            // this block's dK and dQ run
            const uint32_t st2 = (qit + 1) & 1, ph2 = ((qit + 1) >> 1) & 1;
            if (!wait_w(q_full + st2, ph2)) { ok = false; break; }
            fix_q(is + 1, st2);
            tc_fence_after();
            issue_s(st2);
          }
          if (!wait_w(ds_ready, nblocks & 1)) { ok = false; break; }
          tc_fence_after();
          // dQ first (R1 is free once the warpgroups have read dP^T): the drain warps start
          // on it while dK runs
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ = dS K   (K = 128 KV rows; both operands MN-major)
            mma_ss_w(tR1, dsc(mDS, kk * 2048), dsc(mK, kk * 2048), kIdDQ, kk > 0);
          mma_commit_w(dq_full);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // dK += dS^T Q   (dS^T read K-major from shared memory)
            const uint32_t off = (kk >> 2) * L::kBox + (kk & 3) * 32;
            mma_ss_w(tdK, dsc(kDS, off), dsc(mQ, st * L::kTile + kk * 2048), kIdKV,
                     (is > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit_w(q_empty + st);
          ++qit;
          ++nblocks;
        }
        if (!ok) break;
        mma_commit_w(kv_done);
        mma_commit_w(kv_empty);
      }
      mma_commit_w(drain);
      wait_w(drain, 0);
    }
   }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain warpgroup
    // Thread t owns query row t of the block (TMEM lane t); for head-dim column group g
    // (4 floats) the warp's 32 rows are 512 contiguous bytes of the tiled accumulator, and
    // a 32-column chunk of the block (8 groups x 128 rows) is 16 KB contiguous.
    regs_to<kRegsDrain>();
    constexpr int kChunks = D / 32;  // 32-column TMEM loads per row
    constexpr bool kBulk = !kOrdered;
    const int t = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t aStage = smem_u32(smem + L::kStage);
    uint32_t tile_it = 0, nblocks = 0, sit = 0;  // sit: chunks staged so far
    for (;;) {
      const uint32_t slot = tile_it & 1;
      if (!__all_sync(0xffffffffu, bwait(tile_full + slot, (tile_it >> 1) & 1, abort_flag, p.wait_limit, p.status))) break;
      const int tid = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(tile_empty + slot);
      ++tile_it;
      if (tid < 0) break;
      const DevTile tl = p.tiles[tid];
      const DevItem it = p.items[tl.item];
      const int nq = it.q_hi - it.q_lo;
      const int nqb = (nq + kBlockM - 1) / kBlockM;
      float* acc_hd = p.ws_dq + it.ws_dq_offset + (int64_t)(tl.head - it.h_lo) * nqb * (kBlockM * D);
      float* acc = acc_hd + t * 4;
      // ordered adds: this warp's 32-row slice of accumulator block ib has turn counter
      // turns[4 (block) + warp slice]; KV tile b adds when the counter reads b.  A
      // block's turn is passed on at the next block (or the end of the tile), after a
      // fence that by then mostly finds its reductions complete.
      auto turn_of = [&](int ib) {
        return p.turns + 4 * ((acc + (int64_t)ib * (kBlockM * D) - p.ws_dq) / (kBlockM * D)) + (warp & 3);
      };
      auto pass_turn = [&](int ib) {
        fence_acq_rel_gpu();  // this lane's reductions come before the release below
        __syncwarp();
        if (lane == 0) st_release_gpu(turn_of(ib), tl.block + 1);
      };
      int pending = -1;  // block whose turn this warp still holds
      const int start = block_start<kOrdered>(tl.block, nqb);
      bool ok = true;
      for (int is = 0; is < nqb; ++is) {
        const int ib = first_block(is, start, nqb);
        if (!__all_sync(0xffffffffu, bwait(dq_full, nblocks & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
        tc_fence_after();
        float* dst = acc + (int64_t)ib * (kBlockM * D);
        const bool row_ok = ib * kBlockM + t < nq;  // rows past the item hold dS = 0
        // all of the row first: TMEM R1 is released before any reduction is issued
        uint32_t u[kChunks][32];
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tmem_ld32(tmem + lane_base + 128 + 32 * c, u[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(dq_empty);  // the next block's dP^T may overwrite R1
        if constexpr (kBulk) {
          // chunk c (columns 32c..32c+31) of block ib is 16 KB contiguous in the tiled
          // accumulator, [8 column groups][128 rows][4]: each thread writes its row's 8
          // groups into a staging buffer of the same layout, and one thread issues the
          // chunk's bulk reduce-add once all 128 rows are in; a buffer is refilled once
          // the engine has read it (two buffers, so one chunk is staged while the
          // previous one is read)
          float* blk = acc_hd + (int64_t)ib * (kBlockM * D);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const uint32_t b = sit & 1, use = sit >> 1;
            if (!__all_sync(0xffffffffu, bwait(stage_free + b, (use & 1) ^ 1, abort_flag, p.wait_limit, p.status))) {
              ok = false;
              break;
            }
            const uint32_t sb = aStage + b * L::kStageBytes;
#pragma unroll
            for (int g = 0; g < 8; ++g)
              st_shared_v4(sb + (g * kBlockM + t) * 16, u[c][4 * g], u[c][4 * g + 1], u[c][4 * g + 2], u[c][4 * g + 3]);
            fence_proxy_async_smem();
            mbar_arrive(stage_full + b);
            if (warp == 8 && lane == 0 && bwait(stage_full + b, use & 1, abort_flag, p.wait_limit, p.status)) {
              bulk_reduce_add_f32(blk + c * (32 * kBlockM), sb, L::kStageBytes);
              bulk_commit();
              bulk_wait_read_1();  // the other buffer's reduce-add has read it
              if (sit > 0) mbar_arrive(stage_free + (b ^ 1));
            }
            ++sit;
          }
          if (!ok) break;
          ++nblocks;
          continue;
        }
        if constexpr (kOrdered) {
          if (pending >= 0) pass_turn(pending);
          bool mine = true;
          if (lane == 0) mine = wait_turn(turn_of(ib), tl.block, abort_flag, p.wait_limit, p.status);
          __syncwarp();  // the other lanes' reductions follow lane 0's acquire
          if (!__shfl_sync(0xffffffffu, mine ? 1 : 0, 0)) { ok = false; break; }
          pending = ib;
        }
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
#pragma unroll
            for (int g = 0; g < 8; ++g)
              red_add_v4(dst + (8 * c + g) * (4 * kBlockM), u[c][4 * g], u[c][4 * g + 1], u[c][4 * g + 2],
                         u[c][4 * g + 3]);
        }
        ++nblocks;
      }
      if (!ok) break;
      if constexpr (kOrdered) {
        if (pending >= 0) pass_turn(pending);
      }
    }
    // the bulk reduce-adds this thread issued are complete before the kernel ends
    if (kBulk && warp == 8 && lane == 0) bulk_wait_all();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    // Two warpgroups share the TMEM lanes (lane = KV row) and split the columns:
    // warpgroup wg takes queries [64wg, 64wg+64) of S^T and dP^T and head-dim columns
    // [wg d/2, (wg+1) d/2) of dK and dV.
    regs_to<kRegsSoftmax>();
    constexpr int kHalfD = D / 2;
    const int wg = warp >> 2;
    const int t = threadIdx.x & 127;  // KV row of the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int qc0 = 64 * wg;          // this warpgroup's query columns
    const int dc0 = kHalfD * wg;      // this warpgroup's head-dim columns
    const float sl2 = p.scale_log2;
    const uint32_t aDSrow = smem_u32(sDS) + wg * L::kBox + t * 128;  // row t of box wg
    uint32_t tile_it = 0, nblocks = 0, ntiles = 0;
    for (;;) {
      const uint32_t slot = tile_it & 1;
      if (!__all_sync(0xffffffffu, bwait(tile_full + slot, (tile_it >> 1) & 1, abort_flag, p.wait_limit, p.status))) break;
      const int tid = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(tile_empty + slot);
      ++tile_it;
      if (tid < 0) break;
      const DevTile tl = p.tiles[tid];
      const DevItem it = p.items[tl.item];
      const int nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo;
      const int nkv = it.kv_hi - it.kv_lo;
      const int nqb = (nq + kBlockM - 1) / kBlockM;
      const int hl = tl.head - it.h_lo;
      const int kv_local = tl.block * kBlockN + t;
      const bool kv_ok = kv_local < nkv;
      const float* lse_row = p.lse + it.fin_lse_offset + (int64_t)hl * nq;
      const float* d_row = p.ws_d + it.ws_d_offset + (int64_t)hl * nq;
      bool ok = true;
      float lse_n = -kInfB, d_n = 0.f;  // warpgroup 0 stages -LSE*log2(e) and -D of query t of each block
      const int ib0 = block_start<kOrdered>(tl.block, nqb);
      if (wg == 0 && nqb > 0 && ib0 * kBlockM + t < nq) {
        lse_n = -__ldg(lse_row + ib0 * kBlockM + t) * kLog2eB;
        d_n = -__ldg(d_row + ib0 * kBlockM + t);
      }
      for (int is = 0; is < nqb; ++is) {
        // publish this block's LSE / D, prefetch the next block's
        if (wg == 0) {
          sLD[256 * (nblocks & 1) + t] = lse_n;
          sLD[256 * (nblocks & 1) + 128 + t] = d_n;
        }
        mbar_arrive(ld_full);  // bounded stand-in for a barrier of both warpgroups
        if (!__all_sync(0xffffffffu, bwait(ld_full, nblocks & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
        if (wg == 0) {
          const int qn = first_block(is + 1, ib0, nqb) * kBlockM + t;
          lse_n = -kInfB; d_n = 0.f;
          if (is + 1 < nqb && qn < nq) { lse_n = -__ldg(lse_row + qn) * kLog2eB; d_n = -__ldg(d_row + qn); }
        }

        // the warpgroups meet only at ld_full, so warpgroup 0 may stage the next block's
        // LSE / D while warpgroup 1 still reads this block's: one buffer per block parity
        // (warpgroup 0 cannot get two blocks ahead: ld_full needs both)
        const float* sLSE = sLD + 256 * (nblocks & 1);
        const float* sD = sLSE + 128;
        if (!__all_sync(0xffffffffu, bwait(s_full, nblocks & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
        tc_fence_after();
        float pr[64];
        {
          uint32_t u0[32], u1[32];
          tmem_ld32(tmem + lane_base + qc0, u0);
          tmem_ld32(tmem + lane_base + qc0 + 32, u1);
          tmem_ld_wait();
          // exponent arguments two queries per instruction (the staged LSE is negated)
          const float2 sl2v = make_float2(sl2, sl2);
          const float2* nl2 = reinterpret_cast<const float2*>(sLSE + qc0);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x0 = fma2(make_float2(__uint_as_float(u0[2 * e]), __uint_as_float(u0[2 * e + 1])), sl2v, nl2[e]);
            const float2 x1 =
                fma2(make_float2(__uint_as_float(u1[2 * e]), __uint_as_float(u1[2 * e + 1])), sl2v, nl2[16 + e]);
            pr[2 * e] = kv_ok ? ex2(x0.x) : 0.f;
            pr[2 * e + 1] = kv_ok ? ex2(x0.y) : 0.f;
            pr[32 + 2 * e] = kv_ok ? ex2(x1.x) : 0.f;
            pr[32 + 2 * e + 1] = kv_ok ? ex2(x1.y) : 0.f;
          }
        }
        // P^T (bf16) over this warpgroup's S^T columns, already read: dV may start now
        {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) pk[e] = pack_bf16(pr[2 * e], pr[2 * e + 1]);
          tmem_st32(tmem + lane_base + qc0, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_ready);

        // dP^T of this block is issued after the previous block's dQ product, which read
        // the dS^T buffer: once dP^T is complete the buffer may be rewritten
        if (!__all_sync(0xffffffffu, bwait(dp_full, nblocks & 1, abort_flag, p.wait_limit, p.status))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_base + 128 + qc0 + 32 * c, u);
          tmem_ld_wait();
          uint32_t pk[16];
          // dS = P (dP - D), two queries per instruction (the staged D is negated)
          const float2* nd2 = reinterpret_cast<const float2*>(sD + qc0 + 32 * c);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 ds = mul2(add2(make_float2(__uint_as_float(u[2 * e]), __uint_as_float(u[2 * e + 1])), nd2[e]),
                                   make_float2(pr[32 * c + 2 * e], pr[32 * c + 2 * e + 1]));
            pk[e] = pack_bf16(ds.x, ds.y);
          }
          // dS^T row t -> box wg of shared memory, 128-byte swizzle: 16-byte chunk 4c+g
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const int chunk = 4 * c + g;
            st_shared_v4(aDSrow + ((chunk ^ (t & 7)) << 4), pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();  // the dP^T loads are complete: dQ may overwrite R1
        mbar_arrive(ds_ready);

        ++nblocks;
      }
      if (!ok) break;
      // ---- dK, dV of this tile's KV rows (this warpgroup's head-dim columns)
      if (nqb > 0) {
        if (!__all_sync(0xffffffffu, bwait(kv_done, ntiles & 1, abort_flag, p.wait_limit, p.status))) break;
        ++ntiles;
        tc_fence_after();
      }
      const int64_t row_off = it.dkv_offset + (int64_t)kv_local * nh * D + (int64_t)hl * D + dc0;
#pragma unroll
      for (int c = 0; c < kHalfD / 32; ++c) {
        uint32_t uv[32], uk[32];
        if (nqb > 0) {
          tmem_ld32(tmem + lane_base + 256 + dc0 + 32 * c, uv);
          tmem_ld32(tmem + lane_base + 384 + dc0 + 32 * c, uk);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) uv[e] = uk[e] = 0u;
        }
        if (kv_ok) {
          float4* dv4 = reinterpret_cast<float4*>(p.dv + row_off + 32 * c);
          float4* dk4 = reinterpret_cast<float4*>(p.dk + row_off + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4) {
            dv4[v4] = make_float4(__uint_as_float(uv[4 * v4]), __uint_as_float(uv[4 * v4 + 1]),
                                  __uint_as_float(uv[4 * v4 + 2]), __uint_as_float(uv[4 * v4 + 3]));
            dk4[v4] = make_float4(__uint_as_float(uk[4 * v4]) * p.scale, __uint_as_float(uk[4 * v4 + 1]) * p.scale,
                                  __uint_as_float(uk[4 * v4 + 2]) * p.scale, __uint_as_float(uk[4 * v4 + 3]) * p.scale);
          }
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const BwdParams& p, int num_sms, cudaStream_t stream) {
  const int smem = head_dim == 128 ? BwdLayout<128>::kBytes : BwdLayout<64>::kBytes;
  const int smem_launch = smem > 120 * 1024 ? smem : 120 * 1024;
  using Kernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const BwdParams);
  const bool ordered = p.turns != nullptr;  // ordered (deterministic) dQ adds
  const Kernel k = head_dim == 128 ? (ordered ? zl_bwd_kernel<128, true> : zl_bwd_kernel<128, false>)
                                   : (ordered ? zl_bwd_kernel<64, true> : zl_bwd_kernel<64, false>);
  static PerDeviceOnce configured[2][2];
  const int di = head_dim == 128 ? 1 : 0, oi = ordered ? 1 : 0;
  cudaError_t e = configured[di][oi].run([&] {
    cudaError_t r = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_launch);
    if (r != cudaSuccess) return r;
    // the register split adds up to exactly the launch allocation: a kernel built with
    // another per-thread count would leave an increase waiting for registers forever
    cudaFuncAttributes fa;
    r = cudaFuncGetAttributes(&fa, k);
    if (r != cudaSuccess) return r;
    return fa.numRegs == (int)kRegsLaunch ? cudaSuccess : cudaErrorInvalidKernelImage;
  });
  if (e != cudaSuccess) return e;
  const int grid = p.n_tiles < num_sms ? p.n_tiles : num_sms;
  if (grid == 0) return cudaSuccess;
  e = cudaMemsetAsync(p.counter, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  k<<<grid, 512, smem_launch, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace zl
