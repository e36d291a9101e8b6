// Internal tables shared by the host planner and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <vector>

#include "../../include/zl.h"

namespace zl {

constexpr int kBlockM = 128;   // query rows per forward tile / per backward q-step
constexpr int kBlockN = 128;   // KV rows per forward step / per backward tile
constexpr int kFwdBlockM = 256;  // query rows per forward tile of the two-sub-tile kernel

// fp32 dQ accumulator of one item, tiled by backward query block so that one warp's
// 16-byte vector reduction of 32 consecutive rows covers 512 contiguous bytes:
//   acc[hl][qb][c / 4][r][c % 4]   for query q = qb * kBlockM + r, head-dim column c.
// The last query block is padded to kBlockM rows (padding rows are never read).
__host__ __device__ inline int64_t acc_floats(int64_t nq, int64_t nh, int64_t d) {
  return nh * ((nq + kBlockM - 1) / kBlockM) * kBlockM * d;
}
__host__ __device__ inline int64_t acc_index(int64_t q, int64_t hl, int64_t c, int64_t nq, int64_t d) {
  const int64_t nqb = (nq + kBlockM - 1) / kBlockM;
  return ((hl * nqb + q / kBlockM) * (d / 4) + c / 4) * (4 * kBlockM) + (q % kBlockM) * 4 + (c & 3);
}

// Resolved work item as the kernels read it (device copy of the planner's table).
struct DevItem {
  int64_t seq_offset;
  int32_t seq_len, q_lo, q_hi, h_lo, h_hi, kv_lo, kv_hi, emit_lse;
  int64_t out_offset;      // own O block: `o` (bf16) or `o_partial` (fp32)
  int64_t lse_offset;      // own LSE block in `lse`
  int64_t fin_out_offset;  // final O / dO block in `o` (group's block for k-split items)
  int64_t fin_lse_offset;  // final LSE block in `lse`
  int64_t dq_offset;       // [|q|,|h|,d] block in dq
  int64_t dkv_offset;      // [|kv|,|h|,d] block in dk and dv
  int64_t ws_d_offset;     // row sums D, [|h|,|q|] floats in the workspace
  int64_t ws_dq_offset;    // fp32 dQ accumulator (q-block tiled, see acc_floats) from the accumulator base
                           // (which is ws_d_floats floats into the workspace)
  int64_t rowhead_begin;   // prefix of |q|*|h| over items (row-parallel kernels)
};

struct DevTile {           // one scheduler unit
  int32_t item, head, block, cost;
};

struct DevGroup {          // one k-split merge group
  int32_t member_begin, n_members, nq, nh;
  int64_t out_offset;      // merged O block in `o`
  int64_t lse_offset;      // merged LSE block in `lse`
  int64_t rowhead_begin;   // prefix of nq*nh over groups
};

struct DevMember {         // one partial of a merge group
  int64_t o_offset;        // [nq, nh, d] block in o_partial
  int64_t lse_offset;      // [nh, nq] block in lse_partial
};

// Named NVTX range over one ABI call (host side: it covers validation and the enqueue of
// the launches), so timelines and ncu's NVTX filters can find each call.  A no-op
// unless a profiling tool is attached.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Once-per-device setup of a kernel's launch attributes.  cudaFuncSetAttribute acts on
// the current device, so a process that drives several GPUs must set them on each; two
// host threads may both run the setup, which is harmless (it is idempotent).
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return setup();  // outside the mask: set up every time
    const uint64_t bit = 1ull << dev;
    if (done_.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }

 private:
  std::atomic<uint64_t> done_{0};
};

// Scheduler counters and the status word live in one small device block.
enum CounterSlot { kCtrFwd = 0, kCtrBwd = 1, kStatus = 2, kNumCounters = 8 };

}  // namespace zl

struct zl_plan {
  int32_t n_heads = 0, head_dim = 0;
  int64_t total_tokens = 0;
  int device = -1;
  int num_sms = 0;
  bool host_only = false;
  bool test_withhold = false;   // ZL_PLAN_TEST_WITHHOLD_LOAD

  std::vector<zl::DevItem> items;
  std::vector<zl_work_item> resolved;
  std::vector<int32_t> item_group;
  std::vector<zl::DevTile> fwd_tiles, bwd_tiles;
  std::vector<zl::DevGroup> groups;        // every merge group (queries)
  std::vector<zl::DevGroup> merge_groups;  // the groups the merge launch combines (unfused)
  std::vector<uint8_t> group_fused;        // per group: computed as one forward item
  std::vector<zl::DevMember> members;
  std::vector<int32_t> member_items;

  int64_t o_elems = 0, o_partial_elems = 0, lse_elems = 0, dq_elems = 0, dkv_elems = 0;
  int64_t ws_d_floats = 0, ws_dq_floats = 0, workspace_bytes = 0;
  int64_t ws_turn_ints = 0;  // dQ turn counters after the accumulator (ZL_PLAN_DETERMINISTIC_DQ)
  int64_t total_rowheads = 0, group_rowheads = 0, merge_rowheads = 0;
  int32_t n_user = 0;        // work-list items; items[n_user..] are fused forward items
  bool fuse_kmerge = false;  // ZL_PLAN_FUSE_LOCAL_KMERGE
  bool det_dq = false;       // ZL_PLAN_DETERMINISTIC_DQ
  bool fwd_writes_o = false, fwd_writes_partial = false;  // some forward tile writes o / o_partial

  // device copies (one allocation, carved)
  void* dev_blob = nullptr;
  zl::DevItem* d_items = nullptr;
  zl::DevTile* d_fwd_tiles = nullptr;
  zl::DevTile* d_bwd_tiles = nullptr;
  zl::DevGroup* d_groups = nullptr;
  zl::DevMember* d_members = nullptr;
  int32_t* d_counters = nullptr;
  CUtensorMap* d_do_maps = nullptr;          // 1 per item (its final dO block),
                                             // rewritten by every backward call
  std::vector<CUtensorMap> h_do_maps;        // host staging of the same
};
