// Launch interfaces of the kernels (host side).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "zl_internal.h"

namespace zl {

struct FwdParams {
  const DevItem* items;
  const DevTile* tiles;
  int32_t n_tiles;
  int32_t* counter;
  int32_t* status;
  long long wait_limit;   // cycles a bounded wait may spin
  int32_t withhold_load;  // test hook: announce but never issue the first K load
  __nv_bfloat16* o;
  float* o_partial;
  float* lse;
  float scale_log2;
};

struct BwdParams {
  const DevItem* items;
  const DevTile* tiles;
  int32_t n_tiles;
  int32_t* counter;
  int32_t* status;
  long long wait_limit;
  int32_t withhold_load;  // test hook: announce but never issue the first K/V load
  const float* lse;   // final LSE arena
  const float* ws_d;  // row sums D (workspace)
  float* ws_dq;       // fp32 dQ accumulator (workspace, tiled as acc_index)
  int32_t* turns;     // deterministic dQ: turn counter per (query block, warp slice); null otherwise
  float* dk;
  float* dv;
  const CUtensorMap* do_maps;  // one per item: its final dO block as [|q|, |h|, d] (device memory)
  float scale;
  float scale_log2;
};

cudaError_t launch_fwd2(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const FwdParams& p, int num_sms, cudaStream_t stream);

// max_members: the largest member count of the groups (selects the kernel instance)
cudaError_t launch_merge(int head_dim, const DevGroup* groups, int32_t n_groups, const DevMember* members,
                         int64_t total_rowheads, int32_t max_members, const float* o_partial,
                         const float* lse_partial, __nv_bfloat16* o, float* lse_out, int num_sms,
                         cudaStream_t stream);

cudaError_t launch_bwd_pre(int head_dim, const DevItem* items, int32_t n_items, int64_t total_rowheads,
                           const __nv_bfloat16* o, const __nv_bfloat16* d_o, float* ws_d, float* ws_dq,
                           int64_t acc_total, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const BwdParams& p, int num_sms, cudaStream_t stream);

// acc_floats_total: floats of the whole dQ accumulator (every item's, in item order)
cudaError_t launch_dq_finalize(int head_dim, const DevItem* items, int32_t n_items, int64_t acc_floats_total,
                               const float* ws_dq, float* dq, float scale, int num_sms, cudaStream_t stream);

}  // namespace zl
