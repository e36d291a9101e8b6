// C-ABI entry points: argument checks, TMA tensor maps, kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "zl_internal.h"
#include "zl_kernels.h"

using namespace zl;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// [T, H, d] bf16, tiles of 128 tokens x 64 head-dim elements (one 128-byte swizzle
// span); coordinates are (d offset, head, token).
bool make_qkv_map(CUtensorMap* m, const void* base, int64_t T, int32_t H, int32_t d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One [rows, H, d] block of the `o` arena (same tiling as the Q/K/V maps).
bool make_block_map(CUtensorMap* m, const void* base, int64_t rows, int32_t H, int32_t d) {
  return make_qkv_map(m, base, rows, H, d);
}

// A plan that can be launched, with the device it was built on current: its tile lists,
// counters and status word live in that device's memory.
bool launchable(const zl_plan* p) {
  if (!p || p->host_only || !p->d_items) return false;
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == p->device;
}

// Spin budget of a bounded device wait: ~0.5 s at 2 GHz; short for the test hook.
long long wait_limit(const zl_plan* p) { return p->test_withhold ? 20000000LL : 1000000000LL; }

}  // namespace

extern "C" zl_status zl_coalesced_attn_fwd(const zl_plan* p, const void* q, const void* k, const void* v, void* o,
                                           float* o_partial, float* lse, float scale, void* stream) {
  NvtxRange range("zl_coalesced_attn_fwd");
  if (!launchable(p) || !q || !k || !v || !lse) return ZL_ERR_INVALID_ARG;
  if ((p->fwd_writes_o && !o) || (p->fwd_writes_partial && !o_partial)) return ZL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(o_partial) ||
      !aligned16(lse))
    return ZL_ERR_ALIGN;
  if (p->fwd_tiles.empty()) return ZL_OK;
  CUtensorMap tq, tk, tv;
  if (!make_qkv_map(&tq, q, p->total_tokens, p->n_heads, p->head_dim) ||
      !make_qkv_map(&tk, k, p->total_tokens, p->n_heads, p->head_dim) ||
      !make_qkv_map(&tv, v, p->total_tokens, p->n_heads, p->head_dim))
    return ZL_ERR_CUDA;
  FwdParams fp;
  fp.items = p->d_items;
  fp.tiles = p->d_fwd_tiles;
  fp.n_tiles = (int32_t)p->fwd_tiles.size();
  fp.counter = p->d_counters + kCtrFwd;
  fp.status = p->d_counters + kStatus;
  fp.wait_limit = wait_limit(p);
  fp.withhold_load = p->test_withhold ? 1 : 0;
  fp.o = static_cast<__nv_bfloat16*>(o);
  fp.o_partial = o_partial;
  fp.lse = lse;
  fp.scale_log2 = scale * 1.44269504088896340736f;
  cudaError_t e = launch_fwd2(p->head_dim, tq, tk, tv, fp, p->num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

extern "C" zl_status zl_merge_partials(const zl_plan* p, const float* o_partial, const float* lse_partial, void* o,
                                       float* lse_out, void* stream) {
  NvtxRange range("zl_merge_partials");
  if (!launchable(p)) return ZL_ERR_INVALID_ARG;
  if (p->merge_groups.empty()) return ZL_OK;  // none, or all fused into the forward
  if (!o_partial || !lse_partial || !o || !lse_out) return ZL_ERR_INVALID_ARG;
  if (!aligned16(o_partial) || !aligned16(lse_partial) || !aligned16(o) || !aligned16(lse_out)) return ZL_ERR_ALIGN;
  int32_t max_members = 0;
  for (const DevGroup& G : p->merge_groups) max_members = G.n_members > max_members ? G.n_members : max_members;
  cudaError_t e = launch_merge(p->head_dim, p->d_groups, (int32_t)p->merge_groups.size(), p->d_members,
                               p->merge_rowheads, max_members, o_partial, lse_partial,
                               static_cast<__nv_bfloat16*>(o), lse_out, p->num_sms,
                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

extern "C" zl_status zl_bwd_preprocess(const zl_plan* p, const void* o, const void* d_o, void* workspace,
                                       void* stream) {
  NvtxRange range("zl_bwd_preprocess");
  if (!launchable(p) || !o || !d_o || (p->workspace_bytes > 0 && !workspace)) return ZL_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(d_o) || !aligned16(workspace)) return ZL_ERR_ALIGN;
  if (p->items.empty()) return ZL_OK;
  float* ws_d = static_cast<float*>(workspace);
  cudaError_t e = launch_bwd_pre(p->head_dim, p->d_items, p->n_user, p->total_rowheads,
                                 static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(d_o), ws_d,
                                 ws_d + p->ws_d_floats, p->ws_dq_floats + p->ws_turn_ints, p->num_sms,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

extern "C" zl_status zl_bwd_main(const zl_plan* p, const void* q, const void* k, const void* v, const void* d_o,
                                 const float* lse, float* dk, float* dv, void* workspace, float scale, void* stream) {
  NvtxRange range("zl_bwd_main");
  if (!launchable(p) || !q || !k || !v || !d_o || !lse || !dk || !dv || (p->workspace_bytes > 0 && !workspace))
    return ZL_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(d_o) || !aligned16(lse) || !aligned16(dk) ||
      !aligned16(dv) || !aligned16(workspace))
    return ZL_ERR_ALIGN;
  if (p->bwd_tiles.empty()) return ZL_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  if (!make_qkv_map(&tq, q, p->total_tokens, p->n_heads, p->head_dim) ||
      !make_qkv_map(&tk, k, p->total_tokens, p->n_heads, p->head_dim) ||
      !make_qkv_map(&tv, v, p->total_tokens, p->n_heads, p->head_dim))
    return ZL_ERR_CUDA;
  // Per item: its dO (final block in the `o` arena, [|q|, |h|, d] with row stride |h| d)
  // for TMA loads.
  zl_plan* mp = const_cast<zl_plan*>(p);
  float* ws_d = static_cast<float*>(workspace);
  for (int32_t i = 0; i < p->n_user; ++i) {
    const DevItem& it = p->items[i];
    const int64_t nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo;
    if (nq == 0 || nh == 0) continue;
    const void* base = static_cast<const __nv_bfloat16*>(d_o) + it.fin_out_offset;
    if (!make_block_map(&mp->h_do_maps[i], base, nq, (int32_t)nh, p->head_dim)) return ZL_ERR_CUDA;
  }
  if (cudaMemcpyAsync(p->d_do_maps, p->h_do_maps.data(), sizeof(CUtensorMap) * p->n_user,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return ZL_ERR_CUDA;
  BwdParams bp;
  bp.items = p->d_items;
  bp.tiles = p->d_bwd_tiles;
  bp.n_tiles = (int32_t)p->bwd_tiles.size();
  bp.counter = p->d_counters + kCtrBwd;
  bp.status = p->d_counters + kStatus;
  bp.wait_limit = wait_limit(p);
  bp.withhold_load = p->test_withhold ? 1 : 0;
  bp.lse = lse;
  bp.ws_d = ws_d;
  bp.ws_dq = ws_d + p->ws_d_floats;
  bp.turns = p->det_dq ? reinterpret_cast<int32_t*>(bp.ws_dq + p->ws_dq_floats) : nullptr;
  bp.dk = dk;
  bp.dv = dv;
  bp.scale = scale;
  bp.scale_log2 = scale * 1.44269504088896340736f;
  bp.do_maps = p->d_do_maps;
  cudaError_t e = launch_bwd(p->head_dim, tq, tk, tv, bp, p->num_sms, st);
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

extern "C" zl_status zl_bwd_finalize(const zl_plan* p, float* dq, void* workspace, float scale, void* stream) {
  NvtxRange range("zl_bwd_finalize");
  if (!launchable(p) || !dq || (p->workspace_bytes > 0 && !workspace)) return ZL_ERR_INVALID_ARG;
  if (!aligned16(dq) || !aligned16(workspace)) return ZL_ERR_ALIGN;
  if (p->items.empty()) return ZL_OK;
  const float* ws_dq = static_cast<const float*>(workspace) + p->ws_d_floats;
  cudaError_t e = launch_dq_finalize(p->head_dim, p->d_items, p->n_user, p->ws_dq_floats, ws_dq, dq, scale,
                                     p->num_sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

extern "C" zl_status zl_coalesced_attn_bwd(const zl_plan* p, const void* q, const void* k, const void* v,
                                           const void* o, const void* d_o, const float* lse, float* dq, float* dk,
                                           float* dv, void* workspace, float scale, void* stream) {
  NvtxRange range("zl_coalesced_attn_bwd");
  if (!launchable(p) || !q || !k || !v || !o || !d_o || !lse || !dq || !dk || !dv ||
      (p->workspace_bytes > 0 && !workspace))
    return ZL_ERR_INVALID_ARG;
  zl_status s = zl_bwd_preprocess(p, o, d_o, workspace, stream);
  if (s == ZL_OK) s = zl_bwd_main(p, q, k, v, d_o, lse, dk, dv, workspace, scale, stream);
  if (s == ZL_OK) s = zl_bwd_finalize(p, dq, workspace, scale, stream);
  return s;
}

extern "C" zl_status zl_get_device_status(const zl_plan* p, void* stream, int32_t* device_status) {
  if (!launchable(p) || !device_status) return ZL_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, p->d_counters + kStatus, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemsetAsync(p->d_counters + kStatus, 0, sizeof(int32_t), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return ZL_ERR_CUDA;
  *device_status = v;
  return ZL_OK;
}

extern "C" const char* zl_status_string(zl_status s) {
  switch (s) {
    case ZL_OK: return "ok";
    case ZL_ERR_INVALID_ARG: return "invalid argument";
    case ZL_ERR_ALIGN: return "pointer or offset not 16-byte aligned";
    case ZL_ERR_CUDA: return "CUDA error";
    case ZL_ERR_TIMEOUT: return "bounded device wait timed out";
    case ZL_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case ZL_ERR_NO_MEMORY: return "out of memory";
  }
  return "unknown status";
}

extern "C" int32_t zl_version(void) { return 100; }
