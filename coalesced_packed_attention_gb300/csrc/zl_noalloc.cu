// Forward launch that allocates no device memory.
//
// Callers that cannot call cudaMalloc — code running where a device allocator is not
// available or not allowed (a pre-reserved memory pool, a host framework that owns all
// device memory, an embedding that forbids allocation after start-up) — cannot create a
// zl_plan, because a plan uploads its item table, tile list and scheduler counter to
// memory the library allocates.  zl_coalesced_attn_fwd_noalloc takes the work list
// directly, builds the tables on the host and copies them into a fixed scratch area
// compiled into the library (g_zl_noalloc_scratch below), then launches the same
// forward kernel as zl_coalesced_attn_fwd.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "zl_internal.h"
#include "zl_kernels.h"

using namespace zl;

namespace {

// Scratch for the item table, the tile list, the scheduler counter and the status word.
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr size_t kCounterBytes = 256;                     // counter + status word, zeroed per call
// The capacity stated in zl.h (bytes per item and per forward tile) follows these sizes.
static_assert(sizeof(DevItem) == 112 && sizeof(DevTile) == 16, "update the capacity stated in zl.h");

static __device__ __align__(256) unsigned char g_zl_noalloc_scratch[kNoAllocScratchBytes];

struct ScratchSlot {
  void* base = nullptr;  // device address of g_zl_noalloc_scratch on that device
  int num_sms = 0;
  bool ready = false;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
ScratchSlot g_slots[kMaxDevices];

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Once per device, with that device current: the array's device address.  In host
// code g_zl_noalloc_scratch names a host-side stand-in, never a device address.
zl_status scratch_for_current_device(ScratchSlot** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZL_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ZL_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot& s = g_slots[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ZL_ERR_CUDA;
    if (major != 10 || minor != 3) return ZL_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_zl_noalloc_scratch) != cudaSuccess || p == nullptr) return ZL_ERR_CUDA;
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ZL_ERR_CUDA;
    s.base = p;
    s.ready = true;
  }
  *out = &s;
  return ZL_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_noalloc() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool qkv_map(CUtensorMap* m, const void* base, int64_t T, int32_t H, int32_t d) {
  auto fn = encode_fn_noalloc();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" zl_status zl_coalesced_attn_fwd_noalloc(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                                                   int32_t head_dim, int64_t total_tokens, const void* q,
                                                   const void* k, const void* v, void* o, float* o_partial,
                                                   float* lse, float scale, void* stream) {
  if (!q || !k || !v || !lse) return ZL_ERR_INVALID_ARG;
  if (!al16(q) || !al16(k) || !al16(v) || !al16(o) || !al16(o_partial) || !al16(lse)) return ZL_ERR_ALIGN;
  // host tables only: the planner allocates no device memory for a host-only plan
  zl_plan* plan = nullptr;
  zl_status s = zl_plan_worklist(items, n_items, n_heads, head_dim, total_tokens, ZL_PLAN_HOST_ONLY, &plan);
  if (s != ZL_OK) return s;
  bool any_whole = false, any_emit = false;
  for (const auto& it : plan->items) (it.emit_lse ? any_emit : any_whole) = true;
  const size_t item_bytes = align256(sizeof(DevItem) * plan->items.size());
  const size_t tile_bytes = align256(sizeof(DevTile) * plan->fwd_tiles.size());
  if ((any_whole && !o) || (any_emit && !o_partial)) s = ZL_ERR_INVALID_ARG;
  else if (kCounterBytes + item_bytes + tile_bytes > kNoAllocScratchBytes) s = ZL_ERR_INVALID_ARG;  // too large
  ScratchSlot* slot = nullptr;
  if (s == ZL_OK) s = scratch_for_current_device(&slot);
  if (s == ZL_OK && !plan->fwd_tiles.empty()) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* base = static_cast<unsigned char*>(slot->base);
    int32_t* counters = reinterpret_cast<int32_t*>(base);
    DevItem* d_items = reinterpret_cast<DevItem*>(base + kCounterBytes);
    DevTile* d_tiles = reinterpret_cast<DevTile*>(base + kCounterBytes + item_bytes);
    CUtensorMap tq, tk, tv;
    // pageable host sources: each copy is staged before cudaMemcpyAsync returns, so the
    // host tables may be freed right after
    if (cudaMemsetAsync(counters, 0, kCounterBytes, st) != cudaSuccess ||
        cudaMemcpyAsync(d_items, plan->items.data(), sizeof(DevItem) * plan->items.size(), cudaMemcpyHostToDevice,
                        st) != cudaSuccess ||
        cudaMemcpyAsync(d_tiles, plan->fwd_tiles.data(), sizeof(DevTile) * plan->fwd_tiles.size(),
                        cudaMemcpyHostToDevice, st) != cudaSuccess) {
      s = ZL_ERR_CUDA;
    } else if (!qkv_map(&tq, q, total_tokens, n_heads, head_dim) || !qkv_map(&tk, k, total_tokens, n_heads, head_dim) ||
               !qkv_map(&tv, v, total_tokens, n_heads, head_dim)) {
      s = ZL_ERR_CUDA;
    } else {
      FwdParams fp;
      fp.items = d_items;
      fp.tiles = d_tiles;
      fp.n_tiles = (int32_t)plan->fwd_tiles.size();
      fp.counter = counters + kCtrFwd;
      fp.status = counters + kStatus;
      fp.wait_limit = 1000000000LL;
      fp.withhold_load = 0;
      fp.o = static_cast<__nv_bfloat16*>(o);
      fp.o_partial = o_partial;
      fp.lse = lse;
      fp.scale_log2 = scale * 1.44269504088896340736f;
      if (launch_fwd2(head_dim, tq, tk, tv, fp, slot->num_sms, st) != cudaSuccess) s = ZL_ERR_CUDA;
    }
  }
  zl_plan_destroy(plan);  // host-only plan: frees host memory, no device call
  return s;
}

extern "C" zl_status zl_noalloc_get_device_status(void* stream, int32_t* device_status) {
  if (!device_status) return ZL_ERR_INVALID_ARG;
  ScratchSlot* slot = nullptr;
  zl_status s = scratch_for_current_device(&slot);
  if (s != ZL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* word = reinterpret_cast<int32_t*>(slot->base) + kStatus;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess ||
      cudaMemsetAsync(word, 0, sizeof(int32_t), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
    return ZL_ERR_CUDA;
  *device_status = v;
  return ZL_OK;
}
