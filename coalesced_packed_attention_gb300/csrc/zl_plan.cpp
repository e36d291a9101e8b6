// Host planner: validates a work list, places every output block, cuts the list into
// tiles and orders them longest-first for the persistent scheduler.
//
// The work list mixes whole sequences with theta=(q,h,k) shards co-located on one
// rank ("Zellige", pith.science review, "What carries the argument"); the planner is
// what lets one launch run them together in a reproducible order: tiles from every item
// share a single list, ordered by cost with work-list order breaking ties, so the
// schedule is deterministic for a given list.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <new>
#include <set>
#include <tuple>

#include "zl_internal.h"

using namespace zl;

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

zl_status validate(const zl_work_item& it, int32_t H, int64_t T) {
  if (it.seq_offset < 0 || it.seq_len < 1 || it.seq_offset + it.seq_len > T) return ZL_ERR_INVALID_ARG;
  if (it.q_lo < 0 || it.q_lo > it.q_hi || it.q_hi > it.seq_len) return ZL_ERR_INVALID_ARG;
  if (it.kv_lo < 0 || it.kv_lo > it.kv_hi || it.kv_hi > it.seq_len) return ZL_ERR_INVALID_ARG;
  if (it.h_lo < 0 || it.h_lo > it.h_hi || it.h_hi > H) return ZL_ERR_INVALID_ARG;
  if (it.emit_lse != 0 && it.emit_lse != 1) return ZL_ERR_INVALID_ARG;
  if (it.out_offset < -1 || it.lse_offset < -1) return ZL_ERR_INVALID_ARG;
  if (it.out_offset >= 0 && (it.out_offset % 8) != 0) return ZL_ERR_ALIGN;
  return ZL_OK;
}

bool covers_sequence(const zl_work_item& it, int32_t H) {
  return it.q_lo == 0 && it.q_hi == it.seq_len && it.h_lo == 0 && it.h_hi == H;
}

using GroupKey = std::tuple<int64_t, int32_t, int32_t, int32_t, int32_t, int32_t>;
GroupKey group_key(const zl_work_item& it) {
  return std::make_tuple(it.seq_offset, it.seq_len, it.q_lo, it.q_hi, it.h_lo, it.h_hi);
}

// explicit: caller-chosen merge groups (member item ids in member order), or null for
// the default grouping by equal (sequence, rows, heads) keys in list order.
zl_status build(zl_plan* p, const zl_work_item* items, int32_t n,
                const std::vector<std::vector<int32_t>>* explicit_groups) {
  const int32_t H = p->n_heads, d = p->head_dim;
  const int64_t T = p->total_tokens;
  for (int32_t i = 0; i < n; ++i) {
    zl_status s = validate(items[i], H, T);
    if (s != ZL_OK) return s;
  }

  // ---- merge groups
  std::vector<std::vector<int32_t>> gmembers;
  p->item_group.assign(n, -1);
  if (explicit_groups) {
    // every emit_lse item in exactly one group, every member an emit_lse item, members
    // of a group sharing sequence, rows and heads
    for (size_t g = 0; g < explicit_groups->size(); ++g) {
      const std::vector<int32_t>& m = (*explicit_groups)[g];
      if (m.empty()) return ZL_ERR_INVALID_ARG;
      for (int32_t i : m) {
        if (i < 0 || i >= n || !items[i].emit_lse || p->item_group[i] >= 0) return ZL_ERR_INVALID_ARG;
        if (group_key(items[i]) != group_key(items[m[0]])) return ZL_ERR_INVALID_ARG;
        p->item_group[i] = (int32_t)g;
      }
    }
    for (int32_t i = 0; i < n; ++i)
      if (items[i].emit_lse && p->item_group[i] < 0) return ZL_ERR_INVALID_ARG;
    gmembers = *explicit_groups;
  } else {
    // emit_lse items sharing (sequence, rows, heads), list order
    std::map<GroupKey, int32_t> gkey;
    for (int32_t i = 0; i < n; ++i) {
      const zl_work_item& it = items[i];
      if (!it.emit_lse) continue;
      auto f = gkey.find(group_key(it));
      int32_t g;
      if (f == gkey.end()) {
        g = (int32_t)gmembers.size();
        gkey[group_key(it)] = g;
        gmembers.emplace_back();
      } else {
        g = f->second;
      }
      gmembers[g].push_back(i);
      p->item_group[i] = g;
    }
  }
  // KV chunks of one group must be disjoint; with ZL_PLAN_FUSE_LOCAL_KMERGE a group
  // whose chunks tile one contiguous range [kv_lo, kv_hi) is computed as one item
  std::vector<std::pair<int32_t, int32_t>> gspan(gmembers.size(), {0, 0});
  p->group_fused.assign(gmembers.size(), 0);
  for (size_t g = 0; g < gmembers.size(); ++g) {
    std::vector<std::pair<int32_t, int32_t>> r;
    for (int32_t i : gmembers[g]) r.push_back({items[i].kv_lo, items[i].kv_hi});
    std::sort(r.begin(), r.end());
    bool contiguous = true;
    for (size_t j = 1; j < r.size(); ++j) {
      if (r[j].first < r[j - 1].second) return ZL_ERR_INVALID_ARG;
      if (r[j].first != r[j - 1].second) contiguous = false;
    }
    gspan[g] = {r.front().first, r.back().second};
    p->group_fused[g] = p->fuse_kmerge && contiguous ? 1 : 0;
  }
  auto fused_member = [&](int32_t i) { return p->item_group[i] >= 0 && p->group_fused[p->item_group[i]]; };

  // ---- arena placement
  const int64_t packed_o = T * H * (int64_t)d, packed_lse = T * H;
  int64_t o_next = packed_o, lse_next = packed_lse, op_next = 0;
  for (int32_t i = 0; i < n; ++i) {  // user-placed blocks push the automatic ones back
    const zl_work_item& it = items[i];
    const int64_t oblk = (int64_t)(it.q_hi - it.q_lo) * (it.h_hi - it.h_lo) * d;
    const int64_t lblk = (int64_t)(it.q_hi - it.q_lo) * (it.h_hi - it.h_lo);
    if (it.out_offset >= 0) {
      if (it.emit_lse) op_next = std::max(op_next, it.out_offset + oblk);
      else o_next = std::max(o_next, it.out_offset + oblk);
    }
    if (it.lse_offset >= 0) lse_next = std::max(lse_next, it.lse_offset + lblk);
  }
  o_next = align_up(o_next, 8);
  op_next = align_up(op_next, 8);
  std::set<int64_t> packed_claim, grad_claim;

  p->resolved.assign(items, items + n);
  p->n_user = n;
  p->items.resize(n);
  int64_t dq_next = packed_o, dkv_next = packed_o, wsd_next = 0, wsq_next = 0, rh = 0;
  for (int32_t i = 0; i < n; ++i) {
    zl_work_item& it = p->resolved[i];
    DevItem& di = p->items[i];
    const int64_t nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo, nkv = it.kv_hi - it.kv_lo;
    if (!it.emit_lse && it.out_offset < 0 && it.lse_offset < 0 && covers_sequence(it, H) &&
        !packed_claim.count(it.seq_offset)) {
      packed_claim.insert(it.seq_offset);
      it.out_offset = it.seq_offset * H * d;
      it.lse_offset = it.seq_offset * H;
    }
    if (fused_member(i)) {
      // computed and stored through its group's fused item: no partial O, no own LSE
      it.out_offset = -1;
      it.lse_offset = -1;
    } else {
      if (it.out_offset < 0) {
        if (it.emit_lse) { it.out_offset = op_next; op_next += align_up(nq * nh * d, 8); }
        else { it.out_offset = o_next; o_next += align_up(nq * nh * d, 8); }
      }
      if (it.lse_offset < 0) { it.lse_offset = lse_next; lse_next += nq * nh; }
    }
    di.seq_offset = it.seq_offset;
    di.seq_len = it.seq_len;
    di.q_lo = it.q_lo; di.q_hi = it.q_hi;
    di.h_lo = it.h_lo; di.h_hi = it.h_hi;
    di.kv_lo = it.kv_lo; di.kv_hi = it.kv_hi;
    di.emit_lse = it.emit_lse;
    di.out_offset = it.out_offset;
    di.lse_offset = it.lse_offset;
    di.fin_out_offset = it.out_offset;   // replaced below for group members
    di.fin_lse_offset = it.lse_offset;
    const bool whole = !it.emit_lse && covers_sequence(it, H) && it.kv_lo == 0 && it.kv_hi == it.seq_len;
    if (whole && !grad_claim.count(it.seq_offset)) {
      grad_claim.insert(it.seq_offset);
      di.dq_offset = it.seq_offset * H * d;
      di.dkv_offset = it.seq_offset * H * d;
    } else {
      di.dq_offset = dq_next; dq_next += align_up(nq * nh * d, 8);
      di.dkv_offset = dkv_next; dkv_next += align_up(nkv * nh * d, 8);
    }
    di.ws_d_offset = wsd_next; wsd_next += nq * nh;
    di.ws_dq_offset = wsq_next; wsq_next += acc_floats(nq, nh, d);
    di.rowhead_begin = rh; rh += nq * nh;
  }
  p->total_rowheads = rh;

  // group final blocks
  p->groups.clear(); p->members.clear(); p->member_items.clear();
  int64_t grh = 0;
  for (size_t g = 0; g < gmembers.size(); ++g) {
    const zl_work_item& f = p->resolved[gmembers[g][0]];
    DevGroup G;
    G.member_begin = (int32_t)p->members.size();
    G.n_members = (int32_t)gmembers[g].size();
    G.nq = f.q_hi - f.q_lo;
    G.nh = f.h_hi - f.h_lo;
    if (covers_sequence(f, H) && !packed_claim.count(f.seq_offset)) {
      packed_claim.insert(f.seq_offset);
      G.out_offset = f.seq_offset * H * d;
      G.lse_offset = f.seq_offset * H;
    } else {
      G.out_offset = o_next; o_next += align_up((int64_t)G.nq * G.nh * d, 8);
      G.lse_offset = lse_next; lse_next += (int64_t)G.nq * G.nh;
    }
    G.rowhead_begin = grh; grh += (int64_t)G.nq * G.nh;
    for (int32_t i : gmembers[g]) {
      p->members.push_back({p->items[i].out_offset, p->items[i].lse_offset});
      p->member_items.push_back(i);
      p->items[i].fin_out_offset = G.out_offset;
      p->items[i].fin_lse_offset = G.lse_offset;
    }
    p->groups.push_back(G);
  }
  p->group_rowheads = grh;
  // the merge launch covers the unfused groups only (own row-head prefix); each fused
  // group becomes one forward item after the work list's items, whose O (bf16) and
  // LSE land straight in the group's final blocks
  p->merge_groups.clear();
  int64_t mrh = 0;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    DevGroup G = p->groups[g];
    if (p->group_fused[g]) {
      const zl_work_item& f = p->resolved[gmembers[g][0]];
      DevItem fi{};
      fi.seq_offset = f.seq_offset;
      fi.seq_len = f.seq_len;
      fi.q_lo = f.q_lo; fi.q_hi = f.q_hi;
      fi.h_lo = f.h_lo; fi.h_hi = f.h_hi;
      fi.kv_lo = gspan[g].first; fi.kv_hi = gspan[g].second;
      fi.emit_lse = 0;
      fi.out_offset = fi.fin_out_offset = G.out_offset;
      fi.lse_offset = fi.fin_lse_offset = G.lse_offset;
      fi.dq_offset = fi.dkv_offset = -1;  // forward only
      fi.rowhead_begin = rh;              // past every work-list row-head
      p->items.push_back(fi);
      continue;
    }
    G.rowhead_begin = mrh;
    mrh += (int64_t)G.nq * G.nh;
    p->merge_groups.push_back(G);
  }
  p->merge_rowheads = mrh;

  p->o_elems = o_next;
  p->o_partial_elems = op_next;
  p->lse_elems = lse_next;
  p->dq_elems = dq_next;
  p->dkv_elems = dkv_next;
  p->ws_d_floats = align_up(wsd_next, 4);
  p->ws_dq_floats = wsq_next;
  // deterministic dQ: one turn counter per (128-row query block, 32-row warp slice)
  p->ws_turn_ints = p->det_dq ? 4 * (wsq_next / ((int64_t)kBlockM * d)) : 0;
  p->workspace_bytes = 4 * (p->ws_d_floats + p->ws_dq_floats + p->ws_turn_ints);
  // ws_dq_offset is relative to the dQ accumulator region, which starts ws_d_floats
  // floats into the workspace (the launchers pass that base pointer)

  // ---- tiles, longest first (stable: ties keep work-list, head, block order)
  p->fwd_tiles.clear(); p->bwd_tiles.clear();
  for (int32_t i = 0; i < (int32_t)p->items.size(); ++i) {  // work-list items, then fused items
    const DevItem& it = p->items[i];
    const bool user = i < n;
    const int32_t nqb = (int32_t)ceil_div(it.q_hi - it.q_lo, kBlockM);
    const int32_t nfb = (int32_t)ceil_div(it.q_hi - it.q_lo, kFwdBlockM);
    const int32_t nkb = (int32_t)ceil_div(it.kv_hi - it.kv_lo, kBlockN);
    const bool fwd = !user || !fused_member(i);
    for (int32_t h = it.h_lo; h < it.h_hi; ++h) {
      if (fwd)
        for (int32_t b = 0; b < nfb; ++b) p->fwd_tiles.push_back({i, h, b, nkb});
      if (user)
        for (int32_t b = 0; b < nkb; ++b) p->bwd_tiles.push_back({i, h, b, nqb});
    }
  }
  auto by_cost = [](const DevTile& a, const DevTile& b) { return a.cost > b.cost; };
  std::stable_sort(p->fwd_tiles.begin(), p->fwd_tiles.end(), by_cost);
  if (p->det_dq)  // block-major within each cost: one head's KV tiles are claimed far apart
    std::stable_sort(p->bwd_tiles.begin(), p->bwd_tiles.end(),
                     [](const DevTile& a, const DevTile& b) { return a.block < b.block; });
  std::stable_sort(p->bwd_tiles.begin(), p->bwd_tiles.end(), by_cost);
  if (p->fwd_tiles.size() > (size_t)INT32_MAX || p->bwd_tiles.size() > (size_t)INT32_MAX)
    return ZL_ERR_INVALID_ARG;
  for (const auto& t : p->fwd_tiles) (p->items[t.item].emit_lse ? p->fwd_writes_partial : p->fwd_writes_o) = true;
  return ZL_OK;
}

template <typename T>
T* carve(char*& cur, size_t count) {
  T* p = reinterpret_cast<T*>(cur);
  cur += align_up((int64_t)(sizeof(T) * count), 256);
  return p;
}

zl_status upload(zl_plan* p) {
  if (cudaGetDevice(&p->device) != cudaSuccess) return ZL_ERR_CUDA;
  if (cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess)
    return ZL_ERR_CUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, p->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, p->device);
  if (major != 10 || minor != 3) return ZL_ERR_UNSUPPORTED;
  const size_t bytes = align_up(sizeof(DevItem) * p->items.size(), 256) +
                       align_up(sizeof(DevTile) * p->fwd_tiles.size(), 256) +
                       align_up(sizeof(DevTile) * p->bwd_tiles.size(), 256) +
                       align_up(sizeof(DevGroup) * p->merge_groups.size(), 256) +
                       align_up(sizeof(DevMember) * p->members.size(), 256) +
                       align_up(sizeof(int32_t) * kNumCounters, 256) +
                       align_up(sizeof(CUtensorMap) * p->items.size(), 256);
  if (cudaMalloc(&p->dev_blob, bytes) != cudaSuccess) { p->dev_blob = nullptr; return ZL_ERR_NO_MEMORY; }
  char* cur = static_cast<char*>(p->dev_blob);
  p->d_items = carve<DevItem>(cur, p->items.size());
  p->d_fwd_tiles = carve<DevTile>(cur, p->fwd_tiles.size());
  p->d_bwd_tiles = carve<DevTile>(cur, p->bwd_tiles.size());
  p->d_groups = carve<DevGroup>(cur, p->merge_groups.size());
  p->d_members = carve<DevMember>(cur, p->members.size());
  p->d_counters = carve<int32_t>(cur, kNumCounters);
  p->d_do_maps = carve<CUtensorMap>(cur, p->items.size());
  p->h_do_maps.resize(p->items.size());
  auto cp = [](void* dst, const void* src, size_t n) {
    return n == 0 || cudaMemcpy(dst, src, n, cudaMemcpyHostToDevice) == cudaSuccess;
  };
  bool ok = cp(p->d_items, p->items.data(), sizeof(DevItem) * p->items.size()) &&
            cp(p->d_fwd_tiles, p->fwd_tiles.data(), sizeof(DevTile) * p->fwd_tiles.size()) &&
            cp(p->d_bwd_tiles, p->bwd_tiles.data(), sizeof(DevTile) * p->bwd_tiles.size()) &&
            cp(p->d_groups, p->merge_groups.data(), sizeof(DevGroup) * p->merge_groups.size()) &&
            cp(p->d_members, p->members.data(), sizeof(DevMember) * p->members.size()) &&
            cudaMemset(p->d_counters, 0, sizeof(int32_t) * kNumCounters) == cudaSuccess;
  return ok ? ZL_OK : ZL_ERR_CUDA;
}

}  // namespace

namespace {

zl_status plan_impl(const zl_work_item* items, int32_t n_items, int32_t n_heads, int32_t head_dim,
                    int64_t total_tokens, uint32_t flags, const std::vector<std::vector<int32_t>>* groups,
                    zl_plan** out) {
  if (!out) return ZL_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_items < 0 || (n_items > 0 && !items) || n_heads < 1 || total_tokens < 1 ||
      total_tokens >= ((int64_t)1 << 31))
    return ZL_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return ZL_ERR_UNSUPPORTED;
  constexpr uint32_t kKnownFlags =
      ZL_PLAN_HOST_ONLY | ZL_PLAN_TEST_WITHHOLD_LOAD | ZL_PLAN_FUSE_LOCAL_KMERGE | ZL_PLAN_DETERMINISTIC_DQ;
  if (flags & ~kKnownFlags) return ZL_ERR_INVALID_ARG;
  zl_plan* p = new (std::nothrow) zl_plan();
  if (!p) return ZL_ERR_NO_MEMORY;
  p->n_heads = n_heads;
  p->head_dim = head_dim;
  p->total_tokens = total_tokens;
  p->host_only = (flags & ZL_PLAN_HOST_ONLY) != 0;
  p->test_withhold = (flags & ZL_PLAN_TEST_WITHHOLD_LOAD) != 0;
  p->fuse_kmerge = (flags & ZL_PLAN_FUSE_LOCAL_KMERGE) != 0;
  p->det_dq = (flags & ZL_PLAN_DETERMINISTIC_DQ) != 0;
  zl_status s = build(p, items, n_items, groups);
  if (s == ZL_OK && p->det_dq) s = zl_plan_check_bounds(p);  // includes the turn order
  if (s == ZL_OK && !p->host_only) s = upload(p);
  if (s != ZL_OK) {
    zl_plan_destroy(p);
    return s;
  }
  *out = p;
  return ZL_OK;
}

}  // namespace

extern "C" zl_status zl_plan_worklist(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                                      int32_t head_dim, int64_t total_tokens, uint32_t flags,
                                      zl_plan** out) {
  NvtxRange range("zl_plan_worklist");
  return plan_impl(items, n_items, n_heads, head_dim, total_tokens, flags, nullptr, out);
}

extern "C" zl_status zl_plan_worklist_groups(const zl_work_item* items, int32_t n_items, int32_t n_heads,
                                             int32_t head_dim, int64_t total_tokens, uint32_t flags,
                                             const int32_t* group_item_ids, const int32_t* group_ptr,
                                             int32_t n_groups, zl_plan** out) {
  NvtxRange range("zl_plan_worklist_groups");
  if (out) *out = nullptr;
  if (n_groups < 0 || (n_groups > 0 && (!group_item_ids || !group_ptr)) || (group_ptr && group_ptr[0] != 0))
    return ZL_ERR_INVALID_ARG;
  std::vector<std::vector<int32_t>> groups((size_t)n_groups);
  for (int32_t g = 0; g < n_groups; ++g) {
    if (group_ptr[g + 1] < group_ptr[g] || group_ptr[g + 1] > (int64_t)n_items) return ZL_ERR_INVALID_ARG;
    groups[g].assign(group_item_ids + group_ptr[g], group_item_ids + group_ptr[g + 1]);
  }
  return plan_impl(items, n_items, n_heads, head_dim, total_tokens, flags, &groups, out);
}

extern "C" void zl_plan_destroy(zl_plan* plan) {
  if (!plan) return;
  if (plan->dev_blob) cudaFree(plan->dev_blob);
  delete plan;
}

extern "C" zl_status zl_plan_arena_sizes(const zl_plan* p, int64_t* o_elems, int64_t* o_partial_elems,
                                         int64_t* lse_elems, int64_t* dq_elems, int64_t* dkv_elems,
                                         int64_t* workspace_bytes) {
  if (!p) return ZL_ERR_INVALID_ARG;
  if (o_elems) *o_elems = p->o_elems;
  if (o_partial_elems) *o_partial_elems = p->o_partial_elems;
  if (lse_elems) *lse_elems = p->lse_elems;
  if (dq_elems) *dq_elems = p->dq_elems;
  if (dkv_elems) *dkv_elems = p->dkv_elems;
  if (workspace_bytes) *workspace_bytes = p->workspace_bytes;
  return ZL_OK;
}

extern "C" zl_status zl_plan_item(const zl_plan* p, int32_t i, zl_work_item* resolved,
                                  int64_t* fin_out_offset, int64_t* fin_lse_offset,
                                  int64_t* dq_offset, int64_t* dkv_offset, int32_t* group) {
  if (!p || i < 0 || i >= p->n_user) return ZL_ERR_INVALID_ARG;
  if (resolved) *resolved = p->resolved[i];
  if (fin_out_offset) *fin_out_offset = p->items[i].fin_out_offset;
  if (fin_lse_offset) *fin_lse_offset = p->items[i].fin_lse_offset;
  if (dq_offset) *dq_offset = p->items[i].dq_offset;
  if (dkv_offset) *dkv_offset = p->items[i].dkv_offset;
  if (group) *group = p->item_group[i];
  return ZL_OK;
}

extern "C" zl_status zl_plan_count(const zl_plan* p, int32_t which, int64_t* count) {
  if (!p || !count) return ZL_ERR_INVALID_ARG;
  switch (which) {
    case 0: *count = (int64_t)p->fwd_tiles.size(); return ZL_OK;
    case 1: *count = (int64_t)p->bwd_tiles.size(); return ZL_OK;
    case 2: *count = (int64_t)p->groups.size(); return ZL_OK;
    case 3: *count = (int64_t)p->n_user; return ZL_OK;
    case 4: *count = (int64_t)p->merge_groups.size(); return ZL_OK;
    default: return ZL_ERR_INVALID_ARG;
  }
}

extern "C" zl_status zl_plan_tiles(const zl_plan* p, int32_t which, int32_t* out, int64_t n) {
  if (!p || !out || (which != 0 && which != 1)) return ZL_ERR_INVALID_ARG;
  const auto& t = which == 0 ? p->fwd_tiles : p->bwd_tiles;
  if (n < (int64_t)t.size()) return ZL_ERR_INVALID_ARG;
  for (size_t i = 0; i < t.size(); ++i) {
    out[4 * i + 0] = t[i].item;
    out[4 * i + 1] = t[i].head;
    out[4 * i + 2] = t[i].block;
    out[4 * i + 3] = t[i].cost;
  }
  return ZL_OK;
}

extern "C" zl_status zl_plan_group(const zl_plan* p, int32_t g, int32_t* members, int32_t cap,
                                   int32_t* n_members, int64_t* out_offset, int64_t* lse_offset) {
  if (!p || g < 0 || g >= (int32_t)p->groups.size()) return ZL_ERR_INVALID_ARG;
  const DevGroup& G = p->groups[g];
  if (n_members) *n_members = G.n_members;
  if (members)
    for (int32_t j = 0; j < G.n_members && j < cap; ++j) members[j] = p->member_items[G.member_begin + j];
  if (out_offset) *out_offset = G.out_offset;
  if (lse_offset) *lse_offset = G.lse_offset;
  return ZL_OK;
}

// Host-side dry run of every device access the plan's tables imply: each item's and
// group's blocks lie inside the arenas zl_plan_arena_sizes reports, and the workspace
// ranges inside workspace_bytes.  Tile indices address existing items, heads and blocks.
extern "C" zl_status zl_plan_check_bounds(const zl_plan* p) {
  if (!p) return ZL_ERR_INVALID_ARG;
  const int64_t d = p->head_dim;
  auto in = [](int64_t off, int64_t n, int64_t total) { return n == 0 || (off >= 0 && off + n <= total); };
  for (size_t i = 0; i < p->items.size(); ++i) {
    const DevItem& it = p->items[i];
    const int64_t nq = it.q_hi - it.q_lo, nh = it.h_hi - it.h_lo, nkv = it.kv_hi - it.kv_lo;
    const int64_t ob = nq * nh * d;
    const bool user = (int32_t)i < p->n_user;
    const bool fused_member = user && p->item_group[i] >= 0 && p->group_fused[p->item_group[i]];
    if (fused_member) {  // no own blocks: the group's fused item writes its final ones
      if (it.out_offset != -1 || it.lse_offset != -1) return ZL_ERR_INVALID_ARG;
    } else {
      if (!in(it.out_offset, ob, it.emit_lse ? p->o_partial_elems : p->o_elems)) return ZL_ERR_INVALID_ARG;
      if (!in(it.lse_offset, nq * nh, p->lse_elems)) return ZL_ERR_INVALID_ARG;
    }
    if (!in(it.fin_out_offset, ob, p->o_elems) || !in(it.fin_lse_offset, nq * nh, p->lse_elems))
      return ZL_ERR_INVALID_ARG;
    if (!user) {  // a fused forward item: no gradients, no workspace
      if (it.emit_lse) return ZL_ERR_INVALID_ARG;
      continue;
    }
    if (!in(it.dq_offset, ob, p->dq_elems) || !in(it.dkv_offset, nkv * nh * d, p->dkv_elems))
      return ZL_ERR_INVALID_ARG;
    if (!in(it.ws_d_offset, nq * nh, p->ws_d_floats) || !in(it.ws_dq_offset, acc_floats(nq, nh, d), p->ws_dq_floats))
      return ZL_ERR_INVALID_ARG;
    if (4 * (p->ws_d_floats + p->ws_dq_floats + p->ws_turn_ints) > p->workspace_bytes) return ZL_ERR_INVALID_ARG;
    if (p->det_dq && (it.ws_dq_offset % ((int64_t)kBlockM * d) != 0 ||
                      4 * ((it.ws_dq_offset + acc_floats(nq, nh, d)) / ((int64_t)kBlockM * d)) > p->ws_turn_ints))
      return ZL_ERR_INVALID_ARG;
  }
  for (size_t g = 0; g < p->groups.size(); ++g) {
    const DevGroup& G = p->groups[g];
    if (!in(G.out_offset, (int64_t)G.nq * G.nh * d, p->o_elems) || !in(G.lse_offset, (int64_t)G.nq * G.nh, p->lse_elems))
      return ZL_ERR_INVALID_ARG;
    if (p->group_fused[g]) continue;  // no partials to merge
    for (int32_t m = 0; m < G.n_members; ++m) {
      const DevMember& mb = p->members[G.member_begin + m];
      if (!in(mb.o_offset, (int64_t)G.nq * G.nh * d, p->o_partial_elems) ||
          !in(mb.lse_offset, (int64_t)G.nq * G.nh, p->lse_elems))
        return ZL_ERR_INVALID_ARG;
    }
  }
  const int32_t n = (int32_t)p->items.size();
  for (const auto& t : p->fwd_tiles) {
    if (t.item < 0 || t.item >= n) return ZL_ERR_INVALID_ARG;
    const DevItem& it = p->items[t.item];
    if (t.head < it.h_lo || t.head >= it.h_hi || (int64_t)t.block * kFwdBlockM >= it.q_hi - it.q_lo)
      return ZL_ERR_INVALID_ARG;
  }
  // deterministic dQ: the KV tiles of each (item, head) must be claimed in the order of
  // their turns (0, 1, 2, ...), so that a tile only ever waits on tiles claimed before it
  std::vector<int64_t> head_base(p->n_user + 1, 0);
  for (int32_t i = 0; i < p->n_user; ++i) head_base[i + 1] = head_base[i] + (p->items[i].h_hi - p->items[i].h_lo);
  std::vector<int32_t> next_turn(p->det_dq ? head_base[p->n_user] : 0, 0);
  for (const auto& t : p->bwd_tiles) {
    if (t.item < 0 || t.item >= p->n_user) return ZL_ERR_INVALID_ARG;
    const DevItem& it = p->items[t.item];
    if (t.head < it.h_lo || t.head >= it.h_hi || (int64_t)t.block * kBlockN >= it.kv_hi - it.kv_lo)
      return ZL_ERR_INVALID_ARG;
    if (p->det_dq && next_turn[head_base[t.item] + t.head - it.h_lo]++ != t.block) return ZL_ERR_INVALID_ARG;
  }
  return ZL_OK;
}
