// C-ABI front end: argument validation, split plan (grid size), TMA tensor
// maps, workspace layout, launches. Declared in include/zl_decode_attn.h.
#include "../../include/zl_decode_attn.h"
#include "kernels.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

namespace {

using zl::GqaParams;

constexpr double kLog2e = 1.4426950408889634;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// cuTensorMapEncodeTiled from the driver, fetched once through the runtime so
// the library links against cudart only.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A different nonzero tag for every GQA call in this process: the in-kernel
// split merge counts arrivals per tag, so counters left behind by a call that
// stopped early (a device error) are ignored by the next call. The call
// number goes through an invertible 32-bit mix (odd multiplier, xor-shifts),
// so consecutive tags are far apart and unlike small integers or float bits
// that other data may have left in the buffer.
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e = 0;
  while (e == 0) {
    uint32_t x = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    e = x;
  }
  return e;
}

struct DeviceInfo {
  int device = -1;
  int sms = 0;
};

zl_status current_device(DeviceInfo* info) {
  static int sm_count[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ZL_ERR_CUDA;
  if (dev < 0 || dev >= 64) return ZL_ERR_UNSUPPORTED;
  if (sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ZL_ERR_CUDA;
    sm_count[dev] = n;
  }
  info->device = dev;
  info->sms = sm_count[dev];
  return ZL_OK;
}

// ------------------------------------------------------------------ GQA plan
struct GqaPlan {
  int hpc = 0, nhg = 0, g = 0, grid = 0;
  bool fused = false;
  // shared-prefix calls: prefix tiles, sequences per group, groups
  int prefix_tiles = 0, sgs = 0, ng = 0;
  int q_group = 1;  // query tokens per row group
  int gh = 0, hchunks = 1;  // query heads per row group, head chunks per kv head
  int ngroups = 1;          // row groups: ceil(q_len / q_group) x hchunks
  int tg = 1;       // token groups per CTA (2: both groups of a two-group call in every CTA)
  bool unit_cut = false;  // one CTA per (sequence, head group): no cut unit, no merge
  size_t off_lse = 0, off_o = 0, off_pre_lse = 0, off_pre_o = 0;
  size_t off_suf_lse = 0, off_suf_o = 0, bytes = 0;
};

// Query tokens per sequence one call takes, and query heads per kv head (the
// GQA path takes the (token, head) rows of a kv head in groups of at most 16).
constexpr int kMaxQueryTokens = 128;
constexpr int kMaxGroupHeads = 128;
// A call whose longest (sequence, head group) unit has at most
// zl::kGqaUnitCutTiles tiles (known from max_seq_len) gives each unit a
// CTA of its own and skips the merge launch. Without max_seq_len the kernels
// take the same decision on the device (GqaParams::auto_cut).

zl_status gqa_validate_shape(const zl_decode_attn_params* a) {
  if (!a || a->struct_size != sizeof(zl_decode_attn_params)) return ZL_ERR_INVALID_ARG;
  if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->q_len < 1 || a->page_size < 1 ||
      a->num_pages < 1 || a->block_table_stride < 1 || a->D_qk < 1 || a->D_v < 1 ||
      a->num_ctas < 0 || a->max_seq_len < 0)
    return ZL_ERR_INVALID_ARG;
  if (a->Hq % a->Hkv != 0) return ZL_ERR_INVALID_ARG;
  if (a->flags & ~uint32_t(ZL_DECODE_SINGLE_LAUNCH | ZL_DECODE_TEST_STALL))
    return ZL_ERR_INVALID_ARG;
  if (a->num_ctas > 65535) return ZL_ERR_UNSUPPORTED;  // the tile cut needs G^2 < 2^32
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return ZL_ERR_INVALID_ARG;
  if (a->D_qk != zl::kGqaHeadDim || a->D_v != zl::kGqaHeadDim) return ZL_ERR_UNSUPPORTED;
  // (query token, head) rows of one kv head share an m16 tile: at most 16 per
  // row group. A call with g * q_len > 16 takes its query tokens in groups of
  // 16 / g, or with g > 16 each token's heads in ceil(g / 16) chunks (side by
  // side in one launch; one launch per group in single-launch mode). A
  // shared-prefix call keeps all its rows in one group.
  if (a->Hq / a->Hkv > kMaxGroupHeads || a->q_len > kMaxQueryTokens) return ZL_ERR_UNSUPPORTED;
  if (a->shared_prefix_pages > 0 && a->Hq / a->Hkv * a->q_len > 16) return ZL_ERR_UNSUPPORTED;
  if (a->page_size % zl::kGqaTile != 0 || a->page_size > 1024) return ZL_ERR_UNSUPPORTED;
  if (a->B > zl::kMaxBatch) return ZL_ERR_UNSUPPORTED;
  if (a->shared_prefix_pages < 0 || a->shared_prefix_pages > a->block_table_stride)
    return ZL_ERR_INVALID_ARG;
  if (a->shared_prefix_pages > 0 && (a->flags & ZL_DECODE_SINGLE_LAUNCH))
    return ZL_ERR_UNSUPPORTED;
  return ZL_OK;
}

zl_status gqa_plan(const zl_decode_attn_params* a, GqaPlan* plan) {
  zl_status st = gqa_validate_shape(a);
  if (st != ZL_OK) return st;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != ZL_OK) return st;
  plan->g = a->Hq / a->Hkv;
  plan->fused = (a->flags & ZL_DECODE_SINGLE_LAUNCH) != 0;
  plan->hpc = zl::gqa_heads_per_cta(a->Hkv);
  plan->nhg = a->Hkv / plan->hpc;
  if (plan->g <= 16) {  // every head of a token in one group
    plan->gh = plan->g;
    plan->hchunks = 1;
    plan->q_group = std::min(a->q_len, 16 / plan->g);
  } else {  // one token per group, its heads in chunks of at most 16
    plan->hchunks = (plan->g + 15) / 16;
    plan->gh = (plan->g + plan->hchunks - 1) / plan->hchunks;
    plan->q_group = 1;
  }
  plan->ngroups = (a->q_len + plan->q_group - 1) / plan->q_group * plan->hchunks;
  // Exactly two row groups, side by side: every CTA takes both (half the kv
  // heads per CTA, the same number of warps), so that one shared-memory stage
  // serves both groups and each K/V tile crosses from L2 once.
  if (plan->ngroups == 2 && !plan->fused && a->shared_prefix_pages == 0) {
    plan->tg = 2;
    plan->hpc = std::max(1, plan->hpc / 2);
    plan->nhg = a->Hkv / plan->hpc;
  }
  const int rps = plan->gh * plan->q_group;
  if (a->shared_prefix_pages > 0) {
    plan->prefix_tiles = a->shared_prefix_pages * a->page_size / zl::kGqaTile;
    plan->sgs = 16 / rps > 0 ? 16 / rps : 1;
    plan->ng = (a->B + plan->sgs - 1) / plan->sgs;
    if (plan->ng + a->B > zl::kMaxBatch) return ZL_ERR_UNSUPPORTED;  // one tile-count table
  }
  const int rows_per_warp = plan->prefix_tiles > 0 ? plan->sgs * rps : rps;
  int grid = a->num_ctas;
  if (grid == 0) {
    // the kernel's tile-offset table: one entry per unit (prefix groups and
    // sequences) plus the total; the launch takes the same layout
    const bool small = (plan->prefix_tiles > 0 ? plan->ng : 0) + a->B + 1 <= zl::kSmallTable;
    const int per_sm =
        plan->prefix_tiles > 0
            ? zl::gqa_shared_ctas_per_sm(plan->hpc, rows_per_warp > 8, a->q_len > 1, small,
                                         dev.device)
            : zl::gqa_ctas_per_sm(plan->hpc, rps > 8, a->q_len > 1, plan->fused, plan->tg, small,
                                  dev.device);
    if (per_sm < 1) return ZL_ERR_CUDA;
    grid = dev.sms * per_sm;
    if (a->max_seq_len > 0 && plan->prefix_tiles == 0) {
      const int64_t max_tiles = (int64_t(a->max_seq_len) + zl::kGqaTile - 1) / zl::kGqaTile;
      const int64_t units = int64_t(a->B) * plan->nhg;
      if (units <= grid && max_tiles <= zl::kGqaUnitCutTiles) {
        // Short contexts: one CTA per whole unit. Streaming the longest unit
        // alone costs less than cutting units and merging their pieces.
        plan->unit_cut = true;
        plan->fused = false;
        grid = int(units);
      } else {
        // No more CTAs than tiles: B * head groups * ceil(max_seq_len / 16).
        const int64_t tiles = units * max_tiles;
        if (tiles < grid) grid = int(tiles < 1 ? 1 : tiles);
      }
    }
  }
  plan->grid = grid;
  // partial slots: 2 per (token group, CTA) pair and consumer warp
  const size_t rows = size_t(grid) * plan->tg * 2 * plan->hpc * rows_per_warp;
  const size_t store_rows = plan->prefix_tiles > 0 ? size_t(a->B) * a->q_len * a->Hq : 0;
  // [0, off_lse): one arrival counter (8 bytes) per (sequence, kv head); then
  // the partials' lse and outputs; then (shared prefix) each query row's
  // result over its prefix part and over its suffix part when one CTA had the
  // whole unit: base-2 lse and normalised fp32 output.
  plan->off_lse = round_up(size_t(a->B) * a->Hkv * sizeof(unsigned long long), 256);
  plan->off_o = plan->off_lse + round_up(rows * sizeof(float), 256);
  plan->off_pre_lse = plan->off_o + round_up(rows * zl::kGqaHeadDim * sizeof(float), 256);
  plan->off_pre_o = plan->off_pre_lse + round_up(store_rows * sizeof(float), 256);
  plan->off_suf_lse =
      plan->off_pre_o + round_up(store_rows * zl::kGqaHeadDim * sizeof(float), 256);
  plan->off_suf_o = plan->off_suf_lse + round_up(store_rows * sizeof(float), 256);
  plan->bytes = plan->off_suf_o + store_rows * zl::kGqaHeadDim * sizeof(float);
  return ZL_OK;
}

// A call with several groups of query tokens runs them in one launch, side by
// side, unless it merges inside the attention kernel (its arrival counters
// are per sequence and kv head) or has a shared prefix (one group only).
bool groups_together(const GqaPlan& plan) {
  return plan.ngroups > 1 && !plan.fused && plan.prefix_tiles == 0;
}

// ------------------------------------------------------------------ MLA plan
struct MlaPlan {
  int clusters = 0;
  size_t off_split = 0, off_span = 0, off_lse = 0, off_o = 0, bytes = 0;
};

zl_status mla_validate_shape(const zl_decode_attn_params* a) {
  if (!a || a->struct_size != sizeof(zl_decode_attn_params)) return ZL_ERR_INVALID_ARG;
  if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->q_len < 1 || a->page_size < 1 ||
      a->num_pages < 1 || a->block_table_stride < 1 || a->D_qk < 1 || a->D_v < 1 ||
      a->num_ctas < 0 || a->max_seq_len < 0)
    return ZL_ERR_INVALID_ARG;
  if (!(a->scale > 0.f) || !std::isfinite(a->scale)) return ZL_ERR_INVALID_ARG;
  if (a->Hkv != 1) return ZL_ERR_INVALID_ARG;
  if (a->flags & ~uint32_t(ZL_DECODE_SINGLE_LAUNCH | ZL_DECODE_TEST_STALL))
    return ZL_ERR_INVALID_ARG;
  if (a->flags) return ZL_ERR_UNSUPPORTED;  // neither flag exists for MLA
  if (a->shared_prefix_pages != 0) return ZL_ERR_UNSUPPORTED;
  if (a->D_qk != zl::kMlaDqk || a->D_v != zl::kMlaDv) return ZL_ERR_UNSUPPORTED;
  if (a->Hq != zl::kMlaHeads) return ZL_ERR_UNSUPPORTED;
  if (a->page_size % zl::kMlaTile != 0 || a->page_size > 1024) return ZL_ERR_UNSUPPORTED;
  if (int64_t(a->B) * a->q_len > zl::kMlaMaxBatch) return ZL_ERR_UNSUPPORTED;
  return ZL_OK;
}

zl_status mla_plan(const zl_decode_attn_params* a, MlaPlan* plan) {
  zl_status st = mla_validate_shape(a);
  if (st != ZL_OK) return st;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != ZL_OK) return st;
  int clusters = a->num_ctas > 0 ? (a->num_ctas + 1) / 2 : dev.sms / 2;
  if (a->num_ctas == 0 && a->max_seq_len > 0) {
    const int64_t tiles =
        int64_t(a->B) * a->q_len *
        ((int64_t(a->max_seq_len) + zl::kMlaTile - 1) / zl::kMlaTile);
    if (tiles < clusters) clusters = int(tiles < 1 ? 1 : tiles);
  }
  if (clusters < 1) clusters = 1;
  plan->clusters = clusters;
  const size_t rows = size_t(clusters) * 2 * zl::kMlaHeads;
  // tile prefix sums per (sequence, query token) | first tile of each cluster |
  // first and last cluster of each unit | partial lse | partial outputs
  const size_t units = size_t(a->B) * a->q_len;
  plan->off_split = round_up((units + 1) * sizeof(int32_t), 256);
  plan->off_span = plan->off_split + round_up((size_t(clusters) + 1) * sizeof(int32_t), 256);
  plan->off_lse = plan->off_span + round_up(units * 2 * sizeof(int32_t), 256);
  plan->off_o = plan->off_lse + round_up(rows * sizeof(float), 256);
  plan->bytes = plan->off_o + rows * zl::kMlaDv * sizeof(float);
  return ZL_OK;
}

// Tensor maps this thread encoded recently, so a decode loop over the same
// pools skips the driver call (the map is a plain 128-byte value).
struct PoolMapKey {
  const void* pool;
  int64_t page_stride, token_stride, head_stride;
  int32_t D, page_size, Hkv, num_pages, box_heads;
  bool operator==(const PoolMapKey& o) const {
    return pool == o.pool && page_stride == o.page_stride && token_stride == o.token_stride &&
           head_stride == o.head_stride && D == o.D && page_size == o.page_size &&
           Hkv == o.Hkv && num_pages == o.num_pages && box_heads == o.box_heads;
  }
};
constexpr int kMapCache = 8;
thread_local PoolMapKey t_map_keys[kMapCache];
thread_local CUtensorMap t_maps[kMapCache];
thread_local int t_map_used = 0, t_map_next = 0;

zl_status encode_pool_map(CUtensorMap* map, const void* pool, const zl_decode_attn_params* a,
                          int box_heads) {
  const PoolMapKey key{pool, a->page_stride, a->token_stride, a->head_stride, a->D_qk,
                       a->page_size, a->Hkv, a->num_pages, box_heads};
  for (int i = 0; i < t_map_used; ++i)
    if (t_map_keys[i] == key) {
      *map = t_maps[i];
      return ZL_OK;
    }
  auto encode = tensor_map_encoder();
  if (!encode) return ZL_ERR_CUDA;
  const cuuint64_t dims[4] = {cuuint64_t(a->D_qk), cuuint64_t(a->page_size), cuuint64_t(a->Hkv),
                              cuuint64_t(a->num_pages)};
  const cuuint64_t strides[3] = {cuuint64_t(a->token_stride) * 2, cuuint64_t(a->head_stride) * 2,
                                 cuuint64_t(a->page_stride) * 2};
  const cuuint32_t box[4] = {64, cuuint32_t(zl::kGqaTile), cuuint32_t(box_heads), 1};
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool),
                            dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return ZL_ERR_UNSUPPORTED;
  t_map_keys[t_map_next] = key;
  t_maps[t_map_next] = *map;
  t_map_next = (t_map_next + 1) % kMapCache;
  if (t_map_used < kMapCache) ++t_map_used;
  return ZL_OK;
}

zl_status validate_pointers(const zl_decode_attn_params* a, bool need_v) {
  if (!a->q || !a->k_pool || !a->block_table || !a->seq_lens || !a->out)
    return ZL_ERR_INVALID_ARG;
  if (need_v && !a->v_pool) return ZL_ERR_INVALID_ARG;
  if (!need_v && a->v_pool) return ZL_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->out, 16) ||
      (a->v_pool && !aligned(a->v_pool, 16)) || !aligned(a->block_table, 4) ||
      !aligned(a->seq_lens, 4) || (a->lse && !aligned(a->lse, 4)) ||
      (a->err_flags && !aligned(a->err_flags, 4)))
    return ZL_ERR_INVALID_ARG;
  if (a->page_stride <= 0 || a->token_stride <= 0 || a->head_stride <= 0 ||
      a->page_stride % 8 || a->token_stride % 8 || a->head_stride % 8)
    return ZL_ERR_INVALID_ARG;
  // fused KV append: GQA takes k_new and v_new together, MLA k_new alone
  if (!a->k_new && a->v_new) return ZL_ERR_INVALID_ARG;
  if (a->k_new && (need_v != (a->v_new != nullptr))) return ZL_ERR_INVALID_ARG;
  if ((a->k_new && !aligned(a->k_new, 16)) || (a->v_new && !aligned(a->v_new, 16)))
    return ZL_ERR_INVALID_ARG;
  return ZL_OK;
}

}  // namespace

extern "C" {

const char* zl_status_string(zl_status s) {
  switch (s) {
    case ZL_OK: return "ok";
    case ZL_ERR_INVALID_ARG: return "invalid argument";
    case ZL_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case ZL_ERR_WORKSPACE: return "workspace missing or too small";
    case ZL_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

zl_status zl_decode_attn_workspace_size(const zl_decode_attn_params* a, size_t* bytes) {
  if (!bytes) return ZL_ERR_INVALID_ARG;
  GqaPlan plan;
  const zl_status st = gqa_plan(a, &plan);
  if (st != ZL_OK) return st;
  *bytes = plan.bytes;
  return ZL_OK;
}

zl_status zl_decode_attn_launches(const zl_decode_attn_params* a, int32_t* launches) {
  if (!launches) return ZL_ERR_INVALID_ARG;
  GqaPlan plan;
  const zl_status st = gqa_plan(a, &plan);
  if (st != ZL_OK) return st;
  const int per_launch = (plan.fused || plan.unit_cut) ? 1 : 2;
  *launches = groups_together(plan) ? per_launch : plan.ngroups * per_launch;
  return ZL_OK;
}

zl_status zl_decode_attn(const zl_decode_attn_params* a, zl_stream_t stream) {
  zl_status st = gqa_validate_shape(a);
  if (st != ZL_OK) return st;
  if ((st = validate_pointers(a, true)) != ZL_OK) return st;
  GqaPlan plan;
  if ((st = gqa_plan(a, &plan)) != ZL_OK) return st;
  if (!a->workspace || !aligned(a->workspace, 256) || a->workspace_bytes < plan.bytes)
    return ZL_ERR_WORKSPACE;

  GqaParams p;
  std::memset(&p, 0, sizeof(p));
  if ((st = encode_pool_map(&p.tmap_k, a->k_pool, a, plan.hpc)) != ZL_OK) return st;
  if ((st = encode_pool_map(&p.tmap_v, a->v_pool, a, plan.hpc)) != ZL_OK) return st;
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  p.block_table = a->block_table;
  p.seq_lens = a->seq_lens;
  p.bt_stride = a->block_table_stride;
  char* ws = static_cast<char*>(a->workspace);
  p.ws_count = reinterpret_cast<unsigned long long*>(ws);
  p.ws_lse = reinterpret_cast<float*>(ws + plan.off_lse);
  p.ws_o = reinterpret_cast<float*>(ws + plan.off_o);
  p.err_flags = a->err_flags;
  p.epoch = next_epoch();
  p.test_stall = (a->flags & ZL_DECODE_TEST_STALL) ? 1 : 0;
  p.B = a->B;
  p.unit_cut = plan.unit_cut ? 1 : 0;
  p.auto_cut = (a->num_ctas == 0 && !plan.unit_cut && plan.prefix_tiles == 0) ? 1 : 0;
  p.q_total = a->q_len;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.g = plan.g;
  p.gh = plan.gh;
  p.hchunks = plan.hchunks;
  p.hc0 = 0;
  p.page_size = a->page_size;
  p.num_pages = a->num_pages;
  p.hpc = plan.hpc;
  p.nhg = plan.nhg;
  p.scale_log2 = float(double(a->scale) * kLog2e);
  p.prefix_tiles = plan.prefix_tiles;
  p.sgs = plan.sgs;
  p.ng = plan.ng;
  p.pre_lse = reinterpret_cast<float*>(ws + plan.off_pre_lse);
  p.pre_o = reinterpret_cast<float*>(ws + plan.off_pre_o);
  p.suf_lse = reinterpret_cast<float*>(ws + plan.off_suf_lse);
  p.suf_o = reinterpret_cast<float*>(ws + plan.off_suf_o);
  if (a->k_new) {  // the attention launch stores the new tokens' rows first
    p.k_new = static_cast<const uint4*>(a->k_new);
    p.v_new = static_cast<const uint4*>(a->v_new);
    p.k_pool = static_cast<uint4*>(const_cast<void*>(a->k_pool));
    p.v_pool = static_cast<uint4*>(const_cast<void*>(a->v_pool));
    p.page_stride16 = a->page_stride / 8;
    p.token_stride16 = a->token_stride / 8;
    p.head_stride16 = a->head_stride / 8;
  }

  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int ngroups = plan.ngroups;
  if (groups_together(plan)) {
    // Every row group (q_group query tokens, gh heads of each kv head) in one
    // launch, side by side: two share every CTA; more split the grid's CTAs
    // between them, and each cuts the same tile line, so the groups read each
    // K/V tile at about the same time (all but the first read are served by
    // L2). One merge launch covers every group.
    p.q_tok0 = 0;
    p.q_len = plan.q_group;
    p.ngroups = ngroups;
    p.tg = plan.tg;
    // two groups per CTA: each group has every CTA; else the grid is split.
    // The partial slots are sized for plan.grid (group, CTA) pairs: with
    // floor(grid / ngroups) >= 1 CTAs per group the pairs are at most that; a
    // group with one CTA (more groups than CTAs) takes the whole tile line,
    // so it cuts no unit and writes no partial (nor does a unit-cut launch).
    p.group_ctas = plan.unit_cut || plan.tg == 2 ? plan.grid : std::max(1, plan.grid / ngroups);
    const int launch_grid = plan.tg == 2 ? plan.grid : p.group_ctas * ngroups;
    const cudaError_t e = zl::gqa_decode_launch(
        p, launch_grid, false, s, reinterpret_cast<cudaEvent_t>(a->attn_begin),
        reinterpret_cast<cudaEvent_t>(a->attn_end));
    return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
  }
  // One launch (attention, then its merge) per row group: group gg is query
  // tokens from (gg / hchunks) * q_group, head chunk gg % hchunks. attn_begin
  // is recorded before the first, attn_end after the last attention launch.
  // The launches share the workspace: each reads it only after the one before
  // has finished (programmatic dependent launches).
  p.ngroups = 1;
  p.tg = 1;
  p.group_ctas = plan.grid;
  for (int gg = 0; gg < ngroups; ++gg) {
    const int tok0 = gg / plan.hchunks * plan.q_group;
    p.q_tok0 = tok0;
    p.q_len = std::min(plan.q_group, a->q_len - tok0);
    p.hc0 = gg % plan.hchunks;
    if (gg > 0) p.epoch = next_epoch();
    const bool first = gg == 0, last = gg == ngroups - 1;
    cudaEvent_t begin = first ? reinterpret_cast<cudaEvent_t>(a->attn_begin) : nullptr;
    cudaEvent_t end = last ? reinterpret_cast<cudaEvent_t>(a->attn_end) : nullptr;
    const cudaError_t e = plan.prefix_tiles > 0
                              ? zl::gqa_shared_launch(p, plan.grid, s, begin, end)
                              : zl::gqa_decode_launch(p, plan.grid, plan.fused, s, begin, end);
    if (e != cudaSuccess) return ZL_ERR_CUDA;
  }
  return ZL_OK;
}

zl_status zl_decode_attn_mla_workspace_size(const zl_decode_attn_params* a, size_t* bytes) {
  if (!bytes) return ZL_ERR_INVALID_ARG;
  MlaPlan plan;
  const zl_status st = mla_plan(a, &plan);
  if (st != ZL_OK) return st;
  *bytes = plan.bytes;
  return ZL_OK;
}

zl_status zl_decode_attn_mla(const zl_decode_attn_params* a, zl_stream_t stream) {
  zl_status st = mla_validate_shape(a);
  if (st != ZL_OK) return st;
  if ((st = validate_pointers(a, false)) != ZL_OK) return st;
  MlaPlan plan;
  if ((st = mla_plan(a, &plan)) != ZL_OK) return st;
  if (!a->workspace || !aligned(a->workspace, 256) || a->workspace_bytes < plan.bytes)
    return ZL_ERR_WORKSPACE;
  auto encode = tensor_map_encoder();
  if (!encode) return ZL_ERR_CUDA;

  zl::MlaParams p;
  std::memset(&p, 0, sizeof(p));
  {
    const cuuint64_t dims[3] = {cuuint64_t(zl::kMlaDqk), cuuint64_t(a->page_size),
                                cuuint64_t(a->num_pages)};
    const cuuint64_t strides[2] = {cuuint64_t(a->token_stride) * 2, cuuint64_t(a->page_stride) * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(zl::kMlaTile), 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    if (encode(&p.tmap_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a->k_pool), dims,
               strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ZL_ERR_UNSUPPORTED;
  }
  p.q = static_cast<const __nv_bfloat16*>(a->q);
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.lse = a->lse;
  p.block_table = a->block_table;
  p.seq_lens = a->seq_lens;
  p.bt_stride = a->block_table_stride;
  char* ws = static_cast<char*>(a->workspace);
  p.ws_prefix = reinterpret_cast<int32_t*>(ws);
  p.ws_split = reinterpret_cast<int32_t*>(ws + plan.off_split);
  p.ws_span = reinterpret_cast<int32_t*>(ws + plan.off_span);
  p.ws_lse = reinterpret_cast<float*>(ws + plan.off_lse);
  p.ws_o = reinterpret_cast<float*>(ws + plan.off_o);
  p.err_flags = a->err_flags;
  p.B = a->B;
  p.q_len = a->q_len;
  p.page_size = a->page_size;
  p.num_pages = a->num_pages;
  p.scale_log2 = float(double(a->scale) * kLog2e);
  p.out_align32 = aligned(a->out, 32) ? 1 : 0;
  if (a->k_new) {  // the attention launch stores the new tokens' latent rows first
    p.kv_new = static_cast<const uint4*>(a->k_new);
    p.kv_pool = static_cast<uint4*>(const_cast<void*>(a->k_pool));
    p.page_stride16 = a->page_stride / 8;
    p.token_stride16 = a->token_stride / 8;
  }
  const cudaError_t e = zl::mla_decode_launch(p, plan.clusters,
                                              reinterpret_cast<cudaStream_t>(stream),
                                              reinterpret_cast<cudaEvent_t>(a->attn_begin),
                                              reinterpret_cast<cudaEvent_t>(a->attn_end));
  return e == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}

}  // extern "C"
