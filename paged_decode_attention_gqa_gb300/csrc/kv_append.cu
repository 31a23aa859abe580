// Paged KV append: copy the new tokens' K and V rows into their page slots
// (declared in include/zl_decode_attn.h as zl_kv_append).
//
// The new rows are what the fused QKV projection produces ("ZhiLight: Zhihu's
// CUDA Inference Engine ...", section "Dual streams, host all-reduce and the
// memory model": fused kernels for qkv); decode attention then reads them from
// the cache like every older token. New token i of sequence b is logical
// position seq_lens[b] - q_len + i.
//
// One warp per (sequence, new token, kv head): the K row and then the V row
// are cut into 16-byte chunks, one chunk per lane per pass (for D = 128 the
// 16 + 16 chunks are one pass of the warp). Pure copies, so bit-exact.
#include "../../include/zl_decode_attn.h"
#include "kernels.h"
#include "ptx.cuh"

#include <cstring>

namespace zl {
namespace {

struct AppendParams {
  const uint4* k_new;  // [rows][ck]
  const uint4* v_new;  // [rows][cv] or nullptr
  uint4* k_pool;
  uint4* v_pool;       // nullptr for a latent-only pool
  int64_t page_stride, token_stride, head_stride;  // in 16-byte chunks
  const int32_t* block_table;
  int64_t bt_stride;
  const int32_t* seq_lens;
  uint32_t* err_flags;
  int64_t rows;        // B * q_len * Hkv
  int q_len, Hkv, ck, cv, page_size, num_pages;
};

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendParams p) {
  // The attention kernels that follow are programmatic dependents: let them
  // start their prologue now (they wait for this grid before reading memory).
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < p.rows;
       row += warps) {
    const int kh = int(row % p.Hkv);
    const int64_t bi = row / p.Hkv;
    const int i = int(bi % p.q_len);
    const int64_t b = bi / p.q_len;
    const int L = __ldg(p.seq_lens + b);
    if (L < p.q_len || int64_t(L) > p.bt_stride * p.page_size) {
      if (lane == 0 && i == 0 && kh == 0 && p.err_flags) atomicOr(p.err_flags, 2u);
      continue;
    }
    const int t = L - p.q_len + i;
    const int page = __ldg(p.block_table + b * p.bt_stride + t / p.page_size);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0 && kh == 0 && p.err_flags) atomicOr(p.err_flags, 1u);
      continue;
    }
    const int64_t dst =
        int64_t(page) * p.page_stride + int64_t(t % p.page_size) * p.token_stride +
        int64_t(kh) * p.head_stride;
    const int n = p.ck + (p.v_pool ? p.cv : 0);
    for (int c = lane; c < n; c += 32) {
      if (c < p.ck) {
        p.k_pool[dst + c] = __ldg(p.k_new + row * p.ck + c);
      } else {
        const int cv = c - p.ck;
        p.v_pool[dst + cv] = __ldg(p.v_new + row * p.cv + cv);
      }
    }
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

zl_status validate(const zl_kv_append_params* a) {
  if (!a || a->struct_size != sizeof(zl_kv_append_params)) return ZL_ERR_INVALID_ARG;
  if (a->B < 1 || a->q_len < 1 || a->Hkv < 1 || a->page_size < 1 || a->num_pages < 1 ||
      a->block_table_stride < 1 || a->D_k < 8 || a->D_k > 1024 || a->D_k % 8)
    return ZL_ERR_INVALID_ARG;
  if (!a->k_new || !a->k_pool || !a->block_table || !a->seq_lens) return ZL_ERR_INVALID_ARG;
  if (!a->v_pool != !a->v_new) return ZL_ERR_INVALID_ARG;
  if (a->v_pool && (a->D_v < 8 || a->D_v > 1024 || a->D_v % 8)) return ZL_ERR_INVALID_ARG;
  if (!aligned16(a->k_new) || !aligned16(a->k_pool) || (a->v_new && !aligned16(a->v_new)) ||
      (a->v_pool && !aligned16(a->v_pool)) ||
      (reinterpret_cast<uintptr_t>(a->block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(a->seq_lens) & 3u) ||
      (a->err_flags && (reinterpret_cast<uintptr_t>(a->err_flags) & 3u)))
    return ZL_ERR_INVALID_ARG;
  if (a->page_stride <= 0 || a->token_stride <= 0 || a->head_stride <= 0 ||
      a->page_stride % 8 || a->token_stride % 8 || a->head_stride % 8)
    return ZL_ERR_INVALID_ARG;
  return ZL_OK;
}

}  // namespace
}  // namespace zl

extern "C" zl_status zl_kv_append(const zl_kv_append_params* a, zl_stream_t stream) {
  const zl_status st = zl::validate(a);
  if (st != ZL_OK) return st;
  zl::AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.k_new = static_cast<const uint4*>(a->k_new);
  p.v_new = static_cast<const uint4*>(a->v_new);
  p.k_pool = static_cast<uint4*>(a->k_pool);
  p.v_pool = static_cast<uint4*>(a->v_pool);
  p.page_stride = a->page_stride / 8;
  p.token_stride = a->token_stride / 8;
  p.head_stride = a->head_stride / 8;
  p.block_table = a->block_table;
  p.bt_stride = a->block_table_stride;
  p.seq_lens = a->seq_lens;
  p.err_flags = a->err_flags;
  p.rows = int64_t(a->B) * a->q_len * a->Hkv;
  p.q_len = a->q_len;
  p.Hkv = a->Hkv;
  p.ck = a->D_k / 8;
  p.cv = a->v_pool ? a->D_v / 8 : 0;
  p.page_size = a->page_size;
  p.num_pages = a->num_pages;
  const int64_t blocks = (p.rows + 7) / 8;  // 8 warps per block, one row per warp
  const int grid = int(blocks < 65535 ? blocks : 65535);
  zl::kv_append_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? ZL_OK : ZL_ERR_CUDA;
}
