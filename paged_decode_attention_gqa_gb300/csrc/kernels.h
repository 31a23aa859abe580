// Internal interface between the C-ABI front end (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace zl {

constexpr int kGqaTile = 16;     // tokens per pipeline stage of the GQA kernel
constexpr int kGqaHeadDim = 128; // D_qk = D_v
constexpr int kMaxBatch = 4096;  // sequences per call (prefix table lives in smem)
// Entries of the GQA kernel's small tile-offset table (units + 1); calls with
// more units take the full one of kMaxBatch + 1 entries.
constexpr int kSmallTable = 512;
// A call whose longest (sequence, head group) unit has at most this many
// 16-token tiles gives each unit a CTA of its own and merges nothing (when the
// units fit in the grid). With few units a CTA's tiles are latency-bound
// (~0.5 us each, whatever the head count), so a unit this short costs about
// what a merge launch does; longer ones are cut and merged.
constexpr int kGqaUnitCutTiles = 8;

// Everything the GQA attention kernel reads.
struct GqaParams {
  CUtensorMap tmap_k;  // 4-D {D, page_size, Hkv, num_pages}, box {64, 16, HPC, 1}, 128B swizzle
  CUtensorMap tmap_v;  // same geometry over the V pool
  const __nv_bfloat16* q;  // [B, q_len, Hq, 128]
  __nv_bfloat16* out;      // [B, q_len, Hq, 128]
  float* lse;              // [B, q_len, Hq] natural log, or nullptr
  const int32_t* block_table;
  const int32_t* seq_lens;
  int64_t bt_stride;
  unsigned long long* ws_count;  // [B * Hkv] arrivals per split unit: epoch << 32 | count
  // Partial slots: [(row group, CTA) pairs][2][HPC][gh * q_len], pair k * group_ctas + c
  float* ws_o;         // [..][128] normalised partial outputs
  float* ws_lse;       // base-2 lse of the partials (NaN = bad piece)
  uint32_t* err_flags; // or nullptr
  uint32_t epoch;      // nonzero, different for every host call
  // Shared-prefix decode (zero otherwise): the first prefix_tiles tiles of
  // every sequence are the same pages. Groups of sgs sequences (ng groups)
  // attend to them together. A unit one CTA finishes leaves each query row's
  // result over its part in pre_* (prefix) or suf_* (the rest): fp32
  // normalised output [B, q_len, Hq, 128] and base-2 lse [B, q_len, Hq].
  int prefix_tiles, sgs, ng;
  float* pre_o;
  float* pre_lse;
  float* suf_o;
  float* suf_lse;
  int test_stall;      // failure-detection test hook: stall the producer until its wait runs out
  int B, q_len, Hq, Hkv, g, page_size, num_pages;
  // Query tokens: q_total per sequence (q, out and lse rows are [B, q_total,
  // Hq]). A launch covers ngroups groups of up to q_len tokens starting at
  // q_tok0: CTAs [k * group_ctas, (k + 1) * group_ctas) take group k, tokens
  // [q_tok0 + k * q_len, + q_len) (fewer in the last group), and cut the same
  // tile line (every sequence's whole context) so that the groups read each
  // K/V tile at about the same time. With ngroups = 1 the line ends where the
  // group's last token stops seeing.
  int q_total, q_tok0, ngroups, group_ctas;
  // Query heads per row group (gh <= 16) and head chunks per kv head: with g <=
  // 16 a group holds all g heads of its tokens (gh = g, hchunks = 1); with g >
  // 16 each token's g heads go in hchunks = ceil(g / 16) chunks of gh heads
  // (the last may have fewer), one token per group. Group k of a launch is
  // token group (hc0 + k) / hchunks (counted from q_tok0) and head chunk
  // (hc0 + k) % hchunks.
  int gh, hchunks, hc0;
  // Token groups per CTA (1 or 2). With 2, every CTA takes both groups of a
  // two-group launch (consumer warp w: kv head w % hpc, group w / hpc), so a
  // K/V stage serves both; group_ctas is then the whole grid, and group k's
  // CTA c is counted as CTA k * group_ctas + c for its partial slots.
  int tg;
  // 1: CTA c takes unit c (sequence c / nhg, head group c % nhg) whole, so no
  // unit is cut and there is nothing to merge (the host picks this for short
  // contexts, where a merge launch would cost more than the attention).
  int unit_cut;
  // 1: the grid is the default one and the host knew no length bound; the
  // kernels then choose the unit cut above themselves, from seq_lens, when
  // every unit is short and the units fit in the group's CTAs (the attention
  // and merge kernels take the same decision from the same lengths).
  int auto_cut;
  int hpc;             // kv heads per CTA
  int nhg;             // Hkv / hpc head groups
  float scale_log2;    // scale * log2(e)
  // Fused KV append (k_new = nullptr: none). The new tokens' rows [B, q_total,
  // Hkv, 128] bf16 as 16-byte chunks; before loading a tile that holds new
  // tokens, the producer warp stores their rows of the CTA's kv heads into the
  // pools (raw pointers, strides in 16-byte chunks).
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_pool;
  uint4* v_pool;
  int64_t page_stride16, token_stride16, head_stride16;
};

constexpr int kMlaTile = 64;       // tokens per MLA tile (page sizes are multiples of it)
constexpr int kMlaDqk = 576;       // latent 512 + rope 64
constexpr int kMlaDv = 512;        // V = first 512 latent columns
constexpr int kMlaHeads = 128;     // query heads (= TMEM lanes)
constexpr int kMlaMaxBatch = 1024; // (sequence, query token) pairs per MLA call
constexpr int kMlaUnitCost = 4;     // extra cost of a unit (Q load, epilogue) in tiles, for the split

// Everything the MLA kernel and its merge kernel read.
struct MlaParams {
  CUtensorMap tmap_kv;  // 3-D {576, page_size, num_pages}, box {64, 64, 1}, 128B swizzle
  const __nv_bfloat16* q;  // [B, q_len, 128, 576]
  __nv_bfloat16* out;   // [B, q_len, 128, 512]
  float* lse;           // [B, q_len, 128] natural log, or nullptr
  const int32_t* block_table;
  const int32_t* seq_lens;
  int64_t bt_stride;
  int32_t* ws_prefix;   // [B + 1] tile prefix sums
  int32_t* ws_split;    // [clusters + 1] first tile of each cluster's range
  int32_t* ws_span;     // [B][2] first and last cluster holding tiles of each unit
  float* ws_o;          // [clusters][2][128][512] normalised partial outputs (fp32)
  float* ws_lse;        // [clusters][2][128] base-2 lse of partials (NaN = bad piece)
  uint32_t* err_flags;
  int B, q_len, page_size, num_pages;
  float scale_log2;
  int out_align32;      // out is 32-byte aligned: 32-byte stores
  // Fused KV append (kv_new = nullptr: none): the new tokens' latent rows
  // [B, q_len, 576] bf16 as 16-byte chunks; each producer warp stores the
  // columns it loads of the new tokens its cluster's tiles hold, before its
  // first load (raw pool pointer, strides in 16-byte chunks).
  const uint4* kv_new;
  uint4* kv_pool;
  int64_t page_stride16, token_stride16;
};

size_t mla_smem_bytes();
// Launches `clusters` CTA pairs of the MLA kernel, then its merge kernel.
cudaError_t mla_decode_launch(const MlaParams& p, int clusters, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end);

// kv heads handled by one CTA for this Hkv (largest of 8, 4, 2, 1 dividing it).
int gqa_heads_per_cta(int Hkv);
// CTAs of the attention kernel that fit on one SM (0 on error); small: the
// call's units + 1 fit the small table (at most kSmallTable entries).
int gqa_ctas_per_sm(int hpc, bool rows16, bool causal, bool fused, int tg, bool small,
                    int device);
// Shared-prefix decode: CTAs per SM of its attention kernel, and its two
// launches (attention over prefix groups and suffixes, then the merge).
int gqa_shared_ctas_per_sm(int hpc, bool rows16, bool causal, bool small, int device);
cudaError_t gqa_shared_launch(const GqaParams& p, int grid, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end);
// Launches the attention kernel on `grid` CTAs. fused: split units are merged
// inside it (one launch); otherwise a merge kernel follows as a programmatic
// dependent launch.
cudaError_t gqa_decode_launch(const GqaParams& p, int grid, bool fused, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end);

}  // namespace zl
