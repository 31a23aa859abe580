// Paged GQA decode attention for sm_103a: one persistent wave of CTAs, each a
// TMA producer warp plus one tensor-core consumer warp per kv head.
//
// Work decomposition. For sequence b the context is cut into n_b tiles of 16
// tokens. The tiles of all (sequence, kv-head-group) units are laid end to end
// and the line is cut into min(G, tiles) equal ranges, one per CTA ("split-KV" of the
// flash_decoding family named under "技术架构：五层模块化设计" on the
// "ZhiLight：知乎开源的高性能 LLM 推理加速引擎" page). A CTA whose range covers a
// whole unit writes the final output; a unit cut between CTAs leaves one
// normalised partial (o, lse) per CTA in the workspace, and the merge kernel
// that follows (a programmatic dependent launch) combines them by
// log-sum-exp in CTA order. With FUSED the attention kernel merges instead:
// each consumer warp that writes a partial counts its arrival on the
// (sequence, kv head) counter and the last to arrive merges, in the same CTA
// order, so the result does not depend on which CTA finished last. Either way
// the cut depends only on seq_lens and G, so results are deterministic and
// bit-identical under page remapping. MODE kModeShared adds units that cover a
// shared prefix for a group of sequences at once (see gqa_prefix.cu).
//
// Per tile (16 tokens x HPC kv heads), the producer issues four TMA loads (K
// and V, two 64-column halves each, 128-byte swizzled) into a ring of
// shared-memory stages guarded by mbarriers. Consumer warp w owns kv head w of
// the group: its g query heads are the rows of an m16n8k16 tensor-core tile
// ("fused batch attention for decoding using tensor core instructions", the
// "ZhiLight: Zhihu's CUDA Inference Engine..." page, "Dual streams, host
// all-reduce and the memory model"), S = Q K^T and O += P V run on mma.sync,
// and the online softmax (a lazily moved base, the sum) stays in registers
// with quad shuffles. With q_len > 1 query tokens per sequence the rows are
// the (token, head) pairs, at most 16 per row group (more rows go in several
// groups), each with its causal limit (the CAUSAL instances; q_len = 1 runs
// the instances without the limit).
#pragma once

#include "kernels.h"
#include "ptx.cuh"

#include <math_constants.h>

namespace zl {

namespace {

constexpr uint32_t kErrBadPage = 1u;
constexpr uint32_t kErrBadLen = 2u;
constexpr uint32_t kErrTimeout = 4u;
constexpr uint32_t kErrBadPrefix = 8u;
constexpr int kMergeRows = 4;  // rows one warp merges together (single launch; large merges)

// What one launch of the attention kernel covers.
constexpr int kModePlain = 0;   // every sequence over all of its own pages
// Shared prefix: units (group of sgs sequences, head group) over the prefix
// tiles, then units (sequence, head group) over each sequence's tiles past
// the prefix, on one tile line; whole units leave fp32 results in the prefix
// and suffix stores, and the merge kernel combines both parts of every row.
constexpr int kModeShared = 1;
constexpr uint64_t kTestStallNs = 50ull * 1000 * 1000;  // bound of the test-hook wait
// A row's softmax base moves only when a tile's scores exceed it by more than
// this (base 2): P stays at most 2^8 in between.
constexpr float kLazyLog2 = 8.f;

template <int HPC, int TG = 1>
struct GqaCfg {
  static constexpr int kHalfBytes = HPC * kGqaTile * 64 * 2;  // one 64-column half of K or V
  static constexpr int kStageBytes = 4 * kHalfBytes;           // K lo | K hi | V lo | V hi
  // Two row groups per CTA: six stages, and as many CTAs per SM as make 8
  // consumer warps (one at HPC = 4, four at HPC = 1), so that an SM has
  // 192 KB of stages in flight and 8 consumer warps to hide each tile's
  // latency, as at HPC = 8.
  static constexpr int kStages = TG > 1 ? 6 : HPC == 8 ? 3 : HPC == 4 ? 4 : HPC == 2 ? 6 : 8;
  static constexpr int kConsumers = HPC * TG;  // consumer warps
  static constexpr int kThreads = (kConsumers + 1) * 32;
  static constexpr int kMinBlocks = TG > 1 && kConsumers < 8 ? 8 / kConsumers : 1;
  // 1 KB alignment slack + stages + barriers + per-stage flags + abort flag and
  // longest unit + split-piece records (2 per consumer warp); then the table of
  // per-unit tile offsets, sized for the call (see table_entries).
  static constexpr size_t kFixedBytes = 1024 + size_t(kStages) * kStageBytes + kStages * 16 +
                                        kStages * 4 + 16 + kConsumers * 2 * 4;
  static constexpr size_t smem_bytes(bool small_table) {
    return kFixedBytes + size_t(small_table ? kSmallTable : kMaxBatch + 1) * 4;
  }
  static constexpr size_t kSmemBytes = smem_bytes(false);  // the largest, for the attribute
};

// Entries of the tile-offset table a launch needs (one per unit plus the
// total), and whether they fit the small layout. A call with up to
// kSmallTable - 1 units takes the small one: at one kv head per CTA that
// leaves room for a fourth CTA on an SM (4 x 51 KB instead of 4 x 65 KB).
__host__ __device__ __forceinline__ int table_entries(const GqaParams& p, int mode) {
  return (mode == kModeShared ? p.ng : 0) + p.B + 1;
}
__host__ __device__ __forceinline__ bool small_table(const GqaParams& p, int mode) {
  return table_entries(p, mode) <= kSmallTable;
}

__device__ __forceinline__ void raise_error(uint32_t* flags, uint32_t bits) {
  if (flags) atomicOr(flags, bits);
}

// Index of the sequence whose tile range contains global tile `idx`:
// the largest b with nhg * prefix[b] <= idx (sequences with no tiles are skipped
// because the next prefix equals theirs).
__device__ __forceinline__ int locate_seq(const int* prefix, int B, int nhg, int64_t idx) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (int64_t(nhg) * prefix[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// First tile of CTA cc's range when W tiles are cut into G ranges
// [floor(cc W / G), floor((cc+1) W / G)), from Wq = W / G and Wr = W % G:
// floor(cc W / G) = cc Wq + floor(cc Wr / G), and cc Wr < G^2 < 2^32 (G is
// at most 65535), so no 64-bit division is needed. The launches cut into
// G = min(CTAs, W) ranges (at least 1), so every range below G holds a tile:
// a unit cut between CTAs c_lo..c_hi has exactly c_hi - c_lo + 1 pieces, and
// owner() finds c_lo and c_hi without walking the CTAs.
struct TileCut {
  int64_t Wq;
  uint32_t Wr, G;
  __device__ __forceinline__ TileCut(int64_t W, int ctas) {
    const int64_t g = W < int64_t(ctas) ? (W > 0 ? W : 1) : int64_t(ctas);
    G = uint32_t(g);
    Wq = W / g;
    Wr = uint32_t(W % g);
  }
  __device__ __forceinline__ int64_t start(int cc) const {
    return int64_t(cc) * Wq + int64_t((uint32_t(cc) * Wr) / G);
  }
  // The CTA whose range holds tile x: the largest cc with start(cc) <= x,
  // i.e. ceil((x + 1) G / W) - 1.
  __device__ __forceinline__ int owner(int64_t x) const {
    const int64_t W = Wq * G + Wr;
    return int(((x + 1) * int64_t(G) + W - 1) / W) - 1;
  }
};

// Whether every unit of the launch is short enough for a CTA of its own (the
// unit cut): at most kGqaUnitCutTiles tiles in the longest unit (n_max), and
// no more units than the group's CTAs.
__device__ __forceinline__ bool short_units(int64_t units, int n_max, int ctas) {
  return units <= ctas && n_max <= kGqaUnitCutTiles;
}

// 64-bit compare-and-swap with acquire-release semantics at GPU scope: the
// arriving warp's partial rows (ordered before it by __syncwarp) are released
// with its arrival, and the last arrival acquires everyone else's.
__device__ __forceinline__ unsigned long long cas_acq_rel(unsigned long long* addr,
                                                          unsigned long long cmp,
                                                          unsigned long long val) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;"
               : "=l"(old)
               : "l"(addr), "l"(cmp), "l"(val)
               : "memory");
  return old;
}

__device__ __forceinline__ void st_relaxed(unsigned long long* addr, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(addr), "l"(v) : "memory");
}

// Count one arrival on a split unit's counter (epoch << 32 | count; a word
// from another epoch counts as 0, so a call that stopped early cannot confuse
// the next one). Returns true for the last of `pieces` arrivals, which also
// puts the word back to 0. The first CAS guesses the usual state of a unit's
// first arrival (a zero word), so that arrival costs one round trip. The CAS
// retries only while other CTAs update the same word; the bound is a guard,
// never reached by a correct schedule.
__device__ __forceinline__ bool arrive_last(unsigned long long* word, uint32_t epoch, int pieces,
                                            uint32_t* err_flags) {
  unsigned long long old = 0ull;
  for (int tries = 0; tries < (1 << 20); ++tries) {
    const uint32_t cnt = uint32_t(old >> 32) == epoch ? uint32_t(old) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
    const unsigned long long seen = cas_acq_rel(word, old, want);
    if (seen == old) {
      if (int(cnt + 1u) < pieces) return false;
      st_relaxed(word, 0ull);
      return true;
    }
    old = seen;
  }
  raise_error(err_flags, kErrTimeout);
  return false;
}

// The CTAs holding pieces of a split unit (first tile U0, n tiles): c_lo owns
// tile U0, c_hi the last tile. Every range holds a tile, so each CTA from
// c_lo to c_hi has one piece; returns their number.
__device__ __forceinline__ int split_cta_span(const TileCut& cut, int64_t U0, int n, int& c_lo,
                                              int& c_hi) {
  c_lo = cut.owner(U0);
  c_hi = cut.owner(U0 + n - 1);
  return c_hi - c_lo + 1;
}

// Split-KV merge. The R rows of kv head w (of CTA head group hg) are merged
// over the pieces of a split unit by the warp whose arrival was the last
// (single launch, NR = kMergeRows rows per warp) or by the merge kernel (NR =
// 1 or kMergeRows): a running max and rescaled sums per row, always in CTA
// order, so the result depends neither on who merges nor on how many rows a
// warp takes. Pieces go in batches of P: a lane loads every row's lse and its
// own 4 columns of every row of a batch at once, so a batch costs one round
// trip to L2. Merging the same pieces with any batch size gives the same bits.

// Running log-sum-exp merge of NR rows (base-2 lse): a running max, the
// rescaled weight sum and the rescaled sum of normalised outputs. A source row
// with lse NaN (its piece met a bad page) marks that row bad (bit k of
// `bad`); lse -inf weighs 0.
template <int NR>
struct MergeAcc {
  float mx[NR], den[NR];
  float4 acc[NR];
  uint32_t bad;
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      mx[k] = -CUDART_INF_F;
      den[k] = 0.f;
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    bad = 0u;
  }
  // Every product and sum is rounded as written (no contraction left to the
  // compiler), so the bits do not depend on the code around an inlined copy.
  __device__ __forceinline__ void add(int k, float l, float4 o) {
    bad |= isnan(l) ? 1u << k : 0u;
    const float mn = fmaxf(mx[k], l);
    if (mn != -CUDART_INF_F && !isnan(l)) {
      const float a = ex2_approx(__fsub_rn(mx[k], mn)), wgt = ex2_approx(__fsub_rn(l, mn));
      den[k] = __fmaf_rn(den[k], a, wgt);
      acc[k].x = __fmaf_rn(wgt, o.x, __fmul_rn(acc[k].x, a));
      acc[k].y = __fmaf_rn(wgt, o.y, __fmul_rn(acc[k].y, a));
      acc[k].z = __fmaf_rn(wgt, o.z, __fmul_rn(acc[k].z, a));
      acc[k].w = __fmaf_rn(wgt, o.w, __fmul_rn(acc[k].w, a));
      mx[k] = mn;
    }
  }
};

// Adds the partials of rows [row_off + r0, row_off + r0 + nrows) (slot stride
// R) of the pieces of a unit (first tile U0) held by CTAs c_lo..c_hi, in CTA
// order; pieces go in batches of P whose loads are issued together (one L2
// round trip per batch). Every CTA in c_lo..c_hi holds a piece (the launches
// cut into at most as many ranges as tiles, so no range is empty); each
// piece is its CTA's first (slot 0) except where the unit starts inside c_lo's
// range (slot 1).
template <int NR, int P>
__device__ __forceinline__ void merge_add_pieces(MergeAcc<NR>& m, const GqaParams& p,
                                                 const TileCut& cut, int cta0, int64_t U0,
                                                 int c_lo, int c_hi, int w, int R, int row_off,
                                                 int r0, int nrows, int lane) {
  const int sl_lo = U0 > cut.start(c_lo) ? 1 : 0;
  for (int cb = c_lo; cb <= c_hi; cb += P) {
    float lv[P][NR];
    float4 ov[P][NR];
#pragma unroll
    for (int q = 0; q < P; ++q) {
      const int cc = cb + q;
      const int sl = cc == c_lo ? sl_lo : 0;
      const int64_t base = ((int64_t(cta0 + cc) * 2 + sl) * p.hpc + w) * R + row_off + r0;
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        if (cc <= c_hi && k < nrows) {
          lv[q][k] = __ldcg(p.ws_lse + base + k);
          ov[q][k] =
              __ldcg(reinterpret_cast<const float4*>(p.ws_o + (base + k) * kGqaHeadDim) + lane);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < P; ++q)
#pragma unroll
      for (int k = 0; k < NR; ++k)
        if (cb + q <= c_hi && k < nrows) m.add(k, lv[q][k], ov[q][k]);
  }
}

// Adds rows (sequence b, tile rows r0 + k of gh * q_len: token r / gh, head
// head0 + r % gh) from an fp32 store of whole-unit results.
template <int NR>
__device__ __forceinline__ void merge_add_store(MergeAcc<NR>& m, const GqaParams& p,
                                                const float* st_o, const float* st_lse, int b,
                                                int tok0, int head0, int gh, int r0, int nrows,
                                                int lane) {
  float lv[NR];
  float4 ov[NR];
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    if (k < nrows) {
      const int r = r0 + k;
      const int64_t orow = (int64_t(b) * p.q_total + tok0 + r / gh) * p.Hq + head0 + r % gh;
      lv[k] = __ldcg(st_lse + orow);
      ov[k] = __ldcg(reinterpret_cast<const float4*>(st_o + orow * kGqaHeadDim) + lane);
    }
  }
#pragma unroll
  for (int k = 0; k < NR; ++k)
    if (k < nrows) m.add(k, lv[k], ov[k]);
}

// Writes the merged rows of sequence b (row r: token tok0 + r / gh, head
// head0 + r % gh) as bf16 out and natural-log lse; a bad source or a row with
// no weight gives zeros and lse = -inf.
template <int NR>
__device__ __forceinline__ void merge_write_out(const MergeAcc<NR>& m, const GqaParams& p, int b,
                                                int tok0, int head0, int gh, int r0, int nrows,
                                                int lane) {
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    if (k < nrows) {
      const int r = r0 + k;
      const int64_t orow = (int64_t(b) * p.q_total + tok0 + r / gh) * p.Hq + head0 + r % gh;
      const bool none = ((m.bad >> k) & 1u) || !(m.den[k] > 0.f);
      const float inv = none ? 0.f : __frcp_rn(m.den[k]);
      uint2 packed = make_uint2(0u, 0u);
      if (!none) {
        packed.x = pack_bf16x2(__fmul_rn(m.acc[k].x, inv), __fmul_rn(m.acc[k].y, inv));
        packed.y = pack_bf16x2(__fmul_rn(m.acc[k].z, inv), __fmul_rn(m.acc[k].w, inv));
      }
      reinterpret_cast<uint2*>(p.out + orow * kGqaHeadDim)[lane] = packed;
      if (p.lse && lane == 0)
        p.lse[orow] = none ? -CUDART_INF_F
                           : __fmul_rn(__fadd_rn(m.mx[k], log2f(m.den[k])), 0.69314718055994531f);
    }
  }
}

// A plain unit (sequence b, kv head w of the CTA group, first tile U0) cut
// between CTAs c_lo..c_hi: merge rows [r_begin, r_end), NR at a time, and
// write them.
template <int NR, int P>
__device__ __forceinline__ void merge_split_rows(const GqaParams& p, const TileCut& cut, int cta0,
                                                 int64_t U0, int c_lo, int c_hi, int b, int tok0,
                                                 int w, int head0, int gh, int R, int r_begin,
                                                 int r_end, int lane) {
  for (int r0 = r_begin; r0 < r_end; r0 += NR) {
    const int nrows = min(NR, r_end - r0);
    MergeAcc<NR> m;
    m.init();
    merge_add_pieces<NR, P>(m, p, cut, cta0, U0, c_lo, c_hi, w, R, 0, r0, nrows, lane);
    merge_write_out(m, p, b, tok0, head0, gh, r0, nrows, lane);
  }
}

// Tiles of sequence b's own unit for this launch (seq_lens[b] = L): they end
// where the launch's last query token stops seeing, L - (q_total - q_tok0 -
// q_len) tokens; a shared-prefix launch leaves out the prefix tiles. An
// invalid length (negative, or more tokens than the block table maps) has none.
template <int MODE>
__device__ __forceinline__ int seq_unit_tiles(const GqaParams& p, int L) {
  const int64_t cap = p.bt_stride * int64_t(p.page_size);
  if (!(L >= 0 && int64_t(L) <= cap)) return 0;
  const int unseen = p.ngroups > 1 ? 0 : p.q_total - p.q_tok0 - p.q_len;
  const int t = (L - unseen + kGqaTile - 1) / kGqaTile - (MODE == kModeShared ? p.prefix_tiles : 0);
  return t > 0 ? t : 0;
}

// Row group k of a launch: query tokens [tok0, tok0 + qlen) and, of each kv
// head's g query heads, heads [hoff, hoff + gh). Tile row r of the group is
// token tok0 + r / gh, head hoff + r % gh.
struct RowGroup {
  int tok0, qlen, hoff, gh;
};
__device__ __forceinline__ RowGroup row_group(const GqaParams& p, int k) {
  const int gg = p.hc0 + k;
  const int tt = gg / p.hchunks, hc = gg - tt * p.hchunks;
  RowGroup r;
  r.tok0 = p.q_tok0 + tt * p.q_len;
  r.qlen = min(p.q_len, p.q_total - r.tok0);
  r.hoff = hc * p.gh;
  r.gh = min(p.gh, p.g - r.hoff);
  return r;
}

// Fused KV append, by the 32 lanes of a producer warp: new tokens [inew,
// inew + nn) of sequence b, which sit in slots [slot0, slot0 + nn) of page pg,
// for kv heads [kh0, kh0 + HPC): their K and V rows (16 chunks of 16 bytes
// each) are copied from k_new / v_new into the pools. Each lane then fences
// its stores against the bulk copies that read the page next.
template <int HPC>
__device__ __forceinline__ void append_tile_rows(const GqaParams& p, int b, int pg, int slot0,
                                                 int inew, int nn, int kh0, int lane) {
  constexpr int kChunks = kGqaHeadDim * 2 / 16;
  const int total = nn * HPC * 2 * kChunks;
  for (int c0 = 0; c0 < total; c0 += 4 * 32) {
    uint4 v[4];
    uint4* dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + 32 * u + lane;
      dst[u] = nullptr;
      if (c < total) {
        const int cc = c % kChunks, row = c / kChunks;  // row = (j * HPC + hh) * 2 + (K or V)
        const bool is_v = row & 1;
        const int hh = (row >> 1) % HPC, j = (row >> 1) / HPC;
        const int64_t src =
            ((int64_t(b) * p.q_total + inew + j) * p.Hkv + kh0 + hh) * kChunks + cc;
        v[u] = __ldg((is_v ? p.v_new : p.k_new) + src);
        dst[u] = (is_v ? p.v_pool : p.k_pool) + int64_t(pg) * p.page_stride16 +
                 int64_t(slot0 + j) * p.token_stride16 + int64_t(kh0 + hh) * p.head_stride16 +
                 cc;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
  fence_proxy_async_global();
}

template <int HPC, bool ROWS16, bool CAUSAL, bool FUSED, int MODE = kModePlain, int TG = 1>
__global__ void __launch_bounds__(GqaCfg<HPC, TG>::kThreads, GqaCfg<HPC, TG>::kMinBlocks)
gqa_decode_kernel(const __grid_constant__ GqaParams p) {
  static_assert(MODE == kModePlain || !FUSED, "the in-kernel merge is for plain launches");
  static_assert(TG == 1 || (MODE == kModePlain && !FUSED && CAUSAL),
                "two row groups per CTA: plain launches, causal instances, merge launch");
  using Cfg = GqaCfg<HPC, TG>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128B swizzle wants 1 KB-aligned stages
  uint8_t* smem = smem_raw + (sbase - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * Cfg::kStageBytes);
  uint64_t* empty = full + NS;
  int* stage_bad = reinterpret_cast<int*>(empty + NS);
  volatile int* abort_flag = stage_bad + NS;
  int* unit_max = stage_bad + NS + 1;   // tiles of the longest unit
  int* split_rec = stage_bad + NS + 4;  // [HPC][2]: b | hg << 12 of a split piece, or -1
  int* prefix = split_rec + Cfg::kConsumers * 2;  // table_entries(p, MODE) entries

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B;
  const int64_t cap = p.bt_stride * int64_t(p.page_size);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), Cfg::kConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == Cfg::kConsumers && lane == 0) {
    tma_prefetch_desc(&p.tmap_k);
    tma_prefetch_desc(&p.tmap_v);
  }
  // Launched as a programmatic dependent of whatever kernel precedes it on the
  // stream (e.g. the KV append): everything above overlaps that kernel's tail;
  // nothing in global memory is read or written before it has finished.
  griddep_wait();

  // Units of this launch (one "virtual sequence" v each per head group):
  // plain, v = sequence; shared prefix, v < ng a group of sgs sequences over
  // the prefix tiles, v >= ng sequence v - ng over its tiles past the prefix.
  // Their tiles and the exclusive prefix sum (warp 0).
  const int PT = p.prefix_tiles;
  const int NG = MODE == kModeShared ? p.ng : 0;
  const int V = NG + B;
  auto unit_tiles = [&](int v) -> int {
    return v < NG ? PT : seq_unit_tiles<MODE>(p, p.seq_lens[v - NG]);
  };
  if (warp == 0) {
    const int per = (V + 31) / 32;
    const int v0 = lane * per;
    int local = 0, nmax = 0;
    for (int i = 0; i < per; ++i) {
      const int v = v0 + i;
      if (v < V) {
        if (v >= NG && blockIdx.x == 0) {
          const int L = p.seq_lens[v - NG];
          if (!(L >= 0 && int64_t(L) <= cap)) raise_error(p.err_flags, kErrBadLen);
        }
        const int n = unit_tiles(v);
        local += n;
        nmax = max(nmax, n);
      }
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += x;
      nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, off));
    }
    if (lane == 0) unit_max[0] = nmax;
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int v = v0 + i;
      if (v < V) {
        prefix[v] = run;
        run += unit_tiles(v);
      }
    }
    if (lane == 31) prefix[V] = incl;
  } else if (MODE == kModeShared && warp == 1) {
    // The caller states that every sequence starts with the same prefix_tiles
    // tiles of pages and that every query row sees all of them; CTA c checks
    // sequences c, c + G, ... and flags a violation (results are then void).
    const int ppages = PT * kGqaTile / p.page_size;
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
      int bad = 0;
      for (int j = lane; j < ppages; j += 32)
        bad |= p.block_table[int64_t(b) * p.bt_stride + j] != p.block_table[j] ? 1 : 0;
      const int L = p.seq_lens[b];
      if (lane == 0 && (int64_t(L) > cap || L - p.q_total + 1 < PT * kGqaTile)) bad = 1;
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(p.err_flags, kErrBadPrefix);
    }
  }
  __syncthreads();

  if constexpr (!FUSED) {
    // The merge kernel may be scheduled from here on (this grid is past its
    // own dependency wait); it waits for this whole grid to finish before it
    // reads any partial.
    griddep_launch_dependents();
  }

  // This warp's group of query tokens (tokens [tok0, tok0 + qlen)) and the
  // CTA's place c among the group's G CTAs, which cut the tile line between
  // them. One group per CTA: CTAs [tg G, (tg + 1) G) take group tg. Two per
  // CTA: every CTA takes both, consumer warp w group w / HPC. Either way
  // vcta = tg G + c numbers the (group, CTA) pairs for the partial slots.
  const int tg = TG > 1 ? min(warp / HPC, TG - 1) : int(blockIdx.x) / p.group_ctas;
  const int G = TG > 1 ? int(gridDim.x) : p.group_ctas;
  const int c = TG > 1 ? int(blockIdx.x) : int(blockIdx.x) - tg * p.group_ctas;
  const int vcta = tg * G + c;
  // the group's query tokens [tok0, tok0 + qlen) and heads [hoff, hoff + gh)
  // of each kv head's g
  const RowGroup rg = row_group(p, tg);
  const int tok0 = rg.tok0, qlen = rg.qlen, gh = rg.gh;
  const int nhg = p.nhg;
  const int64_t W = int64_t(nhg) * prefix[V];
  const TileCut cut(W, G);
  // CTAs past the cut's G (more CTAs than tiles) take no tiles.
  int64_t s_c = c < int(cut.G) ? cut.start(c) : W;
  int64_t e_c = c < int(cut.G) ? cut.start(c + 1) : W;
  const bool unit_cut =
      MODE == kModePlain &&
      (p.unit_cut || (p.auto_cut && short_units(int64_t(V) * nhg, unit_max[0], G)));
  if (unit_cut) {
    // Unit (v, hg) holds tiles [nhg * prefix[v] + hg * n, + n) of the line.
    s_c = e_c = 0;
    if (c < int64_t(V) * nhg) {
      const int v = c / nhg, n = prefix[v + 1] - prefix[v];
      s_c = int64_t(nhg) * prefix[v] + int64_t(c % nhg) * n;
      e_c = s_c + n;
    }
  }

  if (warp == Cfg::kConsumers) {
    // ------------------------------------------------------------ producer
    if (p.test_stall) {
      // Failure-detection test hook: wait on a word nothing sets until the
      // bound runs out, then stop the CTA the way a stalled pipeline does.
      __shared__ int never_set;
      if (lane == 0) {
        never_set = 0;
        if (!flag_wait(&never_set, kTestStallNs)) {
          raise_error(p.err_flags, kErrTimeout);
          *abort_flag = 1;
        }
      }
      __syncwarp();
      return;
    }
    int it = 0;
    bool aborted = false;
    for (int64_t base = s_c; base < e_c && !aborted; base += 32) {
      // lane i resolves tile base + i: page id, slot and head group
      const int64_t idx = base + lane;
      int page = 0, slot = 0, hg = 0, bad = 0;
      // fused append: new tokens the tile holds (count, index of the first
      // among the call's new tokens, its slot) and their sequence
      int nnew = 0, inew = 0, nslot = 0, nseq = 0;
      if (idx < e_c) {
        const int v = locate_seq(prefix, V, nhg, idx);
        const int n = prefix[v + 1] - prefix[v];
        const int64_t r = idx - int64_t(nhg) * prefix[v];
        hg = int(r / n);
        const bool pre = v < NG;  // a prefix unit
        const int tok0 = (MODE == kModeShared && !pre ? PT * kGqaTile : 0) + int(r % n) * kGqaTile;
        const int trow = pre ? v * p.sgs : v - NG;  // a block-table row to read
        slot = tok0 % p.page_size;
        page = p.block_table[int64_t(trow) * p.bt_stride + tok0 / p.page_size];
        bad = (page < 0 || page >= p.num_pages) ? 1 : 0;
        if (p.k_new && !pre) {
          const int L = p.seq_lens[trow];
          const int t0 = L - p.q_total;  // the call's first new token
          const int lo = max(tok0, t0), hi = min(tok0 + kGqaTile, L);
          if (t0 >= 0 && hi > lo) {
            nnew = hi - lo;
            inew = lo - t0;
            nslot = slot + (lo - tok0);
            nseq = trow;
          }
        }
      }
      const int cnt = int(min(int64_t(32), e_c - base));
      for (int k = 0; k < cnt; ++k, ++it) {
        const int pg = __shfl_sync(0xffffffffu, page, k);
        const int sl = __shfl_sync(0xffffffffu, slot, k);
        const int h = __shfl_sync(0xffffffffu, hg, k);
        const int bd = __shfl_sync(0xffffffffu, bad, k);
        const int nn = __shfl_sync(0xffffffffu, nnew, k);
        if (nn > 0 && !bd) {
          // Store the new tokens' rows of this CTA's kv heads before the tile's
          // loads (every CTA that loads the tile stores the same bytes).
          append_tile_rows<HPC>(p, __shfl_sync(0xffffffffu, nseq, k), pg,
                                __shfl_sync(0xffffffffu, nslot, k),
                                __shfl_sync(0xffffffffu, inew, k), nn, h * HPC, lane);
          __syncwarp();
        }
        int ok = 1;
        if (lane == 0) {
          const int stage = it % NS;
          const uint32_t phase = (it / NS) & 1;
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag)) {
            raise_error(p.err_flags, kErrTimeout);
            *abort_flag = 1;
            ok = 0;
          } else {
            stage_bad[stage] = bd;
            const uint32_t fb = smem_u32(&full[stage]);
            if (bd) {
              mbar_arrive(fb);  // nothing to load; the consumer discards this piece
            } else {
              const uint32_t dst = sbase + stage * Cfg::kStageBytes;
              mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
              tma_load_4d(dst, &p.tmap_k, fb, 0, sl, h * HPC, pg);
              tma_load_4d(dst + Cfg::kHalfBytes, &p.tmap_k, fb, 64, sl, h * HPC, pg);
              tma_load_4d(dst + 2 * Cfg::kHalfBytes, &p.tmap_v, fb, 0, sl, h * HPC, pg);
              tma_load_4d(dst + 3 * Cfg::kHalfBytes, &p.tmap_v, fb, 64, sl, h * HPC, pg);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          aborted = true;
          break;
        }
      }
    }
    // Do not leave the CTA with copies in flight: wait for the last stages.
    if (lane == 0) {
      const int first = it > NS ? it - NS : 0;
      for (int j = first; j < it; ++j) {
        const volatile int never = 0;
        mbar_wait(smem_u32(&full[j % NS]), (j / NS) & 1, &never);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int w = TG > 1 ? warp % HPC : warp;  // kv head within the CTA's head group
  const int gid = lane >> 2, t4 = lane & 3;
  const int g = p.g;
  const float scale_log2 = p.scale_log2;
  int it = 0;
  int64_t idx = s_c;
  if (lane == 0) split_rec[2 * w] = split_rec[2 * w + 1] = -1;
  while (idx < e_c) {
    const int v = locate_seq(prefix, V, nhg, idx);
    const int n = prefix[v + 1] - prefix[v];
    const int64_t unit_start0 = int64_t(nhg) * prefix[v];
    const int hg = int((idx - unit_start0) / n);
    const int j0 = int((idx - unit_start0) % n);
    const int64_t unit_end = unit_start0 + int64_t(hg + 1) * n;
    const int64_t piece_end = min(e_c, unit_end);
    const int ntiles = int(piece_end - idx);
    const bool partial = (j0 > 0) || (piece_end < unit_end);
    const int slot = (idx == s_c) ? 0 : 1;
    // The unit's (first) sequence: a prefix unit covers the sgs sequences b,
    // b + 1, ... (fewer in the last group), any other unit one sequence.
    const bool pre = v < NG;
    const int b = pre ? v * p.sgs : v - NG;
    // Tokens the unit's tiles cover end at L (a prefix unit: the whole prefix).
    const int L = pre ? PT * kGqaTile : p.seq_lens[b];
    const int head0 = (hg * HPC + w) * g + rg.hoff;  // the group's first query head
    // m16 tile rows are (sequence b + r / rps, query token i, head head0 + j)
    // with rps = gh * qlen rows per sequence, r % rps = i * gh + j; R rows per
    // partial slot (the largest group's), R_act of them exist, the rest are
    // zero. Query i (token tok0 + i of the q_total) sees tokens
    // t < L - q_total + 1 + tok0 + i (the new tokens are in the cache; each
    // sees itself and what precedes it); every row sees all of a shared prefix.
    const int rps = gh * qlen;
    const int R = MODE == kModeShared ? p.sgs * rps : p.gh * p.q_len;
    const int R_act = pre ? min(p.sgs, B - b) * rps : rps;
    const int ra = gid, rb = gid + 8;
    const int lim0 = L - p.q_total + 1 + tok0;
    const int lim_a = pre ? (1 << 30) : lim0 + ra / gh;
    const int lim_b = pre ? (1 << 30) : lim0 + rb / gh;
    auto qrow_index = [&](int r) -> int64_t {
      const int rr = r % rps;
      return (int64_t(b + r / rps) * p.q_total + tok0 + rr / gh) * p.Hq + head0 + rr % gh;
    };

    uint32_t qa[8][4];
    {
      const bool r0 = ra < R_act, r1 = ROWS16 && rb < R_act;
      const uint32_t* q0 =
          reinterpret_cast<const uint32_t*>(p.q + (r0 ? qrow_index(ra) : 0) * kGqaHeadDim);
      const uint32_t* q1 =
          reinterpret_cast<const uint32_t*>(p.q + (r1 ? qrow_index(rb) : 0) * kGqaHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int wd = ks * 8 + t4;  // 32-bit word index of d = 16ks + 2t4
        qa[ks][0] = r0 ? __ldg(q0 + wd) : 0u;
        qa[ks][2] = r0 ? __ldg(q0 + wd + 4) : 0u;
        qa[ks][1] = r1 ? __ldg(q1 + wd) : 0u;
        qa[ks][3] = r1 ? __ldg(q1 + wd + 4) : 0u;
      }
    }

    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
    float o[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    // Rows (a, b) of this thread whose visible tokens reach a tile over a bad
    // page: those rows, and only those, are written as zeros.
    bool bad_a = false, bad_b = false;

    // Online softmax in base 2 with a lazy base. Each row exponentiates
    // against a base m that moves only when a tile's max exceeds it by more
    // than kLazyLog2; then every row of the warp takes max(m, tile max) at once
    // (one vote per tile) and O and l are rescaled. Meanwhile P may reach
    // 2^kLazyLog2, well inside bf16 and fp32 range, and a tile costs no
    // rescale of the 64 O values a thread holds. The result is the same
    // softmax up to rounding; the lse is m + log2(l) with the final base.
    // This thread's four scores of a row (tokens 2t4, 2t4+1, 2t4+8, 2t4+9 of
    // the tile), scaled to base 2 with the tokens past vis masked to -inf,
    // and the row's max over the tile (a row that sees nothing gives -inf).
    auto row_scores = [&](float sa, float sb, float sc, float sd, int vis, float (&x)[4]) -> float {
      x[0] = 2 * t4 < vis ? sa * scale_log2 : -CUDART_INF_F;
      x[1] = 2 * t4 + 1 < vis ? sb * scale_log2 : -CUDART_INF_F;
      x[2] = 2 * t4 + 8 < vis ? sc * scale_log2 : -CUDART_INF_F;
      x[3] = 2 * t4 + 9 < vis ? sd * scale_log2 : -CUDART_INF_F;
      float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      return fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    };
    // Moves a row's base to mn >= m; returns the factor for its O and l (0
    // while the row has seen nothing).
    auto move_base = [&](float& m, float mn) -> float {
      const float alpha = m == -CUDART_INF_F ? 0.f : ex2_approx(m - mn);
      m = mn;
      return alpha;
    };
    // P of a row against its base (a row that has seen nothing has P = 0) and
    // its sum, taken over the bf16-rounded P that the PV product uses.
    auto row_p = [&](const float (&x)[4], float m, float& l, uint32_t& p_lo, uint32_t& p_hi) {
      const float base = m == -CUDART_INF_F ? 0.f : m;
      p_lo = pack_bf16x2(ex2_approx(x[0] - base), ex2_approx(x[1] - base));
      p_hi = pack_bf16x2(ex2_approx(x[2] - base), ex2_approx(x[3] - base));
      const float2 f0 = unpack_bf16x2(p_lo), f2 = unpack_bf16x2(p_hi);
      l += (f0.x + f0.y) + (f2.x + f2.y);
    };

    for (int t = 0; t < ntiles; ++t, ++it) {
      const int stage = it % NS;
      const uint32_t phase = (it / NS) & 1;
      const int tok0 = (MODE == kModeShared && !pre ? PT * kGqaTile : 0) + (j0 + t) * kGqaTile;
      const int valid = min(kGqaTile, L - tok0);  // tokens in the cache (V rows to keep)
      // every lane leaves together (the mma.sync below is warp-wide)
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, abort_flag))) {
        if (lane == 0) {
          raise_error(p.err_flags, kErrTimeout);
          *abort_flag = 1;
        }
        return;
      }
      if (stage_bad[stage]) {
        bad_a |= !CAUSAL || tok0 < lim_a;
        bad_b |= !CAUSAL || tok0 < lim_b;
      }
      const uint32_t kbase = sbase + stage * Cfg::kStageBytes + w * (kGqaTile * 128);
      const uint32_t vbase = kbase + 2 * Cfg::kHalfBytes;

      // S = Q K^T over the 16 tokens: two n8 tiles (tokens 0-7, 8-15).
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int tok = (lane & 7) + ((lane >> 4) << 3);
        const uint32_t row = kbase + tok * 128;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int chunk = ((ks & 3) << 1) + ((lane >> 3) & 1);
          const uint32_t addr = row + (ks >> 2) * Cfg::kHalfBytes + ((chunk ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma_bf16_16816(s[0], qa[ks], b0, b1);
          mma_bf16_16816(s[1], qa[ks], b2, b3);
        }
      }

      uint32_t pa[4];
      {
        float xa[4], xb[4];
        const float mxa = row_scores(s[0][0], s[0][1], s[1][0], s[1][1],
                                     CAUSAL ? min(valid, lim_a - tok0) : valid, xa);
        const float mxb = ROWS16 ? row_scores(s[0][2], s[0][3], s[1][2], s[1][3],
                                              CAUSAL ? min(valid, lim_b - tok0) : valid, xb)
                                 : -CUDART_INF_F;
        if (__any_sync(0xffffffffu, mxa > m0 + kLazyLog2 || mxb > m1 + kLazyLog2)) {
          const float aa = move_base(m0, fmaxf(m0, mxa));
          l0 *= aa;
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            o[nt][0] *= aa;
            o[nt][1] *= aa;
          }
          if (ROWS16) {
            const float ab = move_base(m1, fmaxf(m1, mxb));
            l1 *= ab;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
              o[nt][2] *= ab;
              o[nt][3] *= ab;
            }
          }
        }
        row_p(xa, m0, l0, pa[0], pa[2]);
        if (ROWS16) {
          row_p(xb, m1, l1, pa[1], pa[3]);
        } else {
          pa[1] = pa[3] = 0u;
        }
      }

      // O += P V. Token rows of V past the cache end are zeroed in registers so
      // that NaN in unused slots cannot reach the output (0 * NaN = NaN).
      {
        const bool v00 = 2 * t4 < valid, v01 = 2 * t4 + 1 < valid;
        const bool v10 = 2 * t4 + 8 < valid, v11 = 2 * t4 + 9 < valid;
        const uint32_t m01 = (v00 ? 0x0000ffffu : 0u) | (v01 ? 0xffff0000u : 0u);
        const uint32_t m89 = (v10 ? 0x0000ffffu : 0u) | (v11 ? 0xffff0000u : 0u);
        const int tok = (lane & 7) + (((lane >> 3) & 1) << 3);
        const uint32_t row = vbase + tok * 128;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int chunk = ((jj & 3) << 1) + (lane >> 4);
          const uint32_t addr = row + (jj >> 2) * Cfg::kHalfBytes + ((chunk ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(addr, b0, b1, b2, b3);
          if (valid < kGqaTile) {
            b0 &= m01;
            b1 &= m89;
            b2 &= m01;
            b3 &= m89;
          }
          mma_bf16_16816(o[2 * jj], pa, b0, b1);
          mma_bf16_16816(o[2 * jj + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
    }

    // ---- finalize the piece
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if (ROWS16) {
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    if (__any_sync(0xffffffffu, bad_a || bad_b) && lane == 0) raise_error(p.err_flags, kErrBadPage);
#pragma unroll
    for (int half = 0; half < (ROWS16 ? 2 : 1); ++half) {
      const int r = half ? rb : ra;
      if (r >= R_act) continue;
      const float l = half ? l1 : l0;
      const float m = half ? m1 : m0;
      const bool bad = half ? bad_b : bad_a;
      // A row whose piece met a bad page, or a row that saw no token, is
      // written as zeros with lse = -inf (weight 0 in the merge).
      const bool none = bad || !(l > 0.f);
      const float inv = none ? 0.f : 1.f / l;
      const float lse2 = none ? -CUDART_INF_F : m + log2f(l);
      if (!partial && MODE == kModeShared) {
        // a whole unit: the row's result over this part (prefix or suffix),
        // for the merge kernel to combine
        const int64_t orow = qrow_index(r);
        float* st_o = pre ? p.pre_o : p.suf_o;
        float* st_lse = pre ? p.pre_lse : p.suf_lse;
        float2* dst = reinterpret_cast<float2*>(st_o + orow * kGqaHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[nt * 4 + t4] = none ? make_float2(0.f, 0.f)
                                  : make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (t4 == 0) st_lse[orow] = bad ? CUDART_NAN_F : lse2;
      } else if (!partial) {
        const int64_t orow = qrow_index(r);
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + orow * kGqaHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[nt * 4 + t4] =
              none ? 0u : pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (p.lse && t4 == 0) p.lse[orow] = lse2 * 0.69314718055994531f;
      } else {
        // partial slots are per (token group, CTA) pair: every group has its own
        const int64_t wrow = ((int64_t(vcta) * 2 + slot) * HPC + w) * R + r;
        float2* dst = reinterpret_cast<float2*>(p.ws_o + wrow * kGqaHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[nt * 4 + t4] = none ? make_float2(0.f, 0.f)
                                  : make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (t4 == 0) p.ws_lse[wrow] = bad ? CUDART_NAN_F : lse2;
      }
    }
    // A split piece is merged after the CTA's range is done (its partner
    // pieces finish about then too); only its (b, hg) is kept meanwhile.
    if (FUSED && partial && lane == 0) split_rec[2 * w + slot] = b | (hg << 12);
    idx = piece_end;
  }
  // This warp's split pieces (at most two: the range's first and last) are
  // written; count both arrivals at once (lane sl takes record sl; the CAS
  // releases the rows the warp wrote before __syncwarp), then merge the units
  // this warp completed. Without FUSED the merge kernel does it.
  if constexpr (FUSED) {
  __syncwarp();
  int job = -1;
  if (lane < 2) {
    const int rec = split_rec[2 * w + lane];
    if (rec >= 0) {
      const int b = rec & 4095, hg = rec >> 12;
      const int n = prefix[b + 1] - prefix[b];
      int c_lo, c_hi;
      const int pieces = split_cta_span(cut, int64_t(nhg) * prefix[b] + int64_t(hg) * n, n,
                                        c_lo, c_hi);
      if (arrive_last(p.ws_count + int64_t(b) * p.Hkv + hg * HPC + w, p.epoch, pieces,
                      p.err_flags))
        job = rec;
    }
  }
  for (int sl = 0; sl < 2; ++sl) {
    const int rec = __shfl_sync(0xffffffffu, job, sl);
    if (rec < 0) continue;
    const int b = rec & 4095, hg = rec >> 12;
    const int n = prefix[b + 1] - prefix[b];
    const int64_t U0 = int64_t(nhg) * prefix[b] + int64_t(hg) * n;
    int c_lo, c_hi;
    split_cta_span(cut, U0, n, c_lo, c_hi);
    merge_split_rows<kMergeRows, 4>(p, cut, vcta - c, U0, c_lo, c_hi, b, tok0, w,
                                    (hg * HPC + w) * g + rg.hoff, gh, p.gh * p.q_len, 0,
                                    gh * qlen, lane);
  }
  }

  if constexpr (MODE == kModePlain) {
    // Sequences with no tiles (empty or invalid length): zeros, lse = -inf,
    // for every head of the tokens of the CTA's groups: [ztok0, + zlen).
    const RowGroup zlast = row_group(p, TG - 1);
    const int ztok0 = TG > 1 ? row_group(p, 0).tok0 : tok0;
    const int zlen = TG > 1 ? zlast.tok0 + zlast.qlen - ztok0 : qlen;
    constexpr int kStride = Cfg::kConsumers * 32;  // the consumer threads
    for (int b = c; b < B; b += G) {
      if (prefix[b + 1] != prefix[b]) continue;
      const int64_t rows = int64_t(zlen) * p.Hq;
      const int64_t row0 = (int64_t(b) * p.q_total + ztok0) * p.Hq;
      uint4* dst = reinterpret_cast<uint4*>(p.out + row0 * kGqaHeadDim);
      const int64_t n16 = rows * kGqaHeadDim * 2 / 16;
      for (int64_t i = tid; i < n16; i += kStride) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse)
        for (int64_t i = tid; i < rows; i += kStride) p.lse[row0 + i] = -CUDART_INF_F;
    }
  }
}



// Split-KV merge as its own launch (when the attention kernel runs without
// FUSED), one warp per NR rows of a (sequence, kv head), with the same
// arithmetic per row as the in-kernel merge, so both give the same bits.
// launch_merge takes one row per warp while that makes at most 16 warps per
// SM (short chains of dependent steps, many warps in flight), else
// kMergeRows (fewer copies of each warp's fixed set-up).
// Plain: only units cut between CTAs need it. Shared prefix: every row, from
// its prefix part (the group unit's pieces, or the prefix store when one CTA
// had the whole unit) then its suffix part (pieces, the suffix store, or
// nothing when the sequence ends at the prefix), always in that order.
// Launched as a programmatic dependent of the attention kernel: it may start
// early and waits here until that grid has finished and its writes are
// visible.
template <int MODE, int NR, int PIECES>
__global__ void __launch_bounds__(128) gqa_merge_kernel(const __grid_constant__ GqaParams p,
                                                        int G) {
  const int lane = threadIdx.x & 31;
  const int rmax = p.gh * p.q_len;  // rows of a partial slot (the largest group's)
  const int nrb = (rmax + NR - 1) / NR;
  // items: (row group, sequence, kv head, block of NR rows)
  const int64_t per_group = int64_t(p.B) * p.Hkv * nrb;
  const int64_t item = int64_t(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const bool live = item < per_group * p.ngroups;
  const int tg = live ? int(item / per_group) : 0;
  const int64_t gitem = item - tg * per_group;
  const int64_t unit = live ? gitem / nrb : 0;  // b * Hkv + kv head
  const int b = int(unit / p.Hkv), kvh = int(unit % p.Hkv);
  const RowGroup rg = row_group(p, tg);
  const int tok0 = rg.tok0, gh = rg.gh;
  const int rps = gh * rg.qlen;  // this group's rows per sequence
  // Before waiting for the attention grid: the tile line, from seq_lens alone.
  // seq_lens is an input of the call; the attention grid let this kernel
  // launch only after its own dependency wait, so it is final here. Units are
  // the ng prefix groups (prefix_tiles tiles each), then the sequences.
  const int NG = MODE == kModeShared ? p.ng : 0;
  // tiles of sequences before b, of every sequence, of the longest one
  int before = 0, all = 0, nmax = 0;
  if (live) {
    for (int s = lane; s < p.B; s += 32) {
      const int t = seq_unit_tiles<MODE>(p, p.seq_lens[s]);
      all += t;
      before += s < b ? t : 0;
      nmax = max(nmax, t);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      all += __shfl_xor_sync(0xffffffffu, all, off);
      before += __shfl_xor_sync(0xffffffffu, before, off);
      nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, off));
    }
  }
  const int n = live ? seq_unit_tiles<MODE>(p, p.seq_lens[b]) : 0;
  griddep_wait();
  griddep_launch_dependents();  // the next kernels may start their prologue
  const int r0 = int(gitem % nrb) * NR;
  if (!live || r0 >= rps) return;
  const int nrows = min(NR, rps - r0);
  const int cta0 = tg * G;  // the group's first CTA (G = CTAs per group)
  const int hg = kvh / p.hpc, w = kvh % p.hpc;
  const int head0 = kvh * p.g + rg.hoff;  // the group's first query head
  const int PT = MODE == kModeShared ? p.prefix_tiles : 0;
  const int64_t W = int64_t(p.nhg) * (int64_t(NG) * PT + all);
  const TileCut cut(W, G);
  const int64_t U0 = int64_t(p.nhg) * (int64_t(NG) * PT + before) + int64_t(hg) * n;
  const int c_lo = n ? cut.owner(U0) : 0, c_hi = n ? cut.owner(U0 + n - 1) : 0;
  if constexpr (MODE == kModePlain) {
    // a unit-cut launch (chosen on the device, as the attention kernel did)
    // left every unit whole
    if (p.auto_cut && short_units(int64_t(p.B) * p.nhg, nmax, G)) return;
    if (n == 0 || c_lo == c_hi) return;
    // PIECES pieces per round trip to L2 (launch_merge takes the larger batch
    // when the merge grid fits in one wave at the registers that needs).
    merge_split_rows<NR, PIECES>(p, cut, cta0, U0, c_lo, c_hi, b, tok0, w, head0, gh, rmax, r0,
                                 r0 + nrows, lane);
  } else {
    const int R = p.sgs * rps;  // rows of a partial slot
    MergeAcc<NR> m;
    m.init();
    {
      const int vp = b / p.sgs;  // the group's prefix unit (each has PT tiles)
      const int np = PT;
      const int64_t P0 = int64_t(p.nhg) * (int64_t(vp) * PT) + int64_t(hg) * np;
      const int p_lo = cut.owner(P0), p_hi = cut.owner(P0 + np - 1);
      if (p_lo == p_hi)
        merge_add_store(m, p, p.pre_o, p.pre_lse, b, tok0, head0, gh, r0, nrows, lane);
      else
        merge_add_pieces<NR, PIECES>(m, p, cut, cta0, P0, p_lo, p_hi, w, R, (b % p.sgs) * rps,
                                     r0, nrows, lane);
    }
    if (n > 0) {
      if (c_lo == c_hi)
        merge_add_store(m, p, p.suf_o, p.suf_lse, b, tok0, head0, gh, r0, nrows, lane);
      else
        merge_add_pieces<NR, PIECES>(m, p, cut, cta0, U0, c_lo, c_hi, w, R, 0, r0, nrows, lane);
    }
    merge_write_out(m, p, b, tok0, head0, gh, r0, nrows, lane);
  }
}

constexpr int kMaxDevices = 64;

// Launches the merge kernel for the rows of every (row group, sequence, kv
// head) (ngroups * B * Hkv * rows_per_slot rows) as a programmatic dependent
// of the attention kernel: its CTAs may become resident before the attention
// grid ends and wait in griddepcontrol.wait. Rows per warp (1, or kMergeRows
// past 16 warps per SM) and pieces per L2 round trip (the larger batch when
// the grid fits in one wave at the registers that takes) only change how the
// work is spread: every choice gives the same bits.
template <int MODE, int NR, int P>
struct MergeInstance {
  // blocks of 4 warps over the items (unit, block of NR of its rmax rows)
  static int64_t blocks(int64_t units, int rmax) {
    return (units * ((rmax + NR - 1) / NR) + 3) / 4;
  }
  static cudaError_t launch(const GqaParams& p, int64_t units, int rmax, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks(units, rmax)));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa_merge_kernel<MODE, NR, P>, p, p.group_ctas);
  }
  // CTAs of this instance per wave on `device` (0 on error), queried once.
  static int64_t wave(int device, int sms) {
    static int cached[kMaxDevices] = {};
    if (device >= 0 && device < kMaxDevices && cached[device] > 0) return cached[device];
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gqa_merge_kernel<MODE, NR, P>,
                                                      128, 0) != cudaSuccess)
      return 0;
    if (device >= 0 && device < kMaxDevices) cached[device] = per_sm * sms;
    return int64_t(per_sm) * sms;
  }
};

template <int MODE>
cudaError_t launch_merge(const GqaParams& p, cudaStream_t stream) {
  static int sms_of[kMaxDevices] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (sms_of[device] == 0 &&
      (e = cudaDeviceGetAttribute(&sms_of[device], cudaDevAttrMultiProcessorCount, device)) !=
          cudaSuccess)
    return e;
  const int sms = sms_of[device];
  // units (row group, sequence, kv head), each with a partial slot of rmax
  // rows (the largest group's; a shared-prefix launch has one group)
  const int64_t units = int64_t(p.ngroups) * p.B * p.Hkv;
  const int rmax = p.gh * p.q_len;
  if (units * rmax <= 16LL * sms) {  // one row per warp
    using Big = MergeInstance<MODE, 1, 8>;
    if (Big::blocks(units, rmax) <= Big::wave(device, sms))
      return Big::launch(p, units, rmax, stream);
    return MergeInstance<MODE, 1, 4>::launch(p, units, rmax, stream);
  }
  using Big = MergeInstance<MODE, kMergeRows, 4>;
  if (Big::blocks(units, rmax) <= Big::wave(device, sms))
    return Big::launch(p, units, rmax, stream);
  return MergeInstance<MODE, kMergeRows, 2>::launch(p, units, rmax, stream);
}

// Raise the dynamic shared-memory limit of one kernel instance, once per device.
template <int HPC, bool R16, bool C, bool U, int MODE = kModePlain, int TG = 1>
cudaError_t configure(int device) {
  static bool done[kMaxDevices] = {};
  if (device >= 0 && device < kMaxDevices && done[device]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(gqa_decode_kernel<HPC, R16, C, U, MODE, TG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(GqaCfg<HPC, TG>::kSmemBytes));
  if (e == cudaSuccess && device >= 0 && device < kMaxDevices) done[device] = true;
  return e;
}

template <int HPC, bool R16, bool C, bool U, int MODE = kModePlain, int TG = 1>
cudaError_t launch_attn(const GqaParams& p, int grid, cudaStream_t stream) {
  using Cfg = GqaCfg<HPC, TG>;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if ((e = configure<HPC, R16, C, U, MODE, TG>(device)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::smem_bytes(small_table(p, MODE));
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_decode_kernel<HPC, R16, C, U, MODE, TG>, p);
}

// CTAs per SM at the small or the full table layout.
template <int HPC, bool R16, bool C, bool U, int MODE = kModePlain, int TG = 1>
int occupancy(int device, bool small) {
  using Cfg = GqaCfg<HPC, TG>;
  // Queried once per device and layout (it does not change), not on every call.
  static int cached[kMaxDevices][2] = {};
  if (device >= 0 && device < kMaxDevices && cached[device][small] > 0)
    return cached[device][small];
  if (configure<HPC, R16, C, U, MODE, TG>(device) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &n, gqa_decode_kernel<HPC, R16, C, U, MODE, TG>, Cfg::kThreads,
          Cfg::smem_bytes(small)) != cudaSuccess)
    return 0;
  if (device >= 0 && device < kMaxDevices) cached[device][small] = n;
  return n;
}

}  // namespace
}  // namespace zl
