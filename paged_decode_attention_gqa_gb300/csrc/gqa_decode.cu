// Paged GQA decode attention for sm_103a: one persistent wave of CTAs, each a
// TMA producer warp plus one tensor-core consumer warp per kv head.
//
// Work decomposition. For sequence b the context is cut into n_b tiles of 16
// tokens. The tiles of all (sequence, kv-head-group) units are laid end to end
// and the line is cut into G equal ranges, one per CTA ("split-KV" of the
// flash_decoding family named under "技术架构：五层模块化设计" on the
// "ZhiLight：知乎开源的高性能 LLM 推理加速引擎" page). A CTA whose range covers a
// whole unit writes the final output; a unit cut between CTAs leaves one
// normalised partial (o, lse) per CTA in the workspace, and the merge kernel
// combines them by log-sum-exp in CTA order. The cut depends only on
// seq_lens and G, so results are bit-identical under page remapping.
//
// Per tile (16 tokens x HPC kv heads), the producer issues four TMA loads (K
// and V, two 64-column halves each, 128-byte swizzled) into a ring of
// shared-memory stages guarded by mbarriers. Consumer warp w owns kv head w of
// the group: its g query heads are the rows of an m16n8k16 tensor-core tile
// ("fused batch attention for decoding using tensor core instructions", the
// "ZhiLight: Zhihu's CUDA Inference Engine..." page, "Dual streams, host
// all-reduce and the memory model"), S = Q K^T and O += P V run on mma.sync,
// and the online softmax (running max, rescaled sum) stays in registers with
// quad shuffles. With q_len > 1 query tokens per sequence the rows are the
// (token, head) pairs, g * q_len <= 16 of them, each with its causal limit
// (the CAUSAL instances; q_len = 1 runs the instances without the limit).
#include "kernels.h"
#include "ptx.cuh"

#include <math_constants.h>

namespace zl {

namespace {

constexpr uint32_t kErrBadPage = 1u;
constexpr uint32_t kErrBadLen = 2u;
constexpr uint32_t kErrTimeout = 4u;

template <int HPC>
struct GqaCfg {
  static constexpr int kHalfBytes = HPC * kGqaTile * 64 * 2;  // one 64-column half of K or V
  static constexpr int kStageBytes = 4 * kHalfBytes;           // K lo | K hi | V lo | V hi
  static constexpr int kStages = HPC == 8 ? 3 : HPC == 4 ? 4 : HPC == 2 ? 6 : 8;
  static constexpr int kThreads = (HPC + 1) * 32;
  // 1 KB alignment slack + stages + barriers + per-stage flags + abort flag + prefix table
  static constexpr size_t kSmemBytes =
      1024 + size_t(kStages) * kStageBytes + kStages * 16 + kStages * 4 + 16 + (kMaxBatch + 1) * 4;
};

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

template <int HPC, bool ROWS16, bool CAUSAL>
__global__ void __launch_bounds__(GqaCfg<HPC>::kThreads, 1)
gqa_decode_kernel(const __grid_constant__ GqaParams p) {
  using Cfg = GqaCfg<HPC>;
  constexpr int NS = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // 128B swizzle wants 1 KB-aligned stages
  uint8_t* smem = smem_raw + (sbase - raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * Cfg::kStageBytes);
  uint64_t* empty = full + NS;
  int* stage_bad = reinterpret_cast<int*>(empty + NS);
  volatile int* abort_flag = stage_bad + NS;
  int* prefix = stage_bad + NS + 4;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.B;
  const int64_t cap = p.bt_stride * int64_t(p.page_size);

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), HPC);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == HPC && lane == 0) {
    tma_prefetch_desc(&p.tmap_k);
    tma_prefetch_desc(&p.tmap_v);
  }

  // Tiles per sequence and their exclusive prefix sum (warp 0).
  if (warp == 0) {
    const int per = (B + 31) / 32;
    const int b0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int L = p.seq_lens[b];
        const bool ok = L >= 0 && int64_t(L) <= cap;
        if (!ok && blockIdx.x == 0) raise_error(p.err_flags, kErrBadLen);
        local += ok ? (L + kGqaTile - 1) / kGqaTile : 0;
      }
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        prefix[b] = run;
        const int L = p.seq_lens[b];
        run += (L >= 0 && int64_t(L) <= cap) ? (L + kGqaTile - 1) / kGqaTile : 0;
      }
    }
    if (lane == 31) prefix[B] = incl;
  }
  __syncthreads();

  if (blockIdx.x == 0) {
    for (int b = tid; b <= B; b += Cfg::kThreads) p.ws_prefix[b] = prefix[b];
  }

  const int G = gridDim.x, c = blockIdx.x;
  const int nhg = p.nhg;
  const int64_t W = int64_t(nhg) * prefix[B];
  const int64_t s_c = int64_t(c) * W / G;
  const int64_t e_c = int64_t(c + 1) * W / G;

  if (warp == HPC) {
    // ------------------------------------------------------------ producer
    int it = 0;
    bool aborted = false;
    for (int64_t base = s_c; base < e_c && !aborted; base += 32) {
      // lane i resolves tile base + i: page id, slot and head group
      const int64_t idx = base + lane;
      int page = 0, slot = 0, hg = 0, bad = 0;
      if (idx < e_c) {
        const int b = locate_seq(prefix, B, nhg, idx);
        const int n = prefix[b + 1] - prefix[b];
        const int64_t r = idx - int64_t(nhg) * prefix[b];
        hg = int(r / n);
        const int tok0 = int(r % n) * kGqaTile;
        slot = tok0 % p.page_size;
        page = p.block_table[int64_t(b) * p.bt_stride + tok0 / p.page_size];
        bad = (page < 0 || page >= p.num_pages) ? 1 : 0;
      }
      const int cnt = int(min(int64_t(32), e_c - base));
      for (int k = 0; k < cnt; ++k, ++it) {
        const int pg = __shfl_sync(0xffffffffu, page, k);
        const int sl = __shfl_sync(0xffffffffu, slot, k);
        const int h = __shfl_sync(0xffffffffu, hg, k);
        const int bd = __shfl_sync(0xffffffffu, bad, k);
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
  const int w = warp;                 // kv head within the group
  const int gid = lane >> 2, t4 = lane & 3;
  const int g = p.g;
  const float scale_log2 = p.scale_log2;
  int it = 0;
  int64_t idx = s_c;
  while (idx < e_c) {
    const int b = locate_seq(prefix, B, nhg, idx);
    const int n = prefix[b + 1] - prefix[b];
    const int64_t unit_start0 = int64_t(nhg) * prefix[b];
    const int hg = int((idx - unit_start0) / n);
    const int j0 = int((idx - unit_start0) % n);
    const int64_t unit_end = unit_start0 + int64_t(hg + 1) * n;
    const int64_t piece_end = min(e_c, unit_end);
    const int ntiles = int(piece_end - idx);
    const bool partial = (j0 > 0) || (piece_end < unit_end);
    const int slot = (idx == s_c) ? 0 : 1;
    const int L = p.seq_lens[b];
    const int head0 = (hg * HPC + w) * g;  // first query head of this kv head
    // m16 tile rows r < R = g * q_len are (query token i = r / g, head head0 + r % g);
    // the rest are zero. Query i sees tokens t < L - q_len + 1 + i (the new
    // tokens are in the cache; each sees itself and what precedes it).
    const int R = g * p.q_len;
    const int ra = gid, rb = gid + 8;
    const int lim_a = L - p.q_len + 1 + ra / g;
    const int lim_b = L - p.q_len + 1 + rb / g;
    auto qrow_index = [&](int r) -> int64_t {
      return (int64_t(b) * p.q_len + r / g) * p.Hq + head0 + r % g;
    };

    uint32_t qa[8][4];
    {
      const bool r0 = ra < R, r1 = ROWS16 && rb < R;
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
    int bad = 0;

    // One row's online-softmax step in base 2 over this thread's four scores
    // (tokens 2t4, 2t4+1, 2t4+8, 2t4+9 of the tile; vis = visible tokens of
    // the row in this tile). A row with nothing visible yet keeps m = -inf and
    // contributes zeros.
    auto row_step = [&](float sa, float sb, float sc, float sd, int vis, float& m, float& l,
                        uint32_t& p_lo, uint32_t& p_hi) -> float {
      const float x0 = 2 * t4 < vis ? sa * scale_log2 : -CUDART_INF_F;
      const float x1 = 2 * t4 + 1 < vis ? sb * scale_log2 : -CUDART_INF_F;
      const float x2 = 2 * t4 + 8 < vis ? sc * scale_log2 : -CUDART_INF_F;
      const float x3 = 2 * t4 + 9 < vis ? sd * scale_log2 : -CUDART_INF_F;
      float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m, mx);
      const float base = mn == -CUDART_INF_F ? 0.f : mn;
      const float alpha = ex2_approx(m - base);
      m = mn;
      p_lo = pack_bf16x2(ex2_approx(x0 - base), ex2_approx(x1 - base));
      p_hi = pack_bf16x2(ex2_approx(x2 - base), ex2_approx(x3 - base));
      const float2 f0 = unpack_bf16x2(p_lo), f2 = unpack_bf16x2(p_hi);
      l = l * alpha + ((f0.x + f0.y) + (f2.x + f2.y));
      return alpha;
    };

    for (int t = 0; t < ntiles; ++t, ++it) {
      const int stage = it % NS;
      const uint32_t phase = (it / NS) & 1;
      const int tok0 = (j0 + t) * kGqaTile;
      const int valid = min(kGqaTile, L - tok0);  // tokens in the cache (V rows to keep)
      if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag)) {
        if (lane == 0) {
          raise_error(p.err_flags, kErrTimeout);
          *abort_flag = 1;
        }
        return;
      }
      bad |= stage_bad[stage];
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
        const float alpha = row_step(s[0][0], s[0][1], s[1][0], s[1][1],
                                     CAUSAL ? min(valid, lim_a - tok0) : valid, m0, l0, pa[0], pa[2]);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][0] *= alpha;
          o[nt][1] *= alpha;
        }
      }
      if (ROWS16) {
        const float alpha = row_step(s[0][2], s[0][3], s[1][2], s[1][3],
                                     CAUSAL ? min(valid, lim_b - tok0) : valid, m1, l1, pa[1], pa[3]);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          o[nt][2] *= alpha;
          o[nt][3] *= alpha;
        }
      } else {
        pa[1] = pa[3] = 0u;
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
    if (bad && lane == 0) raise_error(p.err_flags, kErrBadPage);
#pragma unroll
    for (int half = 0; half < (ROWS16 ? 2 : 1); ++half) {
      const int r = half ? rb : ra;
      if (r >= R) continue;
      const float l = half ? l1 : l0;
      const float m = half ? m1 : m0;
      // A piece that met a bad page, or a row that saw no token, is written as
      // zeros with lse = -inf (weight 0 in the merge).
      const bool none = bad || !(l > 0.f);
      const float inv = none ? 0.f : 1.f / l;
      const float lse2 = none ? -CUDART_INF_F : m + log2f(l);
      if (!partial) {
        const int64_t orow = qrow_index(r);
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.out + orow * kGqaHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[nt * 4 + t4] =
              none ? 0u : pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (p.lse && t4 == 0) p.lse[orow] = lse2 * 0.69314718055994531f;
      } else {
        const int64_t wrow = ((int64_t(c) * 2 + slot) * HPC + w) * R + r;
        float2* dst = reinterpret_cast<float2*>(p.ws_o + wrow * kGqaHeadDim);
#pragma unroll
        for (int nt = 0; nt < 16; ++nt)
          dst[nt * 4 + t4] = none ? make_float2(0.f, 0.f)
                                  : make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (t4 == 0) p.ws_lse[wrow] = bad ? CUDART_NAN_F : lse2;
      }
    }
    idx = piece_end;
  }

  // Sequences with no tiles (empty or invalid length): zeros, lse = -inf.
  for (int b = c; b < B; b += G) {
    if (prefix[b + 1] != prefix[b]) continue;
    const int64_t rows = int64_t(p.q_len) * p.Hq;
    uint4* dst = reinterpret_cast<uint4*>(p.out + int64_t(b) * rows * kGqaHeadDim);
    const int64_t n16 = rows * kGqaHeadDim * 2 / 16;
    for (int64_t i = tid; i < n16; i += HPC * 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (p.lse)
      for (int64_t i = tid; i < rows; i += HPC * 32) p.lse[int64_t(b) * rows + i] = -CUDART_INF_F;
  }
}

// CTA that owns global tile x when W tiles are cut into G ranges
// [floor(c W / G), floor((c+1) W / G)).
__device__ __forceinline__ int cta_of_tile(int64_t x, int64_t W, int G) {
  return int(((x + 1) * G + W - 1) / W) - 1;
}

// One warp per (sequence, query head): log-sum-exp merge of the partials of
// a unit that was cut between CTAs, in CTA order. Units that one CTA finished
// were written by the attention kernel and are skipped here.
__global__ void __launch_bounds__(128) gqa_merge_kernel(const __grid_constant__ GqaParams p,
                                                        int G) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + warp;  // (b, query token i, head)
  if (row >= int64_t(p.B) * p.q_len * p.Hq) return;
  const int b = int(row / (int64_t(p.q_len) * p.Hq));
  const int i = int((row / p.Hq) % p.q_len), hq = int(row % p.Hq);
  const int kvh = hq / p.g, hg = kvh / p.hpc, w = kvh % p.hpc;
  const int R = p.g * p.q_len, r = i * p.g + hq % p.g;  // row of the m16 tile
  const int* prefix = p.ws_prefix;
  const int n = prefix[b + 1] - prefix[b];
  if (n == 0) return;
  const int64_t W = int64_t(p.nhg) * prefix[p.B];
  const int64_t U0 = int64_t(p.nhg) * prefix[b] + int64_t(hg) * n;
  const int c_lo = cta_of_tile(U0, W, G), c_hi = cta_of_tile(U0 + n - 1, W, G);
  if (c_lo == c_hi) return;

  float M = -CUDART_INF_F;
  bool bad = false;
  for (int c = c_lo; c <= c_hi; ++c) {
    const int64_t s_c = int64_t(c) * W / G, e_c = int64_t(c + 1) * W / G;
    if (s_c == e_c) continue;
    const int slot = (c == c_lo && U0 > s_c) ? 1 : 0;
    const float l = p.ws_lse[((int64_t(c) * 2 + slot) * p.hpc + w) * R + r];
    bad |= isnan(l);
    M = fmaxf(M, l);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (!bad) {
    for (int c = c_lo; c <= c_hi; ++c) {
      const int64_t s_c = int64_t(c) * W / G, e_c = int64_t(c + 1) * W / G;
      if (s_c == e_c) continue;
      const int slot = (c == c_lo && U0 > s_c) ? 1 : 0;
      const int64_t wrow = ((int64_t(c) * 2 + slot) * p.hpc + w) * R + r;
      const float wgt = exp2f(p.ws_lse[wrow] - M);
      const float4 v = reinterpret_cast<const float4*>(p.ws_o + wrow * kGqaHeadDim)[lane];
      acc.x += wgt * v.x;
      acc.y += wgt * v.y;
      acc.z += wgt * v.z;
      acc.w += wgt * v.w;
      den += wgt;
    }
  }
  const float inv = bad ? 0.f : 1.f / den;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(p.out + row * kGqaHeadDim)[lane] = packed;
  if (p.lse && lane == 0)
    p.lse[row] = bad ? -CUDART_INF_F : (M + log2f(den)) * 0.69314718055994531f;
}

constexpr int kMaxDevices = 64;

// Raise the dynamic shared-memory limit of one kernel instance, once per device.
template <int HPC, bool R16, bool C>
cudaError_t configure(int device) {
  static bool done[kMaxDevices] = {};
  if (device >= 0 && device < kMaxDevices && done[device]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(gqa_decode_kernel<HPC, R16, C>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(GqaCfg<HPC>::kSmemBytes));
  if (e == cudaSuccess && device >= 0 && device < kMaxDevices) done[device] = true;
  return e;
}

template <int HPC, bool R16, bool C>
cudaError_t launch_attn(const GqaParams& p, int grid, cudaStream_t stream) {
  using Cfg = GqaCfg<HPC>;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if ((e = configure<HPC, R16, C>(device)) != cudaSuccess) return e;
  gqa_decode_kernel<HPC, R16, C><<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <int HPC, bool R16, bool C>
int occupancy(int device) {
  using Cfg = GqaCfg<HPC>;
  if (configure<HPC, R16, C>(device) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_decode_kernel<HPC, R16, C>, Cfg::kThreads,
                                                    Cfg::kSmemBytes) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace

int gqa_heads_per_cta(int Hkv) {
  if (Hkv % 8 == 0) return 8;
  if (Hkv % 4 == 0) return 4;
  if (Hkv % 2 == 0) return 2;
  return 1;
}

namespace {

// The kernel instance for (heads per CTA, 16 rows, causal rows).
template <template <int, bool, bool> class F, typename... A>
auto dispatch(int hpc, bool r16, bool causal, A... a) -> decltype(F<1, false, false>::run(a...)) {
  using R = decltype(F<1, false, false>::run(a...));
  const int k = (hpc * 2 + (r16 ? 1 : 0)) * 2 + (causal ? 1 : 0);
  switch (k) {
#define ZL_CASE(H, S, C) \
  case (H * 2 + S) * 2 + C: return F<H, bool(S), bool(C)>::run(a...);
    ZL_CASE(1, 0, 0) ZL_CASE(1, 0, 1) ZL_CASE(1, 1, 0) ZL_CASE(1, 1, 1)
    ZL_CASE(2, 0, 0) ZL_CASE(2, 0, 1) ZL_CASE(2, 1, 0) ZL_CASE(2, 1, 1)
    ZL_CASE(4, 0, 0) ZL_CASE(4, 0, 1) ZL_CASE(4, 1, 0) ZL_CASE(4, 1, 1)
    ZL_CASE(8, 0, 0) ZL_CASE(8, 0, 1) ZL_CASE(8, 1, 0) ZL_CASE(8, 1, 1)
#undef ZL_CASE
    default: return R();
  }
}

template <int HPC, bool R16, bool C>
struct Occupancy {
  static int run(int device) { return occupancy<HPC, R16, C>(device); }
};

template <int HPC, bool R16, bool C>
struct Launch {
  static cudaError_t run(const GqaParams* p, int grid, cudaStream_t stream) {
    return launch_attn<HPC, R16, C>(*p, grid, stream);
  }
};

}  // namespace

int gqa_ctas_per_sm(int hpc, bool rows16, bool causal, int device) {
  return dispatch<Occupancy>(hpc, rows16, causal, device);
}

cudaError_t gqa_decode_launch(const GqaParams& p, int grid, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  cudaError_t e = cudaSuccess;
  if (attn_begin && (e = cudaEventRecord(attn_begin, stream)) != cudaSuccess) return e;
  const bool r16 = p.g * p.q_len > 8;
  const bool known = p.hpc == 1 || p.hpc == 2 || p.hpc == 4 || p.hpc == 8;
  if (!known) return cudaErrorInvalidValue;
  e = dispatch<Launch>(p.hpc, r16, p.q_len > 1, &p, grid, stream);
  if (e != cudaSuccess) return e;
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  const int64_t rows = int64_t(p.B) * p.q_len * p.Hq;
  gqa_merge_kernel<<<int((rows + 3) / 4), 128, 0, stream>>>(p, grid);
  return cudaGetLastError();
}

}  // namespace zl
