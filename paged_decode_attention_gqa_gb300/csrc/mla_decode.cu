// Absorbed multi-head latent attention (MLA) decode for sm_103a on tcgen05.
//
// The operation (MLA is listed under "功能生态" and flash_mla under
// "技术架构：五层模块化设计" on "ZhiLight：知乎开源的高性能 LLM 推理加速引擎"; DeepseekV2
// MLA under "Dual streams, host all-reduce and the memory model" on "ZhiLight:
// Zhihu's CUDA Inference Engine..."): every token stores one latent row of 576
// bf16 (512 latent + 64 rope); all 128 query heads attend over it with
// QK over the 576 columns and V = the first 512 columns.
//
// Shape of the problem on one SM: fp32 O for 128 heads x 512 columns is the
// whole of TMEM (512 columns x 128 lanes), and Q (128 x 576 bf16) is 147 KB of
// shared memory. So a cluster of two CTAs shares each tile of 64 tokens:
//   rank 0 loads latent columns [0,256) and the rope [512,576),
//   rank 1 loads latent columns [256,512);
// each rank computes a partial S = Q K^T over its columns into TMEM (M = 128
// heads, N = 64 tokens, K = 320 or 256), the two fp32 partials are swapped
// through distributed shared memory and summed (both ranks then hold the same
// S and make the same softmax decisions), and each rank accumulates its own
// 256 columns of O = P V in TMEM (N = 256, V read MN-major straight from the
// tile it loaded). Every K/V byte leaves HBM once.
//
// Warp roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 2-5 softmax / epilogue, one thread per head row (TMEM lane).
// The running max is only moved when it grows by more than 2^8, so O in TMEM
// is rarely rescaled (P <= 256 meanwhile).
#include "kernels.h"
#include "ptx.cuh"

#include <math_constants.h>

namespace zl {

namespace {

constexpr uint32_t kErrBadPage = 1u;
constexpr uint32_t kErrBadLen = 2u;
constexpr uint32_t kErrTimeout = 4u;

constexpr int kTile = kMlaTile;               // tokens per tile (= page size granule)
constexpr int kRows = 128;                    // query heads = TMEM lanes
constexpr int kBoxQ = kRows * 128;            // 16 KB: 128 rows x 64 bf16
constexpr int kBoxKV = kTile * 128;           // 8 KB: 64 tokens x 64 bf16
constexpr int kMaxBoxes = 5;                  // rank 0: 4 latent + 1 rope
constexpr int kStages = 2;
constexpr int kStageBytes = kMaxBoxes * kBoxKV;  // 40 KB
constexpr int kXStride = 64 * 4 + 16;            // exchange row (padded against bank conflicts)
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMaxBoxes * kBoxQ;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffX = kOffP + kRows * 128;
constexpr int kOffBar = kOffX + kRows * kXStride;
enum : int {
  B_Q_FULL = 0, B_Q_EMPTY, B_KV_FULL0, B_KV_FULL1, B_KV_EMPTY0, B_KV_EMPTY1, B_S_FULL0,
  B_S_FULL1, B_S_EMPTY0, B_S_EMPTY1, B_P_FULL, B_PV_DONE, B_X_FULL, B_X_FREE, B_FINAL, B_COUNT
};
constexpr int kOffMisc = kOffBar + 8 * 16;
constexpr int kOffPrefix = kOffMisc + 64;
constexpr size_t kSmemBytes = 1024 + kOffPrefix + size_t(kMlaMaxBatch + 1) * 4;
static_assert(kSmemBytes <= 232448, "MLA kernel exceeds 227 KB of shared memory");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;    // O half: columns [0, 256)
constexpr uint32_t kTmemS = 256;  // S buffers: [256, 320) and [320, 384)
constexpr int kThreads = 192;

__device__ __forceinline__ void raise_error(uint32_t* flags, uint32_t bits) {
  if (flags) atomicOr(flags, bits);
}

__device__ __forceinline__ int locate(const int* prefix, int B, int64_t idx) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  int* prefix = reinterpret_cast<int*>(smem + kOffPrefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int cid = blockIdx.x >> 1, NC = gridDim.x >> 1;
  const int nbox = rank == 0 ? 5 : 4;
  const int B = p.B;
  const int64_t cap = p.bt_stride * int64_t(p.page_size);

  if (tid == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_EMPTY), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KV_FULL0 + s), 1);
      mbar_init(bar(B_KV_EMPTY0 + s), 1);
      mbar_init(bar(B_S_FULL0 + s), 1);
      mbar_init(bar(B_S_EMPTY0 + s), kRows);
    }
    mbar_init(bar(B_P_FULL), kRows);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_X_FULL), kRows);
    mbar_init(bar(B_X_FREE), kRows);
    mbar_init(bar(B_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_kv);
    tma_prefetch_desc(&p.tmap_q);
  }
  // Tiles (of 64 tokens) per sequence, exclusive prefix sum.
  if (warp == 2) {
    const int per = (B + 31) / 32;
    const int b0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int L = p.seq_lens[b];
        const bool ok = L >= 0 && int64_t(L) <= cap;
        if (!ok && blockIdx.x == 0) raise_error(p.err_flags, kErrBadLen);
        local += ok ? (L + kTile - 1) / kTile : 0;
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
        run += (L >= 0 && int64_t(L) <= cap) ? (L + kTile - 1) / kTile : 0;
      }
    }
    if (lane == 31) prefix[B] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tmem = *tmem_slot;

  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += kThreads) p.ws_prefix[b] = prefix[b];

  const int64_t W = prefix[B];
  const int64_t s_c = int64_t(cid) * W / NC;
  const int64_t e_c = int64_t(cid + 1) * W / NC;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0, piece = 0;
      bool ok = true;
      for (int64_t idx = s_c; idx < e_c && ok;) {
        const int b = locate(prefix, B, idx);
        const int j0 = int(idx - prefix[b]);
        const int64_t pend = min(e_c, int64_t(prefix[b + 1]));
        if (!mbar_wait(bar(B_Q_EMPTY), (piece & 1) ^ 1u, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(B_Q_FULL), nbox * kBoxQ);
        for (int i = 0; i < nbox; ++i) {
          const int col = i < 4 ? int(rank) * 256 + 64 * i : 512;
          tma_load_3d(sbase + kOffQ + i * kBoxQ, &p.tmap_q, bar(B_Q_FULL), col, 0, b);
        }
        for (int j = j0; j < j0 + int(pend - idx); ++j, ++it) {
          const int s = it & 1;
          if (!mbar_wait(bar(B_KV_EMPTY0 + s), ((it >> 1) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int tok0 = j * kTile;
          const int page = p.block_table[int64_t(b) * p.bt_stride + tok0 / p.page_size];
          if (page < 0 || page >= p.num_pages) {
            mbar_arrive(bar(B_KV_FULL0 + s));  // nothing loaded; the piece is discarded
          } else {
            const int slot = tok0 % p.page_size;
            mbar_arrive_expect_tx(bar(B_KV_FULL0 + s), nbox * kBoxKV);
            for (int i = 0; i < nbox; ++i) {
              const int col = i < 4 ? int(rank) * 256 + 64 * i : 512;
              tma_load_3d(sbase + kOffKV + s * kStageBytes + i * kBoxKV, &p.tmap_kv,
                          bar(B_KV_FULL0 + s), col, slot, page);
            }
          }
        }
        ++piece;
        idx = pend;
      }
      if (!ok) {
        raise_error(p.err_flags, kErrTimeout);
        *abort_flag = 1;
      }
      // Leave no copy in flight: wait for the last stages and the last Q.
      const volatile int never = 0;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        mbar_wait(bar(B_KV_FULL0 + (j & 1)), (j >> 1) & 1, &never);
      if (piece > 0) mbar_wait(bar(B_Q_FULL), (piece - 1) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(kRows, kTile, false);
      const uint32_t idesc_pv = umma_idesc_bf16(kRows, 256, true);
      int it = 0, piece = 0, pending = -1;
      bool pending_first = false, ok = true;
      auto issue_pv = [&](int j, bool first) -> bool {
        if (!mbar_wait(bar(B_P_FULL), j & 1, abort_flag)) return false;
        tc_fence_after();
        const int s = j & 1;
        const uint32_t vbase = sbase + kOffKV + s * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t a = umma_smem_desc(sbase + kOffP + kk * 32, 0, 1024, 2);
          const uint64_t bdesc = umma_smem_desc(vbase + kk * 16 * 128, kBoxKV, 1024, 2);
          umma_bf16(tmem + kTmemO, a, bdesc, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(bar(B_KV_EMPTY0 + s));
        umma_commit(bar(B_PV_DONE));
        return true;
      };
      for (int64_t idx = s_c; idx < e_c && ok;) {
        const int b = locate(prefix, B, idx);
        const int64_t pend = min(e_c, int64_t(prefix[b + 1]));
        const int ntiles = int(pend - idx);
        if (!mbar_wait(bar(B_Q_FULL), piece & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int t = 0; t < ntiles; ++t, ++it) {
          const int s = it & 1;
          const uint32_t ph = (it >> 1) & 1;
          if (!mbar_wait(bar(B_KV_FULL0 + s), ph, abort_flag) ||
              !mbar_wait(bar(B_S_EMPTY0 + s), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kvbase = sbase + kOffKV + s * kStageBytes;
          for (int i = 0; i < nbox; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = umma_smem_desc(sbase + kOffQ + i * kBoxQ + kk * 32, 0, 1024, 2);
              const uint64_t bdesc = umma_smem_desc(kvbase + i * kBoxKV + kk * 32, 0, 1024, 2);
              umma_bf16(tmem + kTmemS + 64 * s, a, bdesc, idesc_qk, (i | kk) ? 1u : 0u);
            }
          }
          umma_commit(bar(B_S_FULL0 + s));
          if (t == ntiles - 1) umma_commit(bar(B_Q_EMPTY));
          if (pending >= 0 && !issue_pv(pending, pending_first)) { ok = false; break; }
          pending = it;
          pending_first = (t == 0);  // first PV of a piece overwrites O
        }
        ++piece;
        idx = pend;
      }
      if (ok && pending >= 0 && !issue_pv(pending, pending_first)) ok = false;
      if (!ok) {
        raise_error(p.err_flags, kErrTimeout);
        *abort_flag = 1;
      }
      // Every MMA done before TMEM is released.
      umma_commit(bar(B_FINAL));
      const volatile int never = 0;
      mbar_wait(bar(B_FINAL), 0, &never);
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;                 // query head = TMEM lane
    const uint32_t tl = tmem + (uint32_t(32 * q4) << 16);
    const float c = p.scale_log2;
    const uint32_t my_x = sbase + kOffX + row * kXStride;
    const uint32_t peer_x = mapa_shared(my_x, peer);
    const uint32_t peer_xfull = mapa_shared(bar(B_X_FULL), peer);
    const uint32_t peer_xfree = mapa_shared(bar(B_X_FREE), peer);
    const int stid = tid - 64;                       // 0..127 within the softmax group
    int it = 0;
    bool ok = true;
    for (int64_t idx = s_c; idx < e_c && ok;) {
      const int b = locate(prefix, B, idx);
      const int j0 = int(idx - prefix[b]);
      const int64_t pend = min(e_c, int64_t(prefix[b + 1]));
      const int ntiles = int(pend - idx);
      const bool partial = (j0 > 0) || (pend < prefix[b + 1]);
      const int slot = (idx == s_c) ? 0 : 1;
      const int L = p.seq_lens[b];
      float m_used = -CUDART_INF_F, l = 0.f;
      int bad = 0;
      for (int t = 0; t < ntiles; ++t, ++it) {
        const int s = it & 1;
        const uint32_t ph = (it >> 1) & 1;
        const int tok0 = (j0 + t) * kTile;
        const int valid = min(kTile, L - tok0);
        const int page = p.block_table[int64_t(b) * p.bt_stride + tok0 / p.page_size];
        bad |= (page < 0 || page >= p.num_pages) ? 1 : 0;

        // my partial scores for this tile
        if (!mbar_wait(bar(B_S_FULL0 + s), ph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tmem_ld32(tl + kTmemS + 64 * s, lo);
          tmem_ld32(tl + kTmemS + 64 * s + 32, hi);
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(bar(B_S_EMPTY0 + s));

        // swap partials with the peer through distributed shared memory
        if (!mbar_wait_cluster(bar(B_X_FREE), (it & 1) ^ 1u, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int k = 0; k < 16; ++k)
          st_cluster_v4(peer_x + 16 * k, __uint_as_float(sv[4 * k]), __uint_as_float(sv[4 * k + 1]),
                        __uint_as_float(sv[4 * k + 2]), __uint_as_float(sv[4 * k + 3]));
        mbar_arrive_remote(peer_xfull);
        if (!mbar_wait_cluster(bar(B_X_FULL), it & 1, abort_flag)) { ok = false; break; }
        float x[64];
        {
          const float4* mine = reinterpret_cast<const float4*>(smem + kOffX + row * kXStride);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 v = mine[k];
            x[4 * k] = __uint_as_float(sv[4 * k]) + v.x;
            x[4 * k + 1] = __uint_as_float(sv[4 * k + 1]) + v.y;
            x[4 * k + 2] = __uint_as_float(sv[4 * k + 2]) + v.z;
            x[4 * k + 3] = __uint_as_float(sv[4 * k + 3]) + v.w;
          }
        }
        mbar_arrive_remote(peer_xfree);

        // online softmax (base 2); the max moves only when it grows by > 8
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          x[k] = (k < valid) ? x[k] * c : -CUDART_INF_F;
          mx = fmaxf(mx, x[k]);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (t == 0) {
          m_used = mx;
        } else if (mx > m_used + 8.f) {
          alpha = exp2f(m_used - mx);
          m_used = mx;
          rescale = true;
        }
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          pk[k] = pack_bf16x2(ex2_approx(x[2 * k] - m_used), ex2_approx(x[2 * k + 1] - m_used));
          const float2 f = unpack_bf16x2(pk[k]);
          lsum += f.x + f.y;
        }
        l = l * alpha + lsum;

        // tail tile: zero the V rows past the end (NaN there would poison 0 * V)
        if (valid < kTile) {
          const uint32_t vb = sbase + kOffKV + s * kStageBytes;
          const int nz = (kTile - valid) * 4 * 8;  // 16-byte chunks in 4 latent boxes
          for (int z = stid; z < nz; z += kRows) {
            const int chunk = z & 7, box = (z >> 3) & 3, r = valid + (z >> 5);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + box * kBoxKV + r * 128 + chunk * 16),
                         "r"(0u)
                         : "memory");
          }
        }

        // P buffer and O are free once the previous PV finished
        if (it > 0 && !mbar_wait(bar(B_PV_DONE), (it - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        // tcgen05.ld/st are warp-wide: rescale when any row of the warp needs it
        // (rows that do not need it multiply by exactly 1).
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[32];
            tmem_ld32(tl + kTmemO + 32 * cc, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(tl + kTmemO + 32 * cc, o);
          }
          tmem_wait_st();
        }
        // P row: 64 bf16 in the 128-byte-swizzled K-major layout of the A operand
        {
          const uint32_t prow = sbase + kOffP + row * 128;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             prow + ((k ^ (row & 7)) << 4)),
                         "r"(pk[4 * k]), "r"(pk[4 * k + 1]), "r"(pk[4 * k + 2]), "r"(pk[4 * k + 3])
                         : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL));
      }
      if (!ok) break;

      // ---- epilogue of the piece: O / l
      if (!mbar_wait(bar(B_PV_DONE), (it - 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      if (bad && stid == 0) raise_error(p.err_flags, kErrBadPage);
      const float inv = bad ? 0.f : 1.f / l;
      const float lse2 = bad ? -CUDART_INF_F : m_used + log2f(l);
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t o[32];
        tmem_ld32(tl + kTmemO + 32 * cc, o);
        tmem_wait_ld();
        const int col = int(rank) * 256 + 32 * cc;
        if (!partial) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t(b) * kRows + row) * kMlaDv + col);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = bad ? 0u : pack_bf16x2(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
            v.y = bad ? 0u : pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
            v.z = bad ? 0u : pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
            v.w = bad ? 0u : pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
            dst[k] = v;
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(
              p.ws_o + ((int64_t(cid) * 2 + slot) * kRows + row) * kMlaDv + col);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                         : make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                       __uint_as_float(o[4 * k + 2]) * inv, __uint_as_float(o[4 * k + 3]) * inv);
        }
      }
      if (rank == 0) {
        if (!partial) {
          if (p.lse) p.lse[int64_t(b) * kRows + row] = lse2 * 0.69314718055994531f;
        } else {
          p.ws_lse[(int64_t(cid) * 2 + slot) * kRows + row] = bad ? CUDART_NAN_F : lse2;
        }
      }
      tc_fence_before();
      idx = pend;
    }
    if (!ok) {
      raise_error(p.err_flags, kErrTimeout);
      *abort_flag = 1;
    }
    // Sequences with no tiles: zeros (this rank's columns), lse = -inf.
    for (int b = cid; b < B; b += NC) {
      if (prefix[b + 1] != prefix[b]) continue;
      uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t(b) * kRows + row) * kMlaDv +
                                            int(rank) * 256);
      for (int k = 0; k < 32; ++k) dst[k] = make_uint4(0u, 0u, 0u, 0u);
      if (rank == 0 && p.lse) p.lse[int64_t(b) * kRows + row] = -CUDART_INF_F;
    }
  }

  // ---- teardown: all roles done; release TMEM, then leave the cluster together
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

__device__ __forceinline__ int cluster_of_tile(int64_t x, int64_t W, int NC) {
  return int(((x + 1) * NC + W - 1) / W) - 1;
}

// One warp per (sequence, head): log-sum-exp merge of the partials of a
// sequence cut between clusters, in cluster order.
__global__ void __launch_bounds__(128) mla_merge_kernel(const __grid_constant__ MlaParams p,
                                                        int NC) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + warp;
  if (row >= int64_t(p.B) * kRows) return;
  const int b = int(row / kRows), h = int(row % kRows);
  const int* prefix = p.ws_prefix;
  const int n = prefix[b + 1] - prefix[b];
  if (n == 0) return;
  const int64_t W = prefix[p.B];
  const int64_t U0 = prefix[b];
  const int c_lo = cluster_of_tile(U0, W, NC), c_hi = cluster_of_tile(U0 + n - 1, W, NC);
  if (c_lo == c_hi) return;
  float M = -CUDART_INF_F;
  bool bad = false;
  for (int c = c_lo; c <= c_hi; ++c) {
    const int64_t s_c = int64_t(c) * W / NC, e_c = int64_t(c + 1) * W / NC;
    if (s_c == e_c) continue;
    const int slot = (c == c_lo && U0 > s_c) ? 1 : 0;
    const float l = p.ws_lse[(int64_t(c) * 2 + slot) * kRows + h];
    bad |= isnan(l);
    M = fmaxf(M, l);
  }
  float acc[16] = {};
  float den = 0.f;
  if (!bad) {
    for (int c = c_lo; c <= c_hi; ++c) {
      const int64_t s_c = int64_t(c) * W / NC, e_c = int64_t(c + 1) * W / NC;
      if (s_c == e_c) continue;
      const int slot = (c == c_lo && U0 > s_c) ? 1 : 0;
      const int64_t wrow = (int64_t(c) * 2 + slot) * kRows + h;
      const float wgt = exp2f(p.ws_lse[wrow] - M);
      const float4* src = reinterpret_cast<const float4*>(p.ws_o + wrow * kMlaDv);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = src[lane + 32 * k];
        acc[4 * k] += wgt * v.x;
        acc[4 * k + 1] += wgt * v.y;
        acc[4 * k + 2] += wgt * v.z;
        acc[4 * k + 3] += wgt * v.w;
      }
      den += wgt;
    }
  }
  const float inv = bad ? 0.f : 1.f / den;
  uint2* dst = reinterpret_cast<uint2*>(p.out + row * kMlaDv);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint2 v;
    v.x = pack_bf16x2(acc[4 * k] * inv, acc[4 * k + 1] * inv);
    v.y = pack_bf16x2(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
    dst[lane + 32 * k] = v;
  }
  if (p.lse && lane == 0)
    p.lse[row] = bad ? -CUDART_INF_F : (M + log2f(den)) * 0.69314718055994531f;
}

constexpr int kMaxDevices = 64;

}  // namespace

size_t mla_smem_bytes() { return kSmemBytes; }

cudaError_t mla_decode_launch(const MlaParams& p, int clusters, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  static bool configured[kMaxDevices] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[device]) {
    e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured[device] = true;
  }
  if (attn_begin && (e = cudaEventRecord(attn_begin, stream)) != cudaSuccess) return e;
  mla_decode_kernel<<<2 * clusters, kThreads, kSmemBytes, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  const int64_t rows = int64_t(p.B) * kRows;
  mla_merge_kernel<<<int((rows + 3) / 4), 128, 0, stream>>>(p, clusters);
  return cudaGetLastError();
}

}  // namespace zl
