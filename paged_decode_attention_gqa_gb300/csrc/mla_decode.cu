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
// Warp roles (224 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 2-5 softmax / epilogue, one thread per head row (TMEM lane),
// warp 6 releases the exchange buffer to the peer.
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

constexpr int kTile = kMlaTile;               // tokens per tile
constexpr int kRows = 128;                    // query heads = TMEM lanes
constexpr int kBoxKV = kTile * 128;           // 4 KB: 32 tokens x 64 bf16
constexpr int kMaxBoxes = 5;                  // rank 0: 4 latent + 1 rope
constexpr int kStages = 3;
constexpr int kStageBytes = kMaxBoxes * kBoxKV;  // 40 KB
constexpr int kXRow = kTile * 4;                 // 256 B: one row of fp32 partial scores
constexpr int kXBytes = kRows * kXRow;           // 32 KB
constexpr int kOffKV = 0;
constexpr int kOffX = kOffKV + kStages * kStageBytes;  // received partials (single buffer)
constexpr int kOffStg = kOffX + kXBytes;               // own partials (double buffer)
constexpr int kOffBar = kOffStg + 2 * kXBytes;
enum : int {
  B_Q_FULL = 0,
  B_KV_FULL0, B_KV_EMPTY0 = B_KV_FULL0 + kStages, B_S_FULL = B_KV_EMPTY0 + kStages,
  B_S_EMPTY, B_P_FULL, B_PV_DONE, B_X_FULL, B_X_FREE, B_READ_DONE, B_STAGED0,
  B_FINAL = B_STAGED0 + 2,
  B_COUNT
};
constexpr int kOffMisc = kOffBar + 8 * B_COUNT;
constexpr int kOffPrefix = kOffMisc + 64;
constexpr size_t kSmemBytes = 1024 + kOffPrefix + size_t(kMlaMaxBatch + 1) * 4;
static_assert(kSmemBytes <= 232448, "MLA kernel exceeds 227 KB of shared memory");
static_assert(kOffKV % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle atoms need aligned buffers");
// TMEM columns (fp32 or bf16 pairs), 128 lanes = 128 heads:
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;                // O, this rank's 256 columns of D_v
constexpr uint32_t kTmemS = 256;              // S tile: kTile fp32 columns
constexpr uint32_t kTmemP = kTmemS + kTile;   // P tile: kTile bf16 = kTile / 2 columns
constexpr uint32_t kTmemQ = kTmemP + kTile / 2;  // Q, this rank's 320 or 256 dims
static_assert(kTmemQ + 160 <= kTmemCols, "TMEM holds O, S, P and Q");
constexpr int kThreads = 224;  // producer, MMA, 4 softmax warps, exchange warp

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
  // The units of work are (sequence b, query token i) pairs, v = b * q_len + i:
  // q, out and lse rows of v are contiguous, and v attends causally to the
  // first L_b - q_len + 1 + i tokens of sequence b's pages.
  const int B = p.B * p.q_len;
  const int64_t cap = p.bt_stride * int64_t(p.page_size);
  // Visible tokens of unit v (0 for an invalid sequence length).
  auto vis_len = [&](int v) -> int {
    const int L = p.seq_lens[v / p.q_len];
    if (!(L >= 0 && int64_t(L) <= cap)) return 0;
    const int n = L - p.q_len + 1 + v % p.q_len;
    return n > 0 ? n : 0;
  };

  if (tid == 0) {
    mbar_init(bar(B_Q_FULL), kRows);  // softmax threads wrote this piece's Q into TMEM
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_KV_FULL0 + s), 1);
      mbar_init(bar(B_KV_EMPTY0 + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_EMPTY), kRows);
    mbar_init(bar(B_P_FULL), kRows);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_X_FULL), 1);      // local expect_tx + the peer's bulk-copy bytes
    mbar_init(bar(B_X_FREE), 1);      // the peer has read our previous partial
    mbar_init(bar(B_READ_DONE), kRows);  // all rows of the received partial read
    for (int i = 0; i < 2; ++i)
      mbar_init(bar(B_STAGED0 + i), kRows);  // all rows of the outgoing partial written
    mbar_init(bar(B_FINAL), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Launched as a programmatic dependent of the kernel before it on the
  // stream: wait for it before touching global memory, and before taking
  // TMEM (a kernel still running on this SM may need its own).
  griddep_wait();
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmap_kv);
  }
  // Tiles (of 64 tokens) per sequence, exclusive prefix sum.
  if (warp == 2) {
    const int per = (B + 31) / 32;
    const int b0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int L = p.seq_lens[b / p.q_len];
        const bool ok = L >= 0 && int64_t(L) <= cap;
        if (!ok && blockIdx.x == 0) raise_error(p.err_flags, kErrBadLen);
        local += (vis_len(b) + kTile - 1) / kTile;
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
        run += (vis_len(b) + kTile - 1) / kTile;
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
  // The merge kernel may be scheduled from here on; it waits for this whole
  // grid to finish before it reads anything.
  griddep_launch_dependents();

  const int64_t W = prefix[B];
  const int64_t s_c = int64_t(cid) * W / NC;
  const int64_t e_c = int64_t(cid + 1) * W / NC;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int64_t idx = s_c; idx < e_c && ok;) {
        const int b = locate(prefix, B, idx);
        const int j0 = int(idx - prefix[b]);
        const int64_t pend = min(e_c, int64_t(prefix[b + 1]));
        for (int j = j0; j < j0 + int(pend - idx); ++j, ++it) {
          const int s = it % kStages;
          if (!mbar_wait(bar(B_KV_EMPTY0 + s), ((it / kStages) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const int tok0 = j * kTile;
          const int page =
              p.block_table[int64_t(b / p.q_len) * p.bt_stride + tok0 / p.page_size];
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
        idx = pend;
      }
      if (!ok) {
        raise_error(p.err_flags, kErrTimeout);
        *abort_flag = 1;
      }
      // Leave no copy in flight: wait for the last stages and the last Q.
      const volatile int never = 0;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        mbar_wait(bar(B_KV_FULL0 + j % kStages), (j / kStages) & 1, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // An event loop: issue whichever is ready first, QK of the next tile (its
    // K/V staged and the S tile read out by the softmax warps) or PV of the
    // oldest tile whose P is written.
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_bf16(kRows, kTile, false);
      const uint32_t idesc_pv = umma_idesc_bf16(kRows, 256, true);
      const int total = int(e_c - s_c);
      int qk = 0, pv = 0, qpiece = 0;
      bool ok = true;
      uint64_t last_progress = globaltimer_ns();
      while (pv < total && ok) {
        bool progressed = false;
        if (qk < total) {
          const int64_t idx = s_c + qk;
          const int b = locate(prefix, B, idx);
          const bool first = (qk == 0) || (idx == prefix[b]);
          const bool last = (qk == total - 1) || (idx + 1 == prefix[b + 1]);
          const int s = qk % kStages;
          if (mbar_test(bar(B_KV_FULL0 + s), (qk / kStages) & 1) &&
              mbar_test(bar(B_S_EMPTY), (qk & 1) ^ 1u) &&
              (!first || mbar_test(bar(B_Q_FULL), qpiece & 1))) {
            tc_fence_after();
            const uint32_t kvbase = sbase + kOffKV + s * kStageBytes;
            // S = Q K^T: A = Q from TMEM (16 dims = 8 columns per step), B = K
            // K-major with the 128-byte swizzle.
            for (int i = 0; i < nbox; ++i) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bdesc = umma_smem_desc(kvbase + i * kBoxKV + kk * 32, 0, 1024, 2);
                umma_bf16_tmem_a(tmem + kTmemS, tmem + kTmemQ + 32 * i + 8 * kk, bdesc, idesc_qk,
                                 (i | kk) ? 1u : 0u);
              }
            }
            umma_commit(bar(B_S_FULL));
            if (last) ++qpiece;
            ++qk;
            progressed = true;
          }
        }
        if (pv < qk && mbar_test(bar(B_P_FULL), pv & 1)) {
          const int64_t idx = s_c + pv;
          const int b = locate(prefix, B, idx);
          const bool first = (pv == 0) || (idx == prefix[b]);  // overwrite O
          tc_fence_after();
          // O[:, rank half] (+)= P V: A = P from TMEM (16 tokens = 8 columns per
          // step); B = V, MN-major with the 128-byte swizzle (8-token groups 1 KB
          // apart, the next 64 columns in the next box).
          const int s = pv % kStages;
          const uint32_t vbase = sbase + kOffKV + s * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint64_t bdesc = umma_smem_desc(vbase + kk * 16 * 128, kBoxKV, 1024, 2);
            umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + 8 * kk, bdesc, idesc_pv,
                             (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(bar(B_KV_EMPTY0 + s));
          umma_commit(bar(B_PV_DONE));
          ++pv;
          progressed = true;
        }
        if (progressed) {
          last_progress = globaltimer_ns();
        } else if (*abort_flag || globaltimer_ns() - last_progress > kWaitTimeoutNs) {
          ok = false;
        }
      }
      if (!ok) {
        raise_error(p.err_flags, kErrTimeout);
        *abort_flag = 1;
      }
      // Every MMA done before TMEM is released.
      umma_commit(bar(B_FINAL));
      const volatile int never = 0;
      mbar_wait(bar(B_FINAL), 0, &never);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ exchange warp
    // Once all rows of received tile j are read, tell the peer its next bulk
    // copy may land (the remote arrive's latency stays off the softmax path).
    if (lane == 0) {
      const uint32_t peer_xfree = mapa_shared(bar(B_X_FREE), peer);
      const int total = int(e_c - s_c);
      for (int j = 0; j < total; ++j) {
        if (!mbar_wait(bar(B_READ_DONE), j & 1, abort_flag)) {
          raise_error(p.err_flags, kErrTimeout);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_remote(peer_xfree);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;                 // query head = TMEM lane
    const uint32_t tl = tmem + (uint32_t(32 * q4) << 16);
    const float c = p.scale_log2;
    const uint32_t peer_x = mapa_shared(sbase + kOffX, peer);
    const uint32_t peer_xfull = mapa_shared(bar(B_X_FULL), peer);
    const int stid = tid - 64;                       // 0..127 within the softmax group
    const int total = int(e_c - s_c);                // tiles of this cluster
    // 16-byte chunk k of this row in an exchange buffer (swizzled by row).
    auto xaddr = [&](uint32_t buf, int k) -> uint32_t {
      return buf + uint32_t(row * kXRow) + ((uint32_t(k) ^ uint32_t(row & 7)) << 4);
    };

    // send(j): this rank's partial scores of tile j. The rows go to the local
    // staging buffer j & 1 (they are re-read from there when tile j is summed);
    // once all 128 are there, one thread bulk-copies the buffer into the peer's
    // receive buffer j & 1, crediting the bytes to the peer's X_FULL barrier.
    // No flow-control barrier is needed: the peer sends tile j + 2 into our
    // buffer only after receiving our tile j + 1, which we send after summing
    // tile j; and staging buffer j & 1 is rewritten only after the peer's tile
    // j + 1 reached us, which the peer sent after receiving our tile j.
    auto send = [&](int j) -> bool {
      const int xb = j & 1;
      if (!mbar_wait(bar(B_S_FULL), j & 1, abort_flag)) return false;
      tc_fence_after();
      const uint32_t stg = sbase + kOffStg + xb * kXBytes;
#pragma unroll 1
      for (int h = 0; h < kTile / 32; ++h) {
        uint32_t v[32];
        tmem_ld32(tl + kTmemS + 32 * h, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xaddr(stg, 8 * h + k)),
                       "r"(v[4 * k]), "r"(v[4 * k + 1]), "r"(v[4 * k + 2]), "r"(v[4 * k + 3])
                       : "memory");
      }
      tc_fence_before();
      mbar_arrive(bar(B_S_EMPTY));                   // QK of the next tile may start
      fence_proxy_async_smem();
      mbar_arrive(bar(B_STAGED0 + xb));
      if (stid == 0) {
        if (!mbar_wait(bar(B_STAGED0 + xb), (j >> 1) & 1, abort_flag)) return false;
        // the peer's single receive buffer must have been read (tile j - 1)
        if (j >= 1 && !mbar_wait_cluster(bar(B_X_FREE), (j - 1) & 1, abort_flag)) return false;
        bulk_copy_to_peer(peer_x, stg, kXBytes, peer_xfull);
      }
      return true;
    };

    // Q of sequence b (this rank's columns, 2 bf16 per 32-bit column) into
    // TMEM, one head row per thread; the MMA issuer waits on Q_FULL.
    auto load_q = [&](int b) {
      const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (int64_t(b) * kRows + row) * kMlaDqk);
      for (int i = 0; i < nbox; ++i) {
        const int col = i < 4 ? int(rank) * 256 + 64 * i : 512;
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 u = __ldg(qrow + col / 8 + k);
          v[4 * k] = u.x;
          v[4 * k + 1] = u.y;
          v[4 * k + 2] = u.z;
          v[4 * k + 3] = u.w;
        }
        tmem_st32(tl + kTmemQ + 32 * i, v);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_Q_FULL));
    };

    if (total > 0) load_q(locate(prefix, B, s_c));
    bool ok = total == 0 || send(0);
    int it = 0;
    for (int64_t idx = s_c; idx < e_c && ok;) {
      const int b = locate(prefix, B, idx);
      const int j0 = int(idx - prefix[b]);
      const int64_t pend = min(e_c, int64_t(prefix[b + 1]));
      const int ntiles = int(pend - idx);
      const bool partial = (j0 > 0) || (pend < prefix[b + 1]);
      const int slot = (idx == s_c) ? 0 : 1;
      const int L = vis_len(b);
      const int32_t* bt_row = p.block_table + int64_t(b / p.q_len) * p.bt_stride;
      float m_used = -CUDART_INF_F, l = 0.f;
      int bad = 0;
      int page_cur = bt_row[(j0 * kTile) / p.page_size];
      for (int t = 0; t < ntiles; ++t, ++it) {
        const int xb = it & 1;
        const int tok0 = (j0 + t) * kTile;
        const int valid = min(kTile, L - tok0);
        // block-table entry of the next tile, loaded one tile ahead
        const int page_nxt = (t + 1 < ntiles) ? bt_row[(tok0 + kTile) / p.page_size] : 0;
        bad |= (page_cur < 0 || page_cur >= p.num_pages) ? 1 : 0;

        // receive the peer's partial of this tile; S = own + peer
        if (stid == 0) mbar_arrive_expect_tx(bar(B_X_FULL), kXBytes);
        if (!mbar_wait_cluster(bar(B_X_FULL), it & 1, abort_flag)) { ok = false; break; }
        float x[kTile];
        {
          const uint32_t own = sbase + kOffStg + xb * kXBytes;
          const uint32_t got = sbase + kOffX;
#pragma unroll
          for (int k = 0; k < kTile / 4; ++k) {
            float a0, a1, a2, a3, b0, b1, b2, b3;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(a0), "=f"(a1), "=f"(a2), "=f"(a3) : "r"(xaddr(own, k)) : "memory");
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(b0), "=f"(b1), "=f"(b2), "=f"(b3) : "r"(xaddr(got, k)) : "memory");
            x[4 * k] = a0 + b0;
            x[4 * k + 1] = a1 + b1;
            x[4 * k + 2] = a2 + b2;
            x[4 * k + 3] = a3 + b3;
          }
        }
        mbar_arrive(bar(B_READ_DONE));  // the exchange warp releases the buffer to the peer
        // online softmax (base 2); the max moves only when it grows by > 8
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < kTile; ++k) {
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
        uint32_t pk[kTile / 2];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < kTile / 2; ++k) {
          pk[k] = pack_bf16x2(ex2_approx(x[2 * k] - m_used), ex2_approx(x[2 * k + 1] - m_used));
          const float2 f = unpack_bf16x2(pk[k]);
          lsum += f.x + f.y;
        }
        l = l * alpha + lsum;

        // tail tile: zero the V rows past the end (NaN there would poison 0 * V)
        if (valid < kTile) {
          const uint32_t vb = sbase + kOffKV + (it % kStages) * kStageBytes;
          const int nz = (kTile - valid) * 4 * 8;  // 16-byte chunks in 4 latent boxes
          for (int z = stid; z < nz; z += kRows) {
            const int chunk = z & 7, box = (z >> 3) & 3, r = valid + (z >> 5);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + box * kBoxKV + r * 128 + chunk * 16),
                         "r"(0u)
                         : "memory");
          }
        }

        // The P tile in TMEM is free (and O stable for a rescale) once PV(it - 1)
        // finished.
        if (it >= 1 && !mbar_wait(bar(B_PV_DONE), (it - 1) & 1, abort_flag)) { ok = false; break; }
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
        }
        tmem_st32(tl + kTmemP, pk);                  // P row: 64 bf16 in 32 columns
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL));

        // send the next tile's partial; a new sequence first needs its Q in TMEM
        // (every QK of this one is done: this tile's S was read out)
        if (it + 1 < total && t + 1 == ntiles) load_q(locate(prefix, B, s_c + it + 1));
        if (it + 1 < total && !send(it + 1)) { ok = false; break; }
        page_cur = page_nxt;
      }
      if (!ok) break;

      // ---- epilogue of the piece: O / l
      if (!mbar_wait(bar(B_PV_DONE), (it - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
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
// sequence cut between clusters, in cluster order. A programmatic dependent
// launch of the attention kernel: it waits here until that grid is done.
__global__ void __launch_bounds__(128) mla_merge_kernel(const __grid_constant__ MlaParams p,
                                                        int NC) {
  griddep_wait();
  griddep_launch_dependents();  // the next call's kernels may start their prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + warp;
  if (row >= int64_t(p.B) * p.q_len * kRows) return;
  const int b = int(row / kRows), h = int(row % kRows);
  const int* prefix = p.ws_prefix;
  const int n = prefix[b + 1] - prefix[b];
  if (n == 0) return;
  const int64_t W = prefix[p.B * p.q_len];
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
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(2 * clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, p)) != cudaSuccess) return e;
  }
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  const int64_t rows = int64_t(p.B) * p.q_len * kRows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel, p, clusters);
}

}  // namespace zl
