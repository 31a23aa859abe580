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
// whole of TMEM (512 columns x 128 lanes). So a cluster of two CTAs shares
// each range of 64-token tiles, and each CTA owns half of O: rank r
// accumulates O columns [256r, 256r + 256) in TMEM. Both ranks compute the
// whole score tile S = Q K^T (M = 128 heads, N = 64 tokens, K = 576) and run
// the same softmax; computing S twice costs less tensor time than trading
// fp32 partial scores between the CTAs every tile. Both CTAs load every tile
// at about the same time, so the second load is served by L2.
//
// Where the operands live (per CTA):
//   TMEM: O (256 columns) | S (64) | P (64 bf16 = 32) | Q of this rank's
//         latent half and the rope (320 dims = 160 columns);
//   smem: Q of the other latent half (128 x 256 bf16, 128-byte swizzle) and
//         two stages of K/V, each split into an "E" part (the other latent
//         half and the rope: read by QK only) and an "L" part (this rank's
//         latent half: read by QK and then, as V, by PV).
// The E part of a stage is released when the QK that reads it is done, the L
// part when the PV is done, and every tile's QK starts with its E part, so the
// loads of tile j + 2 have about a whole tile of slack with two stages.
//
// Warp roles (224 threads): warp 0 loads the E parts, warp 6 the L parts
// (TMA), warp 1 issues the MMAs (and owns TMEM), warps 2-5 softmax /
// epilogue, one thread per head row (TMEM lane). The MMA issuer interleaves
// PV of tile j - 1 between the two halves of QK of tile j when P is ready.
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
constexpr int kBox = kTile * 128;             // 8 KB: kTile tokens x 64 bf16
constexpr int kEBoxes = 5;                    // other latent half (4 boxes) + rope
constexpr int kLBoxes = 4;                    // this rank's latent half
constexpr int kStages = 2;
constexpr int kEBytes = kEBoxes * kBox;       // 40 KB
constexpr int kLBytes = kLBoxes * kBox;       // 32 KB
constexpr int kQBox = kRows * 128;            // 16 KB: 128 heads x 64 dims of Q
constexpr int kOffE = 0;
constexpr int kOffL = kOffE + kStages * kEBytes;
constexpr int kOffQ = kOffL + kStages * kLBytes;  // Q of the other latent half
constexpr int kOffBar = kOffQ + 4 * kQBox;
enum : int {
  B_Q_FULL = 0,
  B_E_FULL0, B_E_EMPTY0 = B_E_FULL0 + kStages,
  B_L_FULL0 = B_E_EMPTY0 + kStages, B_L_EMPTY0 = B_L_FULL0 + kStages,
  B_S_FULL = B_L_EMPTY0 + kStages, B_S_EMPTY, B_P_FULL, B_PV_DONE, B_FINAL,
  B_Q_STAGED, B_Q_USED,  // the softmax threads' own syncs around the Q staging buffer
  B_APPEND,  // fused append: the softmax threads stored the new rows
  B_COUNT
};
constexpr int kOffMisc = kOffBar + 8 * B_COUNT;
constexpr int kOffPrefix = kOffMisc + 64;                            // tile prefix sums
constexpr int kOffCost = kOffPrefix + (kMlaMaxBatch + 1) * 4 + 12;  // cost prefix sums
constexpr size_t kSmemBytes = 1024 + kOffCost + size_t(kMlaMaxBatch + 1) * 4;
static_assert(kSmemBytes <= 232448, "MLA kernel exceeds 227 KB of shared memory");
static_assert(kOffL % 1024 == 0 && kOffQ % 1024 == 0 && kEBytes % 1024 == 0 &&
                  kLBytes % 1024 == 0,
              "swizzle atoms need 1024-byte aligned buffers");
// TMEM columns (fp32 or bf16 pairs), 128 lanes = 128 heads:
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;                // O, this rank's 256 columns of D_v
constexpr uint32_t kTmemS = 256;              // S tile: kTile fp32 columns
constexpr uint32_t kTmemP = kTmemS + kTile;   // P tile: kTile bf16 = kTile / 2 columns
constexpr uint32_t kTmemQ = kTmemP + kTile / 2;  // Q: this rank's latent half, then the rope
static_assert(kTmemQ + 160 <= kTmemCols, "TMEM holds O, S, P and Q");
constexpr int kThreads = 224;  // E producer, MMA, 4 softmax warps, L producer

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

// Wait on an mbarrier with the whole warp by polling with test_wait (which
// never suspends the warp, so the MMA issuer sees a completed phase at once);
// true on every lane only if the phase completed, false on every lane after a
// timeout or an abort.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          const volatile int* abort_flag) {
  if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (__all_sync(0xffffffffu, mbar_test(bar, parity))) return true;
    if ((i & 63u) == 0) {
      const bool stop = *abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs;
      if (__any_sync(0xffffffffu, stop)) return false;
    }
  }
}

// Fused KV append, by the softmax threads (thread `tid` of `nthreads`) while
// the first loads are in flight: every new token that the tiles [s_c, e_c) of
// the units `prefix` lays out hold is copied from kv_new into its pool slot
// (all 576 columns), and the stores are fenced against the bulk copies that
// read those pages. Both CTAs of the pair, and every unit of a sequence that
// sees the token, store the same bytes.
__device__ __noinline__ void append_new_rows(const MlaParams& p, const int* prefix, int B,
                                             int64_t s_c, int64_t e_c, int tid, int nthreads) {
  constexpr int kChunks = kMlaDqk / 8;  // 16-byte chunks of a row
  const int64_t cap = p.bt_stride * int64_t(p.page_size);
  for (int u = e_c > s_c ? locate(prefix, B, s_c) : B; u < B && prefix[u] < e_c; ++u) {
    const int64_t j_lo = max(s_c, int64_t(prefix[u])) - prefix[u];
    const int64_t j_hi = min(e_c, int64_t(prefix[u + 1])) - prefix[u];
    if (j_hi <= j_lo) continue;
    const int b = u / p.q_len;
    const int L = p.seq_lens[b];
    if (!(L >= p.q_len && int64_t(L) <= cap)) continue;
    const int t0 = L - p.q_len;            // the call's first new token
    const int vis = t0 + 1 + u % p.q_len;  // tokens unit u sees
    const int t_lo = max(int(j_lo) * kTile, t0);
    const int t_hi = min(int(j_hi) * kTile, vis);
    for (int c = tid; c < (t_hi - t_lo) * kChunks; c += nthreads) {
      const int t = t_lo + c / kChunks, col = c % kChunks;
      const int page = p.block_table[int64_t(b) * p.bt_stride + t / p.page_size];
      if (page < 0 || page >= p.num_pages) continue;
      p.kv_pool[int64_t(page) * p.page_stride16 + int64_t(t % p.page_size) * p.token_stride16 +
                col] = __ldg(p.kv_new + (int64_t(b) * p.q_len + (t - t0)) * kChunks + col);
    }
  }
  fence_proxy_async_global();
}

// APPEND: the instance that also stores the new tokens' rows (p.kv_new); the
// plain instance has none of that code.
template <bool APPEND>
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
  int* cost = reinterpret_cast<int*>(smem + kOffCost);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = int(cluster_ctarank()), other = rank ^ 1;
  const int cid = blockIdx.x >> 1, NC = gridDim.x >> 1;
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
    mbar_init(bar(B_Q_FULL), kRows);  // softmax threads wrote this piece's Q
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_E_FULL0 + s), 1);
      mbar_init(bar(B_E_EMPTY0 + s), 1);
      mbar_init(bar(B_L_FULL0 + s), 1);
      mbar_init(bar(B_L_EMPTY0 + s), 1);
    }
    mbar_init(bar(B_S_FULL), 1);
    mbar_init(bar(B_S_EMPTY), kRows);
    mbar_init(bar(B_P_FULL), kRows);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_FINAL), 1);
    mbar_init(bar(B_Q_STAGED), kRows);
    mbar_init(bar(B_Q_USED), kRows);
    if constexpr (APPEND) mbar_init(bar(B_APPEND), kRows);
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
  if ((warp == 0 || warp == 6) && lane == 0) {
    tma_prefetch_desc(&p.tmap_kv);
  }
  // Tiles (of 64 tokens) per unit, exclusive prefix sum; and the same for the
  // cost of a unit: its tiles plus kMlaUnitCost when it has any (its Q load
  // and epilogue), which the clusters share equally.
  if (warp == 2) {
    const int per = (B + 31) / 32;
    const int b0 = lane * per;
    int local = 0, local_cost = 0;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        const int L = p.seq_lens[b / p.q_len];
        const bool ok = L >= 0 && int64_t(L) <= cap;
        if (!ok && blockIdx.x == 0) raise_error(p.err_flags, kErrBadLen);
        const int n = (vis_len(b) + kTile - 1) / kTile;
        local += n;
        local_cost += n > 0 ? n + kMlaUnitCost : 0;
      }
    }
    int incl = local, incl_cost = local_cost;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      const int vc = __shfl_up_sync(0xffffffffu, incl_cost, off);
      if (lane >= off) {
        incl += v;
        incl_cost += vc;
      }
    }
    int run = incl - local, run_cost = incl_cost - local_cost;
    for (int i = 0; i < per; ++i) {
      const int b = b0 + i;
      if (b < B) {
        prefix[b] = run;
        cost[b] = run_cost;
        const int n = (vis_len(b) + kTile - 1) / kTile;
        run += n;
        run_cost += n > 0 ? n + kMlaUnitCost : 0;
      }
    }
    if (lane == 31) {
      prefix[B] = incl;
      cost[B] = incl_cost;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // This cluster's tiles [s_c, e_c): equal shares of the cost line, mapped
  // back to tiles (a share that starts inside a unit's fixed cost starts at
  // the unit's first tile).
  const int64_t W = prefix[B];
  auto tile_at = [&](int64_t a) -> int64_t {
    if (a >= cost[B]) return W;
    const int u = locate(cost, B, a);
    const int64_t o = a - cost[u] - kMlaUnitCost;
    return prefix[u] + (o > 0 ? o : 0);
  };
  const int64_t s_c = tile_at(int64_t(cid) * cost[B] / NC);
  const int64_t e_c = tile_at(int64_t(cid + 1) * cost[B] / NC);

  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += kThreads) p.ws_prefix[b] = prefix[b];
  if (rank == 0 && tid == 0) {
    p.ws_split[cid] = int32_t(s_c);
    if (cid == NC - 1) p.ws_split[NC] = int32_t(e_c);
  }
  // The merge kernel may be scheduled from here on; it waits for this whole
  // grid to finish before it reads anything.
  griddep_launch_dependents();

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ------------------------------------------------------------ producers
    // Warp 0 streams the E parts (the other latent half and the rope), warp 6
    // the L parts (this rank's latent half) of the tiles of this cluster.
    const bool e_part = warp == 0;
    const int full0 = e_part ? B_E_FULL0 : B_L_FULL0;
    const int empty0 = e_part ? B_E_EMPTY0 : B_L_EMPTY0;
    const uint32_t region = sbase + (e_part ? kOffE : kOffL);
    const int stage_bytes = e_part ? kEBytes : kLBytes;
    const int nbox = e_part ? kEBoxes : kLBoxes;
    const int half = e_part ? other : rank;
    const int total = int(e_c - s_c);
    // Tile `it` is tile j of unit b; the block-table entry of the next tile
    // is read one tile ahead, so its latency is hidden behind the stage wait.
    int b = total > 0 ? locate(prefix, B, s_c) : 0;
    int j = total > 0 ? int(s_c - prefix[b]) : 0;
    int64_t ub_end = total > 0 ? prefix[b + 1] : 0;
    auto page_of = [&](int u, int jt) -> int {
      return p.block_table[int64_t(u / p.q_len) * p.bt_stride + (jt * kTile) / p.page_size];
    };
    int page = total > 0 ? page_of(b, j) : 0;
    bool appended = false;  // the softmax threads stored the new rows (APPEND instance)
    // APPEND: the unit's first new token, read one unit ahead like the pages
    int t0_cur = 0;
    if constexpr (APPEND) t0_cur = total > 0 ? p.seq_lens[b / p.q_len] - p.q_len : 0;
    int it = 0;
    bool ok = true;
    for (; it < total; ++it) {
      const int s = it % kStages;
      const int tok0 = j * kTile;
      // advance to the next tile (skipping units without tiles) and read its page
      const int64_t nidx = s_c + it + 1;
      int nb = b, nj = j + 1;
      if (nidx == ub_end && it + 1 < total) {
        do {
          ++nb;
        } while (prefix[nb + 1] <= nidx);
        nj = 0;
      }
      const int page_next = it + 1 < total ? page_of(nb, nj) : 0;
      int t0_next = t0_cur;
      if constexpr (APPEND) {
        if (nb != b && it + 1 < total) t0_next = p.seq_lens[nb / p.q_len] - p.q_len;
      }
      if (!mbar_wait(bar(empty0 + s), ((it / kStages) & 1) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      if (page < 0 || page >= p.num_pages) {
        mbar_arrive(bar(full0 + s));  // nothing loaded; the piece is discarded
      } else {
        if constexpr (APPEND) {  // a tile that holds a new token waits for its rows
          const int vis = t0_cur + 1 + b % p.q_len;  // tokens unit b sees
          if (!appended && tok0 + kTile > t0_cur && tok0 < vis) {
            if (!mbar_wait(bar(B_APPEND), 0, abort_flag)) {
              ok = false;
              break;
            }
            appended = true;
          }
        }
        const int slot = tok0 % p.page_size;
        mbar_arrive_expect_tx(bar(full0 + s), uint32_t(stage_bytes));
        for (int i = 0; i < nbox; ++i) {
          const int col = i < 4 ? half * 256 + 64 * i : 512;
          tma_load_3d(region + s * stage_bytes + i * kBox, &p.tmap_kv, bar(full0 + s), col, slot,
                      page);
        }
      }
      if (nb != b) ub_end = prefix[nb + 1];
      b = nb;
      j = nj;
      page = page_next;
      t0_cur = t0_next;
    }
    if (!ok) {
      raise_error(p.err_flags, kErrTimeout);
      *abort_flag = 1;
    }
    // Leave no copy in flight: wait for the last stages to land.
    const volatile int never = 0;
    for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
      mbar_wait(bar(full0 + j % kStages), (j / kStages) & 1, &never);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and bookkeeping are warp-uniform);
    // one elected lane issues. Per tile k: QK over the E part (Q from shared
    // memory for the other latent half, from TMEM for the rope), then PV of
    // tile k - 1 if its P is already written, then QK over the L part (Q from
    // TMEM), then PV of tile k - 1 if it was not issued yet.
    const uint32_t idesc_qk = umma_idesc_bf16(kRows, kTile, false);
    const uint32_t idesc_pv = umma_idesc_bf16(kRows, 256, true);
    const uint32_t qs = sbase + kOffQ;
    const int total = int(e_c - s_c);
    int qpiece = 0, pv_next = 0;
    bool ok = true;
    // The unit of the current tile and the end of its tiles, kept in
    // registers: shared memory is only read when a new unit starts.
    int ub = total > 0 ? locate(prefix, B, s_c) : 0;
    int64_t ub_end = total > 0 ? prefix[ub + 1] : 0;
    bool cur_first = true;  // tile k starts a unit (its PV overwrites O)
    // O[:, rank half] (+)= P V: A = P from TMEM (16 tokens = 8 columns per
    // step); B = V, MN-major with the 128-byte swizzle (8-token groups 1 KB
    // apart, the next 64 columns in the next box).
    auto issue_pv = [&](int j, bool first) {
      const int s = j % kStages;
      const uint32_t vbase = sbase + kOffL + s * kLBytes;
      tc_fence_after();
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t bdesc = umma_smem_desc(vbase + kk * 16 * 128, kBox, 1024, 2);
          umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + 8 * kk, bdesc, idesc_pv,
                           (first && kk == 0) ? 0u : 1u);
        }
        umma_commit(bar(B_L_EMPTY0 + s));
        umma_commit(bar(B_PV_DONE));
      }
      __syncwarp();
    };
    for (int k = 0; k < total && ok; ++k) {
      const int64_t idx = s_c + k;
      const bool prev_first = cur_first;  // of tile k - 1
      cur_first = k == 0;
      if (idx == ub_end) {  // the next unit with tiles
        do {
          ++ub;
          ub_end = prefix[ub + 1];
        } while (ub_end <= idx);
        cur_first = true;
      }
      const bool first = cur_first;
      const bool last = (k == total - 1) || (idx + 1 == ub_end);
      const int s = k % kStages;
      // A new unit: finish the previous one first (its last PV is what the
      // epilogue waits for; the new unit's Q may still be loading).
      if (first && pv_next < k) {
        if (!warp_wait(bar(B_P_FULL), (k - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        issue_pv(k - 1, prev_first);
        ++pv_next;
      }
      const uint32_t ph = (k / kStages) & 1;
      // a new unit needs its Q; S must have been read out; the E part loaded
      if ((first && !warp_wait(bar(B_Q_FULL), qpiece & 1, abort_flag)) ||
          !warp_wait(bar(B_S_EMPTY), (k & 1) ^ 1u, abort_flag) ||
          !warp_wait(bar(B_E_FULL0 + s), ph, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const uint32_t ebase = sbase + kOffE + s * kEBytes;
        if (elect_one()) {
          // S = Q K^T over the other latent half: A = Q in shared memory, B =
          // K, both K-major with the 128-byte swizzle (16 dims = 32 bytes per
          // step).
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = umma_smem_desc(qs + i * kQBox + kk * 32, 0, 1024, 2);
              const uint64_t bdesc = umma_smem_desc(ebase + i * kBox + kk * 32, 0, 1024, 2);
              umma_bf16(tmem + kTmemS, adesc, bdesc, idesc_qk, (i | kk) ? 1u : 0u);
            }
          }
          // ... and over the rope: A = Q in TMEM (16 dims = 8 columns per step)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = umma_smem_desc(ebase + 4 * kBox + kk * 32, 0, 1024, 2);
            umma_bf16_tmem_a(tmem + kTmemS, tmem + kTmemQ + 128 + 8 * kk, bdesc, idesc_qk, 1u);
          }
          umma_commit(bar(B_E_EMPTY0 + s));
        }
        __syncwarp();
      }
      if (pv_next < k && __all_sync(0xffffffffu, mbar_test(bar(B_P_FULL), (k - 1) & 1))) {
        issue_pv(k - 1, prev_first);
        ++pv_next;
      }
      if (!warp_wait(bar(B_L_FULL0 + s), ph, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const uint32_t lbase = sbase + kOffL + s * kLBytes;
        if (elect_one()) {
          // S += Q K^T over this rank's latent half, A = Q from TMEM.
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = umma_smem_desc(lbase + i * kBox + kk * 32, 0, 1024, 2);
              umma_bf16_tmem_a(tmem + kTmemS, tmem + kTmemQ + 32 * i + 8 * kk, bdesc, idesc_qk,
                               1u);
            }
          }
          umma_commit(bar(B_S_FULL));
        }
        __syncwarp();
      }
      if (last) ++qpiece;
      if (pv_next < k) {
        if (!warp_wait(bar(B_P_FULL), (k - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        issue_pv(k - 1, prev_first);
        ++pv_next;
      }
    }
    if (ok && pv_next < total) {
      if (warp_wait(bar(B_P_FULL), (total - 1) & 1, abort_flag))
        issue_pv(total - 1, cur_first);
      else
        ok = false;
    }
    if (!ok && lane == 0) {
      raise_error(p.err_flags, kErrTimeout);
      *abort_flag = 1;
    }
    // Every MMA done before TMEM is released.
    if (elect_one()) umma_commit(bar(B_FINAL));
    __syncwarp();
    const volatile int never = 0;
    mbar_wait(bar(B_FINAL), 0, &never);
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;                 // query head = TMEM lane
    const uint32_t tl = tmem + (uint32_t(32 * q4) << 16);
    const float c = p.scale_log2;
    const int stid = tid - 64;                       // 0..127 within the softmax group
    const int total = int(e_c - s_c);                // tiles of this cluster
    const uint32_t qs = sbase + kOffQ;

    // Q of unit v: this rank's latent half and the rope into TMEM (one head
    // row per TMEM lane, 2 bf16 per 32-bit column), the other latent half
    // into shared memory in the 128-byte swizzled K-major layout. Global reads
    // are coalesced (one warp copies one 512-byte row segment per
    // instruction): the latent half bound for TMEM is first staged in the Q
    // buffer (row-contiguous, 16-byte chunk c of row r at c ^ (r % 32)), read
    // back one row per thread and written to TMEM; then the other half is
    // copied into its final place. Phase 1 (q_stage) may start as soon as
    // every QK of the previous piece is done; phase 2 (q_finish) publishes Q
    // to the MMA issuer (Q_FULL).
    // Waits of the softmax warps end the same way on every lane (the TMEM
    // loads and stores after them are warp-wide).
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, abort_flag));
    };
    auto q_base = [&](int v) -> const uint4* {
      return reinterpret_cast<const uint4*>(p.q + int64_t(v) * kRows * kMlaDqk);
    };
    // chunk i * 128 + stid of the 128 x 32 grid of 16-byte chunks of a half
    auto q_stage = [&](int v) {
      const uint4* qb = q_base(v);
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const int c = i * 128 + stid, r = c >> 5, k = c & 31;
        cp_async_16(qs + uint32_t(r * 512 + ((k ^ (r & 31)) << 4)), qb + r * (kMlaDqk / 8) + rank * 32 + k);
      }
    };
    int qn = 0;  // Q loads so far (phase parity of Q_STAGED and Q_USED)
    auto q_finish = [&](int v) -> bool {
      const uint4* qb = q_base(v);
      cp_async_wait_all();
      mbar_arrive(bar(B_Q_STAGED));  // every staged row has landed
      if (!wait_all(bar(B_Q_STAGED), qn & 1)) return false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t r32[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t src = qs + uint32_t(row * 512 + (((8 * i + k) ^ (row & 31)) << 4));
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(r32[4 * k]), "=r"(r32[4 * k + 1]), "=r"(r32[4 * k + 2]),
                         "=r"(r32[4 * k + 3])
                       : "r"(src)
                       : "memory");
        }
        tmem_st32(tl + kTmemQ + 32 * i, r32);
      }
      mbar_arrive(bar(B_Q_USED));  // the staging rows are consumed
      if (!wait_all(bar(B_Q_USED), qn & 1)) return false;
      ++qn;
      // the other latent half, straight into the swizzled operand layout
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const int c = i * 128 + stid, r = c >> 5, k = c & 31;  // k: 16-byte chunk of 32
        cp_async_16(qs + uint32_t((k >> 3) * kQBox + r * 128) + ((uint32_t(k & 7) ^ uint32_t(r & 7)) << 4),
                    qb + r * (kMlaDqk / 8) + other * 32 + k);
      }
      // the rope (128 bytes of this thread's row)
      {
        const uint4* qrow = qb + row * (kMlaDqk / 8) + 64;
        uint32_t r32[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 u = __ldg(qrow + k);
          r32[4 * k] = u.x;
          r32[4 * k + 1] = u.y;
          r32[4 * k + 2] = u.z;
          r32[4 * k + 3] = u.w;
        }
        tmem_st32(tl + kTmemQ + 128, r32);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_Q_FULL));
      return true;
    };
    // L2 prefetch of the Q rows of unit v (128 heads x 576 bf16, contiguous).
    auto q_prefetch = [&](int v) {
      const char* base = reinterpret_cast<const char*>(p.q + int64_t(v) * kRows * kMlaDqk);
      constexpr uint32_t kQBytes = uint32_t(kRows) * kMlaDqk * 2;  // 147456
      for (uint32_t off = 0; off < kQBytes; off += 16384u)
        prefetch_l2_bulk(base + off, min(16384u, kQBytes - off));
    };

    bool ok = true;
    if (total > 0) {
      const int v0 = locate(prefix, B, s_c);
      q_stage(v0);
      ok = q_finish(v0);
      if constexpr (APPEND) {
        // Fused KV append while the first tile's QK runs (the softmax threads
        // wait for its scores anyway); a producer loads a tile that holds a
        // new token only after this.
        append_new_rows(p, prefix, B, s_c, e_c, stid, kRows);
        mbar_arrive(bar(B_APPEND));
      }
    }
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
      // the first and the last cluster holding tiles of unit b, for the merge
      if (rank == 0 && stid == 0) {
        if (j0 == 0) p.ws_span[2 * b] = 2 * cid + slot;  // and its partial's slot
        if (pend == prefix[b + 1]) p.ws_span[2 * b + 1] = cid;
      }
      if (stid == 0 && pend < e_c) q_prefetch(locate(prefix, B, pend));
      int page_cur = bt_row[(j0 * kTile) / p.page_size];
      for (int t = 0; t < ntiles; ++t, ++it) {
        const int tok0 = (j0 + t) * kTile;
        const int valid = min(kTile, L - tok0);
        // block-table entry of the next tile, loaded one tile ahead
        const int page_nxt = (t + 1 < ntiles) ? bt_row[(tok0 + kTile) / p.page_size] : 0;
        bad |= (page_cur < 0 || page_cur >= p.num_pages) ? 1 : 0;

        // S of this tile: TMEM -> registers, then hand the columns back
        if (!wait_all(bar(B_S_FULL), it & 1)) { ok = false; break; }
        tc_fence_after();
        float x[kTile];
        {
          uint32_t s0[32], s1[32];
          tmem_ld32(tl + kTmemS, s0);
          tmem_ld32(tl + kTmemS + 32, s1);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            x[k] = __uint_as_float(s0[k]);
            x[32 + k] = __uint_as_float(s1[k]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_S_EMPTY));  // QK of the next tile may start
        // Every QK of this unit's piece is done: the next piece's Q may go in
        // (the shared-memory part now, the TMEM part once P is written).
        const int v_next = (it + 1 < total && t + 1 == ntiles) ? locate(prefix, B, s_c + it + 1) : -1;
        if (v_next >= 0) q_stage(v_next);

        // online softmax (base 2); the max moves only when it grows by > 8.
        // The max is taken on the raw scores (c > 0, so max(c x) = c max(x)
        // exactly) and the scale goes into the exponent's FFMA; four partial
        // maxima and sums keep the dependency chains short.
        if (valid < kTile) {  // the same for every row: no divergence
#pragma unroll
          for (int k = 0; k < kTile; ++k)
            if (k >= valid) x[k] = -CUDART_INF_F;
        }
        float mq[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int k = 4; k < kTile; ++k) mq[k & 3] = fmaxf(mq[k & 3], x[k]);
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * c;
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
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kTile / 2; ++k) {
          pk[k] = pack_bf16x2(ex2_approx(fmaf(x[2 * k], c, -m_used)),
                              ex2_approx(fmaf(x[2 * k + 1], c, -m_used)));
          const float2 f = unpack_bf16x2(pk[k]);
          ls[k & 3] += f.x + f.y;
        }
        l = l * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));

        // tail tile: zero the V rows past the end (NaN there would poison 0 * V)
        if (valid < kTile) {
          const uint32_t vb = sbase + kOffL + (it % kStages) * kLBytes;
          const int nz = (kTile - valid) * kLBoxes * 8;  // 16-byte chunks in the V boxes
          for (int z = stid; z < nz; z += kRows) {
            const int chunk = z & 7, box = (z >> 3) & 3, r = valid + (z >> 5);
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + box * kBox + r * 128 + chunk * 16),
                         "r"(0u)
                         : "memory");
          }
          fence_proxy_async_smem();  // the PV MMA reads these rows
        }

        // The P tile in TMEM is free (and O stable for a rescale) once PV(it - 1)
        // finished.
        if (it >= 1 && !wait_all(bar(B_PV_DONE), (it - 1) & 1)) { ok = false; break; }
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
        if (v_next >= 0 && !q_finish(v_next)) { ok = false; break; }
        page_cur = page_nxt;
      }
      if (!ok) break;

      // ---- epilogue of the piece: O / l
      if (!wait_all(bar(B_PV_DONE), (it - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (bad && stid == 0) raise_error(p.err_flags, kErrBadPage);
      const float inv = bad ? 0.f : 1.f / l;
      const float lse2 = bad ? -CUDART_INF_F : m_used + log2f(l);
      // O / l, two 32-column chunks per TMEM wait, 32-byte stores
#pragma unroll 1
      for (int cc = 0; cc < 8; cc += 2) {
        uint32_t o[2][32];
        tmem_ld32(tl + kTmemO + 32 * cc, o[0]);
        tmem_ld32(tl + kTmemO + 32 * (cc + 1), o[1]);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int col = rank * 256 + 32 * (cc + h);
          float f[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) f[k] = bad ? 0.f : __uint_as_float(o[h][k]) * inv;
          if (partial) {
            // a piece of a unit: fp32 into this cluster's partial slot
            float* pdst = p.ws_o + ((int64_t(cid) * 2 + slot) * kRows + row) * kMlaDv + col;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              st_global_v8(pdst + 8 * k, __float_as_uint(f[8 * k]), __float_as_uint(f[8 * k + 1]),
                           __float_as_uint(f[8 * k + 2]), __float_as_uint(f[8 * k + 3]),
                           __float_as_uint(f[8 * k + 4]), __float_as_uint(f[8 * k + 5]),
                           __float_as_uint(f[8 * k + 6]), __float_as_uint(f[8 * k + 7]));
            continue;
          }
          // a whole unit: bf16 to out
          __nv_bfloat16* dst = p.out + (int64_t(b) * kRows + row) * kMlaDv + col;
          const bool v8 = p.out_align32;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(f[16 * k + 2 * e], f[16 * k + 2 * e + 1]);
            if (v8) {
              st_global_v8(dst + 16 * k, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * k);
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
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

  // ---- teardown: all roles done; release TMEM
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One warp per (unit, head) row of a unit cut between clusters: log-sum-exp
// merge of its normalised partials, in cluster order. The loads of a batch of
// up to three partials (split bounds, lse, rows) are independent, so a warp
// waits on memory about twice per batch. Three covers the 2-3 pieces a unit
// usually has, at 78 registers: the merge's one warp per row runs in several
// waves, and four (94 registers, fewer warps resident) was 1.4 us slower per
// step. A programmatic dependent launch of the attention kernel: it waits here
// until that grid is done.
__global__ void __launch_bounds__(128) mla_merge_kernel(const __grid_constant__ MlaParams p,
                                                        int NC) {
  griddep_wait();
  griddep_launch_dependents();  // the next call's kernels may start their prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * 4 + warp;
  if (row >= int64_t(p.B) * p.q_len * kRows) return;
  const int b = int(row / kRows), h = int(row % kRows);
  const int u0 = p.ws_prefix[b], u1 = p.ws_prefix[b + 1];
  const int2 span = reinterpret_cast<const int2*>(p.ws_span)[b];
  if (u1 == u0) return;  // no tiles: the attention kernel wrote zeros
  const int c_lo = span.x >> 1, slot_lo = span.x & 1, c_hi = span.y;
  // (always in range unless the attention kernel gave up early, which it
  // reports through err_flags; the check keeps every read in bounds)
  if (span.x < 0 || c_lo == c_hi || c_hi >= NC || c_lo > c_hi) return;
  constexpr int kBatch = 3;
  float M = -CUDART_INF_F, den = 0.f, acc[16] = {};
  bool bad = false;
  for (int c0 = c_lo; c0 <= c_hi; c0 += kBatch) {
    float lse[kBatch];
    bool live[kBatch];
    float4 v[kBatch][4];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int c = min(c0 + i, c_hi);
      const int64_t wrow = (int64_t(c) * 2 + (c == c_lo ? slot_lo : 0)) * kRows + h;
      // clusters without tiles hold no partial of this unit
      live[i] = c0 + i <= c_hi && p.ws_split[c] != p.ws_split[c + 1];
      lse[i] = p.ws_lse[wrow];
      const float4* src = reinterpret_cast<const float4*>(p.ws_o + wrow * kMlaDv);
#pragma unroll
      for (int k = 0; k < 4; ++k) v[i][k] = src[lane + 32 * k];
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (!live[i]) continue;
      if (isnan(lse[i])) {  // a piece over a bad page: the row is zeroed
        bad = true;
        continue;
      }
      if (lse[i] > M) {  // online merge: rescale what is accumulated
        const float r = exp2f(M - lse[i]);
        den *= r;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] *= r;
        M = lse[i];
      }
      const float wgt = exp2f(lse[i] - M);
      den += wgt;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc[4 * k] += wgt * v[i][k].x;
        acc[4 * k + 1] += wgt * v[i][k].y;
        acc[4 * k + 2] += wgt * v[i][k].z;
        acc[4 * k + 3] += wgt * v[i][k].w;
      }
    }
  }
  const float inv = bad ? 0.f : 1.f / den;
  uint2* dst = reinterpret_cast<uint2*>(p.out + row * kMlaDv);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint2 o;
    o.x = pack_bf16x2(acc[4 * k] * inv, acc[4 * k + 1] * inv);
    o.y = pack_bf16x2(acc[4 * k + 2] * inv, acc[4 * k + 3] * inv);
    dst[lane + 32 * k] = o;
  }
  if (p.lse && lane == 0)
    p.lse[row] = bad ? -CUDART_INF_F : (M + log2f(den)) * 0.69314718055994531f;
}

constexpr int kMaxDevices = 64;

}  // namespace

size_t mla_smem_bytes() { return kSmemBytes; }

cudaError_t mla_decode_launch(const MlaParams& p, int clusters, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  static bool configured[kMaxDevices][2] = {};
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return e;
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  const bool append = p.kv_new != nullptr;
  auto kernel = append ? mla_decode_kernel<true> : mla_decode_kernel<false>;
  if (!configured[device][append]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes));
    if (e != cudaSuccess) return e;
    configured[device][append] = true;
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
    if ((e = cudaLaunchKernelEx(&cfg, kernel, p)) != cudaSuccess) return e;
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
