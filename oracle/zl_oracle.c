/*
 * Oracle for paged decode attention: plain, slow, fp64, on the CPU.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file. The CUDA library never includes, links or
 * calls it, and this file includes nothing from the CUDA library.
 *
 * What it computes.
 *   "ZhiLight：知乎开源的高性能 LLM 推理加速引擎", section "4. Tensor Core 上的
 *   Flash Attention": in the decode phase every running sequence adds one new
 *   token and the engine runs one fused, batched attention over all of them.
 *   "ZhiLight: Zhihu's CUDA Inference Engine ...", section "Dual streams, host
 *   all-reduce and the memory model": fused batch attention for decoding,
 *   prefix cache, DeepseekV2 MLA.
 *   The DataFun talk write-up, section "1. 大模型负载分析": attention comes in
 *   head-sharing variants such as multi-query attention (the GQA family).
 *
 *   For sequence b, query row i (< q_len), query head h, with
 *   g = Hq / Hkv and kv head kh = h / g, over the visible tokens t < n_vis:
 *
 *     s_t     = scale * sum_d q[b,i,h,d] * K_b[t,kh,d]
 *     m       = max_t s_t
 *     w_t     = exp(s_t - m) / sum_u exp(s_u - m)
 *     out[d]  = sum_t w_t * V_b[t,kh,d]
 *     lse     = m + ln(sum_t exp(s_t - m))          (natural log)
 *
 *   K_b[t] is row (t mod P) of physical page block_table[b, t / P] of the K
 *   pool, and likewise for V. n_vis = L_b - q_len + 1 + i (the new tokens are
 *   already in the cache and each query sees itself and everything before
 *   it); for q_len = 1 that is all L_b tokens.
 *
 *   MLA (multi-head latent attention, absorbed form): Hkv = 1, the "K" row is
 *   the latent row of width D_qk, and V is its first D_v columns; pass
 *   v_pool = NULL for that.
 *
 * Precision: every bf16 input is decoded exactly (its 16 bits become the high
 * half of an IEEE binary32) and all arithmetic is IEEE binary64, in the plain
 * order written above. No blocking, fusion or reordering.
 *
 * Degenerate cases (stated here, shared with the CUDA library's contract):
 *   n_vis <= 0 (empty context)               -> out = 0, lse = -inf, status 0
 *   seq_len < 0 or > max_pages * P            -> out = 0, lse = -inf, bit 2
 *   a referenced page id outside [0,num_pages) -> out = 0, lse = -inf, bit 1
 * The return value is the OR of those bits over the batch.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ZL_ORACLE_BAD_PAGE 1
#define ZL_ORACLE_BAD_LEN 2

/* bf16 bits -> exact binary32 value -> binary64. */
static double bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Address of row (page, slot, head) in a pool, in elements. */
static int64_t pool_row(int64_t page, int64_t slot, int64_t head, int64_t page_stride,
                        int64_t token_stride, int64_t head_stride) {
  return page * page_stride + slot * token_stride + head * head_stride;
}

/*
 * Attention of one query row over the visible tokens [t_begin, t_end) of one
 * sequence. Writes out[0..D_v) (normalised) and returns lse through *lse_out.
 * weights, if not NULL, receives the normalised softmax weights w_t for
 * t in [t_begin, t_end) (t_end - t_begin entries).
 * Returns 0, or ZL_ORACLE_BAD_PAGE with out = 0 and lse = -inf.
 */
static int attend_row(const uint16_t* q_row, const uint16_t* k_pool, const uint16_t* v_pool,
                      int64_t page_stride, int64_t token_stride, int64_t head_stride,
                      const int32_t* bt_row, int kh, int D_qk, int D_v, int page_size,
                      int num_pages, double scale, int64_t t_begin, int64_t t_end,
                      double* s, double* out, double* lse_out, double* weights) {
  int64_t n = t_end - t_begin;
  for (int d = 0; d < D_v; ++d) out[d] = 0.0;
  *lse_out = -INFINITY;
  if (n <= 0) return 0;

  /* Every page the range touches must be a real page of the pool. */
  for (int64_t t = t_begin; t < t_end; ++t) {
    int32_t page = bt_row[t / page_size];
    if (page < 0 || page >= num_pages) return ZL_ORACLE_BAD_PAGE;
  }

  /* s_t = scale * q . K_t */
  for (int64_t t = t_begin; t < t_end; ++t) {
    int32_t page = bt_row[t / page_size];
    const uint16_t* k_row =
        k_pool + pool_row(page, t % page_size, kh, page_stride, token_stride, head_stride);
    double dot = 0.0;
    for (int d = 0; d < D_qk; ++d) dot += bf16_to_f64(q_row[d]) * bf16_to_f64(k_row[d]);
    s[t - t_begin] = scale * dot;
  }

  /* m = max_t s_t ; denominator = sum_t exp(s_t - m) */
  double m = s[0];
  for (int64_t j = 1; j < n; ++j)
    if (s[j] > m) m = s[j];
  double denom = 0.0;
  for (int64_t j = 0; j < n; ++j) denom += exp(s[j] - m);

  /* out = sum_t w_t V_t */
  for (int64_t t = t_begin; t < t_end; ++t) {
    double w = exp(s[t - t_begin] - m) / denom;
    if (weights) weights[t - t_begin] = w;
    int32_t page = bt_row[t / page_size];
    const uint16_t* v_row =
        (v_pool ? v_pool : k_pool) +
        pool_row(page, t % page_size, kh, page_stride, token_stride, head_stride);
    for (int d = 0; d < D_v; ++d) out[d] += w * bf16_to_f64(v_row[d]);
  }
  *lse_out = m + log(denom);
  return 0;
}

/*
 * Batched paged decode attention.
 *   q            bf16 bits [B, q_len, Hq, D_qk], contiguous
 *   k_pool       bf16 bits, row (page, slot, head) at
 *                page*page_stride + slot*token_stride + head*head_stride
 *   v_pool       same strides as k_pool; NULL means V = first D_v columns of K
 *   block_table  int32 [B, bt_stride]; row b lists the physical pages of b
 *   seq_lens     int32 [B]; tokens in the cache, the new ones included
 *   out          fp64 [B, q_len, Hq, D_v]
 *   lse          fp64 [B, q_len, Hq] or NULL
 *   num_threads  OpenMP threads (<= 0: the runtime default)
 */
int zl_oracle_decode_attn(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                          int64_t page_stride, int64_t token_stride, int64_t head_stride,
                          const int32_t* block_table, int64_t bt_stride,
                          const int32_t* seq_lens, int B, int q_len, int Hq, int Hkv, int D_qk,
                          int D_v, int page_size, int num_pages, double scale, double* out,
                          double* lse, int num_threads) {
  int status = 0;
  int g = Hq / Hkv;
  int64_t capacity = bt_stride * (int64_t)page_size;
  int64_t rows = (int64_t)B * q_len * Hq;
  int64_t max_len = 0;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  if (max_len > capacity) max_len = capacity;

#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads) reduction(| : status)
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < rows; ++r) {
      int h = (int)(r % Hq);
      int i = (int)((r / Hq) % q_len);
      int b = (int)(r / ((int64_t)Hq * q_len));
      double* o = out + r * D_v;
      double row_lse = -INFINITY;
      int64_t L = seq_lens[b];
      if (L < 0 || L > capacity) {
        for (int d = 0; d < D_v; ++d) o[d] = 0.0;
        status |= ZL_ORACLE_BAD_LEN;
      } else {
        int64_t n_vis = L - q_len + 1 + i;
        if (n_vis > L) n_vis = L;
        status |= attend_row(q + r * D_qk, k_pool, v_pool, page_stride, token_stride,
                             head_stride, block_table + (int64_t)b * bt_stride, h / g, D_qk, D_v,
                             page_size, num_pages, scale, 0, n_vis, s, o, &row_lse, NULL);
      }
      if (lse) lse[r] = row_lse;
    }
    free(s);
  }
  return status;
}

/*
 * One query row over an arbitrary token range [t_begin, t_end) of sequence b:
 * the per-split partial result (normalised output and its lse). The caller
 * owns the range; nothing here decides it. weights may be NULL.
 */
int zl_oracle_attend_range(const uint16_t* q_row, const uint16_t* k_pool, const uint16_t* v_pool,
                           int64_t page_stride, int64_t token_stride, int64_t head_stride,
                           const int32_t* bt_row, int kh, int D_qk, int D_v, int page_size,
                           int num_pages, double scale, int64_t t_begin, int64_t t_end,
                           double* out, double* lse, double* weights) {
  int64_t n = t_end - t_begin;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  int st = attend_row(q_row, k_pool, v_pool, page_stride, token_stride, head_stride, bt_row, kh,
                      D_qk, D_v, page_size, num_pages, scale, t_begin, t_end, s, out, lse,
                      weights);
  free(s);
  return st;
}

/*
 * Log-sum-exp merge of S partial results of one query row (split-KV):
 *   M   = max_s lse_s
 *   c_s = exp(lse_s - M)
 *   out = sum_s c_s o_s / sum_s c_s
 *   lse = M + ln(sum_s c_s)
 * A partial with lse = -inf (an empty range) has weight 0. If every partial
 * is empty the result is out = 0, lse = -inf.
 *   parts  fp64 [S, D]   normalised partial outputs
 *   lses   fp64 [S]
 */
void zl_oracle_lse_merge(const double* parts, const double* lses, int S, int D, double* out,
                         double* lse_out) {
  double M = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (lses[s] > M) M = lses[s];
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (M == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double sum_c = 0.0;
  for (int s = 0; s < S; ++s) sum_c += exp(lses[s] - M);
  for (int s = 0; s < S; ++s) {
    double c = exp(lses[s] - M) / sum_c;
    for (int d = 0; d < D; ++d) out[d] += c * parts[(int64_t)s * D + d];
  }
  *lse_out = M + log(sum_c);
}

/*
 * Paged KV append: store the q_len new tokens of every sequence in their page
 * slots, the step that precedes decode attention. The new K and V rows are
 * what the fused QKV projection produces ("ZhiLight: Zhihu's CUDA Inference
 * Engine ...", section "Dual streams, host all-reduce and the memory model":
 * fused kernels for qkv; "ZhiLight：知乎开源的高性能 LLM 推理加速引擎", section
 * "3. 自研 Fusion Kernel": QKV fusion). The pages do not spell the append out;
 * the plain reading used here: seq_lens[b] counts the tokens after the
 * append, so new token i (< q_len) is logical position t = L_b - q_len + i and
 * goes to slot t mod P of physical page block_table[b, t / P], kv head kh.
 *
 *   k_new   bf16 bits [B, q_len, Hkv, D_k], contiguous
 *   v_new   bf16 bits [B, q_len, Hkv, D_v], or NULL (MLA: the latent row only)
 *   k_pool, v_pool   pools addressed as in zl_oracle_decode_attn (updated in place)
 * Errors, per sequence: L_b < q_len or L_b > max_pages * P -> nothing of b is
 * written, bit 2; per token: a page id outside [0, num_pages) -> that token is
 * not written, bit 1. Returns the OR of the bits.
 */
int zl_oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pool,
                        uint16_t* v_pool, int64_t page_stride, int64_t token_stride,
                        int64_t head_stride, const int32_t* block_table, int64_t bt_stride,
                        const int32_t* seq_lens, int B, int q_len, int Hkv, int D_k, int D_v,
                        int page_size, int num_pages) {
  int status = 0;
  int64_t capacity = bt_stride * (int64_t)page_size;
  for (int b = 0; b < B; ++b) {
    int64_t L = seq_lens[b];
    if (L < q_len || L > capacity) {
      status |= ZL_ORACLE_BAD_LEN;
      continue;
    }
    for (int i = 0; i < q_len; ++i) {
      int64_t t = L - q_len + i;
      int64_t page = block_table[(int64_t)b * bt_stride + t / page_size];
      if (page < 0 || page >= num_pages) {
        status |= ZL_ORACLE_BAD_PAGE;
        continue;
      }
      for (int kh = 0; kh < Hkv; ++kh) {
        int64_t dst = pool_row(page, t % page_size, kh, page_stride, token_stride, head_stride);
        int64_t src_row = ((int64_t)b * q_len + i) * Hkv + kh;
        for (int d = 0; d < D_k; ++d) k_pool[dst + d] = k_new[src_row * D_k + d];
        if (v_new)
          for (int d = 0; d < D_v; ++d) v_pool[dst + d] = v_new[src_row * D_v + d];
      }
    }
  }
  return status;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int zl_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
