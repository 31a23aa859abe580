/*
 * zl_decode_attn — paged decode attention for GB300 (sm_103a), C ABI.
 *
 * The operation. Each running sequence adds one new query token and attends
 * to its whole paged K/V cache in one fused, batched launch: the decode-phase
 * "fused batch attention" on tensor cores that "ZhiLight：知乎开源的高性能 LLM
 * 推理加速引擎" describes in section "4. Tensor Core 上的 Flash Attention", and
 * that "ZhiLight: Zhihu's CUDA Inference Engine for Llama and DeepSeek on PCIe
 * GPUs" lists in "Dual streams, host all-reduce and the memory model" (fused
 * batch attention for decoding using tensor core instructions; prefix cache;
 * DeepseekV2 MLA). For sequence b, query head h, kv head kh = h / (Hq/Hkv):
 *
 *   out[b,h,:] = sum_{t < seq_lens[b]} softmax_t(scale * q[b,h,:] . K_b[t,kh,:]) V_b[t,kh,:]
 *   lse[b,h]   = ln sum_t exp(scale * q[b,h,:] . K_b[t,kh,:])
 *
 * where row t of K_b is slot (t mod page_size) of physical page
 * block_table[b, t / page_size] (likewise V). With q_len > 1 new tokens per
 * sequence (speculative or multi-token-prediction decode: all of them are
 * already in the cache, the last q_len of its seq_lens[b] tokens), query
 * token i < q_len attends causally to t < seq_lens[b] - q_len + 1 + i, and
 * q, out, lse gain a q_len axis after B. Grouped-query heads sharing a
 * kv head are evaluated together so each K/V byte is read once per group (the
 * DataFun talk write-up, section "1. 大模型负载分析", names the head-sharing
 * attention variants). Long or ragged contexts are split across CTAs and the
 * partial results merged by log-sum-exp (the split-KV "flash_decoding" idea
 * named under "技术架构：五层模块化设计").
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer. The library never allocates or
 *     frees device memory and never synchronises; it enqueues kernels on the
 *     given stream only. Its state is host-side (per-device attributes), with
 *     one exception: the static scratch array of zl_decode_attn_noalloc
 *     (ZL_NOALLOC_WORKSPACE_BYTES, held by every GPU that loads the library
 *     until the process exits).
 *   - Host errors return synchronously and launch nothing.
 *   - Device data errors (a page id outside [0, num_pages), a seq_len outside
 *     [0, block_table_stride * page_size], a pipeline wait that timed out)
 *     cannot be returned without a sync: the kernel ORs a ZL_DEVERR_* bit into
 *     *err_flags (when err_flags is not NULL) and writes zeros (lse = -inf)
 *     for the affected query rows: every row of a sequence with a bad length,
 *     and every row whose visible tokens reach a bad page. Nothing traps.
 *   - seq_lens[b] = 0 gives out = 0 and lse = -inf; that is not an error.
 *   - Results depend only on logical content: remapping pages gives
 *     bit-identical output, and repeated calls are bit-identical.
 */
#ifndef ZL_DECODE_ATTN_H
#define ZL_DECODE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / cudaEvent_t. NULL stream = the legacy default. */
typedef struct CUstream_st* zl_stream_t;
typedef struct CUevent_st* zl_event_t;

typedef enum {
  ZL_OK = 0,
  ZL_ERR_INVALID_ARG = 1, /* NULL or misaligned pointer, bad size or stride */
  ZL_ERR_UNSUPPORTED = 2, /* a valid shape this build does not implement */
  ZL_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than required */
  ZL_ERR_CUDA = 4         /* a CUDA runtime call or launch failed */
} zl_status;

/* Bits the kernels OR into *err_flags. */
#define ZL_DEVERR_BAD_PAGE 1u    /* block_table entry outside [0, num_pages) */
#define ZL_DEVERR_BAD_SEQ_LEN 2u /* seq_len < 0 or > block_table_stride * page_size */
#define ZL_DEVERR_TIMEOUT 4u     /* a pipeline wait gave up after ~2 s */
#define ZL_DEVERR_BAD_PREFIX 8u  /* shared_prefix_pages does not hold for some sequence */

typedef struct {
  size_t struct_size; /* sizeof(zl_decode_attn_params), for ABI checks */

  /* Query, bf16 [B, q_len, Hq, D_qk], contiguous, 16-byte aligned. */
  const void* q;
  /* K and V pools, bf16. Row (page, slot, head) of D_qk elements starts at
     page*page_stride + slot*token_stride + head*head_stride (elements); the
     row itself is contiguous. Strides are multiples of 8 elements, the base
     16-byte aligned. [num_pages, page_size, Hkv, D] ("NHD") and
     [num_pages, Hkv, page_size, D] ("HND") are both expressible.
     MLA: v_pool must be NULL; V is the first D_v columns of the K row. */
  const void* k_pool;
  const void* v_pool;
  int64_t page_stride, token_stride, head_stride;

  /* int32 [B, block_table_stride]: physical page of each logical page. */
  const int32_t* block_table;
  int64_t block_table_stride;
  /* int32 [B], device: tokens in the cache, the new token included. */
  const int32_t* seq_lens;

  /* Output, bf16 [B, q_len, Hq, D_v], contiguous, 16-byte aligned. */
  void* out;
  /* Optional fp32 [B, q_len, Hq], natural-log log-sum-exp of the scaled
     scores; NULL to skip. */
  float* lse;

  int32_t B, q_len, Hq, Hkv, D_qk, D_v, page_size, num_pages;
  /* Host-side upper bound of seq_lens (0 = unknown); used only to size the
     grid for small problems. Results do not depend on it. */
  int32_t max_seq_len;
  float scale; /* softmax scale, e.g. 1/sqrt(D) */

  /* Caller-owned device scratch of at least zl_decode_attn_workspace_size()
     bytes, 256-byte aligned.
     zl_decode_attn with ZL_DECODE_SINGLE_LAUNCH: its first 8 * B * Hkv bytes
     are one arrival counter per (sequence, kv head), which must be zero
     before the call (zero-fill them, e.g. with cudaMemsetAsync). The
     in-kernel merge counts them up and returns each one it used to zero, so
     a call leaves them ready for the next call of the same or smaller
     B * Hkv; counters left by a call that stopped on a device error are
     recognised (each call tags its counts) and ignored. Anything else
     written into that range (a call without the flag, a call with a larger
     B * Hkv, other data) needs a new zero fill of it first: the tag makes
     such leftovers harmless unless their upper 32 bits happen to equal the
     call's tag, and only a zero fill rules that out.
     Otherwise: contents need no initialisation. */
  void* workspace;
  size_t workspace_bytes;

  /* Optional device word; kernels atomically OR ZL_DEVERR_* bits into it. */
  uint32_t* err_flags;

  /* Number of CTAs of the attention kernel; 0 = one wave on this device.
     Any value >= 1 gives the same result within fp32 rounding: the work is
     split into that many equal token ranges (at most one per 16-token tile;
     CTAs beyond that take none) and merged. With 0 (and no shared prefix),
     zl_decode_attn also decides on the device, from seq_lens, whether every
     (sequence, head group) is short enough for a CTA of its own, the rule
     that max_seq_len lets the host apply before the launch (see
     zl_decode_attn); decided on the device, the merge kernel is still
     launched but has nothing to do. */
  int32_t num_ctas;

  /* Optional profiling events recorded on the stream immediately before and
     after the attention kernel (not the split-KV merge when that is a second
     launch); NULL to skip. */
  zl_event_t attn_begin, attn_end;

  /* ZL_DECODE_* bits; 0 for the defaults. */
  uint32_t flags;

  /* zl_decode_attn only; 0 = none. The first shared_prefix_pages entries of
     every block-table row are the same physical pages (a cached prefix all B
     sequences share), and every query row sees all of them
     (seq_lens[b] - q_len + 1 >= shared_prefix_pages * page_size). Those pages
     are then read once per group of 16 / (g * q_len) sequences instead of
     once per sequence. The kernels check both conditions and set
     ZL_DEVERR_BAD_PREFIX if either fails (results are then undefined). Not
     with ZL_DECODE_SINGLE_LAUNCH. */
  int32_t shared_prefix_pages;

  /* Optional fused KV append; NULL = the cache already holds the new tokens.
     The q_len new tokens' rows, bf16, contiguous, 16-byte aligned:
     zl_decode_attn: k_new [B, q_len, Hkv, D_qk] and v_new [B, q_len, Hkv,
     D_v], both required; zl_decode_attn_mla: k_new [B, q_len, D_qk] (the
     latent rows) and v_new NULL. The attention launch itself stores them in
     their page slots first, exactly as zl_kv_append would (new token i of
     sequence b is position seq_lens[b] - q_len + i; the pools must be
     writable), and attends over the result: a decode step needs no separate
     append launch. After the call the pools hold the new rows, bit-exact,
     except rows on a bad page (skipped and flagged, as zl_kv_append does) and
     the rows of a sequence with fewer than q_len tokens or a bad length
     (skipped; only a bad length is flagged, by the attention). With
     shared_prefix_pages the new tokens must lie past the shared pages. */
  const void* k_new;
  const void* v_new;
} zl_decode_attn_params;

/* zl_decode_attn: merge the split-KV partials inside the attention kernel
   (the last CTA to finish a piece of a (sequence, kv head) merges it, in a
   fixed order), so the call is one launch. Without it the merge is a second,
   programmatically dependent launch. Both give bit-identical results.
   zl_decode_attn_mla accepts no flags. */
#define ZL_DECODE_SINGLE_LAUNCH 1u

/* Test hook for failure detection, not for production calls: the attention
   kernel first waits on a word that nothing ever sets, so its bounded wait
   (about 50 ms) runs out; every CTA then stops, the call reports
   ZL_DEVERR_TIMEOUT in *err_flags, and out / lse are left undefined. The
   context stays usable and the next call without the hook computes normally.
   This is how a stalled pipeline is reported, made to happen on purpose
   without a fault. zl_decode_attn only. */
#define ZL_DECODE_TEST_STALL 0x80000000u

/*
 * GQA / MHA / MQA decode over separate K and V pools.
 *   Supported: D_qk = D_v = 128; Hq % Hkv == 0; g = Hq/Hkv <= 128;
 *   1 <= q_len <= 128; page_size a multiple of 16 (<= 1024); 1 <= B <= 4096.
 *   The (query token, head) rows one kv head serves go in row groups of at
 *   most 16, one 16-row tensor-core tile: when g * q_len > 16 the tokens go in
 *   groups of 16 / g, and when g > 16 each token's g heads go in ceil(g / 16)
 *   chunks (MQA with many query heads). The groups run side by side in one
 *   attention launch (two groups share every CTA and each K/V tile; with
 *   more, each group reads the K/V, mostly from L2 for all but the first);
 *   with ZL_DECODE_SINGLE_LAUNCH, one launch per group, and attn_begin is
 *   recorded before the first and attn_end after the last.
 *   With shared_prefix_pages > 0, g * q_len <= 16. When max_seq_len shows that
 *   every (sequence, head group) is short (at most 8 tiles of 16 tokens), each
 *   gets a CTA of its own and no merge is launched. A query row that
 *   sees no token (seq_lens[b] < q_len) gives out = 0 and lse = -inf. A bad
 *   page id zeroes (out = 0, lse = -inf) every query row whose visible tokens
 *   reach that page, and only those: with q_len > 1, a bad page that holds
 *   only the newest tokens zeroes only the rows of the queries that see them.
 *   Anything else returns ZL_ERR_UNSUPPORTED (or ZL_ERR_INVALID_ARG when the
 *   value is not meaningful at all, e.g. Hkv = 0).
 */
zl_status zl_decode_attn(const zl_decode_attn_params* params, zl_stream_t stream);

/*
 * Absorbed multi-head latent attention (MLA) decode: one shared latent row per
 * token of width D_qk = 576 (512 latent + 64 rope); V is its first D_v = 512
 * columns. The "ZhiLight：知乎开源的高性能 LLM 推理加速引擎" page lists MLA support
 * under "功能生态" and flash_mla under "技术架构：五层模块化设计".
 *   Supported: Hkv = 1, v_pool = NULL, Hq = 128, D_qk = 576, D_v = 512,
 *   page_size a multiple of 64 (<= 1024), q_len >= 1 with B * q_len <= 1024
 *   (query token i attends causally, as for zl_decode_attn; each (sequence,
 *   query token) pair is a unit of work of its own).
 *   head_stride is not used. The kernel runs on clusters of two CTAs;
 *   num_ctas (when > 0) is rounded up to an even count.
 */
zl_status zl_decode_attn_mla(const zl_decode_attn_params* params, zl_stream_t stream);

/* Workspace bytes zl_decode_attn (resp. zl_decode_attn_mla) needs for these
   params. Only the shape fields and num_ctas are read; pointers may be NULL.
   Needs a current CUDA device (the default grid depends on its SM count). */
zl_status zl_decode_attn_workspace_size(const zl_decode_attn_params* params, size_t* bytes);
zl_status zl_decode_attn_mla_workspace_size(const zl_decode_attn_params* params, size_t* bytes);

/* Kernel launches one zl_decode_attn call with these params enqueues: the
   attention kernel and, unless no unit is cut (short contexts given a CTA per
   unit, known from max_seq_len) or ZL_DECODE_SINGLE_LAUNCH merges inside it,
   the merge kernel; with ZL_DECODE_SINGLE_LAUNCH, that once per row group
   (group of query tokens, or of heads when g > 16; see zl_decode_attn). A
   shared-prefix call has one row group. The same inputs and
   rules as zl_decode_attn_workspace_size. (zl_decode_attn_mla always
   enqueues two.) */
zl_status zl_decode_attn_launches(const zl_decode_attn_params* params, int32_t* launches);

/*
 * zl_decode_attn without a caller-provided workspace, for callers that cannot
 * allocate device memory (a host that already reserved all of it for its own
 * pool, a plugin interface with no scratch allocator, a loop that cannot
 * afford cudaMalloc's implicit synchronisation). The pages describe no such
 * entry point; it has no counterpart there.
 *   - Same arguments, checks and results as zl_decode_attn; workspace and
 *     workspace_bytes are ignored.
 *   - The scratch is one array of ZL_NOALLOC_WORKSPACE_BYTES in the library's
 *     own device memory; every GPU that loads the library holds it until the
 *     process exits. With num_ctas = 0, a call whose default grid needs more
 *     workspace than that runs on the largest grid whose workspace fits (the
 *     result is the same within fp32 rounding; only the split differs). With
 *     num_ctas > 0, or when even one CTA does not fit, it returns
 *     ZL_ERR_WORKSPACE.
 *   - The first call on each device looks up the array's device address (with
 *     that device current), and so does the first call in a new context on it
 *     (after cudaDeviceReset); make those calls before any stream capture.
 *   - Calls allocate nothing: no cudaMalloc, cudaFree or allocating library
 *     routine. All calls share the one array, which keeps the last call's
 *     contents. A call with ZL_DECODE_SINGLE_LAUNCH first zero-fills its
 *     arrival counters (the first 8 * B * Hkv bytes of the array) with
 *     cudaMemsetAsync on the stream, so whatever an earlier call left there
 *     never matters; other calls need nothing cleared. Calls that overlap on
 *     the GPU (other streams, other threads) race on the array: serialise
 *     them.
 */
#define ZL_NOALLOC_WORKSPACE_BYTES (8u << 20)
zl_status zl_decode_attn_noalloc(const zl_decode_attn_params* params, zl_stream_t stream);

/*
 * Paged KV append: store the q_len new tokens of every sequence (the K and V
 * rows the fused QKV projection produced; "ZhiLight: Zhihu's CUDA Inference
 * Engine ...", section "Dual streams, host all-reduce and the memory model",
 * lists fused kernels for qkv beside the decode attention) in their page
 * slots, before zl_decode_attn / zl_decode_attn_mla reads them. seq_lens[b]
 * counts the tokens after the append, so new token i (< q_len) of sequence b
 * is logical position t = seq_lens[b] - q_len + i: slot t % page_size of
 * physical page block_table[b, t / page_size]. The pages assign no pages; the
 * caller's block table must already map position t.
 *   - Pools, strides, block table and seq_lens mean exactly what they mean in
 *     zl_decode_attn_params (the same buffers can be passed to both calls).
 *     v_pool = NULL and v_new = NULL for a latent-only (MLA) pool.
 *   - k_new: bf16 [B, q_len, Hkv, D_k], v_new: bf16 [B, q_len, Hkv, D_v],
 *     contiguous, 16-byte aligned; D_k, D_v multiples of 8, <= 1024 (D_v <= D_k
 *     is not required: each pool row is as wide as its own new row).
 *   - Device data errors: seq_lens[b] < q_len or > block_table_stride *
 *     page_size writes nothing of sequence b (ZL_DEVERR_BAD_SEQ_LEN); a page
 *     id outside [0, num_pages) skips that token (ZL_DEVERR_BAD_PAGE).
 *   - Every written element is a copy: the result is bit-exact.
 *   - The writes are ordinary stores on the given stream; a decode call
 *     enqueued after it on the same stream sees them.
 *   - zl_decode_attn_params.k_new / v_new do the same stores inside the
 *     attention launch (one launch less per decode step).
 */
typedef struct {
  size_t struct_size; /* sizeof(zl_kv_append_params) */
  const void* k_new;
  const void* v_new;
  void* k_pool;
  void* v_pool;
  int64_t page_stride, token_stride, head_stride;
  const int32_t* block_table;
  int64_t block_table_stride;
  const int32_t* seq_lens;
  int32_t B, q_len, Hkv, D_k, D_v, page_size, num_pages;
  uint32_t* err_flags; /* optional, as in zl_decode_attn_params */
} zl_kv_append_params;

zl_status zl_kv_append(const zl_kv_append_params* params, zl_stream_t stream);

/* Static description of a status code. */
const char* zl_status_string(zl_status status);

#ifdef __cplusplus
}
#endif

#endif /* ZL_DECODE_ATTN_H */
