// GQA decode over a shared prefix: kernel instances and their launches.
//
// When every sequence starts with the same pages (a prefix cached once and
// shared: the prefix cache of "ZhiLight：知乎开源的高性能 LLM 推理加速引擎",
// sections "技术架构：五层模块化设计" and "功能生态"), the plain launch would stream
// those pages once per sequence. Here they are streamed once per group of sgs
// sequences instead: the rows of one m16 tensor-core tile are the query rows
// of sgs sequences (sgs = 16 / (g * q_len)), so each K/V tile of the prefix
// serves all of them. One attention launch covers the prefix units (group,
// head group) and the suffix units (sequence, head group: its tiles past the
// prefix) on one tile line cut into equal CTA ranges; the merge launch then
// combines, for every query row, its prefix part and its suffix part. The
// merge is a programmatic dependent of the attention kernel.
#include "gqa_kernel.cuh"

namespace zl {
namespace {

template <template <int, bool, bool, bool, int> class F, int MODE, typename... A>
auto dispatch_mode(int hpc, bool r16, bool causal, A... a)
    -> decltype(F<1, false, false, false, MODE>::run(a...)) {
  using Ret = decltype(F<1, false, false, false, MODE>::run(a...));
  const int k = (hpc * 2 + (r16 ? 1 : 0)) * 2 + (causal ? 1 : 0);
  switch (k) {
#define ZL_CASE(H, S, C) \
  case (H * 2 + S) * 2 + C: return F<H, bool(S), bool(C), false, MODE>::run(a...);
#define ZL_CASES(H) ZL_CASE(H, 0, 0) ZL_CASE(H, 0, 1) ZL_CASE(H, 1, 0) ZL_CASE(H, 1, 1)
    ZL_CASES(1) ZL_CASES(2) ZL_CASES(4) ZL_CASES(8)
#undef ZL_CASES
#undef ZL_CASE
    default: return Ret();
  }
}

template <int HPC, bool R16, bool C, bool U, int MODE>
struct Occupancy {
  static int run(bool small, int device) {
    return occupancy<HPC, R16, C, U, MODE>(device, small);
  }
};

template <int HPC, bool R16, bool C, bool U, int MODE>
struct Launch {
  static cudaError_t run(const GqaParams* p, int grid, cudaStream_t stream) {
    return launch_attn<HPC, R16, C, U, MODE>(*p, grid, stream);
  }
};

}  // namespace

int gqa_shared_ctas_per_sm(int hpc, bool rows16, bool causal, bool small, int device) {
  return dispatch_mode<Occupancy, kModeShared>(hpc, rows16, causal, small, device);
}

cudaError_t gqa_shared_launch(const GqaParams& p, int grid, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  const bool known = p.hpc == 1 || p.hpc == 2 || p.hpc == 4 || p.hpc == 8;
  if (!known) return cudaErrorInvalidValue;
  cudaError_t e = cudaSuccess;
  if (attn_begin && (e = cudaEventRecord(attn_begin, stream)) != cudaSuccess) return e;
  const bool r16 = p.sgs * p.gh * p.q_len > 8;
  if ((e = dispatch_mode<Launch, kModeShared>(p.hpc, r16, p.q_total > 1, &p, grid, stream)) !=
      cudaSuccess)
    return e;
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  return launch_merge<kModeShared>(p, stream);
}

}  // namespace zl
