// GQA decode: kernel instances for the plain path (every sequence attends to
// its own pages) and their launch. The kernels live in gqa_kernel.cuh.
#include "gqa_kernel.cuh"

namespace zl {

int gqa_heads_per_cta(int Hkv) {
  if (Hkv % 8 == 0) return 8;
  if (Hkv % 4 == 0) return 4;
  if (Hkv % 2 == 0) return 2;
  return 1;
}

namespace {

// The kernel instance for (heads per CTA, 16 rows, causal rows, fused merge).
template <template <int, bool, bool, bool> class F, typename... A>
auto dispatch(int hpc, bool r16, bool causal, bool fused, A... a)
    -> decltype(F<1, false, false, false>::run(a...)) {
  using R = decltype(F<1, false, false, false>::run(a...));
  const int k = ((hpc * 2 + (r16 ? 1 : 0)) * 2 + (causal ? 1 : 0)) * 2 + (fused ? 1 : 0);
  switch (k) {
#define ZL_CASE(H, S, C, U) \
  case ((H * 2 + S) * 2 + C) * 2 + U: return F<H, bool(S), bool(C), bool(U)>::run(a...);
#define ZL_CASES(H)                                                              \
  ZL_CASE(H, 0, 0, 0) ZL_CASE(H, 0, 0, 1) ZL_CASE(H, 0, 1, 0) ZL_CASE(H, 0, 1, 1) \
  ZL_CASE(H, 1, 0, 0) ZL_CASE(H, 1, 0, 1) ZL_CASE(H, 1, 1, 0) ZL_CASE(H, 1, 1, 1)
    ZL_CASES(1) ZL_CASES(2) ZL_CASES(4) ZL_CASES(8)
#undef ZL_CASES
#undef ZL_CASE
    default: return R();
  }
}

template <int HPC, bool R16, bool C, bool U>
struct Occupancy {
  static int run(int device) { return occupancy<HPC, R16, C, U>(device); }
};

template <int HPC, bool R16, bool C, bool U>
struct Launch {
  static cudaError_t run(const GqaParams* p, int grid, cudaStream_t stream) {
    return launch_attn<HPC, R16, C, U>(*p, grid, stream);
  }
};

}  // namespace

int gqa_ctas_per_sm(int hpc, bool rows16, bool causal, bool fused, int device) {
  return dispatch<Occupancy>(hpc, rows16, causal, fused, device);
}

cudaError_t gqa_decode_launch(const GqaParams& p, int grid, bool fused, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  cudaError_t e = cudaSuccess;
  if (attn_begin && (e = cudaEventRecord(attn_begin, stream)) != cudaSuccess) return e;
  const bool r16 = p.g * p.q_len > 8;
  const bool known = p.hpc == 1 || p.hpc == 2 || p.hpc == 4 || p.hpc == 8;
  if (!known) return cudaErrorInvalidValue;
  e = dispatch<Launch>(p.hpc, r16, p.q_total > 1, fused, &p, grid, stream);
  if (e != cudaSuccess) return e;
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  if (fused || p.unit_cut) return cudaSuccess;  // nothing left to merge
  // The merge as a programmatic dependent launch: its CTAs may become resident
  // before the attention grid ends and wait in griddepcontrol.wait.
  const int64_t items =
      int64_t(p.ngroups) * p.B * p.Hkv * ((p.g * p.q_len + kMergeRows - 1) / kMergeRows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((items + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gqa_merge_kernel<kModePlain>, p, p.group_ctas);
}

}  // namespace zl
