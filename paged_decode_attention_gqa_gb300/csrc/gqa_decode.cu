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
  static int run(bool small, int device) { return occupancy<HPC, R16, C, U>(device, small); }
};

template <int HPC, bool R16, bool C, bool U>
struct Launch {
  static cudaError_t run(const GqaParams* p, int grid, cudaStream_t stream) {
    return launch_attn<HPC, R16, C, U>(*p, grid, stream);
  }
};

// Two row groups per CTA: causal rows (correct for one query token too: the
// limit is then the whole cache), merge launch, heads per CTA 1/2/4 (half of
// a one-group CTA's).
template <int HPC, bool R16>
struct TwoGroups {
  static cudaError_t launch(const GqaParams& p, int grid, cudaStream_t stream) {
    return launch_attn<HPC, R16, true, false, kModePlain, 2>(p, grid, stream);
  }
  static int ctas_per_sm(bool small, int device) {
    return occupancy<HPC, R16, true, false, kModePlain, 2>(device, small);
  }
};

cudaError_t launch_two_groups(const GqaParams& p, bool r16, int grid, cudaStream_t stream) {
  switch (p.hpc * 2 + (r16 ? 1 : 0)) {
    case 2: return TwoGroups<1, false>::launch(p, grid, stream);
    case 3: return TwoGroups<1, true>::launch(p, grid, stream);
    case 4: return TwoGroups<2, false>::launch(p, grid, stream);
    case 5: return TwoGroups<2, true>::launch(p, grid, stream);
    case 8: return TwoGroups<4, false>::launch(p, grid, stream);
    case 9: return TwoGroups<4, true>::launch(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

int two_groups_ctas_per_sm(int hpc, bool r16, bool small, int device) {
  switch (hpc * 2 + (r16 ? 1 : 0)) {
    case 2: return TwoGroups<1, false>::ctas_per_sm(small, device);
    case 3: return TwoGroups<1, true>::ctas_per_sm(small, device);
    case 4: return TwoGroups<2, false>::ctas_per_sm(small, device);
    case 5: return TwoGroups<2, true>::ctas_per_sm(small, device);
    case 8: return TwoGroups<4, false>::ctas_per_sm(small, device);
    case 9: return TwoGroups<4, true>::ctas_per_sm(small, device);
    default: return 0;
  }
}

}  // namespace

int gqa_ctas_per_sm(int hpc, bool rows16, bool causal, bool fused, int tg, bool small,
                    int device) {
  // (two groups per CTA always run the causal instances: with one query token
  // every row's limit is the whole cache)
  if (tg == 2) return fused ? 0 : two_groups_ctas_per_sm(hpc, rows16, small, device);
  return dispatch<Occupancy>(hpc, rows16, causal, fused, small, device);
}

cudaError_t gqa_decode_launch(const GqaParams& p, int grid, bool fused, cudaStream_t stream,
                              cudaEvent_t attn_begin, cudaEvent_t attn_end) {
  cudaError_t e = cudaSuccess;
  if (attn_begin && (e = cudaEventRecord(attn_begin, stream)) != cudaSuccess) return e;
  const bool r16 = p.gh * p.q_len > 8;
  const bool known = p.hpc == 1 || p.hpc == 2 || p.hpc == 4 || p.hpc == 8;
  if (!known) return cudaErrorInvalidValue;
  if (p.tg == 2) {
    if (fused) return cudaErrorInvalidValue;
    e = launch_two_groups(p, r16, grid, stream);
  } else {
    e = dispatch<Launch>(p.hpc, r16, p.q_total > 1, fused, &p, grid, stream);
  }
  if (e != cudaSuccess) return e;
  if (attn_end && (e = cudaEventRecord(attn_end, stream)) != cudaSuccess) return e;
  if (fused || p.unit_cut) return cudaSuccess;  // nothing left to merge
  return launch_merge<kModePlain>(p, stream);
}

}  // namespace zl
