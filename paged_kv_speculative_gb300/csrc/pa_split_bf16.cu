// bf16-KV instantiations of the split kernel (head_dim 64 and 128).
#include "pa_split.cuh"

namespace pav {

template <int D, int NW>
static cudaError_t run_bf16(int units, const CUtensorMap* tmk, const CUtensorMap* tmv, const SplitParams* p,
                            cudaStream_t stream) {
  auto kern = pa_split_kernel<0, D, NW>;
  constexpr int smem = split_smem_bytes(0, D);
  static std::atomic<uint64_t> attr_done{0};  // devices whose limit is raised
  const cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<units, NW * 32, smem, stream>>>(*tmk, *tmv, *p);
  return cudaGetLastError();
}

cudaError_t launch_split_bf16(int head_dim, int warps, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                              const SplitParams* p, cudaStream_t stream) {
#define PAV_CASE(DD, NN) \
  if (head_dim == DD && warps == NN) return run_bf16<DD, NN>(units, tmk, tmv, p, stream);
  PAV_CASE(64, 1) PAV_CASE(64, 2) PAV_CASE(64, 3) PAV_CASE(64, 4) PAV_CASE(64, 8)
  PAV_CASE(128, 1) PAV_CASE(128, 2) PAV_CASE(128, 3) PAV_CASE(128, 4) PAV_CASE(128, 8)
#undef PAV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pav
