// FP8 (E4M3 + per-token fp32 scales) instantiations of the split kernel (head_dim 128).
#include "pa_split.cuh"

namespace pav {

template <int NW>
static cudaError_t run_fp8(int units, const CUtensorMap* tmk, const CUtensorMap* tmv, const SplitParams* p,
                           cudaStream_t stream) {
  auto kern = pa_split_kernel<1, 128, NW>;
  constexpr int smem = split_smem_bytes(1, 128);
  static std::atomic<uint64_t> attr_done{0};  // devices whose limit is raised
  const cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<units, NW * 32, smem, stream>>>(*tmk, *tmv, *p);
  return cudaGetLastError();
}

cudaError_t launch_split_fp8(int head_dim, int warps, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                             const SplitParams* p, cudaStream_t stream) {
  if (head_dim != 128) return cudaErrorInvalidValue;
  switch (warps) {
    case 1: return run_fp8<1>(units, tmk, tmv, p, stream);
    case 2: return run_fp8<2>(units, tmk, tmv, p, stream);
    case 3: return run_fp8<3>(units, tmk, tmv, p, stream);
    case 4: return run_fp8<4>(units, tmk, tmv, p, stream);
    case 8: return run_fp8<8>(units, tmk, tmv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pav
