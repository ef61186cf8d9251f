// Instantiations of the tcgen05 split kernel: bf16 and FP8 KV, head_dim 128,
// q_len * group rows padded to 16, 32, 48 or 64.
#include "pa_tc_split.cuh"

namespace pav {

template <int F8, int NP>
static cudaError_t run_tc(int units, const CUtensorMap* tmk, const CUtensorMap* tmv, const SplitParams* p,
                          cudaStream_t stream) {
  auto kern = pa_tc_split_kernel<F8, NP>;
  constexpr int smem = TcCfg<F8, NP>::kSmem;
  static bool attr_set = false;  // benign race: setting the attribute twice is harmless
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<units, 352, smem, stream>>>(*tmk, *tmv, *p);
  return cudaGetLastError();
}

int tc_rows_pad(int rows_max) { return rows_max <= 16 ? 16 : rows_max <= 32 ? 32 : rows_max <= 48 ? 48 : 64; }

cudaError_t launch_tc_split(int kv_fp8, int rows_max, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                            const SplitParams* p, cudaStream_t stream) {
  const int np = tc_rows_pad(rows_max);
#define PAV_TC(F, N) \
  if (kv_fp8 == F && np == N) return run_tc<F, N>(units, tmk, tmv, p, stream);
  PAV_TC(0, 16) PAV_TC(0, 32) PAV_TC(0, 48) PAV_TC(0, 64)
  PAV_TC(1, 16) PAV_TC(1, 32) PAV_TC(1, 48) PAV_TC(1, 64)
#undef PAV_TC
  return cudaErrorInvalidValue;
}

}  // namespace pav
