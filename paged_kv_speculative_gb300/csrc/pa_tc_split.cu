// Instantiations of the tcgen05 split kernel for head_dim 128 (bf16 and FP8
// KV; FP8 up to 48 rows in 256-token K/V tiles), q_len * group rows padded to
// 16, 32, 48 or 64, and the dispatch over
// head_dim (the FP8 head_dim-256 instances live in their own translation unit
// so that the two compile in parallel).
#include "pa_tc_split.cuh"

namespace pav {

cudaError_t launch_tc_split_d256(int kv_fp8, int rows_max, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                 const SplitParams* p, cudaStream_t stream);

cudaError_t launch_tc_split_d64(int kv_fp8, int rows_max, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                const SplitParams* p, cudaStream_t stream);

cudaError_t launch_tc_split(int head_dim, int kv_fp8, int rows_max, int units, const CUtensorMap* tmk,
                            const CUtensorMap* tmv, const SplitParams* p, cudaStream_t stream) {
  if (head_dim == 256) return launch_tc_split_d256(kv_fp8, rows_max, units, tmk, tmv, p, stream);
  if (head_dim == 64) return launch_tc_split_d64(kv_fp8, rows_max, units, tmk, tmv, p, stream);
  if (head_dim != 128) return cudaErrorInvalidValue;
  const int np = tc_rows_pad(rows_max);
#define PAV_TC(F, N) \
  if (kv_fp8 == F && np == N) return run_tc<F, N, 128, tc_subtiles(F, 128, N)>(units, tmk, tmv, p, stream);
  PAV_TC(0, 16) PAV_TC(0, 32) PAV_TC(0, 48) PAV_TC(0, 64)
  PAV_TC(1, 16) PAV_TC(1, 32) PAV_TC(1, 48) PAV_TC(1, 64)
#undef PAV_TC
  return cudaErrorInvalidValue;
}

}  // namespace pav
