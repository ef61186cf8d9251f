// Instantiations of the tcgen05 split kernel for head_dim 64 with bf16 K/V,
// rows padded to 16..64 (own translation unit, compiled in parallel).
#include "pa_tc_split.cuh"

namespace pav {

cudaError_t launch_tc_split_d64(int kv_fp8, int rows_max, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                const SplitParams* p, cudaStream_t stream) {
  if (kv_fp8) return cudaErrorInvalidValue;
  switch (tc_rows_pad(rows_max)) {
    case 16: return run_tc<0, 16, 64>(units, tmk, tmv, p, stream);
    case 32: return run_tc<0, 32, 64>(units, tmk, tmv, p, stream);
    case 48: return run_tc<0, 48, 64>(units, tmk, tmv, p, stream);
    case 64: return run_tc<0, 64, 64>(units, tmk, tmv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pav
