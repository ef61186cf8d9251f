// Instantiations of the tcgen05 split kernel for head_dim 256: FP8 E4M3 K/V
// (the shape the aiter follow-up on the MTP-5 routing page measures: GQA 8 x
// query length 6 = 48 rows over one KV head) and bf16 K/V, rows padded to
// 16..64.
#include "pa_tc_split.cuh"

namespace pav {

cudaError_t launch_tc_split_d256(int kv_fp8, int rows_max, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                 const SplitParams* p, cudaStream_t stream) {
  if (!kv_fp8) {
    switch (tc_rows_pad(rows_max)) {
      case 16: return run_tc<0, 16, 256>(units, tmk, tmv, p, stream);
      case 32: return run_tc<0, 32, 256>(units, tmk, tmv, p, stream);
      case 48: return run_tc<0, 48, 256>(units, tmk, tmv, p, stream);
      case 64: return run_tc<0, 64, 256>(units, tmk, tmv, p, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (tc_rows_pad(rows_max)) {
    case 16: return run_tc<1, 16, 256>(units, tmk, tmv, p, stream);
    case 32: return run_tc<1, 32, 256>(units, tmk, tmv, p, stream);
    case 48: return run_tc<1, 48, 256>(units, tmk, tmv, p, stream);
    case 64: return run_tc<1, 64, 256>(units, tmk, tmv, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pav
