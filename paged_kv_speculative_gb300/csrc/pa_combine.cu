// Log-sum-exp combine of split-KV partials (the "reducer" of a split decode:
// MTP-5 routing page, Motivation). One CTA per output row (token, q head):
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M)
// where O_s is the normalised partial of split s and lse_s its log2-sum-exp.
// Rows whose (sequence, KV head) was not split were written by the split
// kernel and are skipped here.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pav {

template <int D>
__global__ void __launch_bounds__(128) pa_combine_kernel(const __grid_constant__ SplitParams p) {
  constexpr int kQuads = D / 4;            // float4 columns per row
  constexpr int kLanes = 128 / kQuads;     // split lanes per column
  __shared__ float red_m[128];
  __shared__ float4 red_o[128];
  __shared__ float red_w[128];

  const int rho = blockIdx.x;
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.seq[mid].row_start <= rho) lo = mid; else hi = mid - 1;
  }
  const SeqInfo& si = p.seq[lo];
  const int n = si.n_chunks;
  if (n <= 1) return;
  const int local = rho - si.row_start;
  const int i = local / p.num_q_heads;
  const int h = local - i * p.num_q_heads;
  const int G = p.group;
  const int kvh = h / G;
  const int r = i * G + (h - kvh * G);
  const int u0 = si.unit_start + kvh * n;

  const int tid = threadIdx.x;
  const int quad = tid % kQuads;
  const int sl = tid / kQuads;

  float m = -INFINITY;
  for (int s = sl; s < n; s += kLanes) m = fmaxf(m, p.part_lse[static_cast<size_t>(u0 + s) * p.rows_max + r]);
  red_m[tid] = m;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kLanes; ++k) M = fmaxf(M, red_m[k * kQuads + quad]);

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = sl; s < n; s += kLanes) {
      const size_t base = static_cast<size_t>(u0 + s) * p.rows_max + r;
      const float lse = p.part_lse[base];
      const float w = fast_exp2(lse - M);  // 0 for an empty split (lse = -inf)
      const float4 o = *reinterpret_cast<const float4*>(p.part_o + base * D + 4 * quad);
      wsum += w;
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  red_o[tid] = acc;
  red_w[tid] = wsum;
  __syncthreads();
  if (sl != 0) return;
#pragma unroll
  for (int k = 1; k < kLanes; ++k) {
    const float4 o = red_o[k * kQuads + quad];
    acc.x += o.x; acc.y += o.y; acc.z += o.z; acc.w += o.w;
    wsum += red_w[k * kQuads + quad];
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t orow = (static_cast<size_t>(si.q_off + i) * p.num_q_heads + h) * D + 4 * quad;
  if (p.out_f32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + orow) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  } else {
    uint2 w;
    w.x = pack_bf16(acc.x * inv, acc.y * inv);
    w.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) + orow) = w;
  }
}

cudaError_t launch_combine(int head_dim, const SplitParams* p, cudaStream_t stream) {
  if (p->num_rows <= 0) return cudaSuccess;
  if (head_dim == 64) pa_combine_kernel<64><<<p->num_rows, 128, 0, stream>>>(*p);
  else if (head_dim == 128) pa_combine_kernel<128><<<p->num_rows, 128, 0, stream>>>(*p);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pav
