// Log-sum-exp combine of split-KV partials (the "reducer" of a split decode:
// MTP-5 routing page, Motivation). One CTA per output row (token, q head):
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M)
// where O_s is the normalised partial of split s and lse_s its log2-sum-exp.
// Eight warps stride over the splits (four splits' loads in flight per warp),
// each lane owns D/32 columns; the warps' sums meet in shared memory. Rows
// whose (sequence, KV head) was not split were written by the split kernel.
// Launched as a programmatic dependent of the split kernel: the grid may be
// resident before the split kernel ends and waits for it here.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pav {

template <int D>
__global__ void __launch_bounds__(256) pa_combine_kernel(const __grid_constant__ SplitParams p) {
  constexpr int kPer = D / 32;  // columns per lane
  constexpr int kWarps = 8;
  __shared__ float red_m[kWarps];
  __shared__ float red_o[kWarps][D];
  __shared__ float red_w[kWarps];

  asm volatile("griddepcontrol.wait;\n" ::: "memory");

  const int rho = blockIdx.x;
  const WorkView wv = work_view(p);
  if (rho >= wv.num_rows) return;  // a dynamic plan's grid covers its capacity
  int lo = 0, hi = wv.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wv.seq[mid].row_start <= rho) lo = mid; else hi = mid - 1;
  }
  const SeqInfo si = wv.seq[lo];
  const int local = rho - si.row_start;
  const int i = local / p.num_q_heads;
  const int h = local - i * p.num_q_heads;
  const int G = p.group;
  const int kvh = h / G;
  const int r = i * G + (h - kvh * G);
  int n;
  size_t u0;
  if (p.flat) {
    // pair (lo, kvh) covers tiles [t0, t0 + n_tiles); CTA c wrote its piece at slot c + pair
    const int pair = lo * p.num_kv_heads + kvh;
    const int t0 = si.tile_start + kvh * si.n_tiles;
    const int c0 = t0 / wv.per;
    n = (t0 + si.n_tiles - 1) / wv.per - c0 + 1;
    u0 = static_cast<size_t>(c0) + pair;
  } else {
    n = si.n_chunks;
    u0 = static_cast<size_t>(si.unit_start) + static_cast<size_t>(kvh) * n;
  }
  if (n <= 1) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* lse_base = p.part_lse + u0 * p.rows_max + r;
  const float* o_base = p.part_o + (u0 * p.rows_max + r) * D + lane * kPer;
  const size_t o_stride = static_cast<size_t>(p.rows_max) * D;

  // pass 1: the maximum log2-sum-exp
  float m = -INFINITY;
  for (int s = tid; s < n; s += 256) m = fmaxf(m, lse_base[static_cast<size_t>(s) * p.rows_max]);
#pragma unroll
  for (int k = 16; k >= 1; k >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, k));
  if (lane == 0) red_m[warp] = m;
  __syncthreads();
  float M = red_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red_m[w]);

  // pass 2: weighted sum, four splits per warp in flight
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = warp; s0 < n; s0 += 4 * kWarps) {
      float lse[4];
      float o[4][kPer];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = s0 + j * kWarps;
        lse[j] = -INFINITY;
#pragma unroll
        for (int e = 0; e < kPer; ++e) o[j][e] = 0.f;
        if (s < n) {
          lse[j] = lse_base[static_cast<size_t>(s) * p.rows_max];
          const float* src = o_base + static_cast<size_t>(s) * o_stride;
          if constexpr (kPer == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            o[j][0] = v.x; o[j][1] = v.y; o[j][2] = v.z; o[j][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            o[j][0] = v.x; o[j][1] = v.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = fast_exp2(lse[j] - M);  // 0 for a missing or empty split
        wsum += w;
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, o[j][e], acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < kPer; ++e) red_o[warp][lane * kPer + e] = acc[e];
  if (lane == 0) red_w[warp] = wsum;
  __syncthreads();
  if (tid < D) {
    float x = 0.f, ws = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      x += red_o[w][tid];
      ws += red_w[w];
    }
    const float y = ws > 0.f ? x / ws : 0.f;
    const size_t orow = (static_cast<size_t>(si.q_off + i) * p.num_q_heads + h) * D + tid;
    if (p.out_f32) reinterpret_cast<float*>(p.out)[orow] = y;
    else reinterpret_cast<uint16_t*>(p.out)[orow] = static_cast<uint16_t>(pack_bf16(y, 0.f) & 0xFFFFu);
  }
}

cudaError_t launch_combine(int head_dim, const SplitParams* p, cudaStream_t stream) {
  if (p->num_rows <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p->num_rows);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<64>, *p);
  if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<128>, *p);
  return cudaErrorInvalidValue;
}

}  // namespace pav
