// Log-sum-exp combine of split-KV partials (the "reducer" of a split decode:
// MTP-5 routing page, Motivation):
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M)
// where O_s is the normalised partial of split s and lse_s its log2-sum-exp.
// W warps share an output row (token, q head); W grows with the plan's split
// count (1 up to 8 splits, 8 from 33 on). With W = 1 a CTA is two warps (two
// rows, no shared memory); otherwise a CTA is eight warps, on a 64-column slice
// of its rows when whole rows would occupy at most half of the SMs (a batch of
// few rows with many splits: one sequence over the whole GPU; measured on
// GB300, slicing loses once whole rows reach about one CTA per SM). Each warp
// takes every W-th split, eight splits a
// round, loading their lse values and its lanes' columns together (one
// memory round trip per round; rounds combine online, the running sums
// rescaled when the maximum rises); the W warps of a row then merge in shared
// memory. Rows whose (sequence, KV head) was not split were written by the
// split kernel. Plans built from host lengths pass a table of their split pairs
// (CombineTable), so the grid covers only split rows and a row is found by one
// search of that table; plans whose work table lives on the device (or with
// more split pairs than the table holds) cover every row and find it in the
// work table. A plain stream-ordered launch after the split kernel: launched
// as its programmatic dependent instead, the call measured up to 14 us slower
// on GB300 (batch 1 at head_dim 256) and never faster.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pav {

constexpr int kCombineWarpsWide = 8;  // CTAs with W > 1
constexpr int kCombineWarpsNarrow = 2; // CTAs with W = 1
constexpr int kSliceCols = 64;         // columns of a row per CTA with W > 1

__device__ __forceinline__ float ld_cg(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
  return v;
}
// n = 2 or a multiple of 4 consecutive floats (8-byte or 16-byte aligned), in vector loads.
template <int n>
__device__ __forceinline__ void ld_cg_vec(const float* p, float* v) {
  if constexpr (n == 2) {
    asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];\n" : "=f"(v[0]), "=f"(v[1]) : "l"(p));
  } else {
#pragma unroll
    for (int k = 0; k < n; k += 4)
      asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                   : "=f"(v[k]), "=f"(v[k + 1]), "=f"(v[k + 2]), "=f"(v[k + 3])
                   : "l"(p + k));
  }
}

// Warps per output row for a plan whose rows have at most `max_splits` partials.
int combine_warps_per_row(int max_splits) {
  return max_splits <= 8 ? 1 : max_splits <= 16 ? 2 : max_splits <= 32 ? 4 : 8;
}

// A split row: its partials (n of them from slot u0, row r of each) and its place in `out`.
struct RowRef {
  int n;        // partials (1: not split, nothing to merge)
  int r;        // row of the pair inside a partial
  size_t u0;    // slot of the first partial
  size_t orow;  // (token row * Hq + q head), the output row
};

// Row rho of a plan's work table (every row of the batch).
__device__ __forceinline__ RowRef resolve_row(const SplitParams& p, int rho) {
  RowRef rr{0, 0, 0, 0};
  const WorkView wv = work_view(p);
  if (rho >= wv.num_rows) return rr;  // a dynamic plan's grid covers its capacity
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
  rr.r = i * G + (h - kvh * G);
  rr.orow = static_cast<size_t>(si.q_off + i) * p.num_q_heads + h;
  if (p.flat) {
    // (virtual) pair of this row: a pair of more than 64 rows is two, rows 0-63 and the rest, and the partials
    // hold a virtual pair's rows; it covers tiles [t0, t0 + n_tiles) and CTA c wrote its piece at slot
    // slot_base + c + pair
    const int hv = max(1, si.halves), half = hv > 1 ? rr.r / 64 : 0;
    const int vp = kvh * hv + half;
    const int pair = p.rows_split ? si.unit_start + vp : lo * p.num_kv_heads + kvh;
    const int t0 = si.tile_start + vp * si.n_tiles;
    const int c0 = flat_cta_of(wv, t0);
    rr.n = flat_cta_of(wv, t0 + si.n_tiles - 1) - c0 + 1;
    rr.u0 = static_cast<size_t>(p.slot_base) + c0 + pair;
    rr.r -= 64 * half;
  } else {
    rr.n = si.n_chunks;
    rr.u0 = static_cast<size_t>(si.unit_start) + static_cast<size_t>(kvh) * rr.n;
  }
  return rr;
}

// Row rho of a split-pair table (split rows only).
__device__ __forceinline__ RowRef resolve_row(const CombineTable& t, int rho) {
  RowRef rr{0, 0, 0, 0};
  if (rho >= t.num_rows) return rr;
  int lo = 0, hi = t.n_pairs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t.pair[mid].row_base <= rho) lo = mid; else hi = mid - 1;
  }
  const CombinePair cp = t.pair[lo];
  const int r = rho - cp.row_base;          // row of the partials
  const int R = cp.row0 + r;                // row of the pair's q_len * G rows
  const int i = R / t.group;
  rr.n = cp.n;
  rr.r = r;
  rr.u0 = static_cast<size_t>(cp.u0);
  rr.orow = static_cast<size_t>(cp.q_off + i) * t.num_q_heads + cp.head0 + (R - i * t.group);
  return rr;
}

__device__ __forceinline__ int combine_rows(const SplitParams& p) { return work_view(p).num_rows; }
__device__ __forceinline__ int combine_rows(const CombineTable& t) { return t.num_rows; }

template <typename Args, int D, int kWarps, int CW>
__global__ void __launch_bounds__(32 * kWarps) pa_combine_kernel(const __grid_constant__ Args p, int W) {
  constexpr int kPer = CW / 32;  // columns per lane
  constexpr int kSlices = D / CW;  // column slices of a row (consecutive CTAs)
  constexpr int kRound = 8;     // splits in flight per round
  constexpr int kSm = kWarps > 2 ? kWarps : 1;  // the W = 1 form needs no shared memory
  __shared__ float sm_m[kSm], sm_w[kSm];
  __shared__ float sm_acc[kSm][kWarps > 2 ? CW : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wi = warp % W;  // this warp's share of the row's splits
  const int slice = blockIdx.x % kSlices;
  const int rho = (blockIdx.x / kSlices) * (kWarps / W) + warp / W;
  const int col = slice * CW + lane * kPer;  // this lane's first column
  const RowRef rr = resolve_row(p, rho);
  const int n = rr.n, r = rr.r;
  const size_t u0 = rr.u0;
  const bool live = n > 1;  // (warp-uniform; every warp still reaches the barrier below)

  float M = -INFINITY, wsum = 0.f;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  if (live) {
    const float* lse_base = p.part_lse + u0 * p.rows_max + r;
    const float* o_base = p.part_o + (u0 * p.rows_max + r) * D + col;
    const size_t o_stride = static_cast<size_t>(p.rows_max) * D;
    for (int s0 = wi * kRound; s0 < n; s0 += W * kRound) {
      float lse[kRound];
      float o[kRound][kPer];
#pragma unroll
      for (int j = 0; j < kRound; ++j) {
        const int s = s0 + j;
        lse[j] = -INFINITY;
#pragma unroll
        for (int e = 0; e < kPer; ++e) o[j][e] = 0.f;
        if (s < n) {
          lse[j] = ld_cg(lse_base + static_cast<size_t>(s) * p.rows_max);
          ld_cg_vec<kPer>(o_base + static_cast<size_t>(s) * o_stride, o[j]);
        }
      }
      float m = M;
#pragma unroll
      for (int j = 0; j < kRound; ++j) m = fmaxf(m, lse[j]);
      if (m == -INFINITY) continue;  // every split so far is empty
      const float a = M == -INFINITY ? 0.f : fast_exp2(M - m);  // rescale of the earlier rounds
      wsum *= a;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] *= a;
#pragma unroll
      for (int j = 0; j < kRound; ++j) {
        const float w = fast_exp2(lse[j] - m);  // 0 for a missing or empty split
        wsum += w;
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, o[j][e], acc[e]);
      }
      M = m;
    }
  }
  if (kWarps > 2 && W > 1) {  // the row's W warps merge: each rescales to the row maximum
    if (lane == 0) sm_m[warp] = M;
    __syncthreads();
    const int w0 = warp - wi;
    float Mr = -INFINITY;
    for (int k = 0; k < W; ++k) Mr = fmaxf(Mr, sm_m[w0 + k]);
    const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - Mr);
    if (lane == 0) sm_w[warp] = wsum * a;
#pragma unroll
    for (int e = 0; e < kPer; ++e) sm_acc[warp % kSm][(lane * kPer + e) % (kWarps > 2 ? CW : 1)] = acc[e] * a;
    __syncthreads();
    if (wi == 0) {
      wsum = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
      for (int k = 0; k < W; ++k) {
        wsum += sm_w[w0 + k];
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] += sm_acc[(w0 + k) % kSm][(lane * kPer + e) % (kWarps > 2 ? CW : 1)];
      }
    }
  }
  if (!live || wi != 0) return;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t orow = rr.orow * D + col;
  float y[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) y[e] = acc[e] * inv;
  if (p.out_f32) {  // kPer consecutive floats: 8- or 16-byte stores
    float* dst = reinterpret_cast<float*>(p.out) + orow;
    if constexpr (kPer == 2) {
      *reinterpret_cast<float2*>(dst) = make_float2(y[0], y[1]);
    } else {
#pragma unroll
      for (int e = 0; e < kPer; e += 4) *reinterpret_cast<float4*>(dst + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
    }
  } else {  // kPer bf16: 4-, 8- or 16-byte stores
    uint32_t w[kPer / 2];
#pragma unroll
    for (int e = 0; e < kPer; e += 2) w[e / 2] = pack_bf16(y[e], y[e + 1]);
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + orow;
    if constexpr (kPer == 2) *reinterpret_cast<uint32_t*>(dst) = w[0];
    else if constexpr (kPer == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <typename Args>
static cudaError_t launch_combine_args(int head_dim, const Args& a, int num_rows, int max_splits, int sm_count,
                                       cudaStream_t stream) {
  if (num_rows <= 0) return cudaSuccess;
  const int W = combine_warps_per_row(max_splits);
  const int warps = W == 1 ? kCombineWarpsNarrow : kCombineWarpsWide;
  const int rows_per_cta = warps / W;
  const int row_ctas = (num_rows + rows_per_cta - 1) / rows_per_cta;
  const bool sliced = W > 1 && 2 * row_ctas <= sm_count;
  const int slices = sliced ? head_dim / kSliceCols : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(row_ctas * slices);
  cfg.blockDim = dim3(32 * warps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  if (W == 1) {
    if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 64, kCombineWarpsNarrow, 64>, a, W);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 128, kCombineWarpsNarrow, 128>, a, W);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 256, kCombineWarpsNarrow, 256>, a, W);
  } else if (sliced) {
    if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 64, kCombineWarpsWide, kSliceCols>, a, W);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 128, kCombineWarpsWide, kSliceCols>, a, W);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 256, kCombineWarpsWide, kSliceCols>, a, W);
  } else {
    if (head_dim == 64) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 64, kCombineWarpsWide, 64>, a, W);
    if (head_dim == 128) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 128, kCombineWarpsWide, 128>, a, W);
    if (head_dim == 256) return cudaLaunchKernelEx(&cfg, pa_combine_kernel<Args, 256, kCombineWarpsWide, 256>, a, W);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(int head_dim, const SplitParams* p, const CombineTable* t, int max_splits, int sm_count,
                           cudaStream_t stream) {
  if (t) return launch_combine_args(head_dim, *t, t->num_rows, max_splits, sm_count, stream);
  return launch_combine_args(head_dim, *p, p->num_rows, max_splits, sm_count, stream);
}

}  // namespace pav
