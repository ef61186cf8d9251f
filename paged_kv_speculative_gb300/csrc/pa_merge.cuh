// Log-sum-exp merge of a flat plan's split pairs inside the split kernel (the
// "reducer" of a split decode: MTP-5 routing page, Motivation):
//   M = max_s lse_s,  out = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M)
// for every row of every (sequence, KV head) pair whose tiles were cut over
// several CTAs, O_s being the normalised partial of CTA s and lse_s its
// log2-sum-exp.
//
// When a CTA has finished all of its tiles it arrives on a counter per split
// pair it worked on (at most two: the pairs of its first and last tiles).
// Each of a pair's n CTAs then waits until all n have arrived and merges an
// even share of the pair's rows, so the merge of every pair is spread over the
// CTAs that made it and starts as soon as its last piece is written. With few
// rows per CTA and many splits (one long sequence over the whole GPU), several
// warps share a row, each taking every W-th split, and meet in shared memory.
// The waits are on other CTAs of the same grid: the kernel is launched
// cooperatively (all CTAs resident at once), and every wait is bounded.
//
// The counter of a pair goes 0 -> n (arrivals) -> 2n (departures after the
// merge); the CTA whose departure makes it 2n stores 0 again, so every run
// leaves the counters at zero. A CTA departs only after it saw all n
// arrivals, so a departure can never be mistaken for an arrival.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pav {

__device__ __forceinline__ void red_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("fence.acq_rel.gpu;\n red.relaxed.gpu.global.add.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];\n" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ float ld_cg_f1(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
  return v;
}

// A split pair of a flat plan, as one CTA sees it.
struct SplitPair {
  int pair;      // k * Hkv + g
  int k, g;      // work-table entry and KV head
  int c0, n;     // first CTA and CTA count of the pair
};

// The pair holding flat tile f, and whether CTA range [f_lo, f_hi) leaves part of it to other CTAs.
__device__ __forceinline__ bool split_pair_of(const WorkView& wv, int hkv, int f, int f_lo, int f_hi, SplitPair& sp) {
  sp.k = flat_seq_of(wv, f);
  const SeqInfo& s = wv.seq[sp.k];
  sp.g = (f - s.tile_start) / s.n_tiles;
  sp.pair = sp.k * hkv + sp.g;
  const int t0 = s.tile_start + sp.g * s.n_tiles, t1 = t0 + s.n_tiles;  // the pair's tiles [t0, t1)
  sp.c0 = flat_cta_of(wv, t0);
  sp.n = flat_cta_of(wv, t1 - 1) - sp.c0 + 1;
  return t0 < f_lo || t1 > f_hi;
}

// Waits for all CTAs of split pair `q` to arrive, merges this CTA's share of
// its rows, then departs. Every thread of the CTA calls it.
template <int D, int kThreads>
__device__ __noinline__ void merge_one_pair(const SplitParams& p, const WorkView& wv, int cta, SplitPair q,
                                            float* smem) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kPer = D / 32;  // columns per lane
  constexpr int kRound = 8;     // splits in flight per warp and round
  static_assert(kPer == 4 || kPer == 8, "head_dim 128 or 256");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  float* s_m = smem;                       // [kWarps] maxima
  float* s_w = smem + kWarps;              // [kWarps] weight sums
  float* s_acc = smem + 2 * kWarps;        // [kWarps][D] weighted sums
  int& s_ok = *reinterpret_cast<int*>(smem + (2 + D) * kWarps);
  {
    const int n = q.n;
    uint32_t* cnt = p.pair_count + q.pair;
    if (tid == 0) {
      bool ok = true;
      if (ld_acquire_gpu(cnt) < static_cast<uint32_t>(n)) {
        const uint64_t lim = p.wait_limit_ns ? p.wait_limit_ns : 1000000000ull;
        const uint64_t t0 = global_ns();
        while (ld_acquire_gpu(cnt) < static_cast<uint32_t>(n)) {
          if (global_ns() - t0 > lim) {
            ok = false;
            atomicOr(p.err, 4u);
            break;
          }
        }
      }
      s_ok = ok;
    }
    __syncthreads();
    const SeqInfo& si = wv.seq[q.k];
    const int R = si.q_len * G;
    const int kc = cta - q.c0;  // this CTA's index among the pair's
    const int r0 = kc * R / n, r1 = (kc + 1) * R / n;
    const int rows = r1 - r0;
    if (s_ok && rows > 0) {
      const int W = max(1, min(kWarps / rows, (n + kRound - 1) / kRound));  // warps per row
      const int groups = kWarps / W;
      const size_t u0 = static_cast<size_t>(q.c0) + q.pair;  // slot of the pair's first split
      for (int base = 0; base < rows; base += groups) {
        const int gi = warp / W, wi = warp - gi * W;
        const int r = r0 + base + gi;
        const bool live = gi < groups && base + gi < rows;
        float M = -INFINITY, wsum = 0.f;
        float acc[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
        if (live) {
          const float* lse_base = p.part_lse + u0 * p.rows_max + r;
          const float* o_base = p.part_o + (u0 * p.rows_max + r) * D + lane * kPer;
          const size_t o_stride = static_cast<size_t>(p.rows_max) * D;
          for (int s0 = wi * kRound; s0 < n; s0 += W * kRound) {
            float lse[kRound];
            float o[kRound][kPer];
#pragma unroll
            for (int jj = 0; jj < kRound; ++jj) {
              const int s = s0 + jj;
              lse[jj] = -INFINITY;
#pragma unroll
              for (int e = 0; e < kPer; ++e) o[jj][e] = 0.f;
              if (s < n) {
                lse[jj] = ld_cg_f1(lse_base + static_cast<size_t>(s) * p.rows_max);
#pragma unroll
                for (int e = 0; e < kPer; e += 4) {
                  const float4 v = ld_cg_f4(o_base + static_cast<size_t>(s) * o_stride + e);
                  o[jj][e] = v.x;
                  o[jj][e + 1] = v.y;
                  o[jj][e + 2] = v.z;
                  o[jj][e + 3] = v.w;
                }
              }
            }
            float m = M;
#pragma unroll
            for (int jj = 0; jj < kRound; ++jj) m = fmaxf(m, lse[jj]);
            if (m == -INFINITY) continue;  // no visible key in any split so far
            const float a = M == -INFINITY ? 0.f : fast_exp2(M - m);
            wsum *= a;
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] *= a;
#pragma unroll
            for (int jj = 0; jj < kRound; ++jj) {
              const float w = fast_exp2(lse[jj] - m);  // 0 for a missing or empty split
              wsum += w;
#pragma unroll
              for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, o[jj][e], acc[e]);
            }
            M = m;
          }
        }
        if (W > 1) {  // the row's W warps meet: each rescales to the row maximum
          if (lane == 0) s_m[warp] = M;
          __syncthreads();
          float Mr = -INFINITY;
          if (live)
            for (int w = 0; w < W; ++w) Mr = fmaxf(Mr, s_m[gi * W + w]);
          const float a = (M == -INFINITY) ? 0.f : fast_exp2(M - Mr);
          if (lane == 0) s_w[warp] = wsum * a;
#pragma unroll
          for (int e = 0; e < kPer; ++e) s_acc[warp * D + lane * kPer + e] = acc[e] * a;
          __syncthreads();
          if (live && wi == 0) {
            wsum = 0.f;
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
            for (int w = 0; w < W; ++w) {
              wsum += s_w[gi * W + w];
#pragma unroll
              for (int e = 0; e < kPer; ++e) acc[e] += s_acc[(gi * W + w) * D + lane * kPer + e];
            }
          }
          __syncthreads();  // the shared rows are reused by the next round
        }
        if (live && wi == 0) {
          const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
          const int i = r / G;
          const size_t orow =
              (static_cast<size_t>(si.q_off + i) * p.num_q_heads + q.g * G + (r - i * G)) * D + lane * kPer;
          if (p.out_f32) {
            float* dst = reinterpret_cast<float*>(p.out) + orow;
#pragma unroll
            for (int e = 0; e < kPer; e += 4)
              *reinterpret_cast<float4*>(dst + e) =
                  make_float4(acc[e] * inv, acc[e + 1] * inv, acc[e + 2] * inv, acc[e + 3] * inv);
          } else {  // kPer bf16: one 8- or 16-byte store
            uint32_t w[kPer / 2];
#pragma unroll
            for (int e = 0; e < kPer; e += 2) w[e / 2] = pack_bf16(acc[e] * inv, acc[e + 1] * inv);
            uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + orow;
            if constexpr (kPer == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
    // depart: every read of the pair's partials is done; the last departure resets the counter
    __syncthreads();
    if (tid == 0 && atom_add_acq_rel_gpu(cnt, 1u) == 2u * n - 1u) *cnt = 0u;
  }
}

// Called by every thread of the CTA after its tiles are done (kThreads
// threads; `smem`: (D + 2) * kThreads / 32 + 1 words of free shared memory):
// arrives on the split pairs of the CTA's first and last tiles, then merges
// its share of each. Everything is recomputed from the kernel parameters, so
// the split kernel keeps nothing alive for it.
template <int D, int kThreads>
__device__ __noinline__ void merge_split_pairs(const SplitParams& p, float* smem) {
  const WorkView wv = work_view(p);
  const int cta = blockIdx.x;
  const int f_lo = flat_cta_start(wv, cta), f_hi = flat_cta_start(wv, cta + 1);
  if (f_hi <= f_lo) return;
  const int hkv = p.num_kv_heads;
  SplitPair a, b;
  const bool has_a = split_pair_of(wv, hkv, f_lo, f_lo, f_hi, a);
  const bool has_b = split_pair_of(wv, hkv, f_hi - 1, f_lo, f_hi, b) && !(has_a && b.pair == a.pair);
  if (!has_a && !has_b) return;
  // arrive: the CTA's partials (written before the barrier) are released with the count
  __syncthreads();
  if (threadIdx.x == 0) {
    if (has_a) red_release_gpu(p.pair_count + a.pair, 1u);
    if (has_b) red_release_gpu(p.pair_count + b.pair, 1u);
  }
  if (has_a) merge_one_pair<D, kThreads>(p, wv, cta, a, smem);
  if (has_b) merge_one_pair<D, kThreads>(p, wv, cta, b, smem);
}

}  // namespace pav
