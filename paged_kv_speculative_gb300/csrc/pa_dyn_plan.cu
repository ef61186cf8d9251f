// Device-side planner of a dynamic (capacity) plan: turns the call's device
// context/query lengths into the work table the split and combine kernels
// follow, so that one captured CUDA graph serves every batch that fits the
// plan's capacity. Sequences with query length 0 are padding: they get no
// unit and no output row, so they write nothing (stores masked by row
// liveness: DeepSeek-V4.1 page, description of the in-place KV stores). Plans
// of more than 64 sequences built from host lengths use it too: their table
// is too large for the kernel parameters.
//
// Same rules as the host planner (a pair of more than 64 rows is two virtual
// pairs in flat plans). Chunk plans: the chunk is the smallest
// multiple of the staging tile whose unit count fits `slots` (one wave),
// capped at the page-id staging limit. Flat plans: the pairs' K/V tiles of the
// tensor-core kernel end to end, ceil(tiles / slots) of them per CTA. Sequences are scheduled
// longest first (ties by batch index), padded ones last.
//
// One CTA, one thread per sequence of the capacity (up to 1024): the order is
// a bitonic sort of (length, index) keys in shared memory, the offsets are
// block-wide prefix sums.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pav {

constexpr int kPlanThreads = kMaxBatch;  // one thread per sequence of the capacity
static_assert(kPlanThreads == 1024, "the block reductions assume 32 warps");

struct DynPlanArgs {
  const int32_t* ctx;  // [B] device context lengths
  const int32_t* ql;   // [B] device query lengths (0 = padding)
  DynWork* out;
  uint32_t* err;
  int32_t flat;
  int32_t num_seqs, num_q_heads, num_kv_heads, bt_stride, max_len, max_q, slots, tile, max_chunk;
};

// Inclusive prefix sum over the block's 1024 threads (thread order); *total gets the block sum.
__device__ __forceinline__ long long block_scan(long long v, long long* red, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = red[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    red[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += red[warp - 1];
  *total = red[31];
  __syncthreads();  // red is reused by the next call
  return v;
}

__device__ __forceinline__ long long block_sum(long long v, long long* red) {
  long long total;
  (void)block_scan(v, red, &total);
  return total;
}

__device__ __forceinline__ int block_max(int v, long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, m));
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int r = 0;
  for (int w = 0; w < 32; ++w) r = max(r, static_cast<int>(red[w]));
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kPlanThreads) pa_dyn_plan_kernel(DynPlanArgs a) {
  __shared__ unsigned long long s_key[kPlanThreads];
  __shared__ int s_len[kPlanThreads], s_q[kPlanThreads], s_qoff[kPlanThreads];
  __shared__ long long s_red[32];
  const int b = threadIdx.x;
  const bool live = b < a.num_seqs;
  int L = 0, q = 0;
  if (live) {
    L = a.ctx[b];
    q = a.ql[b];
    const bool ok = q >= 1 && q <= a.max_q && L >= q && L <= a.max_len && (L + kPage - 1) / kPage <= a.bt_stride;
    if (q != 0 && !ok && a.err) atomicOr(a.err, 2u);  // outside the plan's capacity: treated as padding
    if (!ok) { L = 0; q = 0; }
  }
  s_len[b] = L;
  s_q[b] = q;

  const long long work = block_sum(static_cast<long long>(L) * a.num_kv_heads, s_red);
  const int max_l = block_max(L, s_red);
  auto units_for = [&](long long c) { return block_sum(L > 0 ? (L + c - 1) / c : 0, s_red) * a.num_kv_heads; };

  int chunk = a.tile;
  if (max_l > 0 && !a.flat) {
    const long long m_hi = (max_l + a.tile - 1) / a.tile;
    long long m_lo = (work + static_cast<long long>(a.slots) * a.tile - 1) / (static_cast<long long>(a.slots) * a.tile);
    m_lo = max(1LL, min(m_lo, m_hi));
    // smallest m in [m_lo, m_hi] with units(m * tile) <= slots (m_hi if none)
    long long lo = m_lo, hi = m_hi;
    while (lo < hi) {
      const long long mid = (lo + hi) / 2;
      if (units_for(mid * a.tile) <= a.slots) hi = mid; else lo = mid + 1;
    }
    chunk = static_cast<int>(min(lo * a.tile, static_cast<long long>(a.max_chunk)));
  }

  // query-row offsets in batch order
  long long tot_tokens;
  s_qoff[b] = static_cast<int>(block_scan(q, s_red, &tot_tokens) - q);

  // order: live sequences by decreasing length (ties by index), then padding by index; entries past the
  // batch sort last and are not written
  s_key[b] = q > 0 ? (static_cast<unsigned long long>(0x7FFFFFFF - L) << 32) | static_cast<unsigned>(b)
                   : (1ull << 63) | static_cast<unsigned>(b);
  __syncthreads();
  for (int k = 2; k <= kPlanThreads; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int o = b ^ j;
      if (o > b) {
        const unsigned long long x = s_key[b], y = s_key[o];
        if ((x > y) == ((b & k) == 0)) {
          s_key[b] = y;
          s_key[o] = x;
        }
      }
      __syncthreads();
    }
  }

  // thread r builds entry r of the table: the sequence of rank r and its offsets in rank order
  const int r = b;
  const int src = static_cast<int>(s_key[r] & 0xFFFFFFFFu);
  const bool in = r < a.num_seqs;
  const int Ls = in ? s_len[src] : 0, qs = in ? s_q[src] : 0;
  const int n_chunks = a.flat ? 0 : (Ls > 0 ? (Ls + chunk - 1) / chunk : 0);
  const int n_tiles = (Ls + a.tile - 1) / a.tile;  // flat plans (the kernel's K/V tiles); 0 for padding
  // flat plans: a pair of more than 64 rows is two virtual pairs (row halves), each a pass over the context
  const int hv = a.flat && qs * (a.num_q_heads / a.num_kv_heads) > 64 ? 2 : 1;
  const long long units_r = static_cast<long long>(n_chunks) * a.num_kv_heads;
  const long long rows_r = static_cast<long long>(qs) * a.num_q_heads;
  const long long tiles_r = static_cast<long long>(n_tiles) * a.num_kv_heads * hv;
  const long long vps_r = static_cast<long long>(a.num_kv_heads) * hv;
  long long total_units, total_rows, total_tiles, total_vps;
  const long long us = block_scan(units_r, s_red, &total_units) - units_r;
  const long long rs = block_scan(rows_r, s_red, &total_rows) - rows_r;
  const long long ts = block_scan(tiles_r, s_red, &total_tiles) - tiles_r;
  const long long vs = block_scan(vps_r, s_red, &total_vps) - vps_r;
  if (in) {
    SeqInfo si;
    si.ctx_len = Ls;
    si.q_len = qs;
    si.q_off = s_qoff[src];
    si.unit_start = static_cast<int>(a.flat ? vs : us);  // flat plans: the entry's first (virtual) pair
    si.row_start = static_cast<int>(rs);
    si.n_chunks = n_chunks;
    si.b = src;
    si.tile_start = static_cast<int>(ts);
    si.n_tiles = n_tiles;
    si.halves = hv;
    dyn_seq(a.out)[r] = si;
  }
  if (b == 0) {
    long long per = 1, n_cta = 0;
    if (total_tiles > 0) {
      per = (total_tiles + a.slots - 1) / a.slots;
      n_cta = (total_tiles + per - 1) / per;  // <= slots, the grid of a flat plan
    }
    a.out->num_units = a.flat ? static_cast<int>(n_cta) : static_cast<int>(total_units);
    a.out->per = static_cast<int>(per);
    a.out->total_tiles = static_cast<int>(total_tiles);
    a.out->chunk = a.flat ? a.tile : chunk;
    a.out->num_rows = static_cast<int>(total_rows);
    a.out->num_tokens = static_cast<int>(tot_tokens);
  }
}

cudaError_t launch_dyn_plan(const int32_t* ctx, const int32_t* ql, DynWork* out, uint32_t* err, int flat, int num_seqs,
                            int num_q_heads, int num_kv_heads, int bt_stride, int max_len, int max_q, int slots, int tile,
                            int max_chunk, cudaStream_t stream) {
  if (num_seqs > kPlanThreads) return cudaErrorInvalidValue;
  DynPlanArgs a{ctx, ql, out, err, flat, num_seqs, num_q_heads, num_kv_heads, bt_stride, max_len, max_q, slots, tile,
                max_chunk};
  pa_dyn_plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pav
