// Device-side planner of a dynamic (capacity) plan: turns the call's device
// context/query lengths into the work table the split and combine kernels
// follow, so that one captured CUDA graph serves every batch that fits the
// plan's capacity. Sequences with query length 0 are padding: they get no
// unit and no output row, so they write nothing (stores masked by row
// liveness: DeepSeek-V4.1 page, description of the in-place KV stores).
//
// Same rules as the host planner. Chunk plans: the chunk is the smallest
// multiple of the staging tile whose unit count fits `slots` (one wave),
// capped at the page-id staging limit. Flat plans: the pairs' 128-token tiles
// end to end, ceil(tiles / slots) of them per CTA. Sequences are scheduled
// longest first.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pav {

struct DynPlanArgs {
  const int32_t* ctx;  // [B] device context lengths
  const int32_t* ql;   // [B] device query lengths (0 = padding)
  DynWork* out;
  uint32_t* err;
  int32_t flat;
  int32_t num_seqs, num_q_heads, num_kv_heads, bt_stride, max_len, max_q, slots, tile, max_chunk;
};

__global__ void __launch_bounds__(64) pa_dyn_plan_kernel(DynPlanArgs a) {
  __shared__ int s_len[kMaxSeqs], s_q[kMaxSeqs], s_rank_units[kMaxSeqs], s_rank_rows[kMaxSeqs], s_rank_tiles[kMaxSeqs];
  __shared__ int s_red[2];
  __shared__ long long s_red64[2];
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
  const int lane = b & 31, warp = b >> 5;

  // block-wide sums / maximum over the 64 threads
  auto sum64 = [&](long long v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    __syncthreads();
    if (lane == 0) s_red64[warp] = v;
    __syncthreads();
    return s_red64[0] + s_red64[1];
  };
  auto max64 = [&](int v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, m));
    __syncthreads();
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    return max(s_red[0], s_red[1]);
  };
  const long long work = sum64(static_cast<long long>(L) * a.num_kv_heads);
  const int max_l = max64(L);
  const long long n_live = sum64(q > 0 ? 1 : 0);
  auto units_for = [&](long long c) { return sum64(L > 0 ? (L + c - 1) / c : 0) * a.num_kv_heads; };

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
  const int n_chunks = a.flat ? 0 : (L > 0 ? (L + chunk - 1) / chunk : 0);
  const int n_tiles = (L + kFlatTile - 1) / kFlatTile;  // 0 for padding

  // rank: live sequences by decreasing length (ties by index), then padding by index
  int rank = 0;
  for (int c = 0; c < a.num_seqs; ++c) {
    if (c == b) continue;
    const bool other_live = s_q[c] > 0;
    if (q > 0) {
      if (other_live && (s_len[c] > L || (s_len[c] == L && c < b))) ++rank;
    } else {
      if (other_live || c < b) ++rank;
    }
  }
  // query-row offset in batch order
  int q_off = 0;
  for (int c = 0; c < b && c < a.num_seqs; ++c) q_off += s_q[c];
  __syncthreads();
  if (live) {
    s_rank_units[rank] = n_chunks * a.num_kv_heads;
    s_rank_rows[rank] = q * a.num_q_heads;
    s_rank_tiles[rank] = n_tiles * a.num_kv_heads;
  }
  __syncthreads();
  if (live) {
    int us = 0, rs = 0, ts = 0;
    for (int r = 0; r < rank; ++r) {
      us += s_rank_units[r];
      rs += s_rank_rows[r];
      ts += s_rank_tiles[r];
    }
    SeqInfo si;
    si.ctx_len = L;
    si.q_len = q;
    si.q_off = q_off;
    si.unit_start = us;
    si.row_start = rs;
    si.n_chunks = n_chunks;
    si.b = b;
    si.tile_start = ts;
    si.n_tiles = n_tiles;
    si.pad = 0;
    a.out->seq[rank] = si;
  }
  const long long total_units = sum64(static_cast<long long>(n_chunks) * a.num_kv_heads);
  const long long total_rows = sum64(static_cast<long long>(q) * a.num_q_heads);
  const long long total_tokens = sum64(q);
  const long long total_tiles = sum64(static_cast<long long>(n_tiles) * a.num_kv_heads);
  if (b == 0) {
    long long per = 1, n_cta = 0;
    if (total_tiles > 0) {
      per = (total_tiles + a.slots - 1) / a.slots;
      n_cta = (total_tiles + per - 1) / per;  // <= slots, the grid of a flat plan
    }
    a.out->num_units = a.flat ? static_cast<int>(n_cta) : static_cast<int>(total_units);
    a.out->per = static_cast<int>(per);
    a.out->total_tiles = static_cast<int>(total_tiles);
    a.out->chunk = a.flat ? kFlatTile : chunk;
    a.out->num_rows = static_cast<int>(total_rows);
    a.out->num_tokens = static_cast<int>(total_tokens);
  }
  (void)n_live;
}

cudaError_t launch_dyn_plan(const int32_t* ctx, const int32_t* ql, DynWork* out, uint32_t* err, int flat, int num_seqs,
                            int num_q_heads, int num_kv_heads, int bt_stride, int max_len, int max_q, int slots, int tile,
                            int max_chunk, cudaStream_t stream) {
  DynPlanArgs a{ctx, ql, out, err, flat, num_seqs, num_q_heads, num_kv_heads, bt_stride, max_len, max_q, slots, tile,
                max_chunk};
  pa_dyn_plan_kernel<<<1, 64, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pav
