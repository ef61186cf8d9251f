// Internal declarations shared by the host planner / C ABI and the kernels.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace pav {

constexpr int kPage = 16;         // tokens per KV page
constexpr int kMaxSeqs = 64;      // sequences whose table travels in the kernel parameters (plans built on the host)
constexpr int kMaxBatch = 1024;   // sequences per call; above kMaxSeqs the table is built on the device at each run
constexpr int kStages = 3;        // shared-memory ring depth of the split kernel
constexpr int kMaxChunk = 16384;  // context tokens per work unit (bounds the page-id staging array)
constexpr int kMaxRows = 128;     // q_len * group rows per (sequence, KV head)
constexpr int kMaxQueryLen = 8;
constexpr int kWsHeader = 256;    // workspace bytes before the partials (device error word at offset 0)

constexpr int kFlatTile = 128;   // tokens per MMA sub-tile of the tcgen05 kernel (the MMA's M)
// 128-token sub-tiles per K/V tile of the tcgen05 kernel: two for FP8 K/V at head_dim 128 with up to 48
// rows (np: rows padded to the instance's N), one elsewhere. (Measured on GB300, split kernel: MTP-5 FP8
// 174 -> 160 us with two; bf16 slower with two, 65 -> 78 us at MTP-5, as its 64 KB tiles leave room for
// one ring stage each; the 64-row FP8 instance spills with two.)
__host__ __device__ constexpr int tc_subtiles(int kv_fp8, int head_dim, int np) {
  return kv_fp8 && head_dim == 128 && np <= 48 ? 2 : 1;
}
// tokens per tile of a flat plan (the tcgen05 kernel's K/V tile)
__host__ __device__ constexpr int tc_tile_tokens(int kv_fp8, int head_dim, int np) {
  return kFlatTile * tc_subtiles(kv_fp8, head_dim, np);
}
constexpr int kMaxCtaTable = 512; // flat plans: CTAs whose tile ranges a plan can list in the kernel parameters

// Per-sequence entry of the work description, sorted by decreasing context
// length so that the longest units are scheduled first.
//
// Two kinds of plan share it. A chunk plan (warp-MMA kernel) gives every
// (sequence, KV head, chunk) its own CTA. A flat plan (tcgen05 kernel) lays
// the (sequence, KV head) pairs end to end as K/V tiles (tc_tile_tokens), pair p =
// k * Hkv + g for the k-th entry and head g, and hands every CTA the same
// number of consecutive tiles (`per`): CTA c works through the pieces
// ("segments") of the pairs its range [c * per, (c + 1) * per) touches. The
// partial of pair p made by CTA c sits at slot c + p, which is unique and
// increases along the tiles, so the slots of one pair are consecutive.
struct SeqInfo {
  int32_t ctx_len;     // L_b
  int32_t q_len;       // q_b
  int32_t q_off;       // first row of sequence b in q / out (batch order)
  int32_t unit_start;  // chunk plans: first work unit of this sequence (units: kv head major, then chunk);
                       // flat plans with row halves: first virtual pair of this sequence
  int32_t row_start;   // first combine row of this sequence (q_len * Hq rows)
  int32_t n_chunks;    // chunk plans: ceil(L_b / chunk)
  int32_t b;           // index of the sequence in the caller's batch
  int32_t tile_start;  // flat plans: first tile of head 0 (head g, row half h starts at
                       // tile_start + (g * halves + h) * n_tiles)
  int32_t n_tiles;     // flat plans: ceil(L_b / tile) tiles per KV head (0 for a padded sequence)
  int32_t halves;      // flat plans: row halves of each pair, 2 when q_len * G > 64 (rows 0-63, then the
                       // rest: two virtual pairs, each a pass over the context); 0 or 1: one
};

// Work description written on the device by the planner kernel of a
// dynamic (capacity) plan, from the device lengths of the call. The header is
// followed by the per-sequence table, one SeqInfo per sequence of the
// capacity: live sequences by decreasing length, then padded ones.
struct DynWork {
  int32_t num_units;  // split units (flat plans: CTAs with work) of this call
  int32_t chunk;      // context tokens per unit (flat plans: 128)
  int32_t num_rows;   // combine rows of this call (sum of q_b * Hq)
  int32_t num_tokens; // sum of q_b
  int32_t per;        // flat plans: tiles per CTA
  int32_t total_tiles;
  int32_t pad[2];
};
__host__ __device__ inline SeqInfo* dyn_seq(DynWork* w) { return reinterpret_cast<SeqInfo*>(w + 1); }
__host__ __device__ inline const SeqInfo* dyn_seq(const DynWork* w) { return reinterpret_cast<const SeqInfo*>(w + 1); }
// Workspace bytes of a device work table for `capacity` sequences.
inline size_t dyn_work_bytes(int capacity) { return sizeof(DynWork) + static_cast<size_t>(capacity) * sizeof(SeqInfo); }

struct SplitParams {
  const uint16_t* q;            // [T, Hq, D] bf16
  const int32_t* block_table;   // [B, stride]
  const float* k_scale;         // [N_pg, Hkv, 16] or null
  const float* v_scale;
  void* out;                    // [T, Hq, D] bf16 | f32
  float* part_o;                // [U, rows_max, D]
  float* part_lse;              // [U, rows_max], log2 domain
  uint32_t* err;                // device error word
  const int32_t* dev_ctx;       // device copies of the lengths (checked against the plan)
  const int32_t* dev_q;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t bt_stride;
  int32_t num_pages;
  int32_t chunk;
  int32_t num_units;
  int32_t rows_max;             // row stride of the partials
  int32_t slot_base;            // flat plans: first partial slot of this launch (CTA c, pair p: slot_base + c + p)
  int32_t rows_split;           // flat plans: 1 when some entry has two row halves (pair p is then the entry's
                                // unit_start + g * halves + h), else 0 (p = entry * Hkv + g)
  int32_t out_f32;
  int32_t num_rows;             // sum_b q_b * Hq (combine grid)
  int32_t flat;                 // 1: flat plan (tiles per CTA), 0: chunk plan
  int32_t per;                  // flat plans: tiles per CTA (when no range table is given)
  int32_t total_tiles;          // flat plans: tiles of every pair
  int32_t ranged;               // flat plans: 1 when cta_start lists every CTA's first tile
  int32_t cta_start[kMaxCtaTable + 1];  // CTA c covers tiles [cta_start[c], cta_start[c + 1])
  float scale_log2;             // softmax_scale * log2(e)
  const DynWork* dyn;           // dynamic plans: the device-written work table; else null
  uint64_t wait_limit_ns;       // a bounded wait gives up after this long (0: one second)
  int32_t stall_cta;            // test hook: this CTA's MMA issuer first waits on a barrier that nothing
                                // completes, so its bounded wait runs out (-1: none)
  SeqInfo seq[kMaxSeqs];
};

// Device error word and diagnostic counters at the start of a workspace.
constexpr int kWsErrWord = 0;       // PA_DEVERR_* bits
constexpr int kWsRescaleWord = 1;   // in-segment rescales of the O accumulator (tcgen05 kernel)

#ifdef __CUDACC__
// The work table a kernel follows: kernel parameters (plans built from host
// lengths) or the device planner's output (dynamic plans; grids are sized for
// the plan's capacity and CTAs past the call's work return at once).
struct WorkView {
  const SeqInfo* seq;
  int num_seqs, chunk, num_units, num_rows, per, total_tiles;
  const int32_t* cta_start;  // flat plans with a range table, else null (CTA c starts at c * per)
};
__device__ __forceinline__ WorkView work_view(const SplitParams& p) {
  if (p.dyn)
    return WorkView{dyn_seq(p.dyn), p.num_seqs, p.dyn->chunk, p.dyn->num_units, p.dyn->num_rows, p.dyn->per,
                    p.dyn->total_tiles, nullptr};
  return WorkView{p.seq, p.num_seqs, p.chunk, p.num_units, p.num_rows, p.per, p.total_tiles,
                  p.ranged ? p.cta_start : nullptr};
}
// First tile of CTA c of a flat plan (c = num_units gives the end).
__device__ __forceinline__ int flat_cta_start(const WorkView& wv, int c) {
  return wv.cta_start ? wv.cta_start[c] : min(c * wv.per, wv.total_tiles);
}
// The CTA of a flat plan whose range holds tile f.
__device__ __forceinline__ int flat_cta_of(const WorkView& wv, int f) {
  if (!wv.cta_start) return f / wv.per;
  int lo = 0, hi = wv.num_units - 1;  // the last CTA starting at or before f
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wv.cta_start[mid] <= f) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// Index of the entry whose tiles contain flat tile f (the last entry with tile_start <= f).
__device__ __forceinline__ int flat_seq_of(const WorkView& wv, int f) {
  int lo = 0, hi = wv.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wv.seq[mid].tile_start <= f) lo = mid; else hi = mid - 1;
  }
  return lo;
}
#endif

// Tile geometry of the split kernel for a KV element size and head dim.
__host__ __device__ constexpr int row_bytes(int kv_fp8, int d) { return d * (kv_fp8 ? 1 : 2); }
__host__ __device__ constexpr int tile_tokens(int kv_fp8, int d) { return 16384 / row_bytes(kv_fp8, d); }
__host__ __device__ constexpr int stage_bytes(int kv_fp8, int d) {
  return 2 * 16384 + (kv_fp8 ? 2 * 4 * tile_tokens(kv_fp8, d) : 0);
}
__host__ __device__ constexpr int split_smem_bytes(int kv_fp8, int d) {
  // stages + derived per-token scale terms (fp8) + page ids + barriers/flags + alignment slack
  return kStages * stage_bytes(kv_fp8, d) + (kv_fp8 ? 16 * tile_tokens(kv_fp8, d) : 0) +
         4 * (kMaxChunk / kPage) + 64 + 1024;
}
// The tcgen05 kernel instance's N (q_len * group rows padded to 16, 32, 48 or 64).
inline int tc_rows_pad(int rows_max) { return rows_max <= 16 ? 16 : rows_max <= 32 ? 32 : rows_max <= 48 ? 48 : 64; }
// CTAs of the split kernel resident per SM (shared memory bound), used by the planner.
__host__ __device__ constexpr int split_ctas_per_sm(int warps) { return warps <= 4 ? 2 : 1; }

// Raises a kernel's dynamic shared-memory limit on the current device. The
// attribute belongs to one device, so it is set once per device ordinal
// (`done` holds one bit per ordinal below 64; higher ordinals set it on
// every launch). Setting it twice is harmless, so no lock is needed.
template <typename Kern>
inline cudaError_t ensure_smem_attr(Kern kern, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// A (sequence, KV head) pair split over several units, as the combine kernel
// sees it: its n partials sit at slots u0 .. u0 + n - 1, its q_len * G rows are
// rows row_base .. row_base + rows - 1 of the combine grid.
struct CombinePair {
  int32_t u0, n;      // first partial slot, partial count
  int32_t q_off;      // first token row of the sequence in q / out
  int32_t head0;      // first q head of the pair (kv head * G)
  int32_t rows;       // rows of the (virtual) pair: q_len * G, or one row half of it
  int32_t row0;       // first row of the pair's q_len * G rows that it covers (64 for a second row half)
  int32_t row_base;   // combine rows of the pairs before this one
};
constexpr int kMaxCombinePairs = 256;  // split pairs a table can list (else every row is covered)
// The combine's arguments for plans built from host lengths: only split rows.
struct CombineTable {
  const float* part_o;
  const float* part_lse;
  void* out;
  int32_t rows_max, num_q_heads, group, out_f32;
  int32_t n_pairs, num_rows;  // split pairs listed, their rows in all
  CombinePair pair[kMaxCombinePairs];
};

// The combine: over the split rows of `t` when given, else over every row of the plan's work table.
cudaError_t launch_combine(int head_dim, const SplitParams* p, const CombineTable* t, int max_splits, int sm_count,
                           cudaStream_t stream);

}  // namespace pav

typedef struct pa_verify_plan_s* pa_verify_plan_t;

namespace pav {

// pa_verify_run's checks and launches with caller-provided scratch, kernel
// parameters on the stack, nothing allocated (host or device).
int enqueue_with_scratch(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* context_lens, const int32_t* query_lens, float softmax_scale, void* out,
                         uint8_t* scratch, size_t scratch_bytes, cudaStream_t stream);
// Records `msg` as this thread's last error and returns `code`.
int report_error(int code, const char* msg);
// Device address of pa_verify_run_static's fixed scratch on the current device
// (looked up on first use per device).
int static_scratch_address(uint8_t** out);

}  // namespace pav
