// C ABI of the paged verify-attention library: planner, validation, launch.
//
// The planner follows the pages' split-decode structure: a decode kernel
// working over KV partitions plus a reducer, with the feasibility check done
// before any plan or scratch exists ("check feasibility first", MTP-5 routing
// page, review of base_attention.py) and a refusal instead of running outside
// the envelope. The partition count is chosen from the total context and the
// SM count so that one wave of CTAs covers the batch; a batch of one gets
// the ceiling of splits it can use (the page's dense-decode split test).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "pa_internal.h"
#include "../../include/pa_verify.h"

namespace pav {
cudaError_t launch_split_bf16(int head_dim, int warps, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                              const SplitParams* p, cudaStream_t stream);
cudaError_t launch_split_fp8(int head_dim, int warps, int units, const CUtensorMap* tmk, const CUtensorMap* tmv,
                             const SplitParams* p, cudaStream_t stream);
cudaError_t launch_dyn_plan(const int32_t* ctx, const int32_t* ql, DynWork* out, uint32_t* err, int flat, int num_seqs,
                            int num_q_heads, int num_kv_heads, int bt_stride, int max_len, int max_q, int slots, int tile,
                            int max_chunk, cudaStream_t stream);
cudaError_t launch_tc_split(int head_dim, int kv_fp8, int rows_max, int units, const CUtensorMap* tmk,
                            const CUtensorMap* tmv, const SplitParams* p, cudaStream_t stream);
cudaError_t launch_kv_write(int head_dim, int fp8, int n_tokens, int num_kv_heads, int num_pages, const void* k_new,
                            const void* v_new, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                            float* k_scale, float* v_scale, uint32_t* err, cudaStream_t stream);
size_t verdict_workspace_bytes(int num_tokens, int vocab);
cudaError_t launch_verdict(int num_seqs, int num_tokens, int vocab, const void* logits, const int32_t* input_ids,
                           const int32_t* query_lens, int32_t* target_ids, int32_t* accepted, int32_t* next_token,
                           void* workspace, cudaStream_t stream);
}  // namespace pav

using namespace pav;

struct pa_verify_plan_s {
  pa_verify_desc d;
  int32_t tile = 0, chunk = 0, units = 0, rows_max = 0, warps = 0, max_splits = 0, needs_combine = 0;
  int32_t num_tokens = 0, num_rows = 0;
  int32_t kernel = PA_KERNEL_WARP_MMA;
  int32_t n_entries = -1;        // entries of seq[] (-1: one per sequence of the batch)
  int32_t part_rows = 0;         // row stride of the partials (0: rows_max)
  int32_t slot_base = 0;         // first partial slot of this launch
  int32_t rows_split = 0;        // some entry has two row halves (SeqInfo::halves)
  int32_t batch_rows = 0;        // rows of the whole batch, when this plan covers part of it
  pa_verify_plan_s* second = nullptr;  // two-launch plans: the second launch (sequences with more rows)
  int32_t dynamic = 0;           // capacity plan: the work table is built on the device each run
  int32_t host_lengths = 0;      // a capacity plan made by pa_verify_plan (more than kMaxSeqs sequences)
  int32_t flat = 0, per = 0, total_tiles = 0;  // flat plans (tcgen05 kernel): tiles per CTA, tiles in all
  int32_t ranged = 0;            // flat plans: cta_start lists the CTAs' ranges
  int32_t cta_start[kMaxCtaTable + 1];
  int64_t part_units = 0;        // partial slots in the workspace
  // split pairs for the combine (plans built from host lengths; -1: more than the table holds, or none built)
  int32_t n_split_pairs = -1, split_rows = 0;
  int32_t combine_splits = 0;    // the split count the combine is sized for (see combine_width)
  CombinePair split_pairs[kMaxCombinePairs];
  int32_t max_len = 0, max_q = 0, slots = 0;
  size_t off_dyn = 0, off_part = kWsHeader, off_lse = kWsHeader;  // workspace layout
  int64_t kv_bytes = 0;
  size_t ws_bytes = 0;
  SeqInfo seq[kMaxSeqs];
  // tensor maps, re-encoded only when the cache pointers change
  const void* tm_k = nullptr;
  const void* tm_v = nullptr;
  CUtensorMap tmk, tmv;
  // measurement events (pa_verify_profile_enable)
  int profiling = 0;
  int profiled_runs = 0;
  int last_had_combine = 0;
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  // bounded-wait test hook (pa_verify_debug_stall)
  int32_t stall_cta = -1;
  uint64_t wait_limit_ns = 0;
};

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int encode_kv_map(CUtensorMap* map, const void* base, const pa_verify_desc& d) {
  auto enc = get_encoder();
  if (!enc) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int esz = d.kv_dtype == PA_KV_FP8_E4M3 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim),
                        static_cast<cuuint64_t>(d.num_pages) * d.num_kv_heads * kPage};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esz), static_cast<cuuint32_t>(kPage)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return PA_OK;
}

int supported_warps(int rows_max) {
  const int w = (rows_max + 15) / 16;
  return w <= 4 ? w : 8;
}

int check_run_args(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                   const float* k_scale, const float* v_scale, const int32_t* block_table,
                   const int32_t* context_lens, const int32_t* query_lens, float softmax_scale, const void* out) {
  const bool fp8 = plan->d.kv_dtype == PA_KV_FP8_E4M3;
  if (!q || !k_cache || !v_cache || !block_table || !context_lens || !query_lens || !out)
    return fail(PA_ERR_INVALID, "a required pointer is NULL");
  if (fp8 && (!k_scale || !v_scale)) return fail(PA_ERR_INVALID, "FP8 KV needs k_scale and v_scale");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
    return fail(PA_ERR_INVALID, "q, k_cache, v_cache and out must be 16-byte aligned");
  if (fp8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16)))
    return fail(PA_ERR_INVALID, "k_scale and v_scale must be 16-byte aligned");
  if (!aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(query_lens, 4))
    return fail(PA_ERR_INVALID, "int32 arrays must be 4-byte aligned");
  if (!(std::isfinite(softmax_scale) && softmax_scale > 0.f)) return fail(PA_ERR_INVALID, "softmax_scale must be finite and > 0");
  return PA_OK;
}

int encode_maps(pa_verify_plan_t plan, const void* k_cache, const void* v_cache) {
  if (plan->tm_k != k_cache) {
    int rc = encode_kv_map(&plan->tmk, k_cache, plan->d);
    if (rc) return rc;
    plan->tm_k = k_cache;
  }
  if (plan->tm_v != v_cache) {
    int rc = encode_kv_map(&plan->tmv, v_cache, plan->d);
    if (rc) return rc;
    plan->tm_v = v_cache;
  }
  return PA_OK;
}

// The fields that differ between the launches of a two-launch plan: its work table and CTA ranges.
void set_launch_fields(SplitParams& p, const pa_verify_plan_s* plan) {
  p.num_seqs = plan->n_entries >= 0 ? plan->n_entries : plan->d.num_seqs;
  p.chunk = plan->chunk;
  p.num_units = plan->units;
  p.flat = plan->flat;
  p.per = plan->per;
  p.total_tiles = plan->total_tiles;
  p.ranged = plan->ranged;
  if (plan->ranged) std::memcpy(p.cta_start, plan->cta_start, sizeof(int32_t) * (plan->units + 1));
  p.slot_base = plan->slot_base;
  p.rows_split = plan->rows_split;
  std::memcpy(p.seq, plan->seq, sizeof(plan->seq));
}

void fill_params(SplitParams& p, pa_verify_plan_t plan, const void* q, const float* k_scale, const float* v_scale,
                 const int32_t* block_table, const int32_t* context_lens, const int32_t* query_lens,
                 float softmax_scale, void* out, uint8_t* ws) {
  const pa_verify_desc& d = plan->d;
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  p.q = static_cast<const uint16_t*>(q);
  p.block_table = block_table;
  p.k_scale = fp8 ? k_scale : nullptr;
  p.v_scale = fp8 ? v_scale : nullptr;
  p.out = out;
  p.err = reinterpret_cast<uint32_t*>(ws);
  if (plan->needs_combine) {
    p.part_o = reinterpret_cast<float*>(ws + plan->off_part);
    p.part_lse = reinterpret_cast<float*>(ws + plan->off_lse);
  }
  p.dyn = plan->dynamic ? reinterpret_cast<const DynWork*>(ws + plan->off_dyn) : nullptr;
  p.dev_ctx = context_lens;
  p.dev_q = query_lens;
  p.num_q_heads = d.num_q_heads;
  p.num_kv_heads = d.num_kv_heads;
  p.group = d.num_q_heads / d.num_kv_heads;
  p.bt_stride = d.block_table_stride;
  p.num_pages = d.num_pages;
  p.rows_max = plan->part_rows > 0 ? plan->part_rows : plan->rows_max;
  p.out_f32 = d.out_dtype == PA_OUT_F32 ? 1 : 0;
  p.num_rows = plan->num_rows;
  p.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * 1.4426950408889634);
  p.wait_limit_ns = plan->wait_limit_ns;
  p.stall_cta = plan->stall_cta;
  set_launch_fields(p, plan);
}

// Enqueues (dynamic plans: the device planner, then) the split kernel and the
// combine; with `prof`, the plan's events bracket the two kernels.
cudaError_t launch_all(pa_verify_plan_t plan, SplitParams& p, cudaStream_t s, bool prof) {
  const pa_verify_desc& d = plan->d;
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  cudaError_t e = cudaSuccess;
  if (plan->dynamic)
    e = launch_dyn_plan(p.dev_ctx, p.dev_q, const_cast<DynWork*>(p.dyn), p.err, plan->flat, d.num_seqs, d.num_q_heads,
                        d.num_kv_heads, d.block_table_stride, plan->max_len, plan->max_q, plan->slots, plan->tile,
                        kMaxChunk, s);
  prof = prof && plan->profiling && plan->ev[0];
  if (e == cudaSuccess && prof) e = cudaEventRecord(plan->ev[0], s);
  if (e == cudaSuccess)
    e = plan->kernel == PA_KERNEL_TCGEN05
            ? launch_tc_split(d.head_dim, fp8 ? 1 : 0, plan->rows_max, plan->units, &plan->tmk, &plan->tmv, &p, s)
        : fp8 ? launch_split_fp8(d.head_dim, plan->warps, plan->units, &plan->tmk, &plan->tmv, &p, s)
              : launch_split_bf16(d.head_dim, plan->warps, plan->units, &plan->tmk, &plan->tmv, &p, s);
  if (e == cudaSuccess && plan->second) {
    // two-launch plan: the sequences with more rows, on their own instance, into the same workspace
    SplitParams p2 = p;
    set_launch_fields(p2, plan->second);
    e = launch_tc_split(d.head_dim, fp8 ? 1 : 0, plan->second->rows_max, plan->second->units, &plan->tmk, &plan->tmv,
                        &p2, s);
  }
  const bool combine = plan->needs_combine != 0;
  if (e == cudaSuccess && prof) e = cudaEventRecord(plan->ev[1], s);
  if (e == cudaSuccess && combine) {
    if (plan->n_split_pairs >= 0 && !plan->dynamic) {
      CombineTable t;
      t.part_o = p.part_o;
      t.part_lse = p.part_lse;
      t.out = p.out;
      t.rows_max = p.rows_max;
      t.num_q_heads = p.num_q_heads;
      t.group = p.group;
      t.out_f32 = p.out_f32;
      t.n_pairs = plan->n_split_pairs;
      t.num_rows = plan->split_rows;
      std::memcpy(t.pair, plan->split_pairs, sizeof(CombinePair) * plan->n_split_pairs);
      e = launch_combine(d.head_dim, &p, &t, plan->combine_splits, d.sm_count, s);
    } else {
      e = launch_combine(d.head_dim, &p, nullptr, plan->max_splits, d.sm_count, s);
    }
  }
  if (e == cudaSuccess && prof) {
    e = cudaEventRecord(plan->ev[2], s);
    plan->profiled_runs++;
    plan->last_had_combine = combine ? 1 : 0;
  }
  return e;
}

// The split count the combine's warps per row are sized for: the count that
// covers 90 % of the split rows (rows with more splits take further rounds of
// loads). Sized for the largest count instead, a batch whose pairs mostly split
// 3 ways but a few 30 ways ran every row with 4 warps (mixed FP8: combine
// 12.1 us under ncu; 90 %: calls 216.6 -> 212.0 us).
int32_t combine_width(const pa_verify_plan_s* P) {
  if (P->n_split_pairs <= 0) return P->max_splits;
  std::vector<std::pair<int32_t, int32_t>> nr;  // (splits, rows)
  int64_t tot = 0;
  for (int j = 0; j < P->n_split_pairs; ++j) {
    nr.emplace_back(P->split_pairs[j].n, P->split_pairs[j].rows);
    tot += P->split_pairs[j].rows;
  }
  std::sort(nr.begin(), nr.end());
  int64_t acc = 0;
  for (const auto& e : nr) {
    acc += e.second;
    if (acc * 10 >= tot * 9) return e.first;
  }
  return P->max_splits;
}

// Lists the split pairs of a plan built from host lengths for the combine's
// table (in plan order); n_split_pairs stays -1 when they do not fit it.
void list_split_pairs(pa_verify_plan_s* P, int hkv, int G, const std::vector<int32_t>& u0,
                      const std::vector<int32_t>& n, bool flat = false) {
  int32_t cnt = 0, rows = 0;
  bool fits = true;
  const int n_ent = P->n_entries >= 0 ? P->n_entries : P->d.num_seqs;
  for (int k = 0; k < n_ent && fits; ++k) {
    const SeqInfo& s = P->seq[k];
    const int hv = flat ? std::max(1, s.halves) : 1;
    for (int g = 0; g < hkv && fits; ++g)
      for (int h = 0; h < hv; ++h) {
        // (virtual) pair index: flat plans number them from the entry's first one
        const int pr = flat ? s.unit_start + g * hv + h : k * hkv + g;
        if (n[pr] <= 1) continue;
        if (cnt == kMaxCombinePairs) {
          fits = false;
          break;
        }
        CombinePair& c = P->split_pairs[cnt++];
        c.u0 = u0[pr];
        c.n = n[pr];
        c.q_off = s.q_off;
        c.head0 = g * G;
        c.rows = hv > 1 ? std::min(64, s.q_len * G - 64 * h) : s.q_len * G;
        c.row0 = 64 * h;
        c.row_base = rows;
        rows += c.rows;
      }
  }
  P->n_split_pairs = fits ? cnt : -1;
  P->split_rows = fits ? rows : 0;
  P->combine_splits = combine_width(P);
}

// Cost model of a CTA's range, in units of 1/32 of one of the instance's K/V
// tiles, fitted on GB300 to per-CTA run times (%globaltimer at entry and exit)
// of batches whose CTAs hold one to six segments, then checked by timing the
// split kernel under neighbouring tables:
// - A CTA that moves from one (sequence, KV head) pair to the next pays for the
//   switch: the outgoing pair's epilogue, the incoming pair's Q staging and the
//   exact maxima of its first tile, code that largely runs cold while HBM is
//   saturated. In tiles of the instance it grows with the rows (the epilogue's
//   rows, the columns of the maxima): about 2 tiles at 16 rows, 8 (head_dim 256)
//   to 10 (256-token FP8 tiles) at 48 and 13 to 20 at 64, where the instances
//   keep their per-column values in shared memory. (bf16 at head_dim 128: the
//   per-CTA fit gives 6 and 11 tiles at 48 and 64 rows, but the kernel times
//   best at 10 and 13. The 32-row entries and the head_dim-64 row are
//   interpolated or copied, not measured.)
// - A tile costs the same whatever the pair's rows, except in the 64-row
//   instances, which skip the P work of column chunks without rows: there a
//   tile of r rows costs about 1 + r / 320 tiles (a 64-row tile 1.2).
constexpr int64_t kCostUnit = 32;  // cost of one tile of a pair without rows
inline int64_t switch_cost(bool fp8, int head_dim, int np) {
  // half tiles, by N = 16, 32, 48, 64
  static constexpr int kBf16[3][4] = {{4, 10, 20, 26}, {4, 10, 20, 26}, {4, 6, 7, 14}};  // head_dim 64, 128, 256
  static constexpr int kFp8[2][4] = {{4, 11, 20, 26}, {4, 8, 16, 40}};                 // head_dim 128, 256
  const int n = np / 16 - 1, hd = head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2;
  const int half = fp8 ? kFp8[hd - 1][n] : kBf16[hd][n];
  return half * kCostUnit / 2;
}
inline int64_t tile_cost(int np, int rows) { return np == 64 ? kCostUnit + rows / 10 : kCostUnit; }

// Cuts the pairs' tiles (in flat order: pair sizes `nt`, tile costs `w`) into
// consecutive CTA ranges whose cost, the tiles' costs plus `sw` for every pair
// after the first, stays within `tau` (>= every tile cost); returns the CTA
// count and, with `starts`, each CTA's first tile followed by the total.
int64_t pack_ranges(const std::vector<int64_t>& nt, const std::vector<int64_t>& w, int64_t sw, int64_t tau,
                    std::vector<int32_t>* starts) {
  int64_t ctas = 0, load = 0, pos = 0;
  bool open = false;
  if (starts) starts->clear();
  for (size_t k = 0; k < nt.size(); ++k) {
    int64_t rem = nt[k];
    while (rem > 0) {
      if (!open) {
        if (starts) starts->push_back(static_cast<int32_t>(pos));
        open = true;
        load = 0;
      }
      const int64_t enter = load > 0 ? sw : 0;
      const int64_t room = tau - load - enter;
      if (room < w[k]) {  // no tile of this pair fits any more: the next CTA takes it
        ++ctas;
        open = false;
        continue;
      }
      const int64_t take = std::min(rem, room / w[k]);
      load += enter + take * w[k];
      rem -= take;
      pos += take;
    }
  }
  if (open) ++ctas;
  if (starts) starts->push_back(static_cast<int32_t>(pos));
  return ctas;
}

// Flat plan of the tcgen05 kernel: the (sequence, KV head) pairs laid end to
// end as the kernel's K/V tiles (tc_tile_tokens), longest sequences first, cut into one wave of
// consecutive CTA ranges. The cut minimises the largest CTA cost (tile costs
// plus a switch cost per pair switch, the model above): binary search on the
// cost bound, greedy filling at each bound. So long pairs are split evenly while short ones are
// packed whole, and a CTA crosses into the next pair only where that pays.
// (`split_override` = n asks for ceil(longest pair / n) tiles per CTA instead,
// and so do plans needing more CTAs than the range table holds.)
int plan_flat(pa_verify_plan_s* P, const pa_verify_desc& d, const int32_t* ctx, const int32_t* ql, int sms,
              pa_verify_plan_t* plan_out, size_t* workspace_bytes_out, const std::vector<char>* member = nullptr) {
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  const int G = d.num_q_heads / d.num_kv_heads, Hkv = d.num_kv_heads;
  // the sequences this plan covers (all, or those of `member`); q offsets stay the batch's
  std::vector<int> order;
  for (int b = 0; b < d.num_seqs; ++b)
    if (!member || (*member)[b]) order.push_back(b);
  const int n_ent = static_cast<int>(order.size());
  P->n_entries = n_ent;  // before anything walks the table (list_split_pairs)
  int rows_all = 0;
  for (int b : order) rows_all = std::max(rows_all, ql[b] * G);
  const int T = tc_tile_tokens(fp8 ? 1 : 0, d.head_dim, tc_rows_pad(rows_all));  // tokens per tile
  std::stable_sort(order.begin(), order.end(), [&](int a, int c) { return ctx[a] > ctx[c]; });
  std::vector<int32_t> q_off(d.num_seqs);
  int32_t acc = 0;
  for (int b = 0; b < d.num_seqs; ++b) {
    q_off[b] = acc;
    acc += ql[b];
  }
  int64_t tiles = 0, row = 0, work = 0, max_nt = 0, total_tokens = 0, vpairs = 0;
  int rows_max = 0;
  bool split_rows = false;
  for (int k = 0; k < n_ent; ++k) {
    const int b = order[k];
    SeqInfo& s = P->seq[k];
    s.ctx_len = ctx[b];
    s.q_len = ql[b];
    s.q_off = q_off[b];
    const int hv = s.q_len * G > 64 ? 2 : 1;  // row halves: pairs of more than 64 rows are two virtual pairs
    s.unit_start = static_cast<int32_t>(vpairs);
    s.row_start = static_cast<int32_t>(row);
    s.n_chunks = 0;
    s.b = b;
    s.tile_start = static_cast<int32_t>(std::min<int64_t>(tiles, INT32_MAX));
    s.n_tiles = (s.ctx_len + T - 1) / T;
    s.halves = hv;
    tiles += static_cast<int64_t>(s.n_tiles) * Hkv * hv;
    vpairs += static_cast<int64_t>(Hkv) * hv;
    split_rows = split_rows || hv > 1;
    row += static_cast<int64_t>(s.q_len) * d.num_q_heads;
    work += static_cast<int64_t>(s.ctx_len) * Hkv;
    max_nt = std::max<int64_t>(max_nt, s.n_tiles);
    rows_max = std::max(rows_max, s.q_len * G);
    total_tokens += s.q_len;
  }
  if (tiles >= (int64_t(1) << 31) || row >= (int64_t(1) << 31)) {
    delete P;
    return fail(PA_ERR_UNSUPPORTED, "work too large for one call");
  }
  int64_t per = d.split_override > 0 ? (max_nt + d.split_override - 1) / d.split_override : (tiles + sms - 1) / sms;
  per = std::max<int64_t>(per, 1);
  int64_t n_cta = (tiles + per - 1) / per;
  P->ranged = 0;
  if (d.split_override == 0 && tiles > 0) {
    const int np = tc_rows_pad(rows_max);  // the kernel instance's N
    const int64_t sw = switch_cost(fp8, d.head_dim, np);
    std::vector<int64_t> nt, w;
    int64_t total = 0, w_max = 0;
    for (int k = 0; k < n_ent; ++k)
      for (int g = 0; g < Hkv; ++g)
        for (int h = 0; h < P->seq[k].halves; ++h) {
          nt.push_back(P->seq[k].n_tiles);
          w.push_back(tile_cost(np, std::min(64, P->seq[k].q_len * G - 64 * h)));
          total += nt.back() * w.back();
          w_max = std::max(w_max, w.back());
        }
    // a bound of the whole cost always fits one CTA
    int64_t lo = std::max((total + sms - 1) / sms, w_max), hi = total + sw * static_cast<int64_t>(nt.size());
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (pack_ranges(nt, w, sw, mid, nullptr) <= sms) hi = mid; else lo = mid + 1;
    }
    std::vector<int32_t> starts;
    const int64_t n = pack_ranges(nt, w, sw, lo, &starts);
    if (n <= kMaxCtaTable) {
      P->ranged = 1;
      n_cta = n;
      std::copy(starts.begin(), starts.end(), P->cta_start);
      per = (lo + kCostUnit - 1) / kCostUnit;  // the cost bound in tiles, reported as the chunk
    }
  }
  // CTA holding tile f
  auto cta_of = [&](int64_t f) -> int64_t {
    if (!P->ranged) return f / per;
    return static_cast<int64_t>(std::upper_bound(P->cta_start, P->cta_start + n_cta + 1, static_cast<int32_t>(f)) -
                                P->cta_start) - 1;
  };
  int max_splits = 0;
  std::vector<int32_t> pu0(static_cast<size_t>(vpairs)), pn(pu0.size());
  for (int k = 0; k < n_ent; ++k)
    for (int g = 0; g < Hkv; ++g)
      for (int h = 0; h < P->seq[k].halves; ++h) {
        const int vp = g * P->seq[k].halves + h;  // virtual pair of the entry
        const int64_t t0 = P->seq[k].tile_start + static_cast<int64_t>(vp) * P->seq[k].n_tiles;
        const int64_t t1 = t0 + P->seq[k].n_tiles - 1;
        const int pr = P->seq[k].unit_start + vp;
        pn[pr] = static_cast<int32_t>(cta_of(t1) - cta_of(t0) + 1);
        pu0[pr] = static_cast<int32_t>(cta_of(t0) + pr);  // CTA c writes pair p's partial at slot c + p
        max_splits = std::max<int>(max_splits, pn[pr]);
      }
  list_split_pairs(P, Hkv, G, pu0, pn, true);
  P->kernel = PA_KERNEL_TCGEN05;
  P->flat = 1;
  P->tile = T;
  P->per = static_cast<int32_t>(per);
  P->total_tiles = static_cast<int32_t>(tiles);
  P->chunk = static_cast<int32_t>(std::min<int64_t>(per * T, INT32_MAX));
  P->units = static_cast<int32_t>(n_cta);
  P->rows_max = rows_max;
  P->warps = supported_warps(rows_max);
  P->max_splits = max_splits;
  P->needs_combine = max_splits > 1 ? 1 : 0;
  P->num_tokens = static_cast<int32_t>(total_tokens);
  P->num_rows = static_cast<int32_t>(row);
  P->part_units = n_cta + vpairs;  // slot c + p < CTAs + (virtual) pairs
  P->rows_split = split_rows ? 1 : 0;
  P->part_rows = split_rows ? 64 : 0;  // partials hold a virtual pair's rows
  P->kv_bytes = work * (fp8 ? (2 * d.head_dim + 8) : (4 * d.head_dim));
  size_t ws = kWsHeader;
  if (P->needs_combine) {
    P->off_part = ws;
    const int stride = split_rows ? 64 : rows_max;
    ws += align_up(static_cast<size_t>(P->part_units) * stride * d.head_dim * 4, 256);
    P->off_lse = ws;
    ws += align_up(static_cast<size_t>(P->part_units) * stride * 4, 256);
  }
  P->ws_bytes = ws;
  *plan_out = P;
  *workspace_bytes_out = ws;
  return PA_OK;
}

// Two-launch plan for a batch that mixes pairs of up to 48 rows with pairs of
// more (FP8 K/V at head_dim 128): each class gets its own flat plan and kernel
// instance (256-token tiles up to 48 rows, the 64-row instance above), launched
// one after the other into one workspace, followed by one combine over both.
// Measured on GB300 (the mixed FP8 batch, µs a call): one launch of the 64-row
// instance 230; the two classes alone 136 and 79, back to back about 215. The
// second launch's partial slots follow the first's; both use the larger row
// stride. Falls back to one launch when the merged combine table does not fit.
int plan_two_launch(pa_verify_plan_s* P, const pa_verify_desc& d, const int32_t* ctx, const int32_t* ql, int sms,
                    pa_verify_plan_t* plan_out, size_t* workspace_bytes_out) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const pa_verify_desc dd = P->d;
  std::vector<char> lo(d.num_seqs, 0), hi(d.num_seqs, 0);
  for (int b = 0; b < d.num_seqs; ++b) (ql[b] * G <= 48 ? lo : hi)[b] = 1;
  pa_verify_plan_s* B = new (std::nothrow) pa_verify_plan_s();
  if (!B) {
    delete P;
    return fail(PA_ERR_NOMEM, "out of host memory");
  }
  B->d = dd;
  pa_verify_plan_t pa = nullptr, pb = nullptr;
  size_t wa = 0, wb = 0;
  int rc = plan_flat(P, d, ctx, ql, sms, &pa, &wa, &lo);  // deletes P on failure
  if (rc != PA_OK) {
    delete B;
    return rc;
  }
  rc = plan_flat(B, d, ctx, ql, sms, &pb, &wb, &hi);
  if (rc != PA_OK) {
    delete P;
    return rc;
  }
  const bool comb = P->needs_combine || B->needs_combine;
  if (comb && (P->n_split_pairs < 0 || B->n_split_pairs < 0 ||
               P->n_split_pairs + B->n_split_pairs > kMaxCombinePairs)) {
    delete P;
    delete B;
    pa_verify_plan_s* S = new (std::nothrow) pa_verify_plan_s();
    if (!S) return fail(PA_ERR_NOMEM, "out of host memory");
    S->d = dd;
    return plan_flat(S, d, ctx, ql, sms, plan_out, workspace_bytes_out);
  }
  const int stride = std::max(P->part_rows > 0 ? P->part_rows : P->rows_max, B->part_rows > 0 ? B->part_rows : B->rows_max);
  B->slot_base = static_cast<int32_t>(P->part_units);
  const int64_t units_all = P->part_units + B->part_units;
  if (comb) {
    for (int j = 0; j < B->n_split_pairs; ++j) {
      CombinePair c = B->split_pairs[j];
      c.u0 += B->slot_base;
      c.row_base += P->split_rows;
      P->split_pairs[P->n_split_pairs++] = c;
    }
    P->split_rows += B->split_rows;
  }
  P->max_splits = std::max(P->max_splits, B->max_splits);
  P->combine_splits = combine_width(P);
  size_t ws = kWsHeader;
  if (comb) {
    P->off_part = ws;
    ws += align_up(static_cast<size_t>(units_all) * stride * d.head_dim * 4, 256);
    P->off_lse = ws;
    ws += align_up(static_cast<size_t>(units_all) * stride * 4, 256);
  }
  for (pa_verify_plan_s* X : {P, B}) {
    X->part_rows = stride;
    X->needs_combine = comb ? 1 : 0;
    X->off_part = P->off_part;
    X->off_lse = P->off_lse;
    X->ws_bytes = ws;
  }
  P->part_units = units_all;
  P->num_tokens += B->num_tokens;
  P->num_rows += B->num_rows;
  P->kv_bytes += B->kv_bytes;
  P->batch_rows = std::max(P->rows_max, B->rows_max);
  P->second = B;
  *plan_out = P;
  *workspace_bytes_out = ws;
  return PA_OK;
}

// Capacity plan: the work table is built on the device at every run from the
// device lengths (pa_dyn_plan.cu), for batches of up to `d.num_seqs` sequences
// with context lengths <= max_len and query lengths <= max_q. Serves
// pa_verify_plan_dynamic and host-length plans of more than kMaxSeqs
// sequences (whose table does not fit the kernel parameters).
int build_capacity_plan(const pa_verify_desc& d, int sms, int max_len, int max_q, bool use_tc,
                        pa_verify_plan_t* plan_out, size_t* workspace_bytes_out) {
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int rows_max = max_q * G;
  const int max_context_len = max_len, max_query_len = max_q;
  const int warps = supported_warps(rows_max);
  const int64_t slots = static_cast<int64_t>(sms) * (use_tc ? 1 : split_ctas_per_sm(warps));
  const int64_t per_pair = (static_cast<int64_t>(max_context_len) + kMaxChunk - 1) / kMaxChunk;
  const int64_t units_cap =
      use_tc ? slots : std::max<int64_t>(slots, static_cast<int64_t>(d.num_seqs) * d.num_kv_heads * per_pair);
  // partial slots: a flat plan's CTA c writes pair p's partial at c + p (a pair of more than 64 rows is two
  // virtual pairs, whose partials hold 64 rows each)
  const bool halves = use_tc && rows_max > 64;
  const int64_t part_cap =
      use_tc ? units_cap + static_cast<int64_t>(d.num_seqs) * d.num_kv_heads * (halves ? 2 : 1) : units_cap;
  const int stride = halves ? 64 : rows_max;  // rows of a partial
  const int64_t rows_cap = static_cast<int64_t>(d.num_seqs) * max_query_len * d.num_q_heads;
  if (units_cap >= (int64_t(1) << 31) || rows_cap >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "capacity too large for one call");

  pa_verify_plan_s* P = new (std::nothrow) pa_verify_plan_s();
  if (!P) return fail(PA_ERR_NOMEM, "out of host memory");
  P->d = d;
  P->d.sm_count = sms;
  P->dynamic = 1;
  P->max_len = max_context_len;
  P->max_q = max_query_len;
  P->slots = static_cast<int32_t>(slots);
  P->kernel = use_tc ? PA_KERNEL_TCGEN05 : PA_KERNEL_WARP_MMA;
  P->flat = use_tc ? 1 : 0;  // flat: one CTA per SM, the tiles per CTA chosen on the device
  P->tile = use_tc ? tc_tile_tokens(fp8 ? 1 : 0, d.head_dim, tc_rows_pad(rows_max)) : tile_tokens(fp8 ? 1 : 0, d.head_dim);
  P->chunk = 0;  // chosen on the device each run
  P->units = static_cast<int32_t>(units_cap);
  P->rows_max = rows_max;
  P->warps = warps;
  P->max_splits = static_cast<int32_t>(std::min<int64_t>(units_cap, (max_context_len + P->tile - 1) / P->tile));
  P->needs_combine = 1;
  P->num_tokens = d.num_seqs * max_query_len;
  P->num_rows = static_cast<int32_t>(rows_cap);
  const int64_t per_th = fp8 ? (2 * d.head_dim + 8) : (4 * d.head_dim);
  P->kv_bytes = static_cast<int64_t>(d.num_seqs) * max_context_len * d.num_kv_heads * per_th;  // at capacity
  P->part_units = part_cap;
  P->rows_split = halves ? 1 : 0;
  P->part_rows = halves ? 64 : 0;
  size_t ws = kWsHeader;
  P->off_dyn = ws;
  ws += align_up(dyn_work_bytes(d.num_seqs), 256);
  P->off_part = ws;
  ws += align_up(static_cast<size_t>(part_cap) * stride * d.head_dim * 4, 256);
  P->off_lse = ws;
  ws += align_up(static_cast<size_t>(part_cap) * stride * 4, 256);
  P->ws_bytes = ws;
  *plan_out = P;
  *workspace_bytes_out = ws;
  return PA_OK;
}

}  // namespace

extern "C" {

const char* pa_verify_last_error(void) { return g_last_error.c_str(); }

int pa_verify_plan(const pa_verify_desc* desc, const int32_t* context_lens_host, const int32_t* query_lens_host,
                   pa_verify_plan_t* plan_out, size_t* workspace_bytes_out) {
  g_last_error.clear();
  if (plan_out) *plan_out = nullptr;
  if (!desc || !plan_out || !workspace_bytes_out) return fail(PA_ERR_INVALID, "desc, plan_out and workspace_bytes_out must not be NULL");
  const pa_verify_desc& d = *desc;
  if (d.num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs < 0");
  if (d.num_seqs > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "num_seqs above " + std::to_string(kMaxBatch));
  if (d.num_seqs > kMaxSeqs && d.split_override > 0)
    return fail(PA_ERR_UNSUPPORTED, "split_override needs num_seqs <= " + std::to_string(kMaxSeqs));
  if (d.num_seqs > 0 && (!context_lens_host || !query_lens_host))
    return fail(PA_ERR_INVALID, "context_lens_host / query_lens_host must not be NULL");
  if (d.num_q_heads < 1 || d.num_kv_heads < 1 || d.num_q_heads % d.num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "need num_q_heads >= 1, num_kv_heads >= 1 and num_q_heads % num_kv_heads == 0");
  if (d.page_size != kPage) return fail(PA_ERR_UNSUPPORTED, "page_size must be 16");
  if (d.kv_dtype != PA_KV_BF16 && d.kv_dtype != PA_KV_FP8_E4M3) return fail(PA_ERR_INVALID, "unknown kv_dtype");
  if (d.out_dtype != PA_OUT_BF16 && d.out_dtype != PA_OUT_F32) return fail(PA_ERR_INVALID, "unknown out_dtype");
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  if (fp8 ? (d.head_dim != 128 && d.head_dim != 256) : (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256))
    return fail(PA_ERR_UNSUPPORTED, fp8 ? "FP8 KV needs head_dim 128 or 256" : "bf16 KV needs head_dim 64, 128 or 256");
  if (d.num_seqs > 0 && (d.num_pages < 1 || d.block_table_stride < 1))
    return fail(PA_ERR_INVALID, "num_pages and block_table_stride must be >= 1");
  if (static_cast<int64_t>(d.num_pages) * d.num_kv_heads * kPage >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_pages * num_kv_heads * 16 must stay below 2^31");
  if (d.split_override < 0 || d.sm_count < 0) return fail(PA_ERR_INVALID, "split_override and sm_count must be >= 0");
  if (d.kernel < PA_KERNEL_AUTO || d.kernel > PA_KERNEL_TCGEN05) return fail(PA_ERR_INVALID, "unknown kernel");

  const int G = d.num_q_heads / d.num_kv_heads;
  int rows_max = 0, max_len = 0, max_q = 0;
  int64_t total_tokens = 0, work = 0;
  for (int b = 0; b < d.num_seqs; ++b) {
    const int L = context_lens_host[b], q = query_lens_host[b];
    if (q < 1 || q > kMaxQueryLen) return fail(PA_ERR_INVALID, "query_lens must lie in 1..8 (sequence " + std::to_string(b) + ")");
    if (L < q) return fail(PA_ERR_INVALID, "context_len < query_len (sequence " + std::to_string(b) + ")");
    if ((static_cast<int64_t>(L) + kPage - 1) / kPage > d.block_table_stride)
      return fail(PA_ERR_INVALID, "context_len needs more pages than block_table_stride (sequence " + std::to_string(b) + ")");
    if (q * G > kMaxRows) return fail(PA_ERR_UNSUPPORTED, "query_len * group above 128 rows");
    rows_max = std::max(rows_max, q * G);
    max_len = std::max(max_len, L);
    max_q = std::max(max_q, q);
    total_tokens += q;
    work += static_cast<int64_t>(L) * d.num_kv_heads;
  }

  int sms = d.sm_count;
  if (sms == 0 && d.num_seqs > 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("SM count query failed: ") + cudaGetErrorString(e));
  }

  pa_verify_plan_s* P = new (std::nothrow) pa_verify_plan_s();
  if (!P) return fail(PA_ERR_NOMEM, "out of host memory");
  P->d = d;
  P->d.sm_count = sms;
  if (d.num_seqs == 0) {
    P->ws_bytes = kWsHeader;
    *plan_out = P;
    *workspace_bytes_out = P->ws_bytes;
    return PA_OK;
  }
  // Up to 64 rows a pair is one pass of the tcgen05 kernel; 65-128 rows are two row halves (virtual pairs).
  const bool tc_ok = d.head_dim >= 64 && rows_max <= 128;
  if (d.kernel == PA_KERNEL_TCGEN05 && !tc_ok) {
    delete P;
    return fail(PA_ERR_UNSUPPORTED, "the tcgen05 kernel needs q_len * group <= 128");
  }
  const bool use_tc = d.kernel == PA_KERNEL_TCGEN05 || (d.kernel == PA_KERNEL_AUTO && tc_ok);
  if (d.head_dim == 256 && !use_tc) {
    delete P;
    return fail(PA_ERR_UNSUPPORTED, "head_dim 256 runs on the tcgen05 kernel only");
  }
  if (d.num_seqs > kMaxSeqs) {
    // the table is too large for the kernel parameters: the device planner builds it at each run
    delete P;
    pa_verify_desc dd = d;
    dd.sm_count = sms;
    const int rc = build_capacity_plan(dd, sms, max_len, max_q, use_tc, plan_out, workspace_bytes_out);
    if (rc != PA_OK) return rc;
    pa_verify_plan_s* C = *plan_out;
    C->host_lengths = 1;
    C->num_tokens = static_cast<int32_t>(total_tokens);
    C->kv_bytes = work * (fp8 ? (2 * d.head_dim + 8) : (4 * d.head_dim));
    C->rows_max = rows_max;  // the plan's rows (the workspace was sized for max_q * G, the same)
    return PA_OK;
  }
  const int tile = use_tc ? 128 : tile_tokens(fp8 ? 1 : 0, d.head_dim);
  const int warps = supported_warps(rows_max);
  const int64_t slots = static_cast<int64_t>(sms) * (use_tc ? 1 : split_ctas_per_sm(warps));
  auto units_for = [&](int64_t c) {
    int64_t u = 0;
    for (int b = 0; b < d.num_seqs; ++b) u += (context_lens_host[b] + c - 1) / c;
    return u * d.num_kv_heads;
  };
  if (use_tc) {
    bool low = false, high = false;
    for (int b = 0; b < d.num_seqs; ++b) (query_lens_host[b] * G <= 48 ? low : high) = true;
    if (fp8 && d.head_dim == 128 && d.split_override == 0 && low && high)
      return plan_two_launch(P, d, context_lens_host, query_lens_host, sms, plan_out, workspace_bytes_out);
    return plan_flat(P, d, context_lens_host, query_lens_host, sms, plan_out, workspace_bytes_out);
  }
  const int64_t max_tile_len = align_up(static_cast<size_t>(max_len), static_cast<size_t>(tile));
  int64_t chunk;
  if (d.split_override > 0) {
    chunk = align_up(static_cast<size_t>((max_len + d.split_override - 1) / d.split_override), static_cast<size_t>(tile));
  } else {
    // one wave: the smallest tile multiple whose unit count fits the resident CTA slots
    chunk = align_up(static_cast<size_t>((work + slots - 1) / slots), static_cast<size_t>(tile));
    chunk = std::max<int64_t>(chunk, tile);
    while (chunk < max_tile_len && units_for(chunk) > slots) chunk += tile;
  }
  chunk = std::min<int64_t>(chunk, kMaxChunk);
  chunk = std::min<int64_t>(chunk, std::max<int64_t>(max_tile_len, tile));
  chunk = std::max<int64_t>(chunk, tile);

  // sequences by decreasing context length: long units are scheduled first
  std::vector<int> order(d.num_seqs);
  for (int b = 0; b < d.num_seqs; ++b) order[b] = b;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int c) { return context_lens_host[a] > context_lens_host[c]; });
  std::vector<int32_t> q_off(d.num_seqs);
  int32_t acc = 0;
  for (int b = 0; b < d.num_seqs; ++b) {
    q_off[b] = acc;
    acc += query_lens_host[b];
  }
  int64_t unit = 0, row = 0;
  int max_splits = 0;
  for (int k = 0; k < d.num_seqs; ++k) {
    const int b = order[k];
    SeqInfo& s = P->seq[k];
    s.ctx_len = context_lens_host[b];
    s.q_len = query_lens_host[b];
    s.q_off = q_off[b];
    s.unit_start = static_cast<int32_t>(unit);
    s.row_start = static_cast<int32_t>(row);
    s.n_chunks = static_cast<int32_t>((s.ctx_len + chunk - 1) / chunk);
    s.b = b;
    s.halves = 0;
    unit += static_cast<int64_t>(s.n_chunks) * d.num_kv_heads;
    row += static_cast<int64_t>(s.q_len) * d.num_q_heads;
    max_splits = std::max(max_splits, s.n_chunks);
  }
  if (unit >= (int64_t(1) << 31) || row >= (int64_t(1) << 31)) {
    delete P;
    return fail(PA_ERR_UNSUPPORTED, "work too large for one call");
  }
  {
    std::vector<int32_t> pu0(static_cast<size_t>(d.num_seqs) * d.num_kv_heads), pn(pu0.size());
    for (int k = 0; k < d.num_seqs; ++k)
      for (int g = 0; g < d.num_kv_heads; ++g) {
        const int pr = k * d.num_kv_heads + g;
        pn[pr] = P->seq[k].n_chunks;
        pu0[pr] = P->seq[k].unit_start + g * P->seq[k].n_chunks;  // units: KV head major, then chunk
      }
    list_split_pairs(P, d.num_kv_heads, G, pu0, pn);
  }
  P->kernel = use_tc ? PA_KERNEL_TCGEN05 : PA_KERNEL_WARP_MMA;
  P->tile = tile;
  P->chunk = static_cast<int32_t>(chunk);
  P->units = static_cast<int32_t>(unit);
  P->rows_max = rows_max;
  P->warps = warps;
  P->max_splits = max_splits;
  P->needs_combine = max_splits > 1 ? 1 : 0;
  P->num_tokens = static_cast<int32_t>(total_tokens);
  P->num_rows = static_cast<int32_t>(row);
  P->part_units = unit;
  const int64_t per_th = fp8 ? (2 * d.head_dim + 8) : (4 * d.head_dim);
  P->kv_bytes = work * per_th;
  size_t ws = kWsHeader;
  if (P->needs_combine) {
    P->off_part = ws;
    ws += align_up(static_cast<size_t>(unit) * rows_max * d.head_dim * 4, 256);
    P->off_lse = ws;
    ws += align_up(static_cast<size_t>(unit) * rows_max * 4, 256);
  }
  P->ws_bytes = ws;
  *plan_out = P;
  *workspace_bytes_out = ws;
  return PA_OK;
}

int pa_verify_plan_get_cta_starts(pa_verify_plan_t plan, int32_t* starts_out, int32_t capacity) {
  g_last_error.clear();
  if (!plan || !starts_out) return fail(PA_ERR_INVALID, "plan and starts_out must not be NULL");
  if (!plan->flat || plan->dynamic) return fail(PA_ERR_INVALID, "only static flat plans have CTA ranges");
  if (capacity < plan->units + 1) return fail(PA_ERR_INVALID, "capacity below num_units + 1");
  for (int32_t c = 0; c <= plan->units; ++c)
    starts_out[c] = plan->ranged ? plan->cta_start[c]
                                 : static_cast<int32_t>(std::min<int64_t>(static_cast<int64_t>(c) * plan->per, plan->total_tiles));
  return plan->units + 1;
}

int pa_verify_plan_get_info(pa_verify_plan_t plan, pa_verify_plan_info* info) {
  if (!plan || !info) return fail(PA_ERR_INVALID, "plan and info must not be NULL");
  info->num_units = plan->units + (plan->second ? plan->second->units : 0);
  info->chunk_tokens = plan->chunk;
  info->tile_tokens = plan->tile;
  info->rows_max = plan->batch_rows > 0 ? plan->batch_rows : plan->rows_max;
  info->warps = plan->warps;
  info->max_splits = plan->max_splits;
  info->needs_combine = plan->needs_combine;
  info->num_tokens = plan->num_tokens;
  info->kv_bytes = plan->kv_bytes;
  info->workspace_bytes = plan->ws_bytes;
  info->kernel = plan->kernel;
  info->dynamic = plan->dynamic && !plan->host_lengths;
  info->device_table = plan->dynamic;
  info->flat = plan->flat;
  info->total_tiles = plan->dynamic ? 0 : plan->total_tiles + (plan->second ? plan->second->total_tiles : 0);
  info->launches = plan->second ? 2 : 1;
  info->split_pairs = plan->dynamic ? -1 : plan->n_split_pairs;
  return PA_OK;
}

pa_verify_plan_t pa_verify_plan_get_second(pa_verify_plan_t plan) { return plan ? plan->second : nullptr; }

int pa_verify_run(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, const int32_t* block_table, const int32_t* context_lens,
                  const int32_t* query_lens, float softmax_scale, void* out, void* workspace, size_t workspace_bytes,
                  pa_stream_t stream) {
  g_last_error.clear();
  if (!plan) return fail(PA_ERR_INVALID, "plan must not be NULL");
  if (plan->d.num_seqs == 0) return PA_OK;
  int rc = check_run_args(plan, q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, query_lens,
                          softmax_scale, out);
  if (rc) return rc;
  if (!workspace) return fail(PA_ERR_INVALID, "a required pointer is NULL");
  if (!aligned(workspace, 256)) return fail(PA_ERR_INVALID, "workspace must be 256-byte aligned");
  if (workspace_bytes < plan->ws_bytes)
    return fail(PA_ERR_WORKSPACE, "workspace of " + std::to_string(workspace_bytes) + " bytes, plan needs " +
                                      std::to_string(plan->ws_bytes));
  rc = encode_maps(plan, k_cache, v_cache);
  if (rc) return rc;
  SplitParams p{};
  fill_params(p, plan, q, k_scale, v_scale, block_table, context_lens, query_lens, softmax_scale, out,
              static_cast<uint8_t*>(workspace));
  cudaError_t e = launch_all(plan, p, reinterpret_cast<cudaStream_t>(stream), true);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  return PA_OK;
}

}  // extern "C"

namespace pav {

// Enqueue for callers that bring their own scratch and cannot have anything
// allocated on their behalf: the same checks and launches as pa_verify_run,
// with the kernel parameters on the stack and no profiling events.
int enqueue_with_scratch(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* context_lens, const int32_t* query_lens, float softmax_scale, void* out,
                         uint8_t* scratch, size_t scratch_bytes, cudaStream_t s) {
  g_last_error.clear();
  if (!plan) return fail(PA_ERR_INVALID, "plan must not be NULL");
  if (plan->d.num_seqs == 0) return PA_OK;
  int rc = check_run_args(plan, q, k_cache, v_cache, k_scale, v_scale, block_table, context_lens, query_lens,
                          softmax_scale, out);
  if (rc) return rc;
  if (!scratch) return fail(PA_ERR_INVALID, "a required pointer is NULL");
  if (scratch_bytes < plan->ws_bytes)
    return fail(PA_ERR_WORKSPACE, "this plan needs " + std::to_string(plan->ws_bytes) +
                                      " bytes of scratch; the fixed scratch holds " + std::to_string(scratch_bytes));
  rc = encode_maps(plan, k_cache, v_cache);
  if (rc) return rc;
  SplitParams p{};
  fill_params(p, plan, q, k_scale, v_scale, block_table, context_lens, query_lens, softmax_scale, out, scratch);
  // the error word starts each call at zero (the scratch keeps the last call's contents)
  cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = launch_all(plan, p, s, false);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("kernel launch failed: ") + cudaGetErrorString(e));
  return PA_OK;
}

int report_error(int code, const char* msg) { return fail(code, msg); }

}  // namespace pav

extern "C" {

int pa_verify_profile_enable(pa_verify_plan_t plan, int enable) {
  g_last_error.clear();
  if (!plan) return fail(PA_ERR_INVALID, "plan must not be NULL");
  if (enable && !plan->ev[0]) {
    for (int k = 0; k < 3; ++k) {
      cudaError_t e = cudaEventCreate(&plan->ev[k]);
      if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("cudaEventCreate failed: ") + cudaGetErrorString(e));
    }
  }
  plan->profiling = enable ? 1 : 0;
  return PA_OK;
}

int pa_verify_profile_read(pa_verify_plan_t plan, float* split_ms, float* combine_ms) {
  g_last_error.clear();
  if (!plan || !split_ms || !combine_ms) return fail(PA_ERR_INVALID, "plan, split_ms and combine_ms must not be NULL");
  if (!plan->ev[0] || plan->profiled_runs == 0) return fail(PA_ERR_INVALID, "no profiled run recorded");
  cudaError_t e = cudaEventSynchronize(plan->ev[2]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(split_ms, plan->ev[0], plan->ev[1]);
  if (e == cudaSuccess) e = cudaEventElapsedTime(combine_ms, plan->ev[1], plan->ev[2]);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("reading profile events failed: ") + cudaGetErrorString(e));
  if (!plan->last_had_combine) *combine_ms = 0.f;
  return PA_OK;
}

int pa_kv_write(const pa_kv_write_desc* desc, const void* k_new, const void* v_new, const int64_t* slot_mapping,
                void* k_cache, void* v_cache, float* k_scale, float* v_scale, uint32_t* error_flags,
                pa_stream_t stream) {
  g_last_error.clear();
  if (!desc) return fail(PA_ERR_INVALID, "desc must not be NULL");
  const pa_kv_write_desc& d = *desc;
  if (d.num_tokens < 0 || d.num_kv_heads < 1 || d.num_pages < 0)
    return fail(PA_ERR_INVALID, "need num_tokens >= 0, num_kv_heads >= 1, num_pages >= 0");
  if (d.kv_dtype != PA_KV_BF16 && d.kv_dtype != PA_KV_FP8_E4M3) return fail(PA_ERR_INVALID, "unknown kv_dtype");
  if (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256)
    return fail(PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (static_cast<int64_t>(d.num_tokens) * d.num_kv_heads * 32 >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "too many tokens for one call");
  if (d.num_tokens == 0) return PA_OK;
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return fail(PA_ERR_INVALID, "a required pointer is NULL");
  if (fp8 && (!k_scale || !v_scale)) return fail(PA_ERR_INVALID, "FP8 KV needs k_scale and v_scale");
  if (!aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(k_cache, 4) || !aligned(v_cache, 4) ||
      !aligned(slot_mapping, 8))
    return fail(PA_ERR_INVALID, "k_new/v_new/caches must be 4-byte and slot_mapping 8-byte aligned");
  cudaError_t e = launch_kv_write(d.head_dim, fp8 ? 1 : 0, d.num_tokens, d.num_kv_heads, d.num_pages, k_new, v_new,
                                  slot_mapping, k_cache, v_cache, fp8 ? k_scale : nullptr, fp8 ? v_scale : nullptr,
                                  error_flags, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("kv write launch failed: ") + cudaGetErrorString(e));
  return PA_OK;
}

size_t pa_greedy_verdict_workspace_bytes(int32_t num_tokens, int32_t vocab) {
  if (num_tokens < 0 || vocab < 1) return 0;
  return verdict_workspace_bytes(num_tokens, vocab);
}

int pa_greedy_verdict(int32_t num_seqs, int32_t num_tokens, int32_t vocab, const void* logits,
                      const int32_t* input_ids, const int32_t* query_lens, int32_t* target_ids, int32_t* accepted,
                      int32_t* next_token, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  g_last_error.clear();
  if (num_seqs < 0 || num_tokens < 0 || vocab < 1) return fail(PA_ERR_INVALID, "need num_seqs >= 0, num_tokens >= 0, vocab >= 1");
  if (num_tokens < num_seqs || (num_seqs == 0) != (num_tokens == 0))
    return fail(PA_ERR_INVALID, "every sequence needs at least one verify position");
  if (static_cast<int64_t>(num_tokens) * ((vocab + 8191) / 8192) >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "logits too large for one call");
  if (num_seqs == 0) return PA_OK;
  if (!logits || !input_ids || !query_lens || !target_ids || !accepted || !next_token || !workspace)
    return fail(PA_ERR_INVALID, "a required pointer is NULL");
  if (!aligned(logits, 2) || !aligned(workspace, 256)) return fail(PA_ERR_INVALID, "logits must be 2-byte and workspace 256-byte aligned");
  if (workspace_bytes < verdict_workspace_bytes(num_tokens, vocab))
    return fail(PA_ERR_WORKSPACE, "workspace smaller than pa_greedy_verdict_workspace_bytes");
  cudaError_t e = launch_verdict(num_seqs, num_tokens, vocab, logits, input_ids, query_lens, target_ids, accepted,
                                 next_token, workspace, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("verdict launch failed: ") + cudaGetErrorString(e));
  return PA_OK;
}

int pa_verify_plan_dynamic(const pa_verify_desc* desc, int32_t max_context_len, int32_t max_query_len,
                           pa_verify_plan_t* plan_out, size_t* workspace_bytes_out) {
  g_last_error.clear();
  if (plan_out) *plan_out = nullptr;
  if (!desc || !plan_out || !workspace_bytes_out)
    return fail(PA_ERR_INVALID, "desc, plan_out and workspace_bytes_out must not be NULL");
  const pa_verify_desc& d = *desc;
  if (d.num_seqs < 1) return fail(PA_ERR_INVALID, "a dynamic plan needs num_seqs (the batch capacity) >= 1");
  if (d.num_seqs > kMaxBatch) return fail(PA_ERR_UNSUPPORTED, "num_seqs above " + std::to_string(kMaxBatch));
  if (d.num_q_heads < 1 || d.num_kv_heads < 1 || d.num_q_heads % d.num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "need num_q_heads >= 1, num_kv_heads >= 1 and num_q_heads % num_kv_heads == 0");
  if (d.page_size != kPage) return fail(PA_ERR_UNSUPPORTED, "page_size must be 16");
  if (d.kv_dtype != PA_KV_BF16 && d.kv_dtype != PA_KV_FP8_E4M3) return fail(PA_ERR_INVALID, "unknown kv_dtype");
  if (d.out_dtype != PA_OUT_BF16 && d.out_dtype != PA_OUT_F32) return fail(PA_ERR_INVALID, "unknown out_dtype");
  const bool fp8 = d.kv_dtype == PA_KV_FP8_E4M3;
  if (fp8 ? (d.head_dim != 128 && d.head_dim != 256) : (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256))
    return fail(PA_ERR_UNSUPPORTED, fp8 ? "FP8 KV needs head_dim 128 or 256" : "bf16 KV needs head_dim 64, 128 or 256");
  if (d.num_pages < 1 || d.block_table_stride < 1) return fail(PA_ERR_INVALID, "num_pages and block_table_stride must be >= 1");
  if (static_cast<int64_t>(d.num_pages) * d.num_kv_heads * kPage >= (int64_t(1) << 31))
    return fail(PA_ERR_UNSUPPORTED, "num_pages * num_kv_heads * 16 must stay below 2^31");
  if (d.split_override != 0) return fail(PA_ERR_INVALID, "split_override is not available for dynamic plans");
  if (d.sm_count < 0) return fail(PA_ERR_INVALID, "sm_count must be >= 0");
  if (d.kernel < PA_KERNEL_AUTO || d.kernel > PA_KERNEL_TCGEN05) return fail(PA_ERR_INVALID, "unknown kernel");
  if (max_query_len < 1 || max_query_len > kMaxQueryLen) return fail(PA_ERR_INVALID, "max_query_len must lie in 1..8");
  if (max_context_len < max_query_len) return fail(PA_ERR_INVALID, "max_context_len < max_query_len");
  if ((static_cast<int64_t>(max_context_len) + kPage - 1) / kPage > d.block_table_stride)
    return fail(PA_ERR_INVALID, "max_context_len needs more pages than block_table_stride");
  const int G = d.num_q_heads / d.num_kv_heads;
  const int rows_max = max_query_len * G;
  if (rows_max > kMaxRows) return fail(PA_ERR_UNSUPPORTED, "max_query_len * group above 128 rows");
  int sms = d.sm_count;
  if (sms == 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("SM count query failed: ") + cudaGetErrorString(e));
  }
  const bool tc_ok = d.head_dim >= 64 && rows_max <= 128;  // 65-128 rows: row halves (the device planner)
  if (d.kernel == PA_KERNEL_TCGEN05 && !tc_ok)
    return fail(PA_ERR_UNSUPPORTED, "the tcgen05 kernel needs q_len * group <= 128");
  const bool use_tc = d.kernel == PA_KERNEL_TCGEN05 || (d.kernel == PA_KERNEL_AUTO && tc_ok);
  if (d.head_dim == 256 && !use_tc)
    return fail(PA_ERR_UNSUPPORTED, "head_dim 256 runs on the tcgen05 kernel only");
  return build_capacity_plan(d, sms, max_context_len, max_query_len, use_tc, plan_out, workspace_bytes_out);
}

int pa_verify_debug_stall(pa_verify_plan_t plan, int32_t stall_cta, uint32_t wait_limit_us) {
  g_last_error.clear();
  if (!plan) return fail(PA_ERR_INVALID, "plan must not be NULL");
  if (stall_cta < -1) return fail(PA_ERR_INVALID, "stall_cta must be -1 (none) or a CTA index");
  plan->stall_cta = stall_cta;
  plan->wait_limit_ns = static_cast<uint64_t>(wait_limit_us) * 1000u;
  return PA_OK;
}

void pa_verify_free(pa_verify_plan_t plan) {
  if (!plan) return;
  for (auto& e : plan->ev)
    if (e) cudaEventDestroy(e);
  delete plan->second;
  delete plan;
}

int pa_verify_device_errors(void* workspace, uint32_t* flags_out, int clear, pa_stream_t stream) {
  g_last_error.clear();
  if (!flags_out) return fail(PA_ERR_INVALID, "flags_out must not be NULL");
  if (!workspace) {  // the fixed scratch of pa_verify_run_static on the current device
    uint8_t* scratch = nullptr;
    const int rc = static_scratch_address(&scratch);
    if (rc != PA_OK) return rc;
    workspace = scratch;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpy(flags_out, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(workspace, 0, sizeof(uint32_t));
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, std::string("reading the device error word failed: ") + cudaGetErrorString(e));
  return PA_OK;
}

}  // extern "C"
