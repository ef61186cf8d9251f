/*
 * pa_verify — paged-KV attention for speculative-decoding verify steps on one
 * GB300 GPU (sm_103a).
 *
 * The operation. Each sequence b of a batch brings q_b verify tokens
 * (1 <= q_b <= 8; 6 for an MTP-5 / DSpark-5 verify step, 4 for MTP-3, 1 for a
 * draft step). Those tokens are the last q_b tokens of the sequence's context of
 * L_b cached tokens. Query row (token i, q head h) attends, with softmax scale
 * `softmax_scale`, to keys 0 .. L_b - q_b + i of KV head h / (Hq / Hkv): the
 * whole context, causal inside the drafts. The GQA group times the query length
 * forms the rows that share one read of a KV head ("rows = query length x GQA
 * group", e.g. qlen 6 x group 8 = 48 rows: "fix(attention): keep MTP-5 decode
 * on FlyDSL pa_decode past the gluon query-length limit", Motivation). Keys and
 * values live in a pool of 16-token pages, head-major within a page
 * ("[MiniMax-M3.1] P/D from a PP4 prefill into a TP4 decode (2/2: DSpark)",
 * page-16 views, head-major per page), reached through a per-sequence block
 * table, and are bf16 or OCP FP8 E4M3 with per-token, per-head fp32 scales
 * (the MTP-5 page, Motivation and Tests: per-token FP8 KV scales with a
 * trailing singleton dimension).
 *
 * Calls. pa_verify_plan checks a batch description and its host-side lengths,
 * refuses anything outside the supported envelope before any allocation, and
 * picks the KV split (chunk length) from total context and SM count.
 * pa_verify_run enqueues the attention on a stream: a split-KV kernel and, when
 * some (sequence, KV head) was split, a log-sum-exp combine kernel.
 *
 * Conventions. All device pointers refer to memory of the current device.
 * The caller owns every buffer; the library keeps no device memory and no
 * pointer past a call. Nothing throws across this interface. Every function
 * returns a status (PA_OK = 0 or a negative PA_ERR_*) and, on failure, leaves
 * a message for pa_verify_last_error(). A refused call launches nothing and
 * writes nothing.
 */
#ifndef PA_VERIFY_H
#define PA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers. NULL = the legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

/* Opaque plan: host memory only, owned by the library until pa_verify_free. */
typedef struct pa_verify_plan_s* pa_verify_plan_t;

enum {
  PA_KV_BF16 = 0,     /* bf16 K/V */
  PA_KV_FP8_E4M3 = 1  /* OCP E4M3 (max finite 448) K/V with fp32 scales */
};

enum { PA_OUT_BF16 = 0, PA_OUT_F32 = 1 };

enum {
  PA_OK = 0,
  PA_ERR_INVALID = -1,     /* bad argument: null pointer, bad length, misalignment */
  PA_ERR_UNSUPPORTED = -2, /* valid but outside the envelope (head_dim, group, batch) */
  PA_ERR_WORKSPACE = -3,   /* workspace smaller than the plan needs */
  PA_ERR_CUDA = -4,        /* a CUDA call failed (launch, tensor-map encode, device query) */
  PA_ERR_NOMEM = -5        /* host allocation failed */
};

/* Bits of the device error word (pa_verify_device_errors). */
enum {
  PA_DEVERR_PAGE_RANGE = 1u,  /* a block-table entry outside [0, num_pages): zeros were read instead */
  PA_DEVERR_LENGTHS = 2u,     /* device context_lens/query_lens differ from the planned ones */
  PA_DEVERR_TIMEOUT = 4u      /* a bounded wait inside a kernel ran out; that CTA's output is invalid */
};

typedef struct {
  int32_t num_seqs;           /* B, 0 .. 1024 (dynamic plans: the capacity, 1 .. 1024) */
  int32_t num_q_heads;        /* Hq >= 1 */
  int32_t num_kv_heads;       /* Hkv >= 1, Hq % Hkv == 0, group G = Hq / Hkv */
  int32_t head_dim;           /* D: 64, 128 or 256 (bf16 KV); 128 or 256 (FP8 KV). 256 runs on the
                                 tcgen05 kernel only, within its envelope (see `kernel`; FP8: the
                                 aiter follow-up's head-256 shape on the MTP-5 routing page) */
  int32_t page_size;          /* must be 16 */
  int32_t kv_dtype;           /* PA_KV_* */
  int32_t out_dtype;          /* PA_OUT_* */
  int32_t num_pages;          /* pool size N_pg; block-table entries must lie in [0, N_pg) */
  int32_t block_table_stride; /* int32 entries per block-table row, >= ceil(L_b / 16) */
  int32_t split_override;     /* 0: the planner chooses; k > 0: chunk length
                                 ceil(max_b L_b / k) rounded up to the staging tile
                                 (num_seqs <= 64 only) */
  int32_t sm_count;           /* 0: query the current device; > 0: plan for that many SMs */
  int32_t kernel;             /* PA_KERNEL_*: 0 picks the tensor-core (tcgen05) kernel, which takes
                                 every head_dim and up to 128 rows (a pair of more than 64 rows runs
                                 as two row halves); the warp-MMA kernel (head_dim 64 or 128, up to
                                 128 rows) runs only when asked for */
} pa_verify_desc;

enum { PA_KERNEL_AUTO = 0, PA_KERNEL_WARP_MMA = 1, PA_KERNEL_TCGEN05 = 2 };

/*
 * Two plan kinds. Chunk plans (warp-MMA kernel): one CTA per (sequence, KV
 * head, chunk of chunk_tokens). Flat plans (tcgen05 kernel): the (sequence,
 * KV head) pairs laid end to end as tiles of tile_tokens and cut into one wave
 * of consecutive CTA ranges. A static plan picks the ranges that minimise the
 * largest CTA cost, counting tiles plus, for every move to another pair inside
 * a range, a switch cost measured per kernel instance (about 2 tiles at 16
 * rows, 5 to 10 at 48, 13 to 20 at 64); pa_verify_plan_get_cta_starts returns
 * them. With split_override, and in dynamic plans, every CTA gets the same
 * number of tiles (chunk_tokens / tile_tokens of them). Either way one wave
 * ends together whatever the length mix. A static FP8 plan at head_dim 128
 * whose batch mixes pairs of up to 48 rows with pairs of more makes two such
 * cuts, one per class, and runs them as two launches (info.launches).
 */
typedef struct {
  int32_t num_units;       /* CTAs of the split kernel: chunk plans sum_b Hkv * ceil(L_b / chunk),
                              flat plans the number of ranges (at most one per SM) */
  int32_t chunk_tokens;    /* chunk plans: context tokens per unit (a multiple of tile_tokens);
                              flat plans: tile_tokens x the largest range cost (in tiles, a
                              switch of pair counted at the instance's switch cost), or
                              tile_tokens x the tiles per CTA of an even cut; dynamic plans 0
                              (the device picks it each run) */
  int32_t tile_tokens;     /* tokens per shared-memory stage (flat plans: 256 for FP8 K/V at head_dim
                              128 with up to 48 rows, else 128) */
  int32_t rows_max;        /* max_b q_b * G */
  int32_t warps;           /* compute warps per CTA = ceil(rows_max / 16) (warp-MMA kernel) */
  int32_t max_splits;      /* most units one (sequence, KV head) is spread over */
  int32_t needs_combine;   /* 1 when some (sequence, KV head) has more than one unit */
  int32_t num_tokens;      /* T = sum_b q_b */
  int64_t kv_bytes;        /* algorithmic K/V(+scale) bytes one run reads */
  size_t workspace_bytes;  /* bytes pa_verify_run needs in `workspace` */
  int32_t kernel;          /* PA_KERNEL_WARP_MMA or PA_KERNEL_TCGEN05 */
  int32_t dynamic;         /* 1 for pa_verify_plan_dynamic plans (figures above are capacities) */
  int32_t flat;            /* 1 for flat plans */
  int32_t total_tiles;     /* flat plans: sum_b Hkv * ceil(L_b / tile_tokens) (dynamic plans: chosen per
                              run, 0 here) */
  int32_t device_table;    /* 1: each run builds the work table on the device from the device lengths
                              (a one-CTA planner kernel ahead of the split kernel): dynamic plans, and
                              plans of more than 64 sequences, whose table does not fit the kernel
                              parameters */
  int32_t launches;        /* split-kernel launches a run makes: 2 for a static FP8 head_dim-128 plan
                              whose batch mixes pairs of up to 48 rows with pairs of more (each
                              class on its own kernel instance, one combine after both); else 1.
                              num_units and total_tiles then count both launches; the rest of the
                              figures describe the first launch (pa_verify_plan_get_second) */
  int32_t split_pairs;     /* static plans: (sequence, KV head) pairs spread over more than one unit,
                              i.e. the pairs the combine merges, over both launches; -1 when they
                              are not listed (more than 256, or a device-built table) */
} pa_verify_plan_info;

/*
 * Checks the batch and builds a plan. The feasibility check comes first and a
 * batch outside the envelope is refused before any plan or scratch exists
 * (the MTP-5 routing page, review and Change: check feasibility before the
 * plan and scratch are built; raise instead of running outside the envelope);
 * the split of the context into partitions plus a reducer follows the split
 * decode the same page describes (Motivation). Reads context_lens_host[num_seqs] and
 * query_lens_host[num_seqs] (host memory, copied into the plan) and requires
 * 1 <= q_b <= 8, q_b <= L_b, ceil(L_b / 16) <= block_table_stride, and
 * (q_b * G) <= 128. On success *plan_out owns a host-side plan and
 * *workspace_bytes_out is the device workspace a run needs (0 is possible only
 * for an empty batch). On failure *plan_out is NULL; nothing is allocated and
 * no CUDA call is made (with sm_count > 0 the function makes no CUDA call at all).
 *
 * Up to 64 sequences the plan's work table travels in the kernel parameters.
 * From 65 to 1024 sequences (the pages' reducer is sized for batches up to
 * 1024: MTP-5 routing page, Motivation) it is the capacity plan of
 * pa_verify_plan_dynamic with capacity num_seqs and the batch's longest
 * lengths as bounds: each run builds the table on the device from the device
 * lengths, whose values must then lie within those bounds (a length outside
 * them sets PA_DEVERR_LENGTHS and that sequence writes nothing).
 */
int pa_verify_plan(const pa_verify_desc* desc, const int32_t* context_lens_host,
                   const int32_t* query_lens_host, pa_verify_plan_t* plan_out,
                   size_t* workspace_bytes_out);

/*
 * Capacity plan for CUDA-graph replay of padded batches: the lengths are read
 * on the device at every run, so one plan (and one captured graph) serves any
 * batch that fits. desc->num_seqs is the batch capacity (the capture width);
 * at run time sequence b may have query_lens[b] = 0 (a padded slot: no output
 * row, nothing written) or 1 <= query_lens[b] <= max_query_len with
 * query_lens[b] <= context_lens[b] <= max_context_len. Out-of-range lengths set
 * PA_DEVERR_LENGTHS and that sequence is treated as padding. q and out hold the
 * live sequences' rows packed in batch order, capacity num_seqs * max_query_len
 * rows. A run enqueues a one-CTA planner kernel (the split of the context and
 * the schedule, by the same rules as pa_verify_plan), the split kernel with a
 * grid sized for the capacity and the combine. Workspace is sized for the
 * capacity. split_override must be 0. Lengths and padding follow the pages'
 * CUDA-graph capture of fixed batch sizes and stores masked by row liveness
 * ("[DeepSeek-V4.1] High-interactivity monokernel decode", launch flags and
 * description).
 */
int pa_verify_plan_dynamic(const pa_verify_desc* desc, int32_t max_context_len, int32_t max_query_len,
                           pa_verify_plan_t* plan_out, size_t* workspace_bytes_out);

/* Copies the plan's figures into *info. */
int pa_verify_plan_get_info(pa_verify_plan_t plan, pa_verify_plan_info* info);

/*
 * A static flat plan's CTA ranges: starts_out[c] is CTA c's first tile and
 * starts_out[n] = the launch's tiles, n = its CTAs (tile t = tile_tokens
 * tokens of the t-th place in the flat order of (sequence, KV head) pairs).
 * Writes n + 1 values and returns that count; PA_ERR_INVALID for other plans
 * or when `capacity` is smaller. For a two-launch plan these are the first
 * launch's ranges (the second's: pa_verify_plan_get_second). Host only, no
 * CUDA call.
 */
int pa_verify_plan_get_cta_starts(pa_verify_plan_t plan, int32_t* starts_out, int32_t capacity);

/*
 * The second launch of a two-launch plan (info.launches == 2), NULL for
 * other plans. The handle is owned by `plan`: pass it only to
 * pa_verify_plan_get_info and pa_verify_plan_get_cta_starts (its figures
 * describe that launch alone), never to pa_verify_run or pa_verify_free.
 * Host only. No counterpart in the pages: it exposes the planner's split of
 * a mixed batch for tests and tuning.
 */
pa_verify_plan_t pa_verify_plan_get_second(pa_verify_plan_t plan);

/*
 * Enqueues verify attention on `stream` and returns without waiting: the split
 * kernel, then the combine kernel when some (sequence, KV head) is split
 * (dynamic plans: a one-CTA planner kernel first). The operation is the one
 * stated at the top of this header: query rows = query length x GQA group
 * over the paged context, with the block table and lengths handed to the
 * kernel and per-token FP8 scales (MTP-5 routing page, Motivation, Change and
 * Tests). Arguments are checked before anything is enqueued; a refused call
 * launches nothing (same page, review). No host-device copy, no
 * allocation, no synchronisation, so a fixed plan can be captured in a graph.
 *   q            [T, Hq, D] bf16, the q_b rows of each sequence packed in batch order
 *   k_cache      [N_pg, Hkv, 16, D] bf16 or E4M3 bytes, 16-byte aligned base
 *   v_cache      same layout as k_cache
 *   k_scale      [N_pg, Hkv, 16] fp32 (a trailing [.., 1] is the same memory),
 *                16-byte aligned; NULL for bf16 KV, required for FP8 KV
 *   v_scale      same as k_scale
 *   block_table  [B, block_table_stride] int32
 *   context_lens [B] int32, device; must hold the planned values (a mismatch
 *                sets PA_DEVERR_LENGTHS and leaves the output undefined)
 *   query_lens   [B] int32, device; same rule
 *   softmax_scale finite and > 0 (1/sqrt(D) is the usual choice)
 *   out          [T, Hq, D] bf16 or fp32 (desc.out_dtype); every element is written
 *   workspace    >= the planned workspace_bytes, 256-byte aligned; holds the
 *                split partials and the device error word. Zero it once after
 *                allocation; runs never clear the error word.
 * All device buffers must stay valid until the enqueued work completes. Two
 * runs that share a workspace must not overlap on the GPU.
 */
int pa_verify_run(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                  const float* k_scale, const float* v_scale, const int32_t* block_table,
                  const int32_t* context_lens, const int32_t* query_lens, float softmax_scale,
                  void* out, void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * Measurement hooks. After pa_verify_profile_enable(plan, 1), every
 * pa_verify_run with this plan records CUDA events (owned by the plan) on its
 * stream before the split kernel, between the kernels and after the combine.
 * pa_verify_profile_read waits for the last profiled run and returns the
 * device time of its split kernel and of its combine kernel (0 when there was
 * none), in milliseconds. Enabling creates the events (needs a device);
 * disabling keeps them until pa_verify_free.
 */
int pa_verify_profile_enable(pa_verify_plan_t plan, int enable);
int pa_verify_profile_read(pa_verify_plan_t plan, float* split_ms, float* combine_ms);

/*
 * pa_verify_run_static: pa_verify_run without a workspace argument, for
 * callers that cannot allocate device memory. Examples: a serving loop that
 * has reserved nearly all HBM for its KV cache up front, a host application
 * that owns every device allocation and gives plug-ins none, or code that must
 * not call cudaMalloc because it would synchronise the device or break a
 * memory-pool policy. (The pages this library follows have no counterpart.)
 *
 * The scratch this call needs (its device error word and the split partials)
 * is a single file-scope device array of PA_STATIC_SCRATCH_BYTES, which every
 * GPU that loads the library holds until the process exits. The first call on
 * a device looks up that array's device address there (cudaGetSymbolAddress,
 * with the device current); make that first call before any stream capture.
 * A plan that needs more scratch than the array holds is refused with
 * PA_ERR_WORKSPACE before anything is enqueued. The call allocates nothing and
 * calls neither cudaMalloc nor cudaFree. Every call shares the one array, which
 * keeps the last call's contents; the error word at its start is cleared on
 * the stream at the start of each call, and pa_verify_device_errors with a
 * NULL workspace reads it. Calls that overlap on the GPU (two streams, two
 * threads) race on the shared scratch: serialise them. Other arguments,
 * checks and return codes are those of pa_verify_run.
 */
#define PA_STATIC_SCRATCH_BYTES (16u << 20)
int pa_verify_run_static(pa_verify_plan_t plan, const void* q, const void* k_cache, const void* v_cache,
                         const float* k_scale, const float* v_scale, const int32_t* block_table,
                         const int32_t* context_lens, const int32_t* query_lens, float softmax_scale,
                         void* out, pa_stream_t stream);

/* Frees a plan (NULL is allowed). */
void pa_verify_free(pa_verify_plan_t plan);

/*
 * Test hook for the bounded waits of the tensor-core (tcgen05) kernel: every
 * wait of a run with this plan gives up after wait_limit_us microseconds
 * (0: the default of one second), and CTA stall_cta (-1: none) first waits on
 * a barrier that nothing completes, so that wait runs out. A wait that runs
 * out sets PA_DEVERR_TIMEOUT; the CTA then waits (bounded) for its copies and
 * MMAs in flight, frees its tensor memory and returns, and the output of its
 * work is invalid. Nothing faults or waits without a limit. Host only, no CUDA
 * call. (The pages have no counterpart; the MTP-5 routing page's rule of
 * raising instead of running outside the envelope is what the error word
 * reports.)
 */
int pa_verify_debug_stall(pa_verify_plan_t plan, int32_t stall_cta, uint32_t wait_limit_us);

/*
 * Reads the device error word of `workspace` (PA_DEVERR_* bits) after
 * synchronising `stream`; clears it when `clear` is non-zero. workspace = NULL
 * reads the fixed scratch of pa_verify_run_static on the current device (its
 * word is cleared at the start of every static call, so it holds the last
 * static call's flags).
 *
 * Workspace layout seen by callers: the first 256 bytes are a header. Its
 * 32-bit word 0 is the error word; word 1 counts, over all runs since the
 * workspace was zeroed, the tiles on which the tensor-core kernel raised a
 * row's running maximum inside a segment and rescaled the accumulated output
 * (a diagnostic of the online softmax; never cleared by runs).
 */
int pa_verify_device_errors(void* workspace, uint32_t* flags_out, int clear, pa_stream_t stream);

/*
 * Paged KV write (the step before verify attention): stores the K/V rows of
 * num_tokens new tokens into their cache slots, in place.
 *   k_new, v_new  [num_tokens, Hkv, D] bf16 (device), 4-byte aligned
 *   slot_mapping  [num_tokens] int64 (device): slot = page * 16 + offset in the
 *                 pool; -1 marks a padded or dead row, which writes nothing
 *                 (in-place stores masked by row liveness: "[DeepSeek-V4.1]
 *                 High-interactivity monokernel decode", description)
 *   k_cache, v_cache  [N_pg, Hkv, 16, D] bf16 (copied as is) or E4M3
 *   k_scale, v_scale  [N_pg, Hkv, 16] fp32, FP8 only (NULL for bf16)
 *   error_flags   optional device uint32: PA_DEVERR_PAGE_RANGE is or-ed in
 *                 when a slot lies outside the pool (that token is skipped)
 * FP8 quantisation per (token, head): s = amax / 448 (1 when amax = 0),
 * code = E4M3(x / s) with IEEE fp32 divisions, round to nearest even and
 * saturation at +-448 (OCP E4M3). head_dim 64, 128 or 256. Slots of one
 * call must be distinct. Asynchronous on `stream`; allocates nothing.
 */
typedef struct {
  int32_t num_tokens;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t kv_dtype;  /* PA_KV_* */
  int32_t num_pages;
} pa_kv_write_desc;

int pa_kv_write(const pa_kv_write_desc* desc, const void* k_new, const void* v_new,
                const int64_t* slot_mapping, void* k_cache, void* v_cache, float* k_scale,
                float* v_scale, uint32_t* error_flags, pa_stream_t stream);

/*
 * Greedy verify verdict (the step after verify attention): from the target
 * model's logits at the verify positions, the number of accepted drafts per
 * sequence and the next token ("ids + verdict" kept on the device:
 * "[DeepSeek-V4.1] High-interactivity monokernel decode", in-graph head).
 *   logits      [T, vocab] bf16 (device), rows packed by sequence like q
 *   input_ids   [T] int32 (device): per sequence the token fed at each verify
 *               position: the last committed token, then the q_b - 1 drafts
 *   query_lens  [num_seqs] int32 (device), 1 .. 32, summing to T
 *   target_ids  [T] int32 out: first index of each row's maximum (a NaN
 *               counts as the maximum; -0 equals +0)
 *   accepted    [num_seqs] int32 out: the longest prefix of drafts equal to
 *               the target's picks, 0 .. q_b - 1
 *   next_token  [num_seqs] int32 out: the target's pick after the accepted prefix
 *   workspace   >= pa_greedy_verdict_workspace_bytes(T, vocab), 256-byte
 *               aligned; its first word is a device error word (PA_DEVERR_LENGTHS
 *               when query_lens are out of range; pa_verify_device_errors reads it)
 * Asynchronous on `stream`; allocates nothing.
 */
size_t pa_greedy_verdict_workspace_bytes(int32_t num_tokens, int32_t vocab);
int pa_greedy_verdict(int32_t num_seqs, int32_t num_tokens, int32_t vocab, const void* logits,
                      const int32_t* input_ids, const int32_t* query_lens, int32_t* target_ids,
                      int32_t* accepted, int32_t* next_token, void* workspace, size_t workspace_bytes,
                      pa_stream_t stream);

/* Message for the last failing call on this thread ("" when none). */
const char* pa_verify_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_VERIFY_H */
