// Split-KV paged verify attention on 5th-generation tensor cores (tcgen05).
//
// Work. The (sequence, KV head) pairs are laid end to end as K/V tiles of 128
// tokens (256 in the FP8 head_dim-128 instances up to 48 rows: two MMA
// sub-tiles) and CTA c takes a consecutive range of them (the host planner's cost-bounded
// cut, or [c * per, (c + 1) * per)), so every SM gets about the same amount of
// K/V whatever the length mix. A CTA walks its range
// as segments, one per pair the range touches. A segment covering a whole
// pair writes the output; otherwise it writes a normalised partial and its
// log2-sum-exp at slot c + pair for the combine kernel (the "reducer" of a
// split decode: MTP-5 routing page, Motivation).
//
// A pair's q_b * G query rows ("rows = query length x GQA group", same page)
// are the N dimension of the MMAs, padded to NP (a pair of 65-128 rows runs
// as two row halves, virtual pairs of the 64-row instance); the 128 tokens of
// an MMA sub-tile are the M dimension, so every K/V byte reaches the tensor core
// straight from the TMA-staged shared memory, once:
//   S^T[tok, r]  = K[tok, :] . Q[r, :]           (A = K tile, K-major; B = Q, K-major)
//   O^T[d, r]   += V[:, d]^T . P^T[:, r]          (A = V tile, MN-major; B = P, MN-major)
// with both accumulators in tensor memory. head_dim 256 (FP8) runs PV as two
// M = 128 halves of the head dimension, one accumulator each.
//
// Warp roles (32 x (3 + 4 NWG) threads): warps 0 and V = 2 + 4 NWG gather pages through the block
// table with 2-D TMA boxes into a KS-deep K ring and a VS-deep V ring (the K
// producer also fills a ring of FP8 scales), one lane per box, reading page
// ids three tiles ahead; warp 1 allocates tensor memory and issues the MMAs
// (one thread); warps 2 .. V - 1 are NWG softmax warpgroups (three for 48 rows
// at head_dim 256, else two), one thread per token of the tile, each group owning NP / NWG row columns and
// staging its own rows of Q. Stages hand over on mbarriers; every wait is
// bounded. The rings run on across segment boundaries; Q is restaged once the
// last S of a segment is done.
//
// Softmax. Row r keeps a reference maximum M_r, uniform across its group. A
// tile whose scores stay below M_r + 8 (log2 units) uses M_r as is, so P <= 2^8
// and no cross-thread row maximum is needed. Otherwise (a segment's first
// tile, or a score that rose by more than 2^8) the warpgroup takes the exact
// tile row maxima, raises M_r and rescales l_r and the O accumulator. The final
// O / l is the same softmax whatever reference was used.
//
// FP8 E4M3 K/V stay 8-bit all the way (kind::f8f6f4). Q and P are each split
// into two E4M3 terms, x = hi + lo, and both terms go through the tensor core
// (Q's into the same accumulator; P's too at head_dim 128, while at 256 they
// are one operand of N = 64 + NP whose two column blocks are summed at the
// end): Q row r is scaled by a power of two 2^e_r first,
// and P (<= 2^8) has its mantissa cut to 3 bits for hi. The per-token scales
// are constant along the head dimension, so s_k multiplies score column t and
// log2 s_v enters the exponent, with l accumulating P / s_v.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

#include <type_traits>

namespace pav {

template <int KV_FP8, int NP, int D, int SUB = 1>
struct TcCfg {
  static constexpr int kD = D;
  // Tokens per K/V tile: SUB sub-tiles of 128 tokens (the MMA's M) a tile. With two (head_dim 128) every
  // softmax thread takes two tokens of a tile and S has two accumulators, so the hand-offs between the
  // roles, the softmax vote and the ring waits are paid once per 256 tokens.
  static constexpr int kSub = SUB;
  static constexpr int kTile = 128 * SUB;
  static constexpr int kRowB = KV_FP8 ? D : 2 * D;           // bytes per token row
  static constexpr int kHalves = kRowB / 128;                // 128-byte planes of a tile (TMA boxes per page)
  // PV M halves (one O accumulator each). head_dim 64 (bf16) keeps one M = 128 accumulator: its second
  // 64-row atom reads the 16 KB after the V slot (the next slot, or Q and P after the last one, always
  // inside the allocation), which fills only output rows d >= 64, never read.
  static constexpr int kMh = D >= 128 ? D / 128 : 1;
  // FP8 at head_dim 256: P's hi and lo planes form one B operand of N = 64 + NP (the lo plane is the operand's
  // second 64-column atom), so a PV k-step is one MMA; the accumulator then holds O_hi in columns [0, NP) and O_lo
  // from 64 on, and O = O_hi + O_lo. (One N = 112 MMA issues in about 61 clocks, two N = 48 ones in about 108.)
  // Measured on GB300: 139 -> 127 us at batch 8 x 150k; at head_dim 128, 2 us slower, so there the two planes
  // accumulate into the same columns by two MMAs.
  static constexpr bool kStackP = KV_FP8 != 0 && D == 256;
  static constexpr int kOCols = kStackP ? 128 : 64;          // tensor-memory columns of one O accumulator
  static constexpr int kSCols = 128 * SUB;                   // S: 2 buffers x SUB sub-tiles x 64 columns
  static constexpr int kTmemCols = kSCols + kMh * kOCols <= 256 ? 256 : 512;  // S, then the O accumulators
  static constexpr int kTileB = kTile * kRowB;               // 16 KB (fp8 D128) / 32 KB (bf16 D128, fp8 D256)
  // K ring depth (a K slot frees once S is done) and V ring depth (a V slot frees only after PV); bf16 at
  // head_dim 256 (64 KB tiles) has room for one stage of each next to Q (32 KB) and P
  static constexpr int KS = kTileB > 32768 ? 1 : kTileB > 16384 ? 2 : 5;
  static constexpr int VS = kTileB > 32768 ? 1 : kTileB > 16384 ? (KV_FP8 ? 2 : 3) : 5;
  static constexpr int kVStage = kTileB;                     // V data
  static constexpr int SS = KV_FP8 ? KS + 2 : 0;             // FP8 scale ring depth (see the K producer)
  static constexpr int kScB = 2 * 4 * kTile;                 // one slot: k then v scales of a tile's tokens
  static constexpr int kQPlane = 64 * 128;                   // one 128-byte-wide plane of 64 rows
  static constexpr int kQB = (KV_FP8 ? 2 : 1) * kHalves * kQPlane;  // bf16: 64-column halves; fp8: hi, lo by half
  static constexpr int kPPlane = KV_FP8 ? kTile * 64 : kTile * 128;  // bytes of one P plane
  static constexpr int kPBuf = KV_FP8 ? 2 * kPPlane : kPPlane;       // fp8: hi and lo planes
  static constexpr int PB = D > 128 ? 3 : 2;                 // P buffers (head_dim 256: PV takes twice the MMAs)
  // Softmax warpgroups: 48 rows at head_dim 256 take three groups of 16 columns (three warps per SM
  // sub-partition; 480 threads leave 136 registers a thread), elsewhere two. Measured on GB300: three
  // groups take 6 us off a batch-1 call at head_dim 256 and cost 2-4 us at larger batches and at 128.
  static constexpr int NWG = (NP == 48 && D == 256) ? 3 : 2;
  static constexpr int kThreads = 32 * (3 + 4 * NWG);
  static constexpr int kVWarp = 2 + 4 * NWG;                 // the V producer (after the softmax warps)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + KS * kTileB;
  static constexpr int kOffSc = kOffV + ((VS * kVStage + 1023) / 1024) * 1024;
  static constexpr int kOffQ = kOffSc + SS * kScB;
  static constexpr int kOffP = kOffQ + kQB;
  static constexpr int kOffRow = kOffP + PB * kPBuf;         // rowC[2][64] f32, rowLim[2][64] i32 (by segment parity)
  static constexpr int kOffRed = kOffRow + 4 * 64 * 4;       // tile maxima [4 NWG warps][64], 1 / row totals [64], reference maxima [64]
  static constexpr int kOffRedL = kOffRed + (4 * NWG + 2) * 64 * 4;  // row-sum partials [4 NWG warps][64]
  static constexpr int kOffBar = kOffRedL + 4 * NWG * 64 * 4;
  static constexpr int kSmem = kOffBar + 512 + 1024;         // barriers, tmem base, alignment slack
  static_assert(NP % 16 == 0 && NP >= 16 && NP <= 64, "N must be 16..64 in steps of 16");
  static_assert((NP / NWG) % 8 == 0 && NP % NWG == 0, "each softmax warpgroup owns a multiple of 8 columns");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
  static_assert(2 * KS + 2 * VS + 7 + 2 * PB + SS <= 62, "barriers fit their 512 bytes with the tmem slot and abort flag");
  static_assert(D == 128 || D == 256 || (!KV_FP8 && D == 64), "head_dim 128 or 256, or 64 with bf16 K/V");
  static_assert(D != 64 || kOffQ - kOffV - VS * kVStage + kQB + PB * kPBuf >= 16384,
                "head_dim 64: 16 KB of the allocation follow the last V slot");
};

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}
// OR of `pred` over the `nthreads` threads of named barrier `id`.
__device__ __forceinline__ bool named_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %3, 0;\n barrier.red.or.pred po, %1, %2, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}
// Maximum of v over the 32 lanes of the warp, in one instruction.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;\n" : "=f"(r) : "f"(v));
  return r;
}
// Two fp32 -> E4M3 bytes, round to nearest even, saturating (lo -> low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Position in a CTA's tile range: entry k of the work table (plan order), KV
// head g, row half h, tile t of the (virtual) pair, with the entry's figures.
// A pair of more than 64 rows is two virtual pairs, rows 0-63 and the rest,
// each a pass over the context (the two run side by side in neighbouring
// CTA ranges, so the second pass mostly finds the tiles in L2).
// RH: the instance can meet row halves (the 64-row one); elsewhere h stays 0 and costs nothing.
template <bool RH>
struct TileCursor {
  int k, g, h, t;
  int L, QL, q_off, b, n_t;
  __device__ __forceinline__ void load_seq(const WorkView& wv) {
    const SeqInfo& s = wv.seq[k];
    L = s.ctx_len;
    QL = s.q_len;
    q_off = s.q_off;
    b = s.b;
    n_t = s.n_tiles;
  }
  // the entry's row halves (read from the table where needed: registers are scarce in these instances)
  __device__ __forceinline__ int halves(const WorkView& wv) const { return RH ? max(1, wv.seq[k].halves) : 1; }
  __device__ __forceinline__ void seek(const WorkView& wv, int f) {
    k = flat_seq_of(wv, f);
    load_seq(wv);
    const int off = f - wv.seq[k].tile_start;
    const int vp = off / n_t, nh = halves(wv);
    g = vp / nh;
    h = vp - g * nh;
    t = off - vp * n_t;
  }
  // to the next tile; the caller guarantees the range has one
  __device__ __forceinline__ void advance(const WorkView& wv, int hkv) {
    if (++t < n_t) return;
    t = 0;
    if constexpr (RH) {
      if (++h < halves(wv)) return;
      h = 0;
    }
    if (++g < hkv) return;
    g = 0;
    ++k;
    load_seq(wv);
  }
  // index of the (virtual) pair: its partial slots and its place among the pairs
  __device__ __forceinline__ int pair(const WorkView& wv, int hkv, bool split) const {
    if constexpr (RH) {
      if (split) return wv.seq[k].unit_start + g * halves(wv) + h;
    }
    return k * hkv + g;
  }
  // rows of this virtual pair, and the first of the pair's q_len * G rows it covers
  __device__ __forceinline__ int rows(int G) const {
    if constexpr (RH) return min(64, QL * G - 64 * h);
    else return QL * G;
  }
  __device__ __forceinline__ int row0() const { return RH ? 64 * h : 0; }
};

template <int KV_FP8, int NP, int D, int SUB = 1>
__global__ void __launch_bounds__(TcCfg<KV_FP8, NP, D, SUB>::kThreads, 1)
    pa_tc_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const __grid_constant__ SplitParams p) {
  using C = TcCfg<KV_FP8, NP, D, SUB>;
  using Cursor = TileCursor<NP == 64>;  // row halves reach only the 64-row instances
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = sm + C::kOffK;
  uint8_t* sV = sm + C::kOffV;
  uint8_t* sQ = sm + C::kOffQ;
  uint8_t* sSc = sm + C::kOffSc;  // FP8 scale ring
  uint8_t* sP = sm + C::kOffP;
  float* rowC = reinterpret_cast<float*>(sm + C::kOffRow);     // [2][64] score multiplier per row
  int* rowLim = reinterpret_cast<int*>(rowC + 128);             // [2][64] last visible key per row (-1: padding)
  float* red = reinterpret_cast<float*>(sm + C::kOffRed);       // [4 NWG warps][64] maxima, [64] 1 / row totals, [64] M_r
  float* refM = red + (4 * C::NWG + 1) * 64;                    // reference maxima of the segment's rows (log2 units)
  float* redl = reinterpret_cast<float*>(sm + C::kOffRedL);     // [4 NWG warps][64] row-sum partials
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kOffBar);
  uint64_t* kfull = bars;
  uint64_t* kempty = kfull + C::KS;
  uint64_t* vfull = kempty + C::KS;
  uint64_t* vempty = vfull + C::VS;
  uint64_t* sfull = vempty + C::VS;
  uint64_t* sfree = sfull + 2;
  uint64_t* pfull = sfree + 2;
  uint64_t* pfree = pfull + C::PB;
  uint64_t* qready = pfree + C::PB;
  uint64_t* scfull = qready + 1;  // [SS] FP8 scale slots landed
  uint64_t* stall_bar = scfull + C::SS;  // never completed (the bounded-wait test hook waits on it)
  uint64_t* drain_bar = stall_bar + 1;   // the MMA issuer's last MMAs, after a failure
  uint32_t* tbase_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tbase_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ------------------------------------------------------------ the CTA's tiles
  const int cta = blockIdx.x;
  const WorkView wv = work_view(p);
  if (cta >= wv.num_units) return;  // a dynamic plan's grid covers its capacity
  const int f_lo = flat_cta_start(wv, cta);
  const int n_tiles = flat_cta_start(wv, cta + 1) - f_lo;
  const int Hkv = p.num_kv_heads, G = p.group;

  // Work that needs neither the barriers nor tensor memory starts before the
  // set-up, so that its memory reads are ahead of the rings' first TMA traffic:
  // the producers find their first tile and read its page ids, the softmax
  // warps find their first segment and load its Q rows.
  constexpr int NH = NP / C::NWG;               // columns per softmax warpgroup
  constexpr int kRowsPerWarp = NH / 4;          // Q rows each softmax warp stages
  const bool is_prod = warp == 0 || warp == C::kVWarp, is_sm = warp >= 2 && warp < C::kVWarp;
  const int wg = is_sm ? (warp - 2) >> 2 : 0;   // softmax warpgroup
  const int col0 = wg * NH;                     // first column this group owns
  // Column of the MMAs' N <-> row of the pair. In the 64-row instances (the ones that skip empty column
  // chunks) the rows are dealt to the softmax warpgroups in chunks of 8, round robin (row chunk m sits in
  // group m % NWG, as that group's chunk m / NWG), so a pair with fewer rows than N keeps every group about
  // equally busy; each group still owns NH consecutive columns. Elsewhere column = row (the mapping cost
  // the three-warpgroup instance registers).
  auto row_of_col = [](int col) {
    if constexpr (NP != 64) return col;
    const int w = col / NH, c = col - w * NH;
    return ((c >> 3) * C::NWG + w) * 8 + (c & 7);
  };
  constexpr int kHalves = C::kHalves;
  const bool is_k = warp == 0;
  // producer lanes: page (within the tile) of this lane's box, on lanes [0, pages * halves) (pages: none)
  constexpr int kTilePages = C::kTile / kPage;
  static_assert(kTilePages * kHalves <= 32, "one box per lane");
  const int jl = lane < kTilePages * kHalves ? lane / kHalves : kTilePages;
  constexpr int kSmArrive = 4 * C::NWG;         // softmax warps: arrivals on sfree, pfull and qready
  auto npages = [&](const Cursor& cq) {
    return min(C::kTile / kPage, (cq.L - cq.t * C::kTile + kPage - 1) / kPage);
  };
  // this lane's raw page id for a tile (-1: no copy); checked against the pool when issued
  auto fetch = [&](const Cursor& cq) {
    return jl < npages(cq) ? __ldg(p.block_table + static_cast<size_t>(cq.b) * p.bt_stride + cq.t * (C::kTile / kPage) + jl)
                           : -1;
  };
  // a softmax warp's Q rows of a segment: column col0 + (warp - 2) % 4 + 4 m, D / 32 bf16 per lane
  using QV = typename std::conditional<(D > 128), uint4, typename std::conditional<(D == 128), uint2, uint32_t>::type>::type;
  auto q_load = [&](const Cursor& cq, QV (&wq)[kRowsPerWarp]) {
    const int rows = cq.rows(G);
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) {
      const int r = row_of_col(col0 + ((warp - 2) & 3) + 4 * m);
      wq[m] = QV{};
      if (r < rows) {
        const int R = cq.row0() + r, i = R / G;  // row of the pair: query i, head g G + R - i G
        wq[m] = *reinterpret_cast<const QV*>(
            p.q + (static_cast<size_t>(cq.q_off + i) * p.num_q_heads + cq.g * G + (R - i * G)) * C::kD +
            (C::kD / 32) * lane);
      }
    }
  };
  Cursor cu0;  // producers: the first tile; softmax warps: the first segment
  Cursor cu1, cu2;  // producers: the next two tiles (their page ids are read ahead)
  int pg0 = -1, pg1 = -1, pg2 = -1;
  QV wq0[kRowsPerWarp];
  if (is_prod || is_sm) cu0.seek(wv, f_lo);
  if (is_prod) {
    pg0 = fetch(cu0);
    cu1 = cu0;
    cu2 = cu0;
    if (n_tiles > 1) {
      cu1.advance(wv, Hkv);
      pg1 = fetch(cu1);
      cu2 = cu1;
    }
    if (n_tiles > 2) {
      cu2.advance(wv, Hkv);
      pg2 = fetch(cu2);
    }
  }
  if (is_sm) q_load(cu0, wq0);

  if (tid == 0) {
    for (int s = 0; s < C::KS; ++s) { mbar_init(smem_addr(&kfull[s]), 1); mbar_init(smem_addr(&kempty[s]), 1); }
    for (int s = 0; s < C::VS; ++s) { mbar_init(smem_addr(&vfull[s]), 1); mbar_init(smem_addr(&vempty[s]), 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&sfull[s]), 1);
      mbar_init(smem_addr(&sfree[s]), kSmArrive);
    }
    for (int s = 0; s < C::PB; ++s) {
      mbar_init(smem_addr(&pfull[s]), kSmArrive);
      mbar_init(smem_addr(&pfree[s]), 1);
    }
    mbar_init(smem_addr(qready), kSmArrive);  // one phase per segment: each softmax warp staged its rows
    for (int s = 0; s < C::SS; ++s) mbar_init(smem_addr(&scfull[s]), 32);  // the K producer's 32 lanes (cp.async)
    mbar_init(smem_addr(stall_bar), 1);
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
  }
  if (warp == 1) {
    tc::tmem_alloc(tbase_slot, C::kTmemCols);
    tc::tmem_relinquish();
  }
  // Each warp reconverges first: lanes that took different paths must reach the
  // CTA barrier together, or it can release before thread 0's set-up is done.
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tbase_slot;
  const uint32_t tS[2] = {tmem, tmem + 64 * SUB};  // S buffer b, sub-tile h at tS[b] + 64 h
  const uint32_t tO = tmem + C::kSCols;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.err, 4u);
  };

  if (warp == 0 || warp == C::kVWarp) {
    // ============================================================ producers
    // Warp 0 feeds the K ring (and the FP8 scale ring), warp kVWarp the V ring.
    // A TMA issue costs its thread about one memory latency, so every page
    // box (and scale copy) of a tile gets its own lane: lane 0 arms the
    // stages' byte counts, then the lanes issue together.
    //
    // Scale slot k % SS is refilled without a wait of its own: issuing tile k
    // follows the end of S(k - KS) (the K slot's release), which the MMA
    // thread issued only after the softmax released S(k - KS - 2), and the
    // softmax reads a tile's scales before it releases the tile's S. So with
    // SS = KS + 2 the slot's previous tile, k - SS, has been read.
    const int depth = is_k ? C::KS : C::VS;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? kfull : vfull;
    uint64_t* empty = is_k ? kempty : vempty;
    // Page ids are read three tiles ahead (cursors cu, c1, c2 for tiles k, k+1, k+2, rotated by value):
    // a tile's issue is much shorter than a load from the block table, so reading only the next tile's
    // ids would hold the ring to about one tile per memory latency.
    Cursor cu = cu0, c1 = cu1, c2 = cu2;
    int pg_raw = pg0, p1 = pg1, p2 = pg2;
    int issued = 0;
    for (int k = 0; k < n_tiles; ++k) {
      Cursor c3 = c2;
      int p3 = -1;
      if (k + 3 < n_tiles) {
        c3.advance(wv, Hkv);
        p3 = fetch(c3);
      }

      // ring slot and phase of tile k, by the ring's compile-time depth (a division by a run-time depth
      // would put an integer-division sequence on the producer's path every tile)
      const int s = is_k ? k % C::KS : k % C::VS;
      const uint32_t ph = static_cast<uint32_t>(is_k ? k / C::KS : k / C::VS) & 1u;
      if (k >= depth) {
        // lane 0 checks the abort flag (another role failed) and waits for the slot; one verdict for the
        // whole warp, so no lane is left at a warp sync: 0 go on, 1 stop, 2 the wait ran out
        int st = 0;
        if (lane == 0)
          st = *abort_flag ? 1
                           : (mbar_wait_bounded(smem_addr(&empty[s]), ph ^ 1u, p.wait_limit_ns) ? 0 : 2);
        st = __shfl_sync(0xffffffffu, st, 0);
        if (st != 0) {
          if (st == 2 && lane == 0) fail();
          break;
        }
      }
      uint8_t* dst = is_k ? sK + s * C::kTileB : sV + s * C::kVStage;
      const uint32_t bar = smem_addr(&full[s]);
      const int npg = npages(cu);
      // an id outside the pool is flagged and read past the tensor's end, where TMA fills zeros
      int pg = pg_raw;
      if (jl < npg && static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages)) {
        atomicOr(p.err, 1u);
        pg = -1;
      }
      const int sslot = k % (C::SS > 0 ? C::SS : 1);  // scale slot (FP8)
      if (lane == 0) mbar_arrive_expect_tx(bar, npg * (kPage * C::kRowB));
      __syncwarp();
      if (lane < npg * kHalves) {
        const int hf = lane % kHalves;
        // an id outside the pool reads past the tensor's end: TMA fills zeros
        const int row = (pg >= 0 ? pg : p.num_pages) * Hkv * kPage + cu.g * kPage;
        tma_load_2d(smem_addr(dst + hf * (C::kTile * 128) + jl * kPage * 128), map, bar, hf * (KV_FP8 ? 128 : 64), row);
      }
      if constexpr (KV_FP8) {
        if (is_k) {
          // The tile's per-token scales (64 bytes of k and 64 of v a page) by 16-byte cp.async through the
          // load/store path: the lanes split the pages' 128 bytes evenly (128-token tiles: lane l takes
          // page l / 4, 32 bytes; 256-token tiles: page l / 2, 64 bytes), k bytes first. (As TMA copies
          // they doubled the TMA requests of a tile.) Every lane then arrives on the slot's barrier once
          // its copies have landed.
          constexpr int kLanesPage = 32 / kTilePages, kLaneBytes = 128 / kLanesPage;
          const int sp = lane / kLanesPage;
          const int spg = __shfl_sync(0xffffffffu, pg, sp * kHalves);  // page id (after the pool check)
          if (sp < npg && spg >= 0) {
            const int ob = (lane % kLanesPage) * kLaneBytes;  // byte of [k scales | v scales] of the page
            const bool vsc = ob >= 64;
            const int part = (ob & 63) / 4;  // floats
            const float* src = (vsc ? p.v_scale : p.k_scale) + (static_cast<size_t>(spg) * Hkv + cu.g) * kPage + part;
            const uint32_t dst = smem_addr(sSc + sslot * C::kScB + (vsc ? C::kTile * 4 : 0) + sp * kPage * 4 + part * 4);
#pragma unroll
            for (int cpy = 0; cpy < kLaneBytes / 16; ++cpy) cp_async_16(dst + 16 * cpy, src + 4 * cpy);
          }
          cp_async_mbar_arrive(smem_addr(&scfull[sslot]));
        }
      }
      // (after the issue, off its path) the device lengths must be the planned ones
      if (is_k && lane == 0 && cu.t == 0 && cu.g == 0 && (p.dev_ctx[cu.b] != cu.L || p.dev_q[cu.b] != cu.QL))
        atomicOr(p.err, 2u);
      ++issued;
      cu = c1;
      c1 = c2;
      c2 = c3;
      pg_raw = p1;
      p1 = p2;
      p2 = p3;
    }
    // No copy may land after the CTA exits: wait (bounded) for the last
    // copies of each ring slot; only this warp arms these barriers, so the
    // parity of tile k's phase is exact.
    if (lane == 0) {
      for (int k = max(0, issued - depth); k < issued; ++k)
        (void)mbar_wait_bounded(smem_addr(&full[k % depth]), static_cast<uint32_t>(k / depth) & 1u, p.wait_limit_ns);
      if constexpr (KV_FP8) {
        if (is_k)
          for (int k = max(0, issued - C::SS); k < issued; ++k)
            (void)mbar_wait_bounded(smem_addr(&scfull[k % C::SS]), static_cast<uint32_t>(k / C::SS) & 1u, p.wait_limit_ns);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    // One thread issues S^T = K Q^T of tile i and O^T += V^T P^T of tile j in
    // the fixed order S0 S1 | S2 PV0 | S3 PV1 | ...: S(j+2) needs only that the
    // softmax has read S(j) (early in its tile) while PV(j) needs its finished
    // P, so each wait is on the event due first and the thread sleeps in
    // hardware (try_wait) instead of polling. A segment's first S needs that
    // segment's Q, staged by the softmax at the start of the previous tile,
    // after the segment before it may have waited for PV(j) in its epilogue:
    // such an S goes after PV(j) instead.
    if (lane == 0) {
      constexpr uint32_t fa = KV_FP8 ? tc::kE4M3 : tc::kBF16;
      constexpr uint32_t idS = tc::idesc(fa, fa, tc::kKMajor, tc::kKMajor, 128, NP);
      constexpr uint32_t idPV = tc::idesc(fa, fa, tc::kMNMajor, tc::kMNMajor, 128, C::kStackP ? 64 + NP : NP);
      const uint32_t aK = smem_addr(sK), aV = smem_addr(sV), aP = smem_addr(sP);
      // Each MMA's operand descriptors are its stage's base descriptor plus a constant (one add): the issue
      // cost of a thread per MMA is then close to the tensor core's own time for these small N.
      const uint64_t dQ = tc::sdesc(smem_addr(sQ), 16, 1024, tc::kSwizzle128B);
      Cursor cs, cv;  // the next S tile, the next PV tile
      cs.seek(wv, f_lo);
      cv = cs;
      int seg_s = 0;      // segment of the next S tile
      auto issue_s = [&](int i) -> bool {
        const int ks_ = i % C::KS, sb = i & 1;
        if (i > 0 && cs.t == 0) ++seg_s;
        if ((i == 0 || cs.t == 0) && !mbar_wait_bounded(smem_addr(qready), static_cast<uint32_t>(seg_s) & 1u, p.wait_limit_ns))
          return false;
        if (!mbar_wait_bounded(smem_addr(&kfull[ks_]), static_cast<uint32_t>(i / C::KS) & 1u, p.wait_limit_ns)) return false;
        if (i >= 2 && !mbar_wait_bounded(smem_addr(&sfree[sb]), static_cast<uint32_t>((i >> 1) - 1) & 1u, p.wait_limit_ns))
          return false;
        tc::fence_after_sync();
        const uint64_t dK = tc::sdesc(aK + ks_ * C::kTileB, 16, 1024, tc::kSwizzle128B);
        // sub-tile h: tokens [128 h, 128 h + 128) of the tile, 16 KB further into each plane
#pragma unroll
        for (int h = 0; h < SUB; ++h) {
          if (KV_FP8) {
#pragma unroll
            for (int pl = 0; pl < 2; ++pl)  // Q hi then Q lo
#pragma unroll
              for (int hf = 0; hf < kHalves; ++hf)  // 128 head-dim entries per plane
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  tc::mma_f8(tS[sb] + 64 * h, tc::desc_plus(dK, hf * (C::kTile * 128) + h * 16384 + ks * 32),
                             tc::desc_plus(dQ, (pl * kHalves + hf) * C::kQPlane + ks * 32), idS,
                             (pl > 0 || hf > 0 || ks > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int ks = 0; ks < 4 * kHalves; ++ks)  // 16 head-dim entries a k-step, 4 per 128-byte plane
              tc::mma_f16(tS[sb] + 64 * h,
                          tc::desc_plus(dK, (ks >> 2) * (C::kTile * 128) + h * 16384 + (ks & 3) * 32),
                          tc::desc_plus(dQ, (ks >> 2) * C::kQPlane + (ks & 3) * 32), idS, ks > 0 ? 1u : 0u);
          }
        }
        tc::commit(&sfull[sb]);
        tc::commit(&kempty[ks_]);
        if (i + 1 < n_tiles) cs.advance(wv, Hkv);
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        const int vs = j % C::VS, pb = j % C::PB;
        const bool first = j == 0 || cv.t == 0;  // the segment's first PV starts its accumulator
        if (!mbar_wait_bounded(smem_addr(&vfull[vs]), static_cast<uint32_t>(j / C::VS) & 1u, p.wait_limit_ns)) return false;
        if (!mbar_wait_bounded(smem_addr(&pfull[pb]), static_cast<uint32_t>(j / C::PB) & 1u, p.wait_limit_ns)) return false;
        tc::fence_after_sync();
        const uint32_t v0 = aV + vs * C::kVStage;
        const uint32_t p0 = aP + pb * C::kPBuf;
        // only the k-steps holding tokens of the pair: rows past them may be stale or never loaded
        const int nv = min(C::kTile, cv.L - cv.t * C::kTile);
        if (KV_FP8) {
          const int nks = (nv + 31) >> 5;  // 32 tokens per k-step
          const uint64_t dV = tc::sdesc(v0, 16384, 1024, tc::kSwizzle128B);
          if constexpr (C::kStackP) {
            // P: hi plane = the operand's first 64 columns, lo plane (kPPlane further on) the next ones
            const uint64_t dP = tc::sdesc(p0, C::kPPlane, 512, tc::kSwizzle64B);
#pragma unroll
            for (int h = 0; h < C::kMh; ++h)  // head-dim entries [128 h, 128 h + 128): V plane h, O accumulator h
#pragma unroll
              for (int ks = 0; ks < C::kTile / 32; ++ks)
                if (ks < nks)
                  tc::mma_f8(tO + C::kOCols * h, tc::desc_plus(dV, h * (C::kTile * 128) + ks * 4096),
                             tc::desc_plus(dP, ks * 2048), idPV, (!first || ks > 0) ? 1u : 0u);
          } else {
            const uint64_t dP = tc::sdesc(p0, 16384, 512, tc::kSwizzle64B);
#pragma unroll
            for (int h = 0; h < C::kMh; ++h)
#pragma unroll
              for (int pl = 0; pl < 2; ++pl)  // hi then lo plane of P, into the same columns
#pragma unroll
                for (int ks = 0; ks < C::kTile / 32; ++ks)
                  if (ks < nks)
                    tc::mma_f8(tO + C::kOCols * h, tc::desc_plus(dV, h * (C::kTile * 128) + ks * 4096),
                               tc::desc_plus(dP, pl * C::kPPlane + ks * 2048), idPV,
                               (!first || pl > 0 || ks > 0) ? 1u : 0u);
          }
        } else {
          const int nks = (nv + 15) >> 4;  // 16 tokens per k-step
          const uint64_t dV = tc::sdesc(v0, C::kTile * 128, 1024, tc::kSwizzle128B);
          const uint64_t dP = tc::sdesc(p0, 16384, 1024, tc::kSwizzle128B);
#pragma unroll
          for (int h = 0; h < C::kMh; ++h)  // head-dim entries [128 h, 128 h + 128): V planes 2h, 2h + 1
#pragma unroll
            for (int ks = 0; ks < C::kTile / 16; ++ks)
              if (ks < nks)
                tc::mma_f16(tO + C::kOCols * h, tc::desc_plus(dV, 2 * h * (C::kTile * 128) + ks * 2048),
                            tc::desc_plus(dP, ks * 2048), idPV, (!first || ks > 0) ? 1u : 0u);
        }
        tc::commit(&vempty[vs]);
        tc::commit(&pfree[pb]);  // also tells the softmax warpgroups that O holds the segment's tiles up to j
        if (j + 1 < n_tiles) cv.advance(wv, Hkv);
        return true;
      };
      // test hook: a wait on a barrier that nothing completes runs out, and the CTA takes its failure path
      bool ok = cta != p.stall_cta || mbar_wait_bounded(smem_addr(stall_bar), 0u, p.wait_limit_ns);
      for (int i = 0; ok && i < min(2, n_tiles); ++i) ok = issue_s(i);
      for (int j = 0; ok && j < n_tiles && !*abort_flag; ++j) {
        const bool s_next = j + 2 < n_tiles;
        const bool s_new_seg = s_next && cs.t == 0;  // cs stands at tile j + 2
        if (s_next && !s_new_seg) ok = issue_s(j + 2);
        if (ok) ok = issue_pv(j);
        if (ok && s_new_seg) ok = issue_s(j + 2);
      }
      if (!ok) fail();
      // After a failure (here or in another role) MMAs already issued may still be running: wait (bounded)
      // for every one of them before tensor memory is freed. (On the normal path they are done already.)
      tc::commit(drain_bar);
      (void)mbar_wait_bounded(smem_addr(drain_bar), 0u, p.wait_limit_ns);
    }
  } else if (is_sm) {
    // ============================================================ softmax warpgroups
    // NWG warpgroups (warps 2-5, 6-9, 10-13). Each covers the 128 tokens of an MMA
    // sub-tile (one per thread, = tensor-memory lane; a thread takes its token of
    // every sub-tile of the tile) for its own NH = NP / NWG columns (rows of the
    // pair); the groups never wait on each other inside the loop.
    const int gt = tid - 64 - wg * 128;           // 0..127 inside the group
    const int q4 = warp & 3;                      // tensor-memory lane quarter of this warp
    const int tok = q4 * 32 + lane;               // token of the tile this thread owns
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int bar_sync = 1 + 2 * wg, bar_or = 2 + 2 * wg;

    // ---- Q rows of columns [col0, col0 + NH) of a segment into the Q buffer (one warp a row), their
    // constants into slot `sl`; then this warp's arrival on qready
    auto stage_q = [&](const Cursor& cq, const QV (&wq)[kRowsPerWarp], int sl) {
      const int rows = cq.rows(G);
#pragma unroll
      for (int m = 0; m < kRowsPerWarp; ++m) {
        const int r = col0 + ((warp - 2) & 3) + 4 * m;  // column (the Q buffer's row)
        const int pr = row_of_col(r);                   // row of the pair
        const QV w = wq[m];
        float cr = p.scale_log2;
        if constexpr (!KV_FP8) {
          // D / 32 bf16 = D / 16 bytes at byte b = (D / 16) * lane of the row: plane b / 128, 16-byte chunk
          // (b % 128) / 16 (head_dim 128: 8 bytes, half lane / 16; head_dim 64: 4 bytes, one plane)
          const int b = (C::kD / 16) * lane, hf = b >> 7, ch = (b & 127) >> 4;
          uint8_t* dst = sQ + hf * C::kQPlane + r * 128 + ((ch ^ (r & 7)) << 4) + (b & 15);
          *reinterpret_cast<QV*>(dst) = w;
        } else {
          constexpr int kE = C::kD / 32;  // head-dim entries of this lane: [kE * lane, kE * lane + kE)
          const uint32_t* wv32 = reinterpret_cast<const uint32_t*>(&w);
          float x[kE];
#pragma unroll
          for (int e = 0; e < kE / 2; ++e) {
            x[2 * e] = bf16_lo(wv32[e]);
            x[2 * e + 1] = bf16_hi(wv32[e]);
          }
          float mx = 0.f;
#pragma unroll
          for (int e = 0; e < kE; ++e) mx = fmaxf(mx, fabsf(x[e]));
#pragma unroll
          for (int k = 16; k >= 1; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
          int ex = 0;
          if (mx > 0.f) {
            int e2;
            frexpf(mx, &e2);  // mx in [2^(e2-1), 2^e2)
            ex = 8 - e2;      // scaled row max in [128, 256)
          }
          uint32_t hw[kE / 4], lw[kE / 4];
#pragma unroll
          for (int e = 0; e < kE; e += 2) {
            const float a = ldexpf(x[e], ex), c = ldexpf(x[e + 1], ex);
            const float ah = __uint_as_float(__float_as_uint(a) & 0xFFF00000u);  // 3 mantissa bits
            const float ch2 = __uint_as_float(__float_as_uint(c) & 0xFFF00000u);
            const int sh = 8 * (e & 3);
            if ((e & 3) == 0) { hw[e >> 2] = 0; lw[e >> 2] = 0; }
            hw[e >> 2] |= e4m3x2(ah, ch2) << sh;
            lw[e >> 2] |= e4m3x2(a - ah, c - ch2) << sh;
          }
          // kE bytes at byte kE*lane of the D-byte row: plane b / 128, 16-byte chunk (b % 128) / 16
          const int b = kE * lane, hf = b >> 7, ch = (b & 127) >> 4;
          const uint32_t off = hf * C::kQPlane + r * 128 + ((ch ^ (r & 7)) << 4) + (b & 15);
          if constexpr (kE == 4) {
            *reinterpret_cast<uint32_t*>(sQ + off) = hw[0];
            *reinterpret_cast<uint32_t*>(sQ + kHalves * C::kQPlane + off) = lw[0];
          } else {
            *reinterpret_cast<uint2*>(sQ + off) = make_uint2(hw[0], hw[1]);
            *reinterpret_cast<uint2*>(sQ + kHalves * C::kQPlane + off) = make_uint2(lw[0], lw[1]);
          }
          cr = ldexpf(p.scale_log2, -ex);
        }
        if (lane == 0) {
          rowC[sl * 64 + r] = cr;
          rowLim[sl * 64 + r] = pr < rows ? cq.L - cq.QL + (cq.row0() + pr) / G : -1;
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(qready);
    };

    Cursor cu = cu0;
    stage_q(cu, wq0, 0);
    named_sync(bar_sync, 128);  // the group's row constants are visible to the group

    // Per owned column pair, this thread's row-sum partial l. The group-uniform per-column values (the
    // reference maxima M_r, the FP8 score multiplier) are held one of two ways. With FP8 K/V, up to 24
    // columns a group and one token a thread, they sit in registers (as -M_r); at 32 columns, or two
    // tokens a thread (256-token tiles), they would spill, and shared memory (broadcast reads) holds them
    // instead. bf16 reads them from shared memory too: its register way spilled 44-56 bytes a thread
    // and measured 1-2 % slower. (Both ways measured: each is the faster one where it is used.)
    constexpr bool kRegs = NH <= 24 && SUB == 1 && KV_FP8 != 0;
    constexpr int kRP = kRegs ? NH / 2 : 1;
    float2 l[NH / 2];
    float2 negm[kRP], crow2[kRP];
    const float* mref = refM + col0;
    int seg = 0, seg_t0 = 0;

    // A failed wait marks this thread and skips its later waits, but every
    // named barrier below is still reached in order: no thread of the
    // group can be left behind at one.
    bool ok_sm = true;
    auto wait = [&](uint64_t* bar, uint32_t par) {
      if (ok_sm && !mbar_wait_bounded(smem_addr(bar), par, p.wait_limit_ns)) {
        ok_sm = false;
        fail();
      }
    };
    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1, sl = seg & 1;
      const bool seg_first = i == 0 || cu.t == 0;
      const bool pair_last = cu.t == cu.n_t - 1;
      const bool seg_last = i == n_tiles - 1 || pair_last;
      if (seg_first) {
        seg_t0 = cu.t;
#pragma unroll
        for (int c = 0; c < NH / 2; ++c) l[c] = make_float2(0.f, 0.f);
        if constexpr (kRegs) {
#pragma unroll
          for (int c = 0; c < kRP; ++c) {
            negm[c] = make_float2(INFINITY, INFINITY);
            crow2[c] = reinterpret_cast<const float2*>(rowC + sl * 64 + col0)[c];
          }
        }
        // the next segment's Q rows (the pair after this one, if the range reaches it) into L2
        if (NP != 64 && cu.n_t - cu.t < n_tiles - i && gt < NH) {
          Cursor nx = cu;
          nx.t = cu.n_t - 1;
          nx.advance(wv, Hkv);
          const int r = row_of_col(col0 + gt);
          if (r < nx.rows(G)) {
            const int R = nx.row0() + r, qi = R / G;
            const uint16_t* qp =
                p.q + (static_cast<size_t>(nx.q_off + qi) * p.num_q_heads + nx.g * G + (R - qi * G)) * C::kD;
#pragma unroll
            for (int o = 0; o < C::kD; o += 64) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(qp + o));
          }
        }
      }
      if constexpr (NP == 64) {
        // 64-row instances: a few tiles before the segment's end instead (rows fetched when a long segment
        // began have left L2 by its end; L2 turns over in about 30 us at these read rates). Measured 1-4 %
        // faster on 64- and 128-row batches; in the other instances the same code, inside their loops, cost
        // MTP-5 FP8 up to 12 us (the 256-token loop is sensitive to any code added to it).
        constexpr int kQAhead = 3;
        if ((cu.t == cu.n_t - 1 - kQAhead || (seg_first && cu.n_t - 1 - cu.t < kQAhead)) &&
            cu.n_t - cu.t < n_tiles - i && gt < NH) {
          Cursor nx = cu;
          nx.t = cu.n_t - 1;
          nx.advance(wv, Hkv);
          const int r = row_of_col(col0 + gt);
          if (r < nx.rows(G)) {
            const int R = nx.row0() + r, qi = R / G;
            const uint16_t* qp =
                p.q + (static_cast<size_t>(nx.q_off + qi) * p.num_q_heads + nx.g * G + (R - qi * G)) * C::kD;
#pragma unroll
            for (int o = 0; o < C::kD; o += 64) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(qp + o));
          }
        }
      }
      wait(&sfull[sb], static_cast<uint32_t>(i >> 1) & 1u);
      tc::fence_after_sync();
      // Columns of this group that hold rows of the pair (a batch whose pairs have fewer rows than the
      // instance's N): in the 64-row instances (the ones a batch of mixed query lengths runs) the P work of
      // 8-column chunks past them is skipped. Their P columns keep stale values, which reach only output
      // columns that are never read, and their row sums stay zero. (Elsewhere the branch cost registers:
      // the 48-row FP8 instance spilled 116 bytes a thread with it, 64 without.)
      // row chunks of the pair dealt to this group: chunk c0 of the group is live iff c0 < act
      const int act = NP != 64 ? min(NH, max(0, cu.rows(G) - col0))
                               : min(NH, 8 * max(0, ((cu.rows(G) + 7) / 8 - wg + C::NWG - 1) / C::NWG));
      // Scores of the owned columns for this thread's token of every sub-tile, in pairs (packed f32x2
      // arithmetic).
      float2 y[SUB][NH / 2];
      {
        uint32_t r[SUB][NH];
#pragma unroll
        for (int h = 0; h < SUB; ++h)
#pragma unroll
          for (int c0 = 0; c0 < NH; c0 += 8)
            tc::ld8(tS[sb] + 64 * h + lane_off + col0 + c0, *reinterpret_cast<uint32_t(*)[8]>(&r[h][c0]));
        tc::wait_ld();
#pragma unroll
        for (int h = 0; h < SUB; ++h)
#pragma unroll
          for (int c = 0; c < NH / 2; ++c)
            y[h][c] = make_float2(__uint_as_float(r[h][2 * c]), __uint_as_float(r[h][2 * c + 1]));
      }
      float sk[SUB], sv[SUB];
#pragma unroll
      for (int h = 0; h < SUB; ++h) { sk[h] = 1.f; sv[h] = 1.f; }
      if constexpr (KV_FP8) {
        // the tile's scales, read before S is released (that release frees their slot for reuse)
        const int ss = i % C::SS;
        wait(&scfull[ss], static_cast<uint32_t>(i / C::SS) & 1u);
        const float* sc = reinterpret_cast<const float*>(sSc + ss * C::kScB);
#pragma unroll
        for (int h = 0; h < SUB; ++h) {
          sk[h] = sc[tok + 128 * h];
          sv[h] = sc[C::kTile + tok + 128 * h];
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[sb]);
      if (seg_last && i + 1 < n_tiles) {
        // S(i), the last reader of this segment's Q, is done: stage the next segment's rows
        Cursor nx = cu;
        nx.advance(wv, Hkv);
        QV wq[kRowsPerWarp];
        q_load(nx, wq);  // every row's load first: one memory latency for the warp's rows
        stage_q(nx, wq, sl ^ 1);
      }

      const int L = cu.L;
      const int tabs0 = cu.t * C::kTile + tok;  // this thread's token of sub-tile h: tabs0 + 128 h
      const int vs = i % C::VS;
      float inv_sv[SUB];
#pragma unroll
      for (int h = 0; h < SUB; ++h) {
        const int tabs = tabs0 + 128 * h;
        inv_sv[h] = 1.f;
        if (KV_FP8) {
          if (tabs >= L) { sk[h] = 0.f; sv[h] = 1.f; }
          const float svh = fmaxf(sv[h], 7.888609052210118e-31f);  // 2^-100 floor keeps log2 and 1/x finite
          const float2 ls = make_float2(__log2f(svh), __log2f(svh));
          inv_sv[h] = __frcp_rn(svh);
          const float2 sk2 = make_float2(sk[h], sk[h]);
#pragma unroll
          for (int c = 0; c < NH / 2; ++c)
            y[h][c] = __ffma2_rn(__fmul2_rn(y[h][c], sk2),
                                 kRegs ? crow2[c % kRP] : reinterpret_cast<const float2*>(rowC + sl * 64 + col0)[c], ls);
        } else {
          const float2 s2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
          for (int c = 0; c < NH / 2; ++c) y[h][c] = __fmul2_rn(y[h][c], s2);
        }
        // causal mask inside the drafts / pair end / padding rows
        if (tabs >= L) {
#pragma unroll
          for (int c = 0; c < NH / 2; ++c) y[h][c] = make_float2(-INFINITY, -INFINITY);
        } else if (tabs > L - cu.QL) {
          const int* lim = rowLim + sl * 64 + col0;
#pragma unroll
          for (int c = 0; c < NH / 2; ++c) {
            if (tabs > lim[2 * c]) y[h][c].x = -INFINITY;
            if (tabs > lim[2 * c + 1]) y[h][c].y = -INFINITY;
          }
        }
      }
      // d = y - M (log2 units); with M = -inf a finite score gives +inf (and a masked one NaN, dropped
      // below). (Shared-memory way: a segment's first tile has no reference yet and d holds y itself.)
      // The tile maximum runs as four independent chains (a single one is 2 x NH x SUB dependent steps).
      float2 dl[SUB][NH / 2];
      float dmax;
      if constexpr (kRegs) {
        float dm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int h = 0; h < SUB; ++h)
#pragma unroll
          for (int c = 0; c < NH / 2; ++c) {
            dl[h][c] = __fadd2_rn(y[h][c], negm[c % kRP]);
            dm4[(h * (NH / 2) + c) & 3] = fmaxf(dm4[(h * (NH / 2) + c) & 3], fmaxf(dl[h][c].x, dl[h][c].y));
          }
        dmax = fmaxf(fmaxf(dm4[0], dm4[1]), fmaxf(dm4[2], dm4[3]));
      } else {
        dmax = INFINITY;
        if (!seg_first) {
          float dm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < NH / 2; ++c) {
            const float2 m = reinterpret_cast<const float2*>(mref)[c];
#pragma unroll
            for (int h = 0; h < SUB; ++h) {
              dl[h][c] = __fadd2_rn(y[h][c], make_float2(-m.x, -m.y));
              dm4[(c * SUB + h) & 3] = fmaxf(dm4[(c * SUB + h) & 3], fmaxf(dl[h][c].x, dl[h][c].y));
            }
          }
          dmax = fmaxf(fmaxf(dm4[0], dm4[1]), fmaxf(dm4[2], dm4[3]));
        } else {
#pragma unroll
          for (int h = 0; h < SUB; ++h)
#pragma unroll
            for (int c = 0; c < NH / 2; ++c) dl[h][c] = y[h][c];
        }
      }
      if (named_or(bar_or, 128, dmax > 8.f)) {
        // ---- exact tile maxima of the owned columns, raise the references, rescale l and O
        // (registers: the maxima of y; shared memory: of d, plus the group-uniform offset M, so that y is
        // not kept next to d)
#pragma unroll
        for (int c = 0; c < NH; ++c) {
          float v = kRegs ? ((c & 1) ? y[0][c >> 1].y : y[0][c >> 1].x) : ((c & 1) ? dl[0][c >> 1].y : dl[0][c >> 1].x);
#pragma unroll
          for (int h = 1; h < SUB; ++h)
            v = fmaxf(v, kRegs ? ((c & 1) ? y[h][c >> 1].y : y[h][c >> 1].x)
                               : ((c & 1) ? dl[h][c >> 1].y : dl[h][c >> 1].x));
          if constexpr (!kRegs) v += seg_first ? 0.f : mref[c];
          const float m = warp_max(v);
          if (lane == 0) red[(warp - 2) * 64 + col0 + c] = m;
        }
        named_sync(bar_sync, 128);
        // One thread per column takes the new reference M' = max(M, tile max), writes it to refM, and leaves in
        // the group's first two warp rows of red the column's offset for d (the old offset minus M') and its
        // factor 2^(M - M') for l and O (1 where M is unchanged, M' = -inf or on a segment's first tile). Every
        // thread then applies them with a few vector loops: the code runs cold, once per segment, so it is kept
        // short, and each column's new reference is taken once, not in every loop that needs it.
        float* rg = red + wg * 4 * 64 + col0;  // this group's 4 warp rows
        bool scaled = false;
        if (gt < NH) {
          const float mo = seg_first ? -INFINITY : refM[col0 + gt];
          const float mn = fmaxf(mo, fmaxf(fmaxf(rg[gt], rg[64 + gt]), fmaxf(rg[128 + gt], rg[192 + gt])));
          scaled = !seg_first && mn != -INFINITY && mn != mo;
          rg[gt] = (seg_first ? 0.f : mo) - mn;
          rg[64 + gt] = scaled ? fast_exp2(mo - mn) : 1.f;
          refM[col0 + gt] = mn;
        }
        // the group's OR, and the barrier that orders the writes above before the reads below
        if (named_or(bar_or, 128, scaled)) {
          if (gt == 0) atomicAdd(p.err + kWsRescaleWord, 1u);  // diagnostic count of O rescales
          wait(&pfree[(i - 1) % C::PB], static_cast<uint32_t>((i - 1) / C::PB) & 1u);  // PV of tile i-1 done
          tc::fence_after_sync();
#pragma unroll 1
          for (int hc = 0; hc < C::kMh * (C::kStackP ? 2 : 1) * NH; hc += 8) {
            const int h = hc / ((C::kStackP ? 2 : 1) * NH), rem = hc - h * (C::kStackP ? 2 : 1) * NH;
            const int pt = rem / NH, c0 = rem - pt * NH;  // O_hi, then O_lo 64 columns on
            const uint32_t ta = tO + C::kOCols * h + 64 * pt + lane_off + col0 + c0;
            uint32_t r8[8];
            tc::ld8(ta, r8);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) r8[j] = __float_as_uint(__uint_as_float(r8[j]) * rg[64 + c0 + j]);
            tc::st8(ta, r8);
          }
          tc::wait_st();
        }
#pragma unroll
        for (int c = 0; c < NH / 2; ++c) {
          l[c] = __fmul2_rn(l[c], reinterpret_cast<const float2*>(rg + 64)[c]);
          if constexpr (kRegs) {
            const float2 m = reinterpret_cast<const float2*>(refM + col0)[c];
            negm[c % kRP] = make_float2(-m.x, -m.y);
#pragma unroll
            for (int h = 0; h < SUB; ++h) dl[h][c] = __fadd2_rn(y[h][c], negm[c % kRP]);
          } else {
            const float2 dd = reinterpret_cast<const float2*>(rg)[c];
#pragma unroll
            for (int h = 0; h < SUB; ++h) dl[h][c] = __fadd2_rn(dl[h][c], dd);
          }
        }
        // red is rewritten only after the next vote (a barrier of this group), when every read here is done
      }
      // ---- P = 2^(y - M) (<= 2^8), row sums, P into shared memory as the MMA's B operand
      const int pb = i % C::PB;
      if (i >= C::PB) wait(&pfree[pb], static_cast<uint32_t>(i / C::PB - 1) & 1u);
      const int nv = L - cu.t * C::kTile;
      if (nv < C::kTile) {
        // Rows past the pair inside the last MMA k-step (a page's unused slots, or a page never loaded)
        // may hold anything, and P = 0 times NaN would still poison O: they become zeros. The softmax
        // looks at the V ring only here, and its parity wait names tile i only once the slot's previous
        // tile, i - VS, has landed: PV(i - PB) done implies that when VS >= PB; otherwise PV(i - VS),
        // which read it, is awaited first (the slot cannot be past tile i: that needs P(i)).
        if (C::VS < C::PB && i >= C::VS)
          wait(&pfree[(i - C::VS) % C::PB], static_cast<uint32_t>((i - C::VS) / C::PB) & 1u);
        wait(&vfull[vs], static_cast<uint32_t>(i / C::VS) & 1u);
        const int kend = KV_FP8 ? ((nv + 31) & ~31) : ((nv + 15) & ~15);
#pragma unroll
        for (int h = 0; h < SUB; ++h) {
          const int t = tok + 128 * h;  // token of the tile
          if (wg == 0 && t >= nv && t < kend) {
#pragma unroll
            for (int hf = 0; hf < C::kRowB / 128; ++hf) {
              uint4* z = reinterpret_cast<uint4*>(sV + vs * C::kVStage + hf * (C::kTile * 128) + t * 128);
#pragma unroll
              for (int k = 0; k < 8; ++k) z[k] = make_uint4(0, 0, 0, 0);
            }
          }
        }
      }
      uint8_t* prow = sP + pb * C::kPBuf;
#pragma unroll
      for (int c0 = 0; c0 < NH; c0 += 8) {
        if (NP == 64 && c0 >= act) continue;  // no row of the pair in these columns (64-row instances)
        const int cg = col0 + c0;  // first global column of these 8
#pragma unroll
        for (int h = 0; h < SUB; ++h) {
          const int t = tok + 128 * h;  // token of the tile (row of P)
          const float2 iv2 = make_float2(inv_sv[h], inv_sv[h]);
          float2 pv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 d = dl[h][c0 / 2 + j];
            // exp2 of max(d, -200): a masked score (-inf, or NaN against M = -inf) gives 0 after flush-to-zero
            pv[j] = make_float2(fast_exp2(fmaxf(d.x, -200.f)), fast_exp2(fmaxf(d.y, -200.f)));
            l[c0 / 2 + j] = __ffma2_rn(pv[j], iv2, l[c0 / 2 + j]);
          }
          if (!KV_FP8) {
            uint4 w;
            w.x = pack_bf16(pv[0].x, pv[0].y);
            w.y = pack_bf16(pv[1].x, pv[1].y);
            w.z = pack_bf16(pv[2].x, pv[2].y);
            w.w = pack_bf16(pv[3].x, pv[3].y);
            const int ch = cg >> 3;  // 16-byte chunk of the 128-byte token row
            *reinterpret_cast<uint4*>(prow + t * 128 + ((ch ^ (t & 7)) << 4)) = w;
          } else {
            uint32_t hw0 = 0, hw1 = 0, lw0 = 0, lw1 = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 a = pv[j];
              const float2 ah = make_float2(__uint_as_float(__float_as_uint(a.x) & 0xFFF00000u),
                                            __uint_as_float(__float_as_uint(a.y) & 0xFFF00000u));  // 3 mantissa bits
              const float2 al = __ffma2_rn(ah, make_float2(-1.f, -1.f), a);                      // exact remainder
              const uint32_t hb = e4m3x2(ah.x, ah.y), lb = e4m3x2(al.x, al.y);
              if (j < 2) { hw0 |= hb << (16 * j); lw0 |= lb << (16 * j); }
              else { hw1 |= hb << (16 * (j - 2)); lw1 |= lb << (16 * (j - 2)); }
            }
            // 8 bytes at byte cg of the 64-byte token row (64B swizzle: chunk ^= (t/2)%4)
            const int ch = cg >> 4;
            const uint32_t off = t * 64 + ((ch ^ ((t >> 1) & 3)) << 4) + (cg & 8);
            *reinterpret_cast<uint2*>(prow + off) = make_uint2(hw0, hw1);
            *reinterpret_cast<uint2*>(prow + C::kPPlane + off) = make_uint2(lw0, lw1);
          }
        }
      }
      fence_proxy_async();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[pb]);

      if (seg_last) {
        // ---- segment epilogue: O / l for the owned columns (PV(i) done: O holds the segment)
        wait(&pfree[pb], static_cast<uint32_t>(i / C::PB) & 1u);
        tc::fence_after_sync();
        // Row sums over the group's 128 threads. Within a warp, a halving butterfly: at each step a lane
        // keeps half of its columns, sends the other half to its partner and adds what it receives, so
        // the NH columns cost about NH shuffles in all and lane L ends with column L >> (5 - log2 W).
        // Then the group's 4 warps meet in shared memory. (This code runs once per segment: it is kept
        // short, as it usually runs cold in the instruction cache while HBM traffic is at its peak.)
        {
          constexpr int W = NH <= 8 ? 8 : NH <= 16 ? 16 : 32;  // columns padded to a power of two
          float v[W];
#pragma unroll
          for (int c = 0; c < W; ++c) v[c] = c < NH ? ((c & 1) ? l[c >> 1].y : l[c >> 1].x) : 0.f;
#pragma unroll
          for (int w = W, k = 16; w > 1; w >>= 1, k >>= 1) {
            const bool up = (lane & k) != 0;
#pragma unroll
            for (int i = 0; i < w / 2; ++i) {
              const float send = up ? v[i] : v[i + w / 2];
              const float keep = up ? v[i + w / 2] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, k);
            }
          }
#pragma unroll
          for (int k = 32 / W / 2; k >= 1; k >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], k);
          constexpr int kShift = W == 32 ? 0 : W == 16 ? 1 : 2;
          const int col = lane >> kShift;
          if ((lane & ((1 << kShift) - 1)) == 0 && col < NH) redl[(warp - 2) * 64 + col0 + col] = v[0];
        }
        named_sync(bar_sync, 128);
        const int rows = cu.rows(G);
        const bool whole = seg_t0 == 0 && pair_last;  // the segment is the whole pair: no combine
        const size_t u = static_cast<size_t>(p.slot_base) + cta + cu.pair(wv, Hkv, p.rows_split != 0);
        float* rinv = red + 4 * C::NWG * 64;  // 1 / row total (0 for an empty row)
        if (gt < NH) {
          const int cc = col0 + gt;
          const float* rl = redl + wg * 4 * 64 + cc;
          const float s2 = (rl[0] + rl[64]) + (rl[128] + rl[192]);
          rinv[cc] = s2 > 0.f ? __frcp_rn(s2) : 0.f;
          const float mg = refM[cc];  // this column's reference max (a column without a finite score has s2 = 0)
          const int pr = row_of_col(cc);
          if (ok_sm && !whole && pr < rows)
            p.part_lse[u * p.rows_max + pr] = s2 > 0.f ? mg + __log2f(s2) : -INFINITY;
        }
        named_sync(bar_sync, 128);
        if (ok_sm) {
#pragma unroll 1
          for (int hc = 0; hc < C::kMh * NH; hc += 8) {
            const int h = hc / NH, c0 = hc - h * NH;
            const int d = 128 * h + tok;  // O^T lanes are head-dim entries
            uint32_t r8[8], q8[8];
            tc::ld8(tO + C::kOCols * h + lane_off + col0 + c0, r8);
            if constexpr (C::kStackP) tc::ld8(tO + C::kOCols * h + 64 + lane_off + col0 + c0, q8);  // O_lo
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int cj = col0 + c0 + j;
              const int r = row_of_col(cj);  // a chunk's columns hold consecutive rows
              if (r >= rows) break;
              const float o = C::kStackP ? __uint_as_float(r8[j]) + __uint_as_float(q8[j]) : __uint_as_float(r8[j]);
              const float val = o * rinv[cj];
              if (C::kD < 128 && d >= C::kD) continue;  // head_dim 64: lanes past it hold unused rows of O
              if (!whole) {
                p.part_o[(u * p.rows_max + r) * C::kD + d] = val;
              } else {
                const int R = cu.row0() + r, qi = R / G;
                const size_t o =
                    (static_cast<size_t>(cu.q_off + qi) * p.num_q_heads + cu.g * G + (R - qi * G)) * C::kD + d;
                if (p.out_f32) reinterpret_cast<float*>(p.out)[o] = val;
                else reinterpret_cast<uint16_t*>(p.out)[o] = static_cast<uint16_t>(pack_bf16(val, 0.f) & 0xFFFFu);
              }
            }
          }
        }
        tc::fence_before_sync();  // the O reads above come before the next segment's first PV
        ++seg;
      }
      if (i + 1 < n_tiles) cu.advance(wv, Hkv);
    }
  }

  // Lane 0 of the MMA warp and of the producers ran alone until here: reconverge
  // before the CTA barrier, so that the TMEM release below follows every role's last use.
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Launches the kernel for one (KV type, padded rows, head_dim) instance.
template <int F8, int NP, int D, int SUB = 1>
cudaError_t run_tc(int units, const CUtensorMap* tmk, const CUtensorMap* tmv, const SplitParams* p,
                   cudaStream_t stream) {
  auto kern = pa_tc_split_kernel<F8, NP, D, SUB>;
  constexpr int smem = TcCfg<F8, NP, D, SUB>::kSmem;
  static std::atomic<uint64_t> attr_done{0};  // devices whose limit is raised
  const cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  kern<<<units, TcCfg<F8, NP, D, SUB>::kThreads, smem, stream>>>(*tmk, *tmv, *p);
  return cudaGetLastError();
}


}  // namespace pav
