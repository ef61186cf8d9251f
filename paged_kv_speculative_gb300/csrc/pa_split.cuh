// Split-KV paged verify attention for sm_103a.
//
// One CTA processes one work unit: a (sequence b, KV head g, context chunk
// [t0, t1)) triple. The q_b * G query rows that share KV head g ("rows =
// query length x GQA group", MTP-5 routing page, Motivation) are packed onto
// 16-row warp MMA tiles, one warp per tile, so each K/V byte of the chunk
// leaves HBM once per call. K/V pages are gathered through the block table
// with 2-D TMA copies (one 16-token x 128-byte box per page, 128B swizzle) into
// a 3-stage shared-memory ring; FP8 scales ride along as 64-byte bulk copies.
//
// Per 64-token sub-tile a warp computes S = Q K^T (mma.sync m16n8k16, fp32
// accumulate), applies the causal mask inside the drafts (key t is visible to
// draft i iff t <= L - q + i), runs an online softmax in the log2 domain and
// accumulates O += P V. Units that cover a whole (b, g) write the normalised
// output; split units write a normalised partial and its log2-sum-exp for the
// combine kernel.
//
// FP8 E4M3 keys/values are unpacked to f16 in registers (exact). The
// per-token scales are constant along the head dimension, so the K scale
// multiplies score column t and the V scale multiplies P column t:
//   y_t   = softmax_scale*log2(e) * s_k[t] * (Q . K8[t]) + log2 s_v[t]
//   P''_t = 2^(y_t - M),  O += P'' V8,  l += P'' / s_v[t] = 2^(z_t - M)
// so O / l is the attention over the dequantised tensors while P'' <= 1 stays
// in f16 range. Q is brought to f16 with a per-row power-of-two scale that
// the score multiplier undoes.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pav {

template <int KV_FP8, int D, int NW>
struct SplitCfg {
  static constexpr int kRowBytes = row_bytes(KV_FP8, D);   // bytes of one token's K (or V) row
  static constexpr int kHalves = kRowBytes / 128;          // 128-byte swizzle columns per row
  static constexpr int kTile = tile_tokens(KV_FP8, D);     // tokens per stage
  static constexpr int kSub = 64;                          // tokens per compute sub-tile
  static constexpr int kSubs = kTile / kSub;
  static constexpr int kKBytes = 16384;                    // K bytes per stage (V the same)
  static constexpr int kStage = stage_bytes(KV_FP8, D);
  static constexpr int kThreads = 32 * NW;
  static constexpr int kKSteps = D / 16;                   // MMA k-steps over the head dim
  static constexpr int kDTiles = D / 8;                    // n-tiles of the output
  static_assert(kRowBytes % 128 == 0, "rows must fill 128-byte swizzle columns");
  static_assert(kTile % kSub == 0, "stage must hold whole sub-tiles");
  static_assert(!KV_FP8 || D == 128, "FP8 path is written for head_dim 128");
};

// Byte offset of the 16-byte chunk `chunk` (0 .. kRowBytes/16-1) of token `tok`
// inside a stage's K or V block laid out [half][token][128 B], 128B swizzle.
template <int TILE>
__device__ __forceinline__ uint32_t swz_off(int tok, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (TILE * 128) + tok * 128 + ((((chunk & 7) ^ (tok & 7))) << 4));
}

template <int KV_FP8, int D, int NW>
__global__ void __launch_bounds__(NW * 32)
    pa_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const __grid_constant__ SplitParams p) {
  using C = SplitCfg<KV_FP8, D, NW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // carve: stages | derived scale terms (fp8) | page ids | barriers
  uint8_t* stage_base = smem;
  float4* derived = reinterpret_cast<float4*>(smem + kStages * C::kStage);
  int32_t* pids = reinterpret_cast<int32_t*>(smem + kStages * C::kStage + (KV_FP8 ? 16 * C::kTile : 0));
  uint64_t* bars = reinterpret_cast<uint64_t*>(pids + kMaxChunk / kPage);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g8 = lane >> 2;  // row within the 8-row half of an MMA tile / n index of B fragments
  const int c4 = lane & 3;   // column pair index

  // ------------------------------------------------------------ the unit
  const int u = blockIdx.x;
  const WorkView wv = work_view(p);
  if (u >= wv.num_units) return;  // a dynamic plan's grid covers its capacity
  int lo = 0, hi = wv.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (wv.seq[mid].unit_start <= u) lo = mid; else hi = mid - 1;
  }
  const SeqInfo si = wv.seq[lo];
  const int local = u - si.unit_start;
  const int kvh = local / si.n_chunks;
  const int chunk_idx = local - kvh * si.n_chunks;
  const int L = si.ctx_len;
  const int QL = si.q_len;
  const int b = si.b;
  const int G = p.group;
  const int rows = QL * G;
  const int t0 = chunk_idx * wv.chunk;
  const int t_end = min(L, t0 + wv.chunk);
  const int n_stages = (t_end - t0 + C::kTile - 1) / C::kTile;
  const int n_pages = (t_end - t0 + kPage - 1) / kPage;
  const bool split = si.n_chunks > 1;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
    prefetch_tmap(&tmk);
    prefetch_tmap(&tmv);
    if (chunk_idx == 0 && kvh == 0 && (p.dev_ctx[b] != L || p.dev_q[b] != QL)) atomicOr(p.err, 2u);
  }
  {
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.bt_stride + t0 / kPage;
    for (int i = tid; i < n_pages; i += C::kThreads) {
      int pg = __ldg(bt + i);
      if (static_cast<unsigned>(pg) >= static_cast<unsigned>(p.num_pages)) {
        atomicOr(p.err, 1u);
        pg = -1;
      }
      pids[i] = pg;
    }
  }
  __syncwarp();  // thread 0 ran the set-up alone: its warp reconverges before the CTA barrier
  __syncthreads();

  // Stage issue (warp 0): pages of tile `k` into ring slot `s`. A TMA issue
  // costs its thread about one memory latency, so each page box and scale
  // copy gets its own lane: K boxes on lanes 0-7, V boxes on 8-15, FP8 k/v
  // scales on 16-23 / 24-31 (every tile has at most 8 boxes per tensor).
  auto issue = [&](int k, int s) {
    uint8_t* st = stage_base + s * C::kStage;
    const uint32_t bar = smem_addr(&bars[s]);
    const int tok0 = t0 + k * C::kTile;
    const int pg0 = (tok0 - t0) / kPage;
    const int npg = (min(t_end, tok0 + C::kTile) - tok0 + kPage - 1) / kPage;
    if (lane == 0) {
      uint32_t bytes = npg * (2 * kPage * C::kRowBytes);
      if (KV_FP8)
        for (int j = 0; j < npg; ++j)
          if (pids[pg0 + j] >= 0) bytes += 2 * kPage * 4;
      mbar_arrive_expect_tx(bar, bytes);
    }
    __syncwarp();
    const int grp = lane >> 3, idx = lane & 7;  // grp 0: K, 1: V, 2: k scales, 3: v scales
    if (grp < 2 && idx < npg * C::kHalves) {
      const int j = idx / C::kHalves, hf = idx % C::kHalves;
      const int pg = pids[pg0 + j];
      // an invalid page reads past the tensor's end: TMA fills zeros
      const int row = (pg >= 0 ? pg : p.num_pages) * p.num_kv_heads * kPage + kvh * kPage;
      const uint32_t off = hf * (C::kTile * 128) + j * kPage * 128 + (grp ? C::kKBytes : 0);
      tma_load_2d(smem_addr(st + off), grp ? &tmv : &tmk, bar, hf * (128 / (KV_FP8 ? 1 : 2)), row);
    }
    if (KV_FP8 && grp >= 2 && idx < npg) {
      const int pg = pids[pg0 + idx];
      if (pg >= 0) {
        const size_t so = (static_cast<size_t>(pg) * p.num_kv_heads + kvh) * kPage;
        bulk_load(smem_addr(st + 2 * C::kKBytes + (grp == 3 ? C::kTile * 4 : 0) + idx * kPage * 4),
                  (grp == 2 ? p.k_scale : p.v_scale) + so, kPage * 4, bar);
      }
    }
  };
  if (warp == 0) {
    for (int s = 0; s < min(kStages, n_stages); ++s) issue(s, s);
  }

  // ------------------------------------------------------------ Q fragments
  const int r0 = warp * 16 + g8;  // rows held by this thread: r0 and r0 + 8
  const int r1 = r0 + 8;
  const bool warp_active = warp * 16 < rows;
  uint32_t qa[C::kKSteps][4];
  float crow[2] = {p.scale_log2, p.scale_log2};  // score multiplier per held row
  {
    const uint16_t* qrow[2] = {nullptr, nullptr};
    const int rr[2] = {r0, r1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (rr[h] < rows) {
        const int i = rr[h] / G;
        const int head = kvh * G + (rr[h] - i * G);
        qrow[h] = p.q + (static_cast<size_t>(si.q_off + i) * p.num_q_heads + head) * D;
      }
    }
    if (!KV_FP8) {
      // standard m16n8k16 A layout: a0 (r0, k 2c..), a1 (r1, k 2c..), a2 (r0, k 2c+8..), a3 (r1, k 2c+8..)
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint16_t* qp = qrow[j & 1];
          const int d = ks * 16 + 2 * c4 + 8 * (j >> 1);
          qa[ks][j] = qp ? __ldg(reinterpret_cast<const uint32_t*>(qp + d)) : 0u;
        }
      }
    } else {
      // FP8 path: head-dim permutation shared by Q and K. k-step ks, slot pair
      // j>>1 covers d = 32*c4 + 4*ks + 2*(j>>1) + {0,1}; thread c4 holds
      // d in [32*c4, 32*c4+32) so K rows are read with two 16-byte loads.
      float qf[2][32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint16_t* qp = qrow[h];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w = qp ? __ldg(reinterpret_cast<const uint4*>(qp + 32 * c4) + v) : make_uint4(0, 0, 0, 0);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qf[h][8 * v + 2 * e] = bf16_lo(ww[e]);
            qf[h][8 * v + 2 * e + 1] = bf16_hi(ww[e]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(qf[h][e]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        int ex = 0;
        if (mx > 0.f) {
          int e2;
          frexpf(mx, &e2);  // mx in [2^(e2-1), 2^e2)
          ex = 15 - e2;     // scaled row max in [2^14, 2^15)
        }
        crow[h] = ldexpf(p.scale_log2, -ex);
#pragma unroll
        for (int e = 0; e < 32; ++e) qf[h][e] = ldexpf(qf[h][e], ex);
      }
#pragma unroll
      for (int ks = 0; ks < C::kKSteps; ++ks) {
        qa[ks][0] = pack_f16(qf[0][4 * ks], qf[0][4 * ks + 1]);
        qa[ks][1] = pack_f16(qf[1][4 * ks], qf[1][4 * ks + 1]);
        qa[ks][2] = pack_f16(qf[0][4 * ks + 2], qf[0][4 * ks + 3]);
        qa[ks][3] = pack_f16(qf[1][4 * ks + 2], qf[1][4 * ks + 3]);
      }
    }
  }

  // causal limits of the two held rows: last visible key index
  const int lim0 = L - QL + (r0 < rows ? r0 / G : 0);
  const int lim1 = L - QL + (r1 < rows ? r1 / G : 0);

  float o[C::kDTiles][4];
#pragma unroll
  for (int n = 0; n < C::kDTiles; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};  // running max (log2 domain for fp8, raw score for bf16)
  float l_run[2] = {0.f, 0.f};

  // per-lane ldmatrix offsets (bf16)
  const int mi = lane >> 3, r8 = lane & 7;

  int it = 0;
  bool aborted = false;
  for (; it < n_stages; ++it) {
    const int s = it % kStages;
    const uint32_t par = static_cast<uint32_t>(it / kStages) & 1u;
    int my_fail = 0;
    if (!mbar_wait_bounded(smem_addr(&bars[s]), par)) {
      my_fail = 1;
      atomicOr(p.err, 4u);
    }
    uint8_t* st = stage_base + s * C::kStage;
    const int tok_base = t0 + it * C::kTile;
    const int valid = min(C::kTile, t_end - tok_base);  // tokens of this stage inside the unit
    if (KV_FP8 || valid < C::kTile) {
      // Neutralise tokens past the unit's end (stale ring data or NaN-filled
      // slots of a last page) and precompute the fp8 per-token terms.
      if (valid < C::kTile) {
        const int zb = valid * 128;  // first byte to clear in each 128-byte column block
        for (int hf = 0; hf < C::kHalves; ++hf) {
          uint4* kz = reinterpret_cast<uint4*>(st + hf * (C::kTile * 128) + zb);
          uint4* vz = reinterpret_cast<uint4*>(st + C::kKBytes + hf * (C::kTile * 128) + zb);
          const int n16 = (C::kTile - valid) * 8;
          for (int i = tid; i < n16; i += C::kThreads) {
            kz[i] = make_uint4(0, 0, 0, 0);
            vz[i] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      if (KV_FP8) {
        const float* ksc = reinterpret_cast<const float*>(st + 2 * C::kKBytes);
        const float* vsc = ksc + C::kTile;
        for (int t = tid; t < C::kTile; t += C::kThreads) {
          float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
          if (t < valid) {
            const float sv = fmaxf(vsc[t], 7.888609052210118e-31f);  // 2^-100 floor: keeps log2 / 1/x finite
            dv = make_float4(ksc[t], __log2f(sv), __frcp_rn(sv), 0.f);
          }
          derived[t] = dv;
        }
      }
      __syncthreads();
    }

    if (warp_active) {
      const uint32_t kst = smem_addr(st);
      const uint32_t vst = kst + C::kKBytes;
#pragma unroll 1
      for (int sub = 0; sub < C::kSubs; ++sub) {
        const int sub0 = sub * C::kSub;          // token offset inside the stage
        const int tok0 = tok_base + sub0;        // absolute token index
        if (sub0 >= valid) break;
        float sacc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;

        // ---- S = Q K^T
        if (!KV_FP8) {
#pragma unroll
          for (int ks = 0; ks < C::kKSteps; ++ks) {
#pragma unroll
            for (int np = 0; np < 4; ++np) {
              const int tok = sub0 + np * 16 + (mi >> 1) * 8 + r8;
              const int chunk = 2 * ks + (mi & 1);
              uint32_t kb[4];
              ldsm_x4(kb, kst + swz_off<C::kTile>(tok, chunk));
              mma_bf16(sacc[2 * np], qa[ks], kb[0], kb[1]);
              mma_bf16(sacc[2 * np + 1], qa[ks], kb[2], kb[3]);
            }
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const int tok = sub0 + nt * 8 + g8;
            const uint4 w0 = lds128(kst + swz_off<C::kTile>(tok, 2 * c4));
            const uint4 w1 = lds128(kst + swz_off<C::kTile>(tok, 2 * c4 + 1));
            const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint32_t b0 = e4m3x2_to_f16x2(wd[ks]);
              const uint32_t b1 = e4m3x2_to_f16x2(wd[ks] >> 16);
              mma_f16(sacc[nt], qa[ks], b0, b1);
            }
          }
        }

        // ---- scores in the log2 domain (fp8: scaled, with log2 s_v added)
        float inv_sv[8][2];
        if (KV_FP8) {
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const int t = sub0 + nt * 8 + 2 * c4;
            const float4 d0 = derived[t];
            const float4 d1 = derived[t + 1];
            sacc[nt][0] = fmaf(sacc[nt][0] * d0.x, crow[0], d0.y);
            sacc[nt][1] = fmaf(sacc[nt][1] * d1.x, crow[0], d1.y);
            sacc[nt][2] = fmaf(sacc[nt][2] * d0.x, crow[1], d0.y);
            sacc[nt][3] = fmaf(sacc[nt][3] * d1.x, crow[1], d1.y);
            inv_sv[nt][0] = d0.z;
            inv_sv[nt][1] = d1.z;
          }
        }
        // causal mask / unit end: only sub-tiles that reach past the first draft's last key
        if (tok0 + C::kSub > L - QL + 1 || tok0 + C::kSub > t_end) {
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int t = tok0 + nt * 8 + 2 * c4 + (e & 1);
              const int lim = (e < 2) ? lim0 : lim1;
              if (t > lim || t >= t_end) sacc[nt][e] = -INFINITY;
            }
          }
        }
        // ---- online softmax
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          mx[0] = fmaxf(mx[0], fmaxf(sacc[nt][0], sacc[nt][1]));
          mx[1] = fmaxf(mx[1], fmaxf(sacc[nt][2], sacc[nt][3]));
        }
        float sub_ref[2], alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
          mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
          const float m_new = fmaxf(m_run[h], mx[h]);
          if (KV_FP8) {
            sub_ref[h] = (m_new == -INFINITY) ? 0.f : m_new;
            alpha[h] = fast_exp2(m_run[h] - sub_ref[h]);
          } else {
            sub_ref[h] = (m_new == -INFINITY) ? 0.f : m_new * crow[h];
            alpha[h] = fast_exp2(m_run[h] * crow[h] - sub_ref[h]);
          }
          m_run[h] = m_new;
        }
        float lsum[2] = {0.f, 0.f};
        uint32_t pa[4][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          float pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            pv[e] = KV_FP8 ? fast_exp2(sacc[nt][e] - sub_ref[h]) : fast_exp2(fmaf(sacc[nt][e], crow[h], -sub_ref[h]));
          }
          if (KV_FP8) {
            lsum[0] = fmaf(pv[0], inv_sv[nt][0], fmaf(pv[1], inv_sv[nt][1], lsum[0]));
            lsum[1] = fmaf(pv[2], inv_sv[nt][0], fmaf(pv[3], inv_sv[nt][1], lsum[1]));
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_f16(pv[0], pv[1]);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_f16(pv[2], pv[3]);
          } else {
            lsum[0] += pv[0] + pv[1];
            lsum[1] += pv[2] + pv[3];
            pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(pv[0], pv[1]);
            pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(pv[2], pv[3]);
          }
        }
        l_run[0] = l_run[0] * alpha[0] + lsum[0];
        l_run[1] = l_run[1] * alpha[1] + lsum[1];
#pragma unroll
        for (int n = 0; n < C::kDTiles; ++n) {
          o[n][0] *= alpha[0];
          o[n][1] *= alpha[0];
          o[n][2] *= alpha[1];
          o[n][3] *= alpha[1];
        }
        // pa[kt] was filled as {r0 lo-half, r1 lo-half, r0 hi-half, r1 hi-half}; A wants
        // a0 (r0, k 2c..), a1 (r1, k 2c..), a2 (r0, k 2c+8..), a3 (r1, k 2c+8..): same order.

        // ---- O += P V
        if (!KV_FP8) {
#pragma unroll
          for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
            for (int np = 0; np < C::kDTiles / 2; ++np) {
              const int tok = sub0 + kt * 16 + (mi & 1) * 8 + r8;
              const int chunk = 2 * np + (mi >> 1);
              uint32_t vb[4];
              ldsm_x4_t(vb, vst + swz_off<C::kTile>(tok, chunk));
              mma_bf16(o[2 * np], pa[kt], vb[0], vb[1]);
              mma_bf16(o[2 * np + 1], pa[kt], vb[2], vb[3]);
            }
          }
        } else {
          // output-column permutation: n-tile nt, column n <-> d = 16 * n + nt, so
          // thread g8 needs d in [16*g8, 16*g8+16) of four tokens: one 16-byte load each.
#pragma unroll
          for (int kt = 0; kt < 4; ++kt) {
            const int ta = sub0 + kt * 16 + 2 * c4;
            const uint4 A0 = lds128(vst + swz_off<C::kTile>(ta, g8));
            const uint4 A1 = lds128(vst + swz_off<C::kTile>(ta + 1, g8));
            const uint4 B0 = lds128(vst + swz_off<C::kTile>(ta + 8, g8));
            const uint4 B1 = lds128(vst + swz_off<C::kTile>(ta + 9, g8));
            const uint32_t a0w[4] = {A0.x, A0.y, A0.z, A0.w}, a1w[4] = {A1.x, A1.y, A1.z, A1.w};
            const uint32_t b0w[4] = {B0.x, B0.y, B0.z, B0.w}, b1w[4] = {B1.x, B1.y, B1.z, B1.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t xa = __byte_perm(a0w[w], a1w[w], 0x5140);  // d 4w, 4w+1 of tokens 2c, 2c+1
              const uint32_t ya = __byte_perm(a0w[w], a1w[w], 0x7362);  // d 4w+2, 4w+3
              const uint32_t xb = __byte_perm(b0w[w], b1w[w], 0x5140);  // tokens 2c+8, 2c+9
              const uint32_t yb = __byte_perm(b0w[w], b1w[w], 0x7362);
              mma_f16(o[4 * w + 0], pa[kt], e4m3x2_to_f16x2(xa), e4m3x2_to_f16x2(xb));
              mma_f16(o[4 * w + 1], pa[kt], e4m3x2_to_f16x2(xa >> 16), e4m3x2_to_f16x2(xb >> 16));
              mma_f16(o[4 * w + 2], pa[kt], e4m3x2_to_f16x2(ya), e4m3x2_to_f16x2(yb));
              mma_f16(o[4 * w + 3], pa[kt], e4m3x2_to_f16x2(ya >> 16), e4m3x2_to_f16x2(yb >> 16));
            }
          }
        }
      }
    }
    // end of stage: every warp is done with slot s; the verdict on a timed-out wait is CTA-uniform
    if (__syncthreads_or(my_fail)) {
      aborted = true;
      break;
    }
    if (warp == 0 && it + kStages < n_stages) {
      fence_proxy_async();
      issue(it + kStages, s);
    }
  }

  if (aborted) {
    // Let the copies already issued (tiles it .. it+kStages-1) land before the
    // CTA's shared memory is released; each wait is bounded again.
    if (tid == 0) {
      for (int k = it; k < min(n_stages, it + kStages); ++k)
        (void)mbar_wait_bounded(smem_addr(&bars[k % kStages]), static_cast<uint32_t>(k / kStages) & 1u);
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ------------------------------------------------------------ epilogue
  if (!warp_active) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  const int rr[2] = {r0, r1};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = rr[h];
    if (r >= rows) continue;
    const float l = l_run[h];
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    float* dst_f = nullptr;
    uint16_t* dst_h = nullptr;
    if (split) {
      dst_f = p.part_o + (static_cast<size_t>(u) * p.rows_max + r) * D;
      if (c4 == 0) {
        const float mref = KV_FP8 ? m_run[h] : m_run[h] * crow[h];
        p.part_lse[static_cast<size_t>(u) * p.rows_max + r] = l > 0.f ? mref + __log2f(l) : -INFINITY;
      }
    } else {
      const int i = r / G;
      const size_t orow = (static_cast<size_t>(si.q_off + i) * p.num_q_heads + kvh * G + (r - i * G)) * D;
      if (p.out_f32) dst_f = reinterpret_cast<float*>(p.out) + orow;
      else dst_h = reinterpret_cast<uint16_t*>(p.out) + orow;
    }
    if (!KV_FP8) {
      // n-tile n, columns 2c, 2c+1 <-> d = 8n + 2c + {0,1}
#pragma unroll
      for (int n = 0; n < C::kDTiles; ++n) {
        const float x0 = o[n][2 * h] * inv_l, x1 = o[n][2 * h + 1] * inv_l;
        const int d = 8 * n + 2 * c4;
        if (dst_f) *reinterpret_cast<float2*>(dst_f + d) = make_float2(x0, x1);
        else *reinterpret_cast<uint32_t*>(dst_h + d) = pack_bf16(x0, x1);
      }
    } else {
      // n-tile n, column 2c+e <-> d = 16*(2c+e) + n: sixteen consecutive d per e
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int d0 = 32 * c4 + 16 * e;
        if (dst_f) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<float4*>(dst_f + d0 + 4 * v) =
                make_float4(o[4 * v][2 * h + e] * inv_l, o[4 * v + 1][2 * h + e] * inv_l,
                            o[4 * v + 2][2 * h + e] * inv_l, o[4 * v + 3][2 * h + e] * inv_l);
        } else {
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            uint4 w;
            w.x = pack_bf16(o[8 * v + 0][2 * h + e] * inv_l, o[8 * v + 1][2 * h + e] * inv_l);
            w.y = pack_bf16(o[8 * v + 2][2 * h + e] * inv_l, o[8 * v + 3][2 * h + e] * inv_l);
            w.z = pack_bf16(o[8 * v + 4][2 * h + e] * inv_l, o[8 * v + 5][2 * h + e] * inv_l);
            w.w = pack_bf16(o[8 * v + 6][2 * h + e] * inv_l, o[8 * v + 7][2 * h + e] * inv_l);
            *reinterpret_cast<uint4*>(dst_h + d0 + 8 * v) = w;
          }
        }
      }
    }
  }
}

}  // namespace pav
