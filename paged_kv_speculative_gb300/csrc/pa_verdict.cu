// Greedy verify verdict: the target model's picks at the q_b verify positions
// decide how many drafts are accepted (ids + verdict computed on the device:
// DeepSeek-V4.1 page, in-graph head output). Position i of a sequence was fed
// token x_i (x_0 the last committed token, then the drafts). t_i = first
// index of the maximum of logits[i] (a NaN counts as the maximum, -0 equals
// +0); accepted a = the longest prefix with x_{j+1} == t_j; next token t_a.
//
// Pass 1: one CTA per (row, 8192-entry vocab chunk) reduces to a 64-bit key
// (order-preserving value bits << 32 | ~index), so the maximum key is the
// largest value at the lowest index. Pass 2: one warp per sequence reduces
// the chunk keys of its rows and takes the verdict with a ballot.
#include <cuda_runtime.h>
#include <stdint.h>

namespace pav {

constexpr int kVerdictChunk = 8192;

__device__ __forceinline__ uint64_t argmax_key(uint16_t bits, uint32_t idx) {
  uint32_t f = static_cast<uint32_t>(bits) << 16;
  uint32_t ord;
  if ((f & 0x7F800000u) == 0x7F800000u && (f & 0x007FFFFFu)) ord = 0xFFFFFFFFu;  // NaN: the maximum
  else {
    if (f == 0x80000000u) f = 0u;  // -0 == +0
    ord = (f & 0x80000000u) ? ~f : (f | 0x80000000u);
  }
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~idx);
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__global__ void __launch_bounds__(256) pa_argmax_chunks_kernel(const uint16_t* __restrict__ logits, int vocab,
                                                               int n_chunks, uint64_t* __restrict__ keys) {
  const int row = blockIdx.x / n_chunks;
  const int chunk = blockIdx.x - row * n_chunks;
  const int v0 = chunk * kVerdictChunk;
  const int v1 = min(vocab, v0 + kVerdictChunk);
  const uint16_t* lr = logits + static_cast<size_t>(row) * vocab;
  uint64_t best = 0;
  // 16-byte loads where the row is aligned, scalar loads for the ragged edges
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(lr) & 15u) == 0);
  if (vec_ok) {
    const int a0 = (v0 + 7) & ~7, a1 = v1 & ~7;
    for (int v = v0 + threadIdx.x; v < min(a0, v1); v += blockDim.x) best = umax64(best, argmax_key(lr[v], v));
    for (int v = a0 + 8 * threadIdx.x; v < a1; v += 8 * blockDim.x) {
      const uint4 w = *reinterpret_cast<const uint4*>(lr + v);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        best = umax64(best, argmax_key(static_cast<uint16_t>(ww[e] & 0xFFFFu), v + 2 * e));
        best = umax64(best, argmax_key(static_cast<uint16_t>(ww[e] >> 16), v + 2 * e + 1));
      }
    }
    for (int v = max(a1, a0) + threadIdx.x; v < v1; v += blockDim.x) best = umax64(best, argmax_key(lr[v], v));
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) best = umax64(best, argmax_key(lr[v], v));
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, m));
  __shared__ uint64_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (blockDim.x >> 5); ++w) best = umax64(best, red[w]);
    keys[blockIdx.x] = best;
  }
}

__global__ void __launch_bounds__(32) pa_verdict_kernel(int num_seqs, const int32_t* __restrict__ query_lens,
                                                        const int32_t* __restrict__ input_ids, int n_chunks,
                                                        int num_tokens, const uint64_t* __restrict__ keys,
                                                        int32_t* __restrict__ target_ids, int32_t* __restrict__ accepted,
                                                        int32_t* __restrict__ next_token, uint32_t* err) {
  const int b = blockIdx.x;
  const int lane = threadIdx.x;
  // row offset of sequence b: sum of the earlier query lengths
  int off = 0;
  for (int s = lane; s < b; s += 32) off += query_lens[s];
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) off += __shfl_xor_sync(0xffffffffu, off, m);
  const int q = query_lens[b];
  if (q < 1 || q > 32 || off + q > num_tokens) {
    if (lane == 0) {
      if (err) atomicOr(err, 2u);
      accepted[b] = 0;
      next_token[b] = -1;
    }
    return;
  }
  int tgt = -1;
  if (lane < q) {
    uint64_t best = 0;
    const uint64_t* kr = keys + static_cast<size_t>(off + lane) * n_chunks;
    for (int c = 0; c < n_chunks; ++c) best = umax64(best, kr[c]);
    tgt = static_cast<int>(~static_cast<uint32_t>(best & 0xFFFFFFFFu));
    target_ids[off + lane] = tgt;
  }
  const bool match = lane < q - 1 && input_ids[off + lane + 1] == tgt;
  const uint32_t ok = __ballot_sync(0xffffffffu, match);
  const int a = __ffs(~ok) - 1;  // first position whose draft was rejected (or q - 1)
  const int acc = min(a, q - 1);
  const int nxt = __shfl_sync(0xffffffffu, tgt, acc);
  if (lane == 0) {
    accepted[b] = acc;
    next_token[b] = nxt;
  }
}

size_t verdict_workspace_bytes(int num_tokens, int vocab) {
  const int n_chunks = (vocab + kVerdictChunk - 1) / kVerdictChunk;
  return 256 + static_cast<size_t>(num_tokens) * n_chunks * 8;
}

cudaError_t launch_verdict(int num_seqs, int num_tokens, int vocab, const void* logits, const int32_t* input_ids,
                           const int32_t* query_lens, int32_t* target_ids, int32_t* accepted, int32_t* next_token,
                           void* workspace, cudaStream_t stream) {
  const int n_chunks = (vocab + kVerdictChunk - 1) / kVerdictChunk;
  uint32_t* err = static_cast<uint32_t*>(workspace);
  uint64_t* keys = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(workspace) + 256);
  if (num_tokens > 0) {
    pa_argmax_chunks_kernel<<<num_tokens * n_chunks, 256, 0, stream>>>(static_cast<const uint16_t*>(logits), vocab,
                                                                       n_chunks, keys);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (num_seqs > 0)
    pa_verdict_kernel<<<num_seqs, 32, 0, stream>>>(num_seqs, query_lens, input_ids, n_chunks, num_tokens, keys,
                                                   target_ids, accepted, next_token, err);
  return cudaGetLastError();
}

}  // namespace pav
