// Paged KV write with per-token FP8 quantisation: the step that fills the
// cache the verify step reads. New tokens' K/V rows go to their slots
// (slot = page * 16 + offset) in place; a slot of -1 is a padded or dead row
// and stores nothing (masked in-place stores: DeepSeek-V4.1 page,
// description of the hi path's KV writes). FP8: per (token, head)
// s = amax / 448 (1 when amax = 0) and code = E4M3(x / s), both divisions
// IEEE round-to-nearest in fp32, the conversion round-to-nearest-even and
// saturating at +-448.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"

namespace pav {

// Two fp32 -> E4M3 bytes, RNE, saturating (lo -> low byte).
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(256)
    pa_kv_write_kernel(int n_tokens, int num_kv_heads, int num_pages, const uint16_t* __restrict__ k_new,
                       const uint16_t* __restrict__ v_new, const int64_t* __restrict__ slot_mapping,
                       void* __restrict__ k_cache, void* __restrict__ v_cache, float* __restrict__ k_scale,
                       float* __restrict__ v_scale, uint32_t* __restrict__ err) {
  constexpr int kPer = D / 32;  // elements per lane
  const int warp_id = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_id >= n_tokens * num_kv_heads) return;
  const int t = warp_id / num_kv_heads;
  const int g = warp_id - t * num_kv_heads;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;  // padded / dead row: no store
  if (slot >= static_cast<int64_t>(num_pages) * 16) {
    if (lane == 0 && err) atomicOr(err, 1u);
    return;
  }
  const int64_t page = slot >> 4;
  const int off = static_cast<int>(slot & 15);
  const size_t src = (static_cast<size_t>(t) * num_kv_heads + g) * D + lane * kPer;
  const size_t row = (static_cast<size_t>(page) * num_kv_heads + g) * 16 + off;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint16_t* x = (which ? v_new : k_new) + src;
    uint16_t xb[kPer];
#pragma unroll
    for (int e = 0; e < kPer; e += 2) *reinterpret_cast<uint32_t*>(&xb[e]) = *reinterpret_cast<const uint32_t*>(x + e);
    if (!FP8) {
      uint16_t* dst = reinterpret_cast<uint16_t*>(which ? v_cache : k_cache) + row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = *reinterpret_cast<uint32_t*>(&xb[e]);
      continue;
    }
    float xf[kPer];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      xf[e] = __uint_as_float(static_cast<uint32_t>(xb[e]) << 16);
      amax = fmaxf(amax, fabsf(xf[e]));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    uint8_t* dst = reinterpret_cast<uint8_t*>(which ? v_cache : k_cache) + row * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2) {
      const uint32_t two = f32x2_to_e4m3x2(__fdiv_rn(xf[e], s), __fdiv_rn(xf[e + 1], s));
      *reinterpret_cast<uint16_t*>(dst + e) = static_cast<uint16_t>(two);
    }
    if (lane == 0) (which ? v_scale : k_scale)[row] = s;
  }
}

cudaError_t launch_kv_write(int head_dim, int fp8, int n_tokens, int num_kv_heads, int num_pages, const void* k_new,
                            const void* v_new, const int64_t* slot_mapping, void* k_cache, void* v_cache,
                            float* k_scale, float* v_scale, uint32_t* err, cudaStream_t stream) {
  const int64_t warps = static_cast<int64_t>(n_tokens) * num_kv_heads;
  if (warps == 0) return cudaSuccess;
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  auto kn = static_cast<const uint16_t*>(k_new);
  auto vn = static_cast<const uint16_t*>(v_new);
#define PAV_KVW(DD, F8)                                                                                        \
  if (head_dim == DD && fp8 == F8) {                                                                           \
    pa_kv_write_kernel<DD, F8><<<blocks, 256, 0, stream>>>(n_tokens, num_kv_heads, num_pages, kn, vn,         \
                                                           slot_mapping, k_cache, v_cache, k_scale, v_scale, err); \
    return cudaGetLastError();                                                                                 \
  }
  PAV_KVW(64, false) PAV_KVW(128, false) PAV_KVW(256, false)
  PAV_KVW(64, true) PAV_KVW(128, true) PAV_KVW(256, true)
#undef PAV_KVW
  return cudaErrorInvalidValue;
}

}  // namespace pav
