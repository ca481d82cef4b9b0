// Arithmetic of one semantic-kernel mean, shared by the compression kernel
// and the fused decode step so that both write bit-identical kernel means.
//
// [InfLLM v2 > Semantic kernels for block relevance scoring, eq. S_j]: kernel
// j is the mean of keys [16 j, 16 j + 32).  It is formed as the fp32 sum of
// two 16-key chunks (keys added in order within a chunk), times 1/32, and
// stored as hi = bf16(mean), lo = bf16(mean - hi).
#pragma once

#include "common.cuh"

namespace infllmv2 {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& w) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(v[i] << 16);
    acc[2 * i + 1] += __uint_as_float(v[i] & 0xffff0000u);
  }
}

// fp32 sum over keys tok0 .. tok0 + 15 of dims [8 sub, 8 sub + 8) of one
// (b, h_kv) key plane `kbh` ([L_max][128] bf16).  Two batches of eight loads.
// Key `row_new` (if in range) is read from `k_row_new` (a 128-dim bf16 row)
// instead of the plane: a key this launch appends and has not yet stored.
__device__ __forceinline__ void chunk_sum16(float (&acc)[8], const __nv_bfloat16* __restrict__ kbh, int tok0,
                                            int sub, int row_new = -1, const uint4* k_row_new = nullptr) {
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 w[kStride / 2];
#pragma unroll
    for (int t = 0; t < kStride / 2; ++t) {
      const int tok = tok0 + half * 8 + t;
      w[t] = tok == row_new ? k_row_new[sub]
                            : __ldg(reinterpret_cast<const uint4*>(kbh + static_cast<size_t>(tok) * kHeadDim) + sub);
    }
#pragma unroll
    for (int t = 0; t < kStride / 2; ++t) add_bf16x8(acc, w[t]);
  }
}

// Mean of two chunk sums for two adjacent dims, as packed bf16 hi and lo pairs.
__device__ __forceinline__ void kernel_mean_hilo(float a0, float a1, float c0, float c1, uint32_t& hw,
                                                 uint32_t& lw) {
  const float m0 = (a0 + c0) * (1.0f / kKernel), m1 = (a1 + c1) * (1.0f / kKernel);
  const __nv_bfloat162 hv = __floats2bfloat162_rn(m0, m1);
  const float h0 = __bfloat162float(hv.x), h1 = __bfloat162float(hv.y);
  const __nv_bfloat162 lv = __floats2bfloat162_rn(m0 - h0, m1 - h1);
  hw = *reinterpret_cast<const uint32_t*>(&hv);
  lw = *reinterpret_cast<const uint32_t*>(&lv);
}

}  // namespace infllmv2
