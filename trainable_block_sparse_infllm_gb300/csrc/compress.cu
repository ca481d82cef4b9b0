// Stage 1 of InfLLM v2: semantic-kernel key compression.
//
// [InfLLM v2 > Semantic kernels for block relevance scoring, eq. S_j]: kernel
// j covers keys [j s, j s + p) (p = 32, s = 16, adjacent kernels overlap by
// half) and is represented by the mean of its keys, eq. r_kernel.
//
// With s = p / 2 every kernel is the union of two consecutive 16-key chunks,
// so a CTA streams its chunk range once (one fp32 sum per chunk and dim) and
// writes Mean_j = (C_j + C_{j+1}) / 32.  The fp32 mean is stored as two bf16
// planes, hi = bf16(mean) and lo = bf16(mean - hi), so that the selection
// stage can feed both straight to the tensor cores.  HBM-bound: one read of
// the keys, one write of 512 bytes per kernel.
#include "compress.cuh"
#include "kernels.h"

namespace infllmv2 {

namespace {

constexpr int kKernelsPerCta = 32;
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    compress_kernel(const __nv_bfloat16* __restrict__ k, const int32_t* __restrict__ kv_lens,
                    int Hkv, int Lmax, int ncmax, int kbegin, int kend,
                    __nv_bfloat16* __restrict__ kc, uint32_t* status) {
  __shared__ __align__(16) float csum[kKernelsPerCta + 1][kHeadDim];
  const int b = blockIdx.z, h = blockIdx.y;
  pdl_wait();
  pdl_trigger();
  const int L = kv_lens[b];
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(status, kStatusBadKvLen);
    return;
  }
  const int nc = n_complete_kernels(L);
  const int begin = kbegin >= 0 ? kbegin : max(0, nc + kbegin);
  const int end = kend >= 0 ? min(kend, nc) : nc;
  const int j0 = begin + blockIdx.x * kKernelsPerCta;
  const int j1 = min(j0 + kKernelsPerCta, end);
  if (j0 >= j1) return;

  const size_t bh = static_cast<size_t>(b) * Hkv + h;
  const __nv_bfloat16* kbh = k + bh * Lmax * kHeadDim;
  const int nchunk = j1 - j0 + 1;  // chunks j0 .. j1 of 16 keys
  const int sub = threadIdx.x & 15;
  for (int cc = threadIdx.x >> 4; cc < nchunk; cc += kThreads / 16) {
    float acc[8];
    chunk_sum16(acc, kbh, (j0 + cc) * kStride, sub);
    float4* dst = reinterpret_cast<float4*>(&csum[cc][sub * 8]);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  __syncthreads();

  __nv_bfloat16* hi_plane = kc + (bh * 2 + 0) * ncmax * kHeadDim;
  __nv_bfloat16* lo_plane = kc + (bh * 2 + 1) * ncmax * kHeadDim;
  for (int idx = threadIdx.x; idx < (j1 - j0) * 32; idx += kThreads) {
    const int jj = idx >> 5, q4 = idx & 31;
    const float4 a = *reinterpret_cast<const float4*>(&csum[jj][q4 * 4]);
    const float4 c = *reinterpret_cast<const float4*>(&csum[jj + 1][q4 * 4]);
    uint32_t hw[2], lw[2];
    kernel_mean_hilo(a.x, a.y, c.x, c.y, hw[0], lw[0]);
    kernel_mean_hilo(a.z, a.w, c.z, c.w, hw[1], lw[1]);
    const size_t off = static_cast<size_t>(j0 + jj) * kHeadDim + q4 * 4;
    *reinterpret_cast<uint2*>(hi_plane + off) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(lo_plane + off) = make_uint2(lw[0], lw[1]);
  }
}

// Coarse kernels of the LSE approximation ([InfLLM v2 > Efficient LSE
// approximation]): the mean of each complete window of sc keys (stride sc,
// sc a multiple of 16), as hi/lo bf16 planes like the fine kernels.  Sixteen
// threads per window, 8 dims each, summing its 16-key chunks in order.
__global__ void __launch_bounds__(kThreads)
    coarse_kernel(const __nv_bfloat16* __restrict__ k, const int32_t* __restrict__ kv_lens, int Hkv, int Lmax,
                  int nccmax, int sc, __nv_bfloat16* __restrict__ kcc, uint32_t* status) {
  const int b = blockIdx.z, h = blockIdx.y;
  pdl_wait();
  pdl_trigger();
  const int L = kv_lens[b];
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && h == 0) atomicOr(status, kStatusBadKvLen);
    return;
  }
  const int ncc = L / sc;
  const int j = blockIdx.x * (kThreads / 16) + (threadIdx.x >> 4);
  if (j >= ncc) return;
  const int sub = threadIdx.x & 15;
  const size_t bh = static_cast<size_t>(b) * Hkv + h;
  const __nv_bfloat16* kbh = k + bh * Lmax * kHeadDim;
  float tot[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int c = 0; c < sc / kStride; ++c) {
    float acc[8];
    chunk_sum16(acc, kbh, j * sc + c * kStride, sub);
#pragma unroll
    for (int e = 0; e < 8; ++e) tot[e] += acc[e];
  }
  const float inv = 1.0f / static_cast<float>(sc);
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float m0 = tot[2 * e] * inv, m1 = tot[2 * e + 1] * inv;
    const __nv_bfloat162 hv = __floats2bfloat162_rn(m0, m1);
    const __nv_bfloat162 lv = __floats2bfloat162_rn(m0 - __bfloat162float(hv.x), m1 - __bfloat162float(hv.y));
    hw[e] = *reinterpret_cast<const uint32_t*>(&hv);
    lw[e] = *reinterpret_cast<const uint32_t*>(&lv);
  }
  const size_t plane = static_cast<size_t>(nccmax) * kHeadDim;
  const size_t off = bh * 2 * plane + static_cast<size_t>(j) * kHeadDim + sub * 8;
  *reinterpret_cast<uint4*>(kcc + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(kcc + off + plane) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

}  // namespace

cudaError_t launch_coarse(const Shape& s, const void* k, const int32_t* kv_lens, int sc, void* kcc,
                          uint32_t* status, cudaStream_t st) {
  const int nccmax = s.Lmax / sc;
  if (nccmax <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((nccmax + kThreads / 16 - 1) / (kThreads / 16), s.Hkv, s.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, coarse_kernel, static_cast<const __nv_bfloat16*>(k), kv_lens, s.Hkv, s.Lmax,
                            nccmax, sc, static_cast<__nv_bfloat16*>(kcc), status);
}

cudaError_t launch_compress(const Shape& s, const void* k, const int32_t* kv_lens, int kbegin,
                            int kend, void* kc, uint32_t* status, cudaStream_t st) {
  int count;
  if (kbegin < 0) {
    count = min(-kbegin, s.ncmax);
  } else {
    const int e = kend >= 0 ? min(kend, s.ncmax) : s.ncmax;
    count = e - kbegin;
  }
  if (count <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((count + kKernelsPerCta - 1) / kKernelsPerCta, s.Hkv, s.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, compress_kernel, static_cast<const __nv_bfloat16*>(k), kv_lens, s.Hkv, s.Lmax,
                            s.ncmax, kbegin, kend, static_cast<__nv_bfloat16*>(kc), status);
}

}  // namespace infllmv2
