// Cache append of a decode step: the keys and values of the n_q newest
// tokens of each sequence go to cache rows kv_lens[b] - n_q .. kv_lens[b] - 1
// ([InfLLM v2 > Block-level key-value partitioning]: the cache of 64-key
// blocks grows by the decoded tokens; their keys also complete the newest
// semantic kernel, which the decode step recomputes).
//
// Optionally the step's queries are copied too (q_src -> q_dst), so that a
// step whose inputs sit in host memory needs no separate copy: the kernel
// reads k_new, v_new and q_src with ordinary loads, which may be page-locked
// host memory mapped for the device.
//
// One 16-byte chunk per thread (a 128-dim bf16 row is 16 chunks).  The
// launch carries a programmatic dependency: the kernel waits for the
// previous kernel of the stream before writing and lets the next one (the
// decode step, which waits for this one in turn) start launching at once.
#include "common.cuh"
#include "kernels.h"

namespace infllmv2 {

namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(const uint4* k_new, const uint4* v_new, const int32_t* kv_lens, uint4* k_cache, uint4* v_cache,
                  int Hkv, int Lmax, int nq, long long total, const uint4* q_src, uint4* q_dst, long long q_chunks,
                  uint32_t* status) {
  const long long e = static_cast<long long>(blockIdx.x) * kAppendThreads + threadIdx.x;
  pdl_wait();
  if (e >= total) {
    if (e - total < q_chunks) q_dst[e - total] = q_src[e - total];   // the step's queries
  } else {
    const int chunk = static_cast<int>(e & 15);
    const int which = static_cast<int>((e >> 4) & 1);   // 0: key row, 1: value row
    const long long unit = e >> 5;                      // (b, h, t)
    const int t = static_cast<int>(unit % nq);
    const long long bh = unit / nq;
    const int b = static_cast<int>(bh / Hkv);
    const int L = kv_lens[b];
    if (L < nq || L > Lmax) {
      if (e == (bh * nq) * 32 && (bh % Hkv) == 0) atomicOr(status, kStatusBadKvLen);
    } else {
      const long long row = bh * Lmax + (L - nq + t);
      (which ? v_cache : k_cache)[row * 16 + chunk] = (which ? v_new : k_new)[unit * 16 + chunk];
    }
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_append(const Shape& s, const void* k_new, const void* v_new, const int32_t* kv_lens, void* k_cache,
                          void* v_cache, const void* q_src, void* q_dst, uint32_t* status, cudaStream_t st) {
  const long long total = static_cast<long long>(s.B) * s.Hkv * s.nq * 32;
  const long long q_chunks = q_src ? static_cast<long long>(s.B) * s.nq * s.Hkv * kGroup * 16 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((total + q_chunks + kAppendThreads - 1) / kAppendThreads), 1, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                            kv_lens, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), s.Hkv, s.Lmax, s.nq,
                            total, static_cast<const uint4*>(q_src), static_cast<uint4*>(q_dst), q_chunks, status);
}

}  // namespace infllmv2
