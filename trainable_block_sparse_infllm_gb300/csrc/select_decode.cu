// Stage 2 of InfLLM v2, decode / verification path (n_q <= 16 tokens per
// sequence): block relevance and top-k block selection.
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck],
// [> Initial and local tokens always selected].  Per query token of a GQA
// group: z[h, j] = score_scale * q_h . Mean_j over the visible kernels,
// g[j] = (1/16) sum_h exp(z[h, j] - lse_h) with the exact two-pass LSE,
// r[blk] = max of g over the kernels meeting the block, top-k with forced
// blocks.
//
// One thread-block cluster of C CTAs per (b, h_kv) group scores the group's
// n_q tokens together.  The blocks 0 .. floor(i/m) are cut into 16-block
// groups, `per` consecutive groups per CTA; CTA r owns the matching 64-kernel
// chunks (the kernels of blocks [16k, 16k+16) are 64k-1 .. 64k+63).
//   phase A  TMA-stream the CTA's hi/lo chunks (the rest prefetched to L2),
//            z = q.Mean on the tensor cores, z to scratch (L2), per-row
//            (max, sum) partials in shared memory.
//   sync     partials of all CTAs read through distributed shared memory
//            -> exact LSE per head.
//   phase B  g and the block maxima r of the CTA's blocks.
//   sync     the CTA that owns token t (t mod C) pulls the token's block
//            scores into registers and selects (bitmask top-k).
// No global partials, tickets or memsets: cluster barriers order it all.
#include "select_common.cuh"

namespace infllmv2 {

namespace {

constexpr int kClThreads = 256;   // 8 warps: one 8-kernel n-tile each per chunk
constexpr int kClChunk = 64;      // kernels per stage (= 16 blocks)
constexpr int kClStages = 2;      // small enough for two CTAs per SM
constexpr int kClStageBytes = 2 * kClChunk * 256;
constexpr int kClMaxR = 16;       // block scores per thread in the top-k (nbmax <= 4096)

struct ClLayout {
  int stage, q, wpart, cpart, lse, g, rsl, tk, surv, bar, total, rsl_stride;
};

__host__ __device__ inline int cl_per(int groups, int C) { return (groups + C - 1) / C; }

__host__ __device__ inline ClLayout cl_layout(int C, int nq, int nbmax, int kmax) {
  ClLayout l;
  const int per = cl_per((nbmax + 15) / 16, C);   // 16-block groups per CTA
  l.rsl_stride = per * 16;
  l.stage = 0;
  l.q = kClStages * kClStageBytes;
  l.wpart = l.q + nq * 4096;
  l.cpart = l.wpart + 8 * nq * kGroup * 8;
  l.lse = l.cpart + nq * kGroup * 8;
  l.g = l.lse + nq * kGroup * 4;
  l.rsl = l.g + (per * kClChunk + 4) * 4;
  l.tk = (l.rsl + nq * l.rsl_stride * 4 + 15) & ~15;
  l.surv = (l.tk + static_cast<int>(sizeof(BitTopkScratch<kClThreads, kClMaxR>)) + 15) & ~15;
  l.bar = (l.surv + nbmax * 8 + 15) & ~15;
  l.total = l.bar + (2 * kClStages + 1) * 8;
  return l;
}

template <int C>
__global__ void __launch_bounds__(kClThreads, 2)
    sel_cluster_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap q_map,
                       SelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nq = p.nq;
  const ClLayout lay = cl_layout(C, nq, p.nbmax, p.kmax);
  float2* wpart = reinterpret_cast<float2*>(smem + lay.wpart);   // [8 warps][nq*16]
  float2* cpart = reinterpret_cast<float2*>(smem + lay.cpart);   // [nq*16]
  float* lse2 = reinterpret_cast<float*>(smem + lay.lse);        // [nq*16]
  float* gbuf = reinterpret_cast<float*>(smem + lay.g);
  float* rsl = reinterpret_cast<float*>(smem + lay.rsl);         // [nq][rsl_stride]
  BitTopkScratch<kClThreads, kClMaxR>& tk = *reinterpret_cast<BitTopkScratch<kClThreads, kClMaxR>*>(smem + lay.tk);
  unsigned long long* surv = reinterpret_cast<unsigned long long*>(smem + lay.surv);   // [nbmax]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + kClStages;
  uint64_t* qbar = empty + kClStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rank = static_cast<int>(cluster_ctarank());
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const size_t unit0 = static_cast<size_t>(bh) * nq;

  if (tid == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    for (int s = 0; s < kClStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    mbar_init(qbar, 1);
    fence_barrier_init();
  }
  for (int e = tid; e < 8 * nq * kGroup; e += kClThreads) wpart[e] = make_float2(-INFINITY, 0.f);
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int L = p.kv_lens[b];
  if (L < nq || L > p.Lmax) {        // same for every CTA of the cluster
    if (rank == 0) {
      for (int e = tid; e < nq * p.kmax; e += kClThreads) p.block_idx[unit0 * p.kmax + e] = -1;
      for (int e = tid; e < nq; e += kClThreads) p.n_sel[unit0 + e] = 0;
      if (p.write_r)
        for (int e = tid; e < nq * p.nbmax; e += kClThreads) p.r_buf[unit0 * p.nbmax + e] = -INFINITY;
      if (tid == 0) atomicOr(p.status, kStatusBadKvLen);
    }
    return;
  }
  const int nbt = (L - 1) / kBlock + 1;            // blocks visible to the last token
  const int groups = (nbt + 15) / 16;
  const int per = cl_per(groups, C);
  const int k0 = min(groups, rank * per), k1 = min(groups, (rank + 1) * per);
  const int nc = n_complete_kernels(L);
  const int nmy = max(0, min(k1, (nc + kClChunk - 1) / kClChunk) - k0);   // chunks to stream

  auto issue = [&](int it) {
    const int st = it % kClStages;
    const int row = (k0 + it) * kClChunk;
    uint8_t* dst = smem + lay.stage + st * kClStageBytes;
    mbar_arrive_expect_tx(&full[st], kClStageBytes);
    tma_load_2d(dst, &kc_map, 0, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 8192, &kc_map, 64, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 16384, &kc_map, 0, (bh * 2 + 1) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 24576, &kc_map, 64, (bh * 2 + 1) * p.ncmax + row, &full[st]);
  };
  if (tid == 0) {
    if (nmy > 0) {
      mbar_arrive_expect_tx(qbar, nq * 4096);
      const int Hq = p.Hkv * kGroup;
      for (int t = 0; t < nq; ++t) {
        const int row = (b * nq + t) * Hq + h * kGroup;
        tma_load_2d(smem + lay.q + t * 4096, &q_map, 0, row, qbar);
        tma_load_2d(smem + lay.q + t * 4096 + 2048, &q_map, 64, row, qbar);
      }
    }
    for (int it = 0; it < min(kClStages, nmy); ++it) issue(it);
    // The rest of this CTA's chunks go to L2 now, so HBM streams at full
    // rate while the two shared-memory stages trail behind.
    for (int it = kClStages; it < nmy; ++it) {
      const int row = (k0 + it) * kClChunk;
      tma_prefetch_2d(&kc_map, 0, (bh * 2 + 0) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 64, (bh * 2 + 0) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 0, (bh * 2 + 1) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 64, (bh * 2 + 1) * p.ncmax + row);
    }
  }

  // ------------------------------------------------------------ phase A --
  bool ok = true;
  if (nmy > 0) ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  const uint32_t q_b = smem_u32(smem + lay.q);
  uint32_t a[8][4];
  if (nq == 1 && nmy > 0) load_q_frags(a, q_b, lane);   // one token: fragments stay in registers
#pragma unroll 1
  for (int it = 0; it < nmy && ok; ++it) {
    const int st = it % kClStages;
    const uint32_t ph = static_cast<uint32_t>(it / kClStages) & 1u;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st], ph, p.status));
    if (!ok) break;
    const int kbase = (k0 + it) * kClChunk;
    const uint32_t hi_b = smem_u32(smem + lay.stage + st * kClStageBytes);
    const int kj = kbase + warp * 8 + 2 * tq;
#pragma unroll 1
    for (int t = 0; t < nq; ++t) {
      const int nvis = n_complete_kernels(L - nq + t + 1);
      if (nq > 1) load_q_frags(a, q_b + t * 4096, lane);
      float acc[4];
      score_ntile(acc, a, hi_b, hi_b + 16384, warp * 8, kClChunk, lane);
      const bool v0 = kj < nvis, v1 = kj + 1 < nvis;
      const float z0 = v0 ? acc[0] * p.scale2 : -INFINITY;
      const float z1 = v1 ? acc[1] * p.scale2 : -INFINITY;
      const float z2 = v0 ? acc[2] * p.scale2 : -INFINITY;
      const float z3 = v1 ? acc[3] * p.scale2 : -INFINITY;
      float* zrow = p.z + ((unit0 + t) * kGroup + g) * static_cast<size_t>(p.ncpad);
      *reinterpret_cast<float2*>(zrow + kj) = make_float2(z0, z1);
      *reinterpret_cast<float2*>(zrow + 8 * static_cast<size_t>(p.ncpad) + kj) = make_float2(z2, z3);
      float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
      lse_add2(m0, l0, z0, z1);
      lse_add2(m1, l1, z2, z3);
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        lse_merge(m0, l0, __shfl_xor_sync(0xffffffffu, m0, o), __shfl_xor_sync(0xffffffffu, l0, o));
        lse_merge(m1, l1, __shfl_xor_sync(0xffffffffu, m1, o), __shfl_xor_sync(0xffffffffu, l1, o));
      }
      if (tq == 0) {
        float2* w0 = &wpart[warp * nq * kGroup + t * kGroup + g];
        float2 v = *w0;
        lse_merge(v.x, v.y, m0, l0);
        *w0 = v;
        float2* w1 = w0 + 8;
        v = *w1;
        lse_merge(v.x, v.y, m1, l1);
        *w1 = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (tid == 0 && it + kClStages < nmy) {
      if (mbar_wait(&empty[st], ph, p.status)) issue(it + kClStages);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int row = tid; row < nq * kGroup; row += kClThreads) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float2 v = wpart[w * nq * kGroup + row];
      lse_merge(m, l, v.x, v.y);
    }
    cpart[row] = make_float2(m, l);
  }
  cluster_sync();

  // ---------------------------------------------- LSE over the cluster --
  for (int row = tid; row < nq * kGroup; row += kClThreads) {
    float2 v[C];   // all remote loads first, so their round trips overlap
#pragma unroll
    for (int q = 0; q < C; ++q) v[q] = ld_dsmem_f32x2(dsmem_addr(&cpart[row], q));
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int q = 0; q < C; ++q) lse_merge(m, l, v[q].x, v[q].y);
    lse2[row] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  // ------------------------------------------------------------ phase B --
  for (int t = 0; t < nq; ++t) {
    const int i = L - nq + t;
    const int c = i / kBlock;
    const int nvis = n_complete_kernels(i + 1);
    const int jb0 = 16 * k0, jb1 = min(16 * k1, c + 1);
    const int klo = max(0, 4 * jb0 - 1);
    if (jb0 < jb1) {
      const int khi = min(nvis, 4 * (jb1 - 1) + 4);
      const float* zu = p.z + (unit0 + t) * kGroup * static_cast<size_t>(p.ncpad);
      const float* lt = lse2 + t * kGroup;
      for (int k = klo + tid; k < khi; k += kClThreads) {
        float zz[kGroup];
#pragma unroll
        for (int hh = 0; hh < kGroup; ++hh) zz[hh] = __ldcg(zu + static_cast<size_t>(hh) * p.ncpad + k);
        float s = 0.f;
#pragma unroll
        for (int hh = 0; hh < kGroup; ++hh) s += fast_exp2(zz[hh] - lt[hh]);
        gbuf[k - klo] = s * (1.0f / kGroup);
      }
      __syncthreads();
      for (int j = jb0 + tid; j < jb1; j += kClThreads) {
        const int a0 = max(0, 4 * j - 1), e0 = min(nvis - 1, 4 * j + 3);
        float r = -INFINITY;
        for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - klo]);
        rsl[t * lay.rsl_stride + (j - jb0)] = r;
        if (p.write_r) p.r_buf[(unit0 + t) * p.nbmax + j] = r;
      }
    }
    __syncthreads();
  }
  cluster_sync();

  // ------------------------------------------------------------- top-k --
  for (int t = rank; t < nq; t += C) {
    const int nb = (L - nq + t) / kBlock + 1;
    float v[kClMaxR];   // block j = tid + 256 x; owned by CTA (j / 16) / per
#pragma unroll
    for (int x = 0; x < kClMaxR; ++x) {
      const int j = tid + kClThreads * x;
      v[x] = -INFINITY;
      if (j < nb) {
        const int q = (j >> 4) / per;
        v[x] = ld_dsmem_f32(dsmem_addr(&rsl[t * lay.rsl_stride + (j - 16 * per * q)], q));
      }
    }
    if (p.write_r)
      for (int j = nb + tid; j < p.nbmax; j += kClThreads) p.r_buf[(unit0 + t) * p.nbmax + j] = -INFINITY;
    select_topk_bits<kClThreads, kClMaxR>(v, nb, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax,
                                          p.block_idx + (unit0 + t) * p.kmax, p.n_sel + unit0 + t, tk, surv, tid);
    __syncthreads();
  }
  cluster_sync();   // keeps this CTA's shared memory alive for remote readers
}

template <int C>
cudaError_t launch_cluster(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map, const SelParams& p,
                           cudaStream_t st, bool* unsupported) {
  const int smem = cl_layout(C, s.nq, s.nbmax, s.kmax).total + 1024;
  *unsupported = false;
  if (smem > 227 * 1024) {
    *unsupported = true;
    return cudaSuccess;
  }
  cudaError_t e = cudaFuncSetAttribute(sel_cluster_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(sel_cluster_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, s.B * s.Hkv, 1);
  cfg.blockDim = dim3(kClThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = C;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, sel_cluster_kernel<C>, &cfg);
  // The 16-CTA form only pays off when every group's cluster is resident at once.
  const int need = (C > 8) ? s.B * s.Hkv : 1;
  if (e != cudaSuccess || clusters < need) {
    cudaGetLastError();
    *unsupported = true;
    return cudaSuccess;
  }
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sel_cluster_kernel<C>, kc_map, q_map, p);
}

}  // namespace

size_t select_decode_ncpad(const Shape& s) {
  return static_cast<size_t>((s.ncmax + kClChunk - 1) / kClChunk) * kClChunk;
}

bool select_decode_supported(const Shape& s) { return s.nbmax <= kClThreads * kClMaxR; }

cudaError_t launch_select_decode(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                                 const SelParams& p, cudaStream_t st) {
  bool unsupported = false;
  cudaError_t e = cudaSuccess;
  if (s.B * s.Hkv * 16 <= 2 * device_sm_count()) {
    e = launch_cluster<16>(s, kc_map, q_map, p, st, &unsupported);
    if (e != cudaSuccess || !unsupported) return e;
  }
  e = launch_cluster<8>(s, kc_map, q_map, p, st, &unsupported);
  if (e == cudaSuccess && unsupported) return cudaErrorInvalidConfiguration;
  return e;
}

}  // namespace infllmv2
