// The whole InfLLM v2 decode step for one query token per sequence in one
// launch: the newest semantic kernel, block selection and sparse attention of
// a (b, h_kv) group run in one thread-block cluster with no global scratch.
//
// [InfLLM v2 > Semantic kernels for block relevance scoring, eqs. S_j,
// r_kernel, r_block], [> Query group sharing, eq. r_group], [> Top-K
// implementation and the LSE bottleneck], [> Initial and local tokens always
// selected], [> Block-level key-value partitioning], [> Complexity analysis,
// stage 2].
//
// CTA r of the cluster owns the 16-block groups [r per, (r + 1) per) and the
// matching 64-kernel chunks (the kernels of blocks [16k, 16k + 16) are
// 64k - 1 .. 64k + 63).
//   compress  the CTA whose chunks hold the newest complete kernel recomputes
//             it from the keys with the compression kernel's arithmetic,
//             stores it in the kernel-mean planes and patches its own
//             shared-memory copy of the chunk.
//   phase A   hi/lo chunks streamed by TMA; z = score_scale q . Mean on the
//             tensor cores; z stays in registers (4 values per thread and
//             chunk), so nothing is written to global memory.
//   LSE       per-warp maxima, exp2(z - max) in place, per-warp sums; CTA
//             partials merged across the cluster through distributed shared
//             memory -> exact lse per head.
//   phase B   g = (1/16) sum_h exp2(z - lse_h) from the stored exponentials
//             and one weight per (warp, head); block maxima of the CTA's
//             blocks.  The kernel 64k - 1 shared with the previous CTA is
//             merged in when CTA 0 gathers the block scores.
//   top-k     CTA 0 holds all block scores in registers and selects.
//   attend    the selected blocks are dealt round-robin to three warp pairs
//             per CTA; a pair TMA-loads one block's K and V tiles (32 KB) and
//             each warp of the pair takes 32 of its keys: S = Q K^T on the
//             tensor cores, online softmax in base 2, O += P V with P fed as
//             bf16 hi + lo.
//   merge     warps merge in shared memory, CTAs through distributed shared
//             memory: CTA r writes heads [16 r / C, 16 (r + 1) / C).
#include "compress.cuh"
#include "select_common.cuh"

namespace infllmv2 {

namespace {

constexpr int kDsThreads = 256;
constexpr int kDsChunk = 64;          // kernels per phase-A stage
constexpr int kDsStages = 2;          // phase-A stages
constexpr int kDsMaxIt = 8;           // chunks per CTA (their z live in registers)
constexpr int kDsPairs = 3;           // attention warp pairs, one 32 KB stage each
constexpr int kDsStageBytes = 32768;  // 64 kernels hi + lo, or one block's K + V
constexpr int kDsMaxR = 16;           // block scores per thread in the top-k
constexpr int kDsCtaOOff = 16384;     // CTA partial O: stage 0's V half

struct DsParams {
  int B, Hkv, Lmax, ncmax, nbmax, kmax;
  int topk, n_init, n_local, inc_forced;
  float score_scale2, attn_scale2;
  const int32_t* kv_lens;
  const __nv_bfloat16* k;
  __nv_bfloat16* kc;
  int32_t* block_idx;
  int32_t* n_sel;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
};

struct DsLayout {
  int surv, selbuf, q, wpart, cpart, lse, gbuf, rsl, glast, sel, cta_ml, warp_ml, wgt, bar, total;
};

// The stage area (kDsPairs x 32 KB) holds, in turn: the phase-A chunks, CTA
// 0's top-k scratch, the attention K/V tiles, the per-warp O partials.
__host__ __device__ inline DsLayout ds_layout(int nbmax, int kmax) {
  DsLayout l;
  l.surv = (static_cast<int>(sizeof(RegTopkScratch<kDsThreads>)) + 15) & ~15;
  l.selbuf = l.surv + nbmax * 8;
  l.q = kDsPairs * kDsStageBytes;
  l.wpart = l.q + 4096;
  l.cpart = l.wpart + 8 * kGroup * 8;
  l.lse = l.cpart + kGroup * 8;
  l.gbuf = l.lse + kGroup * 4;
  l.rsl = l.gbuf + kDsMaxIt * kDsChunk * 4;
  l.glast = l.rsl + kDsMaxIt * 16 * 4;
  l.sel = l.glast + 16;
  l.cta_ml = (l.sel + kmax * 4 + 15) & ~15;
  l.warp_ml = l.cta_ml + kGroup * 8;
  l.wgt = l.warp_ml + 2 * kDsPairs * kGroup * 8;
  l.bar = (l.wgt + 2 * kDsPairs * kGroup * 4 + 15) & ~15;
  l.total = l.bar + (2 * kDsStages + 1 + kDsPairs) * 8;
  return l;
}

__host__ __device__ inline int ds_per(int groups, int C) { return (groups + C - 1) / C; }

// Barrier of the two warps of attention pair `pair` (ids 1..3; 0 is __syncthreads).
__device__ __forceinline__ void pair_sync(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(pair + 1) : "memory");
}

__device__ __forceinline__ void tma_block(uint8_t* stage, const CUtensorMap* kmap, const CUtensorMap* vmap,
                                          int row, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kDsStageBytes);
  tma_load_2d(stage, kmap, 0, row, bar);
  tma_load_2d(stage + 8192, kmap, 64, row, bar);
  tma_load_2d(stage + 16384, vmap, 0, row, bar);
  tma_load_2d(stage + 24576, vmap, 64, row, bar);
}

template <int C>
__global__ void __launch_bounds__(kDsThreads, 2)
    decode_step_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                       DsParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const DsLayout lay = ds_layout(p.nbmax, p.kmax);
  float2* wpart = reinterpret_cast<float2*>(smem + lay.wpart);   // [8 warps][16 heads]
  float2* cpart = reinterpret_cast<float2*>(smem + lay.cpart);   // [16]
  float* lse2 = reinterpret_cast<float*>(smem + lay.lse);        // [16]
  float* gbuf = reinterpret_cast<float*>(smem + lay.gbuf);       // [kDsMaxIt * 64]
  float* rsl = reinterpret_cast<float*>(smem + lay.rsl);         // [kDsMaxIt * 16]
  float* glast = reinterpret_cast<float*>(smem + lay.glast);
  int32_t* selS = reinterpret_cast<int32_t*>(smem + lay.sel);    // [kmax] ascending, -1 padded
  float2* cta_ml = reinterpret_cast<float2*>(smem + lay.cta_ml);
  float2* warp_ml = reinterpret_cast<float2*>(smem + lay.warp_ml);
  float* wgt = reinterpret_cast<float*>(smem + lay.wgt);
  float* cta_o = reinterpret_cast<float*>(smem + kDsCtaOOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + kDsStages;
  uint64_t* qbar = empty + kDsStages;
  uint64_t* kvfull = qbar + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rank = static_cast<int>(cluster_ctarank());
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const size_t orow = static_cast<size_t>(b) * Hq + static_cast<size_t>(h) * kGroup;

  if (tid == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    for (int s = 0; s < kDsStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    mbar_init(qbar, 1);
    for (int s = 0; s < kDsPairs; ++s) mbar_init(&kvfull[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int L = p.kv_lens[b];
  const int nbt = L >= 1 ? (L - 1) / kBlock + 1 : 0;
  const int groups = (nbt + 15) / 16;
  const int per = ds_per(groups, C);
  if (L < 1 || L > p.Lmax || per > kDsMaxIt) {   // same for every CTA of the cluster
    if (rank == 0) {
      for (int e = tid; e < p.kmax; e += kDsThreads) p.block_idx[static_cast<size_t>(bh) * p.kmax + e] = -1;
      for (int e = tid; e < kGroup * kHeadDim; e += kDsThreads) p.out[orow * kHeadDim + e] = __float2bfloat16(0.f);
      if (tid < kGroup && p.lse) p.lse[orow + tid] = -INFINITY;
      if (tid == 0) {
        p.n_sel[bh] = 0;
        atomicOr(p.status, kStatusBadKvLen);
      }
    }
    return;
  }
  const int i = L - 1, c = i / kBlock;
  const int k0 = min(groups, rank * per), k1 = min(groups, (rank + 1) * per);
  const int nc = n_complete_kernels(L);
  const int nmy = max(0, min(k1, (nc + kDsChunk - 1) / kDsChunk) - k0);
  const int jn = nc - 1;   // newest complete kernel
  const int it_new = (jn >= 0 && jn / kDsChunk >= k0 && jn / kDsChunk < k0 + nmy) ? jn / kDsChunk - k0 : -1;
  const size_t plane_rows = static_cast<size_t>(p.ncmax) * kHeadDim;

  auto issue = [&](int it) {
    const int st = it % kDsStages;
    const int row = (k0 + it) * kDsChunk;
    uint8_t* dst = smem + st * kDsStageBytes;
    mbar_arrive_expect_tx(&full[st], kDsStageBytes);
    tma_load_2d(dst, &kc_map, 0, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 8192, &kc_map, 64, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 16384, &kc_map, 0, (bh * 2 + 1) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 24576, &kc_map, 64, (bh * 2 + 1) * p.ncmax + row, &full[st]);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, 4096);
    tma_load_2d(smem + lay.q, &q_map, 0, static_cast<int>(orow), qbar);
    tma_load_2d(smem + lay.q + 2048, &q_map, 64, static_cast<int>(orow), qbar);
    for (int it = 0; it < min(kDsStages, nmy); ++it) issue(it);
    for (int it = kDsStages; it < nmy; ++it) {
      const int row = (k0 + it) * kDsChunk;
      tma_prefetch_2d(&kc_map, 0, (bh * 2 + 0) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 64, (bh * 2 + 0) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 0, (bh * 2 + 1) * p.ncmax + row);
      tma_prefetch_2d(&kc_map, 64, (bh * 2 + 1) * p.ncmax + row);
    }
  }

  // ---------------------------------------------------- newest kernel --
  // Warp 7: lane = 16 * half + sub sums chunk jn + half over dims [8 sub, 8 sub + 8).
  uint4 new_hi = make_uint4(0, 0, 0, 0), new_lo = make_uint4(0, 0, 0, 0);
  if (it_new >= 0 && warp == 7) {
    const __nv_bfloat16* kbh = p.k + static_cast<size_t>(bh) * p.Lmax * kHeadDim;
    const int sub = lane & 15, half = lane >> 4;
    float acc[8], oth[8];
    chunk_sum16(acc, kbh, (jn + half) * kStride, sub);
#pragma unroll
    for (int e = 0; e < 8; ++e) oth[e] = __shfl_down_sync(0xffffffffu, acc[e], 16);
    if (half == 0) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) kernel_mean_hilo(acc[2 * e], acc[2 * e + 1], oth[2 * e], oth[2 * e + 1], hw[e], lw[e]);
      new_hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      new_lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      const size_t off = (static_cast<size_t>(bh) * 2) * plane_rows + static_cast<size_t>(jn) * kHeadDim + sub * 8;
      *reinterpret_cast<uint4*>(p.kc + off) = new_hi;
      *reinterpret_cast<uint4*>(p.kc + off + plane_rows) = new_lo;
    }
  }

  // ------------------------------------------------------------ phase A --
  bool ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  const uint32_t q_b = smem_u32(smem + lay.q);
  float zr[kDsMaxIt][4];
  float mx0 = -INFINITY, mx1 = -INFINITY;
  {
    uint32_t a[8][4];
    load_q_frags(a, q_b, lane);
#pragma unroll
    for (int it = 0; it < kDsMaxIt; ++it) {
      zr[it][0] = zr[it][1] = zr[it][2] = zr[it][3] = -INFINITY;
      if (it < nmy) {
        const int st = it % kDsStages;
        const uint32_t ph = static_cast<uint32_t>(it / kDsStages) & 1u;
        bool got = ok && mbar_wait(&full[st], ph, p.status);
        ok = __all_sync(0xffffffffu, got);
        if (it == it_new) {   // the same iteration in every warp of the CTA
          ok = __syncthreads_and(ok);
          if (ok && warp == 7 && lane < 16) {
            uint8_t* stg = smem + st * kDsStageBytes;
            const uint32_t off = swz128_offset(jn - (k0 + it) * kDsChunk, lane, kDsChunk);
            *reinterpret_cast<uint4*>(stg + off) = new_hi;
            *reinterpret_cast<uint4*>(stg + 16384 + off) = new_lo;
          }
          __syncthreads();
        }
        if (ok) {
          const uint32_t hi_b = smem_u32(smem + st * kDsStageBytes);
          const int kj = (k0 + it) * kDsChunk + warp * 8 + 2 * tq;
          float acc[4];
          score_ntile(acc, a, hi_b, hi_b + 16384, warp * 8, kDsChunk, lane);
          const bool v0 = kj < nc, v1 = kj + 1 < nc;
          zr[it][0] = v0 ? acc[0] * p.score_scale2 : -INFINITY;
          zr[it][1] = v1 ? acc[1] * p.score_scale2 : -INFINITY;
          zr[it][2] = v0 ? acc[2] * p.score_scale2 : -INFINITY;
          zr[it][3] = v1 ? acc[3] * p.score_scale2 : -INFINITY;
          mx0 = fmaxf(mx0, fmaxf(zr[it][0], zr[it][1]));
          mx1 = fmaxf(mx1, fmaxf(zr[it][2], zr[it][3]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (tid == 0 && ok && it + kDsStages < nmy) {
          if (mbar_wait(&empty[st], ph, p.status)) issue(it + kDsStages);
        }
        __syncwarp();
      }
    }
  }

  // --------------------------------------------------- LSE over the cluster --
  // Row g holds head g, row g + 8 head g + 8; the four tq lanes share a row.
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int it = 0; it < kDsMaxIt; ++it) {
    if (it < nmy) {
      zr[it][0] = (mx0 == -INFINITY) ? 0.f : fast_exp2(zr[it][0] - mx0);
      zr[it][1] = (mx0 == -INFINITY) ? 0.f : fast_exp2(zr[it][1] - mx0);
      zr[it][2] = (mx1 == -INFINITY) ? 0.f : fast_exp2(zr[it][2] - mx1);
      zr[it][3] = (mx1 == -INFINITY) ? 0.f : fast_exp2(zr[it][3] - mx1);
      l0 += zr[it][0] + zr[it][1];
      l1 += zr[it][2] + zr[it][3];
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (tq == 0) {
    wpart[warp * kGroup + g] = make_float2(mx0, l0);
    wpart[warp * kGroup + g + 8] = make_float2(mx1, l1);
  }
  __syncthreads();
  if (tid < kGroup) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float2 v = wpart[w * kGroup + tid];
      lse_merge(m, l, v.x, v.y);
    }
    cpart[tid] = make_float2(m, l);
  }
  cluster_sync();
  if (tid < kGroup) {
    float2 v[C];
#pragma unroll
    for (int q = 0; q < C; ++q) v[q] = ld_dsmem_f32x2(dsmem_addr(&cpart[tid], q));
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int q = 0; q < C; ++q) lse_merge(m, l, v[q].x, v[q].y);
    lse2[tid] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  // ------------------------------------------------------------ phase B --
  {
    const float w0 = (mx0 == -INFINITY) ? 0.f : fast_exp2(mx0 - lse2[g]) * (1.0f / kGroup);
    const float w1 = (mx1 == -INFINITY) ? 0.f : fast_exp2(mx1 - lse2[g + 8]) * (1.0f / kGroup);
#pragma unroll
    for (int it = 0; it < kDsMaxIt; ++it) {
      if (it < nmy) {
        float se = zr[it][0] * w0 + zr[it][2] * w1;   // kernel kj, heads g and g + 8
        float so = zr[it][1] * w0 + zr[it][3] * w1;   // kernel kj + 1
#pragma unroll
        for (int o = 4; o <= 16; o <<= 1) {
          se += __shfl_xor_sync(0xffffffffu, se, o);
          so += __shfl_xor_sync(0xffffffffu, so, o);
        }
        if (g == 0) *reinterpret_cast<float2*>(&gbuf[it * kDsChunk + warp * 8 + 2 * tq]) = make_float2(se, so);
      }
    }
  }
  __syncthreads();
  {
    const int jb0 = 16 * k0, jb1 = min(16 * k1, nbt);
    const int kb0 = kDsChunk * k0;
    for (int j = jb0 + tid; j < jb1; j += kDsThreads) {
      const int a0 = max(4 * j - 1, kb0), e0 = min(nc - 1, 4 * j + 3);
      float r = -INFINITY;
      for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - kb0]);
      rsl[j - jb0] = r;
    }
    if (tid == 0) *glast = (k1 > k0 && kDsChunk * k1 - 1 < nc) ? gbuf[kDsChunk * (k1 - k0) - 1] : -INFINITY;
  }
  cluster_sync();

  // ------------------------------------------------------------- top-k --
  if (rank == 0) {
    float v[kDsMaxR];   // block j = tid + 256 x, scored by CTA (j / 16) / per
#pragma unroll
    for (int x = 0; x < kDsMaxR; ++x) {
      const int j = tid + kDsThreads * x;
      v[x] = -INFINITY;
      if (j < nbt) {
        const int q = (j >> 4) / per;
        const int base = 16 * per * q;
        float r = ld_dsmem_f32(dsmem_addr(&rsl[j - base], q));
        if (j == base && q > 0) r = fmaxf(r, ld_dsmem_f32(dsmem_addr(glast, q - 1)));
        v[x] = r;
      }
    }
    RegTopkScratch<kDsThreads>& tk = *reinterpret_cast<RegTopkScratch<kDsThreads>*>(smem);
    select_topk_regs<kDsThreads, kDsMaxR>(
        v, nbt, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax, p.block_idx + static_cast<size_t>(bh) * p.kmax,
        p.n_sel + bh, tk, reinterpret_cast<unsigned long long*>(smem + lay.surv),
        reinterpret_cast<int*>(smem + lay.selbuf), tid, selS);
  }
  cluster_sync();

  // ------------------------------------------------------------ attend --
  if (rank != 0)
    for (int x = tid; x < p.kmax; x += kDsThreads)
      selS[x] = static_cast<int32_t>(ld_dsmem_u32(dsmem_addr(&selS[x], 0)));
  __syncthreads();

  const int pair = warp >> 1, half = warp & 1;
  if (pair < kDsPairs) {
    uint8_t* stage = smem + pair * kDsStageBytes;
    const uint32_t k_b = smem_u32(stage), v_b = k_b + 16384;
    const int kv_row0 = bh * p.Lmax;
    const int rbase = 32 * half;
    int n = rank + C * pair;
    int j = n < p.kmax ? selS[n] : -1;
    if (j > c) j = -1;
    if (half == 0 && lane == 0 && j >= 0) tma_block(stage, &k_map, &v_map, kv_row0 + j * kBlock, &kvfull[pair]);

    float o[16][4];
#pragma unroll
    for (int x = 0; x < 16; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;
    l0 = 0.f;
    l1 = 0.f;
    uint32_t phase = 0;
#pragma unroll 1
    while (j >= 0) {
      bool got = ok && mbar_wait(&kvfull[pair], phase, p.status);
      got = __all_sync(0xffffffffu, got);
      ok = got;
      phase ^= 1u;
      const int key0 = j * kBlock + rbase;
      if (got && key0 <= i) {
        if (key0 + 31 > i) {
          // Keys past i: zero their V rows so masked probabilities never
          // meet non-finite values that may sit in the cache beyond kv_len.
          const int r0 = i - key0 + 1;
          for (int e = lane; e < (32 - r0) * 16; e += 32) {
            const int row = rbase + r0 + (e >> 4), q16 = e & 15;
            *reinterpret_cast<uint4*>(stage + 16384 + (q16 >> 3) * 8192 + row * 128 + (q16 & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // S = Q K^T over this warp's 32 keys: 4 n-tiles of 8 keys.
        float s[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t qa0[4], qa1[4];
          ldmatrix_x4(qa0, q_b + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 4 * kk + (lane >> 4), 16));
          ldmatrix_x4(qa1, q_b + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 4 * kk + 2 + (lane >> 4), 16));
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            uint32_t kb[4];
            ldmatrix_x4(kb, k_b + swz128_offset(rbase + nt * 8 + (lane & 7), 4 * kk + (lane >> 3), kBlock));
            mma_bf16_16816(s[nt], qa0, kb[0], kb[1]);
            mma_bf16_16816(s[nt], qa1, kb[2], kb[3]);
          }
        }
        float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int x = key0 + nt * 8 + 2 * tq;
          const bool v0 = x <= i, v1 = x + 1 <= i;
          s[nt][0] = v0 ? s[nt][0] * p.attn_scale2 : -INFINITY;
          s[nt][1] = v1 ? s[nt][1] * p.attn_scale2 : -INFINITY;
          s[nt][2] = v0 ? s[nt][2] * p.attn_scale2 : -INFINITY;
          s[nt][3] = v1 ? s[nt][3] * p.attn_scale2 : -INFINITY;
          mxa = fmaxf(mxa, fmaxf(s[nt][0], s[nt][1]));
          mxb = fmaxf(mxb, fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
        }
        // key0 <= i, so every row has a finite maximum here.
        const float mn0 = fmaxf(m0, mxa), mn1 = fmaxf(m1, mxb);
        const float sc0 = fast_exp2(m0 - mn0), sc1 = fast_exp2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        l0 *= sc0;
        l1 *= sc1;
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          o[x][0] *= sc0;
          o[x][1] *= sc0;
          o[x][2] *= sc1;
          o[x][3] *= sc1;
        }
        // P as bf16 hi + lo parts (16 significant bits).
        uint32_t pa[2][4], pl[2][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const float p0 = fast_exp2(s[nt][0] - mn0), p1 = fast_exp2(s[nt][1] - mn0);
          const float p2 = fast_exp2(s[nt][2] - mn1), p3 = fast_exp2(s[nt][3] - mn1);
          l0 += p0 + p1;
          l1 += p2 + p3;
          const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
          const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
          const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
          pa[nt >> 1][(nt & 1) * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
          pa[nt >> 1][(nt & 1) * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
          pl[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0 - f01.x, p1 - f01.y);
          pl[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2 - f23.x, p3 - f23.y);
        }
        // O += P V over the 32 keys: two k-steps of 16.
#pragma unroll
        for (int np = 0; np < 8; ++np) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            uint32_t vb[4];
            ldmatrix_x4_trans(vb, v_b + swz128_offset(rbase + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8,
                                                      2 * np + (lane >> 4), kBlock));
            mma_bf16_16816(o[2 * np], pa[kk], vb[0], vb[1]);
            mma_bf16_16816(o[2 * np + 1], pa[kk], vb[2], vb[3]);
            mma_bf16_16816(o[2 * np], pl[kk], vb[0], vb[1]);
            mma_bf16_16816(o[2 * np + 1], pl[kk], vb[2], vb[3]);
          }
        }
      }
      // Next block of this pair (the same sequence in both warps).
      n += C * kDsPairs;
      int jnext = n < p.kmax ? selS[n] : -1;
      if (jnext > c) jnext = -1;
      if (jnext >= 0) {
        // Both warps are done with the stage; order the zeroed V rows
        // (generic writes) before the TMA refill (async proxy).
        fence_proxy_async_smem();
        pair_sync(pair);
        if (half == 0 && lane == 0 && ok)
          tma_block(stage, &k_map, &v_map, kv_row0 + jnext * kBlock, &kvfull[pair]);
      }
      j = jnext;
    }
    pair_sync(pair);   // the partner has finished reading the stage
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float* o_w = reinterpret_cast<float*>(stage + half * 8192);
#pragma unroll
    for (int x = 0; x < 16; ++x) {
      const int d0 = x * 8 + 2 * tq;
      *reinterpret_cast<float2*>(o_w + g * kHeadDim + d0) = make_float2(o[x][0], o[x][1]);
      *reinterpret_cast<float2*>(o_w + (g + 8) * kHeadDim + d0) = make_float2(o[x][2], o[x][3]);
    }
    if (tq == 0) {
      warp_ml[warp * kGroup + g] = make_float2(m0, l0);
      warp_ml[warp * kGroup + g + 8] = make_float2(m1, l1);
    }
  }
  __syncthreads();
  constexpr int kAw = 2 * kDsPairs;   // warps holding attention partials
  if (tid < kGroup) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAw; ++w) M = fmaxf(M, warp_ml[w * kGroup + tid].x);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kAw; ++w) {
      const float2 v = warp_ml[w * kGroup + tid];
      const float wt = (M == -INFINITY) ? 0.f : fast_exp2(v.x - M);
      wgt[w * kGroup + tid] = wt;
      lsum += wt * v.y;
    }
    cta_ml[tid] = make_float2(M, lsum);
  }
  __syncthreads();
  for (int e = tid; e < kGroup * kHeadDim; e += kDsThreads) {
    const int hd = e >> 7;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kAw; ++w)
      acc += wgt[w * kGroup + hd] *
             reinterpret_cast<const float*>(smem + (w >> 1) * kDsStageBytes + (w & 1) * 8192)[e];
    cta_o[e] = acc;
  }
  cluster_sync();

  // Heads [hpc * rank, hpc * (rank + 1)) of the output from all partials.
  constexpr int hpc = kGroup / C;
  for (int e = tid; e < hpc * kHeadDim; e += kDsThreads) {
    const int hd = rank * hpc + e / kHeadDim;
    const int d = e % kHeadDim;
    float2 ml[C];
    float ov[C];
#pragma unroll
    for (int q = 0; q < C; ++q) {
      ml[q] = ld_dsmem_f32x2(dsmem_addr(&cta_ml[hd], q));
      ov[q] = ld_dsmem_f32(dsmem_addr(&cta_o[hd * kHeadDim + d], q));
    }
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < C; ++q) M = fmaxf(M, ml[q].x);
    float lsum = 0.f, acc = 0.f;
#pragma unroll
    for (int q = 0; q < C; ++q) {
      const float wt = (M == -INFINITY) ? 0.f : fast_exp2(ml[q].x - M);
      lsum += wt * ml[q].y;
      acc += wt * ov[q];
    }
    p.out[(orow + hd) * kHeadDim + d] = __float2bfloat16(lsum > 0.f ? acc / lsum : 0.f);
    if (d == 0 && p.lse)
      p.lse[orow + hd] = lsum > 0.f ? (M + fast_log2(lsum)) * 0.69314718055994531f : -INFINITY;
  }
  cluster_sync();   // keeps this CTA's shared memory alive for remote readers
}

template <int C>
bool ds_fits(const Shape& s) {
  const int groups = (s.nbmax + 15) / 16;
  const DsLayout l = ds_layout(s.nbmax, s.kmax);
  return s.nq == 1 && ds_per(groups, C) <= kDsMaxIt && s.nbmax <= kDsThreads * kDsMaxR &&
         l.selbuf + s.kmax * 4 <= kDsPairs * kDsStageBytes && l.total + 1024 <= 113 * 1024;
}

template <int C>
void ds_config(const Shape& s, cudaLaunchConfig_t* cfg, cudaLaunchAttribute (&attrs)[2], cudaStream_t st) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(C, s.B * s.Hkv, 1);
  cfg->blockDim = dim3(kDsThreads, 1, 1);
  cfg->dynamicSmemBytes = ds_layout(s.nbmax, s.kmax).total + 1024;
  cfg->stream = st;
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = C;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attrs;
  cfg->numAttrs = 2;
}

// True when the C-CTA form fits this shape and, for C = 16, every group's
// cluster can be resident at once (the only case in which it pays off).
template <int C>
bool ds_ready(const Shape& s) {
  if (!ds_fits<C>(s)) return false;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attrs[2];
  ds_config<C>(s, &cfg, attrs, nullptr);
  if (cudaFuncSetAttribute(decode_step_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(cfg.dynamicSmemBytes)) != cudaSuccess)
    return cudaGetLastError(), false;
  if (C > 8 && cudaFuncSetAttribute(decode_step_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                   cudaSuccess)
    return cudaGetLastError(), false;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, decode_step_kernel<C>, &cfg) != cudaSuccess)
    return cudaGetLastError(), false;
  return clusters >= ((C > 8) ? s.B * s.Hkv : 1);
}

}  // namespace

int decode_step_cluster_size(const Shape& s) {
  if (s.B * s.Hkv * 16 <= 2 * device_sm_count() && ds_ready<16>(s)) return 16;
  if (ds_ready<8>(s)) return 8;
  return 0;
}

cudaError_t launch_decode_step(const Shape& s, int cluster, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                               const CUtensorMap& k_map, const CUtensorMap& v_map, const void* k,
                               const int32_t* kv_lens, void* kc, int32_t* block_idx, int32_t* n_sel, void* out,
                               float* lse, uint32_t* status, cudaStream_t st) {
  DsParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.ncmax = s.ncmax;
  p.nbmax = s.nbmax;
  p.kmax = s.kmax;
  p.topk = s.topk;
  p.n_init = s.n_init;
  p.n_local = s.n_local;
  p.inc_forced = s.inc_forced;
  p.score_scale2 = s.score_scale2;
  p.attn_scale2 = s.attn_scale2;
  p.kv_lens = kv_lens;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.kc = static_cast<__nv_bfloat16*>(kc);
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attrs[2];
  if (cluster == 16) {
    ds_config<16>(s, &cfg, attrs, st);
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<16>, kc_map, q_map, k_map, v_map, p);
  }
  if (cluster == 8) {
    ds_config<8>(s, &cfg, attrs, st);
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<8>, kc_map, q_map, k_map, v_map, p);
  }
  return cudaErrorInvalidConfiguration;
}

}  // namespace infllmv2
