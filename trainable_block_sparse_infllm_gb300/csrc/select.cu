// Stage 2 of InfLLM v2: block relevance and top-k block selection.
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck] and
// [> Initial and local tokens always selected].  For one query token of one
// GQA group (16 heads):
//   z[h, j] = score_scale * q_h . Mean_j            (visible kernels j)
//   g[j]    = (1/16) sum_h exp(z[h, j] - lse_h)     (exact two-pass LSE)
//   r[blk]  = max_j g[j] over kernels meeting the block (j in 4 blk - 1 .. 4 blk + 3)
//   top-k over r with forced initial/local blocks.
// Scores are kept in base 2 (z scaled by log2 e) so exp is a single ex2.
//
// q . Mean_j is a 16-row (heads) x 128 contraction against every kernel; it
// runs on the tensor cores (bf16 m16n8k16, fp32 accumulation) as
// q . hi_j + q . lo_j with the kernel means stored pre-split into two bf16
// planes, which keeps 16 significant bits of the fp32 mean.
//
// Two paths, same result:
//  * decode / verify (n_q <= 16): few (b, h_kv) groups and thousands of
//    kernels each, so each group's kernels are spread over a thread-block
//    cluster that exchanges LSE partials and block scores through
//    distributed shared memory (sel_cluster_kernel, one launch).
//  * prefill (n_q > 16): one warp per query token, TT tokens per CTA sharing
//    a TMA pipeline of 64-kernel hi/lo tiles, streamed twice (pass 1: LSE,
//    pass 2: normalised group mean and block maxima), then a warp top-k.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace infllmv2 {

namespace {

struct SelParams {
  int B, Hkv, Lmax, nq, ncmax, ncpad, nbmax, kmax;
  int topk, n_init, n_local, inc_forced;
  float scale2;
  const int32_t* kv_lens;
  int32_t* block_idx;  // [B*Hkv*nq][kmax]
  int32_t* n_sel;      // [B*Hkv*nq]
  float* r_buf;        // [B*Hkv*nq][nbmax] block scores (written when write_r)
  float* z;            // [B*Hkv*nq][16][ncpad] scratch  (decode path)
  int write_r;
  int stages;          // prefill path: pipeline depth
  uint32_t* status;
};

__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    m = -INFINITY;
    l = 0.f;
    return;
  }
  l = l * fast_exp2(m - M) + l2 * fast_exp2(m2 - M);
  m = M;
}

// Add two values of one row to a running (max, sum of exp2).
__device__ __forceinline__ void lse_add2(float& m, float& l, float x0, float x1) {
  const float mx = fmaxf(x0, x1);
  if (mx == -INFINITY) return;
  const float M = fmaxf(m, mx);
  l = l * fast_exp2(m - M) + fast_exp2(x0 - M) + fast_exp2(x1 - M);
  m = M;
}

// A fragments (16 rows x 128) of one query token from a swizzled 16-row tile.
__device__ __forceinline__ void load_q_frags(uint32_t (&a)[8][4], uint32_t tile, int lane) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldmatrix_x4(a[ks], tile + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4), 16));
}

// z for one n-tile (8 kernels at tile row n0) of a hi/lo tile with `rows` rows.
// Four accumulators (hi/lo x even/odd k-step) keep the 16 MMAs in four short
// dependency chains instead of one long one.
__device__ __forceinline__ void score_ntile(float (&acc)[4], const uint32_t (&a)[8][4],
                                            uint32_t hi, uint32_t lo, int n0, int rows, int lane) {
  float c[4][4];
#pragma unroll
  for (int x = 0; x < 4; ++x) c[x][0] = c[x][1] = c[x][2] = c[x][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t bh[4], bl[4];
    const uint32_t off = swz128_offset(n0 + (lane & 7), 4 * kk + (lane >> 3), rows);
    ldmatrix_x4(bh, hi + off);
    ldmatrix_x4(bl, lo + off);
    mma_bf16_16816(c[0], a[2 * kk], bh[0], bh[1]);
    mma_bf16_16816(c[1], a[2 * kk], bl[0], bl[1]);
    mma_bf16_16816(c[2], a[2 * kk + 1], bh[2], bh[3]);
    mma_bf16_16816(c[3], a[2 * kk + 1], bl[2], bl[3]);
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] = (c[0][e] + c[2][e]) + (c[1][e] + c[3][e]);
}

// ------------------------------------------------------------- decode path --
//
// One thread-block cluster of C CTAs per (b, h_kv) group; the group's n_q
// query tokens (<= 16) are scored together.  The blocks 0 .. floor(i/m) are
// cut into C contiguous ranges of 16-block groups; CTA r owns the matching
// 64-kernel chunks (kernels of blocks [16k, 16k+16) are 64k-1 .. 64k+63).
//   phase A  TMA-stream the CTA's hi/lo chunks, z = q.Mean (tensor cores),
//            z to scratch (L2), per-row (max, sum) partials in shared memory.
//   sync     partials of all CTAs read through distributed shared memory
//            -> exact LSE per head.
//   phase B  g = mean_h exp2(z - lse) and the block maxima of the CTA's range,
//            with the range's candidate count and best score.
//   top-k    (cluster-wide, three barriers) each CTA histograms its blocks'
//            scores by leading bits against the cluster's best score; the
//            summed histogram gives the bin holding the k-th best score;
//            the few candidates at or above it are gathered by the CTA that
//            owns token t (t mod C), ranked exactly by (score desc, index
//            asc), and written ascending with the forced blocks.
// No global partials, tickets or memsets: the cluster barriers order it all.

constexpr int kClThreads = 256;   // 8 warps: one 8-kernel n-tile each per chunk
constexpr int kClChunk = 64;      // kernels per stage (= 16 blocks)
constexpr int kClStages = 2;   // small enough for two CTAs per SM
constexpr int kClStageBytes = 2 * kClChunk * 256;

// Per-token top-k bookkeeping shared across the cluster.
struct ClTok {
  int n_cand, n_forced, top, n_take;   // local counts / max (then global in `glob`)
  int bnd, n_surv, n_lsurv, pad;
};

struct ClLayout {
  int stage, q, wpart, cpart, lse, g, rsl, tok, glob, hist, ghist, lsurv, gsurv, sel, bar, total, rsl_stride;
};

__host__ __device__ inline ClLayout cl_layout(int C, int nq, int nbmax, int kmax) {
  ClLayout l;
  const int groups = (nbmax + 15) / 16;
  const int per_cta = (groups + C - 1) / C;     // 16-block groups per CTA (upper bound)
  l.rsl_stride = per_cta * 16;
  l.stage = 0;
  l.q = kClStages * kClStageBytes;
  l.wpart = l.q + nq * 4096;
  l.cpart = l.wpart + 8 * nq * kGroup * 8;
  l.lse = l.cpart + nq * kGroup * 8;
  l.g = l.lse + nq * kGroup * 4;
  l.rsl = l.g + (per_cta * kClChunk + 4) * 4;
  l.tok = (l.rsl + nq * l.rsl_stride * 4 + 15) & ~15;       // local ClTok per token
  l.glob = l.tok + nq * static_cast<int>(sizeof(ClTok));     // cluster-wide ClTok per token
  l.hist = l.glob + nq * static_cast<int>(sizeof(ClTok));    // local histograms [nq][256]
  l.ghist = l.hist + nq * 256 * 4;                           // cluster histograms [nq][256]
  l.lsurv = (l.ghist + nq * 256 * 4 + 15) & ~15;             // local survivors [nq][rsl_stride]
  l.gsurv = l.lsurv + nq * l.rsl_stride * 8;                 // gathered survivors [nbmax]
  l.sel = l.gsurv + nbmax * 8;                               // chosen blocks [kmax]
  l.bar = (l.sel + kmax * 4 + 15) & ~15;
  l.total = l.bar + (2 * kClStages + 1) * 8;
  return l;
}

// Scores are binned by their leading bits (sign, exponent, 6 mantissa bits):
// a bin spans about 1.1 % of the score.
constexpr int kClBinShift = 17;

// A block competes for the scored slots if it is not forced and some visible
// kernel touches it.
__device__ __forceinline__ bool cl_candidate(int j, int c, float r, int n_init, int n_local) {
  return j >= n_init && j <= c - n_local && r > -INFINITY;
}

__device__ __forceinline__ int cl_bin(uint32_t top, float r) {
  return static_cast<int>(min(255u, top - (float_to_ordered(r) >> kClBinShift)));
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
  ClTok* tok = reinterpret_cast<ClTok*>(smem + lay.tok);         // [nq] this CTA's slice
  ClTok* glob = reinterpret_cast<ClTok*>(smem + lay.glob);       // [nq] whole cluster
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + lay.hist);    // [nq][256]
  uint32_t* ghist = reinterpret_cast<uint32_t*>(smem + lay.ghist);  // [nq][256]
  unsigned long long* lsurv = reinterpret_cast<unsigned long long*>(smem + lay.lsurv);  // [nq][rsl_stride]
  unsigned long long* gsurv = reinterpret_cast<unsigned long long*>(smem + lay.gsurv);  // [nbmax]
  int* selbuf = reinterpret_cast<int*>(smem + lay.sel);          // [kmax]
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
  for (int e = tid; e < nq * 256; e += kClThreads) hist[e] = 0u;
  for (int e = tid; e < nq; e += kClThreads) tok[e] = ClTok{0, 0, 0, 0, 0, 0, 0, 0};
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
  const int k0 = (rank * groups) / C, k1 = ((rank + 1) * groups) / C;
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
        float s = 0.f;
#pragma unroll
        for (int hh = 0; hh < kGroup; ++hh) s += fast_exp2(__ldcg(zu + static_cast<size_t>(hh) * p.ncpad + k) - lt[hh]);
        gbuf[k - klo] = s * (1.0f / kGroup);
      }
      __syncthreads();
    }
    int my_cand = 0;
    uint32_t my_top = 0;
    for (int j = jb0 + tid; j < jb1; j += kClThreads) {
      const int a0 = max(0, 4 * j - 1), e0 = min(nvis - 1, 4 * j + 3);
      float r = -INFINITY;
      for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - klo]);
      rsl[t * lay.rsl_stride + (j - jb0)] = r;
      if (p.write_r) p.r_buf[(unit0 + t) * p.nbmax + j] = r;
      if (cl_candidate(j, c, r, p.n_init, p.n_local)) {
        ++my_cand;
        my_top = max(my_top, float_to_ordered(r) >> kClBinShift);
      }
    }
    my_cand = __reduce_add_sync(0xffffffffu, my_cand);
    my_top = __reduce_max_sync(0xffffffffu, my_top);
    if (lane == 0 && my_cand > 0) {
      atomicAdd(&tok[t].n_cand, my_cand);
      atomicMax(&tok[t].top, static_cast<int>(my_top));
    }
    __syncthreads();
  }
  cluster_sync();

  // ------------------------------------------------------------- top-k --
  // 1. cluster-wide candidate count and best leading bits; forced blocks are
  //    known in closed form (first n_init, the n_local ending at block c).
  for (int t = tid; t < nq; t += kClThreads) {
    uint32_t nc[C], tp[C];
#pragma unroll
    for (int q = 0; q < C; ++q) {
      nc[q] = ld_dsmem_u32(dsmem_addr(&tok[t].n_cand, q));
      tp[q] = ld_dsmem_u32(dsmem_addr(&tok[t].top, q));
    }
    int ncand = 0, top = 0;
#pragma unroll
    for (int q = 0; q < C; ++q) {
      ncand += static_cast<int>(nc[q]);
      top = max(top, static_cast<int>(tp[q]));
    }
    const int c = (L - nq + t) / kBlock;
    const int n_first = min(p.n_init, c + 1);
    const int n_forced = n_first + max(0, c - max(n_first, c - p.n_local + 1) + 1);
    const int n_take = max(0, p.inc_forced ? p.topk - n_forced : p.topk);
    glob[t] = ClTok{ncand, n_forced, top, n_take, 255, 0, 0, 0};
  }
  __syncthreads();
  // 2. local histograms of the bins (0 = best bin) where a threshold is needed.
  for (int t = 0; t < nq; ++t) {
    const ClTok gt = glob[t];
    if (gt.n_take > 0 && gt.n_cand > gt.n_take) {
      const int c = (L - nq + t) / kBlock;
      const int jb0 = 16 * k0, jb1 = min(16 * k1, c + 1);
      for (int j = jb0 + tid; j < jb1; j += kClThreads) {
        const float r = rsl[t * lay.rsl_stride + (j - jb0)];
        if (cl_candidate(j, c, r, p.n_init, p.n_local))
          atomicAdd(&hist[t * 256 + cl_bin(static_cast<uint32_t>(gt.top), r)], 1u);
      }
    }
  }
  cluster_sync();
  // 3. cluster histograms -> the bin holding the n_take-th best score; every
  //    candidate at or above it survives.
  for (int t = 0; t < nq; ++t) {
    const ClTok gt = glob[t];
    if (gt.n_take > 0 && gt.n_cand > gt.n_take) {
      uint32_t hv[C];
#pragma unroll
      for (int q = 0; q < C; ++q) hv[q] = ld_dsmem_u32(dsmem_addr(&hist[t * 256 + tid], q));
      uint32_t v = 0;
#pragma unroll
      for (int q = 0; q < C; ++q) v += hv[q];
      ghist[t * 256 + tid] = v;
    }
  }
  __syncthreads();
  for (int t = warp; t < nq; t += kClThreads / 32) {
    const ClTok gt = glob[t];
    int bnd = gt.n_take > 0 ? 255 : -1;
    if (gt.n_take > 0 && gt.n_cand > gt.n_take) {
      int cnt[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        cnt[k] = static_cast<int>(ghist[t * 256 + 8 * lane + k]);
        tot += cnt[k];
      }
      int run = warp_inclusive_scan(tot) - tot;
      int found = -1;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (run < gt.n_take && run + cnt[k] >= gt.n_take) found = 8 * lane + k;
        run += cnt[k];
      }
      bnd = __reduce_max_sync(0xffffffffu, found);
    }
    if (lane == 0) glob[t].bnd = bnd;
  }
  __syncthreads();
  for (int t = 0; t < nq; ++t) {
    const ClTok gt = glob[t];
    if (gt.bnd < 0) continue;
    const int c = (L - nq + t) / kBlock;
    const int jb0 = 16 * k0, jb1 = min(16 * k1, c + 1);
    for (int j = jb0 + tid; j < jb1; j += kClThreads) {
      const float r = rsl[t * lay.rsl_stride + (j - jb0)];
      if (cl_candidate(j, c, r, p.n_init, p.n_local) && cl_bin(static_cast<uint32_t>(gt.top), r) <= gt.bnd) {
        const int pos = atomicAdd(&tok[t].n_lsurv, 1);
        lsurv[t * lay.rsl_stride + pos] =
            (static_cast<unsigned long long>(float_to_ordered(r)) << 32) | static_cast<uint32_t>(~j);
      }
    }
  }
  cluster_sync();
  // 4. the CTA that owns token t gathers the survivors, ranks them by
  //    (score desc, index asc), and writes forced + best blocks ascending.
  __shared__ int offs[C + 1];
  for (int t = rank; t < nq; t += C) {
    const ClTok gt = glob[t];
    const int c = (L - nq + t) / kBlock;
    const int nb = c + 1;
    if (warp == 0) {
      const int v = lane < C ? static_cast<int>(ld_dsmem_u32(dsmem_addr(&tok[t].n_lsurv, lane))) : 0;
      const int incl = warp_inclusive_scan(v);
      if (lane < C) offs[lane] = incl - v;
      if (lane == C - 1) offs[C] = incl;
    }
    if (tid == 0) {   // forced blocks, ascending and without duplicates
      const int n_first = min(p.n_init, nb);
      int n = 0;
      for (int j = 0; j < n_first; ++j) selbuf[n++] = j;
      for (int j = max(n_first, c - p.n_local + 1); j <= c; ++j) selbuf[n++] = j;
    }
    __syncthreads();
    const int n_surv = offs[C];
    // One remote load per thread: survivor x lives in CTA q, slot x - offs[q].
    for (int x = tid; x < n_surv; x += kClThreads) {
      int q = 0;
      while (q + 1 < C && offs[q + 1] <= x) ++q;
      gsurv[x] = ld_dsmem_u64(dsmem_addr(&lsurv[t * lay.rsl_stride + (x - offs[q])], q));
    }
    __syncthreads();
    for (int x = tid; x < n_surv; x += kClThreads) {
      const unsigned long long me = gsurv[x];
      int rk = 0;
      int y = 0;
      for (; y + 4 <= n_surv; y += 4)
        rk += (gsurv[y] > me) + (gsurv[y + 1] > me) + (gsurv[y + 2] > me) + (gsurv[y + 3] > me);
      for (; y < n_surv; ++y) rk += (gsurv[y] > me) ? 1 : 0;
      if (rk < gt.n_take) selbuf[gt.n_forced + rk] = static_cast<int>(~static_cast<uint32_t>(me & 0xffffffffu));
    }
    __syncthreads();
    const int n_total = min(p.kmax, gt.n_forced + min(gt.n_take, n_surv));
    int32_t* out = p.block_idx + (unit0 + t) * p.kmax;
    for (int x = tid; x < n_total; x += kClThreads) {
      const int v = selbuf[x];
      int pos = 0;
      for (int y = 0; y < n_total; ++y) pos += (selbuf[y] < v) ? 1 : 0;
      out[pos] = v;
    }
    for (int x = n_total + tid; x < p.kmax; x += kClThreads) out[x] = -1;
    if (tid == 0) p.n_sel[unit0 + t] = n_total;
    if (p.write_r)
      for (int j = nb + tid; j < p.nbmax; j += kClThreads) p.r_buf[(unit0 + t) * p.nbmax + j] = -INFINITY;
    __syncthreads();
  }
  cluster_sync();
}

// ------------------------------------------------------------ prefill path --

constexpr int kPrefTokens = 8;                  // warps (query tokens) per CTA
constexpr int kPrefChunk = 64;                  // kernels per pipeline stage
constexpr int kPrefStageBytes = 2 * kPrefChunk * 256;  // hi + lo tile

struct PrefLayout {
  int stage_off, q_off, r_off, flag_off, gbuf_off, tk_off, bar_off, total;
};

__host__ __device__ inline PrefLayout pref_layout(int stages, int nbmax) {
  PrefLayout l;
  l.stage_off = 0;
  l.q_off = stages * kPrefStageBytes;
  l.r_off = l.q_off + kPrefTokens * 4096;
  l.flag_off = l.r_off + kPrefTokens * nbmax * 4;
  l.gbuf_off = (l.flag_off + kPrefTokens * nbmax + 15) & ~15;
  l.tk_off = l.gbuf_off + kPrefTokens * 68 * 4;
  l.bar_off = (l.tk_off + kPrefTokens * static_cast<int>(sizeof(TopkScratch<32>)) + 15) & ~15;
  l.total = l.bar_off + (2 * stages + 1) * 8;
  return l;
}

__global__ void __launch_bounds__(kPrefTokens * 32)
    sel_prefill_kernel(const __grid_constant__ CUtensorMap kc_map,
                       const __grid_constant__ CUtensorMap q_map, SelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int S = p.stages;
  const PrefLayout lay = pref_layout(S, p.nbmax);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.Hkv + h;
  const int nq = p.nq;
  const int t = blockIdx.x * kPrefTokens + warp;
  const bool active = t < nq;
  const size_t u = static_cast<size_t>(bh) * nq + t;

  float* r_w = reinterpret_cast<float*>(smem + lay.r_off) + warp * p.nbmax;
  uint8_t* flag_w = smem + lay.flag_off + warp * p.nbmax;
  float* gbuf = reinterpret_cast<float*>(smem + lay.gbuf_off) + warp * 68;
  TopkScratch<32>& tk = reinterpret_cast<TopkScratch<32>*>(smem + lay.tk_off)[warp];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
  uint64_t* empty = full + S;
  uint64_t* qbar = empty + S;

  const int L = p.kv_lens[b];
  if (L < nq || L > p.Lmax) {
    if (active) {
      for (int k = lane; k < p.kmax; k += 32) p.block_idx[u * p.kmax + k] = -1;
      if (p.write_r)
        for (int j = lane; j < p.nbmax; j += 32) p.r_buf[u * p.nbmax + j] = -INFINITY;
      if (lane == 0) {
        p.n_sel[u] = 0;
        atomicOr(p.status, kStatusBadKvLen);
      }
    }
    return;
  }
  const int t_last = min(nq - 1, static_cast<int>(blockIdx.x) * kPrefTokens + kPrefTokens - 1);
  const int nvis_max = n_complete_kernels(L - nq + t_last + 1);
  const int nch = (nvis_max + kPrefChunk - 1) / kPrefChunk;
  const int total = 2 * nch;
  const int i_t = L - nq + (active ? t : t_last);
  const int c_t = i_t / kBlock;
  const int nvis_t = n_complete_kernels(i_t + 1);

  for (int j = lane; j < p.nbmax; j += 32) r_w[j] = -INFINITY;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPrefTokens);
    }
    mbar_init(qbar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int it) {
    const int ch = it % nch, stage = it % S;
    uint8_t* dst = smem + lay.stage_off + stage * kPrefStageBytes;
    mbar_arrive_expect_tx(&full[stage], kPrefStageBytes);
    const int row_hi = (bh * 2 + 0) * p.ncmax + ch * kPrefChunk;
    const int row_lo = (bh * 2 + 1) * p.ncmax + ch * kPrefChunk;
    tma_load_2d(dst, &kc_map, 0, row_hi, &full[stage]);
    tma_load_2d(dst + 8192, &kc_map, 64, row_hi, &full[stage]);
    tma_load_2d(dst + 16384, &kc_map, 0, row_lo, &full[stage]);
    tma_load_2d(dst + 24576, &kc_map, 64, row_lo, &full[stage]);
  };

  if (threadIdx.x == 0) {
    const int n_act = min(kPrefTokens, nq - static_cast<int>(blockIdx.x) * kPrefTokens);
    mbar_arrive_expect_tx(qbar, n_act * 4096);
    const int Hq = p.Hkv * kGroup;
    for (int w = 0; w < n_act; ++w) {
      const int row = (b * nq + blockIdx.x * kPrefTokens + w) * Hq + h * kGroup;
      tma_load_2d(smem + lay.q_off + w * 4096, &q_map, 0, row, qbar);
      tma_load_2d(smem + lay.q_off + w * 4096 + 2048, &q_map, 64, row, qbar);
    }
    for (int it = 0; it < min(S, total); ++it) issue(it);
  }
  bool ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  if (!ok) return;

  uint32_t a[8][4];
  if (active) load_q_frags(a, smem_u32(smem + lay.q_off + warp * 4096), lane);
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
  float lse_g = -INFINITY, lse_g8 = -INFINITY;

#pragma unroll 1
  for (int it = 0; it < total; ++it) {
    const int stage = it % S;
    const uint32_t ph = static_cast<uint32_t>(it / S) & 1u;
    const int pass = it / nch, ch = it % nch;
    const int kbase = ch * kPrefChunk;
    if (pass == 1 && ch == 0) {
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        lse_merge(m0, l0, __shfl_xor_sync(0xffffffffu, m0, o), __shfl_xor_sync(0xffffffffu, l0, o));
        lse_merge(m1, l1, __shfl_xor_sync(0xffffffffu, m1, o), __shfl_xor_sync(0xffffffffu, l1, o));
      }
      lse_g = (m0 == -INFINITY) ? -INFINITY : m0 + fast_log2(l0);
      lse_g8 = (m1 == -INFINITY) ? -INFINITY : m1 + fast_log2(l1);
    }
    ok = mbar_wait(&full[stage], ph, p.status);
    if (!__all_sync(0xffffffffu, ok)) break;
    if (active && kbase < nvis_t) {
      const uint32_t hi_b = smem_u32(smem + lay.stage_off + stage * kPrefStageBytes);
      const uint32_t lo_b = hi_b + 16384;
#pragma unroll 2
      for (int nt = 0; nt < 8; ++nt) {
        float acc[4];
        score_ntile(acc, a, hi_b, lo_b, nt * 8, kPrefChunk, lane);
        const int kj = kbase + nt * 8 + 2 * tq;
        const bool v0 = kj < nvis_t, v1 = kj + 1 < nvis_t;
        const float x0 = acc[0] * p.scale2, x1 = acc[1] * p.scale2;
        const float x2 = acc[2] * p.scale2, x3 = acc[3] * p.scale2;
        if (pass == 0) {
          lse_add2(m0, l0, v0 ? x0 : -INFINITY, v1 ? x1 : -INFINITY);
          lse_add2(m1, l1, v0 ? x2 : -INFINITY, v1 ? x3 : -INFINITY);
        } else {
          float s0 = (v0 ? fast_exp2(x0 - lse_g) : 0.f) + (v0 ? fast_exp2(x2 - lse_g8) : 0.f);
          float s1 = (v1 ? fast_exp2(x1 - lse_g) : 0.f) + (v1 ? fast_exp2(x3 - lse_g8) : 0.f);
#pragma unroll
          for (int o = 4; o <= 16; o <<= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
          }
          if (g == 0) {
            gbuf[1 + nt * 8 + 2 * tq] = s0 * (1.0f / kGroup);
            gbuf[2 + nt * 8 + 2 * tq] = s1 * (1.0f / kGroup);
          }
        }
      }
      if (pass == 1) {
        __syncwarp();
        if (lane < 16) {
          const int j = kbase / 4 + lane;
          if (j <= c_t) {
            const int a0 = max(0, 4 * j - 1), e0 = min(nvis_t - 1, 4 * j + 3);
            float r = -INFINITY;
            for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - kbase + 1]);
            r_w[j] = r;
          }
        }
        __syncwarp();
        if (lane == 0) gbuf[0] = gbuf[64];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (threadIdx.x == 0 && it + S < total) {
      if (mbar_wait(&empty[stage], ph, p.status)) issue(it + S);
    }
    __syncwarp();
  }

  if (!active) return;
  __syncwarp();
  if (p.write_r)
    for (int j = lane; j < p.nbmax; j += 32) p.r_buf[u * p.nbmax + j] = r_w[j];
  select_topk<32, true>(r_w, flag_w, c_t + 1, p.n_init, p.n_local, p.topk, p.inc_forced != 0,
                        p.kmax, p.block_idx + u * p.kmax, p.n_sel + u, tk, lane);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

size_t decode_ncpad(const Shape& s) { return static_cast<size_t>((s.ncmax + kClChunk - 1) / kClChunk) * kClChunk; }

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

size_t select_workspace_bytes(const Shape& s) {
  if (s.nq <= kSelDecodeMaxNq) {
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
    return align256(units * kGroup * decode_ncpad(s) * sizeof(float));
  }
  return 0;  // the prefill path keeps everything on chip
}

cudaError_t launch_select(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                          const void* q, const int32_t* kv_lens, int32_t* block_idx,
                          int32_t* n_sel, float* block_scores, void* ws, uint32_t* status,
                          cudaStream_t st) {
  (void)q;
  SelParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.ncmax = s.ncmax;
  p.nbmax = s.nbmax;
  p.kmax = s.kmax;
  p.topk = s.topk;
  p.n_init = s.n_init;
  p.n_local = s.n_local;
  p.inc_forced = s.inc_forced;
  p.scale2 = s.score_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.status = status;
  p.write_r = block_scores != nullptr;
  p.r_buf = block_scores;

  if (s.nq <= kSelDecodeMaxNq) {
    p.ncpad = static_cast<int>(decode_ncpad(s));
    p.z = static_cast<float*>(ws);
    bool unsupported = false;
    cudaError_t e = cudaSuccess;
    // 16-CTA clusters when every group's cluster can be resident at once.
    if (s.B * s.Hkv * 16 <= 2 * device_sm_count()) {
      e = launch_cluster<16>(s, kc_map, q_map, p, st, &unsupported);
      if (e != cudaSuccess || !unsupported) return e;
    }
    e = launch_cluster<8>(s, kc_map, q_map, p, st, &unsupported);
    if (e == cudaSuccess && unsupported) return cudaErrorInvalidConfiguration;
    return e;
  }

  int stages = 3;
  PrefLayout lay = pref_layout(stages, s.nbmax);
  if (lay.total + 1024 > 227 * 1024) {
    stages = 2;
    lay = pref_layout(stages, s.nbmax);
  }
  if (lay.total + 1024 > 227 * 1024) return cudaErrorInvalidConfiguration;
  p.stages = stages;
  const int psmem = lay.total + 1024;
  cudaError_t e = cudaFuncSetAttribute(sel_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       psmem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.nq + kPrefTokens - 1) / kPrefTokens, s.Hkv, s.B);
  sel_prefill_kernel<<<grid, kPrefTokens * 32, psmem, st>>>(kc_map, q_map, p);
  return cudaGetLastError();
}

}  // namespace infllmv2
