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
//  * decode / verify (n_q <= 16): few (b, h_kv, t) units and up to thousands
//    of kernels each, so kernels are split over CTAs.  sel_score_kernel loads
//    a 128-kernel hi/lo tile and the group's queries with TMA, writes z and
//    per-chunk (max, sum) partials; sel_reduce_kernel merges the partials
//    into lse, forms g and the block maxima for a 64-block range, and the last
//    CTA of each unit (atomic ticket) runs the top-k.
//  * prefill (n_q > 16): one warp per query token, TT tokens per CTA sharing
//    a TMA pipeline of 64-kernel hi/lo tiles, streamed twice (pass 1: LSE,
//    pass 2: normalised group mean and block maxima), then a warp top-k.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace infllmv2 {

namespace {

struct SelParams {
  int B, Hkv, Lmax, nq, ncmax, ncpad, nbmax, kmax, n_chunks;
  int topk, n_init, n_local, inc_forced;
  float scale2;
  const int32_t* kv_lens;
  int32_t* block_idx;  // [B*Hkv*nq][kmax]
  int32_t* n_sel;      // [B*Hkv*nq]
  float* r_buf;        // [B*Hkv*nq][nbmax]
  float* z;            // [B*Hkv*nq][16][ncpad]      (decode path)
  float2* part;        // [B*Hkv*nq][16][n_chunks]   (decode path)
  uint32_t* counters;  // [B*Hkv*nq]                 (decode path)
  int write_r;         // prefill path: write r to r_buf
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
__device__ __forceinline__ void score_ntile(float (&acc)[4], const uint32_t (&a)[8][4],
                                            uint32_t hi, uint32_t lo, int n0, int rows, int lane) {
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    uint32_t bh[4], bl[4];
    const uint32_t off = swz128_offset(n0 + (lane & 7), 4 * kk + (lane >> 3), rows);
    ldmatrix_x4(bh, hi + off);
    ldmatrix_x4(bl, lo + off);
    mma_bf16_16816(acc, a[2 * kk], bh[0], bh[1]);
    mma_bf16_16816(acc, a[2 * kk], bl[0], bl[1]);
    mma_bf16_16816(acc, a[2 * kk + 1], bh[2], bh[3]);
    mma_bf16_16816(acc, a[2 * kk + 1], bl[2], bl[3]);
  }
}

// ------------------------------------------------------------- decode path --

constexpr int kScoreThreads = 128;  // 4 warps x 32 kernels
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kScoreThreads)
    sel_score_kernel(const __grid_constant__ CUtensorMap kc_map,
                     const __grid_constant__ CUtensorMap q_map, SelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nq = p.nq;
  uint8_t* hi_t = smem;                 // 128 rows x 128 bf16, swizzled, 32 KB
  uint8_t* lo_t = smem + 32768;
  uint8_t* q_t = smem + 65536;          // nq tiles of 16 rows, 4 KB each
  float2* part_s = reinterpret_cast<float2*>(q_t + nq * 4096);   // [4][nq*16]
  uint64_t* bar = reinterpret_cast<uint64_t*>(part_s + 4 * nq * 16);

  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int L = p.kv_lens[b];
  if (L < nq || L > p.Lmax) {
    if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(p.status, kStatusBadKvLen);
    return;
  }
  const int nc = n_complete_kernels(L);
  const int j0 = blockIdx.x * kSelChunk;
  if (j0 >= nc) return;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, 2 * kSelChunk * 256 + nq * 4096);
    const int row_hi = (bh * 2 + 0) * p.ncmax + j0;
    const int row_lo = (bh * 2 + 1) * p.ncmax + j0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {      // column halves (64 dims)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {          // row halves (64 kernels)
        tma_load_2d(hi_t + half * 16384 + rh * 8192, &kc_map, half * 64, row_hi + rh * 64, bar);
        tma_load_2d(lo_t + half * 16384 + rh * 8192, &kc_map, half * 64, row_lo + rh * 64, bar);
      }
    }
    const int Hq = p.Hkv * kGroup;
    for (int t = 0; t < nq; ++t) {
      const int row = (b * nq + t) * Hq + h * kGroup;
      tma_load_2d(q_t + t * 4096, &q_map, 0, row, bar);
      tma_load_2d(q_t + t * 4096 + 2048, &q_map, 64, row, bar);
    }
  }
  const bool ok = __syncthreads_and(mbar_wait(bar, 0, p.status));
  if (!ok) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const uint32_t hi_b = smem_u32(hi_t), lo_b = smem_u32(lo_t), q_b = smem_u32(q_t);
  const size_t unit0 = static_cast<size_t>(bh) * nq;

  for (int t = 0; t < nq; ++t) {
    const int i = L - nq + t;
    const int nvis = n_complete_kernels(i + 1);
    uint32_t a[8][4];
    load_q_frags(a, q_b + t * 4096, lane);
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    float* zrow = p.z + ((unit0 + t) * kGroup + g) * static_cast<size_t>(p.ncpad);
#pragma unroll 1
    for (int nt = 0; nt < 4; ++nt) {
      const int n0 = warp * 32 + nt * 8;
      float acc[4];
      score_ntile(acc, a, hi_b, lo_b, n0, kSelChunk, lane);
      const int kj = j0 + n0 + 2 * tq;
      const bool v0 = kj < nvis, v1 = kj + 1 < nvis;
      const float z0 = v0 ? acc[0] * p.scale2 : -INFINITY;
      const float z1 = v1 ? acc[1] * p.scale2 : -INFINITY;
      const float z2 = v0 ? acc[2] * p.scale2 : -INFINITY;
      const float z3 = v1 ? acc[3] * p.scale2 : -INFINITY;
      *reinterpret_cast<float2*>(zrow + kj) = make_float2(z0, z1);
      *reinterpret_cast<float2*>(zrow + 8 * static_cast<size_t>(p.ncpad) + kj) = make_float2(z2, z3);
      lse_add2(m0, l0, z0, z1);
      lse_add2(m1, l1, z2, z3);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      lse_merge(m0, l0, __shfl_xor_sync(0xffffffffu, m0, o), __shfl_xor_sync(0xffffffffu, l0, o));
      lse_merge(m1, l1, __shfl_xor_sync(0xffffffffu, m1, o), __shfl_xor_sync(0xffffffffu, l1, o));
    }
    if (tq == 0) {
      part_s[(warp * nq + t) * kGroup + g] = make_float2(m0, l0);
      part_s[(warp * nq + t) * kGroup + g + 8] = make_float2(m1, l1);
    }
  }
  __syncthreads();
  for (int row = threadIdx.x; row < nq * kGroup; row += kScoreThreads) {
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 v = part_s[w * nq * kGroup + row];
      lse_merge(m, l, v.x, v.y);
    }
    p.part[(unit0 * kGroup + row) * p.n_chunks + blockIdx.x] = make_float2(m, l);
  }
}

__global__ void __launch_bounds__(kReduceThreads) sel_reduce_kernel(SelParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ float lse2[kGroup];
  __shared__ float gs[4 * kSelReduceBlocks + 4];
  __shared__ TopkScratch<kReduceThreads> tk;
  __shared__ int is_last;
  float* r_s = reinterpret_cast<float*>(dsm);
  uint8_t* flag_s = reinterpret_cast<uint8_t*>(r_s + p.nbmax);

  const int tid = threadIdx.x;
  const int u = blockIdx.y;
  const int bh = u / p.nq, t = u % p.nq;
  const int b = bh / p.Hkv;
  const int L = p.kv_lens[b];
  int32_t* idx_out = p.block_idx + static_cast<size_t>(u) * p.kmax;
  float* r_row = p.r_buf + static_cast<size_t>(u) * p.nbmax;
  const int jb0 = blockIdx.x * kSelReduceBlocks;
  const int jend = min(p.nbmax, jb0 + kSelReduceBlocks);

  if (L < p.nq || L > p.Lmax) {
    for (int j = jb0 + tid; j < jend; j += kReduceThreads) r_row[j] = -INFINITY;
    if (blockIdx.x == 0) {
      for (int k = tid; k < p.kmax; k += kReduceThreads) idx_out[k] = -1;
      if (tid == 0) {
        p.n_sel[u] = 0;
        atomicOr(p.status, kStatusBadKvLen);
      }
    }
    return;
  }
  const int i = L - p.nq + t;
  const int c = i / kBlock;
  const int nb = c + 1;
  const int nvis = n_complete_kernels(i + 1);
  if (jb0 >= nb) {
    for (int j = jb0 + tid; j < jend; j += kReduceThreads) r_row[j] = -INFINITY;
    return;
  }
  const int jb1 = min(nb, jb0 + kSelReduceBlocks);

  {  // lse of each head from the scoring CTAs' partials
    const int head = tid >> 4, sub = tid & 15;
    const int n_sc = (nvis + kSelChunk - 1) / kSelChunk;
    float m = -INFINITY, l = 0.f;
    const float2* pp = p.part + (static_cast<size_t>(u) * kGroup + head) * p.n_chunks;
    for (int ch = sub; ch < n_sc; ch += 16) {
      const float2 v = __ldcg(pp + ch);
      lse_merge(m, l, v.x, v.y);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
      lse_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if (sub == 0) lse2[head] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  const int klo = max(0, 4 * jb0 - 1);
  const int khi = min(nvis, 4 * (jb1 - 1) + 4);
  const float* zu = p.z + static_cast<size_t>(u) * kGroup * p.ncpad;
  for (int k = klo + tid; k < khi; k += kReduceThreads) {
    float s = 0.f;
#pragma unroll
    for (int hh = 0; hh < kGroup; ++hh) s += fast_exp2(__ldcg(zu + static_cast<size_t>(hh) * p.ncpad + k) - lse2[hh]);
    gs[k - klo] = s * (1.0f / kGroup);
  }
  __syncthreads();
  for (int j = jb0 + tid; j < jend; j += kReduceThreads) {
    float r = -INFINITY;
    if (j < jb1) {
      const int a = max(0, 4 * j - 1), e = min(nvis - 1, 4 * j + 3);
      for (int k = a; k <= e; ++k) r = fmaxf(r, gs[k - klo]);
    }
    r_row[j] = r;
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t nparts = (nb + kSelReduceBlocks - 1) / kSelReduceBlocks;
    const uint32_t prev = atomicAdd(&p.counters[u], 1u);
    is_last = (prev == nparts - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid == 0) p.counters[u] = 0;
  for (int j = tid; j < nb; j += kReduceThreads) r_s[j] = __ldcg(r_row + j);
  __syncthreads();
  select_topk<kReduceThreads, false>(r_s, flag_s, nb, p.n_init, p.n_local, p.topk, p.inc_forced != 0,
                                     p.kmax, idx_out, p.n_sel + u, tk, tid);
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
#pragma unroll 1
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

struct DecodeWs {
  size_t counters, part, z, r, total;
};

DecodeWs decode_ws(const Shape& s) {
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
  const int n_chunks = (s.ncmax + kSelChunk - 1) / kSelChunk;
  const size_t ncpad = static_cast<size_t>(n_chunks) * kSelChunk;
  DecodeWs w;
  w.counters = 0;
  w.part = align256(units * 4);
  w.z = w.part + align256(units * kGroup * n_chunks * sizeof(float2));
  w.r = w.z + align256(units * kGroup * ncpad * sizeof(float));
  w.total = w.r + align256(units * s.nbmax * sizeof(float));
  return w;
}

}  // namespace

size_t select_workspace_bytes(const Shape& s) {
  if (s.nq <= kSelDecodeMaxNq) return decode_ws(s).total;
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
  uint8_t* base = static_cast<uint8_t*>(ws);

  if (s.nq <= kSelDecodeMaxNq) {
    const DecodeWs w = decode_ws(s);
    p.n_chunks = (s.ncmax + kSelChunk - 1) / kSelChunk;
    p.ncpad = p.n_chunks * kSelChunk;
    p.counters = reinterpret_cast<uint32_t*>(base + w.counters);
    p.part = reinterpret_cast<float2*>(base + w.part);
    p.z = reinterpret_cast<float*>(base + w.z);
    p.r_buf = block_scores ? block_scores : reinterpret_cast<float*>(base + w.r);
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
    cudaError_t e = cudaMemsetAsync(p.counters, 0, units * 4, st);
    if (e != cudaSuccess) return e;
    if (p.n_chunks > 0) {
      const int smem = 1024 + 65536 + s.nq * 4096 + 4 * s.nq * kGroup * 8 + 16;
      e = cudaFuncSetAttribute(sel_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      sel_score_kernel<<<dim3(p.n_chunks, s.B * s.Hkv), kScoreThreads, smem, st>>>(kc_map, q_map, p);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    const int rsmem = s.nbmax * 5 + 16;
    e = cudaFuncSetAttribute(sel_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, rsmem);
    if (e != cudaSuccess) return e;
    const int nrc = (s.nbmax + kSelReduceBlocks - 1) / kSelReduceBlocks;
    sel_reduce_kernel<<<dim3(nrc, static_cast<unsigned>(units)), kReduceThreads, rsmem, st>>>(p);
    return cudaGetLastError();
  }

  p.write_r = block_scores != nullptr;
  p.r_buf = block_scores;
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
