// Stage 3 of InfLLM v2 for decode and speculative verification: exact
// softmax attention over the selected KV blocks of each query token.
//
// [InfLLM v2 > Block-level key-value partitioning, eq. B_j]: the cache is
// split into 64-key blocks that are fetched whole; [> Query group sharing]:
// the 16 query heads of a GQA group share one block set, so every block is
// loaded once for the whole group and the heads form the 16-row M dimension
// of the tensor-core MMA ([> Query group sharing]: "at least 16 heads");
// [> Complexity analysis, stage 2]: each query attends k*m keys.
//
// One thread-block cluster of C CTAs per (b, h_kv, t) unit; the unit's
// selected blocks are dealt round-robin to the cluster's 4*C warps.  Each
// warp TMA-loads a block's K and V tiles (128-byte swizzle) into its own
// 32 KB stage, computes S = Q K^T (16 x 64, bf16 m16n8k16 MMAs, fp32), an
// online softmax in base 2, and O += P V with P fed as bf16 hi + lo parts
// (16 significant bits).  Warps merge in shared memory, CTAs merge through
// distributed shared memory: CTA r produces heads [16 r / C, 16 (r+1) / C)
// of the output from every CTA's (max, sum, O) partial.  No global scratch.
#include "common.cuh"
#include "kernels.h"

namespace infllmv2 {

namespace {

constexpr int kAttnWarps = 3;      // 3 x 32 KB stages: two CTAs fit on one SM
constexpr int kStageBytes = 32768;  // K tile 16 KB + V tile 16 KB

struct AttnParams {
  int B, Hkv, Lmax, nq, kmax;
  float scale2;  // attn_scale * log2(e)
  const int32_t* kv_lens;
  const int32_t* block_idx;
  const int32_t* n_sel;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
};

constexpr int kQOff = kAttnWarps * kStageBytes;         // Q tile, 4 KB
constexpr int kCtaOOff = kQOff + 4096;                   // CTA partial O [16][128] fp32
constexpr int kCtaMlOff = kCtaOOff + kGroup * kHeadDim * 4;  // CTA (max, sum) [16]
constexpr int kWarpMlOff = kCtaMlOff + kGroup * 8;       // per-warp (max, sum) [4][16]
constexpr int kWgtOff = kWarpMlOff + kAttnWarps * kGroup * 8;  // per-warp weights [4][16]
constexpr int kBarOff = kWgtOff + kAttnWarps * kGroup * 4;
constexpr int kAttnSmem = 1024 + kBarOff + (1 + kAttnWarps) * 8;

__device__ __forceinline__ void tma_kv(uint8_t* stage, const CUtensorMap* kmap, const CUtensorMap* vmap,
                                       int row, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kStageBytes);
  tma_load_2d(stage, kmap, 0, row, bar);
  tma_load_2d(stage + 8192, kmap, 64, row, bar);
  tma_load_2d(stage + 16384, vmap, 0, row, bar);
  tma_load_2d(stage + 24576, vmap, 64, row, bar);
}

template <int C>
__global__ void __launch_bounds__(kAttnWarps * 32, 2)
    attn_cluster_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* q_t = smem + kQOff;
  float* cta_o = reinterpret_cast<float*>(smem + kCtaOOff);
  float2* cta_ml = reinterpret_cast<float2*>(smem + kCtaMlOff);
  float2* warp_ml = reinterpret_cast<float2*>(smem + kWarpMlOff);
  float* wgt = reinterpret_cast<float*>(smem + kWgtOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int split = static_cast<int>(cluster_ctarank());
  const int t = blockIdx.x / C;
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const size_t u = static_cast<size_t>(bh) * p.nq + t;
  const size_t orow = (static_cast<size_t>(b) * p.nq + t) * Hq + static_cast<size_t>(h) * kGroup;
  uint64_t* qbar = bars;
  uint64_t* kvbar = bars + 1 + warp;

  if (tid == 0) {
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    mbar_init(qbar, 1);
    for (int w = 0; w < kAttnWarps; ++w) mbar_init(bars + 1 + w, 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int L = p.kv_lens[b];
  if (L < p.nq || L > p.Lmax) {      // same for every CTA of the cluster
    if (split == 0) {
      for (int e = tid; e < kGroup * kHeadDim; e += kAttnWarps * 32) p.out[orow * kHeadDim + e] = __float2bfloat16(0.f);
      if (tid < kGroup && p.lse) p.lse[orow + tid] = -INFINITY;
      if (tid == 0 && t == 0) atomicOr(p.status, kStatusBadKvLen);
    }
    return;
  }
  const int i = L - p.nq + t;
  const int c = i / kBlock;
  const int ns = min(p.n_sel[u], p.kmax);
  const int32_t* sel = p.block_idx + u * p.kmax;
  const size_t kv_row0 = static_cast<size_t>(bh) * p.Lmax;
  constexpr int kStride = C * kAttnWarps;   // warps in the cluster
  if (split == 0 && warp == 0) check_selection_row(sel, p.n_sel[u], p.kmax, c, p.status, lane);
  const int first = split * kAttnWarps + warp;

  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, 4096);
    tma_load_2d(q_t, &q_map, 0, static_cast<int>(orow), qbar);
    tma_load_2d(q_t + 2048, &q_map, 64, static_cast<int>(orow), qbar);
  }
  uint8_t* stage = smem + warp * kStageBytes;
  const uint32_t k_b = smem_u32(stage), v_b = k_b + 16384;
  // Start this warp's first block load before waiting for Q.
  int n = first;
  while (n < ns && (sel[n] < 0 || sel[n] > c)) n += kStride;
  if (lane == 0 && n < ns && kv_row_ok(kv_row0 + static_cast<size_t>(sel[n]) * kBlock, kv_row0, p.Lmax, p.status))
    tma_kv(stage, &k_map, &v_map, static_cast<int>(kv_row0 + static_cast<size_t>(sel[n]) * kBlock), kvbar);

  bool ok = __all_sync(0xffffffffu, mbar_wait(qbar, 0, p.status));
  uint32_t qa[8][4];
  const uint32_t q_b = smem_u32(q_t);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldmatrix_x4(qa[ks], q_b + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4), 16));

  float o[16][4];
#pragma unroll
  for (int x = 0; x < 16; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  uint32_t phase = 0;

#pragma unroll 1
  while (n < ns && ok) {
    const int j = sel[n];
    ok = __all_sync(0xffffffffu, mbar_wait(kvbar, phase, p.status));
    phase ^= 1u;
    if (!ok) break;
    const int key0 = j * kBlock;
    if (key0 + kBlock - 1 > i) {
      // Keys past i: zero their V rows so masked probabilities never meet
      // non-finite values that may sit in the cache beyond kv_len.
      const int r0 = i - key0 + 1;
      for (int e = lane; e < (kBlock - r0) * 16; e += 32) {
        const int row = r0 + (e >> 4), q16 = e & 15;
        *reinterpret_cast<uint4*>(stage + 16384 + (q16 >> 3) * 8192 + row * 128 + (q16 & 7) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys.
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t kb[4];
        ldmatrix_x4(kb, k_b + swz128_offset(nt * 8 + (lane & 7), 4 * kk + (lane >> 3), kBlock));
        mma_bf16_16816(s[nt], qa[2 * kk], kb[0], kb[1]);
        mma_bf16_16816(s[nt], qa[2 * kk + 1], kb[2], kb[3]);
      }
    }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int x = key0 + nt * 8 + 2 * tq;
      const bool v0 = x <= i, v1 = x + 1 <= i;
      s[nt][0] = v0 ? s[nt][0] * p.scale2 : -INFINITY;
      s[nt][1] = v1 ? s[nt][1] * p.scale2 : -INFINITY;
      s[nt][2] = v0 ? s[nt][2] * p.scale2 : -INFINITY;
      s[nt][3] = v1 ? s[nt][3] * p.scale2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
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
    // P enters the tensor cores as hi + lo bf16 parts (16 significant bits),
    // so the only bf16 rounding left in the output is the final store.
    uint32_t pa[4][4], pl[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
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
    // O += P V: A = P (16 x 64 keys), B = V (64 keys x 128 dims) via ldmatrix.trans.
#pragma unroll
    for (int np = 0; np < 8; ++np) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t vb[4];
        ldmatrix_x4_trans(vb, v_b + swz128_offset(kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8,
                                                  2 * np + (lane >> 4), kBlock));
        mma_bf16_16816(o[2 * np], pa[kk], vb[0], vb[1]);
        mma_bf16_16816(o[2 * np + 1], pa[kk], vb[2], vb[3]);
        mma_bf16_16816(o[2 * np], pl[kk], vb[0], vb[1]);
        mma_bf16_16816(o[2 * np + 1], pl[kk], vb[2], vb[3]);
      }
    }
    // Next block of this warp.
    n += kStride;
    while (n < ns && (sel[n] < 0 || sel[n] > c)) n += kStride;
    if (n < ns) {
      // Order the generic writes to the stage (zeroed V rows) before the
      // async-proxy (TMA) writes that refill it.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && kv_row_ok(kv_row0 + static_cast<size_t>(sel[n]) * kBlock, kv_row0, p.Lmax, p.status))
        tma_kv(stage, &k_map, &v_map, static_cast<int>(kv_row0 + static_cast<size_t>(sel[n]) * kBlock), kvbar);
    }
  }
  __syncwarp();
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  // Per-warp results into the warp's own stage (8 KB of fp32).
  float* o_w = reinterpret_cast<float*>(stage);
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
  __syncthreads();
  if (tid < kGroup) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, warp_ml[w * kGroup + tid].x);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float2 v = warp_ml[w * kGroup + tid];
      const float wt = (M == -INFINITY) ? 0.f : fast_exp2(v.x - M);
      wgt[w * kGroup + tid] = wt;
      lsum += wt * v.y;
    }
    cta_ml[tid] = make_float2(M, lsum);
  }
  __syncthreads();
  for (int e = tid; e < kGroup * kHeadDim; e += kAttnWarps * 32) {
    const int hd = e >> 7;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w)
      acc += wgt[w * kGroup + hd] * reinterpret_cast<const float*>(smem + w * kStageBytes)[e];
    cta_o[e] = acc;
  }
  cluster_sync();

  // Heads [hpc * split, hpc * (split + 1)) of the output from all partials.
  constexpr int hpc = kGroup / C;
  for (int e = tid; e < hpc * kHeadDim; e += kAttnWarps * 32) {
    const int hd = split * hpc + e / kHeadDim;
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
  cluster_sync();
}


template <int C>
cudaError_t launch_cluster(const Shape& s, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, const AttnParams& p, cudaStream_t st, bool* unsupported) {
  *unsupported = false;
  cudaError_t e = cudaFuncSetAttribute(attn_cluster_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(attn_cluster_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C * s.nq, s.B * s.Hkv, 1);
  cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = kAttnSmem;
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
  e = cudaOccupancyMaxActiveClusters(&clusters, attn_cluster_kernel<C>, &cfg);
  // The 16-CTA form only pays off when every unit's cluster is resident at once.
  const long long need = (C > 8) ? static_cast<long long>(s.B) * s.Hkv * s.nq : 1;
  if (e != cudaSuccess || clusters < need) {
    cudaGetLastError();
    *unsupported = true;
    return cudaSuccess;
  }
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<C>, q_map, k_map, v_map, p);
}

}  // namespace

size_t attn_workspace_bytes(const Shape& s, bool prefill) {
  (void)s;
  (void)prefill;
  return 0;
}

cudaError_t launch_attn(const Shape& s, bool prefill, const CUtensorMap& q_map,
                        const CUtensorMap& k_map, const CUtensorMap& v_map,
                        const int32_t* kv_lens, const int32_t* block_idx, const int32_t* n_sel,
                        void* out, float* lse, void* ws, uint32_t* status, cudaStream_t st) {
  (void)prefill;
  (void)ws;
  AttnParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.kmax = s.kmax;
  p.scale2 = s.attn_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status;
  // Cluster size: enough warps for one block each where the SM count allows,
  // and no larger than lets every unit's cluster be resident at once (two
  // CTAs per SM): 8 drafts x 8 groups at 128K run 64 clusters of 4 CTAs in
  // 23 us against 28 us for 1.7 waves of 8-CTA clusters.
  const int want = (s.kmax + kAttnWarps - 1) / kAttnWarps;
  const long long units = static_cast<long long>(s.B) * s.Hkv * s.nq;
  bool unsupported = false;
  cudaError_t e;
  if (want > 8 && units * 16 <= 2 * device_sm_count()) {
    e = launch_cluster<16>(s, q_map, k_map, v_map, p, st, &unsupported);
    if (e != cudaSuccess || !unsupported) return e;
  }
  if (want > 4 && units * 8 <= 2 * device_sm_count()) {
    e = launch_cluster<8>(s, q_map, k_map, v_map, p, st, &unsupported);
    if (e != cudaSuccess || !unsupported) return e;
  }
  e = launch_cluster<4>(s, q_map, k_map, v_map, p, st, &unsupported);
  if (e == cudaSuccess && unsupported) return cudaErrorInvalidConfiguration;
  return e;
}

}  // namespace infllmv2
