// Stage 3 of InfLLM v2: exact softmax attention over the selected KV blocks.
//
// [InfLLM v2 > Block-level key-value partitioning, eq. B_j]: the cache is
// split into 64-key blocks that are fetched whole; [> Query group sharing]:
// the 16 query heads of a GQA group share one block set, so every block is
// loaded once for the whole group and the heads form the 16-row M dimension
// of the tensor-core MMA ([> Query group sharing]: "at least 16 heads");
// [> Complexity analysis, stage 2]: each query attends k*m keys.
//
// One CTA handles a contiguous slice ("split") of the selected blocks of one
// (b, h_kv, t) unit.  Each warp owns one 32 KB shared-memory stage into which
// TMA (128-byte swizzle) loads a block's K and V tiles; the warp computes
// S = Q K^T (16 x 64) with bf16 m16n8k16 MMAs, an online softmax in fp32 base
// 2, and O += P V with P rounded to bf16.  The warps of a CTA merge their
// (max, sum, O) in shared memory; with several splits per unit the CTA writes
// an fp32 partial and the last CTA of the unit (atomic ticket) merges them.
#include "common.cuh"
#include "kernels.h"

namespace infllmv2 {

namespace {

constexpr int kAttnWarps = 4;
constexpr int kMaxSplits = 64;
constexpr int kStageBytes = 32768;  // K tile 16 KB + V tile 16 KB

struct AttnParams {
  int B, Hkv, Lmax, nq, kmax, n_splits, bps;
  float scale2;  // attn_scale * log2(e)
  const int32_t* kv_lens;
  const int32_t* block_idx;
  const int32_t* n_sel;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;      // [units][n_splits][16][128]
  float2* part_ml;    // [units][n_splits][16]
  uint32_t* counters; // [units]
  uint32_t* status;
};

__device__ __forceinline__ void tma_kv(uint8_t* stage, const CUtensorMap* kmap,
                                       const CUtensorMap* vmap, int row, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kStageBytes);
  tma_load_2d(stage, kmap, 0, row, bar);
  tma_load_2d(stage + 8192, kmap, 64, row, bar);
  tma_load_2d(stage + 16384, vmap, 0, row, bar);
  tma_load_2d(stage + 24576, vmap, 64, row, bar);
}

__global__ void __launch_bounds__(kAttnWarps * 32)
    attn_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                const __grid_constant__ CUtensorMap v_map, AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* stages = smem;                                   // kAttnWarps x 32 KB
  uint8_t* q_t = smem + kAttnWarps * kStageBytes;           // 4 KB
  float2* ml_s = reinterpret_cast<float2*>(q_t + 4096);     // [kAttnWarps][16]
  float* wgt_s = reinterpret_cast<float*>(ml_s + kAttnWarps * kGroup);  // [kMaxSplits][16]
  float* inv_s = wgt_s + kMaxSplits * kGroup;               // [16]
  float* mtot_s = inv_s + kGroup;                           // [16]
  uint64_t* bars = reinterpret_cast<uint64_t*>(mtot_s + kGroup);  // qbar, kv[kAttnWarps]
  __shared__ int is_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int split = blockIdx.x % p.n_splits;
  const int t = blockIdx.x / p.n_splits;
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const size_t u = static_cast<size_t>(bh) * p.nq + t;
  const size_t orow = (static_cast<size_t>(b) * p.nq + t) * Hq + static_cast<size_t>(h) * kGroup;

  const int L = p.kv_lens[b];
  if (L < p.nq || L > p.Lmax) {
    if (split == 0) {
      for (int e = tid; e < kGroup * kHeadDim; e += kAttnWarps * 32)
        p.out[orow * kHeadDim + e] = __float2bfloat16(0.f);
      if (tid < kGroup && p.lse) p.lse[orow + tid] = -INFINITY;
      if (tid == 0 && t == 0) atomicOr(p.status, kStatusBadKvLen);
    }
    return;
  }
  const int i = L - p.nq + t;
  const int c = i / kBlock;
  const int ns = min(p.n_sel[u], p.kmax);
  const int lo = split * p.bps;
  const int hi = min(ns, lo + p.bps);
  const int32_t* sel = p.block_idx + u * p.kmax;
  const size_t kv_row0 = static_cast<size_t>(bh) * p.Lmax;

  uint64_t* qbar = bars;
  uint64_t* kvbar = bars + 1 + warp;
  if (tid == 0) {
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    mbar_init(qbar, 1);
    for (int w = 0; w < kAttnWarps; ++w) mbar_init(bars + 1 + w, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, 4096);
    tma_load_2d(q_t, &q_map, 0, static_cast<int>(orow), qbar);
    tma_load_2d(q_t + 2048, &q_map, 64, static_cast<int>(orow), qbar);
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(qbar, 0, p.status));

  uint32_t qa[8][4];
  const uint32_t q_b = smem_u32(q_t);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    ldmatrix_x4(qa[ks], q_b + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 2 * ks + (lane >> 4), 16));

  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  uint8_t* stage = stages + warp * kStageBytes;
  const uint32_t k_b = smem_u32(stage), v_b = k_b + 16384;
  uint32_t phase = 0;

#pragma unroll 1
  for (int n = lo + warp; n < hi && ok; n += kAttnWarps) {
    const int j = sel[n];
    if (j < 0 || j > c) continue;
    // Order this warp's earlier generic writes to the stage (zeroed V rows)
    // before the async-proxy (TMA) writes that refill it.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tma_kv(stage, &k_map, &v_map, static_cast<int>(kv_row0 + static_cast<size_t>(j) * kBlock), kvbar);
    ok = mbar_wait(kvbar, phase, p.status);
    phase ^= 1u;
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
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
    for (int n = 0; n < 16; ++n) {
      o[n][0] *= sc0;
      o[n][1] *= sc0;
      o[n][2] *= sc1;
      o[n][3] *= sc1;
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
  }
  __syncwarp();
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  // Per-warp results into the warp's own stage (K half, 8 KB of fp32).
  float* o_w = reinterpret_cast<float*>(stage);
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    const int d0 = n * 8 + 2 * tq;
    *reinterpret_cast<float2*>(o_w + g * kHeadDim + d0) = make_float2(o[n][0], o[n][1]);
    *reinterpret_cast<float2*>(o_w + (g + 8) * kHeadDim + d0) = make_float2(o[n][2], o[n][3]);
  }
  if (tq == 0) {
    ml_s[warp * kGroup + g] = make_float2(m0, l0);
    ml_s[warp * kGroup + g + 8] = make_float2(m1, l1);
  }
  __syncthreads();
  if (tid < kGroup) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, ml_s[w * kGroup + tid].x);
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float2 v = ml_s[w * kGroup + tid];
      const float wt = (M == -INFINITY) ? 0.f : fast_exp2(v.x - M);
      wgt_s[w * kGroup + tid] = wt;
      lsum += wt * v.y;
    }
    mtot_s[tid] = M;
    inv_s[tid] = lsum;
  }
  __syncthreads();

  const bool single = p.n_splits == 1;
  for (int e = tid; e < kGroup * kHeadDim; e += kAttnWarps * 32) {
    const int hd = e >> 7;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w)
      acc += wgt_s[w * kGroup + hd] * reinterpret_cast<const float*>(stages + w * kStageBytes)[e];
    if (single) {
      const float lsum = inv_s[hd];
      p.out[orow * kHeadDim + e] = __float2bfloat16(lsum > 0.f ? acc / lsum : 0.f);
    } else {
      p.part_o[(u * p.n_splits + split) * (kGroup * kHeadDim) + e] = acc;
    }
  }
  if (single) {
    if (tid < kGroup && p.lse) {
      const float lsum = inv_s[tid];
      p.lse[orow + tid] = lsum > 0.f ? (mtot_s[tid] + fast_log2(lsum)) * 0.69314718055994531f : -INFINITY;
    }
    return;
  }
  if (tid < kGroup) p.part_ml[(u * p.n_splits + split) * kGroup + tid] = make_float2(mtot_s[tid], inv_s[tid]);

  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(&p.counters[u], 1u);
    is_last = (prev == static_cast<uint32_t>(p.n_splits) - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  if (tid == 0) p.counters[u] = 0;
  if (tid < kGroup) {
    float M = -INFINITY;
    for (int sp = 0; sp < p.n_splits; ++sp) M = fmaxf(M, __ldcg(&p.part_ml[(u * p.n_splits + sp) * kGroup + tid]).x);
    float lsum = 0.f;
    for (int sp = 0; sp < p.n_splits; ++sp) {
      const float2 v = __ldcg(&p.part_ml[(u * p.n_splits + sp) * kGroup + tid]);
      const float wt = (M == -INFINITY) ? 0.f : fast_exp2(v.x - M);
      wgt_s[sp * kGroup + tid] = wt;
      lsum += wt * v.y;
    }
    mtot_s[tid] = M;
    inv_s[tid] = lsum;
  }
  __syncthreads();
  for (int e = tid; e < kGroup * kHeadDim; e += kAttnWarps * 32) {
    const int hd = e >> 7;
    float acc = 0.f;
    for (int sp = 0; sp < p.n_splits; ++sp)
      acc += wgt_s[sp * kGroup + hd] * __ldcg(&p.part_o[(u * p.n_splits + sp) * (kGroup * kHeadDim) + e]);
    const float lsum = inv_s[hd];
    p.out[orow * kHeadDim + e] = __float2bfloat16(lsum > 0.f ? acc / lsum : 0.f);
  }
  if (tid < kGroup && p.lse) {
    const float lsum = inv_s[tid];
    p.lse[orow + tid] = lsum > 0.f ? (mtot_s[tid] + fast_log2(lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

constexpr int kAttnSmem = 1024 + kAttnWarps * kStageBytes + 4096 + kAttnWarps * kGroup * 8 +
                          kMaxSplits * kGroup * 4 + 2 * kGroup * 4 + (1 + kAttnWarps) * 8;

int decode_splits(const Shape& s) {
  // One block per warp per CTA: ceil(kmax / warps) splits.
  int n = (s.kmax + kAttnWarps - 1) / kAttnWarps;
  return n < 1 ? 1 : (n > kMaxSplits ? kMaxSplits : n);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t attn_workspace_bytes(const Shape& s, bool prefill) {
  if (prefill) return 0;
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
  const int ns = decode_splits(s);
  return align256(units * 4) + align256(units * ns * kGroup * sizeof(float2)) +
         align256(units * ns * kGroup * kHeadDim * sizeof(float));
}

cudaError_t launch_attn(const Shape& s, bool prefill, const CUtensorMap& q_map,
                        const CUtensorMap& k_map, const CUtensorMap& v_map,
                        const int32_t* kv_lens, const int32_t* block_idx, const int32_t* n_sel,
                        void* out, float* lse, void* ws, uint32_t* status, cudaStream_t st) {
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
  const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
  cudaError_t e;
  if (prefill) {
    p.n_splits = 1;
    p.bps = s.kmax;
  } else {
    p.n_splits = decode_splits(s);
    p.bps = kAttnWarps;
    if (p.n_splits * p.bps < s.kmax) p.bps = (s.kmax + p.n_splits - 1) / p.n_splits;
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.counters = reinterpret_cast<uint32_t*>(base);
    p.part_ml = reinterpret_cast<float2*>(base + align256(units * 4));
    p.part_o = reinterpret_cast<float*>(base + align256(units * 4) +
                                        align256(units * p.n_splits * kGroup * sizeof(float2)));
    if (p.n_splits > 1) {
      e = cudaMemsetAsync(p.counters, 0, units * 4, st);
      if (e != cudaSuccess) return e;
    }
  }
  e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem);
  if (e != cudaSuccess) return e;
  const size_t gx = static_cast<size_t>(p.n_splits) * s.nq;
  if (gx > 0x7fffffffull || s.B * s.Hkv > 65535) return cudaErrorInvalidConfiguration;
  attn_kernel<<<dim3(static_cast<unsigned>(gx), s.B * s.Hkv), kAttnWarps * 32, kAttnSmem, st>>>(
      q_map, k_map, v_map, p);
  return cudaGetLastError();
}

}  // namespace infllmv2
