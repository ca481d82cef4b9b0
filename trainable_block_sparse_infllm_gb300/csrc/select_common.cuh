// Pieces shared by the two selection kernels (decode / prefill paths).
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck]:
// scores z = score_scale * q . Mean_j are kept in base 2 (scaled by log2 e)
// so that exp is a single ex2; q . Mean_j runs on the tensor cores as
// q . hi_j + q . lo_j (bf16 m16n8k16, fp32 accumulation) with the kernel
// means stored pre-split into two bf16 planes.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace infllmv2 {

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
  int sc, nccmax;      // prefill path: coarse-LSE window (0 = exact LSE) and windows per cache
  int csize;           // prefill path: CTAs per 8-token tile (1, or a cluster splitting the chunks)
  float* r_scratch;    // prefill path: block scores off chip, [r_slots][8][nbmax] (null: in shared memory)
  int r_slots;         // slots of r_scratch (one per SM identifier)
  int r_rows;          // prefill path: tokens whose block scores a CTA keeps in shared memory
  const uint16_t* q;   // prefill path: q as bf16 bits, [B*nq*Hkv*16][128]
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

}  // namespace infllmv2
