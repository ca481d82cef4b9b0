// Stage 2 of InfLLM v2: block relevance and top-k block selection -- the
// entry point, its scratch accounting, and the prefill path (n_q > 16).
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck] and
// [> Initial and local tokens always selected].  For one query token of one
// GQA group (16 heads):
//   z[h, j] = score_scale * q_h . Mean_j            (visible kernels j)
//   g[j]    = (1/16) sum_h exp(z[h, j] - lse_h)     (exact two-pass LSE)
//   r[blk]  = max_j g[j] over kernels meeting the block (j in 4 blk - 1 .. 4 blk + 3)
//   top-k over r with forced initial/local blocks.
//
// Two paths, same result:
//  * decode / verify (n_q <= 16): select_decode.cu, one thread-block cluster
//    per (b, h_kv) group.
//  * prefill (n_q > 16): select_tc.cu on tcgen05 (8 tokens x 16 heads per
//    128-row tile); here, the mma.sync form of the same two passes, used for
//    caches whose block scores do not fit the tcgen05 kernel's shared
//    memory: one warp per query token, TT
//    tokens per CTA sharing a TMA pipeline of 64-kernel hi/lo tiles, streamed
//    twice (pass 1: LSE, pass 2: normalised group mean and block maxima),
//    then a warp top-k.
#include "select_common.cuh"

namespace infllmv2 {

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

bool select_tc_supported(const Shape& s);
cudaError_t launch_select_tc(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map,
                             const CUtensorMap& q_map, const SelParams& p, cudaStream_t st);
size_t select_decode_ncpad(const Shape& s);
bool select_decode_supported(const Shape& s);
cudaError_t launch_select_decode(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                                 const SelParams& p, cudaStream_t st);

namespace {

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
  l.bar_off = (l.tk_off + kPrefTokens * static_cast<int>(sizeof(WarpTopkScratch)) + 15) & ~15;
  l.total = l.bar_off + (2 * stages + 1) * 8;
  return l;
}

__global__ void __launch_bounds__(kPrefTokens * 32)
    sel_prefill_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap kcc_map,
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
  WarpTopkScratch& tk = reinterpret_cast<WarpTopkScratch*>(smem + lay.tk_off)[warp];
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
  const int t_first = static_cast<int>(blockIdx.x) * kPrefTokens;
  const int t_last = min(nq - 1, t_first + kPrefTokens - 1);
  const int nvis_max = n_complete_kernels(L - nq + t_last + 1);
  const int nch = (nvis_max + kPrefChunk - 1) / kPrefChunk;
  const int i_t = L - nq + (active ? t : t_last);
  const int c_t = i_t / kBlock;
  const int nvis_t = n_complete_kernels(i_t + 1);
  // LSE pass over coarse windows ([InfLLM v2 > Efficient LSE approximation])
  // for tokens that have a complete one, over the fine kernels otherwise.
  // The stream of 64-row tiles: coarse pass (A), fine LSE pass (B), fine
  // normalise pass (C); A and B only when some token of the CTA needs them.
  const int nvis_c_t = p.sc ? (i_t + 1) / p.sc : 0;
  const bool coarse_t = nvis_c_t > 0;
  const int nvis_c_max = p.sc ? (L - nq + t_last + 1) / p.sc : 0;
  const bool need_b = p.sc == 0 || (L - nq + t_first + 1) / p.sc == 0;
  const int nch_a = (nvis_c_max + kPrefChunk - 1) / kPrefChunk;
  const int nch_b = need_b ? nch : 0;
  const int seg_c = nch_a + nch_b;
  const int total = seg_c + nch;

  for (int j = lane; j < p.nbmax; j += 32) r_w[j] = -INFINITY;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&kcc_map);
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
    const int stage = it % S;
    const bool coarse_seg = it < nch_a;
    const int ch = coarse_seg ? it : (it < seg_c ? it - nch_a : it - seg_c);
    const CUtensorMap* map = coarse_seg ? &kcc_map : &kc_map;
    const int rows = coarse_seg ? p.nccmax : p.ncmax;
    uint8_t* dst = smem + lay.stage_off + stage * kPrefStageBytes;
    mbar_arrive_expect_tx(&full[stage], kPrefStageBytes);
    const int row_hi = (bh * 2 + 0) * rows + ch * kPrefChunk;
    const int row_lo = (bh * 2 + 1) * rows + ch * kPrefChunk;
    tma_load_2d(dst, map, 0, row_hi, &full[stage]);
    tma_load_2d(dst + 8192, map, 64, row_hi, &full[stage]);
    tma_load_2d(dst + 16384, map, 0, row_lo, &full[stage]);
    tma_load_2d(dst + 24576, map, 64, row_lo, &full[stage]);
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
    const int pass = it < seg_c ? 0 : 1;
    const int ch = it < nch_a ? it : (it < seg_c ? it - nch_a : it - seg_c);
    const int kbase = ch * kPrefChunk;
    // This token's visible rows of the current tile (0: nothing to do).
    const int nvv = it < nch_a ? (coarse_t ? nvis_c_t : 0) : (it < seg_c ? (coarse_t ? 0 : nvis_t) : nvis_t);
    if (it == seg_c) {
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
    if (active && kbase < nvv) {
      const uint32_t hi_b = smem_u32(smem + lay.stage_off + stage * kPrefStageBytes);
      const uint32_t lo_b = hi_b + 16384;
      // All eight n-tiles' scores first (independent MMA chains), then the
      // exponentials; only the chunk holding the last visible kernel masks.
      float x[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float acc[4];
        score_ntile(acc, a, hi_b, lo_b, nt * 8, kPrefChunk, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[nt][e] = acc[e] * p.scale2;
      }
      if (kbase + kPrefChunk > nvv) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int kj = kbase + nt * 8 + 2 * tq;
          if (kj >= nvv) x[nt][0] = x[nt][2] = -INFINITY;
          if (kj + 1 >= nvv) x[nt][1] = x[nt][3] = -INFINITY;
        }
      }
      if (pass == 0) {
        // Chunk maxima, then one rescale of the running sums per chunk.
        float c0 = x[0][0], c1 = x[0][2];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          c0 = fmaxf(c0, fmaxf(x[nt][0], x[nt][1]));
          c1 = fmaxf(c1, fmaxf(x[nt][2], x[nt][3]));
        }
        const float M0 = fmaxf(m0, c0), M1 = fmaxf(m1, c1);
        if (M0 > -INFINITY) {
          float s0 = l0 * fast_exp2(m0 - M0);
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) s0 += fast_exp2(x[nt][0] - M0) + fast_exp2(x[nt][1] - M0);
          l0 = s0;
          m0 = M0;
        }
        if (M1 > -INFINITY) {
          float s1 = l1 * fast_exp2(m1 - M1);
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) s1 += fast_exp2(x[nt][2] - M1) + fast_exp2(x[nt][3] - M1);
          l1 = s1;
          m1 = M1;
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          float s0 = fast_exp2(x[nt][0] - lse_g) + fast_exp2(x[nt][2] - lse_g8);
          float s1 = fast_exp2(x[nt][1] - lse_g) + fast_exp2(x[nt][3] - lse_g8);
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
  select_topk_warp(r_w, flag_w, c_t + 1, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax,
                   p.block_idx + u * p.kmax, p.n_sel + u, tk, lane);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

cudaError_t launch_prefill_select(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map,
                                  const CUtensorMap& q_map, SelParams p, cudaStream_t st) {
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
  sel_prefill_kernel<<<grid, kPrefTokens * 32, psmem, st>>>(kc_map, kcc_map, q_map, p);
  return cudaGetLastError();
}

bool use_decode_path(const Shape& s) { return s.nq <= kSelDecodeMaxNq && select_decode_supported(s); }

}  // namespace

size_t select_workspace_bytes(const Shape& s) {
  if (use_decode_path(s)) {
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
    return align256(units * kGroup * select_decode_ncpad(s) * sizeof(float));
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

  if (use_decode_path(s)) {
    p.ncpad = static_cast<int>(select_decode_ncpad(s));
    p.z = static_cast<float*>(ws);
    return launch_select_decode(s, kc_map, q_map, p, st);
  }
  // Prefill: the tcgen05 kernel where its shared memory holds the block
  // scores of 8 tokens, the mma.sync kernel otherwise.
  if (select_tc_supported(s)) return launch_select_tc(s, kc_map, kc_map, q_map, p, st);
  return launch_prefill_select(s, kc_map, kc_map, q_map, p, st);
}

cudaError_t launch_select_coarse(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map, int sc,
                                 const CUtensorMap& q_map, const int32_t* kv_lens, int32_t* block_idx,
                                 int32_t* n_sel, float* block_scores, uint32_t* status, cudaStream_t st) {
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
  p.sc = sc;
  p.nccmax = s.Lmax / sc;
  if (select_tc_supported(s)) return launch_select_tc(s, kc_map, kcc_map, q_map, p, st);
  return launch_prefill_select(s, kc_map, kcc_map, q_map, p, st);
}

}  // namespace infllmv2
