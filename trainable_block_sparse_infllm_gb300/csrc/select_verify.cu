// Stage 2 of InfLLM v2 for a few query tokens per sequence (speculative
// verification, 2 <= n_q <= 8): block relevance and top-k block selection of
// every token, in one launch with no global scratch.
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck: the
// exact softmax needs the LSE first, so the kernel means are scored twice],
// [> Initial and local tokens always selected], [> Token-level queries].
//
// One cluster of C CTAs per (b, h_kv) group, one CTA per SM, C chosen at
// launch so that every group's cluster is resident at once.  CTA r owns the
// 16-block groups [r per, (r + 1) per) and the matching 64-kernel chunks.
//   pass 1   the CTA's hi/lo chunks stream through a 3-stage TMA ring (the
//            rest of them head for L2 at once); z = score_scale q_t . Mean
//            for every token t on the tensor cores; each token's running
//            (max, sum of 2^z) per head stays in registers.
//   LSE      the CTA's (max, sum) per (token, head) is pushed into every CTA;
//            one cluster barrier; each CTA merges the C partials.
//   pass 2   the same chunks again, now from L2: z once more, then
//            g = (1/16) sum_h 2^(z_h - lse_h) per token and kernel (the 16
//            heads summed across the lanes of the MMA fragment), kept in
//            shared memory for all of the CTA's kernels and tokens.
//   push     each token's block maxima over the CTA's blocks (and the g of
//            the CTA's last kernel) go to the token's owner CTA (token t:
//            CTA t mod C); one cluster barrier.
//   top-k    the owner selects (exact, the shared top-k routine) and writes
//            the token's list.
// The scores never leave the chip: a second pass over the chunks from L2
// costs less than writing and re-reading one score per (token, head, kernel).
#include "select_common.cuh"

namespace infllmv2 {

namespace {

constexpr int kSvThreads = 512;     // 16 warps: warp w takes n-tile w % 8 of every chunk for the tokens t = w / 8 (mod 2)
constexpr int kSvWarps = kSvThreads / 32;
constexpr int kSvMaxQ = 8;
constexpr int kSvChunk = 64;
constexpr int kSvRing = 3;
constexpr int kSvStageBytes = 32768;
constexpr int kSvMaxC = 16;
constexpr int kSvMaxIt = 16;        // chunks per CTA
constexpr int kSvMaxBlocks = 4096;

struct SvParams {
  int B, Hkv, Lmax, nq, ncmax, nbmax, kmax;
  int topk, n_init, n_local, inc_forced, write_r;
  float scale2;
  const int32_t* kv_lens;
  int32_t* block_idx;
  int32_t* n_sel;
  float* r_buf;
  uint32_t* status;
};

// Shared memory (fixed sizes, so the cluster occupancy is one per device).
// The top-k scratch lies over the ring, free once pass 2 is done; the areas
// other CTAs write into (lse_in, rown, tails) are never overlaid.
constexpr int kSvOwnedRows = 2;     // tokens an owner CTA selects (C >= 4)
struct SvLayout {
  int ring, q, gbuf, rown, tails, lse_in, wpart, cpart, lse, tk, bits, surv, bar, total;
};

__host__ __device__ constexpr SvLayout sv_layout() {
  SvLayout l{};
  l.ring = 0;
  l.tk = 0;                                             // top-k scratch (after pass 2)
  l.bits = 20480;
  l.surv = l.bits + kSvMaxBlocks / 8;
  l.q = kSvRing * kSvStageBytes;                        // [8 tokens][16 rows x 256 B]
  l.gbuf = l.q + kSvMaxQ * 4096;                        // [8 tokens][16 chunks x 64] g of this CTA's kernels
  l.rown = l.gbuf + kSvMaxQ * kSvMaxIt * kSvChunk * 4;  // [2 owned tokens][4096] block scores
  l.tails = l.rown + kSvOwnedRows * kSvMaxBlocks * 4;   // [16 CTAs][8 tokens] last-kernel g
  l.lse_in = l.tails + kSvMaxC * kSvMaxQ * 4;           // [16 CTAs][8 tokens][16 heads] (max, sum)
  l.wpart = l.lse_in + kSvMaxC * kSvMaxQ * kGroup * 8;  // [8 warps][8 tokens][16 heads] (max, sum)
  l.cpart = l.wpart + 8 * kSvMaxQ * kGroup * 8;         // [8 tokens][16 heads]
  l.lse = l.cpart + kSvMaxQ * kGroup * 8;               // [8 tokens][16 heads] lse (base 2)
  l.bar = l.lse + kSvMaxQ * kGroup * 4;
  l.total = l.bar + (2 * kSvRing + 1) * 8;
  return l;
}

constexpr int kSvSmem = sv_layout().total + 1024;
static_assert(kSvSmem <= 227 * 1024, "one CTA per SM");
static_assert(sv_layout().surv + kSvMaxBlocks * 8 <= kSvRing * kSvStageBytes, "top-k scratch inside the ring");

__device__ __forceinline__ uint32_t sv_cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__global__ void __launch_bounds__(kSvThreads, 1)
    sel_verify_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap q_map,
                      SvParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr SvLayout lay = sv_layout();
  float* gbuf = reinterpret_cast<float*>(smem + lay.gbuf);          // [t][it * 64 + x]
  float* rown = reinterpret_cast<float*>(smem + lay.rown);          // [owned row][block]
  float* tails = reinterpret_cast<float*>(smem + lay.tails);        // [src][t]
  float2* lse_in = reinterpret_cast<float2*>(smem + lay.lse_in);    // [src][t][h]
  float2* wpart = reinterpret_cast<float2*>(smem + lay.wpart);      // [w][t][h]
  float2* cpart = reinterpret_cast<float2*>(smem + lay.cpart);      // [t][h]
  float* lse2 = reinterpret_cast<float*>(smem + lay.lse);           // [t][h]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + kSvRing;
  uint64_t* qbar = empty + kSvRing;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rank = static_cast<int>(cluster_ctarank());
  const int C = static_cast<int>(sv_cluster_nctarank());
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int nq = p.nq;
  const size_t unit0 = static_cast<size_t>(bh) * nq;

  if (tid == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    for (int s = 0; s < kSvRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSvWarps);
    }
    mbar_init(qbar, 1);
    fence_barrier_init();
  }
  cluster_arrive_relaxed();
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  const int L = p.kv_lens[b];
  const int nbt = L >= 1 ? (L - 1) / kBlock + 1 : 0;   // blocks visible to the last token
  const int groups = (nbt + 15) / 16;
  const int per = (groups + C - 1) / C;
  if (L < nq || L > p.Lmax || per > kSvMaxIt || nbt > kSvMaxBlocks) {   // same in every CTA
    if (rank == 0) {
      for (int e = tid; e < nq * p.kmax; e += kSvThreads) p.block_idx[unit0 * p.kmax + e] = -1;
      for (int e = tid; e < nq; e += kSvThreads) p.n_sel[unit0 + e] = 0;
      if (p.write_r)
        for (int e = tid; e < nq * p.nbmax; e += kSvThreads) p.r_buf[unit0 * p.nbmax + e] = -INFINITY;
      if (tid == 0) atomicOr(p.status, kStatusBadKvLen);
    }
    cluster_wait();
    return;
  }
  const int k0 = min(groups, rank * per), k1 = min(groups, (rank + 1) * per);
  const int nc = n_complete_kernels(L);
  const int nmy = max(0, min(k1, (nc + kSvChunk - 1) / kSvChunk) - k0);
  const int Hq = p.Hkv * kGroup;

  // Load n (0 <= n < 2 nmy) brings chunk n % nmy: pass 1, then pass 2.
  auto issue = [&](int n) {
    const int st = n % kSvRing;
    const int row = (k0 + n % nmy) * kSvChunk;
    uint8_t* dst = smem + lay.ring + st * kSvStageBytes;
    mbar_arrive_expect_tx(&full[st], kSvStageBytes);
    tma_load_2d(dst, &kc_map, 0, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 8192, &kc_map, 64, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 16384, &kc_map, 0, (bh * 2 + 1) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 24576, &kc_map, 64, (bh * 2 + 1) * p.ncmax + row, &full[st]);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(qbar, nq * 4096);
    for (int t = 0; t < nq; ++t) {
      const int row = (b * nq + t) * Hq + h * kGroup;
      tma_load_2d(smem + lay.q + t * 4096, &q_map, 0, row, qbar);
      tma_load_2d(smem + lay.q + t * 4096 + 2048, &q_map, 64, row, qbar);
    }
    for (int n = 0; n < min(kSvRing, 2 * nmy); ++n) issue(n);
  }
  if (warp == 1) {   // the rest of this CTA's chunks head for L2 now
    for (int x = lane; x < 4 * (nmy - kSvRing); x += 32) {
      const int row = (k0 + kSvRing + (x >> 2)) * kSvChunk;
      tma_prefetch_2d(&kc_map, (x & 1) * 64, (bh * 2 + ((x >> 1) & 1)) * p.ncmax + row);
    }
  }
  bool ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  const uint32_t q_b = smem_u32(smem + lay.q);

  // Visible kernels of token t: those ending at or before its position.
  auto nvis_of = [&](int t) { return n_complete_kernels(L - nq + t + 1); };

  // Scores of this warp's n-tile of chunk `it` (stage st) for token t:
  // z0, z1 (head g, kernels kj, kj + 1) and z2, z3 (head g + 8).
  auto scores = [&](int st, int it, int t, float (&z)[4]) {
    uint32_t a[8][4];
    load_q_frags(a, q_b + t * 4096, lane);
    const uint32_t hi_b = smem_u32(smem + lay.ring + st * kSvStageBytes);
    float acc[4];
    score_ntile(acc, a, hi_b, hi_b + 16384, (warp & 7) * 8, kSvChunk, lane);
    const int kj = (k0 + it) * kSvChunk + (warp & 7) * 8 + 2 * tq;
    const int nv = nvis_of(t);
    const bool v0 = kj < nv, v1 = kj + 1 < nv;
    z[0] = v0 ? acc[0] * p.scale2 : -INFINITY;
    z[1] = v1 ? acc[1] * p.scale2 : -INFINITY;
    z[2] = v0 ? acc[2] * p.scale2 : -INFINITY;
    z[3] = v1 ? acc[3] * p.scale2 : -INFINITY;
  };

  // ------------------------------------------------------------- pass 1 --
  constexpr int kTw = kSvMaxQ / 2;   // tokens per warp: t = (warp >> 3) + 2 x
  const int tpar = warp >> 3;
  float m0[kTw], l0[kTw], m1[kTw], l1[kTw];
#pragma unroll
  for (int x = 0; x < kTw; ++x) m0[x] = m1[x] = -INFINITY, l0[x] = l1[x] = 0.f;
  auto consume = [&](int n) {   // wait for load n, release its stage when done (called by all 8 warps)
    const int st = n % kSvRing;
    bool got = ok && mbar_wait(&full[st], static_cast<uint32_t>(n / kSvRing) & 1u, p.status);
    ok = __all_sync(0xffffffffu, got);
    return st;
  };
  auto release = [&](int n) {
    const int st = n % kSvRing;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
    if (tid == 0 && ok && n + kSvRing < 2 * nmy) {
      if (mbar_wait(&empty[st], static_cast<uint32_t>(n / kSvRing) & 1u, p.status)) issue(n + kSvRing);
    }
    __syncwarp();
  };
#pragma unroll 1
  for (int it = 0; it < nmy; ++it) {
    const int st = consume(it);
    if (ok) {
#pragma unroll
      for (int x = 0; x < kTw; ++x) {
        const int t = tpar + 2 * x;
        if (t >= nq) break;
        float z[4];
        scores(st, it, t, z);
        lse_add2(m0[x], l0[x], z[0], z[1]);
        lse_add2(m1[x], l1[x], z[2], z[3]);
      }
    }
    release(it);
  }
  // Per warp: merge the four tq lanes of each row.
#pragma unroll
  for (int x = 0; x < kTw; ++x) {
    const int t = tpar + 2 * x;
    if (t >= nq) break;
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      lse_merge(m0[x], l0[x], __shfl_xor_sync(0xffffffffu, m0[x], o), __shfl_xor_sync(0xffffffffu, l0[x], o));
      lse_merge(m1[x], l1[x], __shfl_xor_sync(0xffffffffu, m1[x], o), __shfl_xor_sync(0xffffffffu, l1[x], o));
    }
    if (tq == 0) {
      wpart[((warp & 7) * kSvMaxQ + t) * kGroup + g] = make_float2(m0[x], l0[x]);
      wpart[((warp & 7) * kSvMaxQ + t) * kGroup + g + 8] = make_float2(m1[x], l1[x]);
    }
  }
  ok = __syncthreads_and(ok);
  if (tid < nq * kGroup) {   // row tid = (t, h): merge the 8 warps
    float m = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float2 v = wpart[w * kSvMaxQ * kGroup + tid];
      lse_merge(m, l, v.x, v.y);
    }
    cpart[tid] = make_float2(m, l);
  }
  __syncthreads();
  cluster_wait();   // every CTA of the cluster is running
  for (int e = tid; e < C * nq * kGroup; e += kSvThreads) {   // row e % (nq 16) into CTA e / (nq 16)
    const int row = e % (nq * kGroup), dst = e / (nq * kGroup);
    st_dsmem_f32x2(dsmem_addr(&lse_in[(rank * kSvMaxQ) * kGroup + row], dst), cpart[row]);
  }
  cluster_arrive();
  cluster_wait();
  if (tid < nq * kGroup) {   // row (t, h): merge the C partials
    float m = -INFINITY, l = 0.f;
#pragma unroll 1
    for (int q = 0; q < C; ++q) {
      const float2 v = lse_in[(q * kSvMaxQ) * kGroup + tid];
      lse_merge(m, l, v.x, v.y);
    }
    lse2[tid] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  // ------------------------------------------------------------- pass 2 --
  // g of every kernel of the CTA's chunks per token (16 heads summed across
  // the lanes of the MMA fragment), into gbuf; no barrier inside the loop.
#pragma unroll 1
  for (int it = 0; it < nmy; ++it) {
    const int st = consume(nmy + it);
    if (ok) {
#pragma unroll 1
      for (int t = tpar; t < nq; t += 2) {
        float z[4];
        scores(st, it, t, z);
        const float la = lse2[t * kGroup + g], lb = lse2[t * kGroup + g + 8];
        float s0 = 0.f, s1 = 0.f;
        if (la > -INFINITY) {
          s0 += fast_exp2(z[0] - la);
          s1 += fast_exp2(z[1] - la);
        }
        if (lb > -INFINITY) {
          s0 += fast_exp2(z[2] - lb);
          s1 += fast_exp2(z[3] - lb);
        }
        // Sum over the 8 head rows g (lanes tq, tq + 4, ..., tq + 28).
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, o);
          s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        if (g == 0) {
          float* gr = gbuf + t * (kSvMaxIt * kSvChunk) + it * kSvChunk + (warp & 7) * 8 + 2 * tq;
          gr[0] = s0 * (1.0f / kGroup);
          gr[1] = s1 * (1.0f / kGroup);
        }
      }
    }
    release(nmy + it);
  }
  __syncthreads();

  // ------------------------------------------------- block scores to owners --
  // Token t's scores go to CTA t % C, into owned row t / C.  Only kernels
  // visible to the token count; the kernel before the CTA's first is the
  // previous CTA's (merged in by the owner); blocks past the token's own
  // block are not its candidates and are not sent.
  {
    const int jb0 = 16 * k0, jb1 = min(16 * k1, nbt);
    const int kb0 = kSvChunk * k0, kend = kSvChunk * (k0 + nmy);   // kernels held in gbuf: [kb0, kend)
#pragma unroll 1
    for (int e = tid; e < nq * (jb1 - jb0); e += kSvThreads) {
      const int t = e / (jb1 - jb0), j = jb0 + e % (jb1 - jb0);
      if (j > (L - nq + t) / kBlock) continue;
      const int nv = min(nvis_of(t), kend);
      float r = -INFINITY;
      for (int k = max(4 * j - 1, kb0); k <= min(nv - 1, 4 * j + 3); ++k)
        r = fmaxf(r, gbuf[t * (kSvMaxIt * kSvChunk) + (k - kb0)]);
      st_dsmem_f32(dsmem_addr(rown + (t / C) * kSvMaxBlocks + j, t % C), r);
    }
    // The g of this CTA's last kernel (64 k1 - 1), for the next CTA's first block.
    for (int t = tid; t < nq; t += kSvThreads) {
      const int kl = kSvChunk * k1 - 1;
      const float gl = (kl >= kb0 && kl < kend && kl < nvis_of(t)) ? gbuf[t * (kSvMaxIt * kSvChunk) + (kl - kb0)] : -INFINITY;
      st_dsmem_f32(dsmem_addr(tails + rank * kSvMaxQ + t, t % C), gl);
    }
  }
  cluster_arrive();
  cluster_wait();

  // ------------------------------------------------------------- top-k --
#pragma unroll 1
  for (int t = rank; t < nq; t += C) {
    float* r = rown + (t / C) * kSvMaxBlocks;
    const int c = (L - nq + t) / kBlock;
    if (tid > 0 && tid < C && 16 * per * tid <= c)   // block 16 per q starts CTA q's range
      r[16 * per * tid] = fmaxf(r[16 * per * tid], tails[(tid - 1) * kSvMaxQ + t]);
    __syncthreads();
    SmemTopkScratch<kSvThreads>& tk = *reinterpret_cast<SmemTopkScratch<kSvThreads>*>(smem + lay.tk);
    select_topk_smem<kSvThreads>(r, c + 1, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax,
                                 p.block_idx + (unit0 + t) * p.kmax, p.n_sel + unit0 + t, tk,
                                 reinterpret_cast<uint32_t*>(smem + lay.bits),
                                 reinterpret_cast<unsigned long long*>(smem + lay.surv), tid);
    if (p.write_r)
      for (int j = tid; j < p.nbmax; j += kSvThreads) p.r_buf[(unit0 + t) * p.nbmax + j] = j <= c ? r[j] : -INFINITY;
    __syncthreads();
  }
}

// Clusters of C CTAs resident at once on the current device (cached).
int sv_active_clusters(int C) {
  static int cache[64][kSvMaxC + 1];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    const bool ok =
        cudaFuncSetAttribute(sel_verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSvSmem) == cudaSuccess &&
        cudaFuncSetAttribute(sel_verify_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    for (int c = 1; c <= kSvMaxC; ++c) {
      int n = 0;
      if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(kSvThreads, 1, 1);
        cfg.dynamicSmemBytes = kSvSmem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = c;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, sel_verify_kernel, &cfg) != cudaSuccess) n = 0;
      }
      cache[dev][c] = n;
    }
    cudaGetLastError();
    done[dev] = true;
  }
  return cache[dev][C];
}

bool sv_fits(const Shape& s, int C) {
  const int groups = (s.nbmax + 15) / 16;
  return s.nq >= 2 && s.nq <= kSvMaxQ && (s.nq + C - 1) / C <= kSvOwnedRows && (groups + C - 1) / C <= kSvMaxIt &&
         s.nbmax <= kSvMaxBlocks;
}

}  // namespace

// The cluster size for the verify selection of this shape (0 if none fits):
// every group's cluster resident at once, then the most CTAs per group.
int select_verify_cluster_size(const Shape& s) {
  const int G = s.B * s.Hkv;
  for (int C = kSvMaxC; C >= 4; --C)
    if (sv_fits(s, C) && sv_active_clusters(C) >= G) return C;
  return 0;
}

cudaError_t launch_select_verify(const Shape& s, int cluster, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                                 const int32_t* kv_lens, int32_t* block_idx, int32_t* n_sel, float* r_buf,
                                 uint32_t* status, cudaStream_t st) {
  if (cluster < 1 || !sv_fits(s, cluster) || sv_active_clusters(cluster) < 1) return cudaErrorInvalidConfiguration;
  SvParams p{};
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
  p.write_r = r_buf != nullptr;
  p.scale2 = s.score_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.r_buf = r_buf;
  p.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, s.B * s.Hkv, 1);
  cfg.blockDim = dim3(kSvThreads, 1, 1);
  cfg.dynamicSmemBytes = kSvSmem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = cluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sel_verify_kernel, kc_map, q_map, p);
}

}  // namespace infllmv2
