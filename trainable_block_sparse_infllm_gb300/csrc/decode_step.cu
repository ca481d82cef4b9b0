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
//             blocks, pushed to the group's owner CTA.  The kernel 64k - 1
//             shared with the previous CTA is merged in by the owner.
//   top-k     the owner holds all block scores in registers, selects
//             (bitmask top-k) and pushes the list to every CTA.
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
constexpr int kDsCtaOOff = 16384;     // CTA partial O: stage 0's V half
constexpr int kDsZOff = 2 * 32768;    // phase-A scores: the stage slot phase A leaves free
static_assert(kDsMaxIt * kGroup * kDsChunk * 4 <= 32768, "phase-A scores fit one stage slot");

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
  int bits, surv, rfull, glall, q, wpart, cpart, lse, gbuf, wtab, sel, cta_ml, warp_ml, wgt, items, bar, total;
};

// The stage area (kDsPairs x 32 KB) holds, in turn: the phase-A chunks; in
// the owner CTA the gathered block scores and the top-k scratch (other CTAs
// write the scores there only after every CTA's phase A); the attention K/V
// tiles; the per-warp O partials.
__host__ __device__ inline DsLayout ds_layout(int nbmax, int kmax) {
  DsLayout l;
  l.bits = (static_cast<int>(sizeof(SmemTopkScratch<kDsThreads>)) + 15) & ~15;
  l.surv = (l.bits + (nbmax + 31) / 32 * 4 + 15) & ~15;
  l.rfull = l.surv + nbmax * 8;
  l.glall = l.rfull + nbmax * 4;
  l.q = kDsPairs * kDsStageBytes;
  l.wpart = l.q + 4096;
  l.cpart = l.wpart + 8 * kGroup * 8;
  l.lse = l.cpart + kGroup * 8;
  l.gbuf = l.lse + kGroup * 4;
  l.wtab = l.gbuf + kDsMaxIt * kDsChunk * 4;
  l.sel = l.wtab + 8 * kGroup * 4;
  l.cta_ml = (l.sel + kmax * 4 + 15) & ~15;
  l.warp_ml = l.cta_ml + kGroup * 8;
  l.wgt = l.warp_ml + 2 * kDsPairs * kGroup * 8;
  l.items = l.wgt + 2 * kDsPairs * kGroup * 4;   // item counter + two mailbox slots per pair
  l.bar = (l.items + (1 + 2 * kDsPairs) * 4 + 15) & ~15;
  l.total = l.bar + (2 * kDsStages + 1 + kDsPairs) * 8;
  return l;
}

__host__ __device__ inline int ds_per(int groups, int C) { return (groups + C - 1) / C; }

// Barrier of the two warps of attention pair `pair` (ids 1..3; 0 is __syncthreads).
__device__ __forceinline__ void pair_sync(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(pair + 1) : "memory");
}

// K and V tiles of one block into L2 (no shared memory, no completion).
__device__ __forceinline__ void prefetch_block(const CUtensorMap* kmap, const CUtensorMap* vmap, int row) {
  tma_prefetch_2d(kmap, 0, row);
  tma_prefetch_2d(kmap, 64, row);
  tma_prefetch_2d(vmap, 0, row);
  tma_prefetch_2d(vmap, 64, row);
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
  float* wtab = reinterpret_cast<float*>(smem + lay.wtab);       // [8 warps][16 heads] exponential weights
  float* rfull = reinterpret_cast<float*>(smem + lay.rfull);     // owner: [nbmax] all block scores
  float* glall = reinterpret_cast<float*>(smem + lay.glall);     // owner: [C] each CTA's last-kernel g
  int* item_ctr = reinterpret_cast<int*>(smem + lay.items);      // next attention item of this CTA
  int* pair_next = item_ctr + 1;                                 // [pairs][2] mailbox
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
  // The CTA that gathers the block scores and selects; it differs between
  // neighbouring groups so that two clusters sharing SMs do not stack their
  // selections on one SM.
  const int owner = bh % C;
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
    *item_ctr = kDsPairs;
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {   // Q does not depend on the length: start it first
    mbar_arrive_expect_tx(qbar, 4096);
    tma_load_2d(smem + lay.q, &q_map, 0, static_cast<int>(orow), qbar);
    tma_load_2d(smem + lay.q + 2048, &q_map, 64, static_cast<int>(orow), qbar);
  }

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
    mbar_wait(qbar, 0, p.status);   // no copy may still be landing in this CTA's memory
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
  const int kv_row0 = bh * p.Lmax;
  if (rank == owner && warp == 2) {
    // The forced blocks are known now: their K/V head for L2 at once.
    const int n_first = min(p.n_init, c + 1);
    const int lo = max(n_first, c - p.n_local + 1);
    const int n_f = n_first + max(0, c - lo + 1);
    for (int x = lane; x < n_f; x += 32)
      prefetch_block(&k_map, &v_map, kv_row0 + (x < n_first ? x : lo + x - n_first) * kBlock);
  }
  if (it_new >= 0 && warp == 7) {
    // The 32 keys of the newest kernel (8 KB): into L2 while Q and the first chunks load.
    const char* kr = reinterpret_cast<const char*>(p.k + (static_cast<size_t>(bh) * p.Lmax + jn * kStride) * kHeadDim);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + lane * 256));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + lane * 256 + 128));
  }
  if (tid == 0)
    for (int it = 0; it < min(kDsStages, nmy); ++it) issue(it);
  if (warp == 1) {
    // The rest of this CTA's chunks go to L2 now (one box per lane), so HBM
    // streams at full rate while the two shared-memory stages trail behind.
    for (int x = lane; x < 4 * (nmy - kDsStages); x += 32) {
      const int row = (k0 + kDsStages + (x >> 2)) * kDsChunk;
      tma_prefetch_2d(&kc_map, (x & 1) * 64, (bh * 2 + ((x >> 1) & 1)) * p.ncmax + row);
    }
  }

  // ------------------------------------------------------------ phase A --
  bool ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  // Newest kernel, by warp 7 while the other warps start on the chunks.
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

  const uint32_t q_b = smem_u32(smem + lay.q);
  // z (then exp2(z - warp max)) of chunk it, head h, kernel x of the chunk:
  // zs[(it * 16 + h) * 64 + x], in the stage slot phase A leaves free.
  float* zs = reinterpret_cast<float*>(smem + kDsZOff);
  float mx0 = -INFINITY, mx1 = -INFINITY;   // this warp's max of heads g and g + 8
  {
    uint32_t a[8][4];
    load_q_frags(a, q_b, lane);
#pragma unroll 1
    for (int it = 0; it < nmy; ++it) {
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
      float z0 = -INFINITY, z1 = -INFINITY, z2 = -INFINITY, z3 = -INFINITY;
      if (ok) {
        const uint32_t hi_b = smem_u32(smem + st * kDsStageBytes);
        const int kj = (k0 + it) * kDsChunk + warp * 8 + 2 * tq;
        float acc[4];
        score_ntile(acc, a, hi_b, hi_b + 16384, warp * 8, kDsChunk, lane);
        const bool v0 = kj < nc, v1 = kj + 1 < nc;
        z0 = v0 ? acc[0] * p.score_scale2 : -INFINITY;
        z1 = v1 ? acc[1] * p.score_scale2 : -INFINITY;
        z2 = v0 ? acc[2] * p.score_scale2 : -INFINITY;
        z3 = v1 ? acc[3] * p.score_scale2 : -INFINITY;
        mx0 = fmaxf(mx0, fmaxf(z0, z1));
        mx1 = fmaxf(mx1, fmaxf(z2, z3));
      }
      float* zrow = zs + (it * kGroup + g) * kDsChunk + warp * 8 + 2 * tq;
      *reinterpret_cast<float2*>(zrow) = make_float2(z0, z1);
      *reinterpret_cast<float2*>(zrow + 8 * kDsChunk) = make_float2(z2, z3);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (tid == 0 && ok && it + kDsStages < nmy) {
        if (mbar_wait(&empty[st], ph, p.status)) issue(it + kDsStages);
      }
      __syncwarp();
    }
  }

  // --------------------------------------------------- LSE over the cluster --
  // Row g holds head g, row g + 8 head g + 8; the four tq lanes share a row.
  // Each thread turns its own z into exp2(z - warp max) in place.
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  float l0 = 0.f, l1 = 0.f;
#pragma unroll 4
  for (int it = 0; it < nmy; ++it) {
    float2* z01 = reinterpret_cast<float2*>(zs + (it * kGroup + g) * kDsChunk + warp * 8 + 2 * tq);
    float2* z23 = reinterpret_cast<float2*>(reinterpret_cast<float*>(z01) + 8 * kDsChunk);
    float2 u = *z01, w = *z23;
    u.x = (mx0 == -INFINITY) ? 0.f : fast_exp2(u.x - mx0);
    u.y = (mx0 == -INFINITY) ? 0.f : fast_exp2(u.y - mx0);
    w.x = (mx1 == -INFINITY) ? 0.f : fast_exp2(w.x - mx1);
    w.y = (mx1 == -INFINITY) ? 0.f : fast_exp2(w.y - mx1);
    *z01 = u;
    *z23 = w;
    l0 += u.x + u.y;
    l1 += w.x + w.y;
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
  if (tid < 8 * kGroup) {   // head tid / 8, warp tid % 8: a shuffle tree over the 8 warps
    const float2 v = wpart[(tid & 7) * kGroup + (tid >> 3)];
    float m = v.x, l = v.y;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
      lse_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if ((tid & 7) == 0) cpart[tid >> 3] = make_float2(m, l);
  }
  cluster_sync();
  if (tid < C * kGroup) {   // head tid / C, CTA tid % C: one remote load each, then a shuffle tree
    const float2 v = ld_dsmem_f32x2(dsmem_addr(&cpart[tid / C], tid % C));
    float m = v.x, l = v.y;
#pragma unroll
    for (int o = 1; o < C; o <<= 1)
      lse_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if (tid % C == 0) lse2[tid / C] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  // ------------------------------------------------------------ phase B --
  // Weight of warp w's exponentials of head h: exp2(max_wh - lse_h) / 16.
  if (tq == 0) {
    wtab[warp * kGroup + g] = (mx0 == -INFINITY) ? 0.f : fast_exp2(mx0 - lse2[g]) * (1.0f / kGroup);
    wtab[warp * kGroup + g + 8] = (mx1 == -INFINITY) ? 0.f : fast_exp2(mx1 - lse2[g + 8]) * (1.0f / kGroup);
  }
  __syncthreads();
  // g of every kernel of this CTA's chunks (kernel x of a chunk came from warp x / 8).
#pragma unroll 1
  for (int k = tid; k < nmy * kDsChunk; k += kDsThreads) {
    const int it = k / kDsChunk, x = k % kDsChunk;
    const float* zc = zs + it * kGroup * kDsChunk + x;
    const float* wt = wtab + (x >> 3) * kGroup;
    float acc = 0.f;
#pragma unroll
    for (int h = 0; h < kGroup; ++h) acc += zc[h * kDsChunk] * wt[h];
    gbuf[k] = acc;
  }
  __syncthreads();
  {
    const int jb0 = 16 * k0, jb1 = min(16 * k1, nbt);
    const int kb0 = kDsChunk * k0;
#pragma unroll 1
    for (int j = jb0 + tid; j < jb1; j += kDsThreads) {
      const int a0 = max(4 * j - 1, kb0), e0 = min(nc - 1, 4 * j + 3);
      float r = -INFINITY;
      for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - kb0]);
      st_dsmem_f32(dsmem_addr(rfull + j, owner), r);   // the owner gathers every block score
    }
    if (tid == 0) {
      const float gl = (k1 > k0 && kDsChunk * k1 - 1 < nc) ? gbuf[kDsChunk * (k1 - k0) - 1] : -INFINITY;
      st_dsmem_f32(dsmem_addr(glall + rank, owner), gl);
    }
  }
  cluster_sync();

  // ------------------------------------------------------------- top-k --
  if (rank == owner) {
    // Block 16 per q starts CTA q's range; its kernel 64 per q - 1 was scored by CTA q - 1.
    if (tid > 0 && tid < C && 16 * per * tid < nbt)
      rfull[16 * per * tid] = fmaxf(rfull[16 * per * tid], glall[tid - 1]);
    __syncthreads();
    SmemTopkScratch<kDsThreads>& tk = *reinterpret_cast<SmemTopkScratch<kDsThreads>*>(smem);
    select_topk_smem<kDsThreads>(rfull, nbt, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax,
                                 p.block_idx + static_cast<size_t>(bh) * p.kmax, p.n_sel + bh, tk,
                                 reinterpret_cast<uint32_t*>(smem + lay.bits),
                                 reinterpret_cast<unsigned long long*>(smem + lay.surv), tid, selS);
    __syncthreads();
    // Every CTA gets the list in its own shared memory.
#pragma unroll 1
    for (int e = tid; e < C * p.kmax; e += kDsThreads) {
      const int q = e / p.kmax, x = e % p.kmax;
      if (q != owner) st_dsmem_u32(dsmem_addr(selS + x, q), static_cast<uint32_t>(selS[x]));
    }
  }
  cluster_sync();

  // ------------------------------------------------------------ attend --
  const int pair = warp >> 1, half = warp & 1;
  if (pair < kDsPairs) {
    uint8_t* stage = smem + pair * kDsStageBytes;
    const uint32_t k_b = smem_u32(stage), v_b = k_b + 16384;
    const int rbase = 32 * half;
    // Item x of this CTA is list entry rank + C x: items 0..2 go to pairs
    // 0..2, each later one to whichever pair frees its stage first.
    auto block_of = [&](int item) {
      const int n = rank + C * item;
      const int j = n < p.kmax ? selS[n] : -1;
      return j > c ? -1 : j;
    };
    int j = block_of(pair);
    if (half == 0 && lane == 0 && j >= 0) tma_block(stage, &k_map, &v_map, kv_row0 + j * kBlock, &kvfull[pair]);

    float o[16][4];
#pragma unroll
    for (int x = 0; x < 16; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;
    l0 = 0.f;
    l1 = 0.f;
    uint32_t phase = 0;
    int iter = 0;
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
      // Next item of this pair: drawn by the even warp, shared through a
      // two-slot mailbox (a slot is rewritten only two pair barriers later).
      if (half == 0 && lane == 0) pair_next[pair * 2 + (iter & 1)] = atomicAdd(item_ctr, 1);
      // Both warps are done with the stage; order the zeroed V rows
      // (generic writes) before the TMA refill (async proxy).
      fence_proxy_async_smem();
      pair_sync(pair);
      j = block_of(pair_next[pair * 2 + (iter & 1)]);
      ++iter;
      if (j >= 0 && half == 0 && lane == 0 && ok)
        tma_block(stage, &k_map, &v_map, kv_row0 + j * kBlock, &kvfull[pair]);
    }
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
#pragma unroll 1
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
  return s.nq == 1 && ds_per(groups, C) <= kDsMaxIt &&
         l.glall + 16 * 4 <= kDsZOff && l.total + 1024 <= 113 * 1024;
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
