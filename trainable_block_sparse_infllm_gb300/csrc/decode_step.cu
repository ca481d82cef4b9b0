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
// One CTA per SM (its shared memory keeps a second one off); the cluster
// size C (1..16) is chosen at launch so that every group's cluster is
// resident at once.  CTA r owns the 16-block groups [r per, (r + 1) per) and
// the matching 64-kernel chunks (the kernels of blocks [16k, 16k + 16) are
// 64k - 1 .. 64k + 63).  One 192 KB region of shared memory serves, in turn,
// the phase-A ring and scores, the block scores and top-k scratch, and the
// attention stages.
//   append    (infllmv2_append_decode_step only) the phase-A warps load q
//             with ordinary loads instead of the TMA, since it may sit in
//             host memory; CTA 0 stores the token's key and value rows into
//             the caches, which the other CTAs' TMA loads read only after
//             the cluster barrier that follows phase A.
//   compress  the CTA whose chunks hold the newest complete kernel recomputes
//             it from the keys with the compression kernel's arithmetic
//             (an appended key taken from its source row),
//             stores it in the kernel-mean planes and patches its own
//             shared-memory copy of the chunk.
//   phase A   hi/lo chunks streamed by TMA through a 4-stage ring (the rest
//             of the CTA's chunks head for L2 at once); z = score_scale
//             q . Mean on the tensor cores (8 warps), kept in shared memory.
//   LSE       phase A already stores exp2(z - m) with m the running max of
//             the warp's row and keeps the row sums, so the warps' (max, sum)
//             merge at once into the CTA's per head, which is pushed into
//             every CTA of the cluster; after one cluster barrier each CTA
//             merges the C partials itself -> exact lse per head.
//   phase B   g = (1/16) sum_h exp2(z - lse_h) from the stored exponentials
//             and one weight per (chunk, warp, head); block maxima of the
//             CTA's blocks; its candidates ranked among themselves.
//   top-k     each CTA sends every CTA one message (bulk copy, counted on
//             the receiver's mbarrier): its best n_take keys (score, then
//             index) sorted, its first block's partial score and its last
//             kernel's g; each CTA ranks its own entries against all the
//             lists (binary searches) and sends its winners as a bit mask
//             (st.async, a second mbarrier); every CTA assembles the same
//             ascending selection, which CTA 0 writes.
//   attend    the selected blocks rank, rank + C, ... are dealt to six warp
//             pairs; a pair TMA-loads one block's K and V tiles (32 KB) into
//             its stage, and each warp of the pair takes 32 of its keys:
//             S = Q K^T on the tensor cores, online softmax in base 2,
//             O += P V with P fed as bf16 hi + lo.  Blocks of a second round
//             head for L2 as soon as the selection is known.
//   merge     warps merge in shared memory; each head's CTA partial is
//             pushed to the CTA that writes the head (head h: CTA h mod C),
//             which, after one cluster barrier, merges the C partials.
// Every remote access (a store, a bulk copy or an st.async) is complete
// before the last cluster barrier: the stores are released by a barrier
// arrive, the copies and st.async land before their receivers' mbarrier
// waits end.  After the last barrier a CTA only reads its own shared
// memory, so it may exit.
#include "compress.cuh"
#include "select_common.cuh"

namespace infllmv2 {

namespace {

constexpr int kDsThreads = 384;
constexpr int kDsWarps = kDsThreads / 32;
constexpr int kDsAWarps = 8;          // phase-A warps: one 8-kernel n-tile each per chunk
constexpr int kDsProducer = 8;        // warp issuing the phase-A ring loads
constexpr int kDsChunk = 64;          // kernels per phase-A stage
constexpr int kDsRing = 4;            // phase-A stages
constexpr int kDsPairs = kDsWarps / 2;   // attention warp pairs, one stage each
constexpr int kDsStageBytes = 32768;  // 64 kernels hi + lo, or one block's K + V
constexpr int kDsRegion = kDsPairs * kDsStageBytes;
constexpr int kDsZOff = kDsRing * kDsStageBytes;   // phase-A scores after the ring
constexpr int kDsMaxIt = (kDsRegion - kDsZOff) / (kGroup * kDsChunk * 4);   // chunks per CTA
constexpr int kDsMaxC = 16;
constexpr int kDsOutRows = 32;        // C * ceil(16 / C) <= 30 partial rows a CTA may receive
constexpr int kDsMaxBlocks = 4096;    // block scores over the region's first 16 KB
constexpr int kDsGbufOff = 65536;     // g of the CTA's kernels: in the ring, after the phase
constexpr int kDsRmineOff = kDsGbufOff + kDsMaxIt * kDsChunk * 4;
constexpr int kDsListMax = 256;       // best candidates a CTA sends (n_take <= k_max <= 256)
constexpr int kDsMsgBytes = 16 + kDsListMax * 8;   // a CTA's message: DsSummary, then its sorted keys
constexpr int kDsRecvOff = 0;         // [C][kDsMsgBytes] the messages of every CTA (the ring is idle by then)
constexpr int kDsLkeyOff = kDsRmineOff + 16 * kDsMaxIt * 4;   // this CTA's candidate keys
constexpr int kDsSendOff = kDsLkeyOff + 16 * kDsMaxIt * 8;    // this CTA's message
constexpr int kDsMaskWords = 12;      // a CTA's blocks in selection words (16 kDsMaxIt blocks from a 16-aligned start)
// Selection bits [128 words], first-block keys [16], counters [16], this
// CTA's winners [12 words], the winners of every CTA [16][12 words].
constexpr int kDsSelOff = kDsSendOff + kDsMsgBytes;
constexpr int kDsBkeyOff = kDsSelOff + kDsMaxBlocks / 8;
constexpr int kDsCtrOff = kDsBkeyOff + kDsMaxC * 8;
constexpr int kDsRmaskOff = kDsCtrOff + 16 * 4;
constexpr int kDsMinOff = kDsRmaskOff + 64;
static_assert(kDsMaxIt >= 16, "16 chunks per CTA");
static_assert(kDsMsgBytes % 16 == 0 && kDsSendOff % 16 == 0 && kDsMinOff % 16 == 0, "bulk copies and st.async");
static_assert((16 * kDsMaxIt + 31) / 32 + 1 <= kDsMaskWords, "a CTA's blocks fit its mask");
static_assert(kDsRecvOff + kDsMaxC * kDsMsgBytes <= kDsGbufOff, "messages ahead of the phase-B buffers");
static_assert(kDsMinOff + kDsMaxC * kDsMaskWords * 4 <= kDsZOff, "phase-B buffers inside the ring");

// Pushed per CTA before the second barrier.
struct DsSummary {
  float tail;         // g of the CTA's last kernel (-inf if it has none)
  float first;        // score of its first block without the kernel before it (-inf if none)
  int n_list;         // candidates in its sorted list (its first block excluded)
  int pad;
};

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
  uint32_t test_flags;   // checked build: kTestWithholdArrive makes a bounded wait expire
  // Fused cache append (all null when the caller has appended the token):
  // the newest token's q, k and v rows, read with ordinary loads (they may be
  // page-locked host memory), and the caches that take its k and v.
  const uint4* q_src;    // [B][Hq][16 chunks]
  const uint4* k_new;    // [B * Hkv][16 chunks]
  const uint4* v_new;
  uint4* k_w;            // the k and v caches, [B * Hkv * Lmax][16 chunks]
  uint4* v_w;
};

// Fault injection of the checked build's own tests: warp 0 of every CTA
// does not release the ring stage of its first chunk, so the producer's
// bounded wait for that stage expires (TIMEOUT), no later chunk is issued,
// and the phase-A warps' waits for those chunks expire too; every copy that
// was issued has landed before the CTA moves on.
#ifdef INFLLMV2_CHECKED
constexpr uint32_t kTestWithholdArrive = 0x1u;
#endif

// Shared memory after the region (fixed sizes: the footprint, and with it
// the cluster occupancy, does not depend on the shape).
struct DsLayout {
  int q, lse_in, o_in, ml_in, wpart, cpart, lse, sel, nsel, warp_ml, wgt, bar, total;
};

__host__ __device__ constexpr DsLayout ds_layout() {
  DsLayout l{};
  l.q = kDsRegion;                                 // 16 rows x 256 B, two swizzled boxes
  l.lse_in = l.q + 4096;                           // [16 CTAs][16 heads] (max, sum)
  l.o_in = l.lse_in + kDsMaxC * kGroup * 8;        // [32 rows][128] partial O of the heads written here
  l.ml_in = l.o_in + kDsOutRows * kHeadDim * 4;    // [32 rows] their (max, sum)
  l.wpart = l.ml_in + kDsOutRows * 8;              // [8 warps][16 heads] (max, sum)
  l.cpart = l.wpart + kDsAWarps * kGroup * 8;      // [16] CTA (max, sum)
  l.lse = l.cpart + kGroup * 8;                    // [16] lse per head (base 2)
  l.sel = l.lse + kGroup * 4;                      // [kmax <= 256] ascending, -1 padded
  l.nsel = l.sel + 256 * 4;
  l.warp_ml = l.nsel + 16;                         // [12 warps][16 heads] attention (max, sum)
  l.wgt = l.warp_ml + kDsWarps * kGroup * 8;       // [12 warps][16 heads] merge weights, then [16][16]
  l.bar = l.wgt + 16 * 16 * 4;
  l.total = l.bar + (2 * kDsRing + 1 + kDsPairs + 2) * 8;
  return l;
}

constexpr int kDsSmem = ds_layout().total + 1024;   // + 1024-byte alignment slack
// Phase A's running maxima per (chunk, warp, head), turned into phase B's
// weights, lie over the merge's partial-O rows (written only after the
// cluster barrier that follows phase B).
static_assert(kDsMaxIt * kDsAWarps * kGroup <= kDsOutRows * kHeadDim, "weight table inside o_in");
static_assert(kDsSmem <= 227 * 1024, "one CTA per SM");

__host__ __device__ inline int ds_per(int groups, int C) { return (groups + C - 1) / C; }

// Likely winners a CTA prefetches into L2 before the selection is known.
__host__ __device__ inline int ds_prefetch_count(int n_take, int C) { return (n_take + C - 1) / C + 2; }

// Barrier of the two warps of attention pair `pair` (ids 1..6; 0 is __syncthreads).
__device__ __forceinline__ void pair_sync(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(pair + 1) : "memory");
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
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

// kAppend: the cache append is fused in (a separate instantiation, so the
// plain step carries none of its code: this kernel's one-pass code is paced
// by instruction fetch).
template <bool kAppend>
__global__ void __launch_bounds__(kDsThreads, 1)
    decode_step_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap q_map,
                       const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                       DsParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr DsLayout lay = ds_layout();
  float* zs = reinterpret_cast<float*>(smem + kDsZOff);              // [it][16 heads][64]
  float* gbuf = reinterpret_cast<float*>(smem + kDsGbufOff);         // g of this CTA's kernels
  float* rmine = reinterpret_cast<float*>(smem + kDsRmineOff);       // this CTA's first block score
  uint8_t* recv = smem + kDsRecvOff;                                 // [C][kDsMsgBytes] messages
  uint8_t* send = smem + kDsSendOff;                                 // this CTA's message
  unsigned long long* lkeys = reinterpret_cast<unsigned long long*>(smem + kDsLkeyOff);   // this CTA's candidates
  uint32_t* sbits = reinterpret_cast<uint32_t*>(smem + kDsSelOff);                        // [128] selected blocks
  unsigned long long* bkeys = reinterpret_cast<unsigned long long*>(smem + kDsBkeyOff);   // [C] first blocks
  int* sctr = reinterpret_cast<int*>(smem + kDsCtrOff);              // [0] n_loc, [4..16) warp sums
  uint32_t* rmask = reinterpret_cast<uint32_t*>(smem + kDsRmaskOff);                      // this CTA's winners
  uint32_t* minbox = reinterpret_cast<uint32_t*>(smem + kDsMinOff);                      // [C][12] every CTA's
  float2* lse_in = reinterpret_cast<float2*>(smem + lay.lse_in);     // [C][16]
  float* o_in = reinterpret_cast<float*>(smem + lay.o_in);           // [C * hmax][128]
  float2* ml_in = reinterpret_cast<float2*>(smem + lay.ml_in);       // [C * hmax]
  float2* wpart = reinterpret_cast<float2*>(smem + lay.wpart);
  float2* cpart = reinterpret_cast<float2*>(smem + lay.cpart);
  float* lse2 = reinterpret_cast<float*>(smem + lay.lse);
  float* mch = reinterpret_cast<float*>(smem + lay.o_in);            // [chunk][warp][head] (over o_in)
  int32_t* selS = reinterpret_cast<int32_t*>(smem + lay.sel);
  int32_t* nselS = reinterpret_cast<int32_t*>(smem + lay.nsel);
  float2* warp_ml = reinterpret_cast<float2*>(smem + lay.warp_ml);
  float* wgt = reinterpret_cast<float*>(smem + lay.wgt);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bar);
  uint64_t* empty = full + kDsRing;
  uint64_t* qbar = empty + kDsRing;
  uint64_t* kvfull = qbar + 1;
  uint64_t* lbar = kvfull + kDsPairs;   // every CTA's message has landed
  uint64_t* sbar = lbar + 1;            // every CTA's winners have landed

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int rank = static_cast<int>(cluster_ctarank());
  const int C = static_cast<int>(cluster_nctarank());
  const int hmax = (kGroup + C - 1) / C;   // heads a CTA writes at most (head h: CTA h % C)
  const int bh = blockIdx.y;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const size_t orow = static_cast<size_t>(b) * Hq + static_cast<size_t>(h) * kGroup;

  if (tid == 0) {
    prefetch_tensormap(&kc_map);
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    for (int s = 0; s < kDsRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDsAWarps);
    }
    mbar_init(qbar, kAppend ? kDsAWarps : 1);   // the q tile: one TMA load, or the phase-A warps' stores
    for (int s = 0; s < kDsPairs; ++s) mbar_init(&kvfull[s], 1);
    mbar_init(lbar, 1);
    mbar_init(sbar, 1);
    fence_barrier_init();
  }
  // Marks this CTA as running; the matching wait, before the first remote
  // store, makes sure every CTA of the cluster is.
  cluster_arrive_relaxed();
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (kAppend) {
    // Fused append: the group's 16 q rows (4 KB) by the phase-A warps, one
    // 16-byte chunk per thread, into the layout the TMA load would give.
    if (warp < kDsAWarps) {
      const int r = tid >> 4, ch = tid & 15;
      *reinterpret_cast<uint4*>(smem + lay.q + swz128_offset(r, ch, kGroup)) = p.q_src[(orow + r) * 16 + ch];
      __syncwarp();
      if (lane == 0) mbar_arrive(qbar);
    }
  } else if (tid == 0) {   // Q does not depend on the length: start it first
    mbar_arrive_expect_tx(qbar, 4096);
    tma_load_2d(smem + lay.q, &q_map, 0, static_cast<int>(orow), qbar);
    tma_load_2d(smem + lay.q + 2048, &q_map, 64, static_cast<int>(orow), qbar);
  }

  const int L = p.kv_lens[b];
  const int nbt = L >= 1 ? (L - 1) / kBlock + 1 : 0;
  const int groups = (nbt + 15) / 16;
  const int per = ds_per(groups, C);
  if (L < 1 || L > p.Lmax || per > kDsMaxIt || nbt > kDsMaxBlocks) {   // same for every CTA of the cluster
    if (rank == 0) {
#pragma unroll 1
      for (int e = tid; e < p.kmax; e += kDsThreads) p.block_idx[static_cast<size_t>(bh) * p.kmax + e] = -1;
#pragma unroll 1
      for (int e = tid; e < kGroup * kHeadDim; e += kDsThreads) p.out[orow * kHeadDim + e] = __float2bfloat16(0.f);
      if (tid < kGroup && p.lse) p.lse[orow + tid] = -INFINITY;
      if (tid == 0) {
        p.n_sel[bh] = 0;
        atomicOr(p.status, kStatusBadKvLen);
      }
    }
    mbar_wait(qbar, 0, p.status);   // no copy may still be landing in this CTA's memory
    cluster_wait();
    return;
  }
  const int i = L - 1, c = i / kBlock;
  const int k0 = min(groups, rank * per), k1 = min(groups, (rank + 1) * per);
  const int nc = n_complete_kernels(L);
  const int nmy = max(0, min(k1, (nc + kDsChunk - 1) / kDsChunk) - k0);
  const int jn = nc - 1;   // newest complete kernel
  const int it_new = (jn >= 0 && jn / kDsChunk >= k0 && jn / kDsChunk < k0 + nmy) ? jn / kDsChunk - k0 : -1;
  const size_t plane_rows = static_cast<size_t>(p.ncmax) * kHeadDim;
  const int n_first = min(p.n_init, c + 1);
  const int local_lo = max(n_first, c - p.n_local + 1);
  const int n_forced = n_first + max(0, c - local_lo + 1);
  const int n_take = max(0, p.inc_forced ? p.topk - n_forced : p.topk);
  // Power of two >= n_take (and >= 2, so that a message is a multiple of 16 bytes), <= 256.
  const int list_pow = n_take <= 2 ? 2 : 1 << (32 - __clz(n_take - 1));
  const uint32_t msg_bytes = 16 + list_pow * 8;   // a CTA's message to each CTA of the cluster
  if (tid == 0) {   // (no CTA sends before the first cluster barrier, which comes later)
    mbar_arrive_expect_tx(lbar, static_cast<uint32_t>(C) * msg_bytes);
    mbar_arrive_expect_tx(sbar, static_cast<uint32_t>(C) * kDsMaskWords * 4);
  }

  auto issue = [&](int it) {
    const int st = it % kDsRing;
    const int row = (k0 + it) * kDsChunk;
    uint8_t* dst = smem + st * kDsStageBytes;
    mbar_arrive_expect_tx(&full[st], kDsStageBytes);
    tma_load_2d(dst, &kc_map, 0, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 8192, &kc_map, 64, (bh * 2 + 0) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 16384, &kc_map, 0, (bh * 2 + 1) * p.ncmax + row, &full[st]);
    tma_load_2d(dst + 24576, &kc_map, 64, (bh * 2 + 1) * p.ncmax + row, &full[st]);
  };
  const int kv_row0 = bh * p.Lmax;
  if (kAppend && rank == 0 && warp == 10) {
    // Fused append: the token's key and value rows into the caches (row
    // L - 1).  Other CTAs' TMA loads read them only after the cluster barrier
    // that follows phase A (release here, acquire there); the newest kernel
    // below takes the key from k_new itself.
    const size_t row = static_cast<size_t>(kv_row0) + (L - 1);
    const int ch = lane & 15;
    if (lane < 16)
      p.k_w[row * 16 + ch] = p.k_new[static_cast<size_t>(bh) * 16 + ch];
    else
      p.v_w[row * 16 + ch] = p.v_new[static_cast<size_t>(bh) * 16 + ch];
    fence_proxy_async_global();
  }
  if (warp == 9) {
    // The forced blocks are known now: their K/V head for L2 at once, each
    // from one CTA of the cluster.
#pragma unroll 1
    for (int x = rank + C * lane; x < n_forced; x += 32 * C)
      prefetch_block(&k_map, &v_map, kv_row0 + (x < n_first ? x : local_lo + x - n_first) * kBlock);
  }
  if (it_new >= 0 && warp == 11) {
    // The 32 keys of the newest kernel (8 KB): into L2 while Q and the first chunks load.
    const char* kr = reinterpret_cast<const char*>(p.k + (static_cast<size_t>(bh) * p.Lmax + jn * kStride) * kHeadDim);
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + lane * 256));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(kr + lane * 256 + 128));
  }
  if (warp == 10) {
    // The rest of this CTA's chunks go to L2 now (one box per lane), so HBM
    // streams at full rate while the shared-memory stages trail behind.
#pragma unroll 1
    for (int x = lane; x < 4 * (nmy - kDsRing); x += 32) {
      const int row = (k0 + kDsRing + (x >> 2)) * kDsChunk;
      tma_prefetch_2d(&kc_map, (x & 1) * 64, (bh * 2 + ((x >> 1) & 1)) * p.ncmax + row);
    }
  }
  if (tid == kDsProducer * 32)
#pragma unroll 1
    for (int it = 0; it < min(kDsRing, nmy); ++it) issue(it);

  // ------------------------------------------------------------ phase A --
  bool ok = __syncthreads_and(mbar_wait(qbar, 0, p.status));
  // Newest kernel, by warp 11 while warps 0-7 start on the chunks.
  // Warp 11: lane = 16 * half + sub sums chunk jn + half over dims [8 sub, 8 sub + 8).
  uint4 new_hi = make_uint4(0, 0, 0, 0), new_lo = make_uint4(0, 0, 0, 0);
  if (it_new >= 0 && warp == 11) {
    const __nv_bfloat16* kbh = p.k + static_cast<size_t>(bh) * p.Lmax * kHeadDim;
    const int sub = lane & 15, half = lane >> 4;
    float acc[8], oth[8];
    if (kAppend)
      chunk_sum16(acc, kbh, (jn + half) * kStride, sub, L - 1, p.k_new + static_cast<size_t>(bh) * 16);
    else
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
  // exp2(z - m) of chunk it, head h, kernel x of the chunk:
  // zs[(it * 16 + h) * 64 + x], with m the running max of the warp's row of
  // head h up to that chunk, kept in mch[(it * 8 + warp) * 16 + h].  The
  // rows' (max, sum) are thus ready when the last chunk is scored.
  float m0r = -INFINITY, m1r = -INFINITY;   // running max of this warp's rows of heads g and g + 8
  float ls0 = 0.f, ls1 = 0.f;                 // this thread's sums of exp2(z - running max)
  if (warp < kDsAWarps) {
    uint32_t a[8][4];
    load_q_frags(a, q_b, lane);
#pragma unroll 1
    for (int it = 0; it < nmy; ++it) {
      const int st = it % kDsRing;
      const uint32_t ph = static_cast<uint32_t>(it / kDsRing) & 1u;
      bool got = ok && mbar_wait(&full[st], ph, p.status);
      ok = __all_sync(0xffffffffu, got);
      // The chunk holding the newest kernel is read only after warp 11 has
      // patched it (named barrier 7: warps 0-7 and 11).
      if (it == it_new) asm volatile("bar.sync 7, %0;" ::"n"(kDsAWarps * 32 + 32) : "memory");
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
      }
      float c0 = fmaxf(z0, z1), c1 = fmaxf(z2, z3);
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {   // the row's 8 kernels of this chunk (4 tq lanes)
        c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, o));
        c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, o));
      }
      const float n0 = fmaxf(m0r, c0), n1 = fmaxf(m1r, c1);
      if (n0 > -INFINITY) {
        ls0 *= fast_exp2(m0r - n0);
        z0 = fast_exp2(z0 - n0);
        z1 = fast_exp2(z1 - n0);
        ls0 += z0 + z1;
      } else {
        z0 = z1 = 0.f;
      }
      if (n1 > -INFINITY) {
        ls1 *= fast_exp2(m1r - n1);
        z2 = fast_exp2(z2 - n1);
        z3 = fast_exp2(z3 - n1);
        ls1 += z2 + z3;
      } else {
        z2 = z3 = 0.f;
      }
      m0r = n0;
      m1r = n1;
      float* zrow = zs + (it * kGroup + g) * kDsChunk + warp * 8 + 2 * tq;
      *reinterpret_cast<float2*>(zrow) = make_float2(z0, z1);
      *reinterpret_cast<float2*>(zrow + 8 * kDsChunk) = make_float2(z2, z3);
      if (tq == 0) {
        mch[(it * kDsAWarps + warp) * kGroup + g] = n0;
        mch[(it * kDsAWarps + warp) * kGroup + g + 8] = n1;
      }
      __syncwarp();
#ifdef INFLLMV2_CHECKED
      if ((p.test_flags & kTestWithholdArrive) && warp == 0 && it == 0) continue;
#endif
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  } else if (warp == kDsProducer) {
    // Ring refills: chunk it + 4 into the stage chunk it leaves.
    if (lane == 0) {
#pragma unroll 1
      for (int it = 0; it + kDsRing < nmy && ok; ++it) {
        const int st = it % kDsRing;
        if (!mbar_wait(&empty[st], static_cast<uint32_t>(it / kDsRing) & 1u, p.status)) {
          ok = false;
          break;
        }
        issue(it + kDsRing);
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
  } else if (warp == 11 && it_new >= 0) {
    // Patch the newest kernel into its chunk once the chunk has landed,
    // before the phase-A warps read it (named barrier 7: warps 0-7 and 11).
    const int st = it_new % kDsRing;
    bool got = ok && mbar_wait(&full[st], static_cast<uint32_t>(it_new / kDsRing) & 1u, p.status);
    got = __all_sync(0xffffffffu, got);
    if (got && lane < 16) {
      uint8_t* stg = smem + st * kDsStageBytes;
      const uint32_t off = swz128_offset(jn - (k0 + it_new) * kDsChunk, lane, kDsChunk);
      *reinterpret_cast<uint4*>(stg + off) = new_hi;
      *reinterpret_cast<uint4*>(stg + 16384 + off) = new_lo;
    }
    asm volatile("bar.sync 7, %0;" ::"n"(kDsAWarps * 32 + 32) : "memory");
  }

  // --------------------------------------------------- LSE over the cluster --
  // Row g holds head g, row g + 8 head g + 8; the four tq lanes share a row
  // (and its running max) and sum their partial sums.
  if (warp < kDsAWarps) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, o);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, o);
    }
    if (tq == 0) {
      wpart[warp * kGroup + g] = make_float2(m0r, ls0);
      wpart[warp * kGroup + g + 8] = make_float2(m1r, ls1);
    }
  }
  ok = __syncthreads_and(ok);
  if (tid < kDsAWarps * kGroup) {   // head tid / 8, warp tid % 8: a shuffle tree over the 8 warps
    const float2 v = wpart[(tid & 7) * kGroup + (tid >> 3)];
    float m = v.x, l = v.y;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
      lse_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if ((tid & 7) == 0) cpart[tid >> 3] = make_float2(m, l);
  }
  __syncthreads();
  cluster_wait();   // every CTA of the cluster is running
  if (tid < C * kGroup)   // the CTA's partial of head tid % 16 into CTA tid / 16
    st_dsmem_f32x2(dsmem_addr(&lse_in[rank * kGroup + (tid % kGroup)], tid / kGroup), cpart[tid % kGroup]);
  cluster_arrive();
  cluster_wait();
  if (kAppend) fence_proxy_async_global();   // the appended rows, before this CTA's TMA loads of them
  if (tid < kGroup * kDsMaxC) {   // head tid / 16, CTA tid % 16: a shuffle tree over the C partials
    const int q = tid % kDsMaxC, hd = tid / kDsMaxC;
    const float2 v = q < C ? lse_in[q * kGroup + hd] : make_float2(-INFINITY, 0.f);
    float m = v.x, l = v.y;
#pragma unroll
    for (int o = 1; o < kDsMaxC; o <<= 1)
      lse_merge(m, l, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o));
    if (q == 0) lse2[hd] = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
  }
  __syncthreads();

  // ------------------------------------------------------------ phase B --
  // Weight of the exponentials of (chunk, warp, head h): exp2(m - lse_h) / 16
  // with m the running max they were taken against.
#pragma unroll 1
  for (int e = tid; e < nmy * kDsAWarps * kGroup; e += kDsThreads) {
    const float m = mch[e];
    mch[e] = (m == -INFINITY) ? 0.f : fast_exp2(m - lse2[e % kGroup]) * (1.0f / kGroup);
  }
  // (the ring is idle since phase A: the selection's buffers lie in it)
#pragma unroll 1
  for (int w = tid; w < kDsMaxBlocks / 32; w += kDsThreads) sbits[w] = 0u;
  if (tid == 0) sctr[0] = 0;
  __syncthreads();
  // g of every kernel of this CTA's chunks (kernel x of a chunk came from warp x / 8).
#pragma unroll 1
  for (int k = tid; k < nmy * kDsChunk; k += kDsThreads) {
    const int it = k / kDsChunk, x = k % kDsChunk;
    const float* zc = zs + it * kGroup * kDsChunk + x;
    const float* wt = mch + (it * kDsAWarps + (x >> 3)) * kGroup;
    float acc = 0.f;
#pragma unroll
    for (int hh = 0; hh < kGroup; ++hh) acc += zc[hh * kDsChunk] * wt[hh];
    gbuf[k] = acc;
  }
  __syncthreads();
  // ------------------------------------------------------------- top-k --
  // Candidates are the blocks n_first .. local_lo - 1 with a finite score,
  // ordered by one 64-bit key: the score, then the lower index.  Each CTA
  // sorts its own candidates (all but its first block, whose kernel before
  // it was scored by the previous CTA) and sends every CTA one message: the
  // g of its last kernel, its first block's partial score, and its best
  // n_take keys, sorted and zero-padded (one bulk copy per CTA, counted on
  // the receiver's mbarrier).  Once all C messages are in, each CTA
  // completes the C first blocks and ranks its own entries by counting the
  // larger keys of every list (binary searches); rank < n_take wins.  Its
  // winners go to every CTA as a bit mask (st.async, a second mbarrier), and
  // every CTA assembles the same selection.
  const int jb0 = 16 * k0, jb1 = min(16 * k1, nbt);
  const int w0 = jb0 >> 5;   // first selection word of this CTA's blocks
  unsigned long long* skeys = reinterpret_cast<unsigned long long*>(send + 16);
  auto block_key = [](float r, int j) {
    return (static_cast<unsigned long long>(float_to_ordered(r)) << 32) | static_cast<uint32_t>(~j);
  };
  auto msg_keys = [&](int q) { return reinterpret_cast<const unsigned long long*>(recv + q * kDsMsgBytes + 16); };
  auto msg_summary = [&](int q) { return *reinterpret_cast<const DsSummary*>(recv + q * kDsMsgBytes); };
  {
    const int kb0 = kDsChunk * k0;
    const int nrange = max(0, jb1 - jb0);
#pragma unroll 1
    for (int x = tid; x < list_pow; x += kDsThreads) skeys[x] = 0ull;   // 0: below every key
    if (tid < kDsMaskWords) rmask[tid] = 0u;
    // (the trip count is the same in every lane: the warp votes below)
#pragma unroll 1
    for (int x0 = 0; x0 < nrange; x0 += kDsThreads) {
      const int j = jb0 + x0 + tid;
      float r = -INFINITY;
      if (j < jb1) {
        const int a0 = max(4 * j - 1, kb0), e0 = min(nc - 1, 4 * j + 3);
#pragma unroll 1
        for (int k = a0; k <= e0; ++k) r = fmaxf(r, gbuf[k - kb0]);
        if (j == jb0) rmine[0] = r;
      }
      const bool cand = j < jb1 && j > jb0 && j >= n_first && j < local_lo && r > -INFINITY;
      const uint32_t bal = __ballot_sync(0xffffffffu, cand);
      int base = 0;
      if (lane == 0 && bal) base = atomicAdd(&sctr[0], __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      if (cand) lkeys[base + __popc(bal & ((1u << lane) - 1u))] = block_key(r, j);
    }
  }
  __syncthreads();
  const int n_list = min(sctr[0], n_take);
  {
    const int n_loc = sctr[0];
    // Two threads per key, each comparing it with one half of the keys
    // (keys [0, h) and [h, n_loc), h even), eight keys per iteration from
    // four independent 16-byte loads: the loop is bound by load latency.
    const int part = tid & 1;
    const int h = (n_loc / 2 + 1) & ~1;
    const int y0 = part ? h : 0, y1 = part ? n_loc : min(h, n_loc);
#pragma unroll 1
    for (int x0 = 0; x0 < n_loc; x0 += kDsThreads / 2) {   // (same trip count in every lane)
      const int x = x0 + (tid >> 1);
      const unsigned long long me = x < n_loc ? lkeys[x] : 0ull;
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
      int y = y0;
#pragma unroll 1
      for (; y + 8 <= y1; y += 8) {
        const ulonglong2 a0 = *reinterpret_cast<const ulonglong2*>(lkeys + y);
        const ulonglong2 a1 = *reinterpret_cast<const ulonglong2*>(lkeys + y + 2);
        const ulonglong2 a2 = *reinterpret_cast<const ulonglong2*>(lkeys + y + 4);
        const ulonglong2 a3 = *reinterpret_cast<const ulonglong2*>(lkeys + y + 6);
        r0 += (a0.x > me ? 1 : 0) + (a0.y > me ? 1 : 0);
        r1 += (a1.x > me ? 1 : 0) + (a1.y > me ? 1 : 0);
        r2 += (a2.x > me ? 1 : 0) + (a2.y > me ? 1 : 0);
        r3 += (a3.x > me ? 1 : 0) + (a3.y > me ? 1 : 0);
      }
#pragma unroll 1
      for (; y < y1; ++y) r0 += lkeys[y] > me ? 1 : 0;
      int rk = (r0 + r1) + (r2 + r3);
      rk += __shfl_xor_sync(0xffffffffu, rk, 1);
      if (part == 0 && x < n_loc && rk < n_list) skeys[rk] = me;
    }
    if (tid == 0) {
      const float gl = (k1 > k0 && kDsChunk * k1 - 1 < nc) ? gbuf[kDsChunk * (k1 - k0) - 1] : -INFINITY;
      const float first = jb0 < jb1 ? rmine[0] : -INFINITY;
      *reinterpret_cast<float4*>(send) = make_float4(gl, first, __int_as_float(n_list), 0.f);
    }
  }
  fence_proxy_async_smem();   // the message is read by the bulk copies
  __syncthreads();
  if (tid < C)
    bulk_copy_to_cta(dsmem_addr(recv + rank * kDsMsgBytes, static_cast<uint32_t>(tid)), send, msg_bytes,
                     dsmem_addr(lbar, static_cast<uint32_t>(tid)));
  // The CTA's likeliest winners head for L2 while the selection is made
  // (after the copies, which they would otherwise queue ahead of).
  if (warp == 1 && lane < min(ds_prefetch_count(n_take, C), n_list))
    prefetch_block(&k_map, &v_map, kv_row0 + static_cast<int>(~static_cast<uint32_t>(skeys[lane])) * kBlock);
  // (waited for even after an earlier timeout: no copy may still be landing later)
  ok = __syncthreads_and(mbar_wait_cluster(lbar, 0, p.status)) && ok;
  // First block of CTA q (16 per q), completed with CTA q - 1's last kernel.
  if (tid < C) {
    const int q = tid, j = 16 * per * q;
    unsigned long long key = 0ull;   // 0: not a candidate (every candidate's key is larger)
    if (j < nbt) {
      float r = msg_summary(q).first;
      if (q > 0) r = fmaxf(r, msg_summary(q - 1).tail);
      if (j >= n_first && j < local_lo && r > -INFINITY) key = block_key(r, j);
    }
    bkeys[q] = key;
  }
#pragma unroll 1
  for (int j = tid; j < n_first; j += kDsThreads) atomicOr(&sbits[j >> 5], 1u << (j & 31));
#pragma unroll 1
  for (int j = local_lo + tid; j <= c; j += kDsThreads) atomicOr(&sbits[j >> 5], 1u << (j & 31));
  __syncthreads();
  // This CTA's entries (its list, then its first block) against every list:
  // half-warp entry x, lane q searches list q (sorted, zero-padded) and
  // compares first block q; the 16 lanes' counts add up to the entry's rank.
  if (n_take > 0) {
    const int q2 = lane & 15;
#pragma unroll 1
    for (int x0 = 0; x0 <= n_list; x0 += 2 * kDsWarps) {   // (same trip count in every lane)
      const int x = x0 + 2 * warp + (lane >> 4);
      unsigned long long k = 0ull;   // 0: no entry
      if (x <= n_list) k = x < n_list ? msg_keys(rank)[x] : bkeys[rank];
      int pos = 0;
      if (k != 0ull && q2 < C) {
        const unsigned long long* l2 = msg_keys(q2);
        // Branchless binary search: the entries above k form a prefix.
#pragma unroll 1
        for (int step = list_pow >> 1; step >= 1; step >>= 1)
          if (l2[pos + step - 1] > k) pos += step;
        pos += (l2[pos] > k ? 1 : 0) + (bkeys[q2] > k ? 1 : 0);
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) pos += __shfl_xor_sync(0xffffffffu, pos, o);
      if (q2 == 0 && k != 0ull && pos < n_take) {
        const int j = static_cast<int>(~static_cast<uint32_t>(k));
        atomicOr(&rmask[(j >> 5) - w0], 1u << (j & 31));
      }
    }
  }
  __syncthreads();
  if (tid < C) {   // this CTA's winners (words w0 ..) into CTA tid
    const uint32_t dst = dsmem_addr(minbox + rank * kDsMaskWords, static_cast<uint32_t>(tid));
    const uint32_t bar = dsmem_addr(sbar, static_cast<uint32_t>(tid));
#pragma unroll
    for (int x = 0; x < kDsMaskWords / 4; ++x)
      st_async_u32x4(dst + 16 * x, make_uint4(rmask[4 * x], rmask[4 * x + 1], rmask[4 * x + 2], rmask[4 * x + 3]), bar);
  }
  ok = __syncthreads_and(mbar_wait_cluster(sbar, 0, p.status)) && ok;
#pragma unroll 1
  for (int e = tid; e < C * kDsMaskWords; e += kDsThreads) {
    const int q = e / kDsMaskWords, w = ((16 * per * q) >> 5) + e % kDsMaskWords;
    const uint32_t v = minbox[e];
    if (v != 0u && w < kDsMaxBlocks / 32) atomicOr(&sbits[w], v);
  }
  __syncthreads();
  {
    // Ascending list: word w's set bits go to positions [prefix(w), ...).
    const int n_words = (nbt + 31) / 32;   // <= kDsMaxBlocks / 32 <= kDsThreads
    const uint32_t bw = tid < n_words ? sbits[tid] : 0u;
    const int cnt = __popc(bw);
    const int incl = warp_inclusive_scan(cnt);
    if (lane == 31) sctr[4 + warp] = incl;
    __syncthreads();
    int pos = incl - cnt;
#pragma unroll
    for (int w = 0; w < kDsWarps; ++w) pos += (w < warp) ? sctr[4 + w] : 0;
    if (tid == kDsThreads - 1) nselS[0] = min(pos + cnt, p.kmax);
    uint32_t rest = bw;
    while (rest) {
      const int j = tid * 32 + __ffs(rest) - 1;
      rest &= rest - 1u;
      if (pos < p.kmax) selS[pos] = j;
      ++pos;
    }
  }
  __syncthreads();
  const int nsel = nselS[0];
  if (rank == 0) {
#pragma unroll 1
    for (int e = tid; e < p.kmax; e += kDsThreads)
      p.block_idx[static_cast<size_t>(bh) * p.kmax + e] = e < nsel ? selS[e] : -1;
    if (tid == 0) p.n_sel[bh] = nsel;
  }
  if (tid == 32)   // blocks of the second and later rounds: into L2 now
#pragma unroll 1
    for (int n = rank + C * kDsPairs; n < nsel; n += C) prefetch_block(&k_map, &v_map, kv_row0 + selS[n] * kBlock);

  // ------------------------------------------------------------ attend --
  const int pair = warp >> 1, half = warp & 1;
  float l0 = 0.f, l1 = 0.f;
  {
    uint8_t* stage = smem + pair * kDsStageBytes;
    const uint32_t k_b = smem_u32(stage), v_b = k_b + 16384;
    const int rbase = 32 * half;
    // Item x of this CTA is list entry rank + C x; pair `pair` takes items
    // pair, pair + 6, ...
    auto block_of = [&](int item) {
      const int n = rank + C * item;
      const int j = n < nsel ? selS[n] : -1;
      return j > c ? -1 : j;
    };
    int item = pair;
    int j = block_of(item);
    if (half == 0 && lane == 0 && j >= 0 && ok &&
        kv_row_ok(static_cast<size_t>(kv_row0) + static_cast<size_t>(j) * kBlock, kv_row0, p.Lmax, p.status))
      tma_block(stage, &k_map, &v_map, kv_row0 + j * kBlock, &kvfull[pair]);

    float o[16][4];
#pragma unroll
    for (int x = 0; x < 16; ++x) o[x][0] = o[x][1] = o[x][2] = o[x][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;
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
#pragma unroll 1
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
      // Both warps are done with the stage; order the zeroed V rows
      // (generic writes) before the TMA refill (async proxy).
      fence_proxy_async_smem();
      pair_sync(pair);
      item += kDsPairs;
      j = block_of(item);
      if (j >= 0 && half == 0 && lane == 0 && ok &&
          kv_row_ok(static_cast<size_t>(kv_row0) + static_cast<size_t>(j) * kBlock, kv_row0, p.Lmax, p.status))
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
  if (tid < kGroup * 16) {   // head tid / 16, warp tid % 16 (< 12): shuffle trees over the warps
    const int w = tid % 16, hd = tid / 16;
    const float2 v = w < kDsWarps ? warp_ml[w * kGroup + hd] : make_float2(-INFINITY, 0.f);
    float M = v.x;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wt = (M == -INFINITY) ? 0.f : fast_exp2(v.x - M);
    if (w < kDsWarps) wgt[w * kGroup + hd] = wt;
    float lsum = wt * v.y;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    // This CTA's (max, sum) of head hd into the CTA that writes the head.
    if (w == 0) st_dsmem_f32x2(dsmem_addr(&ml_in[rank * hmax + hd / C], hd % C), make_float2(M, lsum));
  }
  __syncthreads();
  // This CTA's partial O of each head into the CTA that writes the head:
  // 4 dims per item, merged over the warps on the way.
#pragma unroll 1
  for (int e = tid; e < kGroup * (kHeadDim / 4); e += kDsThreads) {
    const int hd = e / (kHeadDim / 4), d4 = 4 * (e % (kHeadDim / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kDsWarps; ++w) {
      const float wt = wgt[w * kGroup + hd];
      const float4 v = *reinterpret_cast<const float4*>(smem + (w >> 1) * kDsStageBytes + (w & 1) * 8192 +
                                                          (hd * kHeadDim + d4) * 4);
      acc.x += wt * v.x;
      acc.y += wt * v.y;
      acc.z += wt * v.z;
      acc.w += wt * v.w;
    }
    st_dsmem_f32x4(dsmem_addr(o_in + (rank * hmax + hd / C) * kHeadDim + d4, hd % C), acc);
  }
  cluster_arrive();
  cluster_wait();

  // Heads rank, rank + C, ... of the output from the C partials: first the
  // weight of each (head, source) and each head's sum (16 lanes per head),
  // then the dims.
  float* mw = wgt;   // [hmax][16] source weights / sum, reusing the warp-merge weights
  if (warp < (hmax * 16 + 31) / 32) {   // whole warps: lanes past hmax * 16 carry neutral values
    const int q = tid % 16, hl = tid / 16;
    const float2 ml = (q < C && hl < hmax) ? ml_in[q * hmax + hl] : make_float2(-INFINITY, 0.f);
    float M = ml.x;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wt = (M == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
    float lsum = wt * ml.y;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const int hd = rank + C * hl;
    if (hl < hmax) mw[hl * 16 + q] = lsum > 0.f ? wt / lsum : 0.f;
    if (q == 0 && hl < hmax && hd < kGroup && p.lse)
      p.lse[orow + hd] = lsum > 0.f ? (M + fast_log2(lsum)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
#pragma unroll 1
  for (int e = tid; e < hmax * kHeadDim; e += kDsThreads) {
    const int hl = e / kHeadDim, d = e % kHeadDim;
    const int hd = rank + C * hl;
    if (hd >= kGroup) continue;
    float acc = 0.f;
#pragma unroll 4
    for (int q = 0; q < C; ++q) acc += mw[hl * 16 + q] * o_in[(q * hmax + hl) * kHeadDim + d];
    p.out[(orow + hd) * kHeadDim + d] = __float2bfloat16(acc);
  }
}

bool ds_fits(const Shape& s, int C) {
  const int groups = (s.nbmax + 15) / 16;
  return s.nq == 1 && C >= 1 && C <= kDsMaxC && ds_per(groups, C) <= kDsMaxIt && s.nbmax <= kDsMaxBlocks &&
         s.kmax <= 256;
}

void ds_config(const Shape& s, int C, cudaLaunchConfig_t* cfg, cudaLaunchAttribute (&attrs)[2], cudaStream_t st) {
  *cfg = cudaLaunchConfig_t{};
  cfg->gridDim = dim3(C, s.B * s.Hkv, 1);
  cfg->blockDim = dim3(kDsThreads, 1, 1);
  cfg->dynamicSmemBytes = kDsSmem;
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

// Clusters of C CTAs that can be resident at once on the current device
// (0 if the configuration cannot launch), cached per device.
int ds_active_clusters(int C) {
  static int cache[64][kDsMaxC + 1];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    bool ok = true;
    for (auto* fn : {decode_step_kernel<false>, decode_step_kernel<true>})
      ok = ok && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDsSmem) == cudaSuccess &&
           cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    for (int c = 1; c <= kDsMaxC; ++c) {
      int n = 0;
      if (ok) {
        Shape s{};
        s.B = 1;
        s.Hkv = 1;
        cudaLaunchConfig_t cfg;
        cudaLaunchAttribute attrs[2];
        ds_config(s, c, &cfg, attrs, nullptr);
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, decode_step_kernel<false>, &cfg) != cudaSuccess) n = 0;
      }
      cache[dev][c] = n;
    }
    cudaGetLastError();
    done[dev] = true;
  }
  return cache[dev][C];
}

}  // namespace

// The cluster size for this shape: every group's cluster resident at once
// (a second wave would double the step), then the fewest load rounds and
// the most CTAs per group (more SMs streaming the kernel means).  0 when no
// size fits.
int decode_step_cluster_size(const Shape& s) {
  const int G = s.B * s.Hkv;
  int best = 0;
  double best_cost = 0.0;
  for (int C = kDsMaxC; C >= 1; --C) {
    if (!ds_fits(s, C)) continue;
    const int active = ds_active_clusters(C);
    if (active < 1) continue;
    const int waves = (G + active - 1) / active;
    const int rounds = (s.kmax + C * kDsPairs - 1) / (C * kDsPairs);
    // Per CTA: its share of the kernel means (4 B per element) and of the
    // selected blocks (32 KB each), streamed at ~50 GB/s per SM, plus ~2 us
    // per attention round and ~8 us of fixed latency.
    const double bytes = (static_cast<double>(s.ncmax) * kHeadDim * 4 + static_cast<double>(s.kmax) * 32768) / C;
    const double cost = waves * (8.0 + 2.0 * rounds + bytes / 50e3);
    if (!best || cost < best_cost - 1e-9) {
      best = C;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t launch_decode_step(const Shape& s, int cluster, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                               const CUtensorMap& k_map, const CUtensorMap& v_map, const void* k,
                               const int32_t* kv_lens, void* kc, int32_t* block_idx, int32_t* n_sel, void* out,
                               float* lse, const DsAppend* append, uint32_t* status, uint32_t test_flags,
                               cudaStream_t st) {
  if (cluster < 1 || cluster > kDsMaxC || !ds_fits(s, cluster) || ds_active_clusters(cluster) < 1)
    return cudaErrorInvalidConfiguration;
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
  p.test_flags = test_flags;
  if (append) {
    p.q_src = static_cast<const uint4*>(append->q);
    p.k_new = static_cast<const uint4*>(append->k_new);
    p.v_new = static_cast<const uint4*>(append->v_new);
    p.k_w = static_cast<uint4*>(append->k_cache);
    p.v_w = static_cast<uint4*>(append->v_cache);
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attrs[2];
  ds_config(s, cluster, &cfg, attrs, st);
  return append ? cudaLaunchKernelEx(&cfg, decode_step_kernel<true>, kc_map, q_map, k_map, v_map, p)
                : cudaLaunchKernelEx(&cfg, decode_step_kernel<false>, kc_map, q_map, k_map, v_map, p);
}

}  // namespace infllmv2
