// Stage 3 of InfLLM v2 for prefill on the 5th-generation tensor cores.
//
// [InfLLM v2 > Query group sharing]: the 16 heads of a GQA group share one
// block set, so for a KV block they form 16 rows of one MMA tile; eight
// consecutive query tokens x 16 heads fill the 128-row tcgen05 tile, and
// the CTA walks the union of the eight tokens' selected blocks
// ([InfLLM v2 > Block-level key-value partitioning, eq. B_j]).  Rows whose
// token did not select a block get probability 0 for it, so every row's
// result is exactly its own block-sparse attention.
//
// The union is walked two blocks (128 keys) per item: S = Q K^T is one
// N = 128 product per item and O += P V one K = 128 product, which halves
// the serial work of the issuing thread per key.
//
// Roles (352 threads):
//   warps 0-7  softmax: row r = 32 (w % 4) + lane (token r / 16, head r % 16)
//              is shared by warps w % 4 and w % 4 + 4, which take the
//              item's first and second block (S columns 0-63 / 64-127) and
//              O columns 0-63 / 64-127; they agree on the row's running max
//              through shared memory.  Online softmax in fp32 base 2 with a
//              lazy rescale (the running max only moves when it grows by
//              more than 2^8, which keeps exp2(s - m) <= 256); P (bf16
//              pairs) goes to TMEM; O rows are rescaled in TMEM when needed.
//              Probabilities are computed while the previous P V product
//              runs; a warp whose two tokens both skipped its block only
//              writes zeros.
//   warp 8     MMA issuer (one thread): S_i = Q K_i^T (M 128, N 128, K 128,
//              both operands in shared memory) into one of two TMEM S
//              buffers, and O += P_i V_i (M 128, N 128, K 128; P from TMEM,
//              V an MN-major shared operand), each stream issued as soon as
//              its operands are ready.
//   warp 9     TMA producer: the Q tile, then each item's two K tiles into a
//              3-stage ring (a stage frees once S is computed).
//   warp 10    TMA producer: each item's two V tiles into a 2-stage ring (a
//              stage frees once its P V product is done).
// TMEM: columns [0,256) two S buffers, [256,384) the O accumulator,
// [384,512) two P buffers.
//
// Few tiles (speculative verification: n_q <= 16 drafts per sequence, or a
// short chunk) would leave most SMs idle, so each tile's union is then split
// over a cluster of C CTAs: CTA r walks items [r n / C, (r + 1) n / C) and
// ends with a partial row state (running max m, sum l, unnormalised O in
// TMEM).  After a cluster barrier (every CTA past its last item, its K ring
// free) each CTA pushes row r's partial into CTA r mod C's K ring through
// distributed shared memory; after a second barrier the owner merges
// (M = max m, weights 2^(m - M)) and writes the row.  A block several drafts
// select is thus read once per tile instead of once per draft.
//
// P enters P V as bf16.  One bf16 carries 8 significant bits, and where a
// row averages only a few values the rounding of its probabilities reaches
// the output at 2^-9 |V|.  A tile in which some token attends fewer than
// kSplitKeys keys therefore feeds P as hi = bf16(p) plus lo = bf16(p - hi)
// (16 significant bits): the softmax warps write lo into the S columns they
// have just read, the issuer adds a second product per item, and S of item
// i + 2 waits until P V of item i (which reads that S buffer) is done.
// Longer rows average the rounding away (error below 3e-4 at 1024 keys).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace infllmv2 {

namespace {

constexpr int kTcTokens = 8;
constexpr int kTcKStages = 3;   // K tiles of an item (32 KB): freed as soon as S = Q K^T is done
constexpr int kTcVStages = 2;   // V tiles of an item (32 KB): freed when O += P V is done
constexpr int kTcItemBytes = 32768;
constexpr int kTcSoftmaxWarps = 8;   // two per TMEM lane quadrant, 32 of the 64 S columns each
constexpr int kTcThreads = (kTcSoftmaxWarps + 3) * 32;
constexpr int kTcMmaWarp = kTcSoftmaxWarps, kTcTmaWarp = kTcSoftmaxWarps + 1, kTcVWarp = kTcSoftmaxWarps + 2;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: two S buffers (128 keys each), the O accumulator and two P
// buffers (bf16 pairs, one row per lane: the A operand of O += P V).
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
constexpr float kLazyRescale = 8.0f;
constexpr int kSplitKeys = 2048;   // tiles with a row attending fewer keys feed P as hi + lo
constexpr int kTcMaxSmem = 227 * 1024;
// Cluster merge: C partial rows of ceil(128 / C) rows (O and (m, l)) land in
// the K ring.
__host__ __device__ constexpr int tc_merge_bytes(int C) { return C * ((128 + C - 1) / C) * (512 + 8); }
__host__ __device__ constexpr bool tc_merge_fits(int C) {
  return C > 16 || (tc_merge_bytes(C) <= kTcKStages * kTcItemBytes && tc_merge_fits(C + 1));
}
static_assert(tc_merge_fits(2), "cluster partials fit in the K ring");

struct TcParams {
  int B, Hkv, Lmax, nq, kmax, nbmax;
  int csize;   // CTAs per tile: 1, or a cluster that splits the union's items
  float scale2;
  const int32_t* kv_lens;
  const int32_t* block_idx;
  const int32_t* n_sel;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
};

struct TcLayout {
  int q, kv, vv, bars, slot, bits, ulist, umask, scan, kcnt, xch, total;
};

__host__ __device__ inline TcLayout tc_layout(int nbmax) {
  TcLayout l;
  l.q = 0;                                   // 2 boxes x 128 rows x 128 B
  l.kv = 32768;                              // K ring
  l.vv = l.kv + kTcKStages * kTcItemBytes;   // V ring
  l.bars = l.vv + kTcVStages * kTcItemBytes; // 32 mbarriers max
  l.slot = l.bars + 32 * 8;
  l.bits = l.slot + 16;
  l.ulist = l.bits + ((nbmax + 15) & ~15);
  l.umask = l.ulist + nbmax * 4;
  l.scan = l.umask + ((nbmax + 15) & ~15);
  l.kcnt = l.scan + 64;                      // keys attended per token of the tile
  l.xch = l.kcnt + 64;                       // [2 column halves][128 rows] fp32 exchange
  l.total = l.xch + 2 * 128 * 4;
  return l;
}

// kODone + (m & 1) completes when O += P_m V_m has finished, so the softmax
// warps can wait for the P-V product two blocks back (whose P buffer they
// reuse) without waiting for the one in flight.
// Barrier of the two softmax warps of TMEM lane quadrant q (ids 1..4).
__device__ __forceinline__ void pair_sync(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(q + 1) : "memory");
}

// bf16 pair of the rounding residues p - bf16(p) of two probabilities whose
// rounded pair is `hi` (pack_bf16x2 order: p0 in the low half).
__device__ __forceinline__ uint32_t lo_bf16x2(float p0, float p1, uint32_t hi) {
  const float h0 = __uint_as_float(hi << 16), h1 = __uint_as_float(hi & 0xFFFF0000u);
  return pack_bf16x2(p0 - h0, p1 - h1);
}

// One warp's 64 probabilities of its row for an item (bf16 pairs into w),
// returning their sum.  whole: the row sees all 64 keys or none (sel false),
// so no per-key mask; otherwise keys [0, nv) count.  Every exponential
// goes to the MUFU unit: in a sparse union about half the warps skip each
// block, which leaves the unit room, and a polynomial on the FMA pipe costs
// a dozen instructions per value (with half of the values on it the 32K
// prefill launch took 6.66 ms, against 5.46 ms).
// kSplit: the lo parts p - bf16(p) go to TMEM at lo_addr, 16 pairs at a time.
template <bool kSplit>
__device__ __forceinline__ float row_probs(const uint32_t (&s)[64], uint32_t (&w)[32], bool whole, bool sel,
                                           float m_use, int nv, float scale2, uint32_t lo_addr) {
  float lsum = 0.f;
  if (whole) {
    // A row that skipped the block subtracts +inf: every exp2 is 0.
    const float m_eff = sel ? m_use : INFINITY;
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int x0 = 0; x0 < 32; x0 += 16) {
      uint32_t wl[16];
#pragma unroll
      for (int x = x0; x < x0 + 16; ++x) {
        const float a0 = fmaf(__uint_as_float(s[2 * x]), scale2, -m_eff);
        const float a1 = fmaf(__uint_as_float(s[2 * x + 1]), scale2, -m_eff);
        const float p0 = fast_exp2(a0);
        const float p1 = fast_exp2(a1);
        ls0 += p0;
        ls1 += p1;
        w[x] = pack_bf16x2(p0, p1);
        if (kSplit) wl[x - x0] = lo_bf16x2(p0, p1, w[x]);
      }
      if (kSplit) tc::st16(lo_addr + x0, wl);
    }
    lsum = ls0 + ls1;
  } else {
#pragma unroll
    for (int x0 = 0; x0 < 32; x0 += 16) {
      uint32_t wl[16];
#pragma unroll
      for (int x = x0; x < x0 + 16; ++x) {
        const float a0 = __uint_as_float(s[2 * x]) * scale2 - m_use;
        const float a1 = __uint_as_float(s[2 * x + 1]) * scale2 - m_use;
        const float p0 = (2 * x < nv) ? fast_exp2(a0) : 0.f;
        const float p1 = (2 * x + 1 < nv) ? fast_exp2(a1) : 0.f;
        lsum += p0 + p1;
        w[x] = pack_bf16x2(p0, p1);
        if (kSplit) wl[x - x0] = lo_bf16x2(p0, p1, w[x]);
      }
      if (kSplit) tc::st16(lo_addr + x0, wl);
    }
  }
  return lsum;
}

enum Bar { kQFull = 0, kKFull = 1, kKEmpty = kKFull + kTcKStages, kVFull = kKEmpty + kTcKStages,
           kVEmpty = kVFull + kTcVStages, kSFull = kVEmpty + kTcVStages, kSFree = kSFull + 2,
           kPFull = kSFree + 2, kODone = kPFull + 2, kNumBars = kODone + 2 };
static_assert(kNumBars <= 32, "barrier area holds 32");

// kCluster: the tile's union is split over a cluster of p.csize CTAs (a
// separate instantiation, so the one-CTA form carries none of its code).
template <bool kCluster>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const TcLayout lay = tc_layout(p.nbmax);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.slot);
  uint8_t* bits = smem + lay.bits;
  int32_t* ulist = reinterpret_cast<int32_t*>(smem + lay.ulist);
  uint8_t* umask = smem + lay.umask;
  int* scan = reinterpret_cast<int*>(smem + lay.scan);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.Hkv + h;
  const int Hq = p.Hkv * kGroup;
  const int csize = kCluster ? p.csize : 1;
  const int rank = kCluster ? static_cast<int>(blockIdx.x) % csize : 0;   // == the rank in the cluster
  const int t0 = kCluster ? (static_cast<int>(blockIdx.x) / csize) * kTcTokens : blockIdx.x * kTcTokens;
  const int n_act = min(kTcTokens, p.nq - t0);
  pdl_wait();   // the previous kernel of the stream may still be writing the inputs
  pdl_trigger();
  const int L = p.kv_lens[b];

  if (L < p.nq || L > p.Lmax) {   // the same in every CTA of a cluster: none touches another's memory
    if (kCluster && rank != 0) return;
    for (int e = tid; e < n_act * kGroup * kHeadDim; e += kTcThreads) {
      const int tok = e / (kGroup * kHeadDim), rem = e % (kGroup * kHeadDim);
      p.out[((static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup) * kHeadDim + rem] = __float2bfloat16(0.f);
    }
    if (p.lse)
      for (int e = tid; e < n_act * kGroup; e += kTcThreads)
        p.lse[(static_cast<size_t>(b) * p.nq + t0 + e / kGroup) * Hq + h * kGroup + e % kGroup] = -INFINITY;
    if (tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(p.status, kStatusBadKvLen);
    return;
  }
  const int i_last = L - p.nq + t0 + n_act - 1;
  const int nb = i_last / kBlock + 1;

  // ---- union of the tile's block sets: bit `tok` of bits[j] ----
  uint32_t* bits32 = reinterpret_cast<uint32_t*>(bits);
  int* kcnt = reinterpret_cast<int*>(smem + lay.kcnt);
  for (int w = tid; w < (nb + 3) / 4; w += kTcThreads) bits32[w] = 0u;
  __syncthreads();
  // Warp `tok` (< 8) marks its token's blocks and counts the keys it attends.
  if (warp < kTcTokens) {
    const int tok = warp;
    int keys = 0;
    if (tok < n_act) {
      const size_t u = static_cast<size_t>(bh) * p.nq + t0 + tok;
      const int ns = min(p.n_sel[u], p.kmax);
      const int i_tok = L - p.nq + t0 + tok;
      check_selection_row(p.block_idx + u * p.kmax, p.n_sel[u], p.kmax, i_tok / kBlock, p.status, lane);
      for (int k = lane; k < ns; k += 32) {
        const int j = p.block_idx[u * p.kmax + k];
        if (j >= 0 && j <= i_tok / kBlock) {
          atomicOr(&bits32[j >> 2], (1u << tok) << ((j & 3) * 8));
          keys += min(kBlock, i_tok - j * kBlock + 1);
        }
      }
    }
    keys = warp_sum_int(keys);
    if (lane == 0) kcnt[tok] = keys;
  }
  __syncthreads();
  // Hi + lo probabilities when some token of the tile attends few keys, and
  // always in a cluster (each CTA then sums only a share of a row's keys).
  bool split = false;
  if (kCluster) split = true;
#pragma unroll
  for (int tok = 0; tok < kTcTokens; ++tok) split |= (tok < n_act) && (kcnt[tok] < kSplitKeys);
  {
    const int per = (nb + kTcThreads - 1) / kTcThreads;
    const int lo = tid * per, hi = min(nb, lo + per);
    int cnt = 0;
    for (int j = lo; j < hi; ++j) cnt += bits[j] ? 1 : 0;
    const int incl = warp_inclusive_scan(cnt);
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kTcThreads / 32; ++w) {
      base += (w < warp) ? scan[w] : 0;
      tot += scan[w];
    }
    int pos = base + incl - cnt;
    for (int j = lo; j < hi; ++j) {
      if (bits[j]) {
        ulist[pos] = j;
        umask[pos] = bits[j];
        ++pos;
      }
    }
    __syncthreads();
    if (tid == 0) scan[15] = tot;
  }

  if (tid == 0) {
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    mbar_init(&bars[kQFull], 1);
    for (int s = 0; s < kTcKStages; ++s) {
      mbar_init(&bars[kKFull + s], 1);
      mbar_init(&bars[kKEmpty + s], 1);
    }
    for (int s = 0; s < kTcVStages; ++s) {
      mbar_init(&bars[kVFull + s], 1);
      mbar_init(&bars[kVEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kSFull + s], 1);
      mbar_init(&bars[kSFree + s], kTcSoftmaxWarps);
      mbar_init(&bars[kPFull + s], kTcSoftmaxWarps);
    }
    mbar_init(&bars[kODone], 1);
    mbar_init(&bars[kODone + 1], 1);
    fence_barrier_init();
  }
  if (warp == kTcMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Items of two union blocks (the last may hold one); in a cluster CTA
  // `rank` takes items [it0, it1) of the tile's nit_all.
  const int nu_all = scan[15];
  const int nit_all = (nu_all + 1) / 2;
  const int it0 = kCluster ? rank * nit_all / csize : 0;
  const int it1 = kCluster ? (rank + 1) * nit_all / csize : nit_all;
  const int ubase = kCluster ? 2 * it0 : 0;
  const int nu = kCluster ? max(0, min(nu_all, 2 * it1) - ubase) : nu_all;   // slots ubase .. ubase + nu - 1
  const int nit = kCluster ? it1 - it0 : nit_all;
  const uint32_t q_s = smem_u32(smem + lay.q);
  const uint32_t kv_s = smem_u32(smem + lay.kv);
  const uint32_t vv_s = smem_u32(smem + lay.vv);
  // Block of slot `half` of item `it` (a missing second block repeats the
  // first one's tiles and is masked out).
  auto item_block = [&](int it, int half) { return ulist[ubase + min(2 * it + half, nu - 1)]; };
  float m_fin = -INFINITY, l_fin = 0.f;   // a softmax thread's row state after the last item

  if (warp == kTcTmaWarp) {
    // ------------------------------------------------------- TMA producer
    // Q and the K ring here; the V ring has a warp of its own, so neither
    // producer's waits hold up the other.  An item's stage holds, per
    // 64-column box, 128 rows: the first block's keys then the second's.
    if (lane == 0 && nu > 0) {
      mbar_arrive_expect_tx(&bars[kQFull], n_act * 4096);
      for (int tok = 0; tok < n_act; ++tok) {
        const int row = (b * p.nq + t0 + tok) * Hq + h * kGroup;
        tma_load_2d(smem + lay.q + tok * 2048, &q_map, 0, row, &bars[kQFull]);
        tma_load_2d(smem + lay.q + 16384 + tok * 2048, &q_map, 64, row, &bars[kQFull]);
      }
      for (int it = 0; it < nit; ++it) {
        const int st = it % kTcKStages;
        if (it >= kTcKStages && !mbar_wait(&bars[kKEmpty + st], ((it / kTcKStages) - 1) & 1, p.status)) break;
        uint8_t* dst = smem + lay.kv + st * kTcItemBytes;
        mbar_arrive_expect_tx(&bars[kKFull + st], kTcItemBytes);
        for (int hf = 0; hf < 2; ++hf) {
          const int row = bh * p.Lmax + item_block(it, hf) * kBlock;
          if (!kv_row_ok(row, static_cast<size_t>(bh) * p.Lmax, p.Lmax, p.status)) continue;
          tma_load_2d(dst + hf * 8192, &k_map, 0, row, &bars[kKFull + st]);
          tma_load_2d(dst + 16384 + hf * 8192, &k_map, 64, row, &bars[kKFull + st]);
        }
      }
    }
    __syncwarp();
  } else if (warp == kTcVWarp) {
    // ------------------------------------------------------- V producer
    if (lane == 0 && nu > 0) {
      for (int it = 0; it < nit; ++it) {
        const int st = it % kTcVStages;
        if (it >= kTcVStages && !mbar_wait(&bars[kVEmpty + st], ((it / kTcVStages) - 1) & 1, p.status)) break;
        uint8_t* dst = smem + lay.vv + st * kTcItemBytes;
        mbar_arrive_expect_tx(&bars[kVFull + st], kTcItemBytes);
        for (int hf = 0; hf < 2; ++hf) {
          const int row = bh * p.Lmax + item_block(it, hf) * kBlock;
          if (!kv_row_ok(row, static_cast<size_t>(bh) * p.Lmax, p.Lmax, p.status)) continue;
          tma_load_2d(dst + hf * 8192, &v_map, 0, row, &bars[kVFull + st]);
          tma_load_2d(dst + 16384 + hf * 8192, &v_map, 64, row, &bars[kVFull + st]);
        }
      }
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nu > 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(128, 128, 0, 0);
      constexpr uint32_t kIdO = tc::idesc_bf16(128, 128, 0, 1);
      // Base descriptors; a tile offset is added to the 16-byte address field.
      const uint64_t q_desc0 = tc::sdesc_sw128(q_s, 16, 1024);
      const uint64_t k_desc0 = tc::sdesc_sw128(kv_s, 16, 1024);
      const uint64_t v_desc0 = tc::sdesc_sw128(vv_s, 16384, 1024);
      bool ok = mbar_wait(&bars[kQFull], 0, p.status);
      // Two in-order streams, each issued as soon as its inputs are there:
      // S of item n_s (its K tiles loaded, its S buffer read out two items
      // back) and O += P V of item n_o (its P written, its V tiles loaded).
      // Neither waits behind the other, so a late K tile does not hold back
      // the P V product that frees a V stage.
      int n_s = 0, n_o = 0;
      uint32_t idle = 0;
      while (ok && n_o < nit) {
        bool progressed = false;
        // With split probabilities S buffer n_s & 1 also holds the lo part of
        // item n_s - 2, read by that item's P V product.
        if (n_s < nit && mbar_try_wait(&bars[kKFull + n_s % kTcKStages], (n_s / kTcKStages) & 1) &&
            (n_s < 2 || (mbar_try_wait(&bars[kSFree + (n_s & 1)], ((n_s >> 1) - 1) & 1) &&
                         (!split || mbar_try_wait(&bars[kODone + (n_s & 1)], ((n_s - 2) >> 1) & 1))))) {
          const int st = n_s % kTcKStages, sb = n_s & 1;
          tc::fence_after_sync();
          const uint64_t kd = k_desc0 + static_cast<uint64_t>(st * (kTcItemBytes >> 4));
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t off = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
            tc::mma_ss(tmem + kColS + sb * 128, q_desc0 + off, kd + off, kIdS, k > 0 ? 1u : 0u);
          }
          tc::commit(&bars[kSFull + sb]);
          tc::commit(&bars[kKEmpty + st]);
          ++n_s;
          progressed = true;
        }
        if (n_o < n_s && mbar_try_wait(&bars[kPFull + (n_o & 1)], (n_o >> 1) & 1) &&
            mbar_try_wait(&bars[kVFull + n_o % kTcVStages], (n_o / kTcVStages) & 1)) {
          const int m = n_o, pb = m & 1, st = m % kTcVStages;
          tc::fence_after_sync();
          const uint64_t vd = v_desc0 + static_cast<uint64_t>(st * (kTcItemBytes >> 4));
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc::mma_ts(tmem + kColO, tmem + kColP + pb * 64 + 8 * k, vd + static_cast<uint64_t>((k * 2048) >> 4),
                       kIdO, (m > 0 || k > 0) ? 1u : 0u);
          if (split) {
            // lo parts: keys 64 x + [0, 64) of the item sit in S columns
            // 128 (m & 1) + 64 x + [0, 32).
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_ts(tmem + kColO, tmem + kColS + pb * 128 + 64 * (k >> 2) + 8 * (k & 3),
                         vd + static_cast<uint64_t>((k * 2048) >> 4), kIdO, 1u);
          }
          tc::commit(&bars[kODone + (m & 1)]);
          tc::commit(&bars[kVEmpty + st]);
          ++n_o;
          progressed = true;
        }
        if (progressed) {
          idle = 0;
        } else if (++idle > 4 * kSpinLimit) {
          atomicOr(p.status, kStatusTimeout);
          ok = false;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w: TMEM lane quadrant w % 4 (rows 32 (w % 4) + lane); slot
    // `half` = w / 4 of each item (S columns [64 half, 64 half + 64)) and O
    // columns [64 half, 64 half + 64).  The two warps of a quadrant agree
    // on each row's running max through shared memory; each keeps its own
    // partial row sum.
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;   // TMEM lane == MMA row
    const int tok = r >> 4;
    const bool active = tok < n_act;
    const int i_row = L - p.nq + t0 + tok;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + lay.xch);   // [half][row]
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int it = 0; it < nit; ++it) {
      const int sb = it & 1;
      const int u = 2 * it + half;            // this warp's union slot
      const bool present = u < nu;
      const bool sel = present && active && ((umask[ubase + u] >> tok) & 1);
      const bool warp_sel = __any_sync(0xffffffffu, sel);
      // No early exit from this loop: both warps of a quadrant must meet the
      // same pair barriers, so after a failed (timed-out) wait the warp keeps
      // going without waiting and the status word carries the error.
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kSFull + sb], (it >> 1) & 1, p.status));
      tc::fence_after_sync();
      uint32_t s[64];
      if (warp_sel) {   // a warp none of whose tokens picked its block skips its scores
        tc::ld32(lane_addr + kColS + sb * 128 + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
        tc::ld32(lane_addr + kColS + sb * 128 + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
        tc::wait_ld();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kSFree + sb]);

      // The stage slot holds this block's tiles (a repeat of the item's
      // first block when the item has only one).
      const int key0 = item_block(it, half) * kBlock;
      if (key0 + kBlock > L) {
        // The block holds cache rows past kv_len: clear their V rows so a
        // zero probability never multiplies a non-finite value.
        const int st = it % kTcVStages;
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kVFull + st], (it / kTcVStages) & 1, p.status));
        uint8_t* vt = smem + lay.vv + st * kTcItemBytes + half * 8192;
        const int r0 = L - key0;
        for (int e = lane; e < (kBlock - r0) * 16; e += 32) {
          const int row = r0 + (e >> 4), q16 = e & 15;
          *reinterpret_cast<uint4*>(vt + (q16 >> 3) * 16384 + row * 128 + (q16 & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      const int nv = sel ? min(kBlock, i_row - key0 + 1) : 0;   // keys key0 .. key0 + nv - 1
      // Rows see the whole block or none of it except on a token's own
      // diagonal block; the common case needs no per-key mask.
      const bool whole = __all_sync(0xffffffffu, nv == 0 || nv == kBlock);
      float mx = -INFINITY;
      if (warp_sel) {
        if (whole) {
          float m0 = __uint_as_float(s[0]), m1 = __uint_as_float(s[1]);
#pragma unroll
          for (int x = 2; x < 64; x += 2) {
            m0 = fmaxf(m0, __uint_as_float(s[x]));
            m1 = fmaxf(m1, __uint_as_float(s[x + 1]));
          }
          if (sel) mx = fmaxf(m0, m1) * p.scale2;
        } else {
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (x < nv) mx = fmaxf(mx, __uint_as_float(s[x]) * p.scale2);
        }
      }
      xch[half * 128 + r] = mx;
      pair_sync(quad);
      mx = fmaxf(mx, xch[(half ^ 1) * 128 + r]);
      // Either warp may have selected; both follow the row's combined max.
      const bool row_sel = mx > -INFINITY;
      bool need = false;
      float alpha = 1.f;
      float m_use = m_run;
      if (row_sel) {
        if (m_run == -INFINITY) {
          m_use = mx;
        } else if (mx > m_run + kLazyRescale) {
          need = true;
          alpha = fast_exp2(m_run - mx);
          m_use = mx;
        }
      }
      uint32_t w[32];   // this warp's 64 probabilities of the row, bf16 pairs
      float lsum = 0.f;
      // In split tiles the lo parts go, 16 pairs at a time, over the S
      // columns this warp read for the item (its S buffer is not refilled
      // before this item's P V product is done).
      const uint32_t lo_addr = lane_addr + kColS + sb * 128 + half * 64;
      if (warp_sel) {
        // Probabilities before waiting on the tensor core: only the P store
        // and an O rescale depend on earlier products.
        lsum = split ? row_probs<true>(s, w, whole, sel, m_use, nv, p.scale2, lo_addr)
                     : row_probs<false>(s, w, whole, sel, m_use, nv, p.scale2, lo_addr);
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) w[x] = 0u;
        if (split) {
          uint32_t z16[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) z16[x] = 0u;
          tc::st16(lo_addr, z16);
          tc::st16(lo_addr + 16, z16);
        }
      }
      // P buffer it & 1 was last read by the product of item it - 2.
      if (it >= 2 && ok)
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[kODone + (it & 1)], ((it - 2) >> 1) & 1, p.status));
      if (__any_sync(0xffffffffu, need)) {
        // A rescale touches O: the product of item it - 1 must be done too.
        if (it >= 1 && ok)
          ok = __all_sync(0xffffffffu, mbar_wait(&bars[kODone + ((it - 1) & 1)], ((it - 1) >> 1) & 1, p.status));
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tc::ld32(lane_addr + kColO + half * 64 + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tc::st32(lane_addr + kColO + half * 64 + c * 32, o);
        }
        tc::wait_st();
      }
      l_run = l_run * alpha + lsum;
      m_run = m_use;
      // This warp's 64 probabilities (32 bf16 pairs) into the row's lane of
      // this item's P buffer in TMEM (keys 64 half .. 64 half + 63).
      tc::st32(lane_addr + kColP + (it & 1) * 64 + 32 * half, w);
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPFull + (it & 1)]);
    }
    // ---- epilogue: O / l -> bf16 out, lse ----
    if (nit > 0 && ok)
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[kODone + ((nit - 1) & 1)], ((nit - 1) >> 1) & 1, p.status));
    tc::fence_after_sync();
    xch[half * 128 + r] = l_run;
    pair_sync(quad);
    const float l_row = l_run + xch[(half ^ 1) * 128 + r];
    if (kCluster) {
      m_fin = m_run;
      l_fin = l_row;
    } else {   // (in a cluster the partial rows are merged below)
      const float inv = (l_row > 0.f) ? 1.f / l_row : 0.f;
      __nv_bfloat16* orow = p.out + ((static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)) * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const int col = half * 64 + c * 32;
        uint32_t o[32];
        if (nit > 0) {
          tc::ld32(lane_addr + kColO + col, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        if (active) {
          uint32_t wo[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            wo[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * inv, __uint_as_float(o[2 * x + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + col);
#pragma unroll
          for (int x = 0; x < 4; ++x) dst[x] = make_uint4(wo[4 * x], wo[4 * x + 1], wo[4 * x + 2], wo[4 * x + 3]);
        }
      }
      if (active && half == 0 && p.lse) {
        p.lse[(static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)] =
            (l_row > 0.f) ? (m_run + fast_log2(l_row)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  if (kCluster) {
    // ---- cluster merge: row r of the tile is finished by CTA r % C ----
    // Each CTA's partial row (O relative to its running max m, and the row
    // sum l) goes into the owner's K ring, free once every CTA is past its
    // last item: [source rank][local row r / C][128] O and [source][row] (m, l).
    const int rp = (128 + csize - 1) / csize;
    float* part = reinterpret_cast<float*>(smem + lay.kv);
    float2* pml = reinterpret_cast<float2*>(smem + lay.kv + csize * rp * 512);
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    if (warp < kTcSoftmaxWarps) {
      const int quad = warp & 3, half = warp >> 2;
      const int r = quad * 32 + lane;
      const int dst = r % csize, lr = r / csize;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * 32) << 16);
      const uint32_t a = dsmem_addr(part + (rank * rp + lr) * 128 + half * 64, static_cast<uint32_t>(dst));
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        if (nit > 0) {
          tc::ld32(lane_addr + kColO + half * 64 + c * 32, o);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
#pragma unroll
        for (int x = 0; x < 8; ++x)
          st_dsmem_f32x4(a + c * 128 + 16 * x,
                         make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                     __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3])));
      }
      if (half == 0)
        st_dsmem_f32x2(dsmem_addr(pml + rank * rp + lr, static_cast<uint32_t>(dst)), make_float2(m_fin, l_fin));
    }
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    // Owner: M = max_c m_c, O = sum_c 2^(m_c - M) O_c, l likewise; four
    // columns of one row per thread.
#pragma unroll 1
    for (int e = tid; e < rp * 32; e += kTcThreads) {
      const int lr = e >> 5, c4 = e & 31;
      const int r = lr * csize + rank;
      if (r >= 128 || (r >> 4) >= n_act) continue;
      float mx = -INFINITY;
      for (int c = 0; c < csize; ++c) mx = fmaxf(mx, pml[c * rp + lr].x);
      float l = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if (mx > -INFINITY) {
        for (int c = 0; c < csize; ++c) {
          const float2 ml = pml[c * rp + lr];
          const float w = fast_exp2(ml.x - mx);
          const float4 v = *reinterpret_cast<const float4*>(part + (c * rp + lr) * 128 + 4 * c4);
          l = fmaf(w, ml.y, l);
          o.x = fmaf(w, v.x, o.x);
          o.y = fmaf(w, v.y, o.y);
          o.z = fmaf(w, v.z, o.z);
          o.w = fmaf(w, v.w, o.w);
        }
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const int tok = r >> 4;
      __nv_bfloat16* orow =
          p.out + ((static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)) * kHeadDim + 4 * c4;
      *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(o.x * inv, o.y * inv), pack_bf16x2(o.z * inv, o.w * inv));
      if (c4 == 0 && p.lse)
        p.lse[(static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)] =
            (l > 0.f) ? (mx + fast_log2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Clusters of C CTAs resident at once on the current device (cached; every
// launch of the kernel runs one CTA per SM).
int tc_active_clusters(int C) {
  static int cache[64][17];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    const bool ok =
        cudaFuncSetAttribute(attn_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem) ==
            cudaSuccess &&
        cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem) ==
            cudaSuccess &&
        cudaFuncSetAttribute(attn_tc_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    for (int c = 1; c <= 16; ++c) {
      int n = 0;
      if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c, 1, 1);
        cfg.blockDim = dim3(kTcThreads, 1, 1);
        cfg.dynamicSmemBytes = kTcMaxSmem;
        cudaLaunchAttribute a[1];
        a[0].id = cudaLaunchAttributeClusterDimension;
        a[0].val.clusterDim.x = c;
        a[0].val.clusterDim.y = 1;
        a[0].val.clusterDim.z = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<true>, &cfg) != cudaSuccess) n = 0;
      }
      cache[dev][c] = n;
    }
    cudaGetLastError();
    done[dev] = true;
  }
  return cache[dev][C];
}

}  // namespace

bool attn_tc_fits(const Shape& s) { return tc_layout(s.nbmax).total + 1024 <= kTcMaxSmem; }

// CTAs per tile: 1 while the tiles alone fill half the SMs; otherwise the
// largest cluster (at most 16, and at most one CTA per two union blocks of a
// full selection) with which every tile's cluster is resident at once.
int attn_tc_cluster_size(const Shape& s) {
  const long long units = static_cast<long long>((s.nq + kTcTokens - 1) / kTcTokens) * s.B * s.Hkv;
  if (units * 2 > device_sm_count()) return 1;
  for (int C = std::min(16, s.kmax / 2); C >= 2; --C)
    if (tc_active_clusters(C) >= units) return C;
  return 1;
}

cudaError_t launch_attn_tc(const Shape& s, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, const int32_t* kv_lens, const int32_t* block_idx,
                           const int32_t* n_sel, void* out, float* lse, uint32_t* status, cudaStream_t st) {
  TcParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.kmax = s.kmax;
  p.nbmax = s.nbmax;
  p.scale2 = s.attn_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.status = status;
  if (!attn_tc_fits(s) || tc_active_clusters(1) < 1) return cudaErrorInvalidConfiguration;
  p.csize = attn_tc_cluster_size(s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((s.nq + kTcTokens - 1) / kTcTokens) * p.csize, s.Hkv, s.B);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_layout(s.nbmax).total + 1024;
  cfg.stream = st;
  // Programmatic dependent launch: the CTAs start while the previous kernel
  // drains and wait for it before their first global read.
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = p.csize;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = p.csize > 1 ? 2 : 1;
  return p.csize > 1 ? cudaLaunchKernelEx(&cfg, attn_tc_kernel<true>, q_map, k_map, v_map, p)
                     : cudaLaunchKernelEx(&cfg, attn_tc_kernel<false>, q_map, k_map, v_map, p);
}

}  // namespace infllmv2
