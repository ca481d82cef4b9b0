// Stage 2 of InfLLM v2 for prefill on the 5th-generation tensor cores.
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck]:
// for each query token of a GQA group,
//   z[h, j] = score_scale * q_h . Mean_j        (visible kernels j)
//   g[j]    = (1/16) sum_h 2^(z[h, j] - lse_h)  (exact two-pass LSE, base 2)
//   r[blk]  = max of g over the kernels meeting the block,
// then the top-k with forced blocks ([> Initial and local tokens always
// selected]).
//
// One CTA per 8 consecutive tokens of one (b, h_kv): their 8 x 16 heads are
// the 128 rows of the tcgen05 tile and share every 64-kernel chunk of kernel
// means (causality gives the 8 tokens the same kernels but for the last one
// or two).  z = q . hi + q . lo comes from one product per chunk (M 128,
// N 128, K 128): the chunk's 64 hi rows and 64 lo rows are the 128 rows of B,
// so TMEM receives q . hi and q . lo side by side and the row threads add
// them (an N = 128 product issues at a higher rate than two of N = 64).
// q, the A operand, sits in TMEM too (the row warps write it there), so
// shared memory holds only the chunk ring and the block scores and two CTAs
// fit on an SM while the scores are small.  The chunks are streamed twice:
//   pass 1: each row thread keeps its head's running (max, sum of 2^z)
//           (over coarse windows instead, for the LSE approximation);
//   pass 2: each row thread forms 2^(z - lse) for its head, and the 16 lanes
//           of a token reduce-scatter the warp's 32 kernels so that lane x
//           ends with the group sums of kernels 2x, 2x + 1; two neighbouring
//           lanes and the kernel left of them are exactly the kernels meeting
//           one block.
// Roles (320 threads): warps 0-7 rows (two per TMEM lane quadrant, each with
// 32 of a chunk's 64 kernels; row r = 32 (w % 4) + lane: token r / 16, head
// r % 16), warp 8 MMA issuer (one thread), warp 9 TMA producer.  The row
// warps end with one token's warp top-k each.
//
// Few tiles (2-16 tokens per sequence: speculative verification, short
// chunks) would leave most SMs idle, so a tile's chunks are then split over
// a cluster of C CTAs (CTA r: chunks [r n / C, (r + 1) n / C)).  At the end
// of pass 1 each CTA sends its rows' (max, sum) to every CTA with st.async,
// counted on the receiver's mbarrier (the producer and the MMA issuer go on
// streaming pass 2 meanwhile); each CTA merges the C partials into the LSE.
// Pass 2 writes each block score straight into the shared memory of the
// token's owner (token t: CTA t mod C), plus the g of the CTA's last kernel,
// which the block after its range needs.  After one cluster barrier the
// owner completes those boundary blocks and runs the CTA-wide top-k.
#include "select_common.cuh"
#include "tc.cuh"

namespace infllmv2 {

namespace {

constexpr int kStTokens = 8;
constexpr int kStChunk = 64;               // kernels per chunk
constexpr int kStMaxStages = 3;            // ring depth at one CTA per SM (two stages when two CTAs fit)
constexpr int kStChunkBytes = 32768;       // per 64-dim box: 64 hi rows then 64 lo rows (128 B each)
constexpr int kStRowWarps = 8;             // two per TMEM lane quadrant, 32 of a chunk's 64 kernels each
constexpr int kStThreads = (kStRowWarps + 2) * 32;
constexpr int kStMmaWarp = kStRowWarps, kStTmaWarp = kStRowWarps + 1;
constexpr uint32_t kStTmemCols = 256;      // z (q . hi | q . lo, 64 columns each), then q
constexpr uint32_t kStColQ = 128;          // q: 128 rows x 128 dims as bf16 pairs (the A operand)
constexpr int kStTwoPerSmSmem = 112 * 1024;   // a request this small leaves room for a second CTA on the SM

struct StLayout {
  int ring, r, flag, tk, ctk, cbits, csurv, xch, lse_in, tails, bars, slot, total;
};
constexpr int kStMaxC = 16;
constexpr int kStOnePerSmSmem = 116 * 1024;     // a request this large leaves no room for a second CTA

// The top-k flags and scratch overlay the chunk ring, which is idle once the
// last chunk's products are done (every row warp has waited for them before
// its top-k).
// r_rows: tokens whose block scores this CTA holds (8; in a cluster of C
// the ceil(8 / C) it owns; 0 when they live in global scratch).
__host__ __device__ inline StLayout st_layout(int nbmax, int stages, bool clustered, int r_rows) {
  StLayout l;
  l.ring = 0;
  l.flag = 0;                                           // [8 tokens][nbmax] top-k flags (in the ring)
  l.tk = (kStTokens * nbmax + 15) & ~15;                // one warp top-k scratch per token (in the ring)
  l.ctk = 0;                                            // cluster form: the CTA-wide top-k scratch (in the ring)
  l.cbits = (static_cast<int>(sizeof(SmemTopkScratch<kStThreads>)) + 15) & ~15;
  l.csurv = l.cbits + (((nbmax + 31) / 32 * 4 + 15) & ~15);
  l.r = stages * kStChunkBytes;                         // [r_rows][nbmax] block scores
  l.xch = (l.r + r_rows * nbmax * 4 + 15) & ~15;        // [2][128] (max, sum)
  l.lse_in = l.xch + 2 * 128 * 8;                       // cluster form: [C][128 rows] (max, sum)
  l.tails = l.lse_in + (clustered ? kStMaxC * 128 * 8 : 0);   // cluster form: [C][8 tokens] last-kernel g
  l.bars = l.tails + (clustered ? kStMaxC * kStTokens * 4 : 0);
  l.slot = l.bars + 16 * 8;
  l.total = l.slot + 16;
  const int ring_need = clustered ? l.csurv + nbmax * 8 : l.tk + kStTokens * static_cast<int>(sizeof(WarpTopkScratch));
  if (ring_need > stages * kStChunkBytes) l.total = 1 << 30;   // does not fit: never chosen
  return l;
}

enum StBar { kFull = 0, kEmpty = kFull + kStMaxStages, kQ = kEmpty + kStMaxStages, kZFull = kQ + 1,
             kZFree = kZFull + 1, kLse = kZFree + 1, kStNumBars = kLse + 1 };

// Barrier of the two row warps of TMEM lane quadrant q (ids 1..4).
__device__ __forceinline__ void quad_pair_sync(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(q + 1) : "memory");
}
static_assert(kStNumBars <= 16, "barrier area holds 16");

__global__ void __launch_bounds__(kStThreads, 2)
    sel_tc_kernel(const __grid_constant__ CUtensorMap kc_map, const __grid_constant__ CUtensorMap kcc_map,
                  SelParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int S = p.stages;
  const int csize = p.csize;
  const StLayout lay = st_layout(p.nbmax, S, csize > 1, p.r_rows);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + lay.slot);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.Hkv + h;
  const int nq = p.nq;
  const int rank = static_cast<int>(blockIdx.x) % csize;   // == the rank in the cluster
  const int t0 = (static_cast<int>(blockIdx.x) / csize) * kStTokens;
  const int n_act = min(kStTokens, nq - t0);
  pdl_wait();   // the previous kernel of the stream may still be writing the inputs
  pdl_trigger();
  // Block scores of the tile's 8 tokens: in shared memory, or past that
  // capacity in this SM's slot of the global scratch (that form requests more
  // than half an SM's shared memory, so no two of its CTAs share an SM).
  const uint32_t slot = sm_id();
  if (p.r_scratch && slot >= static_cast<uint32_t>(p.r_slots)) {   // cannot happen with slots from %nsmid
    for (int e = tid; e < n_act * p.kmax; e += kStThreads)
      p.block_idx[(static_cast<size_t>(bh) * nq + t0 + e / p.kmax) * p.kmax + e % p.kmax] = -1;
    if (tid < n_act) p.n_sel[static_cast<size_t>(bh) * nq + t0 + tid] = 0;
    if (tid == 0) atomicOr(p.status, kStatusBounds);
    return;
  }
  float* r_all = p.r_scratch ? p.r_scratch + static_cast<size_t>(slot) * kStTokens * p.nbmax
                             : reinterpret_cast<float*>(smem + lay.r);
  const int r_rows = p.r_scratch ? kStTokens : p.r_rows;
  const int L = p.kv_lens[b];

  if (L < nq || L > p.Lmax) {   // the same in every CTA of a cluster: none touches another's memory
    if (rank != 0) return;
    for (int e = tid; e < n_act * p.kmax; e += kStThreads) {
      const size_t u = static_cast<size_t>(bh) * nq + t0 + e / p.kmax;
      p.block_idx[u * p.kmax + e % p.kmax] = -1;
    }
    if (p.write_r)
      for (int e = tid; e < n_act * p.nbmax; e += kStThreads)
        p.r_buf[(static_cast<size_t>(bh) * nq + t0 + e / p.nbmax) * p.nbmax + e % p.nbmax] = -INFINITY;
    if (tid < n_act) p.n_sel[static_cast<size_t>(bh) * nq + t0 + tid] = 0;
    if (tid == 0) atomicOr(p.status, kStatusBadKvLen);
    return;
  }
  const int nvis_max = n_complete_kernels(L - nq + t0 + n_act);
  const int nch = (nvis_max + kStChunk - 1) / kStChunk;
  const int ch0 = rank * nch / csize, ch1 = (rank + 1) * nch / csize;   // this CTA's fine chunks
  const int nch_my = ch1 - ch0;
  // Stream of chunks: A (coarse windows, the LSE approximation [InfLLM v2 >
  // Efficient LSE approximation]; only with p.sc > 0), B (fine LSE, for the
  // tokens without a complete window; skipped when every token has one), C
  // (fine, normalise and block maxima).  p.sc = 0: B and C only.
  const int nvis_c_max = p.sc ? (L - nq + t0 + n_act) / p.sc : 0;
  const int nch_a = (nvis_c_max + kStChunk - 1) / kStChunk;
  const bool need_b = p.sc == 0 || (L - nq + t0 + 1) / p.sc == 0;
  const int seg_c = nch_a + (need_b ? nch_my : 0);
  const int total = nch_my > 0 ? seg_c + nch_my : 0;

  // Each row thread's q (dims 64 hf .. 64 hf + 63 of row r = token r / 16,
  // head r % 16; see the row warps below): loaded now, so that the loads
  // land while the barriers and TMEM are set up, and stored to TMEM there.
  uint32_t qw[32];
  if (warp < kStRowWarps && total > 0) {
    const int r = (warp & 3) * 32 + lane, tok = r >> 4, hf = warp >> 2;
    if (tok < n_act) {
      const size_t row = (static_cast<size_t>(b) * nq + t0 + tok) * (p.Hkv * kGroup) + h * kGroup + (r & 15);
      const uint4* src = reinterpret_cast<const uint4*>(p.q + row * 128 + 64 * hf);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 u = __ldg(src + i);
        qw[4 * i] = u.x;
        qw[4 * i + 1] = u.y;
        qw[4 * i + 2] = u.z;
        qw[4 * i + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qw[i] = 0u;
    }
  }

  for (int e = tid; e < r_rows * p.nbmax; e += kStThreads) r_all[e] = -INFINITY;
  if (tid == 0) {
    prefetch_tensormap(&kc_map);
    if (p.sc) prefetch_tensormap(&kcc_map);
    for (int s = 0; s < S; ++s) {
      mbar_init(&bars[kFull + s], 1);
      mbar_init(&bars[kEmpty + s], 1);
    }
    mbar_init(&bars[kQ], kStRowWarps);   // q written to TMEM by the row warps
    mbar_init(&bars[kZFull], 1);
    mbar_init(&bars[kZFree], kStRowWarps);   // z read out: the next chunk's product may overwrite it
    mbar_init(&bars[kLse], 1);
    // Cluster form: the C partials of 128 rows arrive by st.async.
    if (csize > 1) mbar_arrive_expect_tx(&bars[kLse], csize * 128 * 8);
    fence_barrier_init();
  }
  if (warp == kStMmaWarp) {
    tc::tmem_alloc(tmem_slot, kStTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (csize > 1) {   // every CTA's barriers and block scores initialised before any remote store
    cluster_arrive();
    cluster_wait();
  }
  const uint32_t tmem = *tmem_slot;
  const uint32_t base_s = smem_u32(smem);

  if (warp == kStTmaWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && total > 0) {
      for (int it = 0; it < total; ++it) {
        const int st = it % S;
        if (it >= S && !mbar_wait(&bars[kEmpty + st], ((it / S) - 1) & 1, p.status)) break;
        const bool coarse_seg = it < nch_a;
        const int ch = coarse_seg ? it : ch0 + (it < seg_c ? it - nch_a : it - seg_c);
        const CUtensorMap* map = coarse_seg ? &kcc_map : &kc_map;
        const int rows = coarse_seg ? p.nccmax : p.ncmax;
        uint8_t* dst = smem + lay.ring + st * kStChunkBytes;
        const int row_hi = (bh * 2 + 0) * rows + ch * kStChunk;
        const int row_lo = (bh * 2 + 1) * rows + ch * kStChunk;
        mbar_arrive_expect_tx(&bars[kFull + st], kStChunkBytes);
        tma_load_2d(dst, map, 0, row_hi, &bars[kFull + st]);
        tma_load_2d(dst + 8192, map, 0, row_lo, &bars[kFull + st]);
        tma_load_2d(dst + 16384, map, 64, row_hi, &bars[kFull + st]);
        tma_load_2d(dst + 24576, map, 64, row_lo, &bars[kFull + st]);
      }
    }
    __syncwarp();
  } else if (warp == kStMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && total > 0) {
      constexpr uint32_t kId = tc::idesc_bf16(128, 128, 0, 0);
      bool ok = mbar_wait(&bars[kQ], 0, p.status);
      for (int it = 0; it < total && ok; ++it) {
        const int st = it % S;
        ok = mbar_wait(&bars[kFull + st], (it / S) & 1, p.status);
        if (ok && it >= 1) ok = mbar_wait(&bars[kZFree], (it - 1) & 1, p.status);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t stage = base_s + lay.ring + st * kStChunkBytes;
        const uint64_t b_desc = tc::sdesc_sw128(stage, 16, 1024);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          // A: q from TMEM (16 dims = 8 columns per step); B: the chunk's 128
          // rows (hi, then lo), dims 16 k .. 16 k + 15 of the 64-dim boxes.
          const uint64_t tb = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
          tc::mma_ts(tmem, tmem + kStColQ + 8 * k, b_desc + tb, kId, k > 0 ? 1u : 0u);
        }
        tc::commit(&bars[kZFull]);
        tc::commit(&bars[kEmpty + st]);
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- rows
    // Warp w: TMEM lane quadrant q = w % 4 (rows 32 q .. 32 q + 31: tokens
    // 2 q and 2 q + 1, lanes 0-15 and 16-31), kernels 32 hf .. 32 hf + 31 of
    // each chunk with hf = w / 4.
    const int q4 = warp & 3, hf = warp >> 2;
    const int r = q4 * 32 + lane;
    const int tok = r >> 4, x = r & 15;
    const bool active = tok < n_act;
    const int i_t = L - nq + t0 + (active ? tok : n_act - 1);
    const int c_t = i_t / kBlock;
    const int nvis_t = active ? n_complete_kernels(i_t + 1) : 0;
    const int nvis_c_t = (active && p.sc) ? (i_t + 1) / p.sc : 0;   // complete coarse windows
    const bool coarse_t = nvis_c_t > 0;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    float2* xch = reinterpret_cast<float2*>(smem + lay.xch);
    float* r_tok = r_all + (tok / csize) * p.nbmax;   // in the owner's rows (token t: CTA t mod C, row t / C)
    const int col0 = 32 * hf;
    // The kernel left of this half's first block: column 31 of the same
    // chunk for the upper half; for the lower half, column 63 of the
    // previous chunk, carried.
    const int xcol = hf ? 31 : 63;
    float m = -INFINITY, l = 0.f, lse2 = -INFINITY;
    float carry = -INFINITY;
    bool ok = true;
    // q of this row, dims 64 hf .. 64 hf + 63, into TMEM columns
    // kStColQ + 32 hf .. + 31 as bf16 pairs: the A operand of the products.
    if (total > 0) {
      tc::st32(lane_addr + kStColQ + 32 * hf, qw);
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kQ]);
    }
    // End of pass 1: merge the two halves' (max, sum) of each row; in a
    // cluster also the C CTAs' partials of the row.
    auto end_pass1 = [&]() {
      xch[hf * 128 + r] = make_float2(m, l);
      quad_pair_sync(q4);
      const float2 o = xch[(hf ^ 1) * 128 + r];
      lse_merge(m, l, o.x, o.y);
      if (csize > 1) {
        float2* lse_in = reinterpret_cast<float2*>(smem + lay.lse_in);
        if (hf == 0)
          for (int d = 0; d < csize; ++d)
            st_async_f32x2(dsmem_addr(lse_in + rank * 128 + r, static_cast<uint32_t>(d)), make_float2(m, l),
                           dsmem_addr(&bars[kLse], static_cast<uint32_t>(d)));
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_cluster(&bars[kLse], 0, p.status));
        m = -INFINITY;
        l = 0.f;
        for (int c = 0; c < csize; ++c) {
          const float2 v = lse_in[c * 128 + r];
          lse_merge(m, l, v.x, v.y);
        }
      }
      lse2 = (m == -INFINITY) ? -INFINITY : m + fast_log2(l);
    };
    // Block score j of this row's token: into its own row here, or into the
    // owner's in a cluster.
    auto put_r = [&](int j, float v) {
      if (csize == 1)
        r_tok[j] = v;
      else
        st_dsmem_f32(dsmem_addr(r_tok + j, static_cast<uint32_t>(tok % csize)), v);
    };
    for (int it = 0; it < total; ++it) {
      const bool pass2 = it >= seg_c;
      const int kbase = (it < nch_a ? it : ch0 + (pass2 ? it - seg_c : it - nch_a)) * kStChunk;
      if (it == seg_c) end_pass1();
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kZFull], it & 1, p.status));
      tc::fence_after_sync();
      uint32_t v[32];
      uint32_t vl[32];   // q . lo of the same kernels, 64 columns on
      tc::ld32(lane_addr + col0, v);
      tc::ld32(lane_addr + 64 + col0, vl);
      uint32_t vx = pass2 ? tc::ld1(lane_addr + xcol) : 0u;
      const uint32_t vxl = pass2 ? tc::ld1(lane_addr + 64 + xcol) : 0u;
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kZFree]);
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) + __uint_as_float(vl[k]));
      vx = __float_as_uint(__uint_as_float(vx) + __uint_as_float(vxl));
      // This row's visible rows of the chunk: coarse windows in segment A for
      // a token that has one, fine kernels in B for a token that has none,
      // fine kernels in C.
      const int nvis_seg = it < nch_a ? (coarse_t ? nvis_c_t : 0) : (pass2 ? nvis_t : (coarse_t ? 0 : nvis_t));
      const int nv = max(0, min(kStChunk, nvis_seg - kbase)) - col0;   // visible among this half's 32
      if (!pass2) {
        if (nv > 0) {
          float cm = -INFINITY;
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (k < nv) cm = fmaxf(cm, __uint_as_float(v[k]));
          const float M = fmaxf(m, cm * p.scale2);
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            s0 += (k < nv) ? fast_exp2(fmaf(__uint_as_float(v[k]), p.scale2, -M)) : 0.f;
            s1 += (k + 1 < nv) ? fast_exp2(fmaf(__uint_as_float(v[k + 1]), p.scale2, -M)) : 0.f;
          }
          l = l * fast_exp2(m - M) + (s0 + s1);
          m = M;
        }
      } else {
        float e[32];
#pragma unroll
        for (int k = 0; k < 32; ++k)
          e[k] = (k < nv) ? fast_exp2(fmaf(__uint_as_float(v[k]), p.scale2, -lse2)) : 0.f;
        // The extra kernel (xcol), summed over the token's 16 heads.
        const int nvx = max(0, min(kStChunk, nvis_seg - kbase));
        float ex = (xcol < nvx) ? fast_exp2(fmaf(__uint_as_float(vx), p.scale2, -lse2)) : 0.f;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ex += __shfl_xor_sync(0xffffffffu, ex, o);
        ex *= 1.0f / kGroup;
        // Reduce-scatter over the token's 16 lanes (xor 8, 4, 2, 1): lane x
        // keeps the half of its range selected by bit 3, 2, 1, 0 of x and adds
        // the partner's copy of that half; it ends with kernels 2x, 2x + 1 of
        // this warp's 32.
        const bool b3 = x & 8, b2 = x & 4, b1 = x & 2, b0 = x & 1;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float send = b3 ? e[k] : e[k + 16];
          const float keep = b3 ? e[k + 16] : e[k];
          e[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float send = b2 ? e[k] : e[k + 8];
          const float keep = b2 ? e[k + 8] : e[k];
          e[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float send = b1 ? e[k] : e[k + 4];
          const float keep = b1 ? e[k + 4] : e[k];
          e[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const float send = b0 ? e[k] : e[k + 2];
          const float keep = b0 ? e[k + 2] : e[k];
          e[k] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
        }
        // Lane x: group values of kernels kbase + col0 + 2x, + 2x + 1.  Block
        // b = x / 2 of the half (kernels 4b .. 4b + 3) is finished by the odd
        // lane, with kernel 4b - 1 from lane x - 2 (or the extra kernel).
        const float g0 = e[0] * (1.0f / kGroup), g1 = e[1] * (1.0f / kGroup);
        const int grp = lane & 16;
        const float p0 = __shfl_sync(0xffffffffu, g0, grp | ((x + 15) & 15));
        const float p1 = __shfl_sync(0xffffffffu, g1, grp | ((x + 15) & 15));
        const float pl = __shfl_sync(0xffffffffu, g1, grp | ((x + 14) & 15));
        const float left = hf ? ex : carry;
        if (!hf) carry = ex;   // column 63 of this chunk, for the next chunk's first block
        if (x & 1) {
          const int j = (kbase + col0) / 4 + (x >> 1);
          const float prev = x == 1 ? left : pl;
          if (active && j <= c_t && j < p.nbmax) {
            const bool has = max(0, 4 * j - 1) < nvis_t;
            put_r(j, has ? fmaxf(fmaxf(prev, fmaxf(p0, p1)), fmaxf(g0, g1)) : -INFINITY);
          }
        }
      }
    }
    if (csize > 1) {
      // A CTA without chunks still sends its (empty) partials.
      if (total == 0) end_pass1();
      // The block after this CTA's range meets its last kernel (4 j - 1):
      // the owner completes that block with it.
      if (hf == 0 && x == 0 && active) {
        float* tails = reinterpret_cast<float*>(smem + lay.tails);
        st_dsmem_f32(dsmem_addr(tails + rank * kStTokens + tok, static_cast<uint32_t>(tok % csize)), carry);
      }
    } else if (nch > 0 && hf == 0 && x == 0 && active) {
      // The block after the last chunk meets one kernel of it (4 j - 1): the
      // lower-half warp carries it.
      const int j = nch * (kStChunk / 4);
      if (j <= c_t && j < p.nbmax && 4 * j - 1 < nvis_t) r_tok[j] = carry;
    }
    quad_pair_sync(q4);
    // The top-k flags and scratch lie over the chunk ring, which the TMA and
    // the tensor cores are done with (every row warp has seen the last
    // chunk's products complete); order these ordinary stores after them.
    fence_proxy_async_smem();
    // Top-k: warp (q, hf) takes token 2 q + hf, whose scores the two warps of
    // the quadrant wrote.
    if (csize == 1) {
      const int tt = 2 * q4 + hf;
      if (tt < n_act) {
        WarpTopkScratch& tk = reinterpret_cast<WarpTopkScratch*>(smem + lay.tk)[tt];
        const size_t u = static_cast<size_t>(bh) * nq + t0 + tt;
        const float* rw = r_all + tt * p.nbmax;
        if (p.write_r)
          for (int jj = lane; jj < p.nbmax; jj += 32) p.r_buf[u * p.nbmax + jj] = rw[jj];
        const int c = (L - nq + t0 + tt) / kBlock;
        select_topk_warp(rw, smem + lay.flag + tt * p.nbmax, c + 1, p.n_init, p.n_local, p.topk,
                         p.inc_forced != 0, p.kmax, p.block_idx + u * p.kmax, p.n_sel + u, tk, lane);
      }
    }
  }

  if (csize > 1) {
    // ---- cluster: the owner CTA's tokens (t mod C == rank) ----
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    fence_proxy_async_smem();   // the top-k scratch lies over the TMA-written ring
    SmemTopkScratch<kStThreads>& tk = *reinterpret_cast<SmemTopkScratch<kStThreads>*>(smem + lay.ctk);
    uint32_t* tbits = reinterpret_cast<uint32_t*>(smem + lay.cbits);
    unsigned long long* tsurv = reinterpret_cast<unsigned long long*>(smem + lay.csurv);
    const float* tails = reinterpret_cast<const float*>(smem + lay.tails);
#pragma unroll 1
    for (int tt = rank; tt < n_act; tt += csize) {
      float* rw = r_all + (tt / csize) * p.nbmax;
      const int i_t = L - nq + t0 + tt, c = i_t / kBlock;
      if (tid == 0) {   // the block after CTA q's range, with q's last kernel (CTAs without chunks share an end)
        const int nvis = n_complete_kernels(i_t + 1);
        for (int q = 0; q < csize; ++q) {
          const int j = 16 * ((q + 1) * nch / csize);
          if (j <= c && j < p.nbmax && 4 * j - 1 < nvis) rw[j] = fmaxf(rw[j], tails[q * kStTokens + tt]);
        }
      }
      __syncthreads();
      const size_t u = static_cast<size_t>(bh) * nq + t0 + tt;
      if (p.write_r)
        for (int jj = tid; jj < p.nbmax; jj += kStThreads) p.r_buf[u * p.nbmax + jj] = rw[jj];
      select_topk_smem<kStThreads>(rw, c + 1, p.n_init, p.n_local, p.topk, p.inc_forced != 0, p.kmax,
                                   p.block_idx + u * p.kmax, p.n_sel + u, tk, tbits, tsurv, tid);
      __syncthreads();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kStMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kStTmemCols);
  }
}

// Clusters of C CTAs of `smem` bytes each resident at once on the current
// device (cached per device, C and smem class: up to kStTwoPerSmSmem, two
// CTAs fit on an SM; past it one).
int st_active_clusters(int C, int smem) {
  static int cache[64][2][kStMaxC + 1];
  static bool done[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!done[dev]) {
    const bool ok =
        cudaFuncSetAttribute(sel_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) == cudaSuccess &&
        cudaFuncSetAttribute(sel_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    for (int k = 0; k < 2; ++k)
      for (int c = 1; c <= kStMaxC; ++c) {
        int n = 0;
        if (ok) {
          cudaLaunchConfig_t cfg = {};
          cfg.gridDim = dim3(c, 1, 1);
          cfg.blockDim = dim3(kStThreads, 1, 1);
          cfg.dynamicSmemBytes = k == 0 ? kStTwoPerSmSmem : kStOnePerSmSmem;
          cudaLaunchAttribute a[1];
          a[0].id = cudaLaunchAttributeClusterDimension;
          a[0].val.clusterDim.x = c;
          a[0].val.clusterDim.y = 1;
          a[0].val.clusterDim.z = 1;
          cfg.attrs = a;
          cfg.numAttrs = 1;
          if (cudaOccupancyMaxActiveClusters(&n, sel_tc_kernel, &cfg) != cudaSuccess) n = 0;
        }
        cache[dev][k][c] = n;
      }
    cudaGetLastError();
    done[dev] = true;
  }
  return cache[dev][smem <= kStTwoPerSmSmem ? 0 : 1][C];
}

// Pipeline depth and dynamic shared memory of a launch with C CTAs per tile.
// Two stages when that leaves room for a second CTA on the SM (each SM then
// streams four chunks at once and overlaps one CTA's row work with the
// other's products); else the deepest ring that fits.  Off chip the block
// scores take one global slot per SM, so one CTA per SM (padded to
// kStOnePerSmSmem).
struct StConfig {
  int stages, smem, r_rows;
};

StConfig st_config(const Shape& s, int csize, bool offchip) {
  StConfig c{0, 0, offchip ? 0 : (kStTokens + csize - 1) / csize};
  const bool clustered = csize > 1;
  const int two = st_layout(s.nbmax, 2, clustered, c.r_rows).total + 1024;
  if (!offchip && two <= kStTwoPerSmSmem) return StConfig{2, two, c.r_rows};
  for (int st = kStMaxStages; st >= 2; --st) {
    const int t = st_layout(s.nbmax, st, clustered, c.r_rows).total + 1024;
    if (t <= 227 * 1024) return StConfig{st, offchip ? std::max(t, kStOnePerSmSmem) : t, c.r_rows};
  }
  return c;
}

}  // namespace

int select_tc_stages(const Shape& s) { return st_config(s, 1, false).stages; }

// The 8 tokens' block scores fit in shared memory (the coarse-LSE selection
// needs this: it takes no workspace).
bool select_tc_onchip(const Shape& s) { return select_tc_stages(s) > 0; }

bool select_tc_supported(const Shape& s) { return select_tc_onchip(s) || st_config(s, 1, true).stages > 0; }

namespace {

__device__ int g_sm_id_bound;

__global__ void sm_id_bound_kernel() { g_sm_id_bound = static_cast<int>(sm_id_bound()); }

// The bound on SM identifiers of the current device (%nsmid), read once per
// device by a one-thread kernel on a private stream (no allocation); without
// a device, twice the SM count.
int device_sm_id_bound() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2 * device_sm_count();
  if (!cache[dev]) {
    int n = 0;
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess) {
      sm_id_bound_kernel<<<1, 1, 0, st>>>();
      if (cudaMemcpyFromSymbolAsync(&n, g_sm_id_bound, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        n = 0;
      cudaStreamDestroy(st);
    }
    cudaGetLastError();
    cache[dev] = n > 0 ? n : 2 * device_sm_count();
  }
  return cache[dev];
}

}  // namespace

// Global scratch for the block scores where they do not fit on chip: one
// [8][nbmax] slot per SM identifier.
int select_tc_scratch_slots(const Shape& s) {
  return (select_tc_onchip(s) || !select_tc_supported(s)) ? 0 : device_sm_id_bound();
}

size_t select_tc_scratch_bytes(const Shape& s) {
  return static_cast<size_t>(select_tc_scratch_slots(s)) * kStTokens * s.nbmax * sizeof(float);
}

// CTAs per 8-token tile: 1 while the tiles alone fill half the SMs (or with
// the coarse LSE); otherwise the largest cluster (at most 16, at least two
// chunks per CTA) with which every tile's cluster is resident at once.
int select_tc_cluster_size(const Shape& s, int sc) {
  if (sc != 0) return 1;
  const long long units = static_cast<long long>((s.nq + kStTokens - 1) / kStTokens) * s.B * s.Hkv;
  if (units * 2 > device_sm_count()) return 1;
  const int nch = (s.ncmax + kStChunk - 1) / kStChunk;
  for (int C = std::min(kStMaxC, nch / 2); C >= 2; --C) {
    const StConfig c = st_config(s, C, false);
    if (c.stages > 0 && st_active_clusters(C, c.smem) >= units) return C;
  }
  return 1;
}

// p.sc > 0: coarse-window LSE from kcc_map (else kcc_map is not read).
cudaError_t launch_select_tc(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map,
                             const SelParams& p, cudaStream_t st) {
  SelParams pp = p;
  if (st_active_clusters(1, kStOnePerSmSmem) < 1 || p.q == nullptr) return cudaErrorInvalidConfiguration;
  const bool offchip = !select_tc_onchip(s);
  if (offchip && (p.r_scratch == nullptr || p.sc != 0)) return cudaErrorInvalidConfiguration;
  if (!offchip) pp.r_scratch = nullptr;
  pp.r_slots = offchip ? select_tc_scratch_slots(s) : 0;
  pp.csize = offchip ? 1 : select_tc_cluster_size(s, p.sc);
  const StConfig c = st_config(s, pp.csize, offchip);
  if (c.stages == 0) return cudaErrorInvalidConfiguration;
  pp.stages = c.stages;
  pp.r_rows = c.r_rows;
  const int smem = c.smem;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(((s.nq + kStTokens - 1) / kStTokens) * pp.csize, s.Hkv, s.B);
  cfg.blockDim = dim3(kStThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // Programmatic dependent launch: the CTAs start while the previous kernel
  // drains and wait for it before their first global read.
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = pp.csize;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = pp.csize > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, sel_tc_kernel, kc_map, kcc_map, pp);
}

}  // namespace infllmv2
