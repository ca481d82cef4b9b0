// Top-k block choice shared by the selection kernels.
//
// [InfLLM v2 > Top-K implementation and the LSE bottleneck, step (3)] and
// [InfLLM v2 > Initial and local tokens always selected]: forced blocks (the
// first n_init blocks and the n_local blocks ending at the query's block c)
// are always taken; among the other blocks with a finite score the best are
// taken in order (score descending, index ascending).  The result is written
// ascending by block index and padded with -1.
//
// The threshold score is found exactly with a 4-pass radix select over the
// order-preserving 32-bit image of the fp32 scores (8-bit digits, one
// shared-memory histogram per pass); ties at the threshold go to the lowest
// indices through a prefix count in index order.  The routine is written for
// a cooperating group of NT threads: a whole CTA (NT = blockDim.x, WARP =
// false) or a single warp (NT = 32, WARP = true).
#pragma once

#include "common.cuh"

namespace infllmv2 {

template <int NT>
struct TopkScratch {
  uint32_t hist[256];
  int ctrl[4];
  int warp_tot[NT / 32 > 0 ? NT / 32 : 1];
};

template <bool WARP>
__device__ __forceinline__ void group_sync() {
  if (WARP) {
    __syncwarp();
  } else {
    __syncthreads();
  }
}

// Exclusive prefix sum of `v` over the group; `total` receives the sum.
template <int NT, bool WARP>
__device__ __forceinline__ int group_exclusive_scan(int v, int& total, TopkScratch<NT>& sm,
                                                    int tid) {
  const int lane = tid & 31;
  int incl = warp_inclusive_scan(v);
  if (WARP) {
    total = __shfl_sync(0xffffffffu, incl, 31);
    return incl - v;
  }
  const int warp = tid >> 5;
  constexpr int NWARP = NT / 32;
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    const int x = sm.warp_tot[w];
    base += (w < warp) ? x : 0;
    tot += x;
  }
  __syncthreads();
  total = tot;
  return base + incl - v;
}

template <int NT, bool WARP>
__device__ __forceinline__ int group_sum(int v, TopkScratch<NT>& sm, int tid) {
  int total;
  group_exclusive_scan<NT, WARP>(v, total, sm, tid);
  return total;
}

// r[0..nb) : block scores of blocks 0..c (c = nb - 1), in shared memory.
// flag[0..nb) : shared scratch (bytes).  Writes out_idx[0..k_max) and *out_n.
template <int NT, bool WARP>
__device__ void select_topk(const float* r, uint8_t* flag, int nb, int n_init, int n_local,
                            int topk, bool includes_forced, int k_max, int32_t* out_idx,
                            int32_t* out_n, TopkScratch<NT>& sm, int tid) {
  const int c = nb - 1;
  const int local_lo = c - n_local + 1;
  int my_cand = 0, my_forced = 0;
  for (int j = tid; j < nb; j += NT) {
    const bool forced = (j < n_init) || (j >= local_lo);
    const bool cand = !forced && (r[j] > -INFINITY);
    flag[j] = forced ? 2 : (cand ? 1 : 0);
    my_cand += cand ? 1 : 0;
    my_forced += forced ? 1 : 0;
  }
  group_sync<WARP>();
  const int n_cand = group_sum<NT, WARP>(my_cand, sm, tid);
  const int n_forced = group_sum<NT, WARP>(my_forced, sm, tid);
  int n_take = includes_forced ? topk - n_forced : topk;
  if (n_take < 0) n_take = 0;

  const int per = (nb + NT - 1) / NT;
  const int lo = tid * per;
  const int hi = min(nb, lo + per);

  if (n_take > 0 && n_cand <= n_take) {
    for (int j = tid; j < nb; j += NT)
      if (flag[j] == 1) flag[j] = 3;
  } else if (n_take > 0) {
    uint32_t prefix = 0, pmask = 0;
    int remaining = n_take;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int b = tid; b < 256; b += NT) sm.hist[b] = 0;
      group_sync<WARP>();
      for (int j = tid; j < nb; j += NT) {
        if (flag[j] == 1) {
          const uint32_t key = float_to_ordered(r[j]);
          if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & 255u], 1u);
        }
      }
      group_sync<WARP>();
      if (tid < 32) {
        // Lane l owns digits 255-8l .. 255-8l-7 (descending).
        int cnt[8];
        int tot = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          cnt[k] = static_cast<int>(sm.hist[255 - 8 * tid - k]);
          tot += cnt[k];
        }
        int run = warp_inclusive_scan(tot) - tot;  // elements with a larger digit
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (run < remaining && run + cnt[k] >= remaining) {
            sm.ctrl[0] = 255 - 8 * tid - k;
            sm.ctrl[1] = remaining - run;
          }
          run += cnt[k];
        }
      }
      group_sync<WARP>();
      prefix |= static_cast<uint32_t>(sm.ctrl[0]) << shift;
      pmask |= 255u << shift;
      remaining = sm.ctrl[1];
      group_sync<WARP>();
    }
    // prefix = exact key of the last element taken; `remaining` of the
    // elements equal to it are taken, lowest indices first.
    int my_eq = 0;
    for (int j = lo; j < hi; ++j)
      if (flag[j] == 1 && float_to_ordered(r[j]) == prefix) ++my_eq;
    int tot_eq;
    int rank = group_exclusive_scan<NT, WARP>(my_eq, tot_eq, sm, tid);
    for (int j = lo; j < hi; ++j) {
      if (flag[j] != 1) continue;
      const uint32_t key = float_to_ordered(r[j]);
      if (key > prefix) {
        flag[j] = 3;
      } else if (key == prefix) {
        if (rank < remaining) flag[j] = 3;
        ++rank;
      }
    }
  }
  group_sync<WARP>();

  int my_sel = 0;
  for (int j = lo; j < hi; ++j) my_sel += (flag[j] >= 2) ? 1 : 0;
  int total;
  int pos = group_exclusive_scan<NT, WARP>(my_sel, total, sm, tid);
  for (int j = lo; j < hi; ++j) {
    if (flag[j] >= 2) {
      if (pos < k_max) out_idx[pos] = j;
      ++pos;
    }
  }
  for (int p = total + tid; p < k_max; p += NT) out_idx[p] = -1;
  if (tid == 0) *out_n = min(total, k_max);
}

// One warp, scores in shared memory, same rule and output as select_topk
// with one histogram pass instead of four radix passes: a 256-bin histogram
// of the candidates' leading bits (sign, exponent, 6 mantissa bits) counted
// down from the best score locates the bin of the n_take-th best; better bins
// are taken and the boundary bin (at most kWarpTopkSurv scores) is ranked
// exactly by (score desc, index asc).  A boundary bin that is the catch-all
// last bin, or holds more scores than that, goes to select_topk.
constexpr int kWarpTopkSurv = 64;

struct WarpTopkScratch {
  union {
    uint32_t hist[256];
    TopkScratch<32> radix;   // the fallback runs after the histogram is read
  };
  unsigned long long surv[kWarpTopkSurv];
  int n_surv;
};

__device__ inline void select_topk_warp(const float* r, uint8_t* flag, int nb, int n_init, int n_local, int topk,
                                 bool includes_forced, int k_max, int32_t* out_idx, int32_t* out_n,
                                 WarpTopkScratch& sm, int lane) {
  constexpr int kShift = 17;
  const int c = nb - 1;
  const int local_lo = c - n_local + 1;
  int my_cand = 0, my_forced = 0;
  uint32_t my_top = 0;
  for (int j = lane; j < nb; j += 32) {
    const bool forced = (j < n_init) || (j >= local_lo);
    const bool cand = !forced && (r[j] > -INFINITY);
    flag[j] = forced ? 2 : (cand ? 1 : 0);
    my_cand += cand ? 1 : 0;
    my_forced += forced ? 1 : 0;
    if (cand) my_top = max(my_top, float_to_ordered(r[j]) >> kShift);
  }
  for (int b = lane; b < 256; b += 32) sm.hist[b] = 0u;
  if (lane == 0) sm.n_surv = 0;
  const int n_cand = __reduce_add_sync(0xffffffffu, my_cand);
  const int n_forced = __reduce_add_sync(0xffffffffu, my_forced);
  const uint32_t top = __reduce_max_sync(0xffffffffu, my_top);
  int n_take = includes_forced ? topk - n_forced : topk;
  if (n_take < 0) n_take = 0;
  __syncwarp();
  if (n_take > 0 && n_cand <= n_take) {
    for (int j = lane; j < nb; j += 32)
      if (flag[j] == 1) flag[j] = 3;
  } else if (n_take > 0) {
    for (int j = lane; j < nb; j += 32)
      if (flag[j] == 1) atomicAdd(&sm.hist[min(255u, top - (float_to_ordered(r[j]) >> kShift))], 1u);
    __syncwarp();
    // Lane l owns bins 8 l .. 8 l + 7 (bin 0 = best).
    int cnt[8], tot = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cnt[k] = static_cast<int>(sm.hist[8 * lane + k]);
      tot += cnt[k];
    }
    int run = warp_inclusive_scan(tot) - tot;
    int my_bnd = -1, my_above = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (run < n_take && run + cnt[k] >= n_take) {
        my_bnd = 8 * lane + k;
        my_above = run;
      }
      run += cnt[k];
    }
    const int src = __ffs(__ballot_sync(0xffffffffu, my_bnd >= 0)) - 1;
    const int bnd = __shfl_sync(0xffffffffu, my_bnd, src);
    const int above = __shfl_sync(0xffffffffu, my_above, src);
    const int in_bnd = static_cast<int>(sm.hist[bnd]);
    if (bnd == 255 || in_bnd > kWarpTopkSurv) {
      __syncwarp();
      select_topk<32, true>(r, flag, nb, n_init, n_local, topk, includes_forced, k_max, out_idx, out_n, sm.radix,
                            lane);
      return;
    }
    for (int j = lane; j < nb; j += 32) {
      if (flag[j] != 1) continue;
      const uint32_t key = float_to_ordered(r[j]);
      const int d = static_cast<int>(min(255u, top - (key >> kShift)));
      if (d < bnd) {
        flag[j] = 3;
      } else if (d == bnd) {
        sm.surv[atomicAdd(&sm.n_surv, 1)] = (static_cast<unsigned long long>(key) << 32) |
                                            static_cast<uint32_t>(~j);
      }
    }
    __syncwarp();
    const int m = sm.n_surv, need = n_take - above;
    for (int x = lane; x < m; x += 32) {
      const unsigned long long me = sm.surv[x];
      int rk = 0;
      for (int y = 0; y < m; ++y) rk += (sm.surv[y] > me) ? 1 : 0;
      if (rk < need) flag[~static_cast<uint32_t>(me & 0xffffffffu)] = 3;
    }
  }
  __syncwarp();
  const int per = (nb + 31) / 32;
  const int lo = lane * per, hi = min(nb, lo + per);
  int my_sel = 0;
  for (int j = lo; j < hi; ++j) my_sel += (flag[j] >= 2) ? 1 : 0;
  const int incl = warp_inclusive_scan(my_sel);
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int pos = incl - my_sel;
  for (int j = lo; j < hi; ++j) {
    if (flag[j] >= 2) {
      if (pos < k_max) out_idx[pos] = j;
      ++pos;
    }
  }
  for (int q = total + lane; q < k_max; q += 32) out_idx[q] = -1;
  if (lane == 0) *out_n = min(total, k_max);
}

// Top-k over scores held in registers: thread tid holds the scores of blocks
// j = tid + NT x (x < MAXR) in v[x].  Same selection rule and output as
// select_topk.  The chosen blocks are marked in a bitmask whose ascending
// scan is the output, so no step sorts or ranks more than the few scores
// tied for the last places:
//   1. a 256-bin histogram of the candidates' leading bits (sign, exponent,
//      6 mantissa bits) counted down from the best score locates the bin
//      holding the n_take-th best; when that is the catch-all last bin and
//      it holds more than NT scores, a second histogram over that bin (16
//      times coarser, reaching 68 octaves below the best) narrows it;
//   2. candidates in better bins are marked, those in the boundary bin are
//      ranked exactly by (score desc, index asc) among themselves;
//   3. forced blocks are marked too, and one warp writes the set bits in
//      ascending order.
// `surv` (shared, nb entries) holds the boundary bin; `sorted_copy`
// (optional, k_max entries) receives the output list too, padded with -1.
// NT >= 256; the caller synchronises before reading sorted_copy.
template <int NT, int MAXR>
struct BitTopkScratch {
  static constexpr int kWords = (NT * MAXR + 31) / 32;
  uint32_t hist[NT / 32][256];
  uint32_t bits[kWords];
  int wred[NT / 32][2];
  int warp_tot[NT / 32];
  int ctrl[4];   // boundary bin, count in better bins, boundary-list length
};

// Bin holding the need-th best entry of the per-warp histograms (bin 0 =
// best); *above = entries in better bins.  Zeroes the histograms for reuse.
// Two barriers.
template <int NT, int MAXR>
__device__ __forceinline__ int topk_boundary_bin(BitTopkScratch<NT, MAXR>& sm, int need, int tid, int* above) {
  constexpr int NWARP = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  int cnt = 0;
  if (tid < 256) {
#pragma unroll
    for (int w = 0; w < NWARP; ++w) cnt += static_cast<int>(sm.hist[w][tid]);
  }
  const int incl = warp_inclusive_scan(cnt);
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0u;
  int before = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) before += (w < warp) ? sm.warp_tot[w] : 0;
  const int run = before + incl - cnt;
  if (tid < 256 && run < need && run + cnt >= need) {
    sm.ctrl[0] = tid;
    sm.ctrl[1] = run;
  }
  __syncthreads();
  *above = sm.ctrl[1];
  return sm.ctrl[0];
}

template <int NT, int MAXR>
__device__ void select_topk_bits(const float (&v)[MAXR], int nb, int n_init, int n_local, int topk,
                                 bool includes_forced, int k_max, int32_t* out_idx, int32_t* out_n,
                                 BitTopkScratch<NT, MAXR>& sm, unsigned long long* surv, int tid,
                                 int32_t* sorted_copy = nullptr) {
  static_assert(NT >= 256, "one thread per histogram bin");
  constexpr int NWARP = NT / 32;
  constexpr int kShift = 17;
  constexpr int kWords = BitTopkScratch<NT, MAXR>::kWords;
  const int lane = tid & 31, warp = tid >> 5;
  const int c = nb - 1;
  const int n_first = min(n_init, nb);
  const int local_lo = max(n_first, c - n_local + 1);
  // 1. candidates, their count and the best leading bits; clear the scratch.
  bool cand[MAXR];
  uint32_t key[MAXR];
  int my_cand = 0;
  uint32_t my_top = 0;
#pragma unroll
  for (int x = 0; x < MAXR; ++x) {
    const int j = tid + NT * x;
    key[x] = float_to_ordered(v[x]);
    cand[x] = j < nb && j >= n_first && j < local_lo && v[x] > -INFINITY;
    if (cand[x]) {
      ++my_cand;
      my_top = max(my_top, key[x] >> kShift);
    }
  }
  for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0u;
  for (int w = tid; w < kWords; w += NT) sm.bits[w] = 0u;
  if (tid == 0) sm.ctrl[2] = 0;
  my_cand = __reduce_add_sync(0xffffffffu, my_cand);
  my_top = __reduce_max_sync(0xffffffffu, my_top);
  if (lane == 0) {
    sm.wred[warp][0] = my_cand;
    sm.wred[warp][1] = static_cast<int>(my_top);
  }
  __syncthreads();
  int n_cand = 0;
  uint32_t top = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    n_cand += sm.wred[w][0];
    top = max(top, static_cast<uint32_t>(sm.wred[w][1]));
  }
  const int n_forced = n_first + max(0, c - local_lo + 1);
  const int n_take = max(0, includes_forced ? topk - n_forced : topk);

  // 2. thresholds: candidates with d < d_sel are taken, d in [d_sel, d_bnd]
  //    (and, at the second level, coarse bin == bnd2) are ranked.
  //    d = distance of a score's leading bits from the best one.
  bool take_all = n_take >= n_cand, take_none = n_take == 0;
  int lvl = 0, bnd = 0, above = 0;
  if (!take_all && !take_none) {
#pragma unroll
    for (int x = 0; x < MAXR; ++x)
      if (cand[x]) atomicAdd(&sm.hist[warp][min(255u, top - (key[x] >> kShift))], 1u);
    __syncthreads();
    bnd = topk_boundary_bin(sm, n_take, tid, &above);
    lvl = 1;
    if (bnd == 255 && n_cand - above > NT) {
#pragma unroll
      for (int x = 0; x < MAXR; ++x) {
        const uint32_t d = top - (key[x] >> kShift);
        if (cand[x] && d >= 255u) atomicAdd(&sm.hist[warp][min(255u, (d - 255u) >> 4)], 1u);
      }
      __syncthreads();
      int above2 = 0;
      bnd = topk_boundary_bin(sm, n_take - above, tid, &above2);
      above += above2;
      lvl = 2;
    }
  }
  // 3. mark the taken candidates and the forced blocks; collect the boundary.
#pragma unroll
  for (int x = 0; x < MAXR; ++x) {
    if (!cand[x] || take_none) continue;
    const int j = tid + NT * x;
    const uint32_t d = top - (key[x] >> kShift);
    bool sel = take_all, tie = false;
    if (lvl == 1) {
      sel = static_cast<int>(min(255u, d)) < bnd;
      tie = static_cast<int>(min(255u, d)) == bnd;
    } else if (lvl == 2) {
      const int d2 = d < 255u ? -1 : static_cast<int>(min(255u, (d - 255u) >> 4));
      sel = d2 < bnd;
      tie = d2 == bnd;
    }
    if (sel) atomicOr(&sm.bits[j >> 5], 1u << (j & 31));
    if (tie) surv[atomicAdd(&sm.ctrl[2], 1)] = (static_cast<unsigned long long>(key[x]) << 32) |
                                              static_cast<uint32_t>(~j);
  }
  for (int j = tid; j < n_first; j += NT) atomicOr(&sm.bits[j >> 5], 1u << (j & 31));
  for (int j = local_lo + tid; j <= c; j += NT) atomicOr(&sm.bits[j >> 5], 1u << (j & 31));
  __syncthreads();
  // 4. the boundary entries that still fit, by exact rank among themselves.
  if (lvl > 0) {
    const int m = sm.ctrl[2];
    const int need = n_take - above;
    for (int x = tid; x < m; x += NT) {
      const unsigned long long me = surv[x];
      int rk = 0;
      for (int y = 0; y < m; ++y) rk += (surv[y] > me) ? 1 : 0;
      if (rk < need) {
        const int j = static_cast<int>(~static_cast<uint32_t>(me & 0xffffffffu));
        atomicOr(&sm.bits[j >> 5], 1u << (j & 31));
      }
    }
    __syncthreads();
  }
  // 5. ascending output from the bitmask (one warp).
  if (warp == 0) {
    constexpr int WPL = (kWords + 31) / 32;
    uint32_t w[WPL];
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      const int wi = lane * WPL + i;
      w[i] = wi < kWords ? sm.bits[wi] : 0u;
      cnt += __popc(w[i]);
    }
    const int incl = warp_inclusive_scan(cnt);
    const int total = min(__shfl_sync(0xffffffffu, incl, 31), k_max);
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < WPL; ++i) {
      uint32_t bw = w[i];
      while (bw) {
        const int j = (lane * WPL + i) * 32 + __ffs(bw) - 1;
        bw &= bw - 1u;
        if (pos < k_max) {
          out_idx[pos] = j;
          if (sorted_copy) sorted_copy[pos] = j;
        }
        ++pos;
      }
    }
    for (int x = total + lane; x < k_max; x += 32) {
      out_idx[x] = -1;
      if (sorted_copy) sorted_copy[x] = -1;
    }
    if (lane == 0) *out_n = total;
  }
}

// Same selection as select_topk_bits for scores held in shared memory
// (r[0..nb)), with every pass a short rolled loop: on this path the code
// fetched once per launch costs more than the arithmetic, so the routine is
// kept small.  `bits` needs (nb + 31) / 32 words of shared scratch.
template <int NT>
struct SmemTopkScratch {
  uint32_t hist[NT / 32][256];
  int wred[NT / 32][2];
  int warp_tot[NT / 32];
  int ctrl[4];   // boundary bin, count in better bins, boundary-list length
};

template <int NT>
__device__ __forceinline__ int smem_topk_boundary(SmemTopkScratch<NT>& sm, int need, int tid, int* above) {
  constexpr int NWARP = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  int cnt = 0;
  if (tid < 256)
    for (int w = 0; w < NWARP; ++w) cnt += static_cast<int>(sm.hist[w][tid]);
  const int incl = warp_inclusive_scan(cnt);
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0u;
  int before = 0;
  for (int w = 0; w < warp; ++w) before += sm.warp_tot[w];
  const int run = before + incl - cnt;
  if (tid < 256 && run < need && run + cnt >= need) {
    sm.ctrl[0] = tid;
    sm.ctrl[1] = run;
  }
  __syncthreads();
  *above = sm.ctrl[1];
  return sm.ctrl[0];
}

template <int NT>
__device__ void select_topk_smem(const float* r, int nb, int n_init, int n_local, int topk, bool includes_forced,
                                 int k_max, int32_t* out_idx, int32_t* out_n, SmemTopkScratch<NT>& sm,
                                 uint32_t* bits, unsigned long long* surv, int tid, int32_t* sorted_copy = nullptr) {
  static_assert(NT >= 256, "one thread per histogram bin");
  constexpr int NWARP = NT / 32;
  constexpr int kShift = 17;
  const int lane = tid & 31, warp = tid >> 5;
  const int c = nb - 1;
  const int n_first = min(n_init, nb);
  const int local_lo = max(n_first, c - n_local + 1);
  const int n_words = (nb + 31) / 32;
  auto is_cand = [&](int j, float x) { return j >= n_first && j < local_lo && x > -INFINITY; };
  int n_cand = 0;
  uint32_t top = 0;
  {
    // 1. candidates, their count and the best leading bits; clear the scratch.
    int my_cand = 0;
    uint32_t my_top = 0;
#pragma unroll 1
    for (int j = tid; j < nb; j += NT) {
      const float x = r[j];
      if (is_cand(j, x)) {
        ++my_cand;
        my_top = max(my_top, float_to_ordered(x) >> kShift);
      }
    }
    for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0u;
    for (int w = tid; w < n_words; w += NT) bits[w] = 0u;
    if (tid == 0) sm.ctrl[2] = 0;
    my_cand = __reduce_add_sync(0xffffffffu, my_cand);
    my_top = __reduce_max_sync(0xffffffffu, my_top);
    if (lane == 0) {
      sm.wred[warp][0] = my_cand;
      sm.wred[warp][1] = static_cast<int>(my_top);
    }
    __syncthreads();
    n_cand = 0;
    top = 0;
    for (int w = 0; w < NWARP; ++w) {
      n_cand += sm.wred[w][0];
      top = max(top, static_cast<uint32_t>(sm.wred[w][1]));
    }
  }
  const int n_forced = n_first + max(0, c - local_lo + 1);
  const int n_take = max(0, includes_forced ? topk - n_forced : topk);
  const bool take_all = n_take >= n_cand, take_none = n_take == 0;
  // 2. thresholds over d = distance of the leading bits from the best (see
  //    select_topk_bits): level 1 bins min(d, 255), level 2 splits bin 255.
  int lvl = 0, bnd = 0, above = 0;
  if (!take_all && !take_none) {
#pragma unroll 1
    for (int j = tid; j < nb; j += NT) {
      const float x = r[j];
      if (is_cand(j, x)) atomicAdd(&sm.hist[warp][min(255u, top - (float_to_ordered(x) >> kShift))], 1u);
    }
    __syncthreads();
    bnd = smem_topk_boundary(sm, n_take, tid, &above);
    lvl = 1;
    if (bnd == 255 && n_cand - above > NT) {
#pragma unroll 1
      for (int j = tid; j < nb; j += NT) {
        const float x = r[j];
        const uint32_t d = top - (float_to_ordered(x) >> kShift);
        if (is_cand(j, x) && d >= 255u) atomicAdd(&sm.hist[warp][min(255u, (d - 255u) >> 4)], 1u);
      }
      __syncthreads();
      int above2 = 0;
      bnd = smem_topk_boundary(sm, n_take - above, tid, &above2);
      above += above2;
      lvl = 2;
    }
  }
  // 3. mark the taken candidates and the forced blocks; collect the boundary.
  if (!take_none) {
    // A warp's 32 consecutive blocks are one bitmask word: one OR per word.
#pragma unroll 1
    for (int j0 = warp * 32; j0 < nb; j0 += NT) {
      const int j = j0 + lane;
      const float x = j < nb ? r[j] : -INFINITY;
      const bool cnd = j < nb && is_cand(j, x);
      const uint32_t key = float_to_ordered(x);
      const uint32_t d = top - (key >> kShift);
      int dd = static_cast<int>(min(255u, d));
      if (lvl == 2) dd = d < 255u ? -1 : static_cast<int>(min(255u, (d - 255u) >> 4));
      const uint32_t take = __ballot_sync(0xffffffffu, cnd && (lvl == 0 || dd < bnd));
      if (lane == 0 && take) atomicOr(&bits[j0 >> 5], take);
      if (cnd && lvl > 0 && dd == bnd)
        surv[atomicAdd(&sm.ctrl[2], 1)] = (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~j);
    }
  }
  for (int j = tid; j < n_first; j += NT) atomicOr(&bits[j >> 5], 1u << (j & 31));
  for (int j = local_lo + tid; j <= c; j += NT) atomicOr(&bits[j >> 5], 1u << (j & 31));
  __syncthreads();
  // 4. the boundary entries that still fit, by exact rank among themselves.
  if (lvl > 0) {
    const int m = sm.ctrl[2];
    const int need = n_take - above;
#pragma unroll 1
    for (int x = tid; x < m; x += NT) {
      const unsigned long long me = surv[x];
      int rk = 0;
#pragma unroll 1
      for (int y = 0; y < m; ++y) rk += (surv[y] > me) ? 1 : 0;
      if (rk < need) {
        const int j = static_cast<int>(~static_cast<uint32_t>(me & 0xffffffffu));
        atomicOr(&bits[j >> 5], 1u << (j & 31));
      }
    }
    __syncthreads();
  }
  // 5. ascending output from the bitmask: warp 0 turns the words' bit counts
  //    into output positions (over the boundary list, which is done), then
  //    every warp expands words, one lane per bit.
  int* wpos = reinterpret_cast<int*>(surv);
  if (warp == 0) {
    int base = 0;
#pragma unroll 1
    for (int w0 = 0; w0 < n_words; w0 += 32) {
      const int cnt = (w0 + lane < n_words) ? __popc(bits[w0 + lane]) : 0;
      const int incl = warp_inclusive_scan(cnt);
      if (w0 + lane < n_words) wpos[w0 + lane] = base + incl - cnt;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sm.ctrl[3] = base;
  }
  __syncthreads();
  const int total = min(sm.ctrl[3], k_max);
#pragma unroll 1
  for (int w = warp; w < n_words; w += NWARP) {
    const uint32_t bw = bits[w];
    if ((bw >> lane) & 1u) {
      const int pos = wpos[w] + __popc(bw & ((1u << lane) - 1u));
      if (pos < k_max) {
        out_idx[pos] = w * 32 + lane;
        if (sorted_copy) sorted_copy[pos] = w * 32 + lane;
      }
    }
  }
  for (int x = total + tid; x < k_max; x += NT) {
    out_idx[x] = -1;
    if (sorted_copy) sorted_copy[x] = -1;
  }
  if (tid == 0) *out_n = total;
}


}  // namespace infllmv2
