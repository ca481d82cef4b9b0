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

// Top-k over scores held in registers: thread tid holds the scores of blocks
// j = tid + NT x (x < MAXR) in v[x].  Same selection rule and output as
// select_topk.  One 256-bin histogram of the scores' leading bits (sign,
// exponent, 6 mantissa bits, counted down from the best score) locates the
// bin holding the n_take-th best score; candidates at or above it are
// ranked exactly by (score desc, index asc).  Every step works on registers
// with a handful of CTA barriers.  `surv` (shared, nb entries) takes the
// survivors, so many-way exact ties are handled too; `sel` (shared, k_max
// entries) collects the chosen blocks; `sorted_copy` (optional, k_max
// entries) receives the ascending output list too, padded with -1.  NT >= 256.
template <int NT>
struct RegTopkScratch {
  uint32_t hist[NT / 32][256];
  int wred[NT / 32][2];
  int warp_tot[NT / 32];
  int ctrl[4];
};

template <int NT, int MAXR>
__device__ void select_topk_regs(const float (&v)[MAXR], int nb, int n_init, int n_local, int topk,
                                 bool includes_forced, int k_max, int32_t* out_idx, int32_t* out_n,
                                 RegTopkScratch<NT>& sm, unsigned long long* surv_buf, int* sel_buf,
                                 int tid, int32_t* sorted_copy = nullptr) {
  static_assert(NT >= 256, "one thread per histogram bin");
  constexpr int NWARP = NT / 32;
  constexpr int kShift = 17;
  const int lane = tid & 31, warp = tid >> 5;
  const int c = nb - 1;
  // 1. candidates, their count and best leading bits.
  bool cand[MAXR];
  int my_cand = 0;
  uint32_t my_top = 0;
#pragma unroll
  for (int x = 0; x < MAXR; ++x) {
    const int j = tid + NT * x;
    cand[x] = j < nb && j >= n_init && j <= c - n_local && v[x] > -INFINITY;
    if (cand[x]) {
      ++my_cand;
      my_top = max(my_top, float_to_ordered(v[x]) >> kShift);
    }
  }
  for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0u;
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
  const int n_first = min(n_init, nb);
  const int n_forced = n_first + max(0, c - max(n_first, c - n_local + 1) + 1);
  const int n_take = max(0, includes_forced ? topk - n_forced : topk);
  // 2. boundary bin (255 = every candidate survives, -1 = none is taken).
  int bnd = n_take > 0 ? 255 : -1;
  if (n_take > 0 && n_cand > n_take) {
#pragma unroll
    for (int x = 0; x < MAXR; ++x)
      if (cand[x]) atomicAdd(&sm.hist[warp][min(255u, top - (float_to_ordered(v[x]) >> kShift))], 1u);
    __syncthreads();
    int cnt = 0;
    for (int b = tid; b < 256; b += NT) {
#pragma unroll
      for (int w = 0; w < NWARP; ++w) cnt += static_cast<int>(sm.hist[w][b]);
    }
    // tid < 256 holds bin tid (NT >= 256); inclusive scan in bin order.
    const int incl = warp_inclusive_scan(cnt);
    if (lane == 31) sm.warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) before += (w < warp) ? sm.warp_tot[w] : 0;
    const int run = before + incl - cnt;
    if (tid < 256 && run < n_take && run + cnt >= n_take) sm.ctrl[0] = tid;
    __syncthreads();
    bnd = sm.ctrl[0];
  }
  // 3. survivors (candidates at or above the boundary bin) into shared memory.
  bool surv[MAXR];
  int my_surv = 0;
#pragma unroll
  for (int x = 0; x < MAXR; ++x) {
    surv[x] = cand[x] && static_cast<int>(min(255u, top - (float_to_ordered(v[x]) >> kShift))) <= bnd;
    my_surv += surv[x] ? 1 : 0;
  }
  const int incl = warp_inclusive_scan(my_surv);
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  int pos = incl - my_surv, n_surv = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    pos += (w < warp) ? sm.warp_tot[w] : 0;
    n_surv += sm.warp_tot[w];
  }
#pragma unroll
  for (int x = 0; x < MAXR; ++x)
    if (surv[x]) surv_buf[pos++] = (static_cast<unsigned long long>(float_to_ordered(v[x])) << 32) |
                                   static_cast<uint32_t>(~(tid + NT * x));
  if (tid == 0) {   // forced blocks first, ascending
    int n = 0;
    for (int j = 0; j < n_first; ++j) sel_buf[n++] = j;
    for (int j = max(n_first, c - n_local + 1); j <= c; ++j) sel_buf[n++] = j;
  }
  __syncthreads();
  // 4. exact rank among survivors; the best n_take follow the forced blocks.
  for (int x = tid; x < n_surv; x += NT) {
    const unsigned long long me = surv_buf[x];
    int rk = 0, y = 0;
    for (; y + 4 <= n_surv; y += 4)
      rk += (surv_buf[y] > me) + (surv_buf[y + 1] > me) + (surv_buf[y + 2] > me) + (surv_buf[y + 3] > me);
    for (; y < n_surv; ++y) rk += (surv_buf[y] > me) ? 1 : 0;
    if (rk < n_take) sel_buf[n_forced + rk] = static_cast<int>(~static_cast<uint32_t>(me & 0xffffffffu));
  }
  __syncthreads();
  // 5. ascending output.
  const int n_total = min(k_max, n_forced + min(n_take, n_surv));
  for (int x = tid; x < n_total; x += NT) {
    const int val = sel_buf[x];
    int p = 0;
    for (int y = 0; y < n_total; ++y) p += (sel_buf[y] < val) ? 1 : 0;
    out_idx[p] = val;
    if (sorted_copy) sorted_copy[p] = val;
  }
  for (int x = n_total + tid; x < k_max; x += NT) {
    out_idx[x] = -1;
    if (sorted_copy) sorted_copy[x] = -1;
  }
  if (tid == 0) *out_n = n_total;
}

// Same contract as select_topk for a whole CTA (NT threads, NT % 32 == 0),
// built for few barriers and no contended atomics: one 256-bin histogram of
// the scores' leading bits (sign, exponent, 6 mantissa bits, counted down
// from the best score; per-warp private copies) finds the bin holding the
// n_take-th best score; every candidate at or above that bin survives, and
// each survivor's exact rank among the survivors, by (score desc, index
// asc), decides whether it is taken.  Falls back to the radix select when
// the survivors exceed NT (many exactly tied or very close scores).
template <int NT>
struct FastTopkScratch {
  uint32_t hist[NT / 32][256];  // per-warp histograms
  unsigned long long surv[NT];  // survivors: (ordered key << 32) | ~index
  int ctrl[8];
  int wcnt[NT / 32][3];
  TopkScratch<NT> radix;
};

template <int NT>
__device__ void select_topk_fast(const float* r, uint8_t* flag, int nb, int n_init, int n_local, int topk,
                                 bool includes_forced, int k_max, int32_t* out_idx, int32_t* out_n,
                                 FastTopkScratch<NT>& sm, int tid) {
  constexpr int NWARP = NT / 32;
  constexpr int kShift = 17;   // 1 sign + 8 exponent + 6 mantissa bits
  const int lane = tid & 31, warp = tid >> 5;
  const int c = nb - 1;
  const int local_lo = c - n_local + 1;
  const int per = (nb + NT - 1) / NT;
  const int lo = tid * per;
  const int hi = min(nb, lo + per);
  // 1. flags (contiguous range per thread), counts, best leading bits.
  int my_cand = 0, my_forced = 0;
  uint32_t my_top = 0;
  for (int j = lo; j < hi; ++j) {
    const bool forced = (j < n_init) || (j >= local_lo);
    const bool cand = !forced && (r[j] > -INFINITY);
    flag[j] = forced ? 2 : (cand ? 1 : 0);
    my_cand += cand ? 1 : 0;
    my_forced += forced ? 1 : 0;
    if (cand) my_top = max(my_top, float_to_ordered(r[j]) >> kShift);
  }
  for (int b = lane; b < 256; b += 32) sm.hist[warp][b] = 0;
  my_cand = __reduce_add_sync(0xffffffffu, my_cand);
  my_forced = __reduce_add_sync(0xffffffffu, my_forced);
  my_top = __reduce_max_sync(0xffffffffu, my_top);
  if (lane == 0) {
    sm.wcnt[warp][0] = my_cand;
    sm.wcnt[warp][1] = my_forced;
    sm.wcnt[warp][2] = static_cast<int>(my_top);
  }
  __syncthreads();
  int n_cand = 0, n_forced = 0;
  uint32_t top = 0;
#pragma unroll
  for (int w = 0; w < NWARP; ++w) {
    n_cand += sm.wcnt[w][0];
    n_forced += sm.wcnt[w][1];
    top = max(top, static_cast<uint32_t>(sm.wcnt[w][2]));
  }
  int n_take = includes_forced ? topk - n_forced : topk;
  if (n_take < 0) n_take = 0;

  bool use_radix = false;
  if (n_take > 0 && n_cand <= n_take) {
    for (int j = lo; j < hi; ++j)
      if (flag[j] == 1) flag[j] = 3;
  } else if (n_take > 0) {
    // 2. per-warp histograms of bins (0 = the best bin).
    for (int j = lo; j < hi; ++j)
      if (flag[j] == 1) atomicAdd(&sm.hist[warp][min(255u, top - (float_to_ordered(r[j]) >> kShift))], 1u);
    __syncthreads();
    // 3. boundary bin: the first whose cumulative count reaches n_take.
    if (warp == 0) {
      int cnt[8], tot = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        int v = 0;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) v += static_cast<int>(sm.hist[w][8 * lane + k]);
        cnt[k] = v;
        tot += v;
      }
      int run = warp_inclusive_scan(tot) - tot;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (run < n_take && run + cnt[k] >= n_take) {
          sm.ctrl[3] = 8 * lane + k;      // boundary bin
          sm.ctrl[4] = run + cnt[k];      // survivors
        }
        run += cnt[k];
      }
    }
    __syncthreads();
    const int bnd = sm.ctrl[3];
    const int n_surv = sm.ctrl[4];
    if (n_surv > NT) {
      use_radix = true;
    } else {
      // 4. survivors into shared memory, positions from a prefix count.
      int my_keep = 0;
      for (int j = lo; j < hi; ++j)
        my_keep += (flag[j] == 1 && static_cast<int>(min(255u, top - (float_to_ordered(r[j]) >> kShift))) <= bnd) ? 1 : 0;
      int tot_keep;
      int pos = group_exclusive_scan<NT, false>(my_keep, tot_keep, sm.radix, tid);
      for (int j = lo; j < hi; ++j) {
        if (flag[j] != 1) continue;
        const uint32_t key = float_to_ordered(r[j]);
        if (static_cast<int>(min(255u, top - (key >> kShift))) <= bnd)
          sm.surv[pos++] = (static_cast<unsigned long long>(key) << 32) | static_cast<uint32_t>(~j);
      }
      __syncthreads();
      // 5. exact rank among the survivors; the best n_take are taken.
      if (tid < n_surv) {
        const unsigned long long me = sm.surv[tid];
        int rank = 0;
        int x = 0;
        for (; x + 4 <= n_surv; x += 4) {
          rank += (sm.surv[x] > me) + (sm.surv[x + 1] > me) + (sm.surv[x + 2] > me) + (sm.surv[x + 3] > me);
        }
        for (; x < n_surv; ++x) rank += (sm.surv[x] > me) ? 1 : 0;
        if (rank < n_take) flag[static_cast<int>(~static_cast<uint32_t>(me & 0xffffffffu))] = 3;
      }
    }
  }
  if (use_radix) {   // uniform: every thread saw the same n_surv
    __syncthreads();
    select_topk<NT, false>(r, flag, nb, n_init, n_local, topk, includes_forced, k_max, out_idx, out_n, sm.radix,
                           tid);
    return;
  }
  __syncthreads();
  // 6. ascending output of forced + taken blocks.
  int my_sel = 0;
  for (int j = lo; j < hi; ++j) my_sel += (flag[j] >= 2) ? 1 : 0;
  int total;
  int pos = group_exclusive_scan<NT, false>(my_sel, total, sm.radix, tid);
  for (int j = lo; j < hi; ++j) {
    if (flag[j] >= 2) {
      if (pos < k_max) out_idx[pos] = j;
      ++pos;
    }
  }
  for (int p = total + tid; p < k_max; p += NT) out_idx[p] = -1;
  if (tid == 0) *out_n = min(total, k_max);
}

}  // namespace infllmv2
