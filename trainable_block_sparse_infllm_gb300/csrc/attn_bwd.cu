// Backward of stage 3 of InfLLM v2: gradients of the block-sparse attention
// output with respect to q, K and V, with the block selection held fixed.
//
// [InfLLM v2 > Training-time considerations]: top-k passes no gradient; the
// keys (and through their means the semantic kernels) are trained by the
// gradient of the stage-2 attention, which is what this file computes.  With
// s = scale q.k over a query's attended keys, P = softmax(s), O = P V and an
// upstream gradient dO:
//     D = rowsum(dO * O),  dP = dO V^T,  dS = P * (dP - D),
//     dq = scale dS K,  dK = scale dS^T q,  dV = P^T dO,
// with P recomputed from the forward's log-sum-exp (P = exp(s - lse)).
//
// Three pieces:
//   * An inverse index: for each (b, h_kv, range of kBkRange query tokens,
//     block j) the tokens of the range whose selection holds j (count, scan,
//     fill), cut into work items of at most kBkChunk tokens.  Items come out
//     ordered by token range, so the CTAs resident at one time share one
//     range's q and dO rows in L2 rather than gathering rows from the whole
//     sequence.
//   * bwd_dq_kernel, query-centric on the warp-level tensor cores: one warp
//     per (b, h_kv, t) unit (its 16 heads are the 16 MMA rows, [InfLLM v2 >
//     Query group sharing]) walks the unit's selected blocks in 16-key quarters
//     (K and V TMA-staged in a per-warp ring) and accumulates dq in
//     registers; it also writes D for the second kernel.
//   * bwd_dkdv_kernel, key-centric on tcgen05/TMEM: one CTA per work item
//     holds block j's K and V in shared memory and takes the item's tokens
//     eight at a time (8 tokens x 16 heads = 128 rows, every row's token
//     selected j, so no work is spent on unselected pairs):
//         S = Q K^T, dP = dO V^T            (M 128 rows, N 64 keys, K 128)
//         P, dS per row                     (4 warps, one row per thread)
//         dV^T += dO^T P, dK^T += Q^T dS    (M 128 dims, N 128 = 64 keys of hi
//                                           then lo parts, K 128 rows)
//     with dV^T and dK^T accumulated in TMEM over the item and added to the
//     fp32 dK / dV rows at the end.
// P and dS enter every bf16 product as hi + lo parts (16 significant bits).
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace infllmv2 {

namespace {

constexpr int kBkChunk = 256;    // tokens per dK/dV work item
constexpr int kBkRange = 2048;   // query tokens per range of the inverse index (a multiple of kIdxTokens)
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  int B, Hkv, Lmax, nq, kmax, nbmax, nr, nl;   // nr: token ranges per (b, h_kv); nl = B Hkv nr nbmax
  float scale;    // attn_scale
  float scale2;   // attn_scale * log2(e)
  const int32_t* kv_lens;
  const int32_t* block_idx;
  const int32_t* n_sel;
  const __nv_bfloat16* q;
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* dq;
  float* dk;
  float* dv;
  float* dsum;      // D, [B, nq, Hq]
  int32_t* cnt;     // [nl] tokens per (b, h, range, j) list
  int32_t* off;     // [nl + 1] first entry of each list
  int32_t* choff;   // [nl + 1] first work item of each list
  int32_t* cursor;  // [nl] fill position
  int32_t* items;   // list of each work item
  int32_t* tok;     // token index of each entry
  uint32_t* status;
};

// ------------------------------------------------------------ inverse index

// Per-CTA histogram of the selected blocks of kIdxTokens consecutive tokens
// of one (b, h_kv), flushed with one global atomic per block; `fill` = true
// reserves a range per block and writes the token indices.
constexpr int kIdxTokens = 64;
static_assert(kBkRange % kIdxTokens == 0, "an index CTA's tokens share one range");
constexpr int kIdxThreads = 256;

template <bool kFill>
__global__ void __launch_bounds__(kIdxThreads) bwd_index_kernel(BwdParams p, bool smem_hist) {
  extern __shared__ int32_t hist[];
  const int bh = blockIdx.y, b = bh / p.Hkv;
  const int t0 = blockIdx.x * kIdxTokens;
  const int n_tok = min(kIdxTokens, p.nq - t0);
  const int L = p.kv_lens[b];
  if (L < p.nq || L > p.Lmax) return;   // such units attend nothing
  const int32_t l0 = (bh * p.nr + t0 / kBkRange) * p.nbmax;
  const int c_last = (L - p.nq + t0 + n_tok - 1) / kBlock;
  if (smem_hist) {
    for (int j = threadIdx.x; j <= c_last; j += kIdxThreads) hist[j] = 0;
    __syncthreads();
  }
  // pass 1: counts (smem) or direct global counts / positions
  for (int e = threadIdx.x; e < n_tok * p.kmax; e += kIdxThreads) {
    const int tt = e / p.kmax, n = e % p.kmax;
    const size_t u = static_cast<size_t>(bh) * p.nq + t0 + tt;
    if (n >= min(p.n_sel[u], p.kmax)) continue;
    const int j = p.block_idx[u * p.kmax + n];
    const int c = (L - p.nq + t0 + tt) / kBlock;
    if (j < 0 || j > c) continue;
    if (smem_hist) {
      atomicAdd(&hist[j], 1);
    } else if (!kFill) {
      atomicAdd(&p.cnt[l0 + j], 1);
    } else {
      p.tok[atomicAdd(&p.cursor[l0 + j], 1)] = t0 + tt;
    }
  }
  if (!smem_hist) return;
  __syncthreads();
  for (int j = threadIdx.x; j <= c_last; j += kIdxThreads) {
    const int v = hist[j];
    if (v == 0) continue;
    if (!kFill)
      atomicAdd(&p.cnt[l0 + j], v);
    else
      hist[j] = atomicAdd(&p.cursor[l0 + j], v);   // this CTA's range starts here
  }
  if (!kFill) return;
  __syncthreads();
  for (int e = threadIdx.x; e < n_tok * p.kmax; e += kIdxThreads) {
    const int tt = e / p.kmax, n = e % p.kmax;
    const size_t u = static_cast<size_t>(bh) * p.nq + t0 + tt;
    if (n >= min(p.n_sel[u], p.kmax)) continue;
    const int j = p.block_idx[u * p.kmax + n];
    const int c = (L - p.nq + t0 + tt) / kBlock;
    if (j < 0 || j > c) continue;
    p.tok[atomicAdd(&hist[j], 1)] = t0 + tt;
  }
}

// One CTA: exclusive scans of the list sizes (entries) and of their work
// item counts, the fill cursors, and the list of each work item.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads) bwd_scan_kernel(BwdParams p) {
  __shared__ int ws_c[32], ws_h[32];
  __shared__ int carry_c, carry_h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry_c = carry_h = 0;
  __syncthreads();
  for (int base = 0; base < p.nl; base += kScanThreads) {
    const int l = base + tid;
    const int c = l < p.nl ? p.cnt[l] : 0;
    const int hc = (c + kBkChunk - 1) / kBkChunk;
    const int ic = warp_inclusive_scan(c), ih = warp_inclusive_scan(hc);
    if (lane == 31) {
      ws_c[warp] = ic;
      ws_h[warp] = ih;
    }
    __syncthreads();
    int pc = 0, ph = 0, tc_ = 0, th = 0;
    for (int w = 0; w < kScanThreads / 32; ++w) {
      if (w < warp) {
        pc += ws_c[w];
        ph += ws_h[w];
      }
      tc_ += ws_c[w];
      th += ws_h[w];
    }
    const int oc = carry_c + pc + ic - c, oh = carry_h + ph + ih - hc;
    if (l < p.nl) {
      p.off[l] = oc;
      p.cursor[l] = oc;
      p.choff[l] = oh;
      for (int k = 0; k < hc; ++k) p.items[oh + k] = l;
    }
    __syncthreads();
    if (tid == 0) {
      carry_c += tc_;
      carry_h += th;
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.off[p.nl] = carry_c;
    p.choff[p.nl] = carry_h;
  }
}

// -------------------------------------------------------------------- dq --

constexpr int kBqWarps = 8;
constexpr int kBqStages = 3;            // 16-key quarters of a block in flight per warp
constexpr int kBqRows = 16;
constexpr int kBqStageBytes = 8192;     // K then V, 16 rows x 128 bf16 each
constexpr int kBqSmem = 1024 + kBqWarps * kBqStages * kBqStageBytes + kBqWarps * kBqStages * 8;

// First valid quarter position (4 n + part) at or after `pos`: entry n must
// name a block in [0, c]; a quarter must start at or before i.
__device__ __forceinline__ int next_part(const int32_t* sel, int ns, int c, int i, int pos) {
  while (pos < 4 * ns) {
    const int n = pos >> 2;
    const int j = sel[n];
    if (j < 0 || j > c || j * kBlock + (pos & 3) * kBqRows > i) {
      pos = 4 * (n + 1);
      continue;
    }
    return pos;
  }
  return 4 * ns;
}

__global__ void __launch_bounds__(kBqWarps * 32, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap k_map16, const __grid_constant__ CUtensorMap v_map16,
                  BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBqWarps * kBqStages * kBqStageBytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  if (tid == 0) {
    prefetch_tensormap(&k_map16);
    prefetch_tensormap(&v_map16);
    for (int s = 0; s < kBqWarps * kBqStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const long long units = static_cast<long long>(p.B) * p.Hkv * p.nq;
  const long long u = static_cast<long long>(blockIdx.x) * kBqWarps + warp;
  if (u >= units) return;
  const int bh = static_cast<int>(u / p.nq), t = static_cast<int>(u % p.nq);
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const size_t orow = (static_cast<size_t>(b) * p.nq + t) * Hq + static_cast<size_t>(h) * kGroup;
  float* dq_rows = p.dq + orow * kHeadDim;
  const int L = p.kv_lens[b];
  if (L < p.nq || L > p.Lmax) {
    for (int e = lane; e < kGroup * kHeadDim; e += 32) dq_rows[e] = 0.f;
    if (lane < kGroup) p.dsum[orow + lane] = 0.f;
    if (lane == 0 && t == 0) atomicOr(p.status, kStatusBadKvLen);
    return;
  }
  const int i = L - p.nq + t;
  const int c = i / kBlock;
  const int ns = min(p.n_sel[u], p.kmax);
  const int32_t* sel = p.block_idx + u * p.kmax;
  check_selection_row(sel, p.n_sel[u], p.kmax, c, p.status, lane);
  uint8_t* ring = smem + warp * kBqStages * kBqStageBytes;
  uint64_t* full = bars + warp * kBqStages;
  const size_t kv_row0 = static_cast<size_t>(bh) * p.Lmax;

  auto issue = [&](int pos, int st) {
    const int row = static_cast<int>(kv_row0 + static_cast<size_t>(sel[pos >> 2]) * kBlock + (pos & 3) * kBqRows);
    if (!kv_row_ok(kv_row0 + static_cast<size_t>(sel[pos >> 2]) * kBlock, kv_row0, p.Lmax, p.status)) return;
    uint8_t* dst = ring + st * kBqStageBytes;
    mbar_arrive_expect_tx(&full[st], kBqStageBytes);
    tma_load_2d(dst, &k_map16, 0, row, &full[st]);
    tma_load_2d(dst + 2048, &k_map16, 64, row, &full[st]);
    tma_load_2d(dst + 4096, &v_map16, 0, row, &full[st]);
    tma_load_2d(dst + 6144, &v_map16, 64, row, &full[st]);
  };
  // Prologue: the first kBqStages quarters.
  int pi = next_part(sel, ns, c, i, 0);
  for (int s = 0; s < kBqStages && pi < 4 * ns; ++s) {
    if (lane == 0) issue(pi, s);
    pi = next_part(sel, ns, c, i, pi + 1);
  }

  // q, dO and O rows of the unit straight from global memory into A
  // fragments (row g / g + 8 = head, 16 columns per k-step).
  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(p.q + orow * kHeadDim);
  const uint32_t* do32 = reinterpret_cast<const uint32_t*>(p.dout + orow * kHeadDim);
  const uint32_t* o32 = reinterpret_cast<const uint32_t*>(p.out + orow * kHeadDim);
  uint32_t qa[8][4], da[8][4];
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c0 = (g * kHeadDim + 16 * ks + 2 * tq) >> 1;
    const int c1 = ((g + 8) * kHeadDim + 16 * ks + 2 * tq) >> 1;
    qa[ks][0] = q32[c0];
    qa[ks][1] = q32[c1];
    qa[ks][2] = q32[c0 + 4];
    qa[ks][3] = q32[c1 + 4];
    da[ks][0] = do32[c0];
    da[ks][1] = do32[c1];
    da[ks][2] = do32[c0 + 4];
    da[ks][3] = do32[c1 + 4];
    const uint32_t oa[4] = {o32[c0], o32[c1], o32[c0 + 4], o32[c1 + 4]};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 dv2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&da[ks][x]));
      const float2 ov2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&oa[x]));
      const float dd = fmaf(dv2.x, ov2.x, dv2.y * ov2.y);
      if (x & 1)
        d1 += dd;
      else
        d0 += dd;
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    d0 += __shfl_xor_sync(0xffffffffu, d0, o);
    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
  }
  if (tq == 0) {
    p.dsum[orow + g] = d0;
    p.dsum[orow + g + 8] = d1;
  }
  const float lse0 = p.lse[orow + g], lse1 = p.lse[orow + g + 8];
  const bool ok0 = lse0 > -INFINITY, ok1 = lse1 > -INFINITY;
  const float m0 = ok0 ? lse0 * kLog2e : 0.f, m1 = ok1 ? lse1 * kLog2e : 0.f;

  float acc[16][4];
#pragma unroll
  for (int x = 0; x < 16; ++x) acc[x][0] = acc[x][1] = acc[x][2] = acc[x][3] = 0.f;

  bool ok = true;
  int pc = next_part(sel, ns, c, i, 0);
  for (int n = 0; pc < 4 * ns; ++n) {
    const int st = n % kBqStages;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (n / kBqStages) & 1, p.status));
    if (!ok) break;
    uint8_t* stage = ring + st * kBqStageBytes;
    const uint32_t k_b = smem_u32(stage), v_b = k_b + 4096;
    const int key0 = sel[pc >> 2] * kBlock + (pc & 3) * kBqRows;
    if (key0 + kBqRows - 1 > i) {
      // Keys past i: zero their K rows (dS is 0 there; the cache rows past
      // kv_len may hold non-finite values).
      const int r0 = i - key0 + 1;
      for (int e = lane; e < (kBqRows - r0) * 16; e += 32) {
        const int row = r0 + (e >> 4), q16 = e & 15;
        *reinterpret_cast<uint4*>(stage + (q16 >> 3) * 2048 + row * 128 + (q16 & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // S = q K^T and dP = dO V^T for 16 keys (2 n-tiles of 8); the four
    // accumulators advance together over the 8 k-steps.
    float s[2][4], dp[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      dp[nt][0] = dp[nt][1] = dp[nt][2] = dp[nt][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t kb[2][4], vb[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint32_t o = swz128_offset(nt * 8 + (lane & 7), 4 * kk + (lane >> 3), kBqRows);
        ldmatrix_x4(kb[nt], k_b + o);
        ldmatrix_x4(vb[nt], v_b + o);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_bf16_16816(s[nt], qa[2 * kk], kb[nt][0], kb[nt][1]);
        mma_bf16_16816(dp[nt], da[2 * kk], vb[nt][0], vb[nt][1]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_bf16_16816(s[nt], qa[2 * kk + 1], kb[nt][2], kb[nt][3]);
        mma_bf16_16816(dp[nt], da[2 * kk + 1], vb[nt][2], vb[nt][3]);
      }
    }
    // dS = P (dP - D) with P = 2^(s scale2 - lse2); 0 past i.
    uint32_t ah[4], al[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int x = key0 + nt * 8 + 2 * tq;
      const bool v0 = x <= i, v1 = x + 1 <= i;
      const float p0 = (v0 && ok0) ? fast_exp2(fmaf(s[nt][0], p.scale2, -m0)) : 0.f;
      const float p1 = (v1 && ok0) ? fast_exp2(fmaf(s[nt][1], p.scale2, -m0)) : 0.f;
      const float p2 = (v0 && ok1) ? fast_exp2(fmaf(s[nt][2], p.scale2, -m1)) : 0.f;
      const float p3 = (v1 && ok1) ? fast_exp2(fmaf(s[nt][3], p.scale2, -m1)) : 0.f;
      const float e0 = p0 != 0.f ? p0 * (dp[nt][0] - d0) : 0.f;
      const float e1 = p1 != 0.f ? p1 * (dp[nt][1] - d0) : 0.f;
      const float e2 = p2 != 0.f ? p2 * (dp[nt][2] - d1) : 0.f;
      const float e3 = p3 != 0.f ? p3 * (dp[nt][3] - d1) : 0.f;
      const __nv_bfloat162 h01 = __floats2bfloat162_rn(e0, e1);
      const __nv_bfloat162 h23 = __floats2bfloat162_rn(e2, e3);
      const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
      ah[nt * 2 + 0] = *reinterpret_cast<const uint32_t*>(&h01);
      ah[nt * 2 + 1] = *reinterpret_cast<const uint32_t*>(&h23);
      al[nt * 2 + 0] = pack_bf16x2(e0 - f01.x, e1 - f01.y);
      al[nt * 2 + 1] = pack_bf16x2(e2 - f23.x, e3 - f23.y);
    }
    // dq += dS K: B = K (16 keys x 128 dims) through ldmatrix.trans.
#pragma unroll
    for (int np = 0; np < 8; ++np) {
      uint32_t kb[4];
      ldmatrix_x4_trans(kb, k_b + swz128_offset((lane & 7) + ((lane >> 3) & 1) * 8, 2 * np + (lane >> 4), kBqRows));
      mma_bf16_16816(acc[2 * np], ah, kb[0], kb[1]);
      mma_bf16_16816(acc[2 * np + 1], ah, kb[2], kb[3]);
      mma_bf16_16816(acc[2 * np], al, kb[0], kb[1]);
      mma_bf16_16816(acc[2 * np + 1], al, kb[2], kb[3]);
    }
    pc = next_part(sel, ns, c, i, pc + 1);
    if (pi < 4 * ns) {
      // The stage is free again (its reads are done); order any zeroed rows
      // before the TMA refill.
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) issue(pi, st);
      pi = next_part(sel, ns, c, i, pi + 1);
    }
  }
  __syncwarp();
#pragma unroll
  for (int x = 0; x < 16; ++x) {
    const int d0c = x * 8 + 2 * tq;
    *reinterpret_cast<float2*>(dq_rows + g * kHeadDim + d0c) = make_float2(acc[x][0] * p.scale, acc[x][1] * p.scale);
    *reinterpret_cast<float2*>(dq_rows + (g + 8) * kHeadDim + d0c) =
        make_float2(acc[x][2] * p.scale, acc[x][3] * p.scale);
  }
}

// ----------------------------------------------------------------- dK, dV --

constexpr int kBkTokens = 8;                 // tokens per 128-row tile
constexpr int kBkStages = 2;                 // q / dO tile stages
constexpr int kBkTileBytes = 65536;          // q 32 KB + dO 32 KB (two 64-column boxes each)
constexpr int kBkThreads = 192;              // warps 0-3 rows, 4 MMA, 5 TMA
constexpr int kBkMmaWarp = 4, kBkTmaWarp = 5;
constexpr uint32_t kBkTmemCols = 512;
// TMEM: two S buffers, two dP buffers (64 columns each), dV^T and dK^T
// (128 columns each: the products of the hi parts, then of the lo parts).
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

// Shared memory (offsets from the 1024-aligned base).
constexpr int kOffKV = 0;                                   // K block 16 KB, V block 16 KB
constexpr int kOffTile = 32768;                             // kBkStages x 64 KB
constexpr int kOffPS = kOffTile + kBkStages * kBkTileBytes; // P hi, P lo, dS hi, dS lo (16 KB each)
constexpr int kOffBars = kOffPS + 65536;
constexpr int kOffSlot = kOffBars + 16 * 8;
constexpr int kOffTok = kOffSlot + 16;
constexpr int kBkSmem = 1024 + kOffTok + kBkChunk * 4;
static_assert(kBkSmem <= 227 * 1024, "dK/dV kernel shared memory");

enum BkBar { kBKv = 0, kBTFull = 1, kBTEmpty = kBTFull + kBkStages, kBSFull = kBTEmpty + kBkStages,
             kBSFree = kBSFull + 2, kBPFull = kBSFree + 2, kBPFree = kBPFull + 1, kBAcc = kBPFree + 1,
             kBNumBars = kBAcc + 1 };
static_assert(kBNumBars <= 16, "barrier area holds 16");

__global__ void __launch_bounds__(kBkThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap do_map,
                    const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                    BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffSlot);
  int32_t* toks = reinterpret_cast<int32_t*>(smem + kOffTok);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int item = blockIdx.x;
  if (item >= p.choff[p.nl]) return;   // grid is an upper bound on the items
  const int l = p.items[item];
  const int e0 = p.off[l] + (item - p.choff[l]) * kBkChunk;
  const int ntok = min(kBkChunk, p.off[l + 1] - e0);
  const int bh = l / (p.nr * p.nbmax), j = l % p.nbmax;
  const int b = bh / p.Hkv, h = bh % p.Hkv;
  const int Hq = p.Hkv * kGroup;
  const int L = p.kv_lens[b];
  const int ntile = (ntok + kBkTokens - 1) / kBkTokens;
  for (int e = tid; e < ntok; e += kBkThreads) toks[e] = p.tok[e0 + e];

  if (tid == 0) {
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&do_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    mbar_init(&bars[kBKv], 1);
    for (int s = 0; s < kBkStages; ++s) {
      mbar_init(&bars[kBTFull + s], 1);
      mbar_init(&bars[kBTEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBSFull + s], 1);
      mbar_init(&bars[kBSFree + s], 4);
    }
    mbar_init(&bars[kBPFull], 4);
    mbar_init(&bars[kBPFree], 1);
    mbar_init(&bars[kBAcc], 1);
    fence_barrier_init();
  }
  if (warp == kBkMmaWarp) {
    tc::tmem_alloc(tmem_slot, kBkTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t base_s = smem_u32(smem);

  if (warp == kBkTmaWarp) {
    // ----------------------------------------------------------- producer
    if (lane == 0 && kv_row_ok(static_cast<size_t>(bh) * p.Lmax + static_cast<size_t>(j) * kBlock,
                               static_cast<size_t>(bh) * p.Lmax, p.Lmax, p.status)) {
      const int row = bh * p.Lmax + j * kBlock;
      mbar_arrive_expect_tx(&bars[kBKv], 32768);
      tma_load_2d(smem + kOffKV, &k_map, 0, row, &bars[kBKv]);
      tma_load_2d(smem + kOffKV + 8192, &k_map, 64, row, &bars[kBKv]);
      tma_load_2d(smem + kOffKV + 16384, &v_map, 0, row, &bars[kBKv]);
      tma_load_2d(smem + kOffKV + 24576, &v_map, 64, row, &bars[kBKv]);
    }
    for (int n = 0; n < ntile; ++n) {
      const int st = n % kBkStages;
      bool ok = true;
      if (n >= kBkStages) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kBTEmpty + st], ((n / kBkStages) - 1) & 1, p.status));
      if (!ok) break;
      uint8_t* tile = smem + kOffTile + st * kBkTileBytes;
      const int nt_tok = min(kBkTokens, ntok - n * kBkTokens);
      if (nt_tok < kBkTokens) {
        // Rows of absent tokens: zeros, so that the dV / dK products see
        // zero operands there.
        const int per = (kBkTokens - nt_tok) * 128;   // 16-byte chunks per 16 KB box
        for (int e = lane; e < 4 * per; e += 32) {
          const int part = e / per, rem = e % per;
          *reinterpret_cast<uint4*>(tile + part * 16384 + nt_tok * 2048 + rem * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      // One box per lane (token tt = lane / 4; q / dO, column half), after
      // lane 0 has set the transaction count.
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBTFull + st], nt_tok * 8192);
      __syncwarp();
      if (lane < nt_tok * 4) {
        const int tt = lane >> 2, part = lane & 3;
        const int row = (b * p.nq + toks[n * kBkTokens + tt]) * Hq + h * kGroup;
        tma_load_2d(tile + part * 16384 + tt * 2048, (part & 2) ? &do_map : &q_map, (part & 1) * 64, row,
                    &bars[kBTFull + st]);
      }
      __syncwarp();
    }
  } else if (warp == kBkMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(128, 64, 0, 0);   // rows x keys, both K-major
      constexpr uint32_t kIdG = tc::idesc_bf16(128, 128, 1, 1);   // dims x (hi | lo keys), both MN-major
      const uint64_t k_desc = tc::sdesc_sw128(base_s + kOffKV, 16, 1024);
      const uint64_t v_desc = tc::sdesc_sw128(base_s + kOffKV + 16384, 16, 1024);
      const uint32_t ps = base_s + kOffPS;
      bool ok = mbar_wait(&bars[kBKv], 0, p.status);
      // Two in-order streams, issued as their inputs arrive: S and dP of tile
      // n_s (its q / dO stage loaded, its S / dP buffer read out by the rows
      // two tiles back) and the dV / dK products of tile n_g (its P and dS
      // written).  Neither waits behind the other: the dV / dK products free
      // a stage for the next load, S feeds the row warps.
      int n_s = 0, n_g = 0;
      uint32_t idle = 0;
      while (ok && n_g < ntile) {
        bool progressed = false;
        if (n_s < ntile && mbar_try_wait(&bars[kBTFull + n_s % kBkStages], (n_s / kBkStages) & 1) &&
            (n_s < 2 || mbar_try_wait(&bars[kBSFree + (n_s & 1)], ((n_s >> 1) - 1) & 1))) {
          const int st = n_s % kBkStages, sb = n_s & 1;
          tc::fence_after_sync();
          const uint32_t tile = base_s + kOffTile + st * kBkTileBytes;
          const uint64_t q_desc = tc::sdesc_sw128(tile, 16, 1024);
          const uint64_t o_desc = tc::sdesc_sw128(tile + 32768, 16, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ta = static_cast<uint64_t>(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
            const uint64_t tb = static_cast<uint64_t>(((k >> 2) * 8192 + (k & 3) * 32) >> 4);
            tc::mma_ss(tmem + kColS + sb * 64, q_desc + ta, k_desc + tb, kIdS, k > 0 ? 1u : 0u);
            tc::mma_ss(tmem + kColDP + sb * 64, o_desc + ta, v_desc + tb, kIdS, k > 0 ? 1u : 0u);
          }
          tc::commit(&bars[kBSFull + sb]);
          ++n_s;
          progressed = true;
        }
        if (n_g < n_s && mbar_try_wait(&bars[kBPFull], n_g & 1)) {
          const int m = n_g, st = m % kBkStages;
          tc::fence_after_sync();
          const uint32_t tile = base_s + kOffTile + st * kBkTileBytes;
          // dO^T and q^T: M = 128 dims in two 64-column boxes (16 KB apart),
          // K = 128 rows; P and dS: K = rows, N = 64 keys.
          const uint64_t qt_desc = tc::sdesc_sw128(tile, 16384, 1024);
          const uint64_t ot_desc = tc::sdesc_sw128(tile + 32768, 16384, 1024);
          const uint64_t ph_desc = tc::sdesc_sw128(ps, 16384, 1024);
          const uint64_t sh_desc = tc::sdesc_sw128(ps + 32768, 16384, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t kd = static_cast<uint64_t>((k * 2048) >> 4);
            const uint32_t first = (m > 0 || k > 0) ? 1u : 0u;
            tc::mma_ss(tmem + kColDV, ot_desc + kd, ph_desc + kd, kIdG, first);
            tc::mma_ss(tmem + kColDK, qt_desc + kd, sh_desc + kd, kIdG, first);
          }
          tc::commit(&bars[kBTEmpty + st]);
          tc::commit(&bars[kBPFree]);
          if (m == ntile - 1) tc::commit(&bars[kBAcc]);
          ++n_g;
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
    // ------------------------------------------------- rows: P and dS
    // Warp w reads TMEM lanes 32 w .. 32 w + 31: row r = token slot r / 16,
    // head r % 16 of the tile.
    const int r = warp * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    uint8_t* ps = smem + kOffPS;
    const int key0 = j * kBlock;
    bool ok = true;
    // The row's lse and D, loaded one tile ahead.
    auto row_inputs = [&](int n, float& lse, float& dsum, int& t) {
      const int slot = n * kBkTokens + (r >> 4);
      lse = -INFINITY;
      dsum = 0.f;
      t = 0;
      if (n < ntile && slot < ntok) {
        t = toks[slot];
        const size_t grow = (static_cast<size_t>(b) * p.nq + t) * Hq + h * kGroup + (r & 15);
        lse = p.lse[grow];
        dsum = p.dsum[grow];
      }
    };
    float lse_n, dsum_n;
    int t_n;
    row_inputs(0, lse_n, dsum_n, t_n);
    for (int n = 0; n < ntile; ++n) {
      const int sb = n & 1;
      float m2 = 0.f;
      const float dsum = dsum_n;
      int nv = 0;
      if (lse_n > -INFINITY) {
        m2 = lse_n * kLog2e;
        nv = min(kBlock, L - p.nq + t_n - key0 + 1);   // keys key0 .. key0 + nv - 1 are <= i
      }
      row_inputs(n + 1, lse_n, dsum_n, t_n);
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kBSFull + sb], (n >> 1) & 1, p.status));
      tc::fence_after_sync();
      uint32_t sv[64], dpv[64];
      tc::ld32(lane_addr + kColS + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tc::ld32(lane_addr + kColS + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tc::ld32(lane_addr + kColDP + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(&dpv[0]));
      tc::ld32(lane_addr + kColDP + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dpv[32]));
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBSFree + sb]);
      // P = 2^(s scale2 - lse2) and dS = P (dP - D) for the row's valid keys,
      // as bf16 hi / lo pairs (two keys per 32-bit word).
      uint32_t phi[32], plo[32], shi[32], slo[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const float p0 = (2 * x < nv) ? fast_exp2(fmaf(__uint_as_float(sv[2 * x]), p.scale2, -m2)) : 0.f;
        const float p1 = (2 * x + 1 < nv) ? fast_exp2(fmaf(__uint_as_float(sv[2 * x + 1]), p.scale2, -m2)) : 0.f;
        const float g0 = (2 * x < nv) ? p0 * (__uint_as_float(dpv[2 * x]) - dsum) : 0.f;
        const float g1 = (2 * x + 1 < nv) ? p1 * (__uint_as_float(dpv[2 * x + 1]) - dsum) : 0.f;
        const __nv_bfloat162 hp = __floats2bfloat162_rn(p0, p1);
        const __nv_bfloat162 hs = __floats2bfloat162_rn(g0, g1);
        const float2 fp = __bfloat1622float2(hp), fs = __bfloat1622float2(hs);
        phi[x] = *reinterpret_cast<const uint32_t*>(&hp);
        shi[x] = *reinterpret_cast<const uint32_t*>(&hs);
        plo[x] = pack_bf16x2(p0 - fp.x, p1 - fp.y);
        slo[x] = pack_bf16x2(g0 - fs.x, g1 - fs.y);
      }
      // The P / dS tiles are read by the previous tile's dV / dK products.
      if (n >= 1 && ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kBPFree], (n - 1) & 1, p.status));
      // Row r of each 128-byte-swizzled tile: 16-byte chunk q at (q ^ (r % 8)).
#pragma unroll
      for (int qc = 0; qc < 8; ++qc) {
        const int off = r * 128 + ((qc ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(ps + off) = make_uint4(phi[4 * qc], phi[4 * qc + 1], phi[4 * qc + 2], phi[4 * qc + 3]);
        *reinterpret_cast<uint4*>(ps + 16384 + off) =
            make_uint4(plo[4 * qc], plo[4 * qc + 1], plo[4 * qc + 2], plo[4 * qc + 3]);
        *reinterpret_cast<uint4*>(ps + 32768 + off) =
            make_uint4(shi[4 * qc], shi[4 * qc + 1], shi[4 * qc + 2], shi[4 * qc + 3]);
        *reinterpret_cast<uint4*>(ps + 49152 + off) =
            make_uint4(slo[4 * qc], slo[4 * qc + 1], slo[4 * qc + 2], slo[4 * qc + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBPFull]);
    }
    // ---- epilogue: TMEM lane d holds dV^T / dK^T row d (64 keys) ----
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kBAcc], 0, p.status));
    tc::fence_after_sync();
    if (ok) {
      const int d = warp * 32 + lane;
      const int nkeys = min(kBlock, p.Lmax - key0);
      float* dvp = p.dv + (static_cast<size_t>(bh) * p.Lmax + key0) * kHeadDim + d;
      float* dkp = p.dk + (static_cast<size_t>(bh) * p.Lmax + key0) * kHeadDim + d;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {   // dV then dK, 32 keys at a time: hi part + lo part
        const uint32_t col = (cc < 2 ? kColDV : kColDK) + (cc & 1) * 32;
        uint32_t gh[32], gl[32];
        tc::ld32(lane_addr + col, gh);
        tc::ld32(lane_addr + col + 64, gl);
        tc::wait_ld();
        float* dst = cc < 2 ? dvp : dkp;
        const float f = cc < 2 ? 1.f : p.scale;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int key = (cc & 1) * 32 + x;
          if (key < nkeys)
            atomicAdd(dst + static_cast<size_t>(key) * kHeadDim,
                      (__uint_as_float(gh[x]) + __uint_as_float(gl[x])) * f);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kBkMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kBkTmemCols);
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct BwdWs {
  size_t dsum, cnt, off, choff, cursor, items, tok, total;
  long long max_items;
};

BwdWs bwd_ws_layout(const Shape& s) {
  BwdWs w{};
  const long long nl = static_cast<long long>(s.B) * s.Hkv * ((s.nq + kBkRange - 1) / kBkRange) * s.nbmax;
  const long long entries = static_cast<long long>(s.B) * s.Hkv * s.nq * s.kmax;
  w.max_items = entries / kBkChunk + nl + 1;
  size_t o = 0;
  w.dsum = o;
  o = align256(o + static_cast<size_t>(s.B) * s.nq * s.Hkv * kGroup * 4);
  w.cnt = o;
  o = align256(o + nl * 4);
  w.off = o;
  o = align256(o + (nl + 1) * 4);
  w.choff = o;
  o = align256(o + (nl + 1) * 4);
  w.cursor = o;
  o = align256(o + nl * 4);
  w.items = o;
  o = align256(o + w.max_items * 4);
  w.tok = o;
  o = align256(o + entries * 4);
  w.total = o;
  return w;
}

}  // namespace

size_t attn_bwd_workspace_bytes(const Shape& s) { return bwd_ws_layout(s).total; }

bool attn_bwd_supported(const Shape& s) {
  const long long nl = static_cast<long long>(s.B) * s.Hkv * ((s.nq + kBkRange - 1) / kBkRange) * s.nbmax;
  const long long entries = static_cast<long long>(s.B) * s.Hkv * s.nq * s.kmax;
  return nl < (1LL << 30) && entries < (1LL << 31) - 1 && bwd_ws_layout(s).max_items < (1LL << 31) - 1;
}

cudaError_t launch_attn_bwd(const Shape& s, const CUtensorMap& q_map, const CUtensorMap& do_map,
                            const CUtensorMap& k_map, const CUtensorMap& v_map, const CUtensorMap& k_map16,
                            const CUtensorMap& v_map16, const void* q, const int32_t* kv_lens,
                            const int32_t* block_idx, const int32_t* n_sel, const void* out, const float* lse,
                            const void* dout, float* dq, float* dk, float* dv, void* ws, uint32_t* status,
                            cudaStream_t st) {
  const BwdWs w = bwd_ws_layout(s);
  uint8_t* wb = static_cast<uint8_t*>(ws);
  BwdParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.kmax = s.kmax;
  p.nbmax = s.nbmax;
  p.nr = (s.nq + kBkRange - 1) / kBkRange;
  p.nl = s.B * s.Hkv * p.nr * s.nbmax;
  p.scale = s.attn_scale;
  p.scale2 = s.attn_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dsum = reinterpret_cast<float*>(wb + w.dsum);
  p.cnt = reinterpret_cast<int32_t*>(wb + w.cnt);
  p.off = reinterpret_cast<int32_t*>(wb + w.off);
  p.choff = reinterpret_cast<int32_t*>(wb + w.choff);
  p.cursor = reinterpret_cast<int32_t*>(wb + w.cursor);
  p.items = reinterpret_cast<int32_t*>(wb + w.items);
  p.tok = reinterpret_cast<int32_t*>(wb + w.tok);
  p.status = status;

  const size_t kv_bytes = static_cast<size_t>(s.B) * s.Hkv * s.Lmax * kHeadDim * sizeof(float);
  cudaError_t e = cudaMemsetAsync(p.cnt, 0, static_cast<size_t>(p.nl) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dk, 0, kv_bytes, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, kv_bytes, st);
  if (e != cudaSuccess) return e;

  // Histogram in shared memory when the blocks of a cache fit (64 KB).
  const bool smem_hist = s.nbmax <= 16384;
  const size_t hist_bytes = smem_hist ? static_cast<size_t>(s.nbmax) * 4 : 0;
  if (hist_bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(bwd_index_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(hist_bytes));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(bwd_index_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(hist_bytes));
    if (e != cudaSuccess) return e;
  }
  const dim3 igrid((s.nq + kIdxTokens - 1) / kIdxTokens, s.B * s.Hkv);
  bwd_index_kernel<false><<<igrid, kIdxThreads, hist_bytes, st>>>(p, smem_hist);
  bwd_scan_kernel<<<1, kScanThreads, 0, st>>>(p);
  bwd_index_kernel<true><<<igrid, kIdxThreads, hist_bytes, st>>>(p, smem_hist);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBqSmem);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(s.B) * s.Hkv * s.nq;
  bwd_dq_kernel<<<static_cast<unsigned>((units + kBqWarps - 1) / kBqWarps), kBqWarps * 32, kBqSmem, st>>>(
      k_map16, v_map16, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBkSmem);
  if (e != cudaSuccess) return e;
  bwd_dkdv_kernel<<<static_cast<unsigned>(w.max_items), kBkThreads, kBkSmem, st>>>(q_map, do_map, k_map, v_map, p);
  return cudaGetLastError();
}

}  // namespace infllmv2
