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
// Roles (192 threads):
//   warps 0-3  softmax: thread r owns row r (token r / 16, head r % 16);
//              reads S from TMEM, online softmax in fp32 base 2 with a lazy
//              rescale (the running max only moves when it grows by more
//              than 2^8, which keeps exp2(s - m) <= 256), writes P (bf16,
//              128-byte swizzled, K-major) to shared memory, rescales its O
//              row in TMEM when needed, and finally writes out / lse.
//   warp 4     TMA producer: Q tile once, then K and V tiles of each union
//              block into a 3-stage ring.
//   warp 5     MMA issuer (one thread): S_n = Q K_n^T (M 128, N 64, K 128)
//              into one of two TMEM S buffers, then O += P_{n-1} V_{n-1}
//              (M 128, N 128, K 64) with V as an MN-major operand.
// TMEM: columns [0,128) two S buffers, [128,256) the O accumulator.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace infllmv2 {

namespace {

constexpr int kTcTokens = 8;
constexpr int kTcStages = 3;
constexpr int kTcThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kLazyRescale = 8.0f;

struct TcParams {
  int B, Hkv, Lmax, nq, kmax, nbmax;
  float scale2;
  const int32_t* kv_lens;
  const int32_t* block_idx;
  const int32_t* n_sel;
  __nv_bfloat16* out;
  float* lse;
  uint32_t* status;
};

struct TcLayout {
  int q, kv, p, bars, slot, bits, ulist, umask, scan, total;
};

__host__ __device__ inline TcLayout tc_layout(int nbmax) {
  TcLayout l;
  l.q = 0;                                   // 2 boxes x 128 rows x 128 B
  l.kv = 32768;                              // stages x (K 16 KB + V 16 KB)
  l.p = l.kv + kTcStages * 32768;            // 2 x 16 KB
  l.bars = l.p + 2 * 16384;                  // 32 mbarriers max
  l.slot = l.bars + 32 * 8;
  l.bits = l.slot + 16;
  l.ulist = l.bits + ((nbmax + 15) & ~15);
  l.umask = l.ulist + nbmax * 4;
  l.scan = l.umask + ((nbmax + 15) & ~15);
  l.total = l.scan + 64;
  return l;
}

enum Bar { kQFull = 0, kKvFull = 1, kKvEmpty = kKvFull + kTcStages, kSFull = kKvEmpty + kTcStages,
           kSFree = kSFull + 2, kPFull = kSFree + 2, kODone = kPFull + 2, kNumBars = kODone + 1 };

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
  const int t0 = blockIdx.x * kTcTokens;
  const int n_act = min(kTcTokens, p.nq - t0);
  const int L = p.kv_lens[b];

  if (L < p.nq || L > p.Lmax) {
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
  for (int w = tid; w < (nb + 3) / 4; w += kTcThreads) bits32[w] = 0u;
  __syncthreads();
  for (int e = tid; e < n_act * p.kmax; e += kTcThreads) {
    const int tok = e / p.kmax, k = e % p.kmax;
    const size_t u = static_cast<size_t>(bh) * p.nq + t0 + tok;
    const int ns = min(p.n_sel[u], p.kmax);
    if (k < ns) {
      const int j = p.block_idx[u * p.kmax + k];
      const int c_tok = (L - p.nq + t0 + tok) / kBlock;
      if (j >= 0 && j <= c_tok) atomicOr(&bits32[j >> 2], (1u << tok) << ((j & 3) * 8));
    }
  }
  __syncthreads();
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
    if (tid == 0) scan[8] = tot;
  }

  if (tid == 0) {
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    mbar_init(&bars[kQFull], 1);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&bars[kKvFull + s], 1);
      mbar_init(&bars[kKvEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kSFull + s], 1);
      mbar_init(&bars[kSFree + s], 4);
      mbar_init(&bars[kPFull + s], 4);
    }
    mbar_init(&bars[kODone], 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int nu = scan[8];
  const uint32_t q_s = smem_u32(smem + lay.q);
  const uint32_t kv_s = smem_u32(smem + lay.kv);
  const uint32_t p_s = smem_u32(smem + lay.p);

  if (warp == 4) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0 && nu > 0) {
      mbar_arrive_expect_tx(&bars[kQFull], n_act * 4096);
      for (int tok = 0; tok < n_act; ++tok) {
        const int row = (b * p.nq + t0 + tok) * Hq + h * kGroup;
        tma_load_2d(smem + lay.q + tok * 2048, &q_map, 0, row, &bars[kQFull]);
        tma_load_2d(smem + lay.q + 16384 + tok * 2048, &q_map, 64, row, &bars[kQFull]);
      }
      for (int n = 0; n < nu; ++n) {
        const int st = n % kTcStages;
        if (n >= kTcStages && !mbar_wait(&bars[kKvEmpty + st], ((n / kTcStages) - 1) & 1, p.status)) break;
        const int row = bh * p.Lmax + ulist[n] * kBlock;
        uint8_t* dst = smem + lay.kv + st * 32768;
        mbar_arrive_expect_tx(&bars[kKvFull + st], 32768);
        tma_load_2d(dst, &k_map, 0, row, &bars[kKvFull + st]);
        tma_load_2d(dst + 8192, &k_map, 64, row, &bars[kKvFull + st]);
        tma_load_2d(dst + 16384, &v_map, 0, row, &bars[kKvFull + st]);
        tma_load_2d(dst + 24576, &v_map, 64, row, &bars[kKvFull + st]);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nu > 0) {
      constexpr uint32_t kIdS = tc::idesc_bf16(128, 64, 0, 0);
      constexpr uint32_t kIdO = tc::idesc_bf16(128, 128, 0, 1);
      bool ok = mbar_wait(&bars[kQFull], 0, p.status);
      for (int n = 0; n <= nu && ok; ++n) {
        if (n < nu) {
          const int st = n % kTcStages, sb = n & 1;
          ok = mbar_wait(&bars[kKvFull + st], (n / kTcStages) & 1, p.status);
          if (ok && n >= 2) ok = mbar_wait(&bars[kSFree + sb], ((n >> 1) - 1) & 1, p.status);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t kb = kv_s + st * 32768;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = tc::sdesc_sw128(q_s + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(kb + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024);
            tc::mma_ss(tmem + sb * 64, ad, bd, kIdS, k > 0 ? 1u : 0u);
          }
          tc::commit(&bars[kSFull + sb]);
        }
        if (n >= 1) {
          const int m = n - 1, pb = m & 1, st = m % kTcStages;
          if (!mbar_wait(&bars[kPFull + pb], (m >> 1) & 1, p.status)) break;
          tc::fence_after_sync();
          const uint32_t vb = kv_s + st * 32768 + 16384;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = tc::sdesc_sw128(p_s + pb * 16384 + k * 32, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(vb + k * 2048, 8192, 1024);
            tc::mma_ss(tmem + 128, ad, bd, kIdO, (m > 0 || k > 0) ? 1u : 0u);
          }
          tc::commit(&bars[kODone]);
          tc::commit(&bars[kKvEmpty + st]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = tid;              // TMEM lane == MMA row
    const int tok = r >> 4;
    const bool active = tok < n_act;
    const int i_row = L - p.nq + t0 + tok;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    uint8_t* prow_base = smem + lay.p + (r >> 3) * 1024 + (r & 7) * 128;
    for (int n = 0; n < nu; ++n) {
      const int sb = n & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[kSFull + sb], (n >> 1) & 1, p.status));
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t s[64];
      tc::ld32(lane_addr + sb * 64, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
      tc::ld32(lane_addr + sb * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kSFree + sb]);

      const bool sel = active && ((umask[n] >> tok) & 1);
      const int key0 = ulist[n] * kBlock;
      if (key0 + kBlock > L) {
        // The block holds cache rows past kv_len: clear their V rows so a
        // zero probability never multiplies a non-finite value.
        const int st = n % kTcStages;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[kKvFull + st], (n / kTcStages) & 1, p.status));
        if (!ok) break;
        uint8_t* vt = smem + lay.kv + st * 32768 + 16384;
        const int r0 = L - key0;
        for (int e = tid; e < (kBlock - r0) * 16; e += 128) {
          const int row = r0 + (e >> 4), q16 = e & 15;
          *reinterpret_cast<uint4*>(vt + (q16 >> 3) * 8192 + row * 128 + (q16 & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      const int nvalid = sel ? min(kBlock, i_row - key0 + 1) : 0;   // keys key0 .. key0+nvalid-1
      float mx = -INFINITY;
#pragma unroll
      for (int x = 0; x < 64; ++x)
        if (x < nvalid) mx = fmaxf(mx, __uint_as_float(s[x]) * p.scale2);
      bool need = false;
      float alpha = 1.f;
      float m_use = m_run;
      if (sel) {
        if (m_run == -INFINITY) {
          m_use = mx;
        } else if (mx > m_run + kLazyRescale) {
          need = true;
          alpha = fast_exp2(m_run - mx);
          m_use = mx;
        }
      }
      if (n >= 1) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars[kODone], (n - 1) & 1, p.status));
        if (!ok) break;
        tc::fence_after_sync();
      }
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::ld32(lane_addr + 128 + c * 32, o);
          tc::wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tc::st32(lane_addr + 128 + c * 32, o);
        }
        tc::wait_st();
      }
      l_run *= alpha;
      m_run = m_use;
      // P row (bf16) into the swizzled K-major tile of this block's buffer.
      uint8_t* prow = prow_base + (n & 1) * 16384;
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int x0 = c * 8 + 2 * e;
          const float p0 = (x0 < nvalid) ? fast_exp2(__uint_as_float(s[x0]) * p.scale2 - m_run) : 0.f;
          const float p1 = (x0 + 1 < nvalid) ? fast_exp2(__uint_as_float(s[x0 + 1]) * p.scale2 - m_run) : 0.f;
          lsum += p0 + p1;
          w[e] = pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l_run += lsum;
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPFull + (n & 1)]);
    }
    // ---- epilogue: O / l -> bf16 out, lse ----
    if (nu > 0 && ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars[kODone], (nu - 1) & 1, p.status));
    tc::fence_after_sync();
    const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
    __nv_bfloat16* orow = p.out + ((static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)) * kHeadDim;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      if (nu > 0) {
        tc::ld32(lane_addr + 128 + c * 32, o);
        tc::wait_ld();
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] = 0u;
      }
      if (active) {
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * inv, __uint_as_float(o[2 * x + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int x = 0; x < 4; ++x) dst[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
      }
    }
    if (active && p.lse) {
      p.lse[(static_cast<size_t>(b) * p.nq + t0 + tok) * Hq + h * kGroup + (r & 15)] =
          (l_run > 0.f) ? (m_run + fast_log2(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

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
  const int smem = tc_layout(s.nbmax).total + 1024;
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.nq + kTcTokens - 1) / kTcTokens, s.Hkv, s.B);
  attn_tc_kernel<<<grid, kTcThreads, smem, st>>>(q_map, k_map, v_map, p);
  return cudaGetLastError();
}

}  // namespace infllmv2
