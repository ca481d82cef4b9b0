// Device helpers shared by the InfLLM v2 kernels: shapes, status word,
// mbarrier + TMA (cp.async.bulk / cp.async.bulk.tensor) wrappers, warp-level
// bf16 tensor-core MMA (m16n8k16) and ldmatrix, and small block primitives.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace infllmv2 {

// Supported shape (the recommended InfLLM v2 configuration).
constexpr int kHeadDim = 128;  // d
constexpr int kGroup = 16;     // query heads per KV head
constexpr int kBlock = 64;     // m, KV block size
constexpr int kKernel = 32;    // p, semantic kernel size
constexpr int kStride = 16;    // s, semantic kernel stride

constexpr uint32_t kStatusBadKvLen = 0x1u;
constexpr uint32_t kStatusTimeout = 0x2u;
constexpr uint32_t kStatusBounds = 0x4u;

// Bounded spin on an mbarrier: ~2^22 polls, each of which may suspend the
// thread for a hardware-chosen time, is far above any legitimate wait here.
// The checked build (INFLLMV2_CHECKED), which its tests drive into expired
// waits on purpose, gives up after 2^16 polls, still far above any
// legitimate wait of its small test cases.
#ifdef INFLLMV2_CHECKED
constexpr uint32_t kSpinLimit = 1u << 16;
#else
constexpr uint32_t kSpinLimit = 1u << 22;
#endif

// `ok`, and in the checked build a false `ok` also records
// INFLLMV2_DEVICE_BOUNDS: every index that comes from the caller (a
// block_idx entry, a selection count) and every K/V tile row built from one
// passes through here before use.  The product build skips the same
// accesses silently.
__device__ __forceinline__ bool bounds_ok(bool ok, uint32_t* status) {
#ifdef INFLLMV2_CHECKED
  if (!ok) atomicOr(status, kStatusBounds);
#else
  (void)status;
#endif
  return ok;
}

// One warp: the checked build verifies a caller-given selection row (its
// count within [0, kmax], every counted entry within [0, c]); the product
// build compiles this to nothing and skips bad entries where they are read.
__device__ __forceinline__ void check_selection_row(const int32_t* row, int n_sel, int kmax, int c,
                                                    uint32_t* status, int lane) {
#ifdef INFLLMV2_CHECKED
  bool ok = n_sel >= 0 && n_sel <= kmax;
  const int n = min(max(n_sel, 0), kmax);
  for (int k = lane; k < n; k += 32) ok = ok && row[k] >= 0 && row[k] <= c;
  if (!__all_sync(0xffffffffu, ok) && lane == 0) atomicOr(status, kStatusBounds);
#else
  (void)row; (void)n_sel; (void)kmax; (void)c; (void)status; (void)lane;
#endif
}

// A K/V tile starting at `row` starts inside its (b, h) plane [plane0,
// plane0 + Lmax).  (The tile of a cache's last, partial block runs past the
// plane; its rows beyond kv_len are masked.)
__device__ __forceinline__ bool kv_row_ok(size_t row, size_t plane0, int Lmax, uint32_t* status) {
  return bounds_ok(row >= plane0 && row < plane0 + static_cast<size_t>(Lmax), status);
}

__host__ __device__ __forceinline__ int n_complete_kernels(int L) {
  return L >= kKernel ? (L - kKernel) / kStride + 1 : 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Round a dynamic shared-memory pointer up to 1024 bytes (the period of the
// 128-byte TMA swizzle); launches reserve 1024 bytes of slack for this.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's ordinary global accesses with its TMA (async proxy)
// accesses: after ordinary stores that another thread's TMA will read (with
// a release / acquire between them), and before a TMA load of such data.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with acquire at cluster scope: for a phase completed by other
// CTAs' remote stores (st.async), whose complete_tx releases at that scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t* status) {
#pragma unroll 1
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
  }
  atomicOr(status, kStatusTimeout);
  return false;
}

// Returns false (and flags the status word) if the phase never completed.
// The spin loops are never unrolled: each wait is inlined at many call
// sites, and an unrolled copy costs kilobytes of instruction fetch at each.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
#pragma unroll 1
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  atomicOr(status, kStatusTimeout);
  return false;
}

// ------------------------------------------------------------------- TMA ----

// 2D tiled tensor load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Bring a 2D tile into L2 ahead of its shared-memory load (no completion
// signal, no shared memory used).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------- tensor-core MMA ----

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Byte offset of 16-byte chunk `chunk` (0..15) of row `row` in a tile of
// 128-column bf16 rows stored as two TMA boxes of 64 columns, each written
// with the 128-byte swizzle (chunk index XOR row % 8 inside a 128-byte row).
// `rows` is the tile height (the first box holds columns 0..63 of all rows).
__device__ __forceinline__ uint32_t swz128_offset(int row, int chunk, int rows) {
  const int box = chunk >> 3;
  const int c = (chunk & 7) ^ (row & 7);
  return static_cast<uint32_t>(box * rows * 128 + row * 128 + (c << 4));
}

// --------------------------------------------- clusters / distributed smem --

// The SM this thread runs on (a slot index for scratch that only one CTA per
// SM uses at a time), and the bound on SM identifiers (which need not be
// contiguous, so it may exceed the number of SMs).
__device__ __forceinline__ uint32_t sm_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t sm_id_bound() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nsmid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier with release/acquire semantics (orders shared and
// global memory accesses of all threads of the cluster).  Every thread of
// every CTA of the cluster must execute it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Split cluster barrier: every thread of every CTA arrives, then waits for
// the phase to complete.  arrive.release orders this thread's earlier
// (including remote) shared-memory writes before the waiters' acquire;
// the relaxed form orders nothing and only marks the CTA as running.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

// Remote loads carry no memory clobber: the data they read is fixed by a
// preceding cluster_sync (which is itself a compiler barrier), and leaving
// them unordered lets independent loads overlap their round trips.
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ unsigned long long ld_dsmem_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ float2 ld_dsmem_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// Remote stores: fire-and-forget; a following cluster_sync (release/acquire)
// makes them visible to the owning CTA.
__device__ __forceinline__ void st_dsmem_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem_f32x2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

__device__ __forceinline__ void st_dsmem_f32x4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory into another CTA's, counted as complete_tx
// on the destination's mbarrier.  dst and bar are shared::cluster addresses
// (dsmem_addr); the source must not change until the copy has landed.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(smem_u32(src)), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void st_async_u32x4(uint32_t addr, uint4 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
               : "memory");
}

// Remote store whose arrival is counted on the destination CTA's mbarrier
// (8 bytes of complete_tx): a receiver that waits on that mbarrier sees the
// value, with no cluster barrier (threads busy in other roles need not join).
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float2 v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(v.x), "f"(v.y), "r"(remote_bar)
               : "memory");
}

// ------------------------------------------- programmatic dependent launch --

// Block until the preceding kernel in the stream has completed and its memory
// is visible (no-op when the launch carries no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to start launching its CTAs.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- math -----

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_to_ordered(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Inclusive prefix sum over a warp.
__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

}  // namespace infllmv2
