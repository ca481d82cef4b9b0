// Internal launch interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Host-side only; every pointer is a device pointer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace infllmv2 {

struct Shape {
  int B, Hkv, Lmax, nq;
  int ncmax;   // complete kernels of a full cache
  int nbmax;   // ceil(Lmax / 64)
  int kmax;    // width of a block_idx row
  int topk, n_init, n_local, inc_forced;
  float score_scale2;  // score_scale * log2(e)
  float attn_scale2;   // attn_scale * log2(e)
  float attn_scale;
};

// SMs of the current device (cached per device).
int device_sm_count();

// ---- stage 1 ---------------------------------------------------------------
cudaError_t launch_compress(const Shape& s, const void* k, const int32_t* kv_lens, int kbegin,
                            int kend, void* kc, uint32_t* status, cudaStream_t st);

// Coarse kernels (means of sc-key windows) for the LSE approximation.
cudaError_t launch_coarse(const Shape& s, const void* k, const int32_t* kv_lens, int sc, void* kcc,
                          uint32_t* status, cudaStream_t st);

// ---- stage 2 ---------------------------------------------------------------
constexpr int kSelDecodeMaxNq = 16;   // n_q at or below this uses the decode path

size_t select_workspace_bytes(const Shape& s);
// The prefill selection (n_q > 16) keeps 8 tokens' block scores in shared
// memory: at most 5115 blocks (327360 tokens) of cache capacity.
bool select_tc_supported(const Shape& s);
bool select_tc_onchip(const Shape& s);   // the prefill path's block scores fit in shared memory
bool select_supported(const Shape& s);
cudaError_t launch_select(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                          const void* q, const int32_t* kv_lens, int32_t* block_idx,
                          int32_t* n_sel, float* block_scores, void* ws, uint32_t* status,
                          cudaStream_t st);
// Prefill path (n_q > 16) with the per-head LSE taken over coarse kernels of
// sc keys (kcc_map over [B, Hkv, 2, Lmax / sc, 128]).
cudaError_t launch_select_coarse(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map, int sc,
                                 const void* q, const int32_t* kv_lens, int32_t* block_idx,
                                 int32_t* n_sel, float* block_scores, uint32_t* status, cudaStream_t st);

// ---- stage 3 ---------------------------------------------------------------
size_t attn_workspace_bytes(const Shape& s, bool prefill);
cudaError_t launch_attn(const Shape& s, bool prefill, const CUtensorMap& q_map,
                        const CUtensorMap& k_map, const CUtensorMap& v_map,
                        const int32_t* kv_lens, const int32_t* block_idx, const int32_t* n_sel,
                        void* out, float* lse, void* ws, uint32_t* status, cudaStream_t st);

// Prefill on tcgen05/TMEM: 8 query tokens x 16 heads per 128-row MMA tile;
// with few tiles (speculative verification, short chunks) each tile's union
// of blocks is split over a cluster.
bool attn_tc_fits(const Shape& s);
int attn_tc_cluster_size(const Shape& s);
cudaError_t launch_attn_tc(const Shape& s, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, const int32_t* kv_lens, const int32_t* block_idx,
                           const int32_t* n_sel, void* out, float* lse, uint32_t* status,
                           cudaStream_t st);

// ---- cache append of a decode step (rows kv_lens[b] - n_q .. kv_lens[b] - 1)
cudaError_t launch_append(const Shape& s, const void* k_new, const void* v_new, const int32_t* kv_lens, void* k_cache,
                          void* v_cache, const void* q_src, void* q_dst, uint32_t* status, cudaStream_t st);

// ---- fused decode step (n_q = 1): newest kernel + selection + attention ----
// Cluster size of the single-launch form on the current device (16 or 8),
// or 0 when it does not apply to this shape.
int decode_step_cluster_size(const Shape& s);
// The cache append fused into the decode step: the newest token's q, k and
// v (device or page-locked host memory) and the caches k and v go into.
struct DsAppend {
  const void* q;
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
};
// append: null when the caller has appended the token (q_map then covers q).
cudaError_t launch_decode_step(const Shape& s, int cluster, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                               const CUtensorMap& k_map, const CUtensorMap& v_map, const void* k,
                               const int32_t* kv_lens, void* kc, int32_t* block_idx, int32_t* n_sel, void* out,
                               float* lse, const DsAppend* append, uint32_t* status, uint32_t test_flags,
                               cudaStream_t st);

// ---- backward of stage 3 (fixed selection) --------------------------------
size_t attn_bwd_workspace_bytes(const Shape& s);
bool attn_bwd_supported(const Shape& s);
// q_map / do_map: 16-row boxes over q / dout; k_map / v_map: 64-row boxes;
// k_map16 / v_map16: 16-row boxes over the caches.
cudaError_t launch_attn_bwd(const Shape& s, const CUtensorMap& q_map, const CUtensorMap& do_map,
                            const CUtensorMap& k_map, const CUtensorMap& v_map, const CUtensorMap& k_map16,
                            const CUtensorMap& v_map16, const void* q, const int32_t* kv_lens,
                            const int32_t* block_idx, const int32_t* n_sel, const void* out, const float* lse,
                            const void* dout, float* dq, float* dk, float* dv, void* ws, uint32_t* status,
                            cudaStream_t st);

}  // namespace infllmv2
