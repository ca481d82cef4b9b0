// Stage 2 of InfLLM v2: block relevance and top-k block selection -- the
// entry point, its scratch accounting, and the prefill path (n_q > 16).
//
// [InfLLM v2 > Semantic kernels, eqs. r_kernel, r_block], [> Query group
// sharing, eq. r_group], [> Top-K implementation and the LSE bottleneck] and
// [> Initial and local tokens always selected].  For one query token of one
// GQA group (16 heads):
//   z[h, j] = score_scale * q_h . Mean_j            (visible kernels j)
//   g[j]    = (1/16) sum_h exp(z[h, j] - lse_h)     (exact two-pass LSE)
//   r[blk]  = max_j g[j] over kernels meeting the block (j in 4 blk - 1 .. 4 blk + 3)
//   top-k over r with forced initial/local blocks.
//
// Paths, same result:
//  * decode (n_q = 1), and up to 16 tokens where nothing below fits:
//    select_decode.cu, one thread-block cluster per (b, h_kv) group.
//  * 2 tokens: select_verify.cu, the two-pass cluster kernel.
//  * 3-16 tokens and prefill: select_tc.cu on tcgen05, 8 tokens x 16 heads
//    per 128-row tile; with few tiles each tile's chunks are split over a
//    cluster.
#include "select_common.cuh"

namespace infllmv2 {

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

int select_tc_cluster_size(const Shape& s, int sc);
size_t select_tc_scratch_bytes(const Shape& s);
cudaError_t launch_select_tc(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map,
                             const SelParams& p, cudaStream_t st);
size_t select_decode_ncpad(const Shape& s);
bool select_decode_supported(const Shape& s);
cudaError_t launch_select_decode(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                                 const SelParams& p, cudaStream_t st);

int select_verify_cluster_size(const Shape& s);
cudaError_t launch_select_verify(const Shape& s, int cluster, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                                 const int32_t* kv_lens, int32_t* block_idx, int32_t* n_sel, float* r_buf,
                                 uint32_t* status, cudaStream_t st);

namespace {

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool use_decode_path(const Shape& s) { return s.nq <= kSelDecodeMaxNq && select_decode_supported(s); }

// Two tokens per sequence: the two-pass mma.sync cluster kernel (on a 128K
// cache 27 us against 32 us for the tensor-core tile, whose cost does not
// shrink with fewer rows); no workspace.
bool use_verify_path(const Shape& s) { return s.nq >= 2 && s.nq <= 8 && select_verify_cluster_size(s) > 0; }

// 3 to 16 tokens per sequence (speculative verification, short chunks): the
// tensor-core tile with its chunks split over a cluster, when such clusters
// fit the device (65 -> 32 us for 8 tokens on a 128K cache); no workspace.
bool use_tc_cluster(const Shape& s) {
  if (s.nq == 2 && use_verify_path(s)) return false;
  return s.nq >= 2 && s.nq <= kSelDecodeMaxNq && select_tc_supported(s) && select_tc_cluster_size(s, 0) > 1;
}

}  // namespace

bool select_supported(const Shape& s) { return use_decode_path(s) || select_tc_supported(s); }

size_t select_workspace_bytes(const Shape& s) {
  if (use_tc_cluster(s) || use_verify_path(s)) return 0;
  if (use_decode_path(s)) {
    const size_t units = static_cast<size_t>(s.B) * s.Hkv * s.nq;
    return align256(units * kGroup * select_decode_ncpad(s) * sizeof(float));
  }
  // The prefill path keeps everything on chip up to 4091 blocks of capacity;
  // past that its block scores take one slot per SM of a global scratch.
  return align256(select_tc_scratch_bytes(s));
}

cudaError_t launch_select(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& q_map,
                          const void* q, const int32_t* kv_lens, int32_t* block_idx,
                          int32_t* n_sel, float* block_scores, void* ws, uint32_t* status,
                          cudaStream_t st) {
  SelParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.ncmax = s.ncmax;
  p.nbmax = s.nbmax;
  p.kmax = s.kmax;
  p.topk = s.topk;
  p.n_init = s.n_init;
  p.n_local = s.n_local;
  p.inc_forced = s.inc_forced;
  p.scale2 = s.score_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.status = status;
  p.write_r = block_scores != nullptr;
  p.r_buf = block_scores;
  p.q = static_cast<const uint16_t*>(q);

  if (use_tc_cluster(s)) return launch_select_tc(s, kc_map, kc_map, p, st);
  if (use_verify_path(s))
    return launch_select_verify(s, select_verify_cluster_size(s), kc_map, q_map, kv_lens, block_idx, n_sel,
                                block_scores, status, st);
  if (use_decode_path(s)) {
    p.ncpad = static_cast<int>(select_decode_ncpad(s));
    p.z = static_cast<float*>(ws);
    return launch_select_decode(s, kc_map, q_map, p, st);
  }
  if (!select_tc_supported(s)) return cudaErrorInvalidConfiguration;   // rejected by the entry points
  p.r_scratch = static_cast<float*>(ws);
  return launch_select_tc(s, kc_map, kc_map, p, st);
}

cudaError_t launch_select_coarse(const Shape& s, const CUtensorMap& kc_map, const CUtensorMap& kcc_map, int sc,
                                 const void* q, const int32_t* kv_lens, int32_t* block_idx,
                                 int32_t* n_sel, float* block_scores, uint32_t* status, cudaStream_t st) {
  SelParams p{};
  p.B = s.B;
  p.Hkv = s.Hkv;
  p.Lmax = s.Lmax;
  p.nq = s.nq;
  p.ncmax = s.ncmax;
  p.nbmax = s.nbmax;
  p.kmax = s.kmax;
  p.topk = s.topk;
  p.n_init = s.n_init;
  p.n_local = s.n_local;
  p.inc_forced = s.inc_forced;
  p.scale2 = s.score_scale2;
  p.kv_lens = kv_lens;
  p.block_idx = block_idx;
  p.n_sel = n_sel;
  p.status = status;
  p.write_r = block_scores != nullptr;
  p.r_buf = block_scores;
  p.q = static_cast<const uint16_t*>(q);
  p.sc = sc;
  p.nccmax = s.Lmax / sc;
  if (!select_tc_onchip(s)) return cudaErrorInvalidConfiguration;   // rejected by the entry point
  return launch_select_tc(s, kc_map, kcc_map, p, st);
}

}  // namespace infllmv2
