// C-ABI layer of the InfLLM v2 library: argument checks, TMA tensor maps,
// workspace accounting and launches.  See include/infllmv2.h for the contract.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <mutex>
#include <string>

#include "infllmv2.h"
#include "common.cuh"
#include "kernels.h"

using namespace infllmv2;

// Device status word (INFLLMV2_DEVICE_* bits), one per device context.
static __device__ uint32_t g_device_status;

// Built-in scratch of infllmv2_select_blocks_static: 8 MiB that every device
// which loads the library keeps until the process exits.  Each call overwrites
// the part it reads before reading it (nothing has to start at zero); calls
// that overlap on the GPU share it and race.
static constexpr size_t kStaticSelectScratchBytes = static_cast<size_t>(8) << 20;
static __device__ __align__(256) unsigned char g_select_scratch[kStaticSelectScratchBytes];

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(INFLLMV2_CUDA_ERROR, "%s: %s", where, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

constexpr int kMaxDevices = 64;

// Fault-injection flags of the checked build's tests (infllmv2_test_hooks).
std::atomic<uint32_t> g_test_flags{0};

uint32_t* status_ptr() {
  static uint32_t* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

// Device address of the built-in selection scratch on the current device.  The
// host name of a __device__ array is only a stand-in, so the address is asked
// of the runtime once per device (on that device's first call) and cached.
void* static_select_scratch(cudaError_t* err) {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = (e != cudaSuccess) ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_select_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    ptrs[dev] = ptr;
  }
  return ptrs[dev];
}

// 2D bf16 view [rows, 128] with boxes of 64 columns x box_rows rows, 128-byte swizzle.
int make_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows, const char* what) {
  auto enc = encode_fn();
  if (!enc) return fail(INFLLMV2_CUDA_ERROR, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(INFLLMV2_CUDA_ERROR, "tensor map for %s failed (CUresult %d)", what, (int)r);
  return INFLLMV2_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_params(const infllmv2_params* p, int32_t n_q, Shape* s) {
  if (!p) return fail(INFLLMV2_INVALID_ARGUMENT, "params is NULL");
  if (p->batch < 1 || p->n_kv_heads < 1 || p->max_kv_len < 1)
    return fail(INFLLMV2_INVALID_ARGUMENT, "batch, n_kv_heads and max_kv_len must be >= 1");
  if (p->head_dim != kHeadDim || p->group_size != kGroup || p->block_size != kBlock ||
      p->kernel_size != kKernel || p->kernel_stride != kStride)
    return fail(INFLLMV2_UNSUPPORTED,
                "supported shape is head_dim 128, group 16, block 64, kernel 32, stride 16 "
                "(got %d, %d, %d, %d, %d)",
                p->head_dim, p->group_size, p->block_size, p->kernel_size, p->kernel_stride);
  if (n_q < 1 || n_q > p->max_kv_len)
    return fail(INFLLMV2_INVALID_ARGUMENT, "n_q = %d outside [1, max_kv_len = %d]", n_q, p->max_kv_len);
  if (p->topk < 1 || p->n_init_blocks < 0 || p->n_local_blocks < 0)
    return fail(INFLLMV2_INVALID_ARGUMENT, "topk must be >= 1 and forced block counts >= 0");
  if (p->topk_includes_forced != 0 && p->topk_includes_forced != 1)
    return fail(INFLLMV2_INVALID_ARGUMENT, "topk_includes_forced must be 0 or 1");
  if (p->topk_includes_forced && p->topk < p->n_init_blocks + p->n_local_blocks)
    return fail(INFLLMV2_INVALID_ARGUMENT, "topk %d < forced blocks %d", p->topk,
                p->n_init_blocks + p->n_local_blocks);
  if (!(std::isfinite(p->score_scale) && p->score_scale > 0.f && std::isfinite(p->attn_scale) &&
        p->attn_scale > 0.f))
    return fail(INFLLMV2_INVALID_ARGUMENT, "scales must be finite and > 0");
  const long long kmax = p->topk_includes_forced
                             ? p->topk
                             : static_cast<long long>(p->topk) + p->n_init_blocks + p->n_local_blocks;
  if (kmax > 4096) return fail(INFLLMV2_UNSUPPORTED, "at most 4096 selected blocks per query");
  if (static_cast<long long>(p->batch) * p->n_kv_heads > 65535)
    return fail(INFLLMV2_UNSUPPORTED, "batch * n_kv_heads must be <= 65535");
  const long long rows = static_cast<long long>(p->batch) * p->n_kv_heads * p->max_kv_len;
  if (rows * 2 > 0x7fffffffLL) return fail(INFLLMV2_UNSUPPORTED, "cache too large for 32-bit row indices");
  if (static_cast<long long>(p->batch) * n_q * p->n_kv_heads * kGroup > 0x7fffffffLL)
    return fail(INFLLMV2_UNSUPPORTED, "too many query rows");
  s->B = p->batch;
  s->Hkv = p->n_kv_heads;
  s->Lmax = p->max_kv_len;
  s->nq = n_q;
  s->ncmax = n_complete_kernels(p->max_kv_len);
  s->nbmax = (p->max_kv_len + kBlock - 1) / kBlock;
  s->kmax = static_cast<int>(kmax);
  s->topk = p->topk;
  s->n_init = p->n_init_blocks;
  s->n_local = p->n_local_blocks;
  s->inc_forced = p->topk_includes_forced;
  s->score_scale2 = p->score_scale * 1.4426950408889634f;
  s->attn_scale2 = p->attn_scale * 1.4426950408889634f;
  s->attn_scale = p->attn_scale;
  return INFLLMV2_OK;
}

size_t workspace_for(const Shape& s, int op) {
  switch (op) {
    case INFLLMV2_OP_SELECT:
      return select_workspace_bytes(s);
    case INFLLMV2_OP_DECODE:
      return attn_workspace_bytes(s, false);
    case INFLLMV2_OP_PREFILL:
      return attn_workspace_bytes(s, true);
    case INFLLMV2_OP_DECODE_STEP:
      return decode_step_cluster_size(s) ? 0 : select_workspace_bytes(s) + attn_workspace_bytes(s, false);
    case INFLLMV2_OP_BACKWARD:
      return attn_bwd_supported(s) ? attn_bwd_workspace_bytes(s) : 0;
    default:
      return 0;
  }
}

int attn_entry(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
               const void* v_cache, const int32_t* kv_lens, const int32_t* block_idx,
               const int32_t* n_selected, void* out, float* lse, void* workspace,
               size_t workspace_bytes, void* stream, bool prefill) {
  Shape s;
  int rc = check_params(p, n_q, &s);
  if (rc) return rc;
  if (!q || !k_cache || !v_cache || !kv_lens || !block_idx || !n_selected || !out)
    return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
  if (!prefill && n_q > kSelDecodeMaxNq)
    return fail(INFLLMV2_INVALID_ARGUMENT, "decode entry point takes n_q <= %d (got %d)", kSelDecodeMaxNq, n_q);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(INFLLMV2_UNSUPPORTED, "q, k_cache, v_cache and out must be 16-byte aligned");
  const size_t need = attn_workspace_bytes(s, prefill);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(INFLLMV2_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
  if (need > 0 && !aligned16(workspace)) return fail(INFLLMV2_UNSUPPORTED, "workspace must be 16-byte aligned");
  uint32_t* status = status_ptr();
  if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
  CUtensorMap qm, km, vm;
  const uint64_t kv_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.Lmax;
  if ((rc = make_map(&qm, q, static_cast<uint64_t>(s.B) * s.nq * s.Hkv * kGroup, 16, "q"))) return rc;
  if ((rc = make_map(&km, k_cache, kv_rows, 64, "k_cache"))) return rc;
  if ((rc = make_map(&vm, v_cache, kv_rows, 64, "v_cache"))) return rc;
  cudaError_t e =
      prefill ? launch_attn_tc(s, qm, km, vm, kv_lens, block_idx, n_selected, out, lse, status,
                               static_cast<cudaStream_t>(stream))
              : launch_attn(s, false, qm, km, vm, kv_lens, block_idx, n_selected, out, lse, workspace, status,
                            static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, prefill ? "sparse_attn_prefill" : "sparse_attn_decode");
  return INFLLMV2_OK;
}

}  // namespace

#define INFLLMV2_GUARD(...)                                                   \
  try {                                                                       \
    __VA_ARGS__;                                                              \
  } catch (...) {                                                             \
    return INFLLMV2_INVALID_ARGUMENT;                                         \
  }

extern "C" {

void infllmv2_default_params(infllmv2_params* p, int32_t batch, int32_t n_kv_heads, int32_t max_kv_len,
                             int32_t topk, int32_t topk_includes_forced) {
  if (!p) return;
  p->batch = batch;
  p->n_kv_heads = n_kv_heads;
  p->group_size = kGroup;
  p->head_dim = kHeadDim;
  p->block_size = kBlock;
  p->kernel_size = kKernel;
  p->kernel_stride = kStride;
  p->topk = topk;
  p->n_init_blocks = 1;
  p->n_local_blocks = 2;
  p->topk_includes_forced = topk_includes_forced;
  p->max_kv_len = max_kv_len;
  p->score_scale = 1.0f / std::sqrt(static_cast<float>(kHeadDim));
  p->attn_scale = p->score_scale;
}

int32_t infllmv2_max_selected(const infllmv2_params* p) {
  Shape s;
  if (check_params(p, 1, &s)) return -1;
  return s.kmax;
}

int32_t infllmv2_num_kernels(const infllmv2_params* p) {
  if (!p || p->max_kv_len < 0) return -1;
  return n_complete_kernels(p->max_kv_len);
}

size_t infllmv2_workspace_size(const infllmv2_params* p, int32_t n_q, int32_t op) {
  Shape s;
  if (check_params(p, n_q, &s)) return 0;
  if ((op == INFLLMV2_OP_DECODE || op == INFLLMV2_OP_DECODE_STEP) && n_q > kSelDecodeMaxNq) return 0;
  return workspace_for(s, op);
}

int infllmv2_compress_keys(const infllmv2_params* p, const void* k_cache, const int32_t* kv_lens,
                           int32_t kernel_begin, int32_t kernel_end, void* kc, void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, 1, &s);
    if (rc) return rc;
    if (!k_cache || !kv_lens || !kc) return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (!aligned16(k_cache) || !aligned16(kc))
      return fail(INFLLMV2_UNSUPPORTED, "k_cache and kc must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    cudaError_t e = launch_compress(s, k_cache, kv_lens, kernel_begin, kernel_end, kc, status,
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "compress_keys");
    return INFLLMV2_OK;
  });
}

int infllmv2_select_blocks(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                           const int32_t* kv_lens, int32_t* block_idx, int32_t* n_selected,
                           float* block_scores, void* workspace, size_t workspace_bytes, void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !kc || !kv_lens || !block_idx || !n_selected)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (!aligned16(q) || !aligned16(kc)) return fail(INFLLMV2_UNSUPPORTED, "q and kc must be 16-byte aligned");
    if (!select_supported(s))
      return fail(INFLLMV2_UNSUPPORTED,
                  "selection for n_q > 16: max_kv_len beyond the supported capacity (about 680K tokens)");
    const size_t need = select_workspace_bytes(s);
    if (need > 0 && (!workspace || workspace_bytes < need))
      return fail(INFLLMV2_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
    if (workspace && !aligned16(workspace)) return fail(INFLLMV2_UNSUPPORTED, "workspace must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap kcm, qm;
    if ((rc = make_map(&qm, q, static_cast<uint64_t>(s.B) * s.nq * s.Hkv * kGroup, 16, "q"))) return rc;
    if (s.ncmax > 0) {
      if ((rc = make_map(&kcm, kc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * s.ncmax, 64, "kc"))) return rc;
    } else {
      kcm = qm;  // no complete kernel fits in the cache: the map is never used
    }
    cudaError_t e = launch_select(s, kcm, qm, q, kv_lens, block_idx, n_selected, block_scores, workspace,
                                  status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "select_blocks");
    return INFLLMV2_OK;
  });
}

int infllmv2_select_blocks_static(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                                  const int32_t* kv_lens, int32_t* block_idx, int32_t* n_selected,
                                  float* block_scores, void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !kc || !kv_lens || !block_idx || !n_selected)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (!aligned16(q) || !aligned16(kc)) return fail(INFLLMV2_UNSUPPORTED, "q and kc must be 16-byte aligned");
    if (!select_supported(s))
      return fail(INFLLMV2_UNSUPPORTED,
                  "selection for n_q > 16: max_kv_len beyond the supported capacity (about 680K tokens)");
    const size_t need = select_workspace_bytes(s);
    if (need > kStaticSelectScratchBytes)
      return fail(INFLLMV2_WORKSPACE_TOO_SMALL,
                  "this selection needs %zu bytes of scratch; the built-in scratch holds %zu bytes "
                  "(use infllmv2_select_blocks with a caller workspace)",
                  need, kStaticSelectScratchBytes);
    void* scratch = nullptr;
    if (need > 0) {
      cudaError_t se = cudaSuccess;
      scratch = static_select_scratch(&se);
      if (!scratch) return cuda_fail(se, "select_blocks_static: address of the built-in scratch");
    }
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap kcm, qm;
    if ((rc = make_map(&qm, q, static_cast<uint64_t>(s.B) * s.nq * s.Hkv * kGroup, 16, "q"))) return rc;
    if (s.ncmax > 0) {
      if ((rc = make_map(&kcm, kc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * s.ncmax, 64, "kc"))) return rc;
    } else {
      kcm = qm;
    }
    cudaError_t e = launch_select(s, kcm, qm, q, kv_lens, block_idx, n_selected, block_scores, scratch, status,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "select_blocks_static");
    return INFLLMV2_OK;
  });
}

int infllmv2_coarse_means(const infllmv2_params* p, const void* k_cache, const int32_t* kv_lens, int32_t coarse,
                          void* kcc, void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, 1, &s);
    if (rc) return rc;
    if (!k_cache || !kv_lens || !kcc) return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (coarse < 32 || coarse > 4096 || coarse % kStride != 0)
      return fail(INFLLMV2_INVALID_ARGUMENT, "coarse window %d: a multiple of 16 in [32, 4096]", coarse);
    if (!aligned16(k_cache) || !aligned16(kcc))
      return fail(INFLLMV2_UNSUPPORTED, "k_cache and kcc must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    cudaError_t e = launch_coarse(s, k_cache, kv_lens, coarse, kcc, status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "coarse_means");
    return INFLLMV2_OK;
  });
}

int infllmv2_select_blocks_coarse_lse(const infllmv2_params* p, const void* q, int32_t n_q, const void* kc,
                                      int32_t coarse, const void* kcc, const int32_t* kv_lens,
                                      int32_t* block_idx, int32_t* n_selected, float* block_scores,
                                      void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !kc || !kcc || !kv_lens || !block_idx || !n_selected)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (coarse < 32 || coarse > 4096 || coarse % kStride != 0)
      return fail(INFLLMV2_INVALID_ARGUMENT, "coarse window %d: a multiple of 16 in [32, 4096]", coarse);
    if (n_q <= kSelDecodeMaxNq)
      return fail(INFLLMV2_UNSUPPORTED,
                  "the coarse LSE applies to the prefill path (n_q > %d); the decode path already "
                  "computes the exact LSE in one pass",
                  kSelDecodeMaxNq);
    if (!aligned16(q) || !aligned16(kc) || !aligned16(kcc))
      return fail(INFLLMV2_UNSUPPORTED, "q, kc and kcc must be 16-byte aligned");
    if (s.ncmax < 1 || s.Lmax / coarse < 1)
      return fail(INFLLMV2_UNSUPPORTED, "max_kv_len must hold a kernel and a coarse window");
    if (!select_tc_onchip(s))
      return fail(INFLLMV2_UNSUPPORTED,
                  "the coarse-LSE selection keeps 8 tokens' block scores on chip: max_kv_len up to 327360");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap kcm, kccm;
    if ((rc = make_map(&kcm, kc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * s.ncmax, 64, "kc"))) return rc;
    if ((rc = make_map(&kccm, kcc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * (s.Lmax / coarse), 64, "kcc")))
      return rc;
    cudaError_t e = launch_select_coarse(s, kcm, kccm, coarse, q, kv_lens, block_idx, n_selected, block_scores,
                                         status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "select_blocks_coarse_lse");
    return INFLLMV2_OK;
  });
}

int infllmv2_sparse_attn_decode(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                                const void* v_cache, const int32_t* kv_lens, const int32_t* block_idx,
                                const int32_t* n_selected, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  INFLLMV2_GUARD(return attn_entry(p, q, n_q, k_cache, v_cache, kv_lens, block_idx, n_selected, out, lse,
                                   workspace, workspace_bytes, stream, false));
}

int infllmv2_sparse_attn_prefill(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                                 const void* v_cache, const int32_t* kv_lens, const int32_t* block_idx,
                                 const int32_t* n_selected, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  INFLLMV2_GUARD(return attn_entry(p, q, n_q, k_cache, v_cache, kv_lens, block_idx, n_selected, out, lse,
                                   workspace, workspace_bytes, stream, true));
}

int infllmv2_append_kv(const infllmv2_params* p, int32_t n_q, const void* k_new, const void* v_new,
                       const int32_t* kv_lens, void* k_cache, void* v_cache, const void* q_src, void* q_dst,
                       void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!k_new || !v_new || !kv_lens || !k_cache || !v_cache)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
      return fail(INFLLMV2_UNSUPPORTED, "k_new, v_new, k_cache and v_cache must be 16-byte aligned");
    if ((q_src == nullptr) != (q_dst == nullptr))
      return fail(INFLLMV2_INVALID_ARGUMENT, "q_src and q_dst are given together or not at all");
    if ((q_src && !aligned16(q_src)) || (q_dst && !aligned16(q_dst)))
      return fail(INFLLMV2_UNSUPPORTED, "q_src and q_dst must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    cudaError_t e = launch_append(s, k_new, v_new, kv_lens, k_cache, v_cache, q_src, q_dst, status,
                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append_kv");
    return INFLLMV2_OK;
  });
}

int infllmv2_decode_step(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                         const void* v_cache, const int32_t* kv_lens, void* kc, int32_t* block_idx,
                         int32_t* n_selected, void* out, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !kv_lens || !kc || !block_idx || !n_selected || !out)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (n_q > kSelDecodeMaxNq)
      return fail(INFLLMV2_INVALID_ARGUMENT, "decode_step takes n_q <= %d (got %d)", kSelDecodeMaxNq, n_q);
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(kc) || !aligned16(out))
      return fail(INFLLMV2_UNSUPPORTED, "q, k_cache, v_cache, kc and out must be 16-byte aligned");
    if (s.ncmax < 1) return fail(INFLLMV2_UNSUPPORTED, "max_kv_len must hold at least one semantic kernel");
    const int cluster = decode_step_cluster_size(s);
    if (!cluster && !select_supported(s))
      return fail(INFLLMV2_UNSUPPORTED,
                  "selection for n_q > 16: max_kv_len beyond the supported capacity (about 680K tokens)");
    const size_t need = cluster ? 0 : select_workspace_bytes(s) + attn_workspace_bytes(s, false);
    if (need > 0 && (!workspace || workspace_bytes < need))
      return fail(INFLLMV2_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
    if (need > 0 && !aligned16(workspace)) return fail(INFLLMV2_UNSUPPORTED, "workspace must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap qm, kcm, km, vm;
    const uint64_t kv_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.Lmax;
    if ((rc = make_map(&qm, q, static_cast<uint64_t>(s.B) * s.nq * s.Hkv * kGroup, 16, "q"))) return rc;
    if ((rc = make_map(&kcm, kc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * s.ncmax, 64, "kc"))) return rc;
    if ((rc = make_map(&km, k_cache, kv_rows, 64, "k_cache"))) return rc;
    if ((rc = make_map(&vm, v_cache, kv_rows, 64, "v_cache"))) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (cluster) {
      e = launch_decode_step(s, cluster, kcm, qm, km, vm, k_cache, kv_lens, kc, block_idx, n_selected, out, lse,
                             nullptr, status, g_test_flags.load(), st);
      if (e != cudaSuccess) return cuda_fail(e, "decode_step");
      return INFLLMV2_OK;
    }
    // Kernels ending inside the last n_q tokens: at most n_q / 16 + 1 of them.
    e = launch_compress(s, k_cache, kv_lens, -(n_q / kStride + 1), -1, kc, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step (compress)");
    const size_t sel_ws = select_workspace_bytes(s);
    e = launch_select(s, kcm, qm, q, kv_lens, block_idx, n_selected, nullptr, workspace, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step (select)");
    e = launch_attn(s, false, qm, km, vm, kv_lens, block_idx, n_selected, out, lse,
                    static_cast<unsigned char*>(workspace) + sel_ws, status, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step (attend)");
    return INFLLMV2_OK;
  });
}

int infllmv2_append_decode_step(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_new,
                                const void* v_new, void* k_cache, void* v_cache, const int32_t* kv_lens, void* kc,
                                int32_t* block_idx, int32_t* n_selected, void* out, float* lse, void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !kv_lens || !kc || !block_idx || !n_selected || !out)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (n_q != 1)
      return fail(INFLLMV2_UNSUPPORTED,
                  "append_decode_step takes n_q = 1 (got %d): use infllmv2_append_kv and infllmv2_decode_step", n_q);
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(kc) || !aligned16(out))
      return fail(INFLLMV2_UNSUPPORTED, "q, k_new, v_new, k_cache, v_cache, kc and out must be 16-byte aligned");
    if (s.ncmax < 1) return fail(INFLLMV2_UNSUPPORTED, "max_kv_len must hold at least one semantic kernel");
    const int cluster = decode_step_cluster_size(s);
    if (!cluster)
      return fail(INFLLMV2_UNSUPPORTED,
                  "the one-launch step does not fit this shape: use infllmv2_append_kv and infllmv2_decode_step");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap kcm, km, vm;
    const uint64_t kv_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.Lmax;
    if ((rc = make_map(&kcm, kc, static_cast<uint64_t>(s.B) * s.Hkv * 2 * s.ncmax, 64, "kc"))) return rc;
    if ((rc = make_map(&km, k_cache, kv_rows, 64, "k_cache"))) return rc;
    if ((rc = make_map(&vm, v_cache, kv_rows, 64, "v_cache"))) return rc;
    const DsAppend app{q, k_new, v_new, k_cache, v_cache};
    // q is read with ordinary loads (it may sit in host memory): the q map
    // slot of the kernel takes the key map, which it then leaves unused.
    cudaError_t e = launch_decode_step(s, cluster, kcm, km, km, vm, k_cache, kv_lens, kc, block_idx, n_selected,
                                       out, lse, &app, status, g_test_flags.load(), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append_decode_step");
    return INFLLMV2_OK;
  });
}

int infllmv2_sparse_attn_backward(const infllmv2_params* p, const void* q, int32_t n_q, const void* k_cache,
                                  const void* v_cache, const int32_t* kv_lens, const int32_t* block_idx,
                                  const int32_t* n_selected, const void* out, const float* lse, const void* dout,
                                  float* dq, float* dk, float* dv, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  INFLLMV2_GUARD({
    Shape s;
    int rc = check_params(p, n_q, &s);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !kv_lens || !block_idx || !n_selected || !out || !lse || !dout || !dq ||
        !dk || !dv)
      return fail(INFLLMV2_INVALID_ARGUMENT, "a required pointer is NULL");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse))
      return fail(INFLLMV2_UNSUPPORTED, "tensor pointers must be 16-byte aligned");
    if (!attn_bwd_supported(s)) return fail(INFLLMV2_UNSUPPORTED, "too many (query, block) pairs for the index");
    const size_t need = attn_bwd_workspace_bytes(s);
    if (!workspace || workspace_bytes < need)
      return fail(INFLLMV2_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes (got %zu)", need, workspace_bytes);
    if (!aligned16(workspace)) return fail(INFLLMV2_UNSUPPORTED, "workspace must be 16-byte aligned");
    uint32_t* status = status_ptr();
    if (!status) return fail(INFLLMV2_CUDA_ERROR, "no device status word (no current CUDA device?)");
    CUtensorMap qm, dom, km, vm, km16, vm16;
    const uint64_t kv_rows = static_cast<uint64_t>(s.B) * s.Hkv * s.Lmax;
    const uint64_t q_rows = static_cast<uint64_t>(s.B) * s.nq * s.Hkv * kGroup;
    if ((rc = make_map(&qm, q, q_rows, 16, "q"))) return rc;
    if ((rc = make_map(&dom, dout, q_rows, 16, "dout"))) return rc;
    if ((rc = make_map(&km, k_cache, kv_rows, 64, "k_cache"))) return rc;
    if ((rc = make_map(&vm, v_cache, kv_rows, 64, "v_cache"))) return rc;
    if ((rc = make_map(&km16, k_cache, kv_rows, 16, "k_cache"))) return rc;
    if ((rc = make_map(&vm16, v_cache, kv_rows, 16, "v_cache"))) return rc;
    cudaError_t e = launch_attn_bwd(s, qm, dom, km, vm, km16, vm16, q, kv_lens, block_idx, n_selected, out, lse,
                                    dout, dq, dk, dv, workspace, status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_attn_backward");
    return INFLLMV2_OK;
  });
}

const char* infllmv2_status_string(int status) {
  switch (status) {
    case INFLLMV2_OK:
      return "INFLLMV2_OK";
    case INFLLMV2_INVALID_ARGUMENT:
      return "INFLLMV2_INVALID_ARGUMENT";
    case INFLLMV2_UNSUPPORTED:
      return "INFLLMV2_UNSUPPORTED";
    case INFLLMV2_WORKSPACE_TOO_SMALL:
      return "INFLLMV2_WORKSPACE_TOO_SMALL";
    case INFLLMV2_CUDA_ERROR:
      return "INFLLMV2_CUDA_ERROR";
    default:
      return "INFLLMV2_UNKNOWN_STATUS";
  }
}

const char* infllmv2_last_error(void) { return g_last_error.c_str(); }

int infllmv2_test_hooks(uint32_t flags) {
  INFLLMV2_GUARD({
#ifdef INFLLMV2_CHECKED
    g_test_flags.store(flags);
    return INFLLMV2_OK;
#else
    (void)flags;
    return fail(INFLLMV2_UNSUPPORTED, "test hooks exist only in the checked build (INFLLMV2_CHECKED)");
#endif
  });
}

int infllmv2_is_checked_build(void) {
#ifdef INFLLMV2_CHECKED
  return 1;
#else
  return 0;
#endif
}

int infllmv2_get_device_status(uint32_t* status_out, int clear) {
  INFLLMV2_GUARD({
    if (!status_out) return fail(INFLLMV2_INVALID_ARGUMENT, "status_out is NULL");
    cudaError_t e = cudaMemcpyFromSymbol(status_out, g_device_status, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "get_device_status");
    if (clear) {
      const uint32_t zero = 0;
      e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(uint32_t));
      if (e != cudaSuccess) return cuda_fail(e, "get_device_status(clear)");
    }
    return INFLLMV2_OK;
  });
}

}  // extern "C"
